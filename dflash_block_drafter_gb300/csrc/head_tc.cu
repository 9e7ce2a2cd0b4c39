// LM head + argmax of a 128-row pass (9..16 sequences of 8 block rows) on the
// tcgen05 tensor cores.  At 128 activation rows the head is a real GEMM
// (logits[128, V] = X[128, H] . W_head[V, H]^T, X as BF16 hi and lo planes):
// the legacy mma.sync GEMV spends most of its time issuing MMAs there, while
// here one thread issues 128 x 256 x 16 MMAs and the pass is bound by the
// 778 MB stream of the head again.
//
// Per CTA: a contiguous range of 256-row vocabulary chunks.  Warp 0 streams,
// per 64-input k-block, the chunk's W box (256 x 64, four 64 x 64 tensor-map
// boxes) and the two X planes (128 x 64 each; the same for every CTA, read
// from L2) into a 3-stage ring; warp 1 allocates 512 TMEM columns and issues
// the MMAs, chunk c accumulating into columns (c % 2) * 256 .. + 256 (A = X:
// TMEM lane = activation row, B = W: column = vocabulary row); warps 2..5
// read a finished accumulator back (one activation row per thread, 256
// logits), keep the row's best (logit, id) and, for the confidence gate,
// its running (max, sum of exp), and hand the columns back.  Each CTA then
// folds its keys into one global packed key per row with a 64-bit atomicMax
// (exact and order-free: keys are order-preserving logit bits over
// 0xffffffff - id, so ties go to the lowest id); the CTA that arrives last
// writes the drafts (and confidences) exactly like the GEMV head, and clears
// the keys and its counter for the next launch.
#include "kernels.h"
#include "common.cuh"
#include "layout.cuh"

namespace dflash {

namespace {

constexpr int kHtRows = 128;                          // activation rows (MMA M)
constexpr int kHtN = 256;                             // vocabulary rows per chunk (MMA N)
constexpr int kHtKB = 64;                             // inputs per k-block (one 128-byte swizzle atom row)
constexpr int kHtStages = 3;
constexpr int kHtXBytes = kHtRows * 128;              // one X plane box: 16 KB
constexpr int kHtWBytes = kHtN * 128;                 // the chunk's W boxes: 32 KB
constexpr int kHtStage = 2 * kHtXBytes + kHtWBytes;   // 64 KB
constexpr int kHtThreads = 192;
constexpr int kHtSmem = 1024 + kHtStages * kHtStage + 1024;

// Instruction descriptor of kind::f16 with BF16 A and B (K-major), FP32
// accumulation, shape M x N.
constexpr uint32_t umma_idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ unsigned long long head_key(float v, int id) {
  return (static_cast<unsigned long long>(float_order_key(v)) << 32) |
         static_cast<unsigned long long>(0xffffffffu - static_cast<uint32_t>(id));
}

__global__ void __launch_bounds__(kHtThreads, 1) head_tc_kernel(const __grid_constant__ HeadTcArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + kHtStages * kHtStage);
  uint64_t* empty = full + kHtStages;
  uint64_t* accf = empty + kHtStages;  // [2] accumulator b complete
  uint64_t* acce = accf + 2;           // [2] accumulator b read back
  uint64_t* mdone = acce + 2;          // every MMA of the CTA has completed
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(mdone + 1);
  int* s_flag = reinterpret_cast<int*>(s_tmem + 1);
  float* s_prob = reinterpret_cast<float*>(s_flag + 4);  // [128]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = static_cast<int>(gridDim.x);
  const int NV = (a.V + kHtN - 1) / kHtN;
  const int c0 = static_cast<int>(static_cast<long long>(blockIdx.x) * NV / G);
  const int c1 = static_cast<int>(static_cast<long long>(blockIdx.x + 1) * NV / G);
  const int nch = c1 - c0;
  const int KB = a.H / kHtKB;

  if (tid == 0) {
    for (int s = 0; s < kHtStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accf[b], 1);
      mbar_init(&acce[b], 4);
    }
    mbar_init(mdone, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(s_tmem, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  bool ok = true;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && nch > 0) {
      prefetch_tensormap(&a.wmap);
      prefetch_tensormap(&a.xmap);
      const uint64_t pol = l2_policy_evict_first();
      const int total = nch * KB;
      auto issue_w = [&](int it) {
        const int s = it % kHtStages, ch = c0 + it / KB, kb = it % KB;
        uint8_t* dst = ring + s * kHtStage + 2 * kHtXBytes;
        for (int b = 0; b < kHtN / 64; ++b)
          tma_load_2d_hint(dst + b * 8192, &a.wmap, kb * kHtKB, ch * kHtN + b * 64, &full[s], pol);
      };
      auto issue_x = [&](int it) {
        const int s = it % kHtStages, kb = it % KB;
        uint8_t* dst = ring + s * kHtStage;
        tma_load_2d(dst, &a.xmap, kb * kHtKB, 0, &full[s]);
        tma_load_2d(dst + kHtXBytes, &a.xmap, kb * kHtKB, kHtRows, &full[s]);
      };
      const int npre = total < kHtStages ? total : kHtStages;
      // the head's boxes do not depend on the previous kernel; the rows do
      for (int it = 0; it < npre; ++it) {
        mbar_arrive_expect_tx(&full[it], kHtStage);
        issue_w(it);
      }
      pdl_wait();
      for (int it = 0; it < npre; ++it) issue_x(it);
      int issued = npre;
      for (int it = npre; it < total; ++it) {
        const int s = it % kHtStages;
        if (!mbar_wait(&empty[s], ((it / kHtStages) - 1) & 1)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&full[s], kHtStage);
        issue_w(it);
        issue_x(it);
        issued = it + 1;
      }
      // every issued copy lands before the CTA may exit
      for (int it = (issued > kHtStages ? issued - kHtStages : 0); it < issued; ++it)
        if (!mbar_wait(&full[it % kHtStages], (it / kHtStages) & 1)) {
          ok = false;
          break;
        }
      if (!ok) set_status(a.status, DFLASH_DEV_TIMEOUT);
    } else if (lane == 0) {
      pdl_wait();
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && nch > 0) {
      constexpr uint32_t idesc = umma_idesc_bf16(kHtRows, kHtN);
      int it = 0;
      for (int lc = 0; lc < nch && ok; ++lc) {
        const int b = lc & 1;
        if (lc >= 2 && !mbar_wait(&acce[b], ((lc >> 1) - 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int s = it % kHtStages;
          if (!mbar_wait(&full[s], (it / kHtStages) & 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t xs = smem_u32(ring + s * kHtStage), ws = xs + 2 * kHtXBytes;
#pragma unroll
          for (int ks = 0; ks < kHtKB / 16; ++ks) {
            const uint64_t db = umma_desc_sw128(ws + ks * 32, 16, 1024);
            umma_f16(tmem + b * kHtN, umma_desc_sw128(xs + ks * 32, 16, 1024), db, idesc, (kb | ks) ? 1u : 0u);
            umma_f16(tmem + b * kHtN, umma_desc_sw128(xs + kHtXBytes + ks * 32, 16, 1024), db, idesc, 1u);
          }
          umma_commit(&empty[s]);
        }
        if (!ok) break;
        umma_commit(&accf[b]);
      }
      // tensor memory may only be freed once every issued MMA has finished
      umma_commit(mdone);
      if (!mbar_wait(mdone, 0)) ok = false;
      if (!ok) set_status(a.status, DFLASH_DEV_TIMEOUT);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    pdl_launch_dependents();
    constexpr float LOG2E = 1.4426950408889634f;
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int r = q * 32 + lane;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(q * 32) << 16);
    const bool sums = a.min_p > 0.f;
    const bool live = r < a.n_seq * 8;
    float best = -INFINITY, m_run = -INFINITY, s_run = 0.f;
    int bid = 0x7fffffff;
    bool bad = false;
    for (int lc = 0; lc < nch; ++lc) {
      const int b = lc & 1;
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&accf[b], (lc >> 1) & 1));
      tc_fence_after();
      const int vbase = (c0 + lc) * kHtN;
#pragma unroll 1
      for (int cc = 0; cc < kHtN / 32; ++cc) {
        uint32_t v32[32];
        tmem_ld32(lane_addr + b * kHtN + cc * 32, v32);
        tmem_wait_ld();
        tmem_reg_fence(v32);
        // ids ascend: a strictly larger logit replaces the best, so ties keep the lowest id
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int id = vbase + cc * 32 + e;
          const float v = __uint_as_float(v32[e]);
          if (id < a.V) {
            if (!isfinite(v)) {
              bad = true;
            } else {
              if (v > best) {
                best = v;
                bid = id;
              }
              if (sums) {
                if (v > m_run) {
                  s_run = s_run * ex2_approx((m_run - v) * LOG2E) + 1.f;
                  m_run = v;
                } else {
                  s_run += ex2_approx((v - m_run) * LOG2E);
                }
              }
            }
          }
        }
      }
      // the accumulator has been read: the chunk after next may overwrite it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acce[b]);
    }
    if (!ok && lane == 0) set_status(a.status, DFLASH_DEV_TIMEOUT);
    if (live) {
      if (bad) set_status(a.status, DFLASH_DEV_NONFINITE);
      if (bid != 0x7fffffff) atomicMax(a.keys + r, head_key(best, bid));
    }
    if (sums) __stcg(a.ms + static_cast<size_t>(blockIdx.x) * kHtRows + r, make_float2(m_run, s_run));
    named_bar_sync(1, 128);
    if (r == 0) s_flag[0] = (atomic_add_acq_rel(a.grid_cnt, 1) == G - 1);
    named_bar_sync(1, 128);
    if (s_flag[0]) {
      // the last CTA: every other CTA's keys and sums are visible (acquire above)
      const unsigned long long k = __ldcg(a.keys + r);
      float prob = -1.f;
      if (sums) {
        float mg = -INFINITY;
        for (int c = 0; c < G; ++c) {
          const float2 v = __ldcg(a.ms + static_cast<size_t>(c) * kHtRows + r);
          if (v.y > 0.f) mg = fmaxf(mg, v.x);
        }
        float S = 0.f;
        for (int c = 0; c < G; ++c) {
          const float2 v = __ldcg(a.ms + static_cast<size_t>(c) * kHtRows + r);
          if (v.y > 0.f) S += v.y * ex2_approx((v.x - mg) * LOG2E);
        }
        prob = S > 0.f ? 1.f / S : 0.f;
      }
      s_prob[r] = prob;
      named_bar_sync(1, 128);
      const int s = r >> 3, i = r & 7;
      if (s < a.n_seq && i >= 1) {
        int B = a.block_len[s];
        B = B < DFLASH_MIN_BLOCK ? DFLASH_MIN_BLOCK : (B > DFLASH_MAX_BLOCK ? DFLASH_MAX_BLOCK : B);
        int out = -1;
        float pr = -1.f;
        if (i < B) {
          if (k == 0ull) {
            set_status(a.status, DFLASH_DEV_NONFINITE);
          } else {
            out = static_cast<int>(0xffffffffu - static_cast<uint32_t>(k & 0xffffffffull));
            if (sums) {
              pr = s_prob[r];
              // offered only if no draft of the block up to this one is below the floor
              for (int i2 = 1; i2 <= i; ++i2)
                if (s_prob[s * 8 + i2] < a.min_p) out = -1;
            }
          }
        }
        a.drafts[s * (DFLASH_MAX_BLOCK - 1) + (i - 1)] = out;
        if (a.probs) a.probs[s * (DFLASH_MAX_BLOCK - 1) + (i - 1)] = pr;
      }
      a.keys[r] = 0ull;
      if (r == 0) *a.grid_cnt = 0;
    }
  }
  // release the tensor memory once every tcgen05 operation of the CTA is done
  // every warp whole again (lanes that finished their role early wait for
  // the one still working) before the CTA-wide barrier
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------
// The LM head of an 8-row pass (one sequence) on tcgen05: A = 128 vocabulary
// rows of the head (two 64 x 64 boxes per 64-input k-block), B = the 16 rows
// hi(0..7), lo(0..7) of the packed activations (one 64 x 16 box: the two
// planes of a chunk are adjacent 8-row blocks), MMA 128 x 16 x 16, so one
// accumulator column pair (r, 8 + r) holds row r's two planes.  The head
// stream is the whole cost (the MMAs are ~1 % of it): a lean consumer lets it
// run at the copy rate.  Per CTA a contiguous range of 128-row vocabulary
// chunks; warp 0 streams them through a 10-stage ring, warp 1 issues the
// MMAs into two 16-column accumulators, warps 2..5 (thread = vocabulary row)
// read a finished chunk back, divide by each row's RMS and keep per row the
// best (logit, id) and the gate's running (max, sum of exp); the CTA then
// reduces over its threads and folds its keys into the global keys, and the
// CTA that arrives last writes the drafts, as the 128-row head does.
constexpr int kH8Rows = 128;                       // vocabulary rows per chunk (MMA M)
constexpr int kH8Stages = 10;
constexpr int kH8WBytes = kH8Rows * 128;           // 16 KB
constexpr int kH8XBytes = 16 * 128;                // 2 KB
constexpr int kH8Stage = kH8WBytes + kH8XBytes;   // 18 KB (a multiple of 1024)
constexpr int kH8Smem = 1024 + kH8Stages * kH8Stage + 1024;

__global__ void __launch_bounds__(kHtThreads, 1) head_tc8_kernel(const __grid_constant__ HeadTcArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + kH8Stages * kH8Stage);
  uint64_t* empty = full + kH8Stages;
  uint64_t* accf = empty + kH8Stages;  // [2]
  uint64_t* acce = accf + 2;           // [2]
  uint64_t* mdone = acce + 2;
  // 8-byte members first (after the barriers, 8-byte aligned), then 4-byte ones
  unsigned long long* s_key = reinterpret_cast<unsigned long long*>(mdone + 1);  // [4 warps][8]
  float2* s_ms = reinterpret_cast<float2*>(s_key + 32);                           // [4 warps][8]
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(s_ms + 32);
  int* s_flag = reinterpret_cast<int*>(s_tmem + 1);
  float* s_rs = reinterpret_cast<float*>(s_flag + 4);    // [8]
  float* s_prob = reinterpret_cast<float*>(s_rs + 8);    // [8]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = static_cast<int>(gridDim.x);
  const int NV = (a.V + kH8Rows - 1) / kH8Rows;
  const int c0 = static_cast<int>(static_cast<long long>(blockIdx.x) * NV / G);
  const int c1 = static_cast<int>(static_cast<long long>(blockIdx.x + 1) * NV / G);
  const int nch = c1 - c0;
  const int KB = a.H / kHtKB;

  if (tid == 0) {
    for (int s = 0; s < kH8Stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accf[b], 1);
      mbar_init(&acce[b], 4);
    }
    mbar_init(mdone, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(s_tmem, 32);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  bool ok = true;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && nch > 0) {
      prefetch_tensormap(&a.wmap);
      prefetch_tensormap(&a.xmap);
      const uint64_t pol = l2_policy_evict_first();
      const int total = nch * KB;
      auto issue_w = [&](int it) {
        const int s = it % kH8Stages, ch = c0 + it / KB, kb = it % KB;
        uint8_t* dst = ring + s * kH8Stage;
        tma_load_2d_hint(dst, &a.wmap, kb * kHtKB, ch * kH8Rows, &full[s], pol);
        tma_load_2d_hint(dst + 8192, &a.wmap, kb * kHtKB, ch * kH8Rows + 64, &full[s], pol);
      };
      auto issue_x = [&](int it) {
        const int s = it % kH8Stages, kb = it % KB;
        // chunk kb / 2 of 128 inputs: its hi and lo planes are rows 16 (kb / 2) .. + 15
        tma_load_2d(ring + s * kH8Stage + kH8WBytes, &a.xmap, (kb & 1) * kHtKB, (kb >> 1) * 16, &full[s]);
      };
      const int npre = total < kH8Stages ? total : kH8Stages;
      for (int it = 0; it < npre; ++it) {
        mbar_arrive_expect_tx(&full[it], kH8Stage);
        issue_w(it);
      }
      pdl_wait();  // the packed rows come from the previous kernel
      for (int it = 0; it < npre; ++it) issue_x(it);
      int issued = npre;
      for (int it = npre; it < total; ++it) {
        const int s = it % kH8Stages;
        if (!mbar_wait(&empty[s], ((it / kH8Stages) - 1) & 1)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&full[s], kH8Stage);
        issue_w(it);
        issue_x(it);
        issued = it + 1;
      }
      for (int it = (issued > kH8Stages ? issued - kH8Stages : 0); it < issued; ++it)
        if (!mbar_wait(&full[it % kH8Stages], (it / kH8Stages) & 1)) {
          ok = false;
          break;
        }
      if (!ok) set_status(a.status, DFLASH_DEV_TIMEOUT);
    } else if (lane == 0) {
      pdl_wait();
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && nch > 0) {
      constexpr uint32_t idesc = umma_idesc_bf16(kH8Rows, 16);
      int it = 0;
      for (int lc = 0; lc < nch && ok; ++lc) {
        const int b = lc & 1;
        if (lc >= 2 && !mbar_wait(&acce[b], ((lc >> 1) - 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int kb = 0; kb < KB; ++kb, ++it) {
          const int s = it % kH8Stages;
          if (!mbar_wait(&full[s], (it / kH8Stages) & 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t ws = smem_u32(ring + s * kH8Stage), xs = ws + kH8WBytes;
#pragma unroll
          for (int ks = 0; ks < kHtKB / 16; ++ks)
            umma_f16(tmem + b * 16, umma_desc_sw128(ws + ks * 32, 16, 1024), umma_desc_sw128(xs + ks * 32, 16, 1024),
                     idesc, (kb | ks) ? 1u : 0u);
          umma_commit(&empty[s]);
        }
        if (!ok) break;
        umma_commit(&accf[b]);
      }
      umma_commit(mdone);
      if (!mbar_wait(mdone, 0)) ok = false;
      if (!ok) set_status(a.status, DFLASH_DEV_TIMEOUT);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    constexpr float LOG2E = 1.4426950408889634f;
    const int et = tid - 64;   // 0..127
    const int q = warp & 3;    // TMEM lane quarter
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(q * 32) << 16);
    const bool sums = a.min_p > 0.f;
    pdl_wait();  // the sums of squares (and x) come from the previous kernel
    pdl_launch_dependents();
    if (et < 8) {
      float ss = 0.f;
      for (int g = 0; g < a.H / 64; ++g) ss += __ldcg(a.ssq + g * 8 + et);
      s_rs[et] = rsqrtf(ss / a.H + a.eps);
    }
    named_bar_sync(1, 128);
    float rs[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) rs[r] = s_rs[r];
    if (a.final_hidden && blockIdx.x == 0)
      for (int i = et; i < 8 * a.H; i += 128) {
        const int r = i / a.H, k = i - r * a.H;
        a.final_hidden[i] = __ldcg(a.x + i) * rs[r] * a.norm_w[k];
      }
    float best[8], m_run[8], s_run[8];
    int bid[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      best[r] = -INFINITY;
      bid[r] = 0x7fffffff;
      m_run[r] = -INFINITY;
      s_run[r] = 0.f;
    }
    bool bad = false;
    for (int lc = 0; lc < nch; ++lc) {
      const int b = lc & 1;
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&accf[b], (lc >> 1) & 1));
      tc_fence_after();
      uint32_t v16[16];
      tmem_ld16(lane_addr + b * 16, v16);
      tmem_wait_ld();
      tmem_reg_fence(v16);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acce[b]);
      const int id = (c0 + lc) * kH8Rows + q * 32 + lane;
      if (id < a.V) {
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          const float v = (__uint_as_float(v16[r]) + __uint_as_float(v16[8 + r])) * rs[r];
          if (!isfinite(v)) {
            bad = true;
          } else {
            if (v > best[r]) {  // a thread's ids ascend: ties keep the lowest
              best[r] = v;
              bid[r] = id;
            }
            if (sums) {
              if (v > m_run[r]) {
                s_run[r] = s_run[r] * ex2_approx((m_run[r] - v) * LOG2E) + 1.f;
                m_run[r] = v;
              } else {
                s_run[r] += ex2_approx((v - m_run[r]) * LOG2E);
              }
            }
          }
        }
      }
    }
    if (!ok && lane == 0) set_status(a.status, DFLASH_DEV_TIMEOUT);
    if (__any_sync(0xffffffffu, bad) && lane == 0) set_status(a.status, DFLASH_DEV_NONFINITE);
    // the CTA's best key and (max, sum) per row: over the warp, then the 4 warps in order
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      unsigned long long k = bid[r] != 0x7fffffff ? head_key(best[r], bid[r]) : 0ull;
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        const unsigned long long k2 = __shfl_xor_sync(0xffffffffu, k, o);
        k = k2 > k ? k2 : k;
      }
      if (lane == 0) s_key[(warp - 2) * 8 + r] = k;
      if (sums) {
        float m = m_run[r], sm = s_run[r];
#pragma unroll
        for (int o = 16; o; o >>= 1) {
          const float m2 = __shfl_xor_sync(0xffffffffu, m, o), s2 = __shfl_xor_sync(0xffffffffu, sm, o);
          const float mx = fmaxf(m, m2);
          sm = (sm > 0.f ? sm * ex2_approx((m - mx) * LOG2E) : 0.f) + (s2 > 0.f ? s2 * ex2_approx((m2 - mx) * LOG2E) : 0.f);
          m = mx;
        }
        if (lane == 0) s_ms[(warp - 2) * 8 + r] = make_float2(m, sm);
      }
    }
    named_bar_sync(1, 128);
    if (et < 8) {
      unsigned long long k = 0ull;
      float m = -INFINITY, sm = 0.f;
      for (int w4 = 0; w4 < 4; ++w4) {
        const unsigned long long k2 = s_key[w4 * 8 + et];
        k = k2 > k ? k2 : k;
        if (sums) {
          const float2 v = s_ms[w4 * 8 + et];
          if (v.y > 0.f) {
            const float mx = fmaxf(m, v.x);
            sm = (sm > 0.f ? sm * ex2_approx((m - mx) * LOG2E) : 0.f) + v.y * ex2_approx((v.x - mx) * LOG2E);
            m = mx;
          }
        }
      }
      if (k) atomicMax(a.keys + et, k);
      if (sums) __stcg(a.ms + static_cast<size_t>(blockIdx.x) * 8 + et, make_float2(m, sm));
    }
    named_bar_sync(1, 128);
    if (et == 0) s_flag[0] = (atomic_add_acq_rel(a.grid_cnt, 1) == G - 1);
    named_bar_sync(1, 128);
    if (s_flag[0]) {
      // the last CTA: every other CTA's keys and sums are visible (acquire above)
      if (et < 8) {
        float prob = -1.f;
        if (sums) {
          float mg = -INFINITY;
          for (int c = 0; c < G; ++c) {
            const float2 v = __ldcg(a.ms + static_cast<size_t>(c) * 8 + et);
            if (v.y > 0.f) mg = fmaxf(mg, v.x);
          }
          float S = 0.f;
          for (int c = 0; c < G; ++c) {
            const float2 v = __ldcg(a.ms + static_cast<size_t>(c) * 8 + et);
            if (v.y > 0.f) S += v.y * ex2_approx((v.x - mg) * LOG2E);
          }
          prob = S > 0.f ? 1.f / S : 0.f;
        }
        s_prob[et] = prob;
      }
      named_bar_sync(1, 128);
      if (et >= 1 && et < 8) {
        const int i = et;
        const unsigned long long k = __ldcg(a.keys + i);
        int B = a.block_len[0];
        B = B < DFLASH_MIN_BLOCK ? DFLASH_MIN_BLOCK : (B > DFLASH_MAX_BLOCK ? DFLASH_MAX_BLOCK : B);
        int out = -1;
        float pr = -1.f;
        if (i < B) {
          if (k == 0ull) {
            set_status(a.status, DFLASH_DEV_NONFINITE);
          } else {
            out = static_cast<int>(0xffffffffu - static_cast<uint32_t>(k & 0xffffffffull));
            if (sums) {
              pr = s_prob[i];
              for (int i2 = 1; i2 <= i; ++i2)
                if (s_prob[i2] < a.min_p) out = -1;
            }
          }
        }
        a.drafts[i - 1] = out;
        if (a.probs) a.probs[i - 1] = pr;
      }
      named_bar_sync(1, 128);
      if (et < 8) a.keys[et] = 0ull;
      if (et == 0) *a.grid_cnt = 0;
    }
  }
  // every warp whole again (lanes that finished their role early wait for
  // the one still working) before the CTA-wide barrier
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 32);
  }
}

}  // namespace

cudaError_t launch_head_tc8(const HeadTcArgs& a, int grid, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(head_tc8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kH8Smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kHtThreads);
  cfg.dynamicSmemBytes = kH8Smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, head_tc8_kernel, a);
}

cudaError_t launch_head_tc(const HeadTcArgs& a, int grid, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(head_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kHtSmem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kHtThreads);
  cfg.dynamicSmemBytes = kHtSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, head_tc_kernel, a);
}

}  // namespace dflash

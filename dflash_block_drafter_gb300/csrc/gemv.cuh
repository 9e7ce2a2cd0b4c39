// Weight-streaming skinny GEMM ("GEMV" over up to 128 activation rows):
//     Y[R, N] = X[R, K] . W[N, K]^T,   R = 8 * NT
// followed by a fused epilogue.  Each weight byte is read from HBM exactly
// once per launch.
//
// Work split: the matrix is cut into units of 64 rows x (32 * CB) inputs;
// units are ordered group-major and the grid is given equal contiguous
// ranges of units (stream-K).  A CTA = 4 consumer warps (one 16-row m-tile
// each) + 1 producer warp.  The producer streams the CTA's range through a
// ring of shared-memory stages with bulk copies (one per unit, plus the
// matching X chunk when X is streamed) completing on mbarriers; weight
// copies for the first stages are issued before the programmatic-dependent-
// launch wait, so they overlap the previous kernel's tail.  Consumers build
// mma.sync m16n8k16 fragments straight from the stage (layout.cuh), apply
// the per-32-block quantisation scales in fp32 between blocks, and
// accumulate in registers.  A group whose units were split between CTAs is
// finished by whichever contributor arrives last (deterministic summation
// order over contributors, no waiting).
#pragma once

#include "layout.cuh"

namespace dflash {

struct GemvArgs {
  CUtensorMap wmap;              // WT_HEAD only
  CUtensorMap xmap;              // X_STREAM_BF16 with KU <= 224: the caller's BF16 rows
                                 // [n_valid_rows, K], boxes of (KU + 32) inputs x n_valid_rows rows
  const uint8_t* W;              // packed weights (fragment-native formats)
  int N, K;                      // logical rows / inputs
  int UPG;                       // units per 64-row group
  int U;                         // total units
  int n_valid_rows;              // activation rows that exist (others read as zero)
  // X_STREAM: activations in the chunked layout (layout.cuh), R = 8 * NT rows
  // X_STREAM_BF16: BF16 rows X[r * ldx + k] (the caller's taps), read through xmap
  const void* X;
  int ldx;
  float eps;
  // X_NORM: X in the chunked layout (two BF16 planes) holding x * w, not yet
  // divided by the row's RMS; ssq[g * 8 + r] = sum of x^2 over inputs
  // [64 g, 64 g + 64) of row r, g < n_ssq; 1 / RMS scales the outputs
  const float* ssq;
  int n_ssq;
  int rs_early;                  // X_NORM: 1 / RMS needed before the first group (final hidden rows)
  // The next kernel's weights (constant, pf_total bytes in pf_U units of
  // pf_unit bytes, its CTA c' of pf_G starting at unit c' * pf_U / pf_G):
  // once this CTA has issued its last unit, it asks L2 for the first
  // pf_bytes of the shares of next CTAs [c * pf_G / G, (c + 1) * pf_G / G),
  // so that the next kernel's stream starts from L2 (pf_bytes 0: none)
  const uint8_t* pf_W;
  size_t pf_total;
  int pf_unit, pf_U, pf_G, pf_bytes;
  // Extra groups (X_NORM, groups aligned to CTAs): the last vgroups of the
  // U / UPG groups re-read weight groups [vwg0, vwg0 + vgroups) with their
  // own activations X2, row sums of squares ssq2 and n_valid2 valid rows (an
  // 8-row draft QKV GEMV that also projects the committed rows' K / V)
  int vgroups, vwg0;
  const void* X2;
  const float* ssq2;
  int n_valid2;
  // Cluster finishing (8-row passes): when cl_parts * cl_gph > 1 the grid is
  // launched in clusters of cl_parts * cl_gph CTAs covering cl_gph whole
  // 64-row groups (one attention head for the per-head epilogue), each group
  // split between cl_parts CTAs.  A group's partial sums go to its first CTA
  // through distributed shared memory, and the groups of a head exchange
  // their results there, instead of through global memory and counters.
  int cl_parts, cl_gph;
  float* partials;               // [gridDim.x, 2, 64, R]
  int* counters;                 // [N / 64]
  int32_t* status;
  unsigned long long* trace;     // diagnostic builds only (DFLASH_TRACE): per-CTA timestamps
};

#ifdef DFLASH_TRACE
#define DFLASH_STAMP(k)                                                                   \
  do {                                                                                    \
    if (a.trace) a.trace[static_cast<size_t>(blockIdx.x) * kTraceSlots + (k)] = globaltimer_ns(); \
  } while (0)
#else
#define DFLASH_STAMP(k) \
  do {                  \
  } while (0)
#endif

template <int WT, int NT, int XMODE>
struct GemvGeom {
  using F = Fmt<WT>;
  static constexpr int R = NT * 8;
  static constexpr int KU = F::CB * 32;                 // inputs per unit
  static constexpr int XSE = KU + 32;                   // streamed X row stride (elements, padded)
  static constexpr int XS_STRIDE = XSE * 2;             // ... in bytes
  static constexpr bool kStream = true;
  // activation type fed to the MMA: FP16 for quantised weights unless X is
  // the caller's BF16 taps
  static constexpr bool kF16 = F::kF16 && (XMODE == X_STREAM || XMODE == X_NORM);
  // BF16 activations computed in fp32 are carried as two BF16 planes, hi and
  // lo = x - hi (about 16 significant bits), each multiplied on the tensor
  // cores; the caller's BF16 taps (X_STREAM_BF16) are exact and need no lo.
  static constexpr bool kSplit = !kF16 && XMODE != X_STREAM_BF16;
  static constexpr int XPLANES = kSplit ? 2 : 1;
  static constexpr int XS_BYTES = kStream ? XPLANES * R * XS_STRIDE : 0;
  static constexpr int STAGE = ((F::UNIT + XS_BYTES + 1023) / 1024) * 1024;
  // Two consumer warpgroups split each unit's CB blocks (K halves): a
  // scheduler runs two consumer warps, hiding the MMA and shared-memory
  // latencies of one behind the other.  At each group end the second
  // warpgroup hands its partial sums to the first through a double buffer.
  // Larger tiles keep fewer threads (register budget).
  static constexpr int CWG = NT <= 4 ? 2 : 1;
  // [2][CWG - 1 warpgroups][128 threads][NT][4] floats
  static constexpr int SBUF = CWG > 1 ? 2 * (CWG - 1) * 128 * NT * 16 : 0;
  static constexpr int RING_BUDGET = 200000 - SBUF;
  static constexpr int STAGES_FIT = RING_BUDGET / STAGE;
  static constexpr int STAGES = STAGES_FIT < 2 ? 2 : (STAGES_FIT < F::STAGES ? STAGES_FIT : F::STAGES);
  static constexpr int RING = STAGES * STAGE;
  static constexpr int THREADS = 128 * CWG + 32;
  // cluster finishing buffers (8-row passes of the backbone formats): the
  // group's partial sums from up to kClMaxParts - 1 other CTAs, and the
  // kClMaxGph groups of a head (kClHeadSlot floats each: 8 x 64 values in mma
  // fragment order, then per-warp partial sums of squares [4][8])
  static constexpr int kClMaxParts = 8, kClMaxGph = 4, kClHeadSlot = 512 + 32;
  static constexpr bool kClusterable = NT == 1 && WT != WT_HEAD;
  static constexpr int CL_RED = kClusterable ? (kClMaxParts - 1) * 128 * 16 : 0;
  static constexpr int CL_HEAD = kClusterable ? kClMaxGph * kClHeadSlot * 4 : 0;
  static constexpr int CLBUF = CL_RED + CL_HEAD;
  static constexpr int MISC = SBUF + CLBUF + 8 * (2 * STAGES + 3) + 64 + 4 * R * 8 + R * 4;
  // smem: [ring][partial-sum double buffer][cluster buffers][barriers][misc]
  static __host__ __device__ constexpr int smem_bytes(int) { return 1024 + RING + MISC; }
};

// Epilogue interface (see gemv_epilogues.cuh):
//   struct Epi {
//     static constexpr bool kAfterGroup;   // needs a CTA-wide step after a group
//     static constexpr bool kFinish;       // needs a CTA-wide step at the end
//     struct Local { ... };                // per-thread registers across groups
//     __device__ void init(Local&) const;
//     __device__ void prologue(const GemvArgs&, int tid) const;     // consumers, after X is ready
//     __device__ void group(const GemvArgs&, Local&, int g, int w, int lane, float (&acc)[NT][4]) const;
//     __device__ void after_group(const GemvArgs&, int g, int tid, int* sflag) const;
//     __device__ void finish(const GemvArgs&, Local&, int w, int lane, int tid, unsigned long long* stage,
//                            int* sflag) const;
//   };

__device__ __forceinline__ int cta_of_unit(long long u, int G, int U) {
  return static_cast<int>(((u + 1) * G - 1) / U);
}

template <int WT, int NT, int XMODE, class Epi>
__global__ void __launch_bounds__(GemvGeom<WT, NT, XMODE>::THREADS, 1)
    gemv_kernel(const __grid_constant__ GemvArgs a, const __grid_constant__ Epi epi) {
  using Geo = GemvGeom<WT, NT, XMODE>;
  using F = Fmt<WT>;
  constexpr int R = Geo::R;
  constexpr int STAGES = Geo::STAGES;
  constexpr bool kF16 = Geo::kF16;
  constexpr bool kStream = Geo::kStream;
  constexpr bool kSplit = Geo::kSplit;
  constexpr int XPLANES = Geo::XPLANES;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;
  float4* sbuf = reinterpret_cast<float4*>(ring + Geo::RING);  // [2][CWG - 1][128][NT] (other warpgroups' sums)
  float4* cl_red = reinterpret_cast<float4*>(ring + Geo::RING + Geo::SBUF);             // [parts - 1][128]
  float* cl_head = reinterpret_cast<float*>(ring + Geo::RING + Geo::SBUF + Geo::CL_RED);  // [gph][8][64]
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + Geo::RING + Geo::SBUF + Geo::CLBUF);
  uint64_t* empty = full + STAGES;
  uint64_t* cl_red_bar = empty + STAGES;   // the other parts' sums have arrived
  uint64_t* cl_head_bar = cl_red_bar + 1;  // the head's other groups have arrived
  int* sflag = reinterpret_cast<int*>(cl_head_bar + 1);                // 16 ints
  float* srs = reinterpret_cast<float*>(sflag + 16);                  // [R] row scales
  unsigned long long* sstage = reinterpret_cast<unsigned long long*>(srs + R);  // [4][R]

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  const int G = gridDim.x;
  if (tid == 0) DFLASH_STAMP(0);
  const int u_begin = static_cast<int>((static_cast<long long>(blockIdx.x) * a.U) / G);
  const int u_end = static_cast<int>((static_cast<long long>(blockIdx.x + 1) * a.U) / G);
  const int n_units = u_end - u_begin;
  const int vu0 = a.U - a.vgroups * a.UPG;  // first unit of the extra groups (U: none)

  const int cl_size = Geo::kClusterable ? a.cl_parts * a.cl_gph : 1;
  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 4 * Geo::CWG);
    }
    if (cl_size > 1) {
      mbar_init(cl_red_bar, a.cl_parts > 1 ? a.cl_parts - 1 : 1);
      mbar_init(cl_head_bar, a.cl_gph > 1 ? a.cl_gph - 1 : 1);
    }
    fence_barrier_init();
  }
  if constexpr (XMODE == X_STREAM_BF16) {
    // rows that are never copied (beyond n_valid_rows) must read as zeros
    if (a.n_valid_rows < R) {
      for (int s = 0; s < STAGES; ++s) {
        uint8_t* xs = ring + s * Geo::STAGE + F::UNIT;
        for (int i = tid; i < (R - a.n_valid_rows) * (Geo::XS_STRIDE / 16); i += Geo::THREADS) {
          const int rr = a.n_valid_rows + i / (Geo::XS_STRIDE / 16);
          reinterpret_cast<uint4*>(xs + rr * Geo::XS_STRIDE)[i % (Geo::XS_STRIDE / 16)] = make_uint4(0, 0, 0, 0);
        }
      }
    }
  }
  __syncthreads();
  // cluster peers may use this CTA's barriers once every CTA has signalled
  // here (the finishing step waits for that before its first remote access)
  if (cl_size > 1) cluster_arrive_relaxed();

  if (warp == 4 * Geo::CWG) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      if constexpr (WT == WT_HEAD) prefetch_tensormap(&a.wmap);
      // a TMA box spans at most 256 inputs: wider units copy row by row
      constexpr bool kXBox = Geo::KU + 32 <= 256;
      if constexpr (XMODE == X_STREAM_BF16 && kXBox) prefetch_tensormap(&a.xmap);
      const uint64_t pol = l2_policy_evict_first();
      uint32_t tx = F::UNIT;
      if constexpr (XMODE == X_STREAM || XMODE == X_NORM) tx += XPLANES * R * Geo::XS_STRIDE;
      if constexpr (XMODE == X_STREAM_BF16) tx += a.n_valid_rows * (kXBox ? Geo::XS_STRIDE : Geo::KU * 2);
      auto issue_w = [&](int it, int u) {
        uint8_t* dst = ring + (it % STAGES) * Geo::STAGE;
        if constexpr (WT == WT_HEAD) {
          const int g = u / a.UPG, j = u - g * a.UPG;
          tma_load_2d_hint(dst, &a.wmap, j * 128, g * 64, &full[it % STAGES], pol);
          tma_load_2d_hint(dst + 8192, &a.wmap, j * 128 + 64, g * 64, &full[it % STAGES], pol);
        } else {
          const int uw = u >= vu0 ? u - vu0 + a.vwg0 * a.UPG : u;
          bulk_g2s_hint(dst, a.W + static_cast<size_t>(uw) * F::UNIT, F::UNIT, &full[it % STAGES], pol);
        }
      };
      auto issue_x = [&](int it, int u) {
        const int j = u % a.UPG;
        uint8_t* dst = ring + (it % STAGES) * Geo::STAGE + F::UNIT;
        if constexpr (XMODE == X_STREAM || XMODE == X_NORM) {
          // one contiguous chunk per plane
          const uint8_t* src = static_cast<const uint8_t*>(u >= vu0 ? a.X2 : a.X) +
                               static_cast<size_t>(j) * XPLANES * R * Geo::XS_STRIDE;
          bulk_g2s(dst, src, XPLANES * R * Geo::XS_STRIDE, &full[it % STAGES]);
        } else if constexpr (XMODE == X_STREAM_BF16) {
          if constexpr (kXBox) {
            // one box: the valid rows x (KU + 32) inputs from input j * KU,
            // landing with the padded row stride; the 32 extra inputs are never read
            tma_load_2d(dst, &a.xmap, j * Geo::KU, 0, &full[it % STAGES]);
          } else {
            const uint8_t* src = static_cast<const uint8_t*>(a.X) + static_cast<size_t>(j) * Geo::KU * 2;
            for (int r = 0; r < a.n_valid_rows; ++r)
              bulk_g2s(dst + r * Geo::XS_STRIDE, src + static_cast<size_t>(r) * a.ldx * 2, Geo::KU * 2,
                       &full[it % STAGES]);
          }
        }
      };
      const int n_pre = n_units < STAGES ? n_units : STAGES;
      for (int it = 0; it < n_pre; ++it) {
        mbar_arrive_expect_tx(&full[it], tx);
        issue_w(it, u_begin + it);
      }
      pdl_wait();  // activations below come from the previous kernel
      DFLASH_STAMP(1);
      epi.producer_start(a, blockIdx.x, G);
      if constexpr (kStream)
        for (int it = 0; it < n_pre; ++it) issue_x(it, u_begin + it);
      int issued = n_pre;
      for (int it = n_pre; it < n_units; ++it) {
        const int s = it % STAGES;
        if (!mbar_wait(&empty[s], ((it / STAGES) - 1) & 1)) {
          set_status(a.status, DFLASH_DEV_TIMEOUT);
          break;
        }
        mbar_arrive_expect_tx(&full[s], tx);
        issue_w(it, u_begin + it);
        if constexpr (kStream) issue_x(it, u_begin + it);
        issued = it + 1;
      }
      if (a.pf_bytes > 0 && issued == n_units) {
        const int n0 = static_cast<int>(static_cast<long long>(blockIdx.x) * a.pf_G / G);
        const int n1 = static_cast<int>(static_cast<long long>(blockIdx.x + 1) * a.pf_G / G);
        for (int c2 = n0; c2 < n1; ++c2) {
          const size_t off = static_cast<size_t>(static_cast<long long>(c2) * a.pf_U / a.pf_G) * a.pf_unit;
          if (off >= a.pf_total) break;
          const size_t left = a.pf_total - off;
          bulk_prefetch_l2_plain(a.pf_W + off, static_cast<uint32_t>(left < size_t(a.pf_bytes) ? left : size_t(a.pf_bytes)));
        }
      }
      // Every issued copy must land before the CTA may exit.
      for (int it = (issued > STAGES ? issued - STAGES : 0); it < issued; ++it)
        if (!mbar_wait(&full[it % STAGES], (it / STAGES) & 1)) {
          set_status(a.status, DFLASH_DEV_TIMEOUT);
          break;
        }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  pdl_wait();
  pdl_launch_dependents();
  // warp w of warpgroup kh: m-tile w, blocks [kh * CB / CWG, (kh + 1) * CB / CWG) of every unit
  const int w = warp & 3, kh = warp >> 2;
  constexpr int BPW = F::CB / Geo::CWG;
  if (tid == 0) DFLASH_STAMP(3);

  // X_NORM: 1 / RMS per row from the producing kernel's partial sums of
  // squares.  The loads are issued here and the sums formed at the first
  // group's end (or at once when the epilogue needs them first), so the
  // weight stream never waits for them.  Warp w owns rows w and w + 4; lane
  // holds groups lane and lane + 32; fixed summation order.
  float ssv[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
  bool rs_ready = XMODE != X_NORM;
  // a CTA's units are all of the extra groups or none (groups aligned to CTAs)
  const bool xcta = u_begin >= vu0;
  const float* ssq = xcta ? a.ssq2 : a.ssq;
  const int nvr = xcta ? a.n_valid2 : a.n_valid_rows;
  auto finish_rs = [&]() {
    if constexpr (XMODE == X_NORM) {
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const int r = w + 4 * rr;
        float ss = ssv[rr][0] + ssv[rr][1];
        for (int g = lane + 64; g < a.n_ssq; g += 32) ss += __ldcg(ssq + g * 8 + r);
#pragma unroll
        for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if (lane == 0 && r < R) srs[r] = (r < nvr) ? rsqrtf(ss / a.K + a.eps) : 0.f;
      }
      named_bar_sync(1, 128);
      rs_ready = true;
    }
  };
  if (kh == 0) {
    if constexpr (XMODE == X_NORM) {
#pragma unroll
      for (int rr = 0; rr < 2; ++rr)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int r = w + 4 * rr, g = lane + 32 * h;
          if (r < R && g < a.n_ssq) ssv[rr][h] = __ldcg(ssq + g * 8 + r);
        }
      if (a.rs_early) finish_rs();
    }
    epi.prologue(a, tid, XMODE == X_NORM ? srs : nullptr);
    named_bar_sync(1, 128);
  }

  typename Epi::Local loc;
  epi.init(loc);
  if constexpr (Geo::kClusterable && Epi::kCluster) {
    // cluster finishing: every peer's barriers are initialised once all have
    // signalled (waited for here, while the ring fills, by the threads that
    // later access peers); the epilogue's per-CTA constants are loaded now
    if (cl_size > 1 && kh == 0) {
      cluster_wait();
      epi.prepare_cluster(a, loc, u_begin / a.UPG, w, lane);
    }
  }
  // Accumulator chains: for the BF16 formats one per k-step and activation
  // plane (acc: hi plane, k-step 0; accb: hi, k-step 1; acc2 / acc2b: the lo
  // plane), so consecutive MMAs never wait on each other; the quantised
  // formats sum each 32-block in its own temporary and scale it into acc.
  // (tiles of more than 16 rows keep one chain per plane: registers)
  constexpr bool kChains = NT <= 2;
  constexpr int NB = kChains ? NT : 1;
  float acc[NT][4], acc2[NT][4], accb_s[NB][4], acc2b_s[NB][4];
#pragma unroll
  for (int t = 0; t < NT; ++t)
    for (int e = 0; e < 4; ++e) acc[t][e] = acc2[t][e] = 0.f;
#pragma unroll
  for (int t = 0; t < NB; ++t)
    for (int e = 0; e < 4; ++e) accb_s[t][e] = acc2b_s[t][e] = 0.f;
  auto accb = [&](int t) -> float(&)[4] {
    if constexpr (kChains) return accb_s[t];
    else return acc[t];
  };
  auto acc2b = [&](int t) -> float(&)[4] {
    if constexpr (kChains) return acc2b_s[t];
    else return acc2[t];
  };

  const int first_group = u_begin / a.UPG;
  const uint32_t ring_s = smem_u32(ring);
  const int xrow = lane >> 2;
  bool ok = true;
  int gcount = 0;  // group ends passed (the same sequence in both warpgroups)
  // blocks of a unit handled together: all their shared-memory loads are
  // issued before their MMAs (fewer at once for large tiles: registers)
  constexpr int IB = NT <= 2 ? BPW : 1;
  constexpr bool kPairs = (WT == WT_Q4_0 || WT == WT_Q5_0) && IB % 2 == 0;

  // After a timeout the loop keeps running (without waiting) so every warp
  // takes the same named barriers; the outputs are then unspecified.
  for (int it = 0; it < n_units; ++it) {
    const int u = u_begin + it;
    const int s = it % STAGES;
    const int g = u / a.UPG, j = u - g * a.UPG;
    if (ok && !mbar_wait(&full[s], (it / STAGES) & 1)) {
      set_status(a.status, DFLASH_DEV_TIMEOUT);
      ok = false;
    }
    if (tid == 0 && it == 0) DFLASH_STAMP(5);
    const uint32_t ubase = ring_s + s * Geo::STAGE;

#pragma unroll
    for (int b0 = 0; b0 < BPW; b0 += IB) {
      BlockFrag f[IB];
      uint4 xf[IB][NT], xl[IB][NT];
#pragma unroll
      for (int i = 0; i < IB; ++i) {
        const int bl = kh * BPW + b0 + i;
        if constexpr (kPairs) {
          if (i % 2 == 0) decode_pair<WT, kF16>(ubase, w, lane, bl >> 1, f[i], f[i + 1]);
        } else {
          f[i] = decode_block<WT, kF16>(ubase, w, lane, bl);
        }
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          const uint32_t xb = ubase + F::UNIT + (t * 8 + xrow) * Geo::XS_STRIDE + bl * 64 + (lane & 3) * 16;
          xf[i][t] = lds128(xb);
          if constexpr (kSplit) xl[i][t] = lds128(xb + R * Geo::XS_STRIDE);
        }
      }
      if constexpr (WT == WT_BF16 || WT == WT_HEAD) {
#pragma unroll
        for (int i = 0; i < IB; ++i)
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            mma_bf16_16816(acc[t], f[i].a[0][0], f[i].a[0][1], f[i].a[0][2], f[i].a[0][3], xf[i][t].x, xf[i][t].y);
            mma_bf16_16816(accb(t), f[i].a[1][0], f[i].a[1][1], f[i].a[1][2], f[i].a[1][3], xf[i][t].z, xf[i][t].w);
            if constexpr (kSplit) {
              mma_bf16_16816(acc2[t], f[i].a[0][0], f[i].a[0][1], f[i].a[0][2], f[i].a[0][3], xl[i][t].x,
                             xl[i][t].y);
              mma_bf16_16816(acc2b(t), f[i].a[1][0], f[i].a[1][1], f[i].a[1][2], f[i].a[1][3], xl[i][t].z,
                             xl[i][t].w);
            }
          }
      } else {
        // one sum per block; its MMAs (k-steps, planes) in rounds over the
        // blocks, so neighbouring MMAs belong to different blocks
        float tmp[IB][NT][4];
#pragma unroll
        for (int i = 0; i < IB; ++i)
#pragma unroll
          for (int t = 0; t < NT; ++t) tmp[i][t][0] = tmp[i][t][1] = tmp[i][t][2] = tmp[i][t][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < 2; ++ks) {
#pragma unroll
          for (int i = 0; i < IB; ++i)
#pragma unroll
            for (int t = 0; t < NT; ++t) {
              const uint32_t b0r = ks ? xf[i][t].z : xf[i][t].x, b1r = ks ? xf[i][t].w : xf[i][t].y;
              if constexpr (kF16)
                mma_f16_16816(tmp[i][t], f[i].a[ks][0], f[i].a[ks][1], f[i].a[ks][2], f[i].a[ks][3], b0r, b1r);
              else
                mma_bf16_16816(tmp[i][t], f[i].a[ks][0], f[i].a[ks][1], f[i].a[ks][2], f[i].a[ks][3], b0r, b1r);
            }
          if constexpr (kSplit) {
#pragma unroll
            for (int i = 0; i < IB; ++i)
#pragma unroll
              for (int t = 0; t < NT; ++t) {
                const uint32_t b0r = ks ? xl[i][t].z : xl[i][t].x, b1r = ks ? xl[i][t].w : xl[i][t].y;
                mma_bf16_16816(tmp[i][t], f[i].a[ks][0], f[i].a[ks][1], f[i].a[ks][2], f[i].a[ks][3], b0r, b1r);
              }
          }
        }
#pragma unroll
        for (int i = 0; i < IB; ++i)
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            acc[t][0] = fmaf(f[i].d_r, tmp[i][t][0], acc[t][0]);
            acc[t][1] = fmaf(f[i].d_r, tmp[i][t][1], acc[t][1]);
            acc[t][2] = fmaf(f[i].d_r8, tmp[i][t][2], acc[t][2]);
            acc[t][3] = fmaf(f[i].d_r8, tmp[i][t][3], acc[t][3]);
          }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
    if (tid == 0 && it == n_units - 1) DFLASH_STAMP(6);

    if (j == a.UPG - 1 || u == u_end - 1) {
      if constexpr (WT == WT_BF16 || WT == WT_HEAD) {
#pragma unroll
        for (int t = 0; t < NT; ++t)
          for (int e = 0; e < 4; ++e) {
            if constexpr (kChains) {
              acc[t][e] = (acc[t][e] + accb_s[t][e]) + (acc2[t][e] + acc2b_s[t][e]);
              accb_s[t][e] = acc2b_s[t][e] = 0.f;
            } else {
              acc[t][e] += acc2[t][e];
            }
            acc2[t][e] = 0.f;
          }
      }
      if constexpr (Geo::CWG > 1) {
        // the other warpgroups hand their K-part sums to the first and go on
        // (barrier 2 + b: buffer b filled; barrier 4 + b: buffer b free again)
        constexpr int NB = 128 * Geo::CWG;
        float4* sbb = sbuf + static_cast<size_t>(gcount & 1) * (Geo::CWG - 1) * 128 * NT;
        if (kh >= 1) {
          float4* sb = sbb + (static_cast<size_t>(kh - 1) * 128 + (w * 32 + lane)) * NT;
          if (gcount >= 2) named_bar_sync(4 + (gcount & 1), NB);
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            sb[t] = make_float4(acc[t][0], acc[t][1], acc[t][2], acc[t][3]);
            acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
          }
          named_bar_arrive(2 + (gcount & 1), NB);
          ++gcount;
          continue;
        }
        named_bar_sync(2 + (gcount & 1), NB);
        // fixed order over the warpgroups (deterministic)
#pragma unroll
        for (int k2 = 0; k2 < Geo::CWG - 1; ++k2) {
          const float4* sb = sbb + (static_cast<size_t>(k2) * 128 + (w * 32 + lane)) * NT;
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            const float4 q = sb[t];
            acc[t][0] += q.x;
            acc[t][1] += q.y;
            acc[t][2] += q.z;
            acc[t][3] += q.w;
          }
        }
        named_bar_arrive(4 + (gcount & 1), NB);
        ++gcount;
      }
      if constexpr (XMODE == X_NORM) {
        // the rows were multiplied unnormalised: scale each output by 1 / RMS of its row
        if (!rs_ready) finish_rs();
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          const int n = t * 8 + (lane & 3) * 2;
          acc[t][0] *= srs[n];
          acc[t][1] *= srs[n + 1];
          acc[t][2] *= srs[n];
          acc[t][3] *= srs[n + 1];
        }
      }
      bool clustered = false;
      if constexpr (Geo::kClusterable && Epi::kCluster) {
        if (cl_size > 1) {
          // ------------------------------------- cluster finishing (DSMEM)
          // this CTA's range lies in one group: part `part` of local group gl
          clustered = true;
          if (tid == 0) DFLASH_STAMP(4);
          const int rank = static_cast<int>(blockIdx.x) % cl_size;
          const int part = rank % a.cl_parts, gl = rank / a.cl_parts;
          const uint32_t leader = static_cast<uint32_t>(gl * a.cl_parts);
          if (part != 0) {
            st_cluster_v4(mapa_shared(smem_u32(cl_red + (part - 1) * 128 + tid), leader), acc[0][0], acc[0][1],
                          acc[0][2], acc[0][3]);
            named_bar_sync(1, 128);
            if (tid == 0) mbar_remote_arrive(mapa_shared(smem_u32(cl_red_bar), leader));
          } else {
            float pre[NT][4];
            float4 wpre = make_float4(0.f, 0.f, 0.f, 0.f);
            if constexpr (Epi::kPreload) epi.template preload<WT, NT>(g, w, lane, pre, wpre);
            if (a.cl_parts > 1) {
              if (ok && !mbar_wait_cluster(cl_red_bar, 0)) {
                set_status(a.status, DFLASH_DEV_TIMEOUT);
                ok = false;
              }
              // the other parts' sums in rank order (deterministic)
              for (int p = 0; p < a.cl_parts - 1; ++p) {
                const float4 q = cl_red[p * 128 + tid];
                acc[0][0] += q.x;
                acc[0][1] += q.y;
                acc[0][2] += q.z;
                acc[0][3] += q.w;
              }
            }
            if constexpr (Epi::kPreload)
              epi.template group_pre<WT, NT>(g, w, lane, acc, pre, wpre);
            else
              ok = epi.template group_cluster<WT>(a, loc, g, gl, a.cl_parts, w, lane, tid, acc, cl_head,
                                                  cl_head_bar, ok);
          }
        }
      }
      const bool complete = (g * a.UPG >= u_begin) && (j == a.UPG - 1);
      if (clustered) {
        // finished above
      } else if (complete) {
        epi.template group<WT, NT>(a, loc, g, w, lane, acc);
        if constexpr (Epi::kAfterGroup) {
          named_bar_sync(1, 128);
          epi.after_group(a, g, tid, sflag);
        }
      } else {
        // ---------------------------------------------- split-group fix-up
        const int which = (g == first_group) ? 0 : 1;
        float* slot = a.partials + (static_cast<size_t>(blockIdx.x) * 2 + which) * 64 * R;
        const int r0 = w * 16 + (lane >> 2);
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          const int c0 = t * 8 + (lane & 3) * 2;
          __stcg(reinterpret_cast<float2*>(slot + r0 * R + c0), make_float2(acc[t][0], acc[t][1]));
          __stcg(reinterpret_cast<float2*>(slot + (r0 + 8) * R + c0), make_float2(acc[t][2], acc[t][3]));
        }
        // the CTA's stores, ordered by the barrier, are released by thread 0's
        // acquire-release counter increment; the last arriver acquires the others'
        float pre[NT][4];
        float4 wpre = make_float4(0.f, 0.f, 0.f, 0.f);
        if constexpr (Epi::kPreload) epi.template preload<WT, NT>(g, w, lane, pre, wpre);
        named_bar_sync(1, 128);
        const long long ufirst = static_cast<long long>(g) * a.UPG;
        const int c_first = cta_of_unit(ufirst, G, a.U);
        const int c_last = cta_of_unit(ufirst + a.UPG - 1, G, a.U);
        if (tid == 0) {
          const int old = atomic_add_acq_rel(&a.counters[g], 1);
          sflag[0] = (old == c_last - c_first);
        }
        named_bar_sync(1, 128);
        if (sflag[0]) {
#pragma unroll
          for (int t = 0; t < NT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
          // the CTAs' partials in ascending order; FB of them are loaded at once
          constexpr int FB = NT <= 2 ? 8 : (NT <= 4 ? 4 : 2);
          for (int cb = c_first; cb <= c_last; cb += FB) {
            float2 p0[FB][NT], p1[FB][NT];
#pragma unroll
            for (int q = 0; q < FB; ++q) {
              const int c = cb + q;
              if (c <= c_last) {
                const int cfg = static_cast<int>((static_cast<long long>(c) * a.U) / G) / a.UPG;
                const int wc = (g == cfg) ? 0 : 1;
                const float* sl = a.partials + (static_cast<size_t>(c) * 2 + wc) * 64 * R;
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                  const int c0 = t * 8 + (lane & 3) * 2;
                  p0[q][t] = __ldcg(reinterpret_cast<const float2*>(sl + r0 * R + c0));
                  p1[q][t] = __ldcg(reinterpret_cast<const float2*>(sl + (r0 + 8) * R + c0));
                }
              } else {
#pragma unroll
                for (int t = 0; t < NT; ++t) p0[q][t] = p1[q][t] = make_float2(0.f, 0.f);
              }
            }
#pragma unroll
            for (int q = 0; q < FB; ++q)
#pragma unroll
              for (int t = 0; t < NT; ++t) {
                acc[t][0] += p0[q][t].x;
                acc[t][1] += p0[q][t].y;
                acc[t][2] += p1[q][t].x;
                acc[t][3] += p1[q][t].y;
              }
          }
          if (tid == 0) a.counters[g] = 0;
          if constexpr (Epi::kPreload)
            epi.template group_pre<WT, NT>(g, w, lane, acc, pre, wpre);
          else
            epi.template group<WT, NT>(a, loc, g, w, lane, acc);
          if constexpr (Epi::kAfterGroup) {
            named_bar_sync(1, 128);
            epi.after_group(a, g, tid, sflag);
          }
        }
        named_bar_sync(1, 128);  // sflag reuse
      }
#pragma unroll
      for (int t = 0; t < NT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
    }
  }
  if constexpr (Geo::CWG > 1) {
    // the first warpgroup's last two buffer releases have no later fill to pair with
    if (kh >= 1)
      for (int gc = (gcount > 2 ? gcount - 2 : 0); gc < gcount; ++gc) named_bar_sync(4 + (gc & 1), 128 * Geo::CWG);
    if (kh >= 1) return;
  }
  if constexpr (Epi::kFinish) epi.template finish<NT>(a, loc, w, lane, tid, sstage, sflag);
  if (tid == 0) DFLASH_STAMP(7);
}

}  // namespace dflash

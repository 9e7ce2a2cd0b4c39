// Weight-streaming GEMM of a 128-row pass (9..16 sequences) on the tcgen05
// tensor cores.  At 128 activation rows every weight is used 128 times: the
// projections are real GEMMs (about 24 GFLOP per layer), which the legacy
// mma.sync GEMV issues far below its throughput.  Here:
//
//   warp 0      streams, per weight unit (64 rows x KU inputs, the packed
//               fragment-native format of the GEMV), the unit and the
//               activation chunk it multiplies (128 rows x KU inputs per
//               plane, as 64-input tensor-map boxes in 128-byte swizzle) into
//               a 2-stage ring;
//   warps 1..4  decode the unit with the GEMV's own decoders (warp w: 16-row
//               m-tile w) and write it, the GGUF block scale folded in (one
//               FP16 rounding of d * (q - offset)), as a 64 x KU K-major
//               operand in 128-byte swizzle;
//   warp 5      issues tcgen05.mma kind::f16, M 128 (activation rows, A from
//               the streamed chunk) x N 64 (the group's weight rows, B from
//               the decoded tile) x K 16, every plane into the group's FP32
//               accumulator -- 64 TMEM columns, 4 groups in flight;
//   warps 6..9  read a finished group back (thread = activation row, its 64
//               outputs) and apply the epilogue: store, residual add, SwiGLU
//               into the down projection's chunked input, or the raw q/k/v,
//               whose per-head norm / RoPE / cell writes heads_rows_kernel
//               then applies with one CTA per (head, sequence).
//
// A CTA owns whole 64-row groups (grid <= groups), or, for matrices of few
// groups (the projections back to the hidden size), one of `parts` slices of
// a group's inputs; the slices' sums meet in global memory and the CTA that
// arrives last adds them in slice order and applies the epilogue.
#include "gemv_launch.cuh"
#include "kernels.h"

namespace dflash {

namespace {

constexpr int kTcThreads = 320;
constexpr int kTcSlots = 4;  // accumulators of 64 TMEM columns in flight

template <int WT>
struct TcGeo {
  using F = Fmt<WT>;
  static constexpr int KU = F::CB * 32;
  static constexpr int PLANES = F::kF16 ? 1 : 2;  // GGUF: FP16 activations; BF16: hi and lo planes
  static constexpr int XBOX = 128 * 128;          // one 128-row x 64-input box: 16 KB
  static constexpr int XBYTES = PLANES * (KU / 64) * XBOX;
  static constexpr int STAGE = ((F::UNIT + XBYTES + 1023) / 1024) * 1024;
  static constexpr int BTILE = 64 * KU * 2;       // decoded unit, 16-bit
  static constexpr int STAGES = 2;
  static constexpr int NB = (1024 + STAGES * STAGE + 2 * BTILE + 1024 <= 227 * 1024) ? 2 : 1;
  static constexpr int SMEM = 1024 + STAGES * STAGE + NB * BTILE + 1024;
};

// Instruction descriptor of kind::f16, FP32 accumulation, K-major A and B,
// shape M x N; bf16: A and B are BF16 (else FP16).
__host__ __device__ constexpr uint32_t idesc_16(int M, int N, bool bf16) {
  return (1u << 4) | (bf16 ? ((1u << 7) | (1u << 10)) : 0u) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// Row R (0..63), inputs k0 .. k0 + 7 (k0 % 8 == 0) of a decoded 64 x KU
// K-major tile in 128-byte swizzle: 64-input columns of 64 rows x 128 bytes.
__device__ __forceinline__ uint32_t btile_addr(uint32_t base, int R, int k0) {
  return base + (k0 >> 6) * (64 * 128) + R * 128 + ((((k0 & 63) >> 3) ^ (R & 7)) << 4);
}

template <int WT>
__device__ __forceinline__ uint32_t scale_pair(uint32_t pair, uint32_t d2) {
  if constexpr (Fmt<WT>::kF16) return hmul2_u32(pair, d2);
  else return pair;
}

template <int WT>
__global__ void __launch_bounds__(kTcThreads, 1) gemv_tc_kernel(const __grid_constant__ GemvArgs a,
                                                                const __grid_constant__ TcEpi epi) {
  using Geo = TcGeo<WT>;
  using F = Fmt<WT>;
  constexpr int KU = Geo::KU, PLANES = Geo::PLANES, STAGES = Geo::STAGES, NB = Geo::NB;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;                          // [STAGES][unit | X boxes]
  uint8_t* btile = ring + STAGES * Geo::STAGE;   // [NB][64 x KU, 16-bit]
  uint64_t* full = reinterpret_cast<uint64_t*>(btile + NB * Geo::BTILE);
  uint64_t* empty = full + STAGES;    // decoders (4) + MMA commit (1)
  uint64_t* bfull = empty + STAGES;   // [NB] decoders (4)
  uint64_t* bempty = bfull + NB;      // [NB] MMA commit
  uint64_t* accf = bempty + NB;       // [kTcSlots] MMA commit at a group's end
  uint64_t* acce = accf + kTcSlots;   // [kTcSlots] epilogue warps (4)
  uint64_t* mdone = acce + kTcSlots;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(mdone + 1);
  int* s_last = reinterpret_cast<int*>(s_tmem + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = static_cast<int>(gridDim.x);
  const int groups = a.U / a.UPG;
  // whole groups [g0, g1) per CTA, or (epi.parts > 1) part p of group g0's
  // inputs: units [ub, ue) of the packed matrix, in order
  int g0, g1, ub, ue;
  if (epi.parts > 1) {
    g0 = blockIdx.x / epi.parts;
    g1 = g0 + 1;
    const int p = blockIdx.x - g0 * epi.parts;
    ub = g0 * a.UPG + p * a.UPG / epi.parts;
    ue = g0 * a.UPG + (p + 1) * a.UPG / epi.parts;
  } else {
    g0 = static_cast<int>(static_cast<long long>(blockIdx.x) * groups / G);
    g1 = static_cast<int>(static_cast<long long>(blockIdx.x + 1) * groups / G);
    ub = g0 * a.UPG;
    ue = g1 * a.UPG;
  }
  const int n_units = ue - ub;

  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 5);
    }
    for (int b = 0; b < NB; ++b) {
      mbar_init(&bfull[b], 4);
      mbar_init(&bempty[b], 1);
    }
    for (int k = 0; k < kTcSlots; ++k) {
      mbar_init(&accf[k], 1);
      mbar_init(&acce[k], 4);
    }
    mbar_init(mdone, 1);
    fence_barrier_init();
  }
  if (warp == 5) {
    tmem_alloc(s_tmem, 64 * kTcSlots);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  bool ok = true;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && n_units > 0) {
      prefetch_tensormap(&a.xmap);
      const uint64_t pol = l2_policy_evict_first();
      const int u0 = ub;
      auto issue_w = [&](int it) {
        uint8_t* dst = ring + (it % STAGES) * Geo::STAGE;
        bulk_g2s_hint(dst, a.W + static_cast<size_t>(u0 + it) * F::UNIT, F::UNIT, &full[it % STAGES], pol);
      };
      auto issue_x = [&](int it) {
        const int j = (u0 + it) % a.UPG;
        uint8_t* dst = ring + (it % STAGES) * Geo::STAGE + F::UNIT;
        // F::UNIT is a multiple of 1024 for every format (16384, 17408, 9216, 11264)
        for (int p = 0; p < PLANES; ++p)
          for (int kb = 0; kb < KU / 64; ++kb)
            tma_load_2d(dst + (p * (KU / 64) + kb) * Geo::XBOX, &a.xmap, kb * 64, (j * PLANES + p) * 128,
                        &full[it % STAGES]);
      };
      const int npre = n_units < STAGES ? n_units : STAGES;
      for (int it = 0; it < npre; ++it) {
        mbar_arrive_expect_tx(&full[it], F::UNIT + Geo::XBYTES);
        issue_w(it);
      }
      pdl_wait();  // the activations come from the previous kernel
      for (int it = 0; it < npre; ++it) issue_x(it);
      int issued = npre;
      for (int it = npre; it < n_units; ++it) {
        const int s = it % STAGES;
        if (!mbar_wait(&empty[s], ((it / STAGES) - 1) & 1)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&full[s], F::UNIT + Geo::XBYTES);
        issue_w(it);
        issue_x(it);
        issued = it + 1;
      }
      for (int it = (issued > STAGES ? issued - STAGES : 0); it < issued; ++it)
        if (!mbar_wait(&full[it % STAGES], (it / STAGES) & 1)) {
          ok = false;
          break;
        }
      if (!ok) set_status(a.status, DFLASH_DEV_TIMEOUT);
    } else if (lane == 0) {
      pdl_wait();
    }
  } else if (warp >= 1 && warp <= 4) {
    // ------------------------------------------------------------ decoders
    const int w = warp - 1;  // m-tile: weight rows 16 w .. 16 w + 15 of the group
    const int gr = lane >> 2, t4 = lane & 3;
    const uint32_t ring_s = smem_u32(ring), bt_s = smem_u32(btile);
    for (int it = 0; it < n_units && ok; ++it) {
      const int s = it % STAGES, b = it % NB;
      if (!mbar_wait(&full[s], (it / STAGES) & 1)) ok = false;
      if (ok && it >= NB && !mbar_wait(&bempty[b], ((it / NB) - 1) & 1)) ok = false;
      if (!ok) break;
      const uint32_t ub = ring_s + s * Geo::STAGE, bb = bt_s + b * Geo::BTILE;
      auto put = [&](int bl, const BlockFrag& f) {
        uint32_t d0 = 0, d8 = 0;
        if constexpr (F::kF16) {
          const __half2 h0 = __float2half2_rn(f.d_r), h8 = __float2half2_rn(f.d_r8);
          d0 = *reinterpret_cast<const uint32_t*>(&h0);
          d8 = *reinterpret_cast<const uint32_t*>(&h8);
        }
        const int k0 = bl * 32 + t4 * 8;
        sts128(btile_addr(bb, w * 16 + gr, k0), scale_pair<WT>(f.a[0][0], d0), scale_pair<WT>(f.a[0][2], d0),
               scale_pair<WT>(f.a[1][0], d0), scale_pair<WT>(f.a[1][2], d0));
        sts128(btile_addr(bb, w * 16 + gr + 8, k0), scale_pair<WT>(f.a[0][1], d8), scale_pair<WT>(f.a[0][3], d8),
               scale_pair<WT>(f.a[1][1], d8), scale_pair<WT>(f.a[1][3], d8));
      };
#pragma unroll
      for (int bl = 0; bl < F::CB; bl += (WT == WT_Q4_0 || WT == WT_Q5_0) ? 2 : 1) {
        if constexpr (WT == WT_Q4_0 || WT == WT_Q5_0) {
          BlockFrag f0, f1;
          decode_pair<WT, F::kF16>(ub, w, lane, bl >> 1, f0, f1);
          put(bl, f0);
          put(bl + 1, f1);
        } else {
          put(bl, decode_block<WT, F::kF16>(ub, w, lane, bl));
        }
      }
      // generic-proxy writes of the tile, then its hand-off to the tensor cores
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&bfull[b]);
        mbar_arrive(&empty[s]);  // the unit's codes have been read
      }
    }
    if (!ok && lane == 0) set_status(a.status, DFLASH_DEV_TIMEOUT);
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n_units > 0) {
      constexpr uint32_t idesc = idesc_16(128, 64, !F::kF16);
      const uint32_t ring_s = smem_u32(ring), bt_s = smem_u32(btile);
      for (int it = 0; it < n_units && ok; ++it) {
        const int s = it % STAGES, b = it % NB;
        const int u = ub + it, gi = u / a.UPG - g0, slot = gi % kTcSlots;
        const bool first = u == ub || u % a.UPG == 0;     // the group's first unit in this CTA
        const bool last = u == ue - 1 || u % a.UPG == a.UPG - 1;
        if (first && gi >= kTcSlots && !mbar_wait(&acce[slot], ((gi / kTcSlots) - 1) & 1)) {
          ok = false;
          break;
        }
        if (!mbar_wait(&full[s], (it / STAGES) & 1) || !mbar_wait(&bfull[b], (it / NB) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t xs = ring_s + s * Geo::STAGE + F::UNIT, bs = bt_s + b * Geo::BTILE;
#pragma unroll
        for (int kk = 0; kk < KU / 16; ++kk) {
          const uint64_t db = umma_desc_sw128(bs + (kk >> 2) * (64 * 128) + (kk & 3) * 32, 16, 1024);
#pragma unroll
          for (int p = 0; p < PLANES; ++p) {
            const uint64_t da =
                umma_desc_sw128(xs + (p * (KU / 64) + (kk >> 2)) * Geo::XBOX + (kk & 3) * 32, 16, 1024);
            umma_f16(tmem + slot * 64, da, db, idesc, (!first || kk || p) ? 1u : 0u);
          }
        }
        umma_commit(&empty[s]);
        umma_commit(&bempty[b]);
        if (last) umma_commit(&accf[slot]);
      }
      // tensor memory may only be freed once every issued MMA has finished
      umma_commit(mdone);
      if (!mbar_wait(mdone, 0)) ok = false;
      if (!ok) set_status(a.status, DFLASH_DEV_TIMEOUT);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    pdl_launch_dependents();
    const int q = warp & 3;               // TMEM lane quarter
    const int n = q * 32 + lane;          // activation row = TMEM lane
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(q * 32) << 16);
    const int ng = g1 - g0;
    for (int gi = 0; gi < ng; ++gi) {
      const int slot = gi % kTcSlots, g = g0 + gi;
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&accf[slot], (gi / kTcSlots) & 1));
      tc_fence_after();
      float v[64];
      {
        uint32_t r0[32], r1[32];
        tmem_ld32(lane_addr + slot * 64, r0);
        tmem_ld32(lane_addr + slot * 64 + 32, r1);
        tmem_wait_ld();
        tmem_reg_fence(r0);
        tmem_reg_fence(r1);
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          v[c] = __uint_as_float(r0[c]);
          v[32 + c] = __uint_as_float(r1[c]);
        }
      }
      // the accumulator has been read: the group kTcSlots later may reuse it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acce[slot]);
      if (epi.parts > 1) {
        // part of the group's sum: published, then the CTA arriving last adds
        // every part in order and applies the epilogue
        float* mine = a.partials + (static_cast<size_t>(blockIdx.x) * 128 + n) * 64;
#pragma unroll
        for (int c = 0; c < 64; c += 4) __stcg(reinterpret_cast<float4*>(mine + c), make_float4(v[c], v[c + 1], v[c + 2], v[c + 3]));
        named_bar_sync(1, 128);
        if (warp == 6 && lane == 0) s_last[0] = atomic_add_acq_rel(&a.counters[g], 1) == epi.parts - 1;
        named_bar_sync(1, 128);
        if (s_last[0]) {
#pragma unroll
          for (int c = 0; c < 64; ++c) v[c] = 0.f;
          for (int p = 0; p < epi.parts; ++p) {
            const float* pp = a.partials + (static_cast<size_t>(g * epi.parts + p) * 128 + n) * 64;
#pragma unroll
            for (int c = 0; c < 64; c += 4) {
              const float4 q4 = __ldcg(reinterpret_cast<const float4*>(pp + c));
              v[c] += q4.x;
              v[c + 1] += q4.y;
              v[c + 2] += q4.z;
              v[c + 3] += q4.w;
            }
          }
          epi.apply(g, n, v);
          if (warp == 6 && lane == 0) a.counters[g] = 0;
        }
        named_bar_sync(1, 128);  // s_last reuse
      } else {
        epi.apply(g, n, v);
      }
    }
    if (!ok && lane == 0) set_status(a.status, DFLASH_DEV_TIMEOUT);
  }
  // release the tensor memory once every tcgen05 operation of the CTA is done
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 64 * kTcSlots);
  }
}

}  // namespace

// Epilogue of one finished 64-row group g for activation row n: v[c] is
// output column g * 64 + c (the weight rows of the packed formats are in
// natural order within a group).
__device__ void TcEpi::apply(int g, int n, const float (&v)[64]) const {
  if (mode == STORE || mode == HEADS) {
    float* o = (mode == STORE ? out : heads.raw) + static_cast<size_t>(n) * (mode == STORE ? ldo : heads.ldr) + g * 64;
#pragma unroll
    for (int c = 0; c < 64; c += 4) __stcg(reinterpret_cast<float4*>(o + c), make_float4(v[c], v[c + 1], v[c + 2], v[c + 3]));
  } else if (mode == RESID) {
    float* o = out + static_cast<size_t>(n) * ldo + g * 64;
#pragma unroll
    for (int c = 0; c < 64; c += 4) {
      float4 x = __ldcg(reinterpret_cast<const float4*>(o + c));
      x.x += v[c];
      x.y += v[c + 1];
      x.z += v[c + 2];
      x.w += v[c + 3];
      __stcg(reinterpret_cast<float4*>(o + c), x);
    }
  } else {  // SWIGLU: per 16-row m-tile, 8 gate rows then the 8 up rows of outputs g * 32 + 8 w' + r
#pragma unroll
    for (int w2 = 0; w2 < 4; ++w2) {
      float hv[8];
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const float gt = v[w2 * 16 + r];
        hv[r] = gt / (1.f + __expf(-gt)) * v[w2 * 16 + 8 + r];
      }
      const int o = g * 32 + w2 * 8;  // 8 consecutive outputs: one 16-byte (FP16) or two (BF16) stores
      if (h_f16) {
        *reinterpret_cast<uint4*>(static_cast<__half*>(h) + xchunk_index(o, n, 0, 128, h_ku, 1)) =
            make_uint4(pack_f16x2(hv[0], hv[1]), pack_f16x2(hv[2], hv[3]), pack_f16x2(hv[4], hv[5]),
                       pack_f16x2(hv[6], hv[7]));
      } else {
        uint4 hi, lo;
        split_bf16x2(hv[0], hv[1], hi.x, lo.x);
        split_bf16x2(hv[2], hv[3], hi.y, lo.y);
        split_bf16x2(hv[4], hv[5], hi.z, lo.z);
        split_bf16x2(hv[6], hv[7], hi.w, lo.w);
        __nv_bfloat16* hp = static_cast<__nv_bfloat16*>(h);
        *reinterpret_cast<uint4*>(hp + xchunk_index(o, n, 0, 128, h_ku, 2)) = hi;
        *reinterpret_cast<uint4*>(hp + xchunk_index(o, n, 1, 128, h_ku, 2)) = lo;
      }
    }
  }
}

// Per-head RMSNorm, RoPE, FP16 rounding and query / cell writes of a 128-row
// pass's raw q/k/v (the GEMV's EpiHeads mode 0), one CTA per (head, sequence)
// over that sequence's 8 block rows.
__global__ void __launch_bounds__(128) heads_rows_kernel(const __grid_constant__ EpiHeads e) {
  const int hh = blockIdx.x, s = blockIdx.y;
  pdl_wait();
  pdl_launch_dependents();
  EpiHeads es = e;
  const int gq = e.n_q / e.n_kv;
  es.raw = e.raw + static_cast<size_t>(s) * 8 * e.ldr;
  es.anchor_pos = e.anchor_pos + s;
  es.block_len = e.block_len + s;
  es.n_seq = 1;
  es.rows_ = 8;
  es.q_ready = e.q_ready + static_cast<size_t>(s) * e.n_kv * gq * 8 * e.d;
  es.Kst = e.Kst + static_cast<size_t>(s) * e.n_kv * e.cap * e.d;
  es.Vst = e.Vst + static_cast<size_t>(s) * e.n_kv * e.cap * e.d;
  es.process_head(hh, threadIdx.x);
}

cudaError_t launch_heads_rows(const EpiHeads& e, int n_heads, int n_seq, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_heads, n_seq);
  cfg.blockDim = dim3(128);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, heads_rows_kernel, e);
}

template <int WT>
static cudaError_t launch_tc(const GemvArgs& a, const TcEpi& e, int grid, cudaStream_t stream) {
  using Geo = TcGeo<WT>;
  cudaError_t err = cudaFuncSetAttribute(gemv_tc_kernel<WT>, cudaFuncAttributeMaxDynamicSharedMemorySize, Geo::SMEM);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kTcThreads);
  cfg.dynamicSmemBytes = Geo::SMEM;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemv_tc_kernel<WT>, a, e);
}

cudaError_t launch_gemv_tc(int wt, const GemvArgs& a, const TcEpi& e, int grid, cudaStream_t stream) {
  switch (wt) {
    case WT_BF16: return launch_tc<WT_BF16>(a, e, grid, stream);
    case WT_Q8_0: return launch_tc<WT_Q8_0>(a, e, grid, stream);
    case WT_Q5_0: return launch_tc<WT_Q5_0>(a, e, grid, stream);
    case WT_Q4_0: return launch_tc<WT_Q4_0>(a, e, grid, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace dflash

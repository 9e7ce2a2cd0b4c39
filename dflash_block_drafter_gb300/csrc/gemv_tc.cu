// Weight-streaming GEMM of a 128-row pass (9..16 sequences) on the tcgen05
// tensor cores.  At 128 activation rows every weight is used 128 times: the
// projections are real GEMMs (about 24 GFLOP per layer), which the legacy
// mma.sync GEMV issues far below its throughput.  Here:
//
//   warp 0      streams the CTA's weight units (64 rows x KU inputs, the
//               packed fragment-native format of the GEMV) into a ring of
//               3..4 stages that the decoders free;
//   warp 10     streams the activation chunks the units multiply (128 rows x
//               KU inputs per plane, 64-input tensor-map boxes in 128-byte
//               swizzle) in half chunks (KU / 2 inputs) into a ring of 3..4
//               half stages that the MMAs free;
//   warps 1..4  decode each unit with the GEMV's own decoders (warp w: 16-row
//               m-tile w) and write it, the GGUF block scale folded in (one
//               FP16 rounding of d * (q - offset)), as a 64 x KU K-major
//               operand in 128-byte swizzle (two tiles);
//   warp 5      issues tcgen05.mma kind::f16, M 128 (activation rows, A from
//               the chunk) x N 64 (the group's weight rows, B from the decoded
//               tile) x K 16, every plane, half by half as the chunk arrives,
//               into the group's FP32 accumulator -- 64 TMEM columns, 4 groups
//               in flight;
//   warps 6..9  read a finished group back (thread = activation row, its 64
//               outputs) and apply the epilogue: store, residual add, SwiGLU
//               into the down projection's chunked input, or the raw q/k/v,
//               whose per-head norm / RoPE / cell writes heads_rows_kernel
//               then applies with one CTA per (head, sequence).
//
// The weights and the activations travel separately, so the weight stream
// (HBM) runs ahead of the tensor cores by its ring and the decoders never
// wait for activations; a CTA with at most 4 groups takes its units
// input-major (for each chunk, every group's unit), one chunk serving all its
// groups.
//
// A CTA owns whole 64-row groups (grid <= groups), or, for matrices of few
// groups (the projections back to the hidden size), one of `parts` slices of
// a group's inputs; the slices' sums meet in global memory and the CTA that
// arrives last adds them in slice order and applies the epilogue.
#include "gemv_launch.cuh"
#include "kernels.h"

namespace dflash {

namespace {

constexpr int kTcThreads = 352;
constexpr int kTcSlots = 4;  // accumulators of 64 TMEM columns in flight
constexpr int kMaxParts = 4;  // input slices per group (the host plans at most this many)

template <int WT>
struct TcGeo {
  using F = Fmt<WT>;
  static constexpr int KU = F::CB * 32;
  static constexpr int PLANES = F::kF16 ? 1 : 2;  // GGUF: FP16 activations; BF16: hi and lo planes
  static constexpr int XBOX = 128 * 128;          // one 128-row x 64-input box: 16 KB
  static constexpr int BOXES = PLANES * (KU / 64);  // boxes of a unit's activation chunk (4 for every format)
  static constexpr int KBH = KU / 128;            // 64-input columns per half chunk and plane
  static constexpr int XHALF = (BOXES / 2) * XBOX;  // half a chunk: inputs [h * KU / 2, (h + 1) * KU / 2)
  static constexpr int BTILE = 64 * KU * 2;       // decoded unit, 16-bit
  static constexpr int NB = 2;  // decoded tiles, interleaved by 64-input column (btile_addr)
  static constexpr int BUDGET = 227 * 1024 - 2048;  // alignment slack and barriers
  // half-chunk stages and weight-unit stages: 4 and at least 3 where they fit, else 3
  static constexpr int XS = (BUDGET - 4 * XHALF - NB * BTILE) / F::UNIT >= 3 ? 4 : 3;
  static constexpr int WS0 = (BUDGET - XS * XHALF - NB * BTILE) / F::UNIT;
  static constexpr int WS = WS0 > 6 ? 6 : WS0;
  static constexpr int SMEM = 1024 + XS * XHALF + NB * BTILE + WS * F::UNIT + 1024;
  static_assert(BOXES == 4 && WS >= 2 && SMEM <= 227 * 1024, "GEMM stage plan");
  static_assert(F::UNIT % 1024 == 0, "weight units keep the 1024-byte alignment of what follows");
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
// K-major tile in 128-byte swizzle, 64-input columns of 64 rows x 128 bytes.
// The two tiles are interleaved column by column (tile t's column kb at
// (2 kb + t) * 8 KB), so that a column of both is one 128-row operand.
__device__ __forceinline__ uint32_t btile_addr(uint32_t tile_base, int R, int k0) {
  return tile_base + (k0 >> 6) * (2 * 64 * 128) + R * 128 + ((((k0 & 63) >> 3) ^ (R & 7)) << 4);
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
  constexpr int KU = Geo::KU, PLANES = Geo::PLANES, NB = Geo::NB, XS = Geo::XS, WS = Geo::WS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* xring = smem;                          // [XS][half chunk: BOXES / 2 boxes]
  uint8_t* btile = xring + XS * Geo::XHALF;       // [NB][64 x KU, 16-bit]
  uint8_t* wring = btile + NB * Geo::BTILE;       // [WS][weight unit]
  uint64_t* xfull = reinterpret_cast<uint64_t*>(wring + WS * F::UNIT);
  uint64_t* xempty = xfull + XS;      // MMA commit
  uint64_t* wfull = xempty + XS;
  uint64_t* wempty = wfull + WS;      // decoders (4)
  uint64_t* bfull = wempty + WS;      // [NB][2 halves] decoders (4)
  uint64_t* bempty = bfull + 2 * NB;  // [NB][2 halves] MMA commit
  uint64_t* accf = bempty + 2 * NB;   // [kTcSlots] MMA commit at a group's end
  uint64_t* acce = accf + kTcSlots;   // [kTcSlots] epilogue warps (4)
  uint64_t* mdone = acce + kTcSlots;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(mdone + 1);
  int* s_last = reinterpret_cast<int*>(s_tmem + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = static_cast<int>(gridDim.x);
  const int groups = a.U / a.UPG;
  // whole groups [g0, g1) per CTA, or (epi.parts > 1) part p of group g0's
  // inputs: units j in [jb, je) of each of the CTA's groups
  int g0, g1, jb, je, slice = blockIdx.x;
  if (epi.parts > 1) {
    // CTA p * groups + g
    const int p = blockIdx.x / groups;
    g0 = blockIdx.x - p * groups;
    g1 = g0 + 1;
    slice = g0 * epi.parts + p;
    jb = p * a.UPG / epi.parts;
    je = (p + 1) * a.UPG / epi.parts;
  } else {
    g0 = static_cast<int>(static_cast<long long>(blockIdx.x) * groups / G);
    g1 = static_cast<int>(static_cast<long long>(blockIdx.x + 1) * groups / G);
    jb = 0;
    je = a.UPG;
  }
  const int ng = g1 - g0, nj = je - jb;
  const int n_units = ng * nj;
  // Unit order.  With at most kTcSlots groups the units go input-major
  // (j outer, group inner): one activation chunk serves all the CTA's groups,
  // every group in its own accumulator.  Else group-major, a chunk per unit.
  const bool jmajor = ng <= kTcSlots;
  const int n_chunks = jmajor ? nj : n_units;
  auto unit_of = [&](int it, int& gi, int& j) {
    if (jmajor) {
      j = jb + it / ng;
      gi = it - (it / ng) * ng;
    } else {
      gi = it / nj;
      j = jb + it - gi * nj;
    }
  };
#ifdef DFLASH_TRACE
  unsigned long long* tr = a.trace ? a.trace + static_cast<size_t>(blockIdx.x) * kTraceSlots : nullptr;
  if (tr && tid == 0) tr[0] = globaltimer_ns();
  long long tw_a = 0, tw_b = 0;
#define TW(acc, expr) ([&]() { const long long t0_ = clock64(); const bool r_ = (expr); acc += clock64() - t0_; return r_; }())
#else
#define TW(acc, expr) (expr)
#endif

  if (tid == 0) {
    for (int s = 0; s < XS; ++s) {
      mbar_init(&xfull[s], 1);
      mbar_init(&xempty[s], 1);
    }
    for (int s = 0; s < WS; ++s) {
      mbar_init(&wfull[s], 1);
      mbar_init(&wempty[s], 4);
    }
    for (int b = 0; b < NB; ++b) {
      for (int h = 0; h < 2; ++h) {
        mbar_init(&bfull[2 * b + h], 4);
        mbar_init(&bempty[2 * b + h], 1);
      }
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
    // ---------------------------------------------------- weight producer
    if (lane == 0 && n_units > 0) {
      const uint64_t pol = l2_policy_evict_first();
      int issued = 0;
      for (int it = 0; it < n_units; ++it) {
        const int s = it % WS;
        if (it >= WS && !TW(tw_a, mbar_wait(&wempty[s], ((it / WS) - 1) & 1))) {
          ok = false;
          break;
        }
        int gi, j;
        unit_of(it, gi, j);
        mbar_arrive_expect_tx(&wfull[s], F::UNIT);
        bulk_g2s_hint(wring + s * F::UNIT, a.W + (static_cast<size_t>(g0 + gi) * a.UPG + j) * F::UNIT, F::UNIT,
                      &wfull[s], pol);
        issued = it + 1;
      }
      // every issued copy must land before the CTA may exit
      for (int it = (issued > WS ? issued - WS : 0); it < issued; ++it)
        if (!mbar_wait(&wfull[it % WS], (it / WS) & 1)) ok = false;
      if (!ok) set_status(a.status, DFLASH_DEV_TIMEOUT);
    }
  } else if (warp == 10) {
    // ------------------------------------------------ activation producer
    if (lane == 0 && n_units > 0) {
      prefetch_tensormap(&a.xmap);
      pdl_wait();  // the activations come from the previous kernel
#ifdef DFLASH_TRACE
      if (tr) tr[9] = globaltimer_ns();
#endif
      // half chunk q = 2 c + h of chunk c (inputs j's half h), stage q % XS
      const int nq = 2 * n_chunks;
      int issued = 0;
      for (int q = 0; q < nq; ++q) {
        const int s = q % XS, c = q >> 1, h = q & 1;
        if (q >= XS && !TW(tw_b, mbar_wait(&xempty[s], ((q / XS) - 1) & 1))) {
          ok = false;
          break;
        }
        int gi, j;
        unit_of(jmajor ? c * ng : c, gi, j);
        mbar_arrive_expect_tx(&xfull[s], Geo::XHALF);
        uint8_t* dst = xring + s * Geo::XHALF;
#pragma unroll
        for (int p = 0; p < PLANES; ++p)
#pragma unroll
          for (int kh = 0; kh < Geo::KBH; ++kh) {
            const int i = p * Geo::KBH + kh;  // box of the half
            const int x = (h * Geo::KBH + kh) * 64, y = (j * PLANES + p) * 128;
            tma_load_2d(dst + i * Geo::XBOX, &a.xmap, x, y, &xfull[s]);
          }
        issued = q + 1;
      }
      for (int q = (issued > XS ? issued - XS : 0); q < issued; ++q)
        if (!mbar_wait(&xfull[q % XS], (q / XS) & 1)) ok = false;
      if (!ok) set_status(a.status, DFLASH_DEV_TIMEOUT);
    } else if (lane == 0) {
      pdl_wait();
    }
  } else if (warp >= 1 && warp <= 4) {
    // ------------------------------------------------------------ decoders
    const int w = warp - 1;  // m-tile: weight rows 16 w .. 16 w + 15 of the group
    const int gr = lane >> 2, t4 = lane & 3;
    const uint32_t w_s = smem_u32(wring), bt_s = smem_u32(btile);
    // Units in steps (two units when the MMA pairs them, else one), each
    // step's tiles written half by half (inputs [0, KU / 2) of every unit of
    // the step, then the rest), so the MMA starts on a step's first half
    // while its second is decoded.
    const bool pair = jmajor && ng == 2;
    const int per = pair ? 2 : 1;
    for (int it0 = 0; it0 < n_units && ok; it0 += per) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        for (int t = 0; t < per && ok; ++t) {
          const int it = it0 + t;
          const int s = it % WS, b = it % NB;
          if (h == 0 && !TW(tw_a, mbar_wait(&wfull[s], (it / WS) & 1))) ok = false;
          if (ok && it >= NB && !TW(tw_b, mbar_wait(&bempty[2 * b + h], ((it / NB) - 1) & 1))) ok = false;
          if (!ok) break;
          const uint32_t ub = w_s + s * F::UNIT, bb = bt_s + b * (64 * 128);
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
            sts128(btile_addr(bb, w * 16 + gr + 8, k0), scale_pair<WT>(f.a[0][1], d8),
                   scale_pair<WT>(f.a[0][3], d8), scale_pair<WT>(f.a[1][1], d8), scale_pair<WT>(f.a[1][3], d8));
          };
          constexpr int HB = F::CB / 2;  // 32-input blocks per half
#pragma unroll
          for (int bl = h * HB; bl < (h + 1) * HB; bl += (WT == WT_Q4_0 || WT == WT_Q5_0) ? 2 : 1) {
            if constexpr (WT == WT_Q4_0 || WT == WT_Q5_0) {
              BlockFrag f0, f1;
              decode_pair<WT, F::kF16>(ub, w, lane, bl >> 1, f0, f1);
              put(bl, f0);
              put(bl + 1, f1);
            } else {
              put(bl, decode_block<WT, F::kF16>(ub, w, lane, bl));
            }
          }
          // generic-proxy writes of the half tile, then its hand-off to the
          // tensor cores (and, after the second half, the unit's codes are read)
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&bfull[2 * b + h]);
            if (h == 1) mbar_arrive(&wempty[s]);
          }
        }
      }
    }
    if (!ok && lane == 0) set_status(a.status, DFLASH_DEV_TIMEOUT);
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && n_units > 0) {
      // Two groups taken input-major: their units of one chunk sit in the
      // two decoded tiles, which make one 128-row operand -- one MMA of
      // N 128 into both groups' accumulators (adjacent TMEM columns).
      const bool pair = jmajor && ng == 2;
      const uint32_t idesc = pair ? idesc_16(128, 128, !F::kF16) : idesc_16(128, 64, !F::kF16);
      const uint32_t x_s = smem_u32(xring), bt_s = smem_u32(btile);
      const int n_steps = pair ? n_units / 2 : n_units;
      for (int stp = 0; stp < n_steps && ok; ++stp) {
        const int it = pair ? 2 * stp : stp;
        const int b = it % NB;
        int gi, j;
        unit_of(it, gi, j);
        const int slot = gi % kTcSlots;
        const int c = jmajor ? it / ng : it;             // the unit's chunk
        const bool new_chunk = !jmajor || gi == 0;
        const bool end_chunk = pair || !jmajor || gi == ng - 1;  // the chunk's last unit
        const bool first = j == jb, last = j == je - 1;  // the group's first / last unit here
        if (first && !jmajor && gi >= kTcSlots && !mbar_wait(&acce[slot], ((gi / kTcSlots) - 1) & 1)) {
          ok = false;
          break;
        }
        const uint32_t bs = bt_s + b * (64 * 128);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int q = 2 * c + h, s = q % XS;
          // this half of the step's decoded tiles
          if (!TW(tw_b, mbar_wait(&bfull[2 * b + h], (it / NB) & 1)) ||
              (pair && !TW(tw_b, mbar_wait(&bfull[2 * (b + 1) + h], ((it + 1) / NB) & 1)))) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (new_chunk) {
            if (!TW(tw_a, mbar_wait(&xfull[s], (q / XS) & 1))) {
              ok = false;
              break;
            }
            tc_fence_after();
          }
          const uint32_t xs = x_s + s * Geo::XHALF;
#pragma unroll
          for (int kq = 0; kq < KU / 32; ++kq) {  // the half's k-steps of 16 inputs
            const int kk = h * (KU / 32) + kq;
            const uint64_t db = umma_desc_sw128(bs + (kk >> 2) * (NB * 64 * 128) + (kk & 3) * 32, 16, 1024);
#pragma unroll
            for (int p = 0; p < PLANES; ++p) {
              const uint64_t da =
                  umma_desc_sw128(xs + (p * Geo::KBH + (kq >> 2)) * Geo::XBOX + (kq & 3) * 32, 16, 1024);
              umma_f16(tmem + slot * 64, da, db, idesc, (!first || kk || p) ? 1u : 0u);
            }
          }
          // the half chunk may be refilled once its last unit's MMAs are done,
          // the half tiles once these are
          if (end_chunk) umma_commit(&xempty[s]);
          umma_commit(&bempty[2 * b + h]);
          if (pair) umma_commit(&bempty[2 * (b + 1) + h]);
        }
        if (!ok) break;
        if (last) {
          umma_commit(&accf[slot]);
          if (pair) umma_commit(&accf[slot + 1]);
        }
      }
#ifdef DFLASH_TRACE
      if (tr) tr[10] = globaltimer_ns();
#endif
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
    bool staged_ok = false;
    for (int gi = 0; gi < ng; ++gi) {
      const int slot = gi % kTcSlots, g = g0 + gi;
      if (ok) ok = __all_sync(0xffffffffu, TW(tw_a, mbar_wait(&accf[slot], (gi / kTcSlots) & 1)));
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
        // part of the group's sum: published ([slice][16-byte column][row],
        // so that a warp's accesses are consecutive), then the CTA arriving
        // last adds every part in order and applies the epilogue
        float4* part4 = reinterpret_cast<float4*>(a.partials);
        float4* mine = part4 + static_cast<size_t>(slice) * 16 * 128 + n;
#pragma unroll
        for (int c4 = 0; c4 < 16; ++c4)
          __stcg(mine + c4 * 128, make_float4(v[4 * c4], v[4 * c4 + 1], v[4 * c4 + 2], v[4 * c4 + 3]));
        named_bar_sync(1, 128);
#ifdef DFLASH_TRACE
        if (tr && warp == 6 && lane == 0) tr[12] = globaltimer_ns();
#endif
        if (warp == 6 && lane == 0) s_last[0] = atomic_add_acq_rel(&a.counters[g], 1) == epi.parts - 1;
        named_bar_sync(1, 128);
#ifdef DFLASH_TRACE
        if (tr && warp == 6 && lane == 0) tr[13] = globaltimer_ns();
#endif
        const bool last_part = s_last[0] != 0;
        named_bar_sync(1, 128);  // s_last may be reused
        if (!last_part) continue;
        // every part's row, this CTA's own included, in part order; a quarter
        // row's loads of all parts are issued together, then added
#pragma unroll
        for (int c0 = 0; c0 < 16; c0 += 4) {
          float4 q4[kMaxParts][4];
#pragma unroll
          for (int p = 0; p < kMaxParts; ++p)
            if (p < epi.parts) {
              const float4* pp = part4 + static_cast<size_t>(g * epi.parts + p) * 16 * 128 + n;
#pragma unroll
              for (int c4 = 0; c4 < 4; ++c4) q4[p][c4] = __ldcg(pp + (c0 + c4) * 128);
            }
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            float4 acc4 = q4[0][c4];
#pragma unroll
            for (int p = 1; p < kMaxParts; ++p)
              if (p < epi.parts) {
                acc4.x += q4[p][c4].x;
                acc4.y += q4[p][c4].y;
                acc4.z += q4[p][c4].z;
                acc4.w += q4[p][c4].w;
              }
            const int c = 4 * (c0 + c4);
            v[c] = acc4.x;
            v[c + 1] = acc4.y;
            v[c + 2] = acc4.z;
            v[c + 3] = acc4.w;
          }
        }
#ifdef DFLASH_TRACE
        if (tr && warp == 6 && lane == 0) tr[11] = globaltimer_ns();
#endif
        if (warp == 6 && lane == 0) a.counters[g] = 0;
      }
      if (jmajor) {
        // every MMA is done once the last group's are (input-major order):
        // the activation ring is free, and each warp stages its 32 rows
        // there to write them out row-contiguously
        if (!staged_ok) {
          if (ok) ok = __all_sync(0xffffffffu, mbar_wait(mdone, 0));
          staged_ok = true;
        }
        epi.apply_staged(g, q, lane, v, reinterpret_cast<float*>(xring) + (warp - 6) * 32 * TcEpi::kStageLd);
      } else {
        epi.apply(g, n, v);
      }
    }
    if (!ok && lane == 0) set_status(a.status, DFLASH_DEV_TIMEOUT);
#ifdef DFLASH_TRACE
    if (tr && warp == 6 && lane == 0) tr[14] = globaltimer_ns();
#endif
  }
  // release the tensor memory once every tcgen05 operation of the CTA is done
#ifdef DFLASH_TRACE
  if (tr) {
    if (warp == 0 && lane == 0) { tr[1] = tw_a; }
    if (warp == 1 && lane == 0) { tr[2] = tw_a; tr[3] = tw_b; }
    if (warp == 5 && lane == 0) { tr[4] = tw_a; tr[5] = tw_b; }
    if (warp == 6 && lane == 0) { tr[6] = tw_a; tr[8] = n_units; }
  }
#endif
  // every warp whole again (lanes that finished their role early wait for
  // the one still working) before the CTA-wide barrier
  __syncwarp();
  tc_fence_before();
  __syncthreads();
#ifdef DFLASH_TRACE
  if (tr && tid == 0) tr[15] = globaltimer_ns();
#endif
#ifdef DFLASH_TRACE
  if (tr && threadIdx.x == 0) tr[7] = globaltimer_ns();
#endif
  if (warp == 5) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 64 * kTcSlots);
  }
#undef TW
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
    // the row's 16 loads first (in flight together), then the adds and stores
    float4* o = reinterpret_cast<float4*>(out + static_cast<size_t>(n) * ldo + g * 64);
    float4 x[16];
#pragma unroll
    for (int c4 = 0; c4 < 16; ++c4) x[c4] = __ldcg(o + c4);
#pragma unroll
    for (int c4 = 0; c4 < 16; ++c4) {
      x[c4].x += v[4 * c4];
      x[c4].y += v[4 * c4 + 1];
      x[c4].z += v[4 * c4 + 2];
      x[c4].w += v[4 * c4 + 3];
      __stcg(o + c4, x[c4]);
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

__device__ void TcEpi::apply_staged(int g, int q, int lane, const float (&v)[64], float* S) const {
  float* mine = S + lane * kStageLd;  // 272-byte rows: a quarter warp's 16-byte stores hit all 32 banks once
  if (mode == SWIGLU) {
    // per 16-row m-tile, 8 gate rows then the 8 up rows of outputs g * 32 + 8 w' + r
#pragma unroll
    for (int w2 = 0; w2 < 4; ++w2) {
      float hv[8];
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const float gt = v[w2 * 16 + r];
        hv[r] = gt / (1.f + __expf(-gt)) * v[w2 * 16 + 8 + r];
      }
      reinterpret_cast<float4*>(mine)[2 * w2] = make_float4(hv[0], hv[1], hv[2], hv[3]);
      reinterpret_cast<float4*>(mine)[2 * w2 + 1] = make_float4(hv[4], hv[5], hv[6], hv[7]);
    }
  } else {
#pragma unroll
    for (int c4 = 0; c4 < 16; ++c4)
      reinterpret_cast<float4*>(mine)[c4] = make_float4(v[4 * c4], v[4 * c4 + 1], v[4 * c4 + 2], v[4 * c4 + 3]);
  }
  __syncwarp();
  if (mode == SWIGLU) {
    // row r's 32 outputs are 64 contiguous bytes of its chunk row (per plane):
    // four lanes per row, eight rows per step
#pragma unroll
    for (int it = 0; it < 4; ++it) {
      const int r = it * 8 + (lane >> 2), pc = lane & 3;
      const float4 a = reinterpret_cast<const float4*>(S + r * kStageLd)[2 * pc];
      const float4 b = reinterpret_cast<const float4*>(S + r * kStageLd)[2 * pc + 1];
      const int o = g * 32 + pc * 8, n = q * 32 + r;
      if (h_f16) {
        *reinterpret_cast<uint4*>(static_cast<__half*>(h) + xchunk_index(o, n, 0, 128, h_ku, 1)) =
            make_uint4(pack_f16x2(a.x, a.y), pack_f16x2(a.z, a.w), pack_f16x2(b.x, b.y), pack_f16x2(b.z, b.w));
      } else {
        uint4 hi, lo;
        split_bf16x2(a.x, a.y, hi.x, lo.x);
        split_bf16x2(a.z, a.w, hi.y, lo.y);
        split_bf16x2(b.x, b.y, hi.z, lo.z);
        split_bf16x2(b.z, b.w, hi.w, lo.w);
        __nv_bfloat16* hp = static_cast<__nv_bfloat16*>(h);
        *reinterpret_cast<uint4*>(hp + xchunk_index(o, n, 0, 128, h_ku, 2)) = hi;
        *reinterpret_cast<uint4*>(hp + xchunk_index(o, n, 1, 128, h_ku, 2)) = lo;
      }
    }
  } else {
    // two rows per step: lanes 0..15 and 16..31 each cover one row's 64 outputs
    float* base = mode == HEADS ? heads.raw : out;
    const int ld = mode == HEADS ? heads.ldr : ldo;
    const int c4 = lane & 15;
    if (mode == RESID) {
      float4 x[16];
#pragma unroll
      for (int it = 0; it < 16; ++it) {
        const int n = q * 32 + 2 * it + (lane >> 4);
        x[it] = __ldcg(reinterpret_cast<const float4*>(base + static_cast<size_t>(n) * ld + g * 64) + c4);
      }
#pragma unroll
      for (int it = 0; it < 16; ++it) {
        const int r = 2 * it + (lane >> 4), n = q * 32 + r;
        const float4 y = reinterpret_cast<const float4*>(S + r * kStageLd)[c4];
        x[it].x += y.x;
        x[it].y += y.y;
        x[it].z += y.z;
        x[it].w += y.w;
        __stcg(reinterpret_cast<float4*>(base + static_cast<size_t>(n) * ld + g * 64) + c4, x[it]);
      }
    } else {
#pragma unroll
      for (int it = 0; it < 16; ++it) {
        const int r = 2 * it + (lane >> 4), n = q * 32 + r;
        __stcg(reinterpret_cast<float4*>(base + static_cast<size_t>(n) * ld + g * 64) + c4,
               reinterpret_cast<const float4*>(S + r * kStageLd)[c4]);
      }
    }
  }
  __syncwarp();  // S is reused by the next group
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
  if (e.parts > kMaxParts) return cudaErrorInvalidValue;
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

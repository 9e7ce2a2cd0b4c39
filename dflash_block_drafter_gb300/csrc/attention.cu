// Non-causal GQA block attention of the draft pass ("#1426 dflash:
// experimental standalone DeepSpec DFlash block drafter", sections "Target
// feature taps" -- non-causal block attention, scale 1/16 -- and "Drafter
// runtime" -- GQA 24 Q / 2 KV, head dim 256).
//
// For one slot and one kv head the queries are the GQ = n_q / n_kv q heads
// of the block's 8 rows: M = 8 * GQ rows (96 for DFlash) sharing every key,
// so QK^T and PV are real matrix products and run on the tcgen05 tensor
// cores.  The keys are the slot's position-addressed cells [0, p + B): the
// fused context plus the block's own rows, which the QKV epilogue wrote at
// [p, p + B).  The keys are split into chunks of 128-key super-tiles
// (split-K / flash-decode): a pass of n_seq sequences has n_seq * C chunks
// (one CTA each per kv head), shared out by chunk_plan so that sequences
// with longer contexts get more of them and every chunk has about the same
// number of super-tiles.  With C > 1 every chunk writes (O unnormalised,
// running max, sum) and attn_combine_kernel merges each sequence's chunks
// with the log-sum-exp rule; with C == 1 (one chunk per sequence) the CTA
// normalises and writes the output directly.
#include "kernels.h"
#include "layout.cuh"

namespace dflash {

struct AttnArgs {
  CUtensorMap qmap;  // queries [slots * n_kv * M, d] fp16, 64 x M boxes (normed, rotated, scaled by 1/sqrt(d))
  CUtensorMap kmap;  // K arena as [rows, d] fp16
  CUtensorMap vmap;
  const int32_t* anchor_pos;
  const int32_t* block_len;
  CUtensorMap pmap;       // chunk partials O / l: [slots * n_kv * C * M, d] fp16, 64 x M boxes
  float2* ml;             // [slots, n_kv, C, M]: running max (log2 units) and sum per row
  void* out;              // attention output in the o-projection's chunked X layout (C == 1)
  int out_f16;            // 1: one FP16 plane; 0: BF16 hi and lo planes
  int out_rows, out_ku;   // chunked layout: rows R of the pass and inputs per unit
  int layer, n_slots, n_kv, n_q, gq, cap, n_seq;
  int Q;                  // chunks of the pass per kv head (grid x; chunk_plan shares them out)
  int window;             // 0: keys [0, p + B), cell = position; W > 0: keys
                          // [max(0, p + B - W), p + B) in a ring, cell = position mod cap
  int32_t* status;
  unsigned long long* trace;  // diagnostic builds only (DFLASH_TRACE): per-CTA timestamps
  const __half* kbase_ptr;    // the K / V arenas (rows of d halves) the maps address
  const __half* vbase_ptr;
  int* plan;                  // [n_seq] out (passes of several sequences): start_s | c_s << 16
};

#ifdef DFLASH_TRACE
#define DFLASH_ATTN_STAMP(k)                                                                                  \
  do {                                                                                                        \
    if (a.trace)                                                                                              \
      a.trace[(static_cast<size_t>(blockIdx.z) * gridDim.y * gridDim.x + blockIdx.y * gridDim.x + blockIdx.x) * kTraceSlots + \
              (k)] = globaltimer_ns();                                                                        \
  } while (0)
#else
#define DFLASH_ATTN_STAMP(k) \
  do {                       \
  } while (0)
#endif

// ---------------------------------------------------------------------------
// tcgen05 attention.  Per CTA (chunk, kv head, slot) the M = 8 * GQ query rows
// (96 for DFlash) are multiplied against the chunk's keys in super-tiles of
// 128 keys:
//   warp 0       TMA producer: Q once (one barrier per 64-column box), then
//                per super-tile two 64-key K tiles and two V tiles (64 x 64
//                boxes, 128-byte swizzle; a K box's two tiles back to back);
//   warp 1       owns the tensor memory and, from one thread, issues
//                tcgen05.mma: S[j % 2] = Q K_j^T (M 128, N 128, K 16 per
//                instruction, FP32 in TMEM) and O += P_j V_j (N = d, V read
//                MN-major straight from its TMA tile);
//   warps 2..17  softmax: warp w reads TMEM lane quarter w % 4 (query rows
//                32 (w % 4) ..) and key slice (w - 2) / 4 (32 of the 128 keys;
//                d / 4 columns of O).  Row maxima are combined across the 4
//                slices through shared memory; P = 2^(s - m) goes to shared
//                memory as FP16 in the 128-byte-swizzled K-major layout the
//                MMA reads; O is rescaled in TMEM when a row's maximum grows.
// S is double-buffered in TMEM so the next super-tile's QK^T overlaps the
// softmax; O (d columns) accumulates in TMEM across the chunk.
//
// Q occupies only its M rows per 64-column box; the MMA's rows M..127 read
// whatever follows (the next box, or the K buffer): values whose scores,
// probabilities and outputs stay in those rows and are never used.
// A lane quarter with no query row skips the softmax arithmetic.
//
// Every wait is bounded.  After a timeout a warp stops waiting but still
// takes every named barrier of the softmax group, so all warps finish.
constexpr int kTcKT = 64;                             // keys per TMA tile
constexpr int kTcKS = 2 * kTcKT;                      // keys per super-tile
constexpr int kTcTmemCols = 512;                      // S0 [0,128), S1 [128,256), O [256, 256 + d)
constexpr int kTcSoftWarps = 16;                      // 4 per TMEM lane quarter
constexpr int kTcSoftThreads = 32 * kTcSoftWarps;
constexpr int kTcThreads = 64 + kTcSoftThreads;

template <int D>
struct TcGeom {
  static constexpr int BOXES = D / 64;
  static constexpr int TILE_BYTES = kTcKT * D * 2;
  static constexpr int P_BYTES = 128 * kTcKS * 2;
  static constexpr int RED_BYTES = (2 * 4 * 128 + 4 * 128) * 4;  // row maxima (double-buffered), row sums
  // Q rows: M x D FP16 (a multiple of 1024 bytes for M % 16 == 0)
  static __host__ __device__ constexpr int q_bytes(int M) { return M * D * 2; }
  static __host__ __device__ constexpr int smem(int M) {
    return 1024 + q_bytes(M) + 4 * TILE_BYTES + P_BYTES + RED_BYTES + 256;
  }
};

// N consecutive columns (16, 32 or 64) of this thread's TMEM lane, times `scale`.
template <int N>
__device__ __forceinline__ void tmem_load_cols(uint32_t addr, float (&v)[N], float scale) {
  if constexpr (N == 16) {
    uint32_t r[16];
    tmem_ld16(addr, r);
    tmem_wait_ld();
    tmem_reg_fence(r);
#pragma unroll
    for (int e = 0; e < 16; ++e) v[e] = __uint_as_float(r[e]) * scale;
  } else {
    static_assert(N % 32 == 0 && N <= 64, "column count");
    uint32_t r[N / 32][32];
#pragma unroll
    for (int h = 0; h < N / 32; ++h) tmem_ld32(addr + h * 32, r[h]);
    tmem_wait_ld();
#pragma unroll
    for (int h = 0; h < N / 32; ++h) {
      tmem_reg_fence(r[h]);
#pragma unroll
      for (int e = 0; e < 32; ++e) v[h * 32 + e] = __uint_as_float(r[h][e]) * scale;
    }
  }
}

// Multiply N consecutive columns of this thread's TMEM lane by `scale` in place.
template <int N>
__device__ __forceinline__ void tmem_scale_cols(uint32_t addr, float scale) {
  if constexpr (N == 16) {
    uint32_t r[16];
    tmem_ld16(addr, r);
    tmem_wait_ld();
    tmem_reg_fence(r);
    uint32_t w[32];
#pragma unroll
    for (int e = 0; e < 16; ++e) w[e] = __float_as_uint(__uint_as_float(r[e]) * scale);
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            addr),
        "r"(w[0]), "r"(w[1]), "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7]), "r"(w[8]), "r"(w[9]),
        "r"(w[10]), "r"(w[11]), "r"(w[12]), "r"(w[13]), "r"(w[14]), "r"(w[15])
        : "memory");
  } else {
#pragma unroll 1
    for (int h = 0; h < N / 32; ++h) {
      uint32_t r[32];
      tmem_ld32(addr + h * 32, r);
      tmem_wait_ld();
      tmem_reg_fence(r);
#pragma unroll
      for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * scale);
      tmem_st32(addr + h * 32, r);
    }
  }
  tmem_wait_st();
}

// Key super-tiles of sequence s in a pass: positions [lo, T) taken from the
// tile-aligned base kbase (lo = 0, or T - window with a ring of cells).
struct SeqKeys {
  int p, B, T, lo, kbase, tiles;
};
__device__ __forceinline__ SeqKeys seq_keys(const int32_t* anchor_pos, const int32_t* block_len, int s, int window,
                                            int cap) {
  SeqKeys k;
  k.p = anchor_pos[s];
  int B = block_len[s];
  k.B = B < DFLASH_MIN_BLOCK ? DFLASH_MIN_BLOCK : (B > DFLASH_MAX_BLOCK ? DFLASH_MAX_BLOCK : B);
  int T = k.p + k.B;
  int lo = 0;
  if (window > 0) {
    T = T < 0 ? 0 : T;
    lo = T - window < 0 ? 0 : T - window;
  } else {
    T = T < 0 ? 0 : (T > cap ? cap : T);
  }
  k.T = T;
  k.lo = lo;
  k.kbase = lo - lo % kTcKS;
  k.tiles = (T - k.kbase + kTcKS - 1) / kTcKS;
  return k;
}

// Chunk plan of a pass, computed by a whole warp (lane s holds sequence s,
// n_seq <= 32): the pass's Q chunks (per kv head) are shared out so that the
// longest chunk is as short as possible -- sequence s takes
// c_s = max(1, ceil(tiles_s / t)) chunks of t super-tiles (its last one
// shorter), t the smallest count with sum_s c_s <= Q (found by bisection; a
// single sequence gets t = ceil(tiles / Q) directly).  Chunks are numbered
// sequence after sequence: sequence s owns [start_s, start_s + c_s).
// Returns t; this lane's c_s and start_s in *cs / *start (lanes >= n_seq: 0).
__device__ int chunk_plan(const int32_t* anchor_pos, const int32_t* block_len, int n_seq, int Q, int window,
                          int cap, int lane, int* cs, int* start) {
  const int tiles = lane < n_seq ? seq_keys(anchor_pos, block_len, lane, window, cap).tiles : 0;
  int t;
  if (n_seq == 1) {
    t = (tiles + Q - 1) / Q;
    t = __shfl_sync(0xffffffffu, t, 0);
    if (t < 1) t = 1;
  } else {
    int hi = tiles;
#pragma unroll
    for (int o = 16; o; o >>= 1) hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    hi = hi < 1 ? 1 : hi;
    int lo = 1;
    while (lo < hi) {  // uniform across the warp
      const int mid = (lo + hi) >> 1;
      int cnt = lane < n_seq ? max(1, (tiles + mid - 1) / mid) : 0;
#pragma unroll
      for (int o = 16; o; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
      if (cnt <= Q) hi = mid;
      else lo = mid + 1;
    }
    t = lo;
  }
  const int c = lane < n_seq ? max(1, (tiles + t - 1) / t) : 0;
  int incl = c;  // inclusive prefix sum over the lanes
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  *cs = c;
  *start = incl - c;
  return t;
}

template <int D>
__global__ void __launch_bounds__(kTcThreads, 1) attn_tc_kernel(const __grid_constant__ AttnArgs a) {
  using Geo = TcGeom<D>;
  constexpr int OC = D / 4;  // O columns per softmax warp
  const int M = a.gq * 8;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sq = smem;                                  // [D/64 boxes][M rows][128 B]
  uint8_t* sk = sq + Geo::q_bytes(M);                  // 2 tiles of [D/64 boxes][64 keys][128 B]
  uint8_t* sv = sk + 2 * Geo::TILE_BYTES;              // 2 tiles
  uint8_t* sp = sv + 2 * Geo::TILE_BYTES;              // [2 boxes][128 rows][128 B]
  float* red_max = reinterpret_cast<float*>(sp + Geo::P_BYTES);  // [2][4 slices][128 rows]
  float* red_l = red_max + 2 * 4 * 128;                          // [4 slices][128 rows]
  uint64_t* bars = reinterpret_cast<uint64_t*>(red_l + 4 * 128);
  uint64_t* qfull = bars + 0;   // [D / 64]: one per 64-column box of Q
  uint64_t* kfull = bars + 4;
  uint64_t* kfree = bars + 5;
  uint64_t* vfull = bars + 6;   // [2]: one per 64-key V tile
  uint64_t* vfree = bars + 8;   // [2]
  uint64_t* sfull = bars + 10;  // [2]
  uint64_t* sfree = bars + 12;  // [2]
  uint64_t* pfull = bars + 14;
  uint64_t* pfree = bars + 15;
  uint64_t* mdone = bars + 16;  // every MMA of the CTA has completed
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + 17);
  int* s_plan = reinterpret_cast<int*>(s_tmem + 1);  // [4]: sequence, its chunk, super-tiles per chunk, idle

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = blockIdx.y;
  if (tid == 0) DFLASH_ATTN_STAMP(0);

  // this CTA's chunk q of the pass (grid x: Q of them) -> its
  // sequence s and chunk c of that sequence (chunk_plan; none: idle)
  // (formed by warp 0 and handed to the others through shared memory; the
  // first CTA also publishes the plan for the merge kernel)
  const int q = blockIdx.x;
  int s = 0, c = blockIdx.x, spc;
  bool idle = false;
  if (a.n_seq == 1) {
    // one sequence: its C chunks, as the plan would give them
    spc = max(1, (seq_keys(a.anchor_pos, a.block_len, 0, a.window, a.cap).tiles + a.Q - 1) / a.Q);
  } else {
    // several sequences (comment above)
    if (warp == 0) {
      int cs_l, start_l;
      const int t = chunk_plan(a.anchor_pos, a.block_len, a.n_seq, a.Q, a.window, a.cap, lane, &cs_l, &start_l);
      const unsigned own = __ballot_sync(0xffffffffu, lane < a.n_seq && q >= start_l && q < start_l + cs_l);
      const int so = own ? __ffs(own) - 1 : 0;
      const int co = q - __shfl_sync(0xffffffffu, start_l, so);
      if (lane == 0) {
        s_plan[0] = so;
        s_plan[1] = own ? co : 0;
        s_plan[2] = t;
        s_plan[3] = own ? 0 : 1;
      }
      if (a.plan && q == 0 && g == 0 && lane < a.n_seq) a.plan[lane] = start_l | (cs_l << 16);
    }
    __syncthreads();
    s = s_plan[0];
    c = s_plan[1];
    spc = s_plan[2];
    idle = s_plan[3] != 0;
  }
  // key positions [lo, T), in super-tiles of kTcKS positions from `kbase`
  // (lo rounded down to a super-tile); with a window the cells are a ring and
  // a super-tile (cap % kTcKS == 0) is one contiguous run of cells
  const SeqKeys sk_ = seq_keys(a.anchor_pos, a.block_len, s, a.window, a.cap);
  const int p = sk_.p, T = sk_.T, lo = sk_.lo, kbase = sk_.kbase;
  const int nst_all = sk_.tiles;
  const int st0 = c * spc;
  const int st1 = min(nst_all, st0 + spc);
  const int nst = (!idle && st1 > st0) ? st1 - st0 : 0;
  const int row0 = ((a.layer * a.n_slots + s) * a.n_kv + g) * a.cap;

  if (tid == 0) {
    for (int b = 0; b < Geo::BOXES; ++b) mbar_init(&qfull[b], 1);
    mbar_init(kfull, 1);
    mbar_init(kfree, 1);
    for (int t = 0; t < 2; ++t) {
      mbar_init(&vfull[t], 1);
      mbar_init(&vfree[t], 1);
    }
    mbar_init(&sfull[0], 1);
    mbar_init(&sfull[1], 1);
    mbar_init(&sfree[0], kTcSoftWarps);
    mbar_init(&sfree[1], kTcSoftWarps);
    mbar_init(pfull, kTcSoftWarps);
    mbar_init(pfree, 1);
    mbar_init(mdone, 1);
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(s_tmem, kTcTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  bool ok = true;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0 && nst > 0) {
      prefetch_tensormap(&a.qmap);
      prefetch_tensormap(&a.kmap);
      prefetch_tensormap(&a.vmap);
      auto tile_row = [&](int j) {
        const int pos = kbase + (st0 + j) * kTcKS;
        return row0 + (a.window > 0 ? pos % a.cap : pos);
      };
      auto issue_k = [&](int j) {
        const int y = tile_row(j);
        mbar_arrive_expect_tx(kfull, 2 * Geo::TILE_BYTES);
        for (int t = 0; t < 2; ++t)
          for (int b = 0; b < Geo::BOXES; ++b)
            tma_load_2d(sk + b * (kTcKS * 128) + t * (kTcKT * 128), &a.kmap, b * 64, y + t * kTcKT, kfull);
      };
      // tiles kLookAhead super-tiles ahead are asked of L2, so that long
      // chunks find their next K / V there instead of waiting on HBM
      constexpr int kLookAhead = 2;
      auto prefetch_tile = [&](int j) {
        if (j >= nst) return;
        const int row = tile_row(j);
        // the super-tile's cells that exist in this (layer, slot, kv head) slab
        const int n_rows = min(kTcKS, row0 + a.cap - row);
        if (n_rows <= 0) return;
        const uint32_t bytes = static_cast<uint32_t>(n_rows * D * 2);
        bulk_prefetch_l2_plain(a.kbase_ptr + static_cast<size_t>(row) * D, bytes);
        bulk_prefetch_l2_plain(a.vbase_ptr + static_cast<size_t>(row) * D, bytes);
      };
      // V tile t of super-tile j: its buffer is refilled as soon as the PV
      // MMAs of the previous super-tile's tile t are done
      auto issue_v_tile = [&](int j, int t) {
        const int y = tile_row(j);
        mbar_arrive_expect_tx(&vfull[t], Geo::TILE_BYTES);
        for (int b = 0; b < Geo::BOXES; ++b)
          tma_load_2d(sv + t * Geo::TILE_BYTES + b * kTcKT * 128, &a.vmap, b * 64, y + t * kTcKT, &vfull[t]);
      };
      auto issue_v = [&](int j) {
        issue_v_tile(j, 0);
        issue_v_tile(j, 1);
      };
      // A first super-tile wholly before the block's positions does not
      // depend on the previous kernel (which writes the block cells; in a
      // ring they cannot be the cells of a position inside the window).
      const bool early = kbase + (st0 + 1) * kTcKS <= p;
      if (early) {
        issue_k(0);
        issue_v(0);
      }
      pdl_wait();
      DFLASH_ATTN_STAMP(8);
      for (int b = 0; b < Geo::BOXES; ++b) {
        mbar_arrive_expect_tx(&qfull[b], M * 128);
        tma_load_2d(sq + b * (M * 128), &a.qmap, b * 64, (s * a.n_kv + g) * M, &qfull[b]);
      }
      if (!early) {
        issue_k(0);
        issue_v(0);
      }
      for (int j = 1; j <= kLookAhead; ++j) prefetch_tile(j);
      int nk = 1, nv = 1;  // super-tiles issued
      for (int j = 1; j < nst; ++j) {
        prefetch_tile(j + kLookAhead);
        if (!mbar_wait(kfree, (j - 1) & 1)) { ok = false; break; }
        issue_k(j);
        ++nk;
        if (!mbar_wait(&vfree[0], (j - 1) & 1)) { ok = false; break; }
        issue_v_tile(j, 0);
        if (!mbar_wait(&vfree[1], (j - 1) & 1)) { ok = false; break; }
        issue_v_tile(j, 1);
        ++nv;
      }
      // Only the last K and V copies can still be in flight (each earlier one
      // was consumed before its buffer was refilled); they and Q must land
      // before the CTA may exit, also after a timeout.
      for (int b = 0; b < Geo::BOXES; ++b)
        if (!mbar_wait(&qfull[b], 0)) ok = false;
      if (!mbar_wait(kfull, (nk - 1) & 1)) ok = false;
      for (int t = 0; t < 2; ++t)
        if (!mbar_wait(&vfull[t], (nv - 1) & 1)) ok = false;
      if (!ok) set_status(a.status, DFLASH_DEV_TIMEOUT);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && nst > 0) {
      // one MMA covers the super-tile's 128 keys: the two 64-key tiles of a
      // 64-column box lie back to back, 128 rows of 128 bytes
      constexpr uint32_t idesc_qk = umma_idesc_f16(128, kTcKS, false, false);
      constexpr uint32_t idesc_pv = umma_idesc_f16(128, D, false, true);
      const uint32_t q_s = smem_u32(sq), k_s = smem_u32(sk), v_s = smem_u32(sv), p_s = smem_u32(sp);
      const uint32_t q_box = static_cast<uint32_t>(M) * 128;
      // S[j % 2] = Q K_j^T; the K buffer is released when it completes.  The
      // first super-tile takes each 64-column box of Q as it lands (rows M..127
      // of a box's MMAs read the next box's memory, landed or not: values
      // confined to those rows, which nothing uses).
      auto issue_qk = [&](int j) -> bool {
        if (!mbar_wait(kfull, j & 1)) return false;
        if (j == 0) DFLASH_ATTN_STAMP(10);
        if (j >= 2 && !mbar_wait(&sfree[j & 1], ((j >> 1) - 1) & 1)) return false;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          if (j == 0 && (kk & 3) == 0) {
            if (!mbar_wait(&qfull[kk >> 2], 0)) return false;
            tc_fence_after();
          }
          const uint64_t da = umma_desc_sw128(q_s + (kk >> 2) * q_box + (kk & 3) * 32, 16, 1024);
          const uint64_t db = umma_desc_sw128(k_s + (kk >> 2) * (kTcKS * 128) + (kk & 3) * 32, 16, 1024);
          umma_f16(tmem + (j & 1) * kTcKS, da, db, idesc_qk, kk > 0);
        }
        umma_commit(&sfull[j & 1]);
        umma_commit(kfree);
        return true;
      };
      // QK^T of super-tile j + 1 runs while the softmax warps work on S[j % 2]:
      // it is issued as soon as its K tile (and S buffer) is there, and the PV
      // of super-tile j as soon as P_j and V_j are -- whichever is ready first
      // goes first, so a late K tile never holds up the PV before it.
      DFLASH_ATTN_STAMP(9);
      if (!issue_qk(0)) ok = false;
      DFLASH_ATTN_STAMP(11);
      for (int j = 0; j < nst && ok; ++j) {
        bool qk_next = j + 1 < nst;
        // wait for `ready`, issuing QK^T of super-tile j + 1 meanwhile if its
        // K tile and S buffer come first
        auto spin_until = [&](auto ready) -> bool {
          const unsigned long long t0 = globaltimer_ns();
          for (int spin = 0;; ++spin) {
            if (qk_next && mbar_test(kfull, (j + 1) & 1) &&
                (j + 1 < 2 || mbar_test(&sfree[(j + 1) & 1], (((j + 1) >> 1) - 1) & 1))) {
              if (!issue_qk(j + 1)) return false;
              qk_next = false;
            }
            if (ready()) return true;
            if ((spin & 63) == 63 && globaltimer_ns() - t0 > kWaitTimeoutNs) return false;
          }
        };
        // PV tile by tile: each V tile's buffer is released once its MMAs are done
        for (int t = 0; t < 2 && ok; ++t) {
          if (!spin_until([&]() { return (t > 0 || mbar_test(pfull, j & 1)) && mbar_test(&vfull[t], j & 1); })) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kTcKT / 16; ++kk) {
            const uint64_t da = umma_desc_sw128(p_s + t * 16384 + kk * 32, 16, 1024);
            const uint64_t db = umma_desc_sw128(v_s + t * Geo::TILE_BYTES + kk * 2048, kTcKT * 128, 1024);
            umma_f16(tmem + 2 * kTcKS, da, db, idesc_pv, (j > 0 || t > 0 || kk > 0) ? 1u : 0u);
          }
          if (t == 1) umma_commit(pfree);
          umma_commit(&vfree[t]);
        }
        if (!ok) break;
        if (qk_next && !issue_qk(j + 1)) { ok = false; break; }
      }
      // tensor memory may only be freed once every issued MMA has finished
      umma_commit(mdone);
      if (!mbar_wait(mdone, 0)) ok = false;
      if (!ok) set_status(a.status, DFLASH_DEV_TIMEOUT);
    }
  } else {
    // ------------------------------------------------------------ softmax
    pdl_wait();
    pdl_launch_dependents();
    constexpr float LOG2E = 1.4426950408889634f;
    const int q4 = warp & 3;                 // TMEM lane quarter this warp may access
    const int cs = (warp - 2) >> 2;          // key slice (32 of 128) and O column slice (d / 4)
    const int m = q4 * 32 + lane;            // query row = TMEM lane
    const bool live = q4 * 32 < M;           // warp-uniform: the quarter holds query rows
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(q4 * 32) << 16);
    const uint32_t o_addr = lane_addr + 2 * kTcKS + cs * OC;
    float m_run = -INFINITY, l_part = 0.f;
    for (int j = 0; j < nst; ++j) {
      const int b = j & 1;
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(&sfull[b], (j >> 1) & 1));
      if (tid == 64 && j == 0) DFLASH_ATTN_STAMP(1);
      tc_fence_after();
      uint32_t r[32];
      if (live) {
        tmem_ld32(lane_addr + b * kTcKS + cs * 32, r);
        tmem_wait_ld();
        tmem_reg_fence(r);
      }
      // S[b] has been read: the next-but-one QK^T may overwrite it
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&sfree[b]);
      // keys e of this slice with lo <= position < T take weight (the last
      // super-tile's tail and, with a window, the first one's head take none)
      const int spos = kbase + (st0 + j) * kTcKS + cs * 32;
      const int khi = min(T - spos, 32), klo = max(lo - spos, 0);
      const bool full_slice = klo == 0 && khi >= 32;
      float mx = -INFINITY;
      if (live) {
        if (full_slice) {
#pragma unroll
          for (int e = 0; e < 32; ++e) mx = fmaxf(mx, __uint_as_float(r[e]));
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (e >= klo && e < khi) mx = fmaxf(mx, __uint_as_float(r[e]));
        }
      }
      if (tid == 64 && j == 0) DFLASH_ATTN_STAMP(2);
      // row maximum over the 4 key slices
      red_max[b * 512 + cs * 128 + m] = mx;
      named_bar_sync(1, kTcSoftThreads);
      {
        const float* rm = red_max + b * 512 + m;
        mx = fmaxf(fmaxf(rm[0], rm[128]), fmaxf(rm[256], rm[384]));
      }
      if (tid == 64 && j == 0) DFLASH_ATTN_STAMP(3);
      const float m_new = fmaxf(m_run, mx * LOG2E);
      const float base = m_new == -INFINITY ? 0.f : m_new;
      const float alpha = ex2_approx(m_run - base);  // 0 on the first super-tile
      // P buffer and O are free once the previous super-tile's PV is done
      if (j > 0) {
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(pfree, (j - 1) & 1));
        tc_fence_after();
        if (live && __any_sync(0xffffffffu, alpha < 1.f)) tmem_scale_cols<OC>(o_addr, alpha);
      }
      // P = 2^(s - m) as FP16: keys 32 cs .. 32 cs + 31 are box cs / 2,
      // 16-byte chunks (cs % 2) * 4 .. + 3 of the row
      float ls = 0.f;
      if (live) {
        uint32_t pk[16];
        if (full_slice) {
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float p0 = ex2_approx(fmaf(__uint_as_float(r[e]), LOG2E, -base));
            const float p1 = ex2_approx(fmaf(__uint_as_float(r[e + 1]), LOG2E, -base));
            ls += p0 + p1;
            pk[e >> 1] = pack_f16x2(p0, p1);
          }
        } else {
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float p0 =
                (e >= klo && e < khi) ? ex2_approx(fmaf(__uint_as_float(r[e]), LOG2E, -base)) : 0.f;
            const float p1 =
                (e + 1 >= klo && e + 1 < khi) ? ex2_approx(fmaf(__uint_as_float(r[e + 1]), LOG2E, -base)) : 0.f;
            ls += p0 + p1;
            pk[e >> 1] = pack_f16x2(p0, p1);
          }
        }
        uint8_t* prow = sp + (cs >> 1) * 16384 + m * 128;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int ch = ((cs & 1) * 4 + q) ^ (m & 7);
          *reinterpret_cast<uint4*>(prow + ch * 16) = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        }
      }
      if (tid == 64 && j == 0) DFLASH_ATTN_STAMP(4);
      l_part = l_part * alpha + ls;
      m_run = m_new;
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(pfull);
      if (tid == 64 && j == 0) DFLASH_ATTN_STAMP(5);
    }
    // final O (after the last PV)
    if (ok && nst > 0) ok = __all_sync(0xffffffffu, mbar_wait(pfree, (nst - 1) & 1));
    tc_fence_after();
    if (tid == 64) DFLASH_ATTN_STAMP(6);
    if (!ok && lane == 0) set_status(a.status, DFLASH_DEV_TIMEOUT);
    // row sum over the 4 key slices, in a fixed order
    red_l[cs * 128 + m] = l_part;
    named_bar_sync(1, kTcSoftThreads);
    const float l_run = (red_l[m] + red_l[128 + m]) + (red_l[256 + m] + red_l[384 + m]);
    const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
    if (a.Q == a.n_seq) {  // one chunk per sequence
      // normalised rows straight into the o-projection's input layout
      if (live) {
        float v[OC];
        if (nst > 0) {
          tmem_load_cols<OC>(o_addr, v, inv);
        } else {
#pragma unroll
          for (int e = 0; e < OC; ++e) v[e] = 0.f;
        }
        if (m < M) {
          if (cs == 0 && !(l_run > 0.f)) set_status(a.status, DFLASH_DEV_NONFINITE);
          const int hl = m >> 3, i = m & 7;
          const int P = a.out_f16 ? 1 : 2;
          const int row = s * 8 + i, col0 = (g * a.gq + hl) * D + cs * OC;
          const size_t lo_off = static_cast<size_t>(a.out_rows) * (a.out_ku + 32);
#pragma unroll
          for (int e8 = 0; e8 < OC; e8 += 8) {
            const size_t o = xchunk_index(col0 + e8, row, 0, a.out_rows, a.out_ku, P);
            if (a.out_f16) {
              *reinterpret_cast<uint4*>(static_cast<__half*>(a.out) + o) =
                  make_uint4(pack_f16x2(v[e8], v[e8 + 1]), pack_f16x2(v[e8 + 2], v[e8 + 3]),
                             pack_f16x2(v[e8 + 4], v[e8 + 5]), pack_f16x2(v[e8 + 6], v[e8 + 7]));
            } else {
              uint4 hi, lo;
              split_bf16x2(v[e8], v[e8 + 1], hi.x, lo.x);
              split_bf16x2(v[e8 + 2], v[e8 + 3], hi.y, lo.y);
              split_bf16x2(v[e8 + 4], v[e8 + 5], hi.z, lo.z);
              split_bf16x2(v[e8 + 6], v[e8 + 7], hi.w, lo.w);
              *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) + o) = hi;
              *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) + o + lo_off) = lo;
            }
          }
        }
      }
    } else {
      // The chunk's partial: O / l as FP16 rows plus (m, l) per row.  The rows
      // are staged in the K buffer (free: the last QK^T completed before the
      // last softmax) as D/64 boxes of M rows x 128 bytes with the 128-byte
      // swizzle, then written by tensor-map stores.  An empty chunk writes
      // only (m, l) = (-inf, 0); the merge gives it no weight.
      // chunk partials of kv head g: [Q chunks of the pass][M] (chunk_plan's numbering)
      const size_t pbase = (static_cast<size_t>(g) * a.Q + q) * M;
      if (nst > 0) {
        if (live) {
          float v[OC];
          tmem_load_cols<OC>(o_addr, v, inv);
          if (m < M) {
            const int col0 = cs * OC;
            uint8_t* row = sk + (col0 >> 6) * (M * 128) + m * 128;
#pragma unroll
            for (int q = 0; q < OC / 8; ++q)
              *reinterpret_cast<uint4*>(row + (((((col0 & 63) >> 3) + q) ^ (m & 7)) << 4)) =
                  make_uint4(pack_f16x2(v[8 * q], v[8 * q + 1]), pack_f16x2(v[8 * q + 2], v[8 * q + 3]),
                             pack_f16x2(v[8 * q + 4], v[8 * q + 5]), pack_f16x2(v[8 * q + 6], v[8 * q + 7]));
          }
        }
        fence_proxy_async_smem();
        named_bar_sync(1, kTcSoftThreads);
        if (tid == 64) {
          for (int h = 0; h < D / 64; ++h) tma_store_2d(&a.pmap, h * 64, static_cast<int>(pbase), sk + h * (M * 128));
          bulk_commit_group();
          DFLASH_ATTN_STAMP(12);
          bulk_wait_group_read_0();  // the staging buffer may be released; the writes land with the grid
          DFLASH_ATTN_STAMP(13);
        }
      }
      if (cs == 0 && m < M) __stcg(a.ml + pbase + m, make_float2(m_run, l_run));
    }
  }
  // release the tensor memory once every tcgen05 operation of the CTA is done
  // every warp whole again (lanes that finished their role early wait for
  // the one still working) before the CTA-wide barrier
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (tid == 0) DFLASH_ATTN_STAMP(7);
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTcTmemCols);
  }
}

// Log-sum-exp merge of the chunk partials of a one-sequence pass, per q head:
// all 8 block rows, a 32-column slice of the head (blockIdx.y).  Chunk c of
// row m carries
// O_c / l_c (FP16) and (m_c, l_c); the row's output is
//   sum_c w_c O_c / l_c,   w_c = l_c 2^(m_c - mx) / sum_c' l_c' 2^(m_c' - mx).
// Lane = (row i = lane / 4, 8 columns from (lane % 4) * 8); warp w takes
// chunks w, w + 8, ...  Each thread issues the loads of up to 9 of its chunks
// (partial values and (m, l)) at once and folds them into a running
// (max, sum, sum of weighted rows); the 8 warps' results are then combined
// through shared memory in a fixed order (deterministic).
struct CombineArgs {
  const __half* part;
  const float2* ml;
  void* out;
  int out_f16;
  int out_rows, out_ku;
  int d, n_q, n_kv, gq, Q;  // Q: chunks of the pass per kv head
  // the pass's chunk plan (chunk_plan): sequence s owns chunks [start_s, start_s + c_s)
  const int32_t* anchor_pos;
  const int32_t* block_len;
  int n_seq, window, cap;
  const int* plan;  // [n_seq] start_s | c_s << 16, written by the attention kernel (n_seq > 1)
  int32_t* status;
  unsigned long long* trace;  // diagnostic builds only (DFLASH_TRACE): per-CTA timestamps
};

__global__ void __launch_bounds__(256) attn_combine_kernel(const __grid_constant__ CombineArgs a) {
  __shared__ float smx[8][32];
  __shared__ float ssum[8][32];
  __shared__ float4 sacc[8][32][2];
  const int hq = blockIdx.x, cb = blockIdx.y, s = 0;
  const int g = hq / a.gq, hl = hq - g * a.gq;
  const int M = a.gq * 8;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) DFLASH_ATTN_STAMP(0);
  // the sequence's chunks, as the attention kernel's plan gives them, formed
  // here while that kernel finishes (it depends only on the pass's inputs)
  const int tiles = seq_keys(a.anchor_pos, a.block_len, 0, a.window, a.cap).tiles;
  const int t_per = max(1, (tiles + a.Q - 1) / a.Q);
  const int n_ch = max(1, (tiles + t_per - 1) / t_per), start = 0;
  pdl_wait();
  if (threadIdx.x == 0) DFLASH_ATTN_STAMP(1);
  pdl_launch_dependents();
  const size_t base = (static_cast<size_t>(g) * a.Q + start) * M;
  const int i = lane >> 2, mrow = hl * 8 + i, col = cb * 32 + (lane & 3) * 8;
  const __half* pr = a.part + (base + mrow) * a.d + col;
  const float2* pml = a.ml + base + mrow;
  const size_t cstride = static_cast<size_t>(M) * a.d;
  float mw = -INFINITY, lw = 0.f, acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;
  constexpr int U = 9;  // 8 warps x 9 loads cover the default 65 chunks in one round
  for (int c0 = warp; c0 < n_ch; c0 += 8 * U) {
    uint4 v[U];
    float2 ml[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int c = c0 + 8 * u;
      if (c < n_ch) {
        ml[u] = __ldcg(pml + static_cast<size_t>(c) * M);
        v[u] = __ldcg(reinterpret_cast<const uint4*>(pr + c * cstride));
      } else {
        ml[u] = make_float2(-INFINITY, 0.f);
        v[u] = make_uint4(0, 0, 0, 0);
      }
    }
    float bm = mw;
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (ml[u].y > 0.f) bm = fmaxf(bm, ml[u].x);
    const float sc = mw == -INFINITY ? 0.f : ex2_approx(mw - bm);
    lw *= sc;
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] *= sc;
    mw = bm;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (ml[u].y > 0.f) {  // chunks without keys hold no partial
        const float w = ml[u].y * ex2_approx(ml[u].x - bm);
        lw += w;
        const __half2* h = reinterpret_cast<const __half2*>(&v[u]);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __half22float2(h[e]);
          acc[2 * e] = fmaf(f.x, w, acc[2 * e]);
          acc[2 * e + 1] = fmaf(f.y, w, acc[2 * e + 1]);
        }
      }
    }
  }
  smx[warp][lane] = mw;
  ssum[warp][lane] = lw;
  sacc[warp][lane][0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
  sacc[warp][lane][1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
  __syncthreads();
  if (threadIdx.x == 0) DFLASH_ATTN_STAMP(2);
  if (warp == 0) {
    float mx = -INFINITY;
#pragma unroll
    for (int w = 0; w < 8; ++w) mx = fmaxf(mx, smx[w][lane]);
    float L = 0.f, r[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) r[e] = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      const float sc = smx[w][lane] == -INFINITY ? 0.f : ex2_approx(smx[w][lane] - mx);
      L = fmaf(ssum[w][lane], sc, L);
      const float4 x = sacc[w][lane][0], y = sacc[w][lane][1];
      r[0] = fmaf(x.x, sc, r[0]);
      r[1] = fmaf(x.y, sc, r[1]);
      r[2] = fmaf(x.z, sc, r[2]);
      r[3] = fmaf(x.w, sc, r[3]);
      r[4] = fmaf(y.x, sc, r[4]);
      r[5] = fmaf(y.y, sc, r[5]);
      r[6] = fmaf(y.z, sc, r[6]);
      r[7] = fmaf(y.w, sc, r[7]);
    }
    if (!(L > 0.f)) {
      if ((lane & 3) == 0) set_status(a.status, DFLASH_DEV_NONFINITE);
      L = 1.f;
    }
    const float inv = 1.f / L;
#pragma unroll
    for (int e = 0; e < 8; ++e) r[e] *= inv;
    const int P = a.out_f16 ? 1 : 2;
    const size_t ob = xchunk_index(hq * a.d + col, s * 8 + i, 0, a.out_rows, a.out_ku, P);
    if (a.out_f16) {
      *reinterpret_cast<uint4*>(static_cast<__half*>(a.out) + ob) =
          make_uint4(pack_f16x2(r[0], r[1]), pack_f16x2(r[2], r[3]), pack_f16x2(r[4], r[5]), pack_f16x2(r[6], r[7]));
    } else {
      uint4 hi, lo;
      split_bf16x2(r[0], r[1], hi.x, lo.x);
      split_bf16x2(r[2], r[3], hi.y, lo.y);
      split_bf16x2(r[4], r[5], hi.z, lo.z);
      split_bf16x2(r[6], r[7], hi.w, lo.w);
      const size_t lo_off = static_cast<size_t>(a.out_rows) * (a.out_ku + 32);
      *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) + ob) = hi;
      *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) + ob + lo_off) = lo;
    }
    if (threadIdx.x == 0) DFLASH_ATTN_STAMP(7);
  }
}

// The same merge for a pass of several sequences, whose sequences own few
// chunks each: one thread per (sequence, q head, block row, 8 columns) folds
// all of its sequence's chunks, loading up to kMultiU of them at once; a
// warp covers one row of a head (256 columns: 32 consecutive 16-byte pieces).
constexpr int kMultiU = 8;

__global__ void __launch_bounds__(256) attn_combine_multi_kernel(const __grid_constant__ CombineArgs a) {
  const int s = blockIdx.y;
  const int t = blockIdx.x * blockDim.x + threadIdx.x;
  const int n8 = a.d / 8;
  pdl_wait();
  pdl_launch_dependents();
  if (t >= a.n_q * 8 * n8) return;
  const int c8 = t % n8, i = (t / n8) % 8, hq = t / (n8 * 8);
  const int g = hq / a.gq, hl = hq - g * a.gq;
  const int M = a.gq * 8;
  const int pl = __ldcg(a.plan + s);
  const int start = pl & 0xffff, n_ch = pl >> 16;
  const size_t base = (static_cast<size_t>(g) * a.Q + start) * M;
  const int mrow = hl * 8 + i, col = c8 * 8;
  const __half* pr = a.part + (base + mrow) * a.d + col;
  const float2* pml = a.ml + base + mrow;
  const size_t cstride = static_cast<size_t>(M) * a.d;
  float mw = -INFINITY, lw = 0.f, acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;
  for (int c0 = 0; c0 < n_ch; c0 += kMultiU) {
    uint4 v[kMultiU];
    float2 ml[kMultiU];
#pragma unroll
    for (int u = 0; u < kMultiU; ++u) {
      const int c = c0 + u;
      if (c < n_ch) {
        ml[u] = __ldcg(pml + static_cast<size_t>(c) * M);
        v[u] = __ldcg(reinterpret_cast<const uint4*>(pr + c * cstride));
      } else {
        ml[u] = make_float2(-INFINITY, 0.f);
        v[u] = make_uint4(0, 0, 0, 0);
      }
    }
    float bm = mw;
#pragma unroll
    for (int u = 0; u < kMultiU; ++u)
      if (ml[u].y > 0.f) bm = fmaxf(bm, ml[u].x);
    const float sc = mw == -INFINITY ? 0.f : ex2_approx(mw - bm);
    lw *= sc;
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] *= sc;
    mw = bm;
#pragma unroll
    for (int u = 0; u < kMultiU; ++u) {
      if (ml[u].y > 0.f) {  // chunks without keys hold no partial
        const float w = ml[u].y * ex2_approx(ml[u].x - bm);
        lw += w;
        const __half2* h = reinterpret_cast<const __half2*>(&v[u]);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __half22float2(h[e]);
          acc[2 * e] = fmaf(f.x, w, acc[2 * e]);
          acc[2 * e + 1] = fmaf(f.y, w, acc[2 * e + 1]);
        }
      }
    }
  }
  if (!(lw > 0.f)) {
    set_status(a.status, DFLASH_DEV_NONFINITE);
    lw = 1.f;
  }
  const float inv = 1.f / lw;
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] *= inv;
  const int P = a.out_f16 ? 1 : 2;
  const size_t ob = xchunk_index(hq * a.d + col, s * 8 + i, 0, a.out_rows, a.out_ku, P);
  if (a.out_f16) {
    *reinterpret_cast<uint4*>(static_cast<__half*>(a.out) + ob) =
        make_uint4(pack_f16x2(acc[0], acc[1]), pack_f16x2(acc[2], acc[3]), pack_f16x2(acc[4], acc[5]),
                   pack_f16x2(acc[6], acc[7]));
  } else {
    uint4 hi, lo;
    split_bf16x2(acc[0], acc[1], hi.x, lo.x);
    split_bf16x2(acc[2], acc[3], hi.y, lo.y);
    split_bf16x2(acc[4], acc[5], hi.z, lo.z);
    split_bf16x2(acc[6], acc[7], hi.w, lo.w);
    const size_t lo_off = static_cast<size_t>(a.out_rows) * (a.out_ku + 32);
    *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) + ob) = hi;
    *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(a.out) + ob + lo_off) = lo;
  }
}

static cudaError_t launch_attn_impl(int D, const AttnArgs& a, dim3 grid, cudaStream_t st, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kTcThreads);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.stream = st;
  switch (D) {
#define DFLASH_ATTN_CASE(DD)                                                                                  \
  case DD: {                                                                                                  \
    cfg.dynamicSmemBytes = TcGeom<DD>::smem(a.gq * 8);                                                        \
    cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<DD>, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448); \
    if (e != cudaSuccess) return e;                                                                           \
    return cudaLaunchKernelEx(&cfg, attn_tc_kernel<DD>, a);                                                   \
  }
    DFLASH_ATTN_CASE(64)
    DFLASH_ATTN_CASE(128)
    DFLASH_ATTN_CASE(256)
#undef DFLASH_ATTN_CASE
  }
  return cudaErrorInvalidValue;
}

int attn_smem_bytes(int D, int M) {
  switch (D) {
    case 64: return TcGeom<64>::smem(M);
    case 128: return TcGeom<128>::smem(M);
    case 256: return TcGeom<256>::smem(M);
  }
  return 0;
}

// One layer's attention for slots [0, n_seq): chunked kernel plus, when the
// context is split, the merge.
// Chunks of a pass per kv head: C per sequence; a pass of several sequences
// on the default C takes at least one wave of CTAs (one per SM), shared out
// by context length (chunk_plan), within the partial buffers' n_slots * C_max.
int attn_pass_chunks(const Model& m, const State& st, int n_seq) {
  const int base = n_seq * st.attn_chunks;
  if (n_seq == 1 || st.attn_chunks_set) return base;
  int wave = m.sm_count / m.cfg.n_kv_heads;
  const int cap = st.n_slots * st.attn_chunks_max;
  if (wave > cap) wave = cap;
  return wave > base ? wave : base;
}

cudaError_t launch_attention(const Model& m, State& st, int layer, int n_seq, int pass_nt, const int32_t* anchor_pos,
                             const int32_t* block_len, int32_t* status, cudaStream_t stream) {
  const dflash_config& c = m.cfg;
  AttnArgs a;
  a.kmap = st.k_map;
  a.vmap = st.v_map;
  a.anchor_pos = anchor_pos;
  a.block_len = block_len;
  a.pmap = st.part_map;
  a.ml = st.attn_ml;
  a.out = st.attn_out;
  a.out_f16 = m.wtype != DFLASH_WT_BF16;
  a.out_rows = 8 * pass_nt;
  a.out_ku = m.wtype == DFLASH_WT_BF16 ? 128 : 256;
  a.layer = layer;
  a.n_slots = st.n_slots;
  a.n_kv = c.n_kv_heads;
  a.n_q = c.n_q_heads;
  a.gq = c.n_q_heads / c.n_kv_heads;
  a.cap = st.capacity;
  a.window = c.attn_window;
  a.Q = attn_pass_chunks(m, st, n_seq);
  a.n_seq = n_seq;
  a.status = status;
  a.qmap = st.q_map;
  a.trace = a.Q * a.n_kv <= st.max_grid ? trace_slot(st) : nullptr;
  a.kbase_ptr = st.K;
  a.vbase_ptr = st.V;
  a.plan = n_seq > 1 ? st.attn_plan : nullptr;
  cudaError_t e = launch_attn_impl(c.head_dim, a, dim3(a.Q, a.n_kv, 1), stream, true);
  if (e != cudaSuccess || a.Q == n_seq) return e;
  if (st.prof_n > 0 && st.prof_k < st.prof_n)
    cudaEventRecordWithFlags(static_cast<cudaEvent_t>(st.prof_events[st.prof_k++]), stream, cudaEventRecordExternal);
  CombineArgs cb;
  cb.part = st.attn_part;
  cb.ml = st.attn_ml;
  cb.out = st.attn_out;
  cb.out_f16 = a.out_f16;
  cb.out_rows = a.out_rows;
  cb.out_ku = a.out_ku;
  cb.d = c.head_dim;
  cb.n_q = c.n_q_heads;
  cb.n_kv = c.n_kv_heads;
  cb.gq = a.gq;
  cb.Q = a.Q;
  cb.anchor_pos = anchor_pos;
  cb.block_len = block_len;
  cb.n_seq = n_seq;
  cb.window = a.window;
  cb.cap = a.cap;
  cb.plan = st.attn_plan;
  cb.status = status;
  // (diagnostic builds: a grid larger than a trace slot records nothing)
  cb.trace = n_seq == 1 && c.n_q_heads * (c.head_dim / 32) <= st.max_grid ? trace_slot(st) : nullptr;
  cudaLaunchConfig_t cfg = {};
  // one sequence: many chunks, spread over the warps of a CTA per (head, 32
  // columns); several: a thread per (sequence, head, row, 8 columns)
  const int per_seq = c.n_q_heads * 8 * (c.head_dim / 8);
  cfg.gridDim = n_seq == 1 ? dim3(c.n_q_heads, c.head_dim / 32, 1) : dim3((per_seq + 255) / 256, n_seq, 1);
  cfg.blockDim = dim3(256);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.stream = stream;
  return n_seq == 1 ? cudaLaunchKernelEx(&cfg, attn_combine_kernel, cb)
                    : cudaLaunchKernelEx(&cfg, attn_combine_multi_kernel, cb);
}

}  // namespace dflash

// Non-causal GQA block attention of the draft pass ("#1426 dflash:
// experimental standalone DeepSpec DFlash block drafter", sections "Target
// feature taps" -- non-causal block attention, scale 1/16 -- and "Drafter
// runtime" -- GQA 24 Q / 2 KV, head dim 256).
//
// For one slot and one kv head the queries are the GQ = n_q / n_kv q heads
// of the block's 8 rows: M = 8 * GQ rows (96 for DFlash) sharing every key.
// The keys are the slot's position-addressed cells [0, p + B): the fused
// context plus the block's own rows, which the QKV epilogue wrote at
// [p, p + B).  The context is split into C chunks (split-K / flash-decode):
// CTA (chunk, kv head, slot) streams its 64-key K and V tiles through a
// 2-stage ring with 2-D TMA copies (64 x 64 boxes, 128-byte swizzle) issued
// by a producer warp, and each consumer warp owns 16 query rows:
//   S = Q K^T (mma.sync m16n8k16, fp16 in, fp32 out) -> online softmax in
//   base 2 -> O += P V.
// With C > 1 every chunk writes (O unnormalised, running max, sum) and
// attn_combine_kernel merges them with the log-sum-exp rule; with C == 1 the
// CTA normalises and writes the output directly.
#include "kernels.h"
#include "layout.cuh"

namespace dflash {

struct AttnArgs {
  CUtensorMap qmap;  // queries [slots * n_kv * M, d] fp16, 64 x M boxes (normed, rotated, scaled by 1/sqrt(d))
  CUtensorMap kmap;  // K arena as [rows, d] fp16
  CUtensorMap vmap;
  const int32_t* anchor_pos;
  const int32_t* block_len;
  float* part;            // [slots, n_kv, C, M, d]
  float2* ml;             // [slots, n_kv, C, M]
  void* out;              // attention output in the o-projection's chunked X layout (C == 1)
  int out_f16;            // 1: one FP16 plane; 0: BF16 hi and lo planes
  int out_rows, out_ku;   // chunked layout: rows R of the pass and inputs per unit
  int layer, n_slots, n_kv, n_q, gq, cap, C, n_seq;
  int32_t* status;
};

constexpr int kAttnKT = 64;      // keys per tile
constexpr int kAttnStages = 2;

template <int D>
struct AttnGeom {
  static constexpr int BOXES = D / 64;
  static constexpr int TILE_BYTES = kAttnKT * D * 2;  // one K (or V) tile
  static __host__ __device__ constexpr int q_bytes(int M) { return M * D * 2; }
  static __host__ __device__ constexpr int smem(int M) {
    return 1024 + q_bytes(M) + 2 * kAttnStages * TILE_BYTES + 4 * kAttnStages * 8 + 64 + 8;
  }
};

// Address of element-chunk (row, 16-byte chunk q within the 64-wide box)
// inside a run of 64-column boxes of `rows` rows with the 128-byte swizzle.
__device__ __forceinline__ uint32_t swz(uint32_t base, int rows, int row, int col8) {
  const int box = col8 >> 3, q = col8 & 7;
  return base + box * rows * 128 + row * 128 + ((q ^ (row & 7)) << 4);
}

template <int D>
__global__ void __launch_bounds__(256, 1) attn_kernel(const __grid_constant__ AttnArgs a) {
  using Geo = AttnGeom<D>;
  const int M = a.gq * 8;
  const int NW = M / 16;  // consumer warps
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sq = smem;
  uint8_t* sk = sq + ((Geo::q_bytes(M) + 1023) / 1024) * 1024;
  uint8_t* sv = sk + kAttnStages * Geo::TILE_BYTES;
  uint64_t* kfull = reinterpret_cast<uint64_t*>(sv + kAttnStages * Geo::TILE_BYTES);
  uint64_t* vfull = kfull + kAttnStages;
  uint64_t* empty = vfull + kAttnStages;
  uint64_t* qbar = empty + kAttnStages;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x, g = blockIdx.y, s = blockIdx.z;

  // key range of this chunk
  const int p = a.anchor_pos[s];
  int B = a.block_len[s];
  B = B < DFLASH_MIN_BLOCK ? DFLASH_MIN_BLOCK : (B > DFLASH_MAX_BLOCK ? DFLASH_MAX_BLOCK : B);
  int T = p + B;
  T = T < 0 ? 0 : (T > a.cap ? a.cap : T);
  const int ntiles = (T + kAttnKT - 1) / kAttnKT;
  const int tpc = (ntiles + a.C - 1) / a.C;
  const int t0 = c * tpc;
  const int t1 = min(ntiles, t0 + tpc);
  const int nt = t1 > t0 ? t1 - t0 : 0;
  const int row0 = ((a.layer * a.n_slots + s) * a.n_kv + g) * a.cap;

  if (tid == 0) {
    for (int i = 0; i < kAttnStages; ++i) {
      mbar_init(&kfull[i], 1);
      mbar_init(&vfull[i], 1);
      mbar_init(&empty[i], NW);
    }
    mbar_init(qbar, 1);
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == NW) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&a.qmap);
      prefetch_tensormap(&a.kmap);
      prefetch_tensormap(&a.vmap);
      auto issue = [&](int it) {
        const int st = it % kAttnStages;
        const int y = row0 + (t0 + it) * kAttnKT;
        mbar_arrive_expect_tx(&kfull[st], Geo::TILE_BYTES);
        for (int b = 0; b < Geo::BOXES; ++b)
          tma_load_2d(sk + st * Geo::TILE_BYTES + b * kAttnKT * 128, &a.kmap, b * 64, y, &kfull[st]);
        mbar_arrive_expect_tx(&vfull[st], Geo::TILE_BYTES);
        for (int b = 0; b < Geo::BOXES; ++b)
          tma_load_2d(sv + st * Geo::TILE_BYTES + b * kAttnKT * 128, &a.vmap, b * 64, y, &vfull[st]);
      };
      // Tiles wholly inside the fused context [0, p) do not depend on the
      // previous kernel (which writes the block cells) and may start early.
      int it = 0;
      const int n_pre = nt < kAttnStages ? nt : kAttnStages;
      for (; it < n_pre && (t0 + it + 1) * kAttnKT <= p; ++it) issue(it);
      pdl_wait();
      // the queries (written by the previous kernel): one 64-column box each
      mbar_arrive_expect_tx(qbar, Geo::q_bytes(M));
      for (int b = 0; b < Geo::BOXES; ++b)
        tma_load_2d(sq + b * M * 128, &a.qmap, b * 64, (s * a.n_kv + g) * M, qbar);
      int issued = it;
      for (; it < nt; ++it) {
        if (it >= kAttnStages && !mbar_wait(&empty[it % kAttnStages], ((it / kAttnStages) - 1) & 1)) {
          set_status(a.status, DFLASH_DEV_TIMEOUT);
          break;
        }
        issue(it);
        issued = it + 1;
      }
      for (int j = (issued > kAttnStages ? issued - kAttnStages : 0); j < issued; ++j) {
        if (!mbar_wait(&kfull[j % kAttnStages], (j / kAttnStages) & 1) ||
            !mbar_wait(&vfull[j % kAttnStages], (j / kAttnStages) & 1)) {
          set_status(a.status, DFLASH_DEV_TIMEOUT);
          break;
        }
      }
    }
    return;
  }
  if (warp > NW) return;

  // -------------------------------------------------------------- consumers
  pdl_wait();
  pdl_launch_dependents();
  if (!mbar_wait(qbar, 0)) set_status(a.status, DFLASH_DEV_TIMEOUT);

  constexpr float LOG2E = 1.4426950408889634f;
  constexpr int NDT = D / 8;  // output n-tiles
  float o[NDT][4];
#pragma unroll
  for (int i = 0; i < NDT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m_r = -INFINITY, m_r8 = -INFINITY, l_r = 0.f, l_r8 = 0.f;

  const uint32_t qb = smem_u32(sq);
  const int wr0 = warp * 16;
  // ldmatrix row/col selectors
  const int a_row = wr0 + (lane & 7) + ((lane >> 3) & 1) * 8;
  const int a_c8 = lane >> 4;
  const int b_key = (lane & 7) + (lane >> 4) * 8;
  const int b_c8 = (lane >> 3) & 1;
  const int v_key = (lane & 7) + ((lane >> 3) & 1) * 8;
  const int v_c8 = lane >> 4;

  bool ok = true;
  for (int it = 0; it < nt && ok; ++it) {
    const int st = it % kAttnStages;
    const uint32_t par = (it / kAttnStages) & 1;
    if (!mbar_wait(&kfull[st], par)) {
      set_status(a.status, DFLASH_DEV_TIMEOUT);
      ok = false;
      break;
    }
    const uint32_t kb = smem_u32(sk + st * Geo::TILE_BYTES);
    const uint32_t vb = smem_u32(sv + st * Geo::TILE_BYTES);
    float sacc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) sacc[i][0] = sacc[i][1] = sacc[i][2] = sacc[i][3] = 0.f;
#pragma unroll 4
    for (int kk = 0; kk < D / 16; ++kk) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4(a0, a1, a2, a3, swz(qb, M, a_row, kk * 2 + a_c8));
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4(b0, b1, b2, b3, swz(kb, kAttnKT, np * 16 + b_key, kk * 2 + b_c8));
        mma_f16_16816(sacc[2 * np], a0, a1, a2, a3, b0, b1);
        mma_f16_16816(sacc[2 * np + 1], a0, a1, a2, a3, b2, b3);
      }
    }
    // mask keys beyond T, scale to base 2, online softmax
    const int kbase = (t0 + it) * kAttnKT + (lane & 3) * 2;
    float mx = -INFINITY, mx8 = -INFINITY;
#pragma unroll
    for (int n = 0; n < 8; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int key = kbase + n * 8 + (e & 1);
        const float v = key < T ? sacc[n][e] * LOG2E : -INFINITY;
        sacc[n][e] = v;
        if (e < 2) mx = fmaxf(mx, v); else mx8 = fmaxf(mx8, v);
      }
#pragma unroll
    for (int off = 1; off <= 2; off <<= 1) {
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      mx8 = fmaxf(mx8, __shfl_xor_sync(0xffffffffu, mx8, off));
    }
    const float mn = fmaxf(m_r, mx), mn8 = fmaxf(m_r8, mx8);
    const float base = mn == -INFINITY ? 0.f : mn;
    const float base8 = mn8 == -INFINITY ? 0.f : mn8;
    const float corr = exp2f(m_r - base), corr8 = exp2f(m_r8 - base8);
    m_r = mn;
    m_r8 = mn8;
    float ls = 0.f, ls8 = 0.f;
    uint32_t pa[4][4];  // P as A fragments, 4 k-steps of 16 keys
#pragma unroll
    for (int n = 0; n < 8; ++n) {
      const float p0 = exp2f(sacc[n][0] - base), p1 = exp2f(sacc[n][1] - base);
      const float p2 = exp2f(sacc[n][2] - base8), p3 = exp2f(sacc[n][3] - base8);
      ls += p0 + p1;
      ls8 += p2 + p3;
      const int ks = n >> 1, hi = n & 1;
      pa[ks][hi * 2 + 0] = pack_f16x2(p0, p1);
      pa[ks][hi * 2 + 1] = pack_f16x2(p2, p3);
    }
    l_r = l_r * corr + ls;
    l_r8 = l_r8 * corr8 + ls8;
#pragma unroll
    for (int i = 0; i < NDT; ++i) {
      o[i][0] *= corr; o[i][1] *= corr;
      o[i][2] *= corr8; o[i][3] *= corr8;
    }
    if (!mbar_wait(&vfull[st], par)) {
      set_status(a.status, DFLASH_DEV_TIMEOUT);
      ok = false;
      break;
    }
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
#pragma unroll
      for (int dp = 0; dp < D / 16; ++dp) {
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(b0, b1, b2, b3, swz(vb, kAttnKT, ks * 16 + v_key, dp * 2 + v_c8));
        mma_f16_16816(o[2 * dp], pa[ks][0], pa[ks][1], pa[ks][2], pa[ks][3], b0, b1);
        mma_f16_16816(o[2 * dp + 1], pa[ks][0], pa[ks][1], pa[ks][2], pa[ks][3], b2, b3);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
  }

  // row sums across the quad
#pragma unroll
  for (int off = 1; off <= 2; off <<= 1) {
    l_r += __shfl_xor_sync(0xffffffffu, l_r, off);
    l_r8 += __shfl_xor_sync(0xffffffffu, l_r8, off);
  }
  const int m0 = wr0 + (lane >> 2), m1 = m0 + 8;
  if (a.C == 1) {
    const float inv = l_r > 0.f ? 1.f / l_r : 0.f, inv8 = l_r8 > 0.f ? 1.f / l_r8 : 0.f;
    if (!(l_r > 0.f) || !(l_r8 > 0.f)) set_status(a.status, DFLASH_DEV_NONFINITE);
    const int P = a.out_f16 ? 1 : 2;
    const int row0 = s * 8 + (m0 & 7), row1 = s * 8 + (m1 & 7);
    const int c0 = (g * a.gq + (m0 >> 3)) * D, c1 = (g * a.gq + (m1 >> 3)) * D;
#pragma unroll
    for (int i = 0; i < NDT; ++i) {
      const int col = i * 8 + (lane & 3) * 2;
      const size_t o0 = xchunk_index(c0 + col, row0, 0, a.out_rows, a.out_ku, P);
      const size_t o1 = xchunk_index(c1 + col, row1, 0, a.out_rows, a.out_ku, P);
      if (a.out_f16) {
        *reinterpret_cast<uint32_t*>(static_cast<__half*>(a.out) + o0) = pack_f16x2(o[i][0] * inv, o[i][1] * inv);
        *reinterpret_cast<uint32_t*>(static_cast<__half*>(a.out) + o1) = pack_f16x2(o[i][2] * inv8, o[i][3] * inv8);
      } else {
        uint32_t h0, l0, h1, l1;
        split_bf16x2(o[i][0] * inv, o[i][1] * inv, h0, l0);
        split_bf16x2(o[i][2] * inv8, o[i][3] * inv8, h1, l1);
        __nv_bfloat16* ob = static_cast<__nv_bfloat16*>(a.out);
        const size_t lo_off = static_cast<size_t>(a.out_rows) * (a.out_ku + 32);  // next plane of the chunk
        *reinterpret_cast<uint32_t*>(ob + o0) = h0;
        *reinterpret_cast<uint32_t*>(ob + o1) = h1;
        *reinterpret_cast<uint32_t*>(ob + o0 + lo_off) = l0;
        *reinterpret_cast<uint32_t*>(ob + o1 + lo_off) = l1;
      }
    }
  } else {
    const size_t pbase = ((static_cast<size_t>(s) * a.n_kv + g) * a.C + c) * M;
#pragma unroll
    for (int i = 0; i < NDT; ++i) {
      const int col = i * 8 + (lane & 3) * 2;
      __stcg(reinterpret_cast<float2*>(a.part + (pbase + m0) * D + col), make_float2(o[i][0], o[i][1]));
      __stcg(reinterpret_cast<float2*>(a.part + (pbase + m1) * D + col), make_float2(o[i][2], o[i][3]));
    }
    if ((lane & 3) == 0) {
      __stcg(a.ml + pbase + m0, make_float2(m_r, l_r));
      __stcg(a.ml + pbase + m1, make_float2(m_r8, l_r8));
    }
  }
}

// Log-sum-exp merge of the C chunk partials of one (slot, q head): all 8 block
// rows, a 64-column slice of the head (blockIdx.y).  The per-row merge weights
// 2^(m_c - M) / L are computed once into shared memory; then 8 groups of 32
// threads each sum every 8th chunk for 2 columns x 8 rows with independent
// loads, and the groups are reduced through shared memory.
struct CombineArgs {
  const float* part;
  const float2* ml;
  void* out;
  int out_f16;
  int out_rows, out_ku;
  int d, n_q, n_kv, gq, C;
  int32_t* status;
};

constexpr int kCombineMaxC = 512;

__global__ void __launch_bounds__(256) attn_combine_kernel(const __grid_constant__ CombineArgs a) {
  __shared__ float sw[8][kCombineMaxC];
  __shared__ float2 sacc[8][8][32];  // [chunk group][row][lane] partial sums of 2 columns
  const int hq = blockIdx.x, cb = blockIdx.y, s = blockIdx.z;
  const int g = hq / a.gq, hl = hq - g * a.gq;
  const int M = a.gq * 8;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_wait();
  pdl_launch_dependents();
  const size_t base = (static_cast<size_t>(s) * a.n_kv + g) * a.C * M;
  {
    // warp i: merge weights of block row i
    const int m = hl * 8 + warp;
    float mx = -INFINITY;
    for (int c = lane; c < a.C; c += 32) {
      const float2 v = __ldcg(a.ml + base + static_cast<size_t>(c) * M + m);
      if (v.y > 0.f) mx = fmaxf(mx, v.x);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float L = 0.f;
    for (int c = lane; c < a.C; c += 32) {
      const float2 v = __ldcg(a.ml + base + static_cast<size_t>(c) * M + m);
      const float e = v.y > 0.f ? exp2f(v.x - mx) : 0.f;
      sw[warp][c] = e;
      L += v.y * e;
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    if (!(L > 0.f)) {
      if (lane == 0) set_status(a.status, DFLASH_DEV_NONFINITE);
      L = 1.f;
    }
    const float inv = 1.f / L;
    __syncwarp();
    for (int c = lane; c < a.C; c += 32) sw[warp][c] *= inv;
  }
  __syncthreads();
  // chunk group = warp; columns cb*64 + 2*lane, +1
  const int col = cb * 64 + lane * 2;
  float2 acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = make_float2(0.f, 0.f);
#pragma unroll 4
  for (int c = warp; c < a.C; c += 8) {
    const float* pc = a.part + (base + static_cast<size_t>(c) * M + hl * 8) * a.d + col;
    float2 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __ldcg(reinterpret_cast<const float2*>(pc + static_cast<size_t>(i) * a.d));
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float wgt = sw[i][c];
      acc[i].x = fmaf(v[i].x, wgt, acc[i].x);
      acc[i].y = fmaf(v[i].y, wgt, acc[i].y);
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) sacc[warp][i][lane] = acc[i];
  __syncthreads();
  // warp i writes row i
  {
    const int i = warp;
    float2 r = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      r.x += sacc[k][i][lane].x;
      r.y += sacc[k][i][lane].y;
    }
    const int P = a.out_f16 ? 1 : 2;
    const size_t ob = xchunk_index(hq * a.d + col, s * 8 + i, 0, a.out_rows, a.out_ku, P);
    if (a.out_f16) {
      *reinterpret_cast<uint32_t*>(static_cast<__half*>(a.out) + ob) = pack_f16x2(r.x, r.y);
    } else {
      uint32_t hi, lo;
      split_bf16x2(r.x, r.y, hi, lo);
      const size_t lo_off = static_cast<size_t>(a.out_rows) * (a.out_ku + 32);
      *reinterpret_cast<uint32_t*>(static_cast<__nv_bfloat16*>(a.out) + ob) = hi;
      *reinterpret_cast<uint32_t*>(static_cast<__nv_bfloat16*>(a.out) + ob + lo_off) = lo;
    }
  }
}

static cudaError_t launch_attn_impl(int D, const AttnArgs& a, dim3 grid, cudaStream_t st, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  const int M = a.gq * 8;
  cfg.blockDim = dim3((M / 16 + 1) * 32);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.stream = st;
  switch (D) {
    case 64: {
      cfg.dynamicSmemBytes = AttnGeom<64>::smem(M);
      cudaError_t e = cudaFuncSetAttribute(attn_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
      if (e != cudaSuccess) return e;
      return cudaLaunchKernelEx(&cfg, attn_kernel<64>, a);
    }
    case 128: {
      cfg.dynamicSmemBytes = AttnGeom<128>::smem(M);
      cudaError_t e = cudaFuncSetAttribute(attn_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
      if (e != cudaSuccess) return e;
      return cudaLaunchKernelEx(&cfg, attn_kernel<128>, a);
    }
    case 256: {
      cfg.dynamicSmemBytes = AttnGeom<256>::smem(M);
      cudaError_t e = cudaFuncSetAttribute(attn_kernel<256>, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
      if (e != cudaSuccess) return e;
      return cudaLaunchKernelEx(&cfg, attn_kernel<256>, a);
    }
  }
  return cudaErrorInvalidValue;
}

int attn_smem_bytes(int D, int gq) {
  const int M = gq * 8;
  switch (D) {
    case 64: return AttnGeom<64>::smem(M);
    case 128: return AttnGeom<128>::smem(M);
    case 256: return AttnGeom<256>::smem(M);
  }
  return 0;
}

// One layer's attention for slots [0, n_seq): chunked kernel plus, when the
// context is split, the merge.
cudaError_t launch_attention(const Model& m, State& st, int layer, int n_seq, int pass_nt, const int32_t* anchor_pos,
                             const int32_t* block_len, int32_t* status, cudaStream_t stream) {
  const dflash_config& c = m.cfg;
  AttnArgs a;
  a.kmap = st.k_map;
  a.vmap = st.v_map;
  a.anchor_pos = anchor_pos;
  a.block_len = block_len;
  a.part = st.attn_part;
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
  a.C = st.attn_chunks;
  a.n_seq = n_seq;
  a.status = status;
  a.qmap = st.q_map;
  cudaError_t e = launch_attn_impl(c.head_dim, a, dim3(a.C, a.n_kv, n_seq), stream, true);
  if (e != cudaSuccess || a.C == 1) return e;
  if (st.prof_n > 0 && st.prof_k < st.prof_n)
    cudaEventRecord(static_cast<cudaEvent_t>(st.prof_events[st.prof_k++]), stream);
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
  cb.C = a.C;
  cb.status = status;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(c.n_q_heads, c.head_dim / 64, n_seq);
  cfg.blockDim = dim3(256);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, attn_combine_kernel, cb);
}

}  // namespace dflash

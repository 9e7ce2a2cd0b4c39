// Host-side launchers of the GEMV kernel family.  The templates are defined
// here and explicitly instantiated once per weight type in gemv_<type>.cu, so
// the heavy kernel instantiations compile in parallel translation units.
#pragma once

#include "gemv_epilogues.cuh"

namespace dflash {

struct LaunchCfg {
  cudaStream_t stream;
  int grid;
  bool pdl;
  int cluster = 1;  // CTAs per cluster (GemvArgs::cl_parts * cl_gph; 1: no clusters)
};

struct ArgmaxParams {
  int vocab, n_seq, H;
  const int32_t* block_len;
  int32_t* drafts;
  unsigned long long* slots;
  float2* ms;      // [grid, R] per-CTA (max logit, sum of exp) for the draft probabilities
  float* probs;    // [n_seq, 7] out, or null
  float min_p;     // confidence floor (0: every draft offered)
  int* grid_cnt;
  float* final_hidden;
  const float* x;
  const float* norm_w;
  int32_t* status;
};

constexpr int kMaxDynSmem = 232448;  // 227 KB, the sm_100 per-CTA limit

template <int WT, int NT, int XMODE>
inline int gemv_smem(int K) {
  return GemvGeom<WT, NT, XMODE>::smem_bytes(K);
}

// Raise the dynamic shared-memory cap once per (kernel instantiation, device)
// to what the per-CTA limit leaves beside the kernel's static shared memory;
// returns that cap in *cap.
template <int WT, int NT, int XMODE, class Epi>
inline cudaError_t ensure_smem_attr(int* cap) {
  static unsigned set_mask = 0;
  static int dyn_cap = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned bit = 1u << (dev & 31);
  if (__atomic_load_n(&set_mask, __ATOMIC_ACQUIRE) & bit) {
    *cap = __atomic_load_n(&dyn_cap, __ATOMIC_ACQUIRE);
    return cudaSuccess;
  }
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, gemv_kernel<WT, NT, XMODE, Epi>);
  if (e != cudaSuccess) return e;
  const int c = kMaxDynSmem - static_cast<int>(fa.sharedSizeBytes);
  e = cudaFuncSetAttribute(gemv_kernel<WT, NT, XMODE, Epi>, cudaFuncAttributeMaxDynamicSharedMemorySize, c);
  if (e != cudaSuccess) return e;
  __atomic_store_n(&dyn_cap, c, __ATOMIC_RELEASE);
  __atomic_fetch_or(&set_mask, bit, __ATOMIC_RELEASE);
  *cap = c;
  return cudaSuccess;
}

template <int WT, int NT, int XMODE, class Epi>
inline cudaError_t launch_gemv(const GemvArgs& a, const Epi& epi, const LaunchCfg& lc) {
  auto kern = gemv_kernel<WT, NT, XMODE, Epi>;
  int cap = 0;
  cudaError_t e = ensure_smem_attr<WT, NT, XMODE, Epi>(&cap);
  if (e != cudaSuccess) return e;
  const int smem = GemvGeom<WT, NT, XMODE>::smem_bytes(a.K);
  if (smem > cap) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(lc.grid);
  cfg.blockDim = dim3(GemvGeom<WT, NT, XMODE>::THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = lc.stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = lc.pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (lc.cluster > 1) {
    if (!GemvGeom<WT, NT, XMODE>::kClusterable || !Epi::kCluster || lc.grid % lc.cluster ||
        a.cl_parts * a.cl_gph != lc.cluster)
      return cudaErrorInvalidValue;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = static_cast<unsigned>(lc.cluster);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  } else if (a.cl_parts * a.cl_gph > 1) {
    return cudaErrorInvalidValue;
  }
  return cudaLaunchKernelEx(&cfg, kern, a, epi);
}

#define DFLASH_NT_SWITCH(nt, ...)                 \
  switch (nt) {                                   \
    case 1: { constexpr int NT = 1; __VA_ARGS__ } \
    case 2: { constexpr int NT = 2; __VA_ARGS__ } \
    case 4: { constexpr int NT = 4; __VA_ARGS__ } \
    case 8: { constexpr int NT = 8; __VA_ARGS__ } \
    case 16: { constexpr int NT = 16; __VA_ARGS__ } \
    default: return cudaErrorInvalidValue;        \
  }

// X (the caller's BF16 taps) streamed, raw fp32 result stored (fusion fc).
template <int WT>
cudaError_t gemv_store(int nt, const GemvArgs& a, const EpiStore& e, const LaunchCfg& lc) {
  switch (nt) {
    case 1: return launch_gemv<WT, 1, X_STREAM_BF16>(a, e, lc);
    case 16: return launch_gemv<WT, 16, X_STREAM_BF16>(a, e, lc);
    default: return cudaErrorInvalidValue;
  }
}

// X streamed, residual add (attention output projection, MLP down).
template <int WT>
cudaError_t gemv_resid(int nt, const GemvArgs& a, const EpiResid& e, const LaunchCfg& lc) {
  DFLASH_NT_SWITCH(nt, return launch_gemv<WT, NT, X_STREAM>(a, e, lc);)
}

// The RMSNorm-fed GEMVs (q/k/v, gate/up, LM head, fusion K/V) of an 8-row
// pass stream x * w in two BF16 planes written by the kernel that produced x,
// and scale their outputs by 1 / RMS (X_NORM); larger passes stream the
// output of a separate RMSNorm kernel.
inline bool fused_norm(int nt) { return nt == 1; }

// SwiGLU gate/up.
template <int WT>
cudaError_t gemv_swiglu(int nt, const GemvArgs& a, void* h, const LaunchCfg& lc) {
  // h is written in the format the down projection streams (FP16 for quantised weights)
  const EpiSwiglu<Fmt<WT>::kF16> e{h};
  if (fused_norm(nt)) return launch_gemv<WT, 1, X_NORM>(a, e, lc);
  DFLASH_NT_SWITCH(nt, return launch_gemv<WT, NT, X_STREAM>(a, e, lc);)
}

// Per-head epilogue (draft QKV / fusion K/V).
template <int WT>
cudaError_t gemv_heads(int nt, const GemvArgs& a, const EpiHeads& e, const LaunchCfg& lc) {
  if (fused_norm(nt)) return launch_gemv<WT, 1, X_NORM>(a, e, lc);
  if (e.mode == 1) {
    switch (nt) {
      case 1: return launch_gemv<WT, 1, X_STREAM>(a, e, lc);
      case 16: return launch_gemv<WT, 16, X_STREAM>(a, e, lc);
      default: return cudaErrorInvalidValue;
    }
  }
  DFLASH_NT_SWITCH(nt, return launch_gemv<WT, NT, X_STREAM>(a, e, lc);)
}

// Epilogue of the tcgen05 GEMM of 128-row passes (gemv_tc.cu): applied per
// finished 64-row group by the thread of each activation row.
struct TcEpi {
  enum { STORE = 0, RESID = 1, SWIGLU = 2, HEADS = 3 };
  int mode;
  float* out;     // STORE: out[n][m]; RESID: x[n][m] += (fp32, row stride ldo)
  int ldo;
  void* h;        // SWIGLU: the down projection's chunked input (128 rows, h_ku inputs per unit)
  int h_ku;
  int h_f16;      // one FP16 plane, else BF16 hi and lo planes
  EpiHeads heads; // HEADS: raw q/k/v into heads.raw (launch_heads_rows finishes them)
  int parts;      // > 1: the grid is groups x parts slices of each group's inputs
                  // (partial sums in GemvArgs::partials, arrivals in GemvArgs::counters)
  __device__ void apply(int g, int n, const float (&v)[64]) const;
  // The same for the 32 rows q * 32 .. q * 32 + 31 of one warp, row q * 32 +
  // lane's values in this lane, staged in S ([32][kStageLd] floats of shared
  // memory) so that the warp's global accesses cover whole row segments.
  static constexpr int kStageLd = 68;
  __device__ void apply_staged(int g, int q, int lane, const float (&v)[64], float* S) const;
};

// The 128-row GEMM on tcgen05: a.xmap maps the chunked activations as
// [K / KU * planes * 128 rows, KU + 32] 16-bit, 64 x 128 boxes, 128-byte
// swizzle; grid <= the group count (every CTA owns whole 64-row groups).
// With slices (e.parts > 1), slice p of group g is CTA p * groups + g.
cudaError_t launch_gemv_tc(int wt, const GemvArgs& a, const TcEpi& e, int grid, cudaStream_t stream);
// The per-head epilogue of a 128-row pass's raw q/k/v (mode 0), one CTA per (head, sequence).
cudaError_t launch_heads_rows(const EpiHeads& e, int n_heads, int n_seq, cudaStream_t stream);

// LM head + argmax over the borrowed row-major BF16 head.
inline cudaError_t gemv_argmax_impl(int nt, const GemvArgs& a, const ArgmaxParams& p, const LaunchCfg& lc) {
  DFLASH_NT_SWITCH(
      nt, EpiArgmax<NT> e{p.vocab, p.n_seq, p.block_len, p.drafts, p.slots, p.ms, p.probs, p.min_p, p.grid_cnt,
                          p.final_hidden, p.x,
                          p.norm_w, p.H, p.status};
      if constexpr (NT == 1) {
        if (fused_norm(nt)) return launch_gemv<WT_HEAD, NT, X_NORM>(a, e, lc);
      } return launch_gemv<WT_HEAD, NT, X_STREAM>(a, e, lc);)
}

}  // namespace dflash

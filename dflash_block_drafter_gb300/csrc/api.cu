// C ABI of libdflash (include/dflash.h): argument validation, model and state
// creation (weight repacking, tensor maps, workspace) and the launch sequence
// of each step of the DFlash block-draft pass.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>

#include "gemv_launch.cuh"
#include "kernels.h"

namespace dflash {
// GEMV launchers, instantiated in gemv_<type>.cu
#define DFLASH_DECLARE_GEMV(WT)                                                                           \
  extern template cudaError_t gemv_store<WT>(int, const GemvArgs&, const EpiStore&, const LaunchCfg&);  \
  extern template cudaError_t gemv_resid<WT>(int, const GemvArgs&, const EpiResid&, const LaunchCfg&);  \
  extern template cudaError_t gemv_swiglu<WT>(int, const GemvArgs&, void*, const LaunchCfg&);             \
  extern template cudaError_t gemv_heads<WT>(int, const GemvArgs&, const EpiHeads&, const LaunchCfg&);
DFLASH_DECLARE_GEMV(WT_BF16)
DFLASH_DECLARE_GEMV(WT_Q8_0)
DFLASH_DECLARE_GEMV(WT_Q5_0)
DFLASH_DECLARE_GEMV(WT_Q4_0)
cudaError_t gemv_argmax(int nt, const GemvArgs& a, const ArgmaxParams& p, const LaunchCfg& lc);

// Diagnostic builds: the next per-CTA timestamp slot of a launch.
unsigned long long* trace_slot(State& st) {
#ifdef DFLASH_TRACE
  if (st.trace && st.trace_k < st.trace_launches)
    return st.trace + static_cast<size_t>(st.trace_k++) * st.max_grid * kTraceSlots;
#endif
  (void)st;
  return nullptr;
}
}  // namespace dflash

using namespace dflash;


namespace {

thread_local char g_cuda_err[256] = "";

int cuda_fail(cudaError_t e, const char* what) {
  std::snprintf(g_cuda_err, sizeof(g_cuda_err), "%s: %s", what, cudaGetErrorString(e));
  if (e == cudaErrorMemoryAllocation) return DFLASH_ERR_OUT_OF_MEMORY;
  return DFLASH_ERR_CUDA;
}

#define CK(call)                                    \
  do {                                              \
    cudaError_t e_ = (call);                        \
    if (e_ != cudaSuccess) return cuda_fail(e_, #call); \
  } while (0)

int cb_of(int wt) { return wt == WT_BF16 ? Fmt<WT_BF16>::CB : Fmt<WT_Q8_0>::CB; }
// inputs per streaming unit of a weight type (the chunked X layout's KU)
int ku_of(int wt) { return 32 * cb_of(wt); }

__global__ void bf16_to_f32_kernel(const uint16_t* __restrict__ in, float* __restrict__ out, int n) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) out[i] = __uint_as_float(static_cast<uint32_t>(in[i]) << 16);
}

int convert_norm(const void* src, float* dst, int n, cudaStream_t st) {
  bf16_to_f32_kernel<<<(n + 255) / 256, 256, 0, st>>>(static_cast<const uint16_t*>(src), dst, n);
  CK(cudaGetLastError());
  return DFLASH_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// The caller's BF16 rows [rows, cols] for a streamed-input GEMV: boxes of
// (ku + 32) columns x box_rows rows without swizzle, so a box lands with the
// GEMV's padded row stride; columns past the tensor read as zeros.
int make_rows_map(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint32_t ku, uint32_t box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = get_encode();
  if (!enc) {
    std::snprintf(g_cuda_err, sizeof(g_cuda_err), "cuTensorMapEncodeTiled unavailable");
    return DFLASH_ERR_CUDA;
  }
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {ku + 32, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    std::snprintf(g_cuda_err, sizeof(g_cuda_err), "cuTensorMapEncodeTiled (rows) failed (%d)", static_cast<int>(r));
    return DFLASH_ERR_CUDA;
  }
  return DFLASH_OK;
}

// 2-D row-major 16-bit tensor [rows, cols] with 64-column x box_rows boxes, 128-byte swizzle.
int make_map_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, CUtensorMapDataType dt,
                uint32_t box_rows = 64) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = get_encode();
  if (!enc) {
    std::snprintf(g_cuda_err, sizeof(g_cuda_err), "cuTensorMapEncodeTiled unavailable");
    return DFLASH_ERR_CUDA;
  }
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    std::snprintf(g_cuda_err, sizeof(g_cuda_err), "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
    return DFLASH_ERR_CUDA;
  }
  return DFLASH_OK;
}

template <class T>
int dev_alloc(T** p, size_t bytes, size_t* total) {
  void* v = nullptr;
  CK(cudaMalloc(&v, bytes ? bytes : 16));
  *p = static_cast<T*>(v);
  *total += bytes;
  return DFLASH_OK;
}

#define TRY(x)                    \
  do {                            \
    int rc_ = (x);                \
    if (rc_ != DFLASH_OK) return rc_; \
  } while (0)

int alloc_packed(PackedMatrix& pm, int wt, int n, int k, size_t* total) {
  pm.wtype = wt;
  pm.n = n;
  pm.k = k;
  pm.bytes = packed_bytes(wt, n, k);
  TRY(dev_alloc(&pm.data, pm.bytes, total));
  CK(cudaMemset(pm.data, 0, pm.bytes));
  return DFLASH_OK;
}

int repack_into(PackedMatrix& pm, const void* src, int rows, int row_off, int interleave) {
  CK(launch_repack(pm.wtype, src, rows, pm.k, pm.data, row_off, interleave, 0));
  return DFLASH_OK;
}

void free_model(Model* m) {
  if (!m) return;
  auto f = [](void* p) { if (p) cudaFree(p); };
  f(m->fc.data);
  f(m->kv_all.data);
  for (int l = 0; l < DFLASH_MAX_LAYERS; ++l) {
    f(m->qkv[l].data);
    f(m->o[l].data);
    f(m->gu[l].data);
    f(m->down[l].data);
  }
  f(m->hidden_norm);
  f(m->attn_norm);
  f(m->q_norm);
  f(m->k_norm);
  f(m->mlp_norm);
  f(m->final_norm);
  f(m->rope_turns);
}

void free_state(State* s) {
  if (!s) return;
  auto f = [](void* p) { if (p) cudaFree(p); };
  f(s->K); f(s->V); f(s->x); f(s->qkv_raw); f(s->q_ready); f(s->attn_out); f(s->hbuf); f(s->xnorm);
  f(s->xn); f(s->ssq); f(s->attn_part); f(s->attn_ml); f(s->attn_plan); f(s->partials); f(s->counters); f(s->argmax_slots); f(s->argmax_ms); f(s->draft_probs); f(s->nonfinite);
  f(s->head_keys); f(s->head_keys8); f(s->h_raw); f(s->kv_raw); f(s->fuse_xnorm); f(s->fuse_xn); f(s->fuse_ssq); f(s->status);
}

int pow2ceil(int v) {
  int p = 1;
  while (p < v) p <<= 1;
  return p;
}


GemvArgs base_args(const PackedMatrix& pm, State& st, int region, int32_t* status) {
  GemvArgs a;
  std::memset(&a, 0, sizeof(a));
  a.trace = trace_slot(st);
  a.W = pm.data;
  a.N = pm.n;
  a.K = pm.k;
  a.UPG = pm.k / (32 * cb_of(pm.wtype));
  a.U = (pm.n / 64) * a.UPG;
  a.partials = st.partials;
  a.counters = st.counters + static_cast<size_t>(region) * st.counter_stride;
  a.status = status;
  return a;
}

// The GEMV asks L2 for the first kPrefetchUnits units of each share of the
// next projection's weights once it has issued its last unit (the next
// kernel's stream then starts from L2); the shares follow the next GEMV's grid.
constexpr int kPrefetchUnits = 8;
int grid_for(const Model& m, const GemvArgs& a);
void set_prefetch(const Model& m, GemvArgs& a, const PackedMatrix& next) {
  GemvArgs t;
  std::memset(&t, 0, sizeof(t));
  t.UPG = next.k / (32 * cb_of(next.wtype));
  t.U = (next.n / 64) * t.UPG;
  if (t.U <= 0) return;
  a.pf_W = next.data;
  a.pf_total = next.bytes;
  a.pf_U = t.U;
  a.pf_unit = static_cast<int>(next.bytes / static_cast<size_t>(t.U));
  a.pf_G = grid_for(m, t);
  a.pf_bytes = kPrefetchUnits * a.pf_unit;
}

// Grid of a GEMV: one CTA per SM at most, with the CTAs' unit ranges aligned
// to the 64-row groups where the counts allow, so that no CTA meets a group
// end in the middle of its range (a split group's fix-up, or a whole head's
// epilogue, then waits for the CTA's own tail instead of stalling its
// stream).  Groups <= SMs: every group is split into the same number of
// parts; more groups than SMs: whole groups per CTA if the group count has a
// divisor within 70 % of the SM count; otherwise plain stream-K over all SMs.
int grid_for(const Model& m, const GemvArgs& a) {
  const int sm = m.sm_count;
  const int groups = a.UPG > 0 ? a.U / a.UPG : 0;
  if (groups >= 1 && groups <= sm) {
    const int parts = sm / groups < a.UPG ? sm / groups : a.UPG;  // at least one unit per CTA
    return groups * parts;
  }
  for (int g = sm; g * 10 >= sm * 7; --g)
    if (g >= 1 && groups % g == 0) return g;
  int g = sm;
  if (g > a.U) g = a.U;
  return g < 1 ? 1 : g;
}

// Cluster finishing of an 8-row GEMV whose grid splits every 64-row group
// into the same number of parts (grid_for with groups <= SMs): clusters of
// parts x gph CTAs (gph = groups per attention head for the per-head
// epilogue, else 1), at most 8.  Sets a.cl_parts / a.cl_gph and returns the
// cluster size, or 1 (no clusters: the counter-based finishing) when the
// shape does not allow it.
int plan_cluster(GemvArgs& a, int grid, int gph) {
  a.cl_parts = a.cl_gph = 0;
  const int groups = a.UPG > 0 ? a.U / a.UPG : 0;
  if (groups < 1 || grid % groups) return 1;
  const int parts = grid / groups;
  if (parts > a.UPG || groups % gph) return 1;
  const int cs = parts * gph;
  if (cs <= 1 || cs > 8 || gph > 4) return 1;
  a.cl_parts = parts;
  a.cl_gph = gph;
  return cs;
}

int check_gemv(cudaError_t e, const char* what) {
  if (e != cudaSuccess) return cuda_fail(e, what);
  return DFLASH_OK;
}

cudaError_t gemv_store_any(int wt, int nt, const GemvArgs& a, const EpiStore& e, const LaunchCfg& lc) {
  switch (wt) {
    case WT_BF16: return gemv_store<WT_BF16>(nt, a, e, lc);
    case WT_Q8_0: return gemv_store<WT_Q8_0>(nt, a, e, lc);
    case WT_Q5_0: return gemv_store<WT_Q5_0>(nt, a, e, lc);
    case WT_Q4_0: return gemv_store<WT_Q4_0>(nt, a, e, lc);
  }
  return cudaErrorInvalidValue;
}
cudaError_t gemv_resid_any(int wt, int nt, const GemvArgs& a, const EpiResid& e, const LaunchCfg& lc) {
  switch (wt) {
    case WT_BF16: return gemv_resid<WT_BF16>(nt, a, e, lc);
    case WT_Q8_0: return gemv_resid<WT_Q8_0>(nt, a, e, lc);
    case WT_Q5_0: return gemv_resid<WT_Q5_0>(nt, a, e, lc);
    case WT_Q4_0: return gemv_resid<WT_Q4_0>(nt, a, e, lc);
  }
  return cudaErrorInvalidValue;
}
cudaError_t gemv_swiglu_any(int wt, int nt, const GemvArgs& a, void* h, const LaunchCfg& lc) {
  switch (wt) {
    case WT_BF16: return gemv_swiglu<WT_BF16>(nt, a, h, lc);
    case WT_Q8_0: return gemv_swiglu<WT_Q8_0>(nt, a, h, lc);
    case WT_Q5_0: return gemv_swiglu<WT_Q5_0>(nt, a, h, lc);
    case WT_Q4_0: return gemv_swiglu<WT_Q4_0>(nt, a, h, lc);
  }
  return cudaErrorInvalidValue;
}
cudaError_t gemv_heads_any(int wt, int nt, const GemvArgs& a, const EpiHeads& e, const LaunchCfg& lc) {
  switch (wt) {
    case WT_BF16: return gemv_heads<WT_BF16>(nt, a, e, lc);
    case WT_Q8_0: return gemv_heads<WT_Q8_0>(nt, a, e, lc);
    case WT_Q5_0: return gemv_heads<WT_Q5_0>(nt, a, e, lc);
    case WT_Q4_0: return gemv_heads<WT_Q4_0>(nt, a, e, lc);
  }
  return cudaErrorInvalidValue;
}

// Record the next profiling event on `stream` (no-op unless profiling is on).
void prof_mark(State* s, cudaStream_t stream) {
  if (s->prof_n > 0 && s->prof_k < s->prof_n)
    cudaEventRecordWithFlags(static_cast<cudaEvent_t>(s->prof_events[s->prof_k++]), stream, cudaEventRecordExternal);
}

bool is_dev_ptr(const void* p) {
  if (!p) return false;
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged;
}

}  // namespace

extern "C" {

const char* dflash_status_string(int status) {
  switch (status) {
    case DFLASH_OK: return "ok";
    case DFLASH_ERR_INVALID_ARG: return "invalid argument";
    case DFLASH_ERR_UNSUPPORTED: return "unsupported configuration";
    case DFLASH_ERR_CAPACITY: return "request exceeds the state's capacity";
    case DFLASH_ERR_CUDA: return "CUDA error";
    case DFLASH_ERR_NO_DEVICE: return "no usable sm_100+ GPU";
    case DFLASH_ERR_OUT_OF_MEMORY: return "out of device memory";
  }
  return "unknown status";
}

const char* dflash_last_cuda_error(void) { return g_cuda_err; }

int dflash_config_check(const dflash_config* c) {
  if (!c) return DFLASH_ERR_INVALID_ARG;
  if (c->n_layers < 1 || c->n_layers > DFLASH_MAX_LAYERS) return DFLASH_ERR_UNSUPPORTED;
  if (c->head_dim != 64 && c->head_dim != 128 && c->head_dim != 256) return DFLASH_ERR_UNSUPPORTED;
  if (c->n_q_heads < 1 || c->n_kv_heads < 1 || c->n_q_heads % c->n_kv_heads) return DFLASH_ERR_UNSUPPORTED;
  const int gq = c->n_q_heads / c->n_kv_heads;
  if ((gq * 8) % 16 || gq * 8 > 128) return DFLASH_ERR_UNSUPPORTED;
  // the attention CTA holds the M = 8 * gq query rows, two K and two V tiles and P in shared memory
  if (attn_smem_bytes(c->head_dim, gq * 8) > 232448) return DFLASH_ERR_UNSUPPORTED;
  // (the row RMSNorm holds a row of at most 8192 values in one CTA's registers)
  if (c->hidden < 256 || c->hidden % 256 || c->hidden > 8192) return DFLASH_ERR_UNSUPPORTED;
  if ((c->n_q_heads * c->head_dim) % 256 || c->intermediate < 256 || c->intermediate % 256)
    return DFLASH_ERR_UNSUPPORTED;
  if ((c->n_kv_heads * c->head_dim) % 64) return DFLASH_ERR_UNSUPPORTED;
  if (c->n_taps < 1 || c->n_taps > 64) return DFLASH_ERR_UNSUPPORTED;
  if (c->vocab < 2) return DFLASH_ERR_UNSUPPORTED;
  if (c->attn_window < 0) return DFLASH_ERR_INVALID_ARG;
  if (c->mask_token_id < 0 || c->mask_token_id >= c->vocab) return DFLASH_ERR_INVALID_ARG;
  if (!(c->rope_theta > 0.f) || !std::isfinite(c->rope_theta)) return DFLASH_ERR_INVALID_ARG;
  if (!(c->norm_eps >= 0.f) || !std::isfinite(c->norm_eps)) return DFLASH_ERR_INVALID_ARG;
  if (c->weight_type < DFLASH_WT_BF16 || c->weight_type > DFLASH_WT_Q4_0) return DFLASH_ERR_UNSUPPORTED;
  // (head rows fit 32-bit tensor-map coordinates: vocab is an int32; the K/V
  // arena's rows are checked when a state is created)
  return DFLASH_OK;
}

size_t dflash_model_device_bytes(const dflash_model* m) { return m ? m->device_bytes : 0; }
size_t dflash_state_device_bytes(const dflash_state* s) { return s ? s->device_bytes : 0; }

int dflash_model_create(const dflash_config* cfg, const dflash_weights* w, dflash_model** out) {
  if (!cfg || !w || !out) return DFLASH_ERR_INVALID_ARG;
  *out = nullptr;
  TRY(dflash_config_check(cfg));
  const dflash_config& c = *cfg;
  const int L = c.n_layers, H = c.hidden, d = c.head_dim, nq = c.n_q_heads, nkv = c.n_kv_heads, I = c.intermediate;
  if (!w->fc || !w->hidden_norm || !w->final_norm || !w->embed || !w->head) return DFLASH_ERR_INVALID_ARG;
  for (int l = 0; l < L; ++l) {
    const dflash_layer_weights& lw = w->layers[l];
    const void* ps[] = {lw.attn_norm, lw.wq, lw.wk, lw.wv, lw.q_norm, lw.k_norm, lw.wo, lw.mlp_norm,
                        lw.w_gate, lw.w_up, lw.w_down};
    for (const void* p : ps)
      if (!p) return DFLASH_ERR_INVALID_ARG;
  }
  if (reinterpret_cast<uintptr_t>(w->head) % 16) return DFLASH_ERR_INVALID_ARG;
  int dev = 0;
  int ndev = 0;
  if (cudaGetDeviceCount(&ndev) != cudaSuccess || ndev == 0) {
    cudaGetLastError();
    return DFLASH_ERR_NO_DEVICE;
  }
  CK(cudaGetDevice(&dev));
  cudaDeviceProp prop;
  CK(cudaGetDeviceProperties(&prop, dev));
  if (prop.major < 10) return DFLASH_ERR_NO_DEVICE;
  if (!is_dev_ptr(w->fc) || !is_dev_ptr(w->head) || !is_dev_ptr(w->embed)) return DFLASH_ERR_INVALID_ARG;

  dflash_model* m = new (std::nothrow) dflash_model();
  if (!m) return DFLASH_ERR_OUT_OF_MEMORY;
  m->cfg = c;
  m->wtype = c.weight_type;
  m->device = dev;
  m->sm_count = prop.multiProcessorCount;
  m->embed = static_cast<const uint16_t*>(w->embed);
  m->head = static_cast<const uint16_t*>(w->head);
  size_t total = 0;
  const int wt = c.weight_type;
  auto fail = [&](int rc) {
    free_model(m);
    delete m;
    return rc;
  };
  int rc;
#define MTRY(x)                      \
  do {                               \
    if ((rc = (x)) != DFLASH_OK) return fail(rc); \
  } while (0)
  const int nqkv = (nq + 2 * nkv) * d;
  MTRY(alloc_packed(m->fc, wt, H, c.n_taps * H, &total));
  MTRY(repack_into(m->fc, w->fc, H, 0, -1));
  MTRY(alloc_packed(m->kv_all, wt, L * 2 * nkv * d, H, &total));
  for (int l = 0; l < L; ++l) {
    const dflash_layer_weights& lw = w->layers[l];
    MTRY(alloc_packed(m->qkv[l], wt, nqkv, H, &total));
    MTRY(repack_into(m->qkv[l], lw.wq, nq * d, 0, -1));
    MTRY(repack_into(m->qkv[l], lw.wk, nkv * d, nq * d, -1));
    MTRY(repack_into(m->qkv[l], lw.wv, nkv * d, (nq + nkv) * d, -1));
    MTRY(repack_into(m->kv_all, lw.wk, nkv * d, l * 2 * nkv * d, -1));
    MTRY(repack_into(m->kv_all, lw.wv, nkv * d, l * 2 * nkv * d + nkv * d, -1));
    MTRY(alloc_packed(m->o[l], wt, H, nq * d, &total));
    MTRY(repack_into(m->o[l], lw.wo, H, 0, -1));
    MTRY(alloc_packed(m->gu[l], wt, 2 * I, H, &total));
    MTRY(repack_into(m->gu[l], lw.w_gate, I, 0, 0));
    MTRY(repack_into(m->gu[l], lw.w_up, I, 0, 1));
    MTRY(alloc_packed(m->down[l], wt, H, I, &total));
    MTRY(repack_into(m->down[l], lw.w_down, H, 0, -1));
  }
  MTRY(dev_alloc(&m->hidden_norm, H * 4, &total));
  MTRY(dev_alloc(&m->attn_norm, size_t(L) * H * 4, &total));
  MTRY(dev_alloc(&m->q_norm, size_t(L) * d * 4, &total));
  MTRY(dev_alloc(&m->k_norm, size_t(L) * d * 4, &total));
  MTRY(dev_alloc(&m->mlp_norm, size_t(L) * H * 4, &total));
  MTRY(dev_alloc(&m->final_norm, H * 4, &total));
  MTRY(convert_norm(w->hidden_norm, m->hidden_norm, H, 0));
  MTRY(convert_norm(w->final_norm, m->final_norm, H, 0));
  for (int l = 0; l < L; ++l) {
    const dflash_layer_weights& lw = w->layers[l];
    MTRY(convert_norm(lw.attn_norm, m->attn_norm + size_t(l) * H, H, 0));
    MTRY(convert_norm(lw.q_norm, m->q_norm + size_t(l) * d, d, 0));
    MTRY(convert_norm(lw.k_norm, m->k_norm + size_t(l) * d, d, 0));
    MTRY(convert_norm(lw.mlp_norm, m->mlp_norm + size_t(l) * H, H, 0));
  }
  // RoPE frequencies as 0.64 fixed-point turns: inv_freq_i / (2 pi) * 2^64.
  {
    uint64_t turns[128];
    const double two_pi = 6.283185307179586476925286766559;
    for (int i = 0; i < d / 2; ++i) {
      const double inv_freq = std::pow(static_cast<double>(c.rope_theta), -2.0 * i / d);
      const double t = std::ldexp(inv_freq / two_pi, 64);
      turns[i] = t >= 18446744073709551615.0 ? ~0ull : static_cast<uint64_t>(t);
    }
    MTRY(dev_alloc(&m->rope_turns, sizeof(uint64_t) * (d / 2), &total));
    if (cudaMemcpy(m->rope_turns, turns, sizeof(uint64_t) * (d / 2), cudaMemcpyHostToDevice) != cudaSuccess)
      return fail(cuda_fail(cudaGetLastError(), "cudaMemcpy rope turns"));
  }
  MTRY(make_map_2d(&m->head_map, w->head, static_cast<uint64_t>(c.vocab), static_cast<uint64_t>(H),
                   CU_TENSOR_MAP_DATA_TYPE_BFLOAT16));
  {
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return fail(cuda_fail(e, "model create"));
  }
  m->device_bytes = total;
#undef MTRY
  *out = m;
  return DFLASH_OK;
}

int dflash_model_destroy(dflash_model* m) {
  if (!m) return DFLASH_ERR_INVALID_ARG;
  free_model(m);
  delete m;
  return DFLASH_OK;
}

int dflash_state_create(const dflash_model* m, int32_t n_slots, int32_t capacity, dflash_state** out) {
  if (!m || !out) return DFLASH_ERR_INVALID_ARG;
  *out = nullptr;
  if (n_slots < 1 || n_slots > DFLASH_MAX_SLOTS) return DFLASH_ERR_INVALID_ARG;
  if (capacity < DFLASH_MAX_BLOCK) return DFLASH_ERR_INVALID_ARG;
  const dflash_config& c = m->cfg;
  const int L = c.n_layers, H = c.hidden, d = c.head_dim, nq = c.n_q_heads, nkv = c.n_kv_heads, I = c.intermediate;
  const long long arena_rows = static_cast<long long>(L) * n_slots * nkv * capacity;
  if (arena_rows > 0x7fffffffLL) return DFLASH_ERR_CAPACITY;
  // a ring of cells (attention window) must hold the window and keep every
  // 128-position super-tile of the attention in one contiguous run of cells
  if (m->cfg.attn_window > 0 && (capacity < m->cfg.attn_window || capacity % 128)) return DFLASH_ERR_UNSUPPORTED;
  dflash_state* s = new (std::nothrow) dflash_state();
  if (!s) return DFLASH_ERR_OUT_OF_MEMORY;
  auto fail = [&](int rc) {
    free_state(s);
    delete s;
    return rc;
  };
  int rc;
#define STRY(x)                      \
  do {                               \
    if ((rc = (x)) != DFLASH_OK) return fail(rc); \
  } while (0)
  s->model = m;
  s->n_slots = n_slots;
  s->capacity = capacity;
  s->nt = pow2ceil(n_slots);
  s->rows = s->nt * 8;
  const int R = s->rows;
  const int gq = nq / nkv;
  const int M = gq * 8;
  {
    // default: one 128-key super-tile per CTA, at most one CTA per SM (each
    // holds 225 KB of shared memory and 512 TMEM columns); buffers sized for
    // up to 4 CTAs' worth of chunks per SM (and at most 512 chunks, the merge
    // kernel's limit)
    // positions one block attends to: the window (plus alignment), else the whole state
    const long long span = m->cfg.attn_window > 0 ? static_cast<long long>(m->cfg.attn_window) + 128 : capacity;
    const long long tiles = (span + 127) / 128;
    const long long per = static_cast<long long>(n_slots) * nkv;
    long long cmax = (4LL * m->sm_count) / per;
    cmax = cmax < 1 ? 1 : (cmax > 512 ? 512 : cmax);
    if (cmax > tiles) cmax = tiles;
    long long cdef = tiles;
    const long long cap1 = m->sm_count / per;
    if (cdef > cap1) cdef = cap1;
    if (cdef > cmax) cdef = cmax;
    if (cdef < 1) cdef = 1;
    s->attn_chunks = static_cast<int>(cdef);
    s->attn_chunks_max = static_cast<int>(cmax);
  }
  size_t total = 0;
  const size_t kv_elems = static_cast<size_t>(arena_rows) * d;
  STRY(dev_alloc(&s->K, kv_elems * 2, &total));
  STRY(dev_alloc(&s->V, kv_elems * 2, &total));
  if (cudaMemset(s->K, 0, kv_elems * 2) != cudaSuccess || cudaMemset(s->V, 0, kv_elems * 2) != cudaSuccess)
    return fail(cuda_fail(cudaGetLastError(), "cudaMemset K/V"));
  const int nqkv = (nq + 2 * nkv) * d;
  STRY(dev_alloc(&s->x, size_t(R) * H * 4, &total));
  STRY(dev_alloc(&s->qkv_raw, size_t(R) * nqkv * 4, &total));
  STRY(dev_alloc(&s->q_ready, size_t(R) * nq * d * 2, &total));
  // activations for streamed-X GEMVs: two 16-bit planes (BF16 hi and lo, or FP16 in the first)
  STRY(dev_alloc(&s->attn_out, xchunk_elems(nq * d, R, 128, 2) * 2, &total));
  // rows of a tile's unused slots are never written by a pass: keep them zero
  if (cudaMemset(s->attn_out, 0, xchunk_elems(nq * d, R, 128, 2) * 2) != cudaSuccess)
    return fail(cuda_fail(cudaGetLastError(), "cudaMemset attn_out"));
  STRY(dev_alloc(&s->hbuf, xchunk_elems(I, R, 128, 2) * 2, &total));
  STRY(dev_alloc(&s->xnorm, xchunk_elems(H, R, 128, 2) * 2, &total));
  STRY(dev_alloc(&s->xn, xchunk_elems(H, 8, 128, 2) * 2, &total));  // largest for 128 inputs per unit
  STRY(dev_alloc(&s->ssq, size_t(H / 64) * 8 * 4, &total));
  STRY(dev_alloc(&s->attn_part, size_t(n_slots) * nkv * s->attn_chunks_max * M * d * 2, &total));
  STRY(dev_alloc(&s->attn_ml, size_t(n_slots) * nkv * s->attn_chunks_max * M * 8, &total));
  STRY(dev_alloc(&s->attn_plan, 32 * 4, &total));
  s->max_grid = 2 * m->sm_count;
  const int rmax = 128;
  STRY(dev_alloc(&s->partials, size_t(s->max_grid) * 2 * 64 * rmax * 4, &total));
  {
    int stride = c.vocab / 64 + 1;
    const int cands[] = {nqkv / 64, H / 64, 2 * I / 64, L * 2 * nkv * d / 64, nq + 2 * nkv, L * 2 * nkv, 16};
    for (int v : cands) stride = stride > v ? stride : v + 1;
    s->counter_stride = stride;
  }
  STRY(dev_alloc(&s->counters, size_t(CNT_REGIONS) * s->counter_stride * 4, &total));
  if (cudaMemset(s->counters, 0, size_t(CNT_REGIONS) * s->counter_stride * 4) != cudaSuccess)
    return fail(cuda_fail(cudaGetLastError(), "cudaMemset counters"));
  STRY(dev_alloc(&s->argmax_slots, size_t(s->max_grid) * rmax * 8, &total));
  STRY(dev_alloc(&s->argmax_ms, size_t(s->max_grid) * rmax * 8, &total));
  STRY(dev_alloc(&s->draft_probs, size_t(n_slots) * (DFLASH_MAX_BLOCK - 1) * 4, &total));
  STRY(dev_alloc(&s->nonfinite, 16, &total));
  s->fuse_rows = 128;
  STRY(dev_alloc(&s->h_raw, size_t(s->fuse_rows) * H * 4, &total));
  STRY(dev_alloc(&s->kv_raw, size_t(s->fuse_rows) * L * 2 * nkv * d * 4, &total));
  STRY(dev_alloc(&s->fuse_xnorm, xchunk_elems(H, 128, 128, 2) * 2, &total));
  STRY(dev_alloc(&s->fuse_xn, xchunk_elems(H, 8, 128, 2) * 2, &total));
  STRY(dev_alloc(&s->fuse_ssq, size_t(H / 64) * 8 * 4, &total));
  STRY(dev_alloc(&s->status, 16, &total));
  if (cudaMemset(s->status, 0, 16) != cudaSuccess) return fail(cuda_fail(cudaGetLastError(), "cudaMemset"));
  STRY(make_map_2d(&s->q_map, s->q_ready, static_cast<uint64_t>(s->nt) * nkv * M, d, CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                   static_cast<uint32_t>(M)));
  STRY(make_map_2d(&s->part_map, s->attn_part, static_cast<uint64_t>(n_slots) * nkv * s->attn_chunks_max * M, d,
                   CU_TENSOR_MAP_DATA_TYPE_FLOAT16, static_cast<uint32_t>(M)));
  STRY(make_map_2d(&s->k_map, s->K, static_cast<uint64_t>(arena_rows), d, CU_TENSOR_MAP_DATA_TYPE_FLOAT16));
  STRY(make_map_2d(&s->v_map, s->V, static_cast<uint64_t>(arena_rows), d, CU_TENSOR_MAP_DATA_TYPE_FLOAT16));
  if (R == 128 && H % 256 == 0 && (nq * d) % 256 == 0 && I % 256 == 0) {
    // the chunked activations of a 128-row pass as rows of one unit's inputs
    // (K / KU * planes * 128 rows of KU + 32), for the tcgen05 layer GEMMs
    const int ku = ku_of(m->wtype), pl = m->wtype == WT_BF16 ? 2 : 1;
    const CUtensorMapDataType dt = m->wtype == WT_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    STRY(make_map_2d(&s->tc_xnorm_map, s->xnorm, static_cast<uint64_t>(H / ku) * pl * 128, ku + 32, dt, 128));
    STRY(make_map_2d(&s->tc_attn_map, s->attn_out, static_cast<uint64_t>(nq * d / ku) * pl * 128, ku + 32, dt, 128));
    STRY(make_map_2d(&s->tc_hbuf_map, s->hbuf, static_cast<uint64_t>(I / ku) * pl * 128, ku + 32, dt, 128));
    s->tc_maps = 1;
  }
  if (H % 128 == 0) {
    // the packed rows the LM head of a one-sequence pass reads: per 128-input
    // chunk the 8 hi rows then the 8 lo rows (row stride 160)
    STRY(make_map_2d(&s->xn_map, s->xn, static_cast<uint64_t>(H / 128) * 16, 160, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 16));
  }
  STRY(dev_alloc(&s->head_keys8, 8 * 8, &total));
  if (cudaMemset(s->head_keys8, 0, 8 * 8) != cudaSuccess)
    return fail(cuda_fail(cudaGetLastError(), "cudaMemset head_keys8"));
  if (R == 128) {
    // the final normed rows of a 128-row pass, one chunk of H inputs per row (row stride H + 32)
    STRY(make_map_2d(&s->xhead_map, s->xnorm, 2 * 128, static_cast<uint64_t>(H) + 32, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                     128));
    STRY(dev_alloc(&s->head_keys, 128 * 8, &total));
    if (cudaMemset(s->head_keys, 0, 128 * 8) != cudaSuccess)
      return fail(cuda_fail(cudaGetLastError(), "cudaMemset head_keys"));
  }
  {
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return fail(cuda_fail(e, "state create"));
  }
  s->device_bytes = total;
#undef STRY
  *out = s;
  return DFLASH_OK;
}

int dflash_state_destroy(dflash_state* s) {
  if (!s) return DFLASH_ERR_INVALID_ARG;
  free_state(s);
  delete s;
  return DFLASH_OK;
}

// K/V of every layer for `rows` fused rows (positions[rows] of `slot`) from
// their x * hidden_norm: X in the chunked layout with the sums of squares ssq
// (8-row tiles), or the rows already normalised (larger tiles, ssq null).
static int launch_fuse_kv(const dflash_model* m, dflash_state* s, const void* X, const float* ssq, int rows,
                          int nt, int32_t slot, const int32_t* positions, int32_t* status, cudaStream_t stream) {
  const dflash_config& c = m->cfg;
  const int H = c.hidden, d = c.head_dim, nkv = c.n_kv_heads, L = c.n_layers;
  GemvArgs a = base_args(m->kv_all, *s, CNT_KV, status);
  a.n_valid_rows = rows;
  a.eps = c.norm_eps;
  a.X = X;
  a.ldx = H;
  if (ssq) {
    a.ssq = ssq;
    a.n_ssq = H / 64;
  }
  EpiHeads e;
  std::memset(&e, 0, sizeof(e));
  e.mode = 1;
  e.raw = s->kv_raw;
  e.ldr = L * 2 * nkv * d;
  e.d = d;
  e.n_q = c.n_q_heads;
  e.n_kv = nkv;
  e.gph = d / 64;
  e.head_cnt = s->counters + static_cast<size_t>(CNT_KV_HEADS) * s->counter_stride;
  e.k_norm = m->k_norm;
  e.turns = m->rope_turns;
  e.eps = c.norm_eps;
  e.q_scale = 1.f;
  e.Kst = s->K;
  e.Vst = s->V;
  e.n_slots = s->n_slots;
  e.cap = s->capacity;
  e.ring = c.attn_window > 0;
  e.slot = slot;
  e.positions = positions;
  e.n_valid = rows;
  e.status = status;
  e.rows_ = nt * 8;
  LaunchCfg lc{stream, grid_for(*m, a), true};
  if (nt == 1) lc.cluster = plan_cluster(a, lc.grid, e.gph);
  prof_mark(s, stream);
  return check_gemv(gemv_heads_any(m->wtype, nt, a, e, lc), "fuse kv");
}

// Projects the K/V of a deferred 8-row fusion now (a separate GEMV).
static int flush_deferred(const dflash_model* m, dflash_state* s, cudaStream_t stream) {
  if (s->pend_n <= 0) return DFLASH_OK;
  const int rows = s->pend_n;
  s->pend_n = 0;
  return launch_fuse_kv(m, s, s->fuse_xn, s->fuse_ssq, rows, 1, s->pend_slot, s->pend_pos, s->pend_status, stream);
}

int dflash_fuse_context(const dflash_model* m, dflash_state* s, int32_t slot, const uint16_t* taps,
                        const int32_t* positions, int32_t n, int32_t* dev_status, dflash_stream_t stream_) {
  if (!m || !s || s->model != m) return DFLASH_ERR_INVALID_ARG;
  if (slot < 0 || slot >= s->n_slots || n < 0) return DFLASH_ERR_INVALID_ARG;
  if (n == 0) return DFLASH_OK;
  if (!taps || !positions) return DFLASH_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(taps) % 16) return DFLASH_ERR_INVALID_ARG;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const dflash_config& c = m->cfg;
  const int H = c.hidden;
  const int wt = m->wtype;
  int32_t* status = dev_status ? dev_status : s->status;
  const int tw = c.n_taps * H;
  s->prof_k = 0;
  // an earlier deferred fusion is projected first (its rows may be re-fused here)
  TRY(flush_deferred(m, s, stream));
  for (int base = 0; base < n; base += s->fuse_rows) {
    const int rows = (n - base) < s->fuse_rows ? (n - base) : s->fuse_rows;
    const int nt = rows <= 8 ? 1 : 16;
    // with 8 rows the fc epilogue also packs h * hidden_norm for the K/V GEMV
    const bool fpacked = fused_norm(nt);
    // a single 8-row tile of a deferring state leaves its K/V to the next draft pass
    const bool defer = s->defer_kv && fpacked && n <= 8;
    // fc: h_raw = taps . W_fc^T
    {
      GemvArgs a = base_args(m->fc, *s, CNT_FC, status);
      a.n_valid_rows = rows;
      // a deferring fusion is followed by a draft pass, which starts with layer 0's QKV
      if (defer) set_prefetch(*m, a, m->qkv[0]);
      a.X = taps + static_cast<size_t>(base) * tw;
      a.ldx = tw;
      if (ku_of(wt) + 32 <= 256)
        TRY(make_rows_map(&a.xmap, a.X, static_cast<uint64_t>(rows), static_cast<uint64_t>(tw),
                          static_cast<uint32_t>(ku_of(wt)), static_cast<uint32_t>(rows)));
      EpiStore e{s->h_raw, H,
                 PackNext{fpacked ? (defer ? s->fuse_xn : s->xn) : nullptr, defer ? s->fuse_ssq : s->ssq,
                          m->hidden_norm, ku_of(wt), wt != WT_BF16}};
      LaunchCfg lc{stream, grid_for(*m, a), true};
      if (nt == 1) lc.cluster = plan_cluster(a, lc.grid, 1);
      prof_mark(s, stream);
      TRY(check_gemv(gemv_store_any(wt, nt, a, e, lc), "fuse fc"));
    }
    if (defer) {
      s->pend_n = rows;
      s->pend_slot = slot;
      s->pend_pos = positions + base;
      s->pend_status = status;
      continue;
    }
    // K/V of every layer from rmsnorm(h_raw) * hidden_norm
    if (fpacked) {
      TRY(launch_fuse_kv(m, s, s->xn, s->ssq, rows, nt, slot, positions + base, status, stream));
    } else {
      NormArgs na{s->h_raw, m->hidden_norm, s->fuse_xnorm, wt != WT_BF16, H, rows, c.norm_eps, nullptr, 0,
                  ku_of(wt)};
      prof_mark(s, stream);
      TRY(check_gemv(launch_rmsnorm_rows(na, nt * 8, stream), "fuse norm"));
      TRY(launch_fuse_kv(m, s, s->fuse_xnorm, nullptr, rows, nt, slot, positions + base, status, stream));
    }
  }
  prof_mark(s, stream);
  return DFLASH_OK;
}

int dflash_draft_block(const dflash_model* m, dflash_state* s, int32_t n_seq, const int32_t* anchor_tok,
                       const int32_t* anchor_pos, const int32_t* block_len, int32_t* drafts, float* final_hidden,
                       int32_t* dev_status, dflash_stream_t stream_) {
  if (!m || !s || s->model != m) return DFLASH_ERR_INVALID_ARG;
  if (n_seq < 1 || n_seq > s->n_slots) return DFLASH_ERR_INVALID_ARG;
  if (!anchor_tok || !anchor_pos || !block_len || !drafts) return DFLASH_ERR_INVALID_ARG;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const dflash_config& c = m->cfg;
  const int L = c.n_layers, H = c.hidden, d = c.head_dim, nq = c.n_q_heads, nkv = c.n_kv_heads, I = c.intermediate;
  const int wt = m->wtype;
  const int nt = pow2ceil(n_seq);
  const int R = nt * 8;
  int32_t* status = dev_status ? dev_status : s->status;
  const bool f16 = wt != WT_BF16;

  s->prof_k = 0;
  // one-slot passes: every RMSNorm-fed GEMV reads the packed rows that the
  // kernel producing x wrote (embed, o-proj and down residual epilogues)
  const bool packed = fused_norm(nt);
  auto set_packed = [&](GemvArgs& a) {
    a.X = s->xn;
    a.ldx = H;
    a.ssq = s->ssq;
    a.n_ssq = H / 64;
  };
  // A deferred fusion's rows ride in this pass's QKV GEMVs when every group
  // of the widened GEMV gets CTAs of its own in clusters of one head:
  // each layer's W_k / W_v groups are then read by two sets of CTAs at about
  // the same time (block rows, committed rows) instead of once more in a
  // separate launch.  Otherwise they are projected first, separately.
  const int kv_groups = 2 * nkv * d / 64;
  bool carry = false;
  if (s->pend_n > 0 && packed) {
    GemvArgs t = base_args(m->qkv[0], *s, CNT_QKV, status);
    t.U += kv_groups * t.UPG;
    carry = plan_cluster(t, grid_for(*m, t), d / 64) > 1 && (t.U / t.UPG) <= m->sm_count;
  }
  if (s->pend_n > 0 && !carry) TRY(flush_deferred(m, s, stream));
  {
    EmbedArgs ea{m->embed, anchor_tok, anchor_pos, block_len, s->x, H, c.vocab, c.mask_token_id, n_seq,
                 s->capacity, c.attn_window > 0, status, nullptr, nullptr, nullptr, 0, 0};
    if (packed) {
      ea.xn = s->xn;
      ea.ku = ku_of(wt);
      ea.f16 = wt != WT_BF16;
      ea.ssq = s->ssq;
      ea.w_next = m->attn_norm;
    }
    prof_mark(s, stream);
    TRY(check_gemv(launch_embed(ea, nt, stream), "embed"));
  }
  // 128-row passes: the layer GEMMs on the tcgen05 tensor cores, every CTA
  // owning whole 64-row groups
  const bool tc = nt == 16 && s->tc_maps;
  // few groups (outputs of the hidden size): each group's inputs in slices
  auto tc_parts = [&](const GemvArgs& a) {
    const int groups = a.U / a.UPG;
    int p = m->sm_count / groups;
    p = p > a.UPG ? a.UPG : p;
    p = p > 4 ? 4 : p;  // the GEMM sums at most 4 slices
    return p < 2 ? 1 : p;
  };
  // The grid of a 128-row GEMM: slices, groups x parts CTAs; whole groups,
  // the largest grid of at most one CTA per SM (and at least 70 % of that)
  // that gives every CTA the same number of groups, else one group range
  // per CTA over min(groups, SMs) CTAs.
  auto tc_launch = [&](const GemvArgs& a, const TcEpi& te) {
    const int groups = a.U / a.UPG;
    if (te.parts > 1) return groups * te.parts;
    const int gmax = groups < m->sm_count ? groups : m->sm_count;
    for (int G = gmax; G >= 1 && G * 10 >= gmax * 7; --G)
      if (groups % G == 0) return G;
    return gmax;
  };
  TcEpi tc_resid;
  std::memset(&tc_resid, 0, sizeof(tc_resid));
  tc_resid.mode = TcEpi::RESID;
  tc_resid.out = s->x;
  tc_resid.ldo = H;
  for (int l = 0; l < L; ++l) {
    // q, k, v projections with per-head norm, RoPE and block K/V cells
    {
      GemvArgs a = base_args(m->qkv[l], *s, CNT_QKV, status);
      a.n_valid_rows = R;
      a.eps = c.norm_eps;
      set_prefetch(*m, a, m->o[l]);
      if (packed) {
        set_packed(a);
      } else {
        NormArgs na{s->x, m->attn_norm + size_t(l) * H, s->xnorm, f16, H, R, c.norm_eps, nullptr, 0,
                    ku_of(wt)};
        prof_mark(s, stream);
        TRY(check_gemv(launch_rmsnorm_rows(na, R, stream), "attn norm"));
        a.X = s->xnorm;
        a.ldx = H;
      }
      EpiHeads e;
      std::memset(&e, 0, sizeof(e));
      e.mode = 0;
      e.raw = s->qkv_raw;
      e.ldr = (nq + 2 * nkv) * d;
      e.d = d;
      e.n_q = nq;
      e.n_kv = nkv;
      e.gph = d / 64;
      e.head_cnt = s->counters + static_cast<size_t>(CNT_QKV_HEADS) * s->counter_stride;
      e.q_norm = m->q_norm + size_t(l) * d;
      e.k_norm = m->k_norm + size_t(l) * d;
      e.turns = m->rope_turns;
      e.eps = c.norm_eps;
      e.q_scale = 1.f / std::sqrt(static_cast<float>(d));
      e.q_ready = s->q_ready;
      e.Kst = s->K;
      e.Vst = s->V;
      e.layer = l;
      e.n_slots = s->n_slots;
      e.cap = s->capacity;
      e.ring = c.attn_window > 0;
      e.n_seq = n_seq;
      e.window = c.attn_window;
      e.prefetch_kv = 1;
      e.anchor_pos = anchor_pos;
      e.block_len = block_len;
      e.status = status;
      e.rows_ = R;
      if (carry) {
        // the committed rows' K/V of this layer: W_k / W_v groups again, as
        // extra groups over the deferred fusion's packed rows
        a.U += kv_groups * a.UPG;
        a.vgroups = kv_groups;
        a.vwg0 = nq * d / 64;
        a.X2 = s->fuse_xn;
        a.ssq2 = s->fuse_ssq;
        a.n_valid2 = s->pend_n;
        e.n_heads0 = nq + 2 * nkv;
        e.vpositions = s->pend_pos;
        e.vn_valid = s->pend_n;
        e.vslot = s->pend_slot;
      }
      if (tc) {
        a.xmap = s->tc_xnorm_map;
        TcEpi te;
        std::memset(&te, 0, sizeof(te));
        te.mode = TcEpi::HEADS;
        te.heads = e;
        prof_mark(s, stream);
        const int grid = tc_launch(a, te);
        TRY(check_gemv(launch_gemv_tc(wt, a, te, grid, stream), "qkv"));
        prof_mark(s, stream);
        TRY(check_gemv(launch_heads_rows(e, nq + 2 * nkv, n_seq, stream), "qkv heads"));
      } else {
        LaunchCfg lc{stream, grid_for(*m, a), true};
        if (nt == 1) lc.cluster = plan_cluster(a, lc.grid, e.gph);
        prof_mark(s, stream);
        TRY(check_gemv(gemv_heads_any(wt, nt, a, e, lc), "qkv"));
      }
    }
    prof_mark(s, stream);
    TRY(check_gemv(launch_attention(*m, *s, l, n_seq, nt, anchor_pos, block_len, status, stream), "attention"));
    {
      GemvArgs a = base_args(m->o[l], *s, CNT_O, status);
      a.n_valid_rows = R;
      set_prefetch(*m, a, m->gu[l]);
      a.X = s->attn_out;
      a.ldx = nq * d;
      EpiResid e{s->x, H,
                 PackNext{packed ? s->xn : nullptr, s->ssq, m->mlp_norm + size_t(l) * H, ku_of(wt), wt != WT_BF16}};
      if (tc) {
        a.xmap = s->tc_attn_map;
        TcEpi te = tc_resid;
        te.parts = tc_parts(a);
        const int grid = tc_launch(a, te);
        prof_mark(s, stream);
        TRY(check_gemv(launch_gemv_tc(wt, a, te, grid, stream), "o proj"));
      } else {
        LaunchCfg lc{stream, grid_for(*m, a), true};
        if (nt == 1) lc.cluster = plan_cluster(a, lc.grid, 1);
        prof_mark(s, stream);
        TRY(check_gemv(gemv_resid_any(wt, nt, a, e, lc), "o proj"));
      }
    }
    {
      GemvArgs a = base_args(m->gu[l], *s, CNT_GU, status);
      a.n_valid_rows = R;
      set_prefetch(*m, a, m->down[l]);
      a.eps = c.norm_eps;
      if (packed) {
        set_packed(a);
      } else {
        NormArgs na{s->x, m->mlp_norm + size_t(l) * H, s->xnorm, f16, H, R, c.norm_eps, nullptr, 0,
                    ku_of(wt)};
        prof_mark(s, stream);
        TRY(check_gemv(launch_rmsnorm_rows(na, R, stream), "mlp norm"));
        a.X = s->xnorm;
        a.ldx = H;
      }
      if (tc) {
        a.xmap = s->tc_xnorm_map;
        TcEpi te;
        std::memset(&te, 0, sizeof(te));
        te.mode = TcEpi::SWIGLU;
        te.h = s->hbuf;
        te.h_ku = ku_of(wt);
        te.h_f16 = wt != WT_BF16;
        prof_mark(s, stream);
        const int grid = tc_launch(a, te);
        TRY(check_gemv(launch_gemv_tc(wt, a, te, grid, stream), "gate/up"));
      } else {
        LaunchCfg lc{stream, grid_for(*m, a), true};
        prof_mark(s, stream);
        TRY(check_gemv(gemv_swiglu_any(wt, nt, a, s->hbuf, lc), "gate/up"));
      }
    }
    {
      GemvArgs a = base_args(m->down[l], *s, CNT_DOWN, status);
      a.n_valid_rows = R;
      if (l + 1 < L) {
        set_prefetch(*m, a, m->qkv[l + 1]);
      } else if (nt == 1) {
        // the LM head of a one-sequence pass: 128-row chunks, CTA c' of
        // min(chunks, SMs) starting at chunk c' * chunks / grid
        const int nv = (c.vocab + 127) / 128;
        a.pf_W = reinterpret_cast<const uint8_t*>(m->head);
        a.pf_total = static_cast<size_t>(c.vocab) * H * 2;
        a.pf_U = nv;
        a.pf_unit = 128 * H * 2;
        a.pf_G = nv < m->sm_count ? nv : m->sm_count;
        a.pf_bytes = 128 * 1024;
      }
      a.X = s->hbuf;
      a.ldx = I;
      EpiResid e{s->x, H,
                 PackNext{packed ? s->xn : nullptr, s->ssq,
                          l + 1 < L ? m->attn_norm + size_t(l + 1) * H : m->final_norm,
                          l + 1 < L ? ku_of(wt) : 32 * Fmt<WT_HEAD>::CB, l + 1 < L && wt != WT_BF16}};
      if (tc) {
        a.xmap = s->tc_hbuf_map;
        TcEpi te = tc_resid;
        te.parts = tc_parts(a);
        const int grid = tc_launch(a, te);
        prof_mark(s, stream);
        TRY(check_gemv(launch_gemv_tc(wt, a, te, grid, stream), "down"));
      } else {
        LaunchCfg lc{stream, grid_for(*m, a), true};
        if (nt == 1) lc.cluster = plan_cluster(a, lc.grid, 1);
        prof_mark(s, stream);
        TRY(check_gemv(gemv_resid_any(wt, nt, a, e, lc), "down"));
      }
    }
  }
  // final norm + LM head + argmax
  {
    GemvArgs a;
    std::memset(&a, 0, sizeof(a));
    a.wmap = m->head_map;
    a.N = ((c.vocab + 63) / 64) * 64;
    a.K = H;
    a.UPG = H / 128;
    a.U = (a.N / 64) * a.UPG;
    a.n_valid_rows = R;
    a.eps = c.norm_eps;
    a.partials = s->partials;
    a.counters = s->counters + static_cast<size_t>(CNT_HEAD) * s->counter_stride;
    a.status = status;
    a.trace = trace_slot(*s);
    ArgmaxParams p;
    p.vocab = c.vocab;
    p.n_seq = n_seq;
    p.H = H;
    p.block_len = block_len;
    p.drafts = drafts;
    p.slots = s->argmax_slots;
    p.ms = s->argmax_ms;
    p.probs = s->draft_probs;
    p.min_p = s->spec_min_p;
    p.grid_cnt = s->counters + static_cast<size_t>(CNT_ARGMAX) * s->counter_stride;
    p.final_hidden = final_hidden;
    a.rs_early = final_hidden != nullptr;
    p.x = s->x;
    p.norm_w = m->final_norm;
    p.status = status;
    if (packed && H % 128 == 0) {
      // one sequence: the head on tcgen05, 128 vocabulary rows per MMA
      HeadTcArgs ha;
      std::memset(&ha, 0, sizeof(ha));
      ha.wmap = m->head_map;
      ha.xmap = s->xn_map;
      ha.V = c.vocab;
      ha.H = H;
      ha.n_seq = 1;
      ha.block_len = block_len;
      ha.drafts = drafts;
      ha.probs = s->draft_probs;
      ha.min_p = s->spec_min_p;
      ha.keys = s->head_keys8;
      ha.ms = s->argmax_ms;
      ha.grid_cnt = p.grid_cnt;
      ha.status = status;
      ha.ssq = s->ssq;
      ha.eps = c.norm_eps;
      ha.final_hidden = final_hidden;
      ha.x = s->x;
      ha.norm_w = m->final_norm;
      const int nv = (c.vocab + 127) / 128;
      if (s->head_ev_begin) CK(cudaEventRecordWithFlags(static_cast<cudaEvent_t>(s->head_ev_begin), stream, cudaEventRecordExternal));
      prof_mark(s, stream);
      TRY(check_gemv(launch_head_tc8(ha, nv < m->sm_count ? nv : m->sm_count, stream), "lm head"));
      if (s->head_ev_end) CK(cudaEventRecordWithFlags(static_cast<cudaEvent_t>(s->head_ev_end), stream, cudaEventRecordExternal));
    } else if (packed) {
      set_packed(a);
      LaunchCfg lc{stream, grid_for(*m, a), true};
      if (s->head_ev_begin) CK(cudaEventRecordWithFlags(static_cast<cudaEvent_t>(s->head_ev_begin), stream, cudaEventRecordExternal));
      prof_mark(s, stream);
      TRY(check_gemv(gemv_argmax(nt, a, p, lc), "lm head"));
      if (s->head_ev_end) CK(cudaEventRecordWithFlags(static_cast<cudaEvent_t>(s->head_ev_end), stream, cudaEventRecordExternal));
    } else if (nt == 16 && H % 64 == 0) {
      // 128 rows: the head is a GEMM for the tcgen05 tensor cores
      NormArgs na{s->x, m->final_norm, s->xnorm, 0, H, R, c.norm_eps, final_hidden, n_seq * 8, H};
      prof_mark(s, stream);
      TRY(check_gemv(launch_rmsnorm_rows(na, R, stream), "final norm"));
      HeadTcArgs ha;
      ha.wmap = m->head_map;
      ha.xmap = s->xhead_map;
      ha.V = c.vocab;
      ha.H = H;
      ha.n_seq = n_seq;
      ha.block_len = block_len;
      ha.drafts = drafts;
      ha.probs = s->draft_probs;
      ha.min_p = s->spec_min_p;
      ha.keys = s->head_keys;
      ha.ms = s->argmax_ms;
      ha.grid_cnt = p.grid_cnt;
      ha.status = status;
      const int nv = (c.vocab + 255) / 256;
      if (s->head_ev_begin) CK(cudaEventRecordWithFlags(static_cast<cudaEvent_t>(s->head_ev_begin), stream, cudaEventRecordExternal));
      prof_mark(s, stream);
      TRY(check_gemv(launch_head_tc(ha, nv < m->sm_count ? nv : m->sm_count, stream), "lm head"));
      if (s->head_ev_end) CK(cudaEventRecordWithFlags(static_cast<cudaEvent_t>(s->head_ev_end), stream, cudaEventRecordExternal));
    } else {
      // Up to 8 slots (64 rows) per head launch: a 128-row mma.sync tile would
      // spill the argmax epilogue's registers, so wider passes take launches of
      // 8 slots, each over its own rows (the head is streamed once per launch).
      const int halves = nt > 8 ? nt / 8 : 1;
      const int hnt = nt > 8 ? 8 : nt;
      const int hr = hnt * 8;
      const size_t half_elems = xchunk_elems(H, hr, 32 * Fmt<WT_HEAD>::CB, 2);
      for (int h = 0; h < halves; ++h) {
        const int rows_f32 = n_seq * 8 - h * hr;
        NormArgs na{s->x + static_cast<size_t>(h) * hr * H, m->final_norm,
                    static_cast<__nv_bfloat16*>(s->xnorm) + h * half_elems, 0, H, hr, c.norm_eps,
                    final_hidden ? final_hidden + static_cast<size_t>(h) * hr * H : nullptr,
                    rows_f32 < 0 ? 0 : (rows_f32 > hr ? hr : rows_f32), 32 * Fmt<WT_HEAD>::CB};
        prof_mark(s, stream);
        TRY(check_gemv(launch_rmsnorm_rows(na, hr, stream), "final norm"));
        GemvArgs ah = a;
        ah.n_valid_rows = hr;
        ah.X = static_cast<__nv_bfloat16*>(s->xnorm) + h * half_elems;
        ah.ldx = H;
        ArgmaxParams ph = p;
        ph.final_hidden = nullptr;
        ph.n_seq = n_seq - h * hnt > hnt ? hnt : n_seq - h * hnt;
        ph.block_len = block_len + h * hnt;
        ph.drafts = drafts + static_cast<size_t>(h) * hnt * (DFLASH_MAX_BLOCK - 1);
        ph.probs = s->draft_probs + static_cast<size_t>(h) * hnt * (DFLASH_MAX_BLOCK - 1);
        if (ph.n_seq <= 0) break;
        LaunchCfg lc{stream, grid_for(*m, ah), true};
        if (h == 0 && s->head_ev_begin)
          CK(cudaEventRecordWithFlags(static_cast<cudaEvent_t>(s->head_ev_begin), stream, cudaEventRecordExternal));
        prof_mark(s, stream);
        TRY(check_gemv(gemv_argmax(hnt, ah, ph, lc), "lm head"));
      }
      if (s->head_ev_end) CK(cudaEventRecordWithFlags(static_cast<cudaEvent_t>(s->head_ev_end), stream, cudaEventRecordExternal));
    }
  }
  if (carry) s->pend_n = 0;
  prof_mark(s, stream);
  return DFLASH_OK;
}

int dflash_accept(const int32_t* drafts, const int32_t* target_ids, const int32_t* block_len, int32_t n_seq,
                  int32_t max_block_len, int32_t* accept_len, int32_t* next_anchor, int32_t* anchor_pos_inout,
                  dflash_stream_t stream) {
  if (!drafts || !target_ids || !block_len || !accept_len || !next_anchor) return DFLASH_ERR_INVALID_ARG;
  if (n_seq < 1 || max_block_len < DFLASH_MIN_BLOCK || max_block_len > DFLASH_MAX_BLOCK)
    return DFLASH_ERR_INVALID_ARG;
  TRY(check_gemv(launch_accept(drafts, target_ids, block_len, n_seq, max_block_len, accept_len, next_anchor,
                               anchor_pos_inout, reinterpret_cast<cudaStream_t>(stream)),
                 "accept"));
  return DFLASH_OK;
}

int dflash_commit_positions(const int32_t* anchor_pos, const int32_t* accept_len, int32_t n_seq,
                            int32_t* positions, dflash_stream_t stream) {
  if (!anchor_pos || !accept_len || !positions || n_seq < 1) return DFLASH_ERR_INVALID_ARG;
  TRY(check_gemv(launch_commit_positions(anchor_pos, accept_len, n_seq, positions,
                                         reinterpret_cast<cudaStream_t>(stream)),
                 "commit positions"));
  return DFLASH_OK;
}

int dflash_state_read_kv(const dflash_state* s, int32_t slot, int32_t layer, int32_t pos0, int32_t n, float* k_out,
                         float* v_out, dflash_stream_t stream) {
  if (!s) return DFLASH_ERR_INVALID_ARG;
  const dflash_config& c = s->model->cfg;
  const bool ring = c.attn_window > 0;
  if (slot < 0 || slot >= s->n_slots || layer < 0 || layer >= c.n_layers || pos0 < 0 || n < 0 || n > s->capacity ||
      (!ring && static_cast<long long>(pos0) + n > s->capacity))
    return DFLASH_ERR_INVALID_ARG;
  const size_t off = static_cast<size_t>((layer * s->n_slots + slot) * c.n_kv_heads) * s->capacity * c.head_dim;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // cells of a deferred fusion are projected before they are read
  TRY(flush_deferred(static_cast<const dflash_model*>(s->model), const_cast<dflash_state*>(s), st));
  if (k_out)
    TRY(check_gemv(launch_kv_copy(false, s->K + off, s->capacity, ring, c.head_dim, c.n_kv_heads, pos0, n, k_out, nullptr, st),
                   "read k"));
  if (v_out)
    TRY(check_gemv(launch_kv_copy(false, s->V + off, s->capacity, ring, c.head_dim, c.n_kv_heads, pos0, n, v_out, nullptr, st),
                   "read v"));
  return DFLASH_OK;
}

int dflash_state_write_kv(dflash_state* s, int32_t slot, int32_t layer, int32_t pos0, int32_t n, const uint16_t* k_in,
                          const uint16_t* v_in, dflash_stream_t stream) {
  if (!s) return DFLASH_ERR_INVALID_ARG;
  const dflash_config& c = s->model->cfg;
  const bool ring = c.attn_window > 0;
  if (slot < 0 || slot >= s->n_slots || layer < 0 || layer >= c.n_layers || pos0 < 0 || n < 0 || n > s->capacity ||
      (!ring && static_cast<long long>(pos0) + n > s->capacity))
    return DFLASH_ERR_INVALID_ARG;
  const size_t off = static_cast<size_t>((layer * s->n_slots + slot) * c.n_kv_heads) * s->capacity * c.head_dim;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // a deferred fusion's cells are written first, so later writes win as in call order
  TRY(flush_deferred(static_cast<const dflash_model*>(s->model), s, st));
  if (k_in)
    TRY(check_gemv(launch_kv_copy(true, s->K + off, s->capacity, ring, c.head_dim, c.n_kv_heads, pos0, n, nullptr, k_in, st),
                   "write k"));
  if (v_in)
    TRY(check_gemv(launch_kv_copy(true, s->V + off, s->capacity, ring, c.head_dim, c.n_kv_heads, pos0, n, nullptr, v_in, st),
                   "write v"));
  return DFLASH_OK;
}

int dflash_state_status(dflash_state* s, int32_t* status_out, dflash_stream_t stream) {
  if (!s || !status_out) return DFLASH_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  CK(cudaMemcpyAsync(status_out, s->status, 4, cudaMemcpyDeviceToHost, st));
  CK(cudaMemsetAsync(s->status, 0, 4, st));
  CK(cudaStreamSynchronize(st));
  return DFLASH_OK;
}

int dflash_model_dequantize(const dflash_model* m, int32_t which, float* out, dflash_stream_t stream) {
  if (!m || !out) return DFLASH_ERR_INVALID_ARG;
  const dflash_config& c = m->cfg;
  const int L = c.n_layers, H = c.hidden, d = c.head_dim, nq = c.n_q_heads, nkv = c.n_kv_heads, I = c.intermediate;
  if (which < 0 || which > 7 * L) return DFLASH_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const PackedMatrix* pm;
  int row_off = 0, rows = 0, inter = -1;
  if (which == 0) {
    pm = &m->fc;
    rows = H;
  } else {
    const int l = (which - 1) / 7, k = (which - 1) % 7;
    switch (k) {
      case 0: pm = &m->qkv[l]; rows = nq * d; break;
      case 1: pm = &m->qkv[l]; rows = nkv * d; row_off = nq * d; break;
      case 2: pm = &m->qkv[l]; rows = nkv * d; row_off = (nq + nkv) * d; break;
      case 3: pm = &m->o[l]; rows = H; break;
      case 4: pm = &m->gu[l]; rows = I; inter = 0; break;
      case 5: pm = &m->gu[l]; rows = I; inter = 1; break;
      default: pm = &m->down[l]; rows = H; break;
    }
  }
  TRY(check_gemv(launch_dequant(pm->wtype, pm->data, pm->n, pm->k, out, row_off, rows, inter, st), "dequant"));
  return DFLASH_OK;
}

int32_t dflash_draft_launches(const dflash_state* s, int32_t n_seq) {
  if (!s || n_seq < 1 || n_seq > s->n_slots) return -1;
  const int L = s->model->cfg.n_layers;
  const int nt = pow2ceil(n_seq);
  const bool streamed = !fused_norm(nt);  // separate RMSNorm kernels
  const int per_layer = 5 + (attn_pass_chunks(*s->model, *s, n_seq) > n_seq ? 1 : 0) + (streamed ? 2 : 0) +
                        (nt == 16 && s->tc_maps ? 1 : 0);  // the per-head step after a tcgen05 QKV GEMM
  const int head_launches = (nt > 8 && !(nt == 16 && s->model->cfg.hidden % 64 == 0)) ? (n_seq + 7) / 8 : 1;
  return 1 + L * per_layer + head_launches * (streamed ? 2 : 1);
}

int32_t dflash_fuse_launches(const dflash_state* s, int32_t n) {
  if (!s || n < 0) return -1;
  int k = 0;
  for (int base = 0; base < n; base += s->fuse_rows) {
    const int rows = (n - base) < s->fuse_rows ? (n - base) : s->fuse_rows;
    k += fused_norm(rows <= 8 ? 1 : 16) ? ((s->defer_kv && n <= 8) ? 1 : 2) : 3;
  }
  return k;
}

int dflash_state_set_attn_chunks(dflash_state* s, int32_t chunks, int32_t* max_chunks) {
  if (!s) return DFLASH_ERR_INVALID_ARG;
  if (max_chunks) *max_chunks = s->attn_chunks_max;
  if (chunks == 0) return DFLASH_OK;
  if (chunks < 1 || chunks > s->attn_chunks_max) return DFLASH_ERR_INVALID_ARG;
  s->attn_chunks = chunks;
  s->attn_chunks_set = 1;
  return DFLASH_OK;
}

int dflash_state_set_defer_kv(dflash_state* s, int32_t on) {
  if (!s || (on != 0 && on != 1)) return DFLASH_ERR_INVALID_ARG;
  if (!on && s->pend_n > 0) return DFLASH_ERR_INVALID_ARG;  // dflash_state_flush first
  s->defer_kv = on;
  return DFLASH_OK;
}

int dflash_state_flush(dflash_state* s, dflash_stream_t stream) {
  if (!s) return DFLASH_ERR_INVALID_ARG;
  return flush_deferred(static_cast<const dflash_model*>(s->model), s, reinterpret_cast<cudaStream_t>(stream));
}

int dflash_state_set_spec_min_p(dflash_state* s, float floor) {
  if (!s || !(floor >= 0.f && floor <= 1.f)) return DFLASH_ERR_INVALID_ARG;
  s->spec_min_p = floor;
  return DFLASH_OK;
}

int dflash_state_read_draft_probs(const dflash_state* s, float* out, dflash_stream_t stream) {
  if (!s || !out) return DFLASH_ERR_INVALID_ARG;
  CK(cudaMemcpyAsync(out, s->draft_probs, size_t(s->n_slots) * (DFLASH_MAX_BLOCK - 1) * 4, cudaMemcpyDeviceToDevice,
                     reinterpret_cast<cudaStream_t>(stream)));
  return DFLASH_OK;
}

int dflash_state_set_profile_events(dflash_state* s, void* const* events, int32_t n_events) {
  if (!s || n_events < 0 || n_events > 256 || (n_events > 0 && !events)) return DFLASH_ERR_INVALID_ARG;
  for (int i = 0; i < n_events; ++i) s->prof_events[i] = events[i];
  s->prof_n = n_events;
  s->prof_k = 0;
  return DFLASH_OK;
}

int dflash_state_set_head_events(dflash_state* s, void* ev_begin, void* ev_end) {
  if (!s || (ev_begin == nullptr) != (ev_end == nullptr)) return DFLASH_ERR_INVALID_ARG;
  s->head_ev_begin = ev_begin;
  s->head_ev_end = ev_end;
  return DFLASH_OK;
}

#ifdef DFLASH_TRACE
// Diagnostic builds only: per-CTA timestamps of the next GEMV launches.
int dflash_state_set_trace(dflash_state* s, unsigned long long* buf, int32_t max_launches) {
  if (!s) return DFLASH_ERR_INVALID_ARG;
  s->trace = buf;
  s->trace_launches = buf ? max_launches : 0;
  s->trace_k = 0;
  return DFLASH_OK;
}
#endif

}  // extern "C"

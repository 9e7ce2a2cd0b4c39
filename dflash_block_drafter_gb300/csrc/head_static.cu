// dflash_head_argmax_static: greedy ids over the target's LM head for up to
// 8 rows of final hidden states, for callers that cannot allocate device
// memory -- code that runs while a CUDA graph is being captured (where
// cudaMalloc is not allowed), engines whose device memory is one arena
// reserved up front and owned by someone else, or real-time loops that must
// never enter the allocator.  Such callers cannot create a dflash_state (which
// allocates its workspace), so this entry point keeps its scratch in a fixed
// array inside the library instead.
//
// The work is the LM-head GEMV + argmax kernel of the draft pass (the same
// kernel template, streaming the borrowed row-major BF16 head through 2-D
// tensor-map copies), instantiated with an epilogue that writes one id per
// input row.  Its scratch -- the hidden rows rounded to BF16, the split-group
// partial sums and their counters, and the per-CTA argmax keys -- lives in
// g_head_scratch below: a file-scope __device__ array of kStaticScratchBytes
// (about 1.35 MB) that every GPU that loads the library holds until exit.
//
// Host code never uses the symbol itself as an address (in host code it is
// only a stand-in): on the first call on each device, with that device
// current, the address is looked up with cudaGetSymbolAddress and cached.
// That first call therefore must not happen while a stream is being captured.
//
// Every call shares the one array: calls that overlap on the GPU (on
// different streams, or from several host threads without ordering) race and
// give wrong ids.  The counters that must start at zero are cleared by each
// call (an asynchronous memset on the call's stream); the rest is fully
// rewritten by each call before it is read.
#include <cstring>
#include <mutex>

#include "gemv_launch.cuh"

namespace dflash {
namespace {

constexpr int kStaticMaxRows = 8;        // one 8-row MMA tile
constexpr int kStaticMaxHidden = 8192;   // hidden size H
constexpr int kStaticMaxVocab = 262144;  // vocabulary V
constexpr int kStaticMaxGrid = 256;      // CTAs of the GEMV

// byte offsets of the scratch regions
constexpr size_t kOffCounters = 0;                                              // int[V/64 + 1]
constexpr size_t kCountersBytes = (kStaticMaxVocab / 64 + 1) * 4;
constexpr size_t kOffGridCnt = ((kOffCounters + kCountersBytes + 255) / 256) * 256;  // int
constexpr size_t kOffSlots = kOffGridCnt + 256;                                 // u64[grid][8]
constexpr size_t kOffPartials = kOffSlots + size_t(kStaticMaxGrid) * kStaticMaxRows * 8;  // f32[grid][2][64][8]
constexpr size_t kOffX = kOffPartials + size_t(kStaticMaxGrid) * 2 * 64 * kStaticMaxRows * 4;  // bf16[8][H]
// the rows in the head GEMV's chunked X layout: 8 rows, 128-input units, BF16 hi + lo planes
constexpr size_t kStaticScratchBytes = kOffX + size_t(kStaticMaxHidden / 128) * 2 * kStaticMaxRows * (128 + 32) * 2;

static __device__ __align__(256) uint8_t g_head_scratch[kStaticScratchBytes];

// Device address of g_head_scratch, looked up once per device.
constexpr int kMaxDevices = 64;
uint8_t* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mutex;

cudaError_t scratch_for_current_device(uint8_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_head_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = static_cast<uint8_t*>(p);
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

// Rows -> the head GEMV's streamed X: BF16 hi = bf16(v) and lo = bf16(v - hi)
// planes in the chunked layout of 8 rows and 128-input units; rows n..7 are
// zero.
__global__ void __launch_bounds__(256) rows_to_bf16_kernel(const float* __restrict__ in, int n, int H,
                                                           __nv_bfloat16* __restrict__ out) {
  pdl_wait();
  pdl_launch_dependents();
  const int total = kStaticMaxRows * H;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
    const int r = i / H, k = i - r * H;
    const float v = r < n ? in[i] : 0.f;
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    out[xchunk_index(k, r, 0, kStaticMaxRows, 128, 2)] = hi;
    out[xchunk_index(k, r, 1, kStaticMaxRows, 128, 2)] = __float2bfloat16_rn(v - __bfloat162float(hi));
  }
}

// The draft pass's argmax epilogue, finishing with one id per input row.
struct EpiArgmaxRows : public EpiArgmax<1> {
  int n_rows;
  int32_t* ids;

  template <int NT>
  __device__ void finish(const GemvArgs&, Local& L, int w, int lane, int tid, unsigned long long* sstage,
                         int* sflag) const {
    constexpr int R = 8;
    const bool any_bad = __any_sync(0xffffffffu, L.bad);
    if (any_bad && lane == 0) set_status(status, DFLASH_DEV_NONFINITE);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      unsigned long long k = pack(L.v[0][h], L.id[0][h]);
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        const unsigned long long k2 = __shfl_xor_sync(0xffffffffu, k, o);
        k = k2 > k ? k2 : k;
      }
      if (lane < 4) sstage[w * R + lane * 2 + h] = k;
    }
    named_bar_sync(1, 128);
    if (tid < R) {
      unsigned long long k = sstage[tid];
      for (int ww = 1; ww < 4; ++ww) {
        const unsigned long long k2 = sstage[ww * R + tid];
        k = k2 > k ? k2 : k;
      }
      __stcg(slots + static_cast<size_t>(blockIdx.x) * R + tid, k);
    }
    named_bar_sync(1, 128);
    if (tid == 0) {
      const int old = atomic_add_acq_rel(grid_cnt, 1);
      sflag[2] = (old == static_cast<int>(gridDim.x) - 1);
    }
    named_bar_sync(1, 128);
    if (!sflag[2]) return;
    const unsigned long long k = grid_max<R>(tid, w, lane, sstage);
    if (tid < n_rows) {
      int out = -1;
      if (k == 0ull) set_status(status, DFLASH_DEV_NONFINITE);
      else out = static_cast<int>(0xffffffffu - static_cast<uint32_t>(k & 0xffffffffull));
      ids[tid] = out;
    }
    if (tid == 0) *grid_cnt = 0;
  }
};

}  // namespace
}  // namespace dflash

using namespace dflash;

extern "C" int dflash_head_argmax_static(const dflash_model* m, const float* hidden, int32_t n_rows, int32_t* ids,
                                         int32_t* dev_status, dflash_stream_t stream_) {
  if (!m || !hidden || !ids) return DFLASH_ERR_INVALID_ARG;
  if (n_rows < 1) return DFLASH_ERR_INVALID_ARG;
  const dflash_config& c = m->cfg;
  // sizes beyond the fixed scratch array are refused, never truncated
  if (n_rows > kStaticMaxRows || c.hidden > kStaticMaxHidden || c.vocab > kStaticMaxVocab)
    return DFLASH_ERR_CAPACITY;
  // the model's tensors (and the scratch array used below) belong to the
  // device that was current at model creation: it must be current now
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return DFLASH_ERR_CUDA;
  if (dev != m->device) return DFLASH_ERR_INVALID_ARG;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  uint8_t* scratch = nullptr;
  if (scratch_for_current_device(&scratch) != cudaSuccess) return DFLASH_ERR_CUDA;

  GemvArgs a;
  memset(&a, 0, sizeof(a));
  a.wmap = m->head_map;
  a.N = ((c.vocab + 63) / 64) * 64;
  a.K = c.hidden;
  a.UPG = c.hidden / 128;
  a.U = (a.N / 64) * a.UPG;
  a.n_valid_rows = kStaticMaxRows;  // rows n_rows..7 of the staged X are zero
  a.X = scratch + kOffX;
  a.ldx = c.hidden;
  a.partials = reinterpret_cast<float*>(scratch + kOffPartials);
  a.counters = reinterpret_cast<int*>(scratch + kOffCounters);
  a.status = dev_status;
  int grid = m->sm_count < a.U ? m->sm_count : a.U;
  if (grid > kStaticMaxGrid) grid = kStaticMaxGrid;
  if (grid < 1) grid = 1;

  EpiArgmaxRows e;
  memset(&e, 0, sizeof(e));
  e.vocab = c.vocab;
  e.n_seq = 1;
  e.H = c.hidden;
  e.slots = reinterpret_cast<unsigned long long*>(scratch + kOffSlots);
  e.grid_cnt = reinterpret_cast<int*>(scratch + kOffGridCnt);
  e.status = dev_status;
  e.n_rows = n_rows;
  e.ids = ids;

  // zero what the kernel counts on: the split-group counters and the grid counter
  if (cudaMemsetAsync(scratch + kOffCounters, 0, kOffSlots - kOffCounters, stream) != cudaSuccess)
    return DFLASH_ERR_CUDA;
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((kStaticMaxRows * c.hidden + 255) / 256);
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, rows_to_bf16_kernel, hidden, static_cast<int>(n_rows), static_cast<int>(c.hidden),
                           reinterpret_cast<__nv_bfloat16*>(scratch + kOffX)) != cudaSuccess)
      return DFLASH_ERR_CUDA;
  }
  LaunchCfg lc{stream, grid, true};
  if (launch_gemv<WT_HEAD, 1, X_STREAM>(a, e, lc) != cudaSuccess) return DFLASH_ERR_CUDA;
  return DFLASH_OK;
}

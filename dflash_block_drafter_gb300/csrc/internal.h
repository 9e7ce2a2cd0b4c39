// Internal structures of libdflash shared by the C-ABI implementation and
// the kernel translation units.  Not part of the public interface.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dflash.h"

namespace dflash {

// Weight storage formats inside the library.  The four backbone types are
// repacked at model creation into a "fragment-native" streaming layout (see
// layout.cuh); the borrowed LM head stays row-major BF16 and is read through
// a 2-D tensor map.
enum WType : int { WT_BF16 = 0, WT_Q8_0 = 1, WT_Q5_0 = 2, WT_Q4_0 = 3, WT_HEAD = 4 };

// How a GEMV kernel obtains its activation rows X.
enum XMode : int {
  X_STREAM = 1,    // X chunks copied from global memory with each weight unit
  X_STREAM_BF16 = 2,  // as X_STREAM, but X is BF16 whatever the weight type (the caller's taps)
  X_NORM = 3          // as X_STREAM with two BF16 planes of x * w written by the kernel that
                      // produced x, plus its per-64-column sums of squares; the outputs are
                      // scaled by 1 / RMS of their row (RMSNorm-fed GEMVs)
};

// One repacked backbone matrix (library-owned, device memory).
struct PackedMatrix {
  uint8_t* data = nullptr;
  int wtype = 0;
  int n = 0;  // output rows (multiple of 64)
  int k = 0;  // input columns (multiple of 256)
  size_t bytes = 0;
};

struct Model {
  dflash_config cfg{};
  int wtype = 0;
  int sm_count = 0;
  int device = 0;
  // backbone matrices, repacked
  PackedMatrix fc;                          // [H, n_taps*H]
  PackedMatrix kv_all;                      // [L * 2 * n_kv*d, H]: per layer W_k then W_v (fusion)
  PackedMatrix qkv[DFLASH_MAX_LAYERS];      // [(n_q + 2 n_kv) d, H]
  PackedMatrix o[DFLASH_MAX_LAYERS];        // [H, n_q d]
  PackedMatrix gu[DFLASH_MAX_LAYERS];       // [2 I, H], gate/up rows interleaved in groups of 8
  PackedMatrix down[DFLASH_MAX_LAYERS];     // [H, I]
  // float copies of the norm weights
  float* hidden_norm = nullptr;             // [H]
  float* attn_norm = nullptr;               // [L, H]
  float* q_norm = nullptr;                  // [L, d]
  float* k_norm = nullptr;                  // [L, d]
  float* mlp_norm = nullptr;                // [L, H]
  float* final_norm = nullptr;              // [H]
  uint64_t* rope_turns = nullptr;           // [d/2] inv_freq_i / (2 pi) as 0.64 fixed point
  // borrowed target tensors
  const uint16_t* embed = nullptr;          // [V, H] BF16
  const uint16_t* head = nullptr;           // [V, H] BF16
  CUtensorMap head_map;         // 64-row x 64-col boxes, 128-byte swizzle
  size_t device_bytes = 0;
};

// Per-GEMV-kind counter regions inside a state's counter array.
enum CounterRegion : int {
  CNT_QKV = 0, CNT_O, CNT_GU, CNT_DOWN, CNT_HEAD, CNT_FC, CNT_KV, CNT_QKV_HEADS, CNT_KV_HEADS,
  CNT_ARGMAX, CNT_REGIONS
};

struct State {
  const Model* model = nullptr;
  int n_slots = 0;
  int capacity = 0;
  int rows = 0;            // R = 8 * NT activation rows of a pass
  int nt = 0;              // n8 tiles of a pass (power of two >= n_slots)
  int attn_chunks = 0;     // context chunks per (slot, kv head)
  int attn_chunks_max = 0; // chunks the partial buffers are sized for
  int attn_chunks_set = 0; // the caller chose attn_chunks (dflash_state_set_attn_chunks)
  // per-layer FP16 K/V arenas: [L][slot][n_kv][capacity][d]
  __half* K = nullptr;
  __half* V = nullptr;
  // pass workspace
  float* x = nullptr;          // [R, H] residual stream
  float* qkv_raw = nullptr;    // [R, (n_q + 2 n_kv) d]
  __half* q_ready = nullptr;   // [slots, n_kv, M = 8 n_q / n_kv, d] normed, rotated, pre-scaled queries
  void* attn_out = nullptr;    // [R, n_q d] activation type
  void* hbuf = nullptr;        // [R, I] activation type (SwiGLU output)
  void* xnorm = nullptr;       // [R, H] activation type (normed rows for streamed-X GEMVs)
  __nv_bfloat16* xn = nullptr;  // 8-row passes: BF16 hi/lo planes of x * w (chunked) for the next RMSNorm-fed GEMV
  float* ssq = nullptr;         // [H / 64, 8] partial sums of squares of x
  __half* attn_part = nullptr;  // [slots, n_kv, C, Gq*8, d] chunk partials O / l
  float2* attn_ml = nullptr;   // [slots, n_kv, C, Gq*8] (max in log2 units, sum)
  int* attn_plan = nullptr;    // [32] the attention chunk plan of the last multi-sequence pass
  float* partials = nullptr;   // GEMV split fix-up slots [max_grid, 2, 64, R_max]
  int* counters = nullptr;     // [CNT_REGIONS][counter_stride]
  int counter_stride = 0;
  unsigned long long* argmax_slots = nullptr;  // [max_grid, R]
  float2* argmax_ms = nullptr;  // [max_grid, R]: per-CTA (max logit, sum of exp) of the LM head
  float* draft_probs = nullptr; // [n_slots, 7]: softmax probability of each draft of the last pass
  float spec_min_p = 0.f;       // confidence floor of the drafts (0: every draft offered)
  int* nonfinite = nullptr;    // [1] scratch flag
  // fusion workspace (tiles of up to fuse_rows positions)
  int fuse_rows = 0;
  float* h_raw = nullptr;      // [fuse_rows, H]
  float* kv_raw = nullptr;     // [fuse_rows, L * 2 * n_kv * d]
  void* fuse_xnorm = nullptr;  // [fuse_rows, H] activation type
  // deferred K/V projection of an 8-row fusion (dflash_state_set_defer_kv):
  // the committed rows' x * hidden_norm (chunked, like xn) and sums of
  // squares, kept until the next draft pass projects them in its QKV GEMVs
  int defer_kv = 0;
  __nv_bfloat16* fuse_xn = nullptr;
  float* fuse_ssq = nullptr;
  int pend_n = 0;                     // rows waiting (0: none)
  int pend_slot = 0;
  const int32_t* pend_pos = nullptr;  // the caller's positions array of that fusion
  int32_t* pend_status = nullptr;
  int32_t* status = nullptr;   // [1] the state's own device status word
  int max_grid = 0;
  void* prof_events[256] = {};     // optional per-kernel event marks
  int prof_n = 0;
  int prof_k = 0;
  unsigned long long* trace = nullptr;  // diagnostic builds: [launch][max_grid][8] timestamps
  int trace_launches = 0;
  int trace_k = 0;
  void* head_ev_begin = nullptr;  // optional cudaEvent_t pair around the LM head
  void* head_ev_end = nullptr;
  CUtensorMap q_map;     // q_ready as [slots*n_kv*M, d], 64 x M boxes, 128-byte swizzle
  CUtensorMap part_map;  // attn_part as [slots*n_kv*C_max*M, d], 64 x M boxes, 128-byte swizzle
  CUtensorMap k_map;  // K arena as [L*slots*n_kv*cap, d], 64x64 boxes, 128-byte swizzle
  CUtensorMap v_map;
  // 128-row passes: xnorm as [2 * 128, H + 32] BF16 rows for the tcgen05 LM head, and its keys
  CUtensorMap xhead_map;
  CUtensorMap xn_map;  // one-sequence passes: xn as [H / 128 * 16, 160] BF16 rows for the tcgen05 LM head
  unsigned long long* head_keys8 = nullptr;  // [8], zero between passes
  CUtensorMap tc_xnorm_map, tc_attn_map, tc_hbuf_map;  // 128-row passes: the layer GEMMs' activations
  int tc_maps = 0;
  unsigned long long* head_keys = nullptr;  // [128], zero between passes
  size_t device_bytes = 0;
};

}  // namespace dflash

// The opaque handles of the C ABI (include/dflash.h) are the library's model
// and state; defined once here for every translation unit that uses them.
struct dflash_model : public dflash::Model {};
struct dflash_state : public dflash::State {};

// Argument structs and host launchers of the small kernels (misc.cu,
// attention.cu), shared with the C-ABI implementation.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"

namespace dflash {

struct EmbedArgs {
  const uint16_t* embed;
  const int32_t* anchor_tok;
  const int32_t* anchor_pos;
  const int32_t* block_len;
  float* x;
  int H, vocab, mask_id, n_seq, cap;
  int ring;  // cells form a ring (attention window): any position >= 0 fits
  int32_t* status;
  // optional (one slot): the first QKV GEMV's input, as PackNext writes it
  // (x * w_next in the chunked layout of 8 rows and ku inputs per unit: one
  // FP16 plane when f16, else BF16 hi/lo planes; per-64-column sums of
  // squares)
  void* xn;
  float* ssq;
  const float* w_next;
  int ku;
  int f16;
};

// out = RMSNorm(x) * w in the chunked streamed-X layout (layout.cuh) of a
// GEMV with R = gridDim.x rows: FP16 (out_f16) or BF16 hi and lo planes.
struct NormArgs {
  const float* x;
  const float* w;
  void* out;
  int out_f16;
  int H, rows_valid;
  float eps;
  float* f32_out;  // optional fp32 copy of rows [0, rows_f32)
  int rows_f32;
  int ku;           // chunked layout of the consuming GEMV: inputs per unit
};

// LM head + argmax of a 128-row pass on the tcgen05 tensor cores (head_tc.cu)
struct HeadTcArgs {
  CUtensorMap wmap;  // the head [V, H] BF16: 64 x 64 boxes, 128-byte swizzle
  CUtensorMap xmap;  // the final normed rows as [2 * 128, H + 32] BF16 (hi rows, then lo rows):
                     // 64 x 128 boxes, 128-byte swizzle
  int V, H, n_seq;
  const int32_t* block_len;
  int32_t* drafts;   // [n_seq, 7]
  float* probs;      // [n_seq, 7] or null
  float min_p;       // confidence floor (0: none, confidences -1)
  unsigned long long* keys;  // [128] packed (logit, id) keys, zero between launches
  float2* ms;        // [grid, 128] per-CTA (max logit, sum of exp) when min_p > 0
  int* grid_cnt;     // zero between launches
  int32_t* status;
  // 8-row passes (launch_head_tc8): xmap maps the packed rows x * w_final (the
  // chunked layout of 8 rows and 128 inputs per unit, BF16 hi then lo plane)
  // as [H / 128 * 16 rows, 160] with 64 x 16 boxes; outputs are divided by
  // each row's RMS from ssq [H / 64][8]; optional final_hidden [8, H] =
  // x * (1 / RMS) * norm_w
  const float* ssq;
  float eps;
  float* final_hidden;
  const float* x;
  const float* norm_w;
};
cudaError_t launch_head_tc(const HeadTcArgs& a, int grid, cudaStream_t stream);
cudaError_t launch_head_tc8(const HeadTcArgs& a, int grid, cudaStream_t stream);

cudaError_t launch_repack(int wtype, const void* src, int rows, int K, uint8_t* dst, int row_off, int interleave,
                          cudaStream_t st);
cudaError_t launch_dequant(int wtype, const uint8_t* packed, int N, int K, float* out, int row_off, int rows_out,
                           int interleave, cudaStream_t st);
cudaError_t launch_embed(const EmbedArgs& a, int nt, cudaStream_t st);
cudaError_t launch_rmsnorm_rows(const NormArgs& a, int rows, cudaStream_t st);
cudaError_t launch_accept(const int32_t* drafts, const int32_t* tgt, const int32_t* block_len, int n_seq, int maxB,
                          int32_t* accept_len, int32_t* next_anchor, int32_t* anchor_pos, cudaStream_t st);
cudaError_t launch_commit_positions(const int32_t* anchor_pos, const int32_t* accept_len, int n_seq, int32_t* out,
                                    cudaStream_t st);
cudaError_t launch_kv_copy(bool write, __half* cells, int cap, bool ring, int d, int n_kv, int pos0, int n, float* out,
                           const uint16_t* in, cudaStream_t st);
int attn_pass_chunks(const Model& m, const State& st, int n_seq);
cudaError_t launch_attention(const Model& m, State& st, int layer, int n_seq, int pass_nt, const int32_t* anchor_pos,
                             const int32_t* block_len, int32_t* status, cudaStream_t stream);
// Dynamic shared memory of the attention kernel for head dim D and M query rows.
int attn_smem_bytes(int D, int M);
// Diagnostic builds: the next per-CTA timestamp slot of a launch (else null).
unsigned long long* trace_slot(State& st);

}  // namespace dflash

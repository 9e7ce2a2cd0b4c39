/*
 * dflash.h -- C ABI of libdflash, a GB300 (sm_103a) implementation of the
 * DFlash block-draft pass of a speculative-decoding LLM engine.
 *
 * The pass has five steps, all executed by hand-written CUDA kernels of this
 * library:
 *   (1) feature fusion: h = rmsnorm(fc(concat(target taps))) for newly
 *       committed positions, projected into each draft layer's own FP16
 *       context K/V state and written by position     -> dflash_fuse_context
 *   (2)-(4) the draft pass over the block [anchor at p, mask tokens at p+1..]:
 *       five dense layers (NeoX RoPE, non-causal GQA block attention, SwiGLU
 *       MLP over BF16 / Q8_0 / Q5_0 / Q4_0 weights), final norm, the target's
 *       LM head and a per-row argmax                    -> dflash_draft_block
 *   (5) greedy acceptance of the candidates against the verifier's argmax
 *       ids                                             -> dflash_accept
 *
 * Sources (page title, section):
 *   "#1426 dflash: experimental standalone DeepSpec DFlash block drafter for
 *    Qwen3.8-Flash-Next (greedy, correctness-first)" -- sections "Drafter
 *    runtime", "Owned DFlash K/V state", "Target feature taps", "Speculative
 *    decode integration", "DFlash artifact", "Current limitations".
 *   "#3322 [Engine] support the official Flash-Next DFlash2 checkpoint" --
 *    section "Approach" (Q8_0 / Q5_0 / Q4_0 backbone quantisation of the 36
 *    backbone matrices, norms kept BF16, shared target output head).
 *   "#366 [RFC] EXPERIMENTAL Investigate DFlash2 support" -- section
 *    "Verification and state management" (full / partial / first-candidate
 *    rejection; commit accepted tokens plus the verifier's continuation).
 *
 * Conventions (apply to every entry point):
 *   - Every function returns an int status (dflash_status).  Arguments are
 *     validated synchronously on the host before anything is enqueued; on a
 *     non-zero return nothing was enqueued.
 *   - Tensor arguments are DEVICE pointers owned by the caller, unless a
 *     comment says otherwise.  Work is enqueued on the caller's cudaStream_t
 *     (0 = legacy default stream) and is asynchronous; kernels read dynamic
 *     scalars (positions, block lengths, token ids) from device memory, so a
 *     captured CUDA graph of a call stays valid as those values change.
 *   - Errors that only the device can see (non-finite values, token ids out
 *     of range, positions beyond the state's capacity, a pipeline wait that
 *     timed out) are OR-ed as DFLASH_DEV_* bits into a device status word
 *     that the caller reads after synchronising.  Kernels never trap; on such
 *     an error they skip the offending access and the outputs of that call
 *     are unspecified.
 *   - No call allocates device memory except dflash_model_create and
 *     dflash_state_create.
 *   - Calls that share a dflash_state must not overlap in time (the state
 *     owns the pass's workspace).  Different states may run concurrently on
 *     different streams against one dflash_model, which is read-only after
 *     creation.
 */
#ifndef DFLASH_H_
#define DFLASH_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t without including the CUDA headers. */
typedef struct CUstream_st* dflash_stream_t;

/* ---------------------------------------------------------------- status */
enum dflash_status {
  DFLASH_OK = 0,
  DFLASH_ERR_INVALID_ARG = 1,  /* null pointer, size out of range, bad slot */
  DFLASH_ERR_UNSUPPORTED = 2,  /* geometry or weight type this build cannot run */
  DFLASH_ERR_CAPACITY = 3,     /* request does not fit the state */
  DFLASH_ERR_CUDA = 4,         /* a CUDA runtime call failed (see dflash_last_cuda_error) */
  DFLASH_ERR_NO_DEVICE = 5,    /* no usable sm_100+ GPU */
  DFLASH_ERR_OUT_OF_MEMORY = 6
};

/* Device-detected error bits, OR-ed into the caller's status word. */
enum dflash_device_error {
  DFLASH_DEV_NONFINITE = 1,   /* a logit or hidden value was NaN/Inf ("non-finite refusal") */
  DFLASH_DEV_BAD_TOKEN = 2,   /* anchor token id outside [0, vocab) */
  DFLASH_DEV_CAPACITY = 4,    /* p + block_len > capacity, or a fuse position >= capacity (negative
                                 fuse positions are skipped rows; ring states accept any p >= 0) */
  DFLASH_DEV_BAD_BLOCK = 8,   /* a block_len outside [2, 8] (clamped) */
  DFLASH_DEV_TIMEOUT = 16     /* a pipeline wait exceeded its time limit (should never happen) */
};

/* Backbone weight storage types ("#3322 ...", "Approach"). */
enum dflash_weight_type {
  DFLASH_WT_BF16 = 0,
  DFLASH_WT_Q8_0 = 1,  /* 34-byte blocks: f16 d, int8 q[32];            w = d*q        */
  DFLASH_WT_Q5_0 = 2,  /* 22-byte blocks: f16 d, u32 qh, u8 qs[16];     w = d*(q - 16) */
  DFLASH_WT_Q4_0 = 3   /* 18-byte blocks: f16 d, u8 qs[16];             w = d*(q - 8)  */
};
/* GGUF-style block layout (little endian): d is IEEE half; for Q4_0/Q5_0
 * element j (< 16) is the low nibble of qs[j] and element j + 16 its high
 * nibble; for Q5_0 bit j of qh is the fifth (most significant) bit of element
 * j.  Blocks of 32 weights run along the input dimension inside each output
 * row; rows are consecutive. */

#define DFLASH_MAX_LAYERS 8
#define DFLASH_MAX_BLOCK 8   /* "--spec 2..8" ("#1426 ...", "DFlash artifact") */
#define DFLASH_MIN_BLOCK 2
#define DFLASH_MAX_SLOTS 16  /* sequences drafted together in one call */

/* ---------------------------------------------------------------- model */
typedef struct dflash_config {
  int32_t n_layers;      /* 5 for DFlash                              */
  int32_t hidden;        /* H = 2560                                   */
  int32_t n_q_heads;     /* 24                                         */
  int32_t n_kv_heads;    /* 2  (q head h reads kv head h / (n_q/n_kv)) */
  int32_t head_dim;      /* d = 256; softmax scale 1/sqrt(d)           */
  int32_t intermediate;  /* I = 7680 (SwiGLU)                          */
  int32_t vocab;         /* V of the target's embedding / LM head      */
  int32_t n_taps;        /* 5 target feature taps of width H           */
  float rope_theta;      /* 1e7, full-head NeoX RoPE                   */
  float norm_eps;        /* RMSNorm epsilon (1e-6)                     */
  int32_t mask_token_id; /* token of the block's mask rows             */
  int32_t weight_type;   /* dflash_weight_type of the 36 backbone matrices */
  int32_t attn_window;   /* 0: a block at p attends over positions [0, p + B)
                          * and position pos lives in cell pos (< capacity).
                          * W > 0: drafter attention window ("#1426 ...",
                          * "Additional constraints": 32768 cells by default
                          * there): the block attends over positions
                          * [max(0, p + B - W), p + B), and the state's cells
                          * form a ring, position pos living in cell
                          * pos mod capacity (capacity >= W, a multiple of
                          * 128), so positions may grow without bound.    */
} dflash_config;

/* Per-layer tensors; names follow the pages' stage names.  Matrices are
 * [out, in] row-major (out rows of `in` weights): BF16 (uint16 bits) when
 * weight_type == DFLASH_WT_BF16, else GGUF-style blocks.  Norm weights are
 * BF16 vectors. */
typedef struct dflash_layer_weights {
  const void* attn_norm;  /* [H]                 */
  const void* wq;         /* [n_q*d, H]          */
  const void* wk;         /* [n_kv*d, H]         */
  const void* wv;         /* [n_kv*d, H]         */
  const void* q_norm;     /* [d] per-head RMSNorm */
  const void* k_norm;     /* [d]                 */
  const void* wo;         /* [H, n_q*d]          */
  const void* mlp_norm;   /* [H]                 */
  const void* w_gate;     /* [I, H]              */
  const void* w_up;       /* [I, H]              */
  const void* w_down;     /* [H, I]              */
} dflash_layer_weights;

typedef struct dflash_weights {
  const void* fc;           /* [H, n_taps*H]  fusion projection                */
  const void* hidden_norm;  /* [H]            RMSNorm after fc                  */
  dflash_layer_weights layers[DFLASH_MAX_LAYERS];
  const void* final_norm;   /* [H]                                              */
  const void* embed;        /* [V, H] BF16 -- the TARGET's embedding, borrowed  */
  const void* head;         /* [V, H] BF16 -- the TARGET's LM head, borrowed    */
} dflash_weights;

typedef struct dflash_model dflash_model;
typedef struct dflash_state dflash_state;

/* Human-readable name of a dflash_status value (static string). */
const char* dflash_status_string(int status);

/* Text of the last CUDA error seen by this thread's calls (static buffer). */
const char* dflash_last_cuda_error(void);

/* Host-only check of a configuration: DFLASH_OK if this build can run it.
 * Requirements: 1 <= n_layers <= DFLASH_MAX_LAYERS; head_dim in {64, 128,
 * 256}; n_q_heads % n_kv_heads == 0 and (n_q_heads / n_kv_heads) * 8 a
 * multiple of 16 and at most 128 (the attention's query rows per kv head
 * fill one 128-row tensor-core tile; at most 112 when head_dim is 256, for
 * shared memory); hidden, n_q_heads*head_dim, intermediate multiples of 256,
 * hidden at most 8192;
 * vocab >= 2; 0 <= mask_token_id < vocab; n_taps >= 1; rope_theta > 0;
 * norm_eps >= 0; a known weight_type.  No device is touched. */
int dflash_config_check(const dflash_config* cfg);

/* Create a model on the current CUDA device.
 *   w:  device pointers as described above, all non-null.  The 36 backbone
 *       matrices and the norm vectors are COPIED into library-owned device
 *       memory (repacked into the library's streaming layout), so the caller
 *       may free them once this call returns.  embed and head are BORROWED
 *       (the drafter has no embedding or LM head of its own, "#1426 ...",
 *       "DFlash artifact"): they must stay valid and unchanged until
 *       dflash_model_destroy.  head must be 16-byte aligned.
 * Synchronises the device.  Returns DFLASH_ERR_UNSUPPORTED for a geometry
 * dflash_config_check rejects. */
int dflash_model_create(const dflash_config* cfg, const dflash_weights* w, dflash_model** out);
int dflash_model_destroy(dflash_model* model);

/* Bytes of device memory the model owns (repacked weights and tables). */
size_t dflash_model_device_bytes(const dflash_model* model);

/* Create a drafter state: n_slots independent sequences, each with its own
 * per-layer FP16 K/V of `capacity` positions ("#1426 ...", "Owned DFlash K/V
 * state": five independent draft-layer states in drafter-owned arenas), plus
 * the workspace of one draft pass over n_slots sequences.  Cells start as
 * zeros.  1 <= n_slots <= DFLASH_MAX_SLOTS, capacity >= DFLASH_MAX_BLOCK;
 * with a model attention window W > 0, capacity >= W and capacity % 128 == 0
 * (else DFLASH_ERR_UNSUPPORTED): the cells are a ring, position pos in cell
 * pos mod capacity.
 * Layout of the K (and V) arena, FP16: [layer][slot][kv_head][capacity][d]. */
int dflash_state_create(const dflash_model* model, int32_t n_slots, int32_t capacity,
                        dflash_state** out);
int dflash_state_destroy(dflash_state* state);
size_t dflash_state_device_bytes(const dflash_state* state);

/* Step (1): fuse n newly committed positions of one slot.
 *   taps:      [n, n_taps*H] BF16 (uint16 bits), the five taps of a position
 *              concatenated in tap order.
 *   positions: [n] int32, distinct, each in [0, capacity) (ring states: >= 0,
 *              and distinct modulo capacity); a negative position skips its
 *              row (nothing written, no error), so a fixed-size call can fuse
 *              a device-determined number of positions (dflash_commit_positions).
 * For every position and layer l: k = RoPE(rmsnorm_head(W_k,l h), pos) and
 * v = W_v,l h are rounded to FP16 and written to the slot's cells,
 * overwriting what was there (a cell is addressed by its position, so a
 * position committed again replaces its cell: "#1426 ...", "Speculative
 * decode integration").
 *   dev_status: device int32 status word (DFLASH_DEV_* bits OR-ed in), or
 *               NULL to use the state's own word (dflash_state_status).
 * n may be 0 (nothing is enqueued). */
int dflash_fuse_context(const dflash_model* model, dflash_state* state, int32_t slot,
                        const uint16_t* taps, const int32_t* positions, int32_t n,
                        int32_t* dev_status, dflash_stream_t stream);

/* Steps (2)-(4): one draft pass for slots 0 .. n_seq-1.
 *   anchor_tok: [n_seq] int32, the bonus token that anchors each block.
 *   anchor_pos: [n_seq] int32, p = the slot's context length; context cells
 *               [0, p) must have been fused.
 *   block_len:  [n_seq] int32 in [2, 8]: block rows B (anchor + B-1 masks).
 *   drafts:     [n_seq, 7] int32 out: drafts[s][j] = argmax over the vocab of
 *               row j + 1 (ties to the lowest id), j < B-1; entries j >= B-1
 *               are set to -1.
 *   final_hidden: optional [n_seq, 8, H] float out (NULL to skip): the final
 *               RMSNorm output of every block row, rows >= B unspecified.
 * The pass writes each layer's block K/V into the slot's cells [p, p + B)
 * (FP16) and attends over cells [0, p + B), non-causally; no rollback is
 * needed because later fusion overwrites those cells (the drafter keeps no
 * undo log for cells of rejected drafts: same section).  With an attention window W
 * (ring state) the cells are those of positions [max(0, p + B - W), p + B),
 * each at pos mod capacity; those positions must have been fused. */
int dflash_draft_block(const dflash_model* model, dflash_state* state, int32_t n_seq,
                       const int32_t* anchor_tok, const int32_t* anchor_pos,
                       const int32_t* block_len, int32_t* drafts, float* final_hidden,
                       int32_t* dev_status, dflash_stream_t stream);

/* Step (5): greedy acceptance for n_seq windows.
 *   drafts:     [n_seq, max_block_len - 1] int32, the candidates.
 *   target_ids: [n_seq, max_block_len] int32, the verifier's argmax after
 *               each window row [anchor, candidates...].
 *   block_len:  [n_seq] int32 in [2, max_block_len].
 *   accept_len: [n_seq] int32 out: n = number of leading candidates equal to
 *               the verifier's ids.
 *   next_anchor: [n_seq] int32 out: target_ids[s][n], the verifier's own
 *               continuation (the next block's anchor).  May alias anchor
 *               arrays of the next dflash_draft_block call.
 *   anchor_pos_inout: optional [n_seq] int32: p += n + 1 (the next anchor's
 *               position) when non-NULL.
 * 2 <= max_block_len <= 8. */
/* The positions the next fusion commits after dflash_accept advanced
 * anchor_pos: the verify window's anchor and its n accepted candidates sit at
 * p .. p + n (p = anchor_pos - n - 1, with n = accept_len), so
 * positions[s][j] = p + j for j <= n and -1 for n < j < 8 ("#1426 ...",
 * "Speculative decode integration": the committed prefix is fused, the
 * bonus token anchors the next block).  With the target's taps of those rows
 * this lets fuse -> draft -> accept -> commit run on the device with no host
 * round trip (a fixed 8-row dflash_fuse_context skips the -1 rows).
 *   anchor_pos, accept_len: [n_seq] int32 device, as left by dflash_accept.
 *   positions: [n_seq, 8] int32 device out. */
int dflash_commit_positions(const int32_t* anchor_pos, const int32_t* accept_len, int32_t n_seq,
                            int32_t* positions, dflash_stream_t stream);

int dflash_accept(const int32_t* drafts, const int32_t* target_ids, const int32_t* block_len,
                  int32_t n_seq, int32_t max_block_len, int32_t* accept_len,
                  int32_t* next_anchor, int32_t* anchor_pos_inout, dflash_stream_t stream);

/* Debug / parity: copy the cells of positions [pos0, pos0 + n) of one slot
 * and layer out as float (exact widening of the FP16 cells), k_out/v_out
 * [n_kv, n, d] device buffers (either may be NULL).  Ring states (attention
 * window > 0) address position pos at cell pos mod capacity and take any
 * pos0 >= 0 with n <= capacity. */
int dflash_state_read_kv(const dflash_state* state, int32_t slot, int32_t layer, int32_t pos0,
                         int32_t n, float* k_out, float* v_out, dflash_stream_t stream);

/* Set the cells of positions [pos0, pos0 + n) (ring states: pos mod
 * capacity, as for dflash_state_read_kv) of one slot and layer from FP16 (uint16 bits)
 * arrays [n_kv, n, d] on the device (pre-filled contexts). */
int dflash_state_write_kv(dflash_state* state, int32_t slot, int32_t layer, int32_t pos0,
                          int32_t n, const uint16_t* k_in, const uint16_t* v_in,
                          dflash_stream_t stream);

/* Read and clear the state's own device status word (used when a call got
 * dev_status == NULL).  Synchronises the stream. */
int dflash_state_status(dflash_state* state, int32_t* status_out, dflash_stream_t stream);

/* Debug / parity: the model's copy of one backbone matrix, dequantised to
 * float [out, in] row-major through the same in-register decode the GEMV
 * kernels use (bit-exact: w = d * (q - offset) in float; BF16 widened).
 *   which: 0 = fc; 1 + 7*l + {0..6} = layer l's {wq, wk, wv, wo, w_gate,
 *   w_up, w_down}. */
int dflash_model_dequantize(const dflash_model* model, int32_t which, float* out,
                            dflash_stream_t stream);

/* Number of kernels one dflash_draft_block call with n_seq sequences
 * launches on this state, and one dflash_fuse_context call with n positions
 * (host-only; for launch accounting). */
int32_t dflash_draft_launches(const dflash_state* state, int32_t n_seq);
int32_t dflash_fuse_launches(const dflash_state* state, int32_t n);

/* Profiling aid: when both are non-NULL (cudaEvent_t handles created by the
 * caller), every following dflash_draft_block on this state records
 * ev_begin on its stream immediately before the LM-head kernel and ev_end
 * right after it, so the dominant kernel can be timed inside a running
 * pass; during stream capture the records become event-record nodes of the
 * graph, so every replay records them.  NULL, NULL switches it off. */
int dflash_state_set_head_events(dflash_state* state, void* ev_begin, void* ev_end);

/* Profiling aid: with n_events > 0, every following dflash_fuse_context and
 * dflash_draft_block call on this state records events[0], events[1], ... on
 * its stream, one immediately before each kernel it launches and one after
 * the last, up to n_events (cudaEvent_t handles created by the caller; the
 * array is copied).  Elapsed time between consecutive events is the time of
 * one kernel (recording between kernels removes their launch overlap, so
 * this is for breakdowns, not for headline timing).  n_events = 0 switches it
 * off.  At most 256 events. */
int dflash_state_set_profile_events(dflash_state* state, void* const* events, int32_t n_events);

/* Tuning: number of context chunks C the attention of a draft pass splits
 * each (sequence, kv head) into (split-context / flash-decode).  A pass of n
 * sequences has n * C chunks per kv head, shared out among its sequences in
 * proportion to their key counts (a longer context gets more chunks, every
 * chunk about as long).  The default C is chosen at state creation from the
 * capacity and the SM count, and a pass of several sequences on the default
 * takes at least one chunk per SM; once C is set here, every pass takes
 * exactly n * C.  Valid values are 1 .. the maximum the state was sized for
 * (returned in *max_chunks when non-NULL; pass chunks = 0 to only query).
 * Applies to later calls. */
int dflash_state_set_attn_chunks(dflash_state* state, int32_t chunks, int32_t* max_chunks);

/* Deferred K/V projection of committed rows ("#1426 ...", "Speculative decode
 * integration": the rows the verifier commits are fused into the drafter's
 * context before its next block).  With on = 1, a dflash_fuse_context call
 * of at most 8 positions on this state runs only the tap projection (fc,
 * RMSNorm) and keeps the rows; the next dflash_draft_block with n_seq = 1
 * then projects their K/V in each layer's own q/k/v GEMV, next to the
 * block's (the layer's W_k / W_v are read by both row sets at the same
 * time instead of once more by a separate launch), so that layer's
 * attention already sees them.  The positions array (and the dev_status
 * word) given to that fusion must stay valid and unchanged until then;
 * device errors of the kept rows are reported in the status word of the
 * draft pass that projects them, or in the fusion's when a separate launch
 * does.  The choice is made on the host when the calls are issued,
 * so a CUDA graph should capture such a fusion together with the draft pass
 * that projects its rows.  Any other call that needs the
 * cells first projects the kept rows with a separate launch on its own
 * stream: a draft pass with n_seq > 1, dflash_fuse_context,
 * dflash_state_read_kv, dflash_state_write_kv and dflash_state_flush.
 * Results are the same either way.  on = 0 is refused (INVALID_ARG) while
 * rows are kept: call dflash_state_flush first.  Default 0. */
int dflash_state_set_defer_kv(dflash_state* state, int32_t on);

/* Projects the K/V of rows kept by a deferring dflash_fuse_context now
 * (nothing to do: returns DFLASH_OK without enqueuing work). */
int dflash_state_flush(dflash_state* state, dflash_stream_t stream);

/* Confidence gate of the proposals ("--spec-min-p", "#3322 ...", "Long-prompt
 * diagnosis and fix": floor 0.5 by default there, 0.7 in its 256K run).  A
 * draft's confidence is the drafter's softmax probability of the drafted
 * token (its LM-head logits, all V of them).  After this call every
 * dflash_draft_block on the state writes -1 (not offered) for the first
 * draft of a block whose confidence is below `floor` and for every later
 * draft of that block, so acceptance stops there.  floor in [0, 1] (else
 * DFLASH_ERR_INVALID_ARG); 0, the default, offers every draft and skips the
 * confidences altogether (the LM head then runs a plain argmax). */
int dflash_state_set_spec_min_p(dflash_state* state, float floor);

/* Copy the confidences of the last dflash_draft_block into out, a caller
 * device buffer of [n_slots, 7] float, on the stream: entry [s][j] is the
 * confidence of draft j of slot s (whether or not the gate offered it), or
 * -1 where the block has no draft j (j >= B - 1, or non-finite logits) and
 * everywhere when that pass ran with floor 0. */
int dflash_state_read_draft_probs(const dflash_state* state, float* out, dflash_stream_t stream);

/* Greedy ids over the target's LM head for n_rows (1..8) rows of final
 * hidden states, for callers that cannot allocate device memory: code that
 * runs while a CUDA graph is being captured, engines that own all device
 * memory as one arena reserved up front, or loops that must never enter the
 * allocator.  It needs no dflash_state: its scratch is a fixed array of about
 * 1.35 MB inside the library (held by every GPU that loads it until exit), and
 * it allocates nothing.  The pages have no counterpart of this entry point.
 *   hidden: [n_rows, H] float, rows already through the final RMSNorm (the
 *           final_hidden output of dflash_draft_block is such a row set).
 *   ids:    [n_rows] int32 out: argmax over the vocabulary of head . row
 *           (ties to the lowest id), computed exactly as the draft pass does.
 * Returns DFLASH_ERR_CAPACITY when n_rows > 8, hidden > 8192 or vocab >
 * 262144 (the fixed scratch's limits), and DFLASH_ERR_INVALID_ARG when the
 * current device is not the one the model was created on.  ids[n_rows..7]
 * are not written.  The first call on each device looks up the scratch
 * array's device address; make it before any stream capture.  All calls
 * share the one scratch array: calls that overlap on the GPU race (order
 * them on one stream).  Each call clears the counters it relies on. */
int dflash_head_argmax_static(const dflash_model* model, const float* hidden, int32_t n_rows, int32_t* ids,
                              int32_t* dev_status, dflash_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* DFLASH_H_ */

// Fused epilogues of the weight-streaming GEMV (gemv.cuh).  Each receives the
// fp32 result of one 16-row m-tile for all activation rows, as the mma.sync
// C fragment: lane (r = lane/4, c = lane%4) holds, for n-tile t,
//   acc[t][0..1] = Y[row t*8 + 2c + {0,1}][weight row m = r]
//   acc[t][2..3] = Y[row t*8 + 2c + {0,1}][weight row m = r + 8]
// where the weight row of the 64-row group is frag_row<WT>(w, m).
#pragma once

#include "gemv.cuh"

namespace dflash {

struct NoLocal {};

// Y stored as fp32 [R, ldo] (activation row major).  Feature fusion: fc.
// Optional output of an epilogue that produces the rows x of a pass with 8
// rows: the next RMSNorm-fed GEMV's input.  For each finished 64-column
// group g: x[n][m] * w_next[m] in the chunked layout of 8 rows and `ku`
// inputs per unit (see xchunk_index) -- one FP16 plane when the consumer has
// GGUF weights (f16), else BF16 hi and lo = bf16(v - hi) planes -- and
// ssq[g * 8 + n] = sum of x[n][m]^2 over the group.  The GEMV divides its
// outputs by the row's RMS.  Null xn: none.
struct PackNext {
  void* xn;
  float* ssq;
  const float* w_next;
  int ku;
  int f16;

  // the four norm weights thread (w, lane) applies in group g (a load with no
  // dependence on the GEMV, so a finisher can issue it early)
  __device__ float4 load_w(int g, int w, int lane) const {
    const int q = (w * 32 + lane) & 15;
    return __ldg(reinterpret_cast<const float4*>(w_next + g * 64 + 4 * q));
  }

  template <int WT, int NT>
  __device__ void operator()(int g, int w, int lane, const float (&v)[NT][4], const float4* wpre = nullptr) const {
    if constexpr (NT == 1) {
      if (xn == nullptr) return;
      __shared__ __align__(16) float tile[8][64 + 4];
      // thread (row = tid / 16, q = tid % 16): columns 4q .. 4q + 3 of the group
      const int tid = w * 32 + lane, row = tid >> 4, q = tid & 15;
      const int m = g * 64 + 4 * q;
      const float4 wv = wpre ? *wpre : load_w(g, w, lane);
      const int r0 = frag_row<WT>(w, lane >> 2), r1 = frag_row<WT>(w, (lane >> 2) + 8);
      const int n = (lane & 3) * 2;
      tile[n][r0] = v[0][0];
      tile[n + 1][r0] = v[0][1];
      tile[n][r1] = v[0][2];
      tile[n + 1][r1] = v[0][3];
      named_bar_sync(1, 128);
      const float4 xv = *reinterpret_cast<const float4*>(&tile[row][4 * q]);
      if (f16) {
        *reinterpret_cast<uint2*>(static_cast<__half*>(xn) + xchunk_index(m, row, 0, 8, ku, 1)) =
            make_uint2(pack_f16x2(xv.x * wv.x, xv.y * wv.y), pack_f16x2(xv.z * wv.z, xv.w * wv.w));
      } else {
        uint2 hi, lo;
        split_bf16x2(xv.x * wv.x, xv.y * wv.y, hi.x, lo.x);
        split_bf16x2(xv.z * wv.z, xv.w * wv.w, hi.y, lo.y);
        __nv_bfloat16* xb = static_cast<__nv_bfloat16*>(xn);
        *reinterpret_cast<uint2*>(xb + xchunk_index(m, row, 0, 8, ku, 2)) = hi;
        *reinterpret_cast<uint2*>(xb + xchunk_index(m, row, 1, 8, ku, 2)) = lo;
      }
      float ss = xv.x * xv.x + xv.y * xv.y + xv.z * xv.z + xv.w * xv.w;
#pragma unroll
      for (int off = 8; off; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
      if (q == 0) ssq[g * 8 + row] = ss;
      named_bar_sync(1, 128);  // the tile is reused by the next group
    }
  }
};

struct EpiStore {
  static constexpr bool kAfterGroup = false, kFinish = false, kPreload = false, kCluster = true;
  using Local = NoLocal;
  float* out;
  int ldo;
  PackNext pack;  // optional (the fusion's fc output feeds the context K/V GEMV)
  __device__ void init(Local&) const {}
  __device__ void prologue(const GemvArgs&, int, const float*) const {}
  __device__ void producer_start(const GemvArgs&, int, int) const {}
  template <int WT, int NT>
  __device__ void group(const GemvArgs&, Local&, int g, int w, int lane, float (&acc)[NT][4]) const {
    const int m0 = g * 64 + frag_row<WT>(w, lane >> 2), m1 = g * 64 + frag_row<WT>(w, (lane >> 2) + 8);
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const int n = t * 8 + (lane & 3) * 2;
      out[static_cast<size_t>(n) * ldo + m0] = acc[t][0];
      out[static_cast<size_t>(n + 1) * ldo + m0] = acc[t][1];
      out[static_cast<size_t>(n) * ldo + m1] = acc[t][2];
      out[static_cast<size_t>(n + 1) * ldo + m1] = acc[t][3];
    }
    pack.template operator()<WT, NT>(g, w, lane, acc);
  }
  // cluster finishing: the group's first CTA holds the complete sums
  template <int WT>
  __device__ bool group_cluster(const GemvArgs& a, const Local&, int g, int, int, int w, int lane, int,
                                float (&acc)[1][4], float*, uint64_t*, bool ok) const {
    Local loc;
    group<WT, 1>(a, loc, g, w, lane, acc);
    return ok;
  }
  __device__ void prepare_cluster(const GemvArgs&, Local&, int, int, int) const {}
  __device__ void after_group(const GemvArgs&, int, int, int*) const {}
  template <int NT>
  __device__ void finish(const GemvArgs&, Local&, int, int, int, unsigned long long*, int*) const {}
};

// Residual update x[R, ldx] += Y: attention output projection and MLP down
// projection.  Every element has exactly one owner thread.
struct EpiResid {
  static constexpr bool kAfterGroup = false, kFinish = false, kCluster = true;
  // a split group's finisher loads its residual values before it knows it
  // is the finisher, overlapping that load with the arrival counter
  static constexpr bool kPreload = true;
  using Local = NoLocal;
  float* x;
  int ldx;
  PackNext pack;  // optional: the next RMSNorm-fed GEMV's operand from x_new

  __device__ void init(Local&) const {}
  __device__ void prologue(const GemvArgs&, int, const float*) const {}
  __device__ void producer_start(const GemvArgs&, int, int) const {}
  __device__ void prepare_cluster(const GemvArgs&, Local&, int, int, int) const {}

  template <int WT, int NT>
  __device__ void group(const GemvArgs&, Local&, int g, int w, int lane, float (&acc)[NT][4]) const {
    const int m0 = g * 64 + frag_row<WT>(w, lane >> 2), m1 = g * 64 + frag_row<WT>(w, (lane >> 2) + 8);
    float v[NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const int n = t * 8 + (lane & 3) * 2;
      float* p00 = x + static_cast<size_t>(n) * ldx + m0;
      float* p10 = x + static_cast<size_t>(n + 1) * ldx + m0;
      float* p01 = x + static_cast<size_t>(n) * ldx + m1;
      float* p11 = x + static_cast<size_t>(n + 1) * ldx + m1;
      v[t][0] = *p00 + acc[t][0];
      v[t][1] = *p10 + acc[t][1];
      v[t][2] = *p01 + acc[t][2];
      v[t][3] = *p11 + acc[t][3];
      *p00 = v[t][0];
      *p10 = v[t][1];
      *p01 = v[t][2];
      *p11 = v[t][3];
    }
    pack.template operator()<WT, NT>(g, w, lane, v);
  }
  template <int WT, int NT>
  __device__ void preload(int g, int w, int lane, float (&pre)[NT][4], float4& wpre) const {
    if (NT == 1 && pack.xn != nullptr) wpre = pack.load_w(g, w, lane);
    const int m0 = g * 64 + frag_row<WT>(w, lane >> 2), m1 = g * 64 + frag_row<WT>(w, (lane >> 2) + 8);
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const int n = t * 8 + (lane & 3) * 2;
      pre[t][0] = __ldcg(x + static_cast<size_t>(n) * ldx + m0);
      pre[t][1] = __ldcg(x + static_cast<size_t>(n + 1) * ldx + m0);
      pre[t][2] = __ldcg(x + static_cast<size_t>(n) * ldx + m1);
      pre[t][3] = __ldcg(x + static_cast<size_t>(n + 1) * ldx + m1);
    }
  }
  template <int WT, int NT>
  __device__ void group_pre(int g, int w, int lane, const float (&acc)[NT][4], const float (&pre)[NT][4],
                            const float4& wpre) const {
    const int m0 = g * 64 + frag_row<WT>(w, lane >> 2), m1 = g * 64 + frag_row<WT>(w, (lane >> 2) + 8);
    float v[NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const int n = t * 8 + (lane & 3) * 2;
#pragma unroll
      for (int e = 0; e < 4; ++e) v[t][e] = pre[t][e] + acc[t][e];
      x[static_cast<size_t>(n) * ldx + m0] = v[t][0];
      x[static_cast<size_t>(n + 1) * ldx + m0] = v[t][1];
      x[static_cast<size_t>(n) * ldx + m1] = v[t][2];
      x[static_cast<size_t>(n + 1) * ldx + m1] = v[t][3];
    }
    pack.template operator()<WT, NT>(g, w, lane, v, &wpre);
  }
  __device__ void after_group(const GemvArgs&, int, int, int*) const {}
  template <int NT>
  __device__ void finish(const GemvArgs&, Local&, int, int, int, unsigned long long*, int*) const {}
};

// SwiGLU: the packed gate/up matrix holds, in every 16-row m-tile, 8 gate
// rows then the 8 up rows of the same outputs, so a lane owns gate (m = r)
// and up (m = r + 8) of output o = g*32 + w*8 + r:  h[n][o] = silu(g) * u,
// written in the chunked layout the down projection streams (FP16, or BF16
// hi and lo planes).
template <bool kF16>
struct EpiSwiglu {
  static constexpr bool kAfterGroup = false, kFinish = false, kPreload = false, kCluster = false;
  using Local = NoLocal;
  void* h;
  __device__ void init(Local&) const {}
  __device__ void prologue(const GemvArgs&, int, const float*) const {}
  __device__ void producer_start(const GemvArgs&, int, int) const {}
  __device__ static float silu(float v) { return v / (1.f + __expf(-v)); }
  template <int WT, int NT>
  __device__ void group(const GemvArgs&, Local&, int g, int w, int lane, float (&acc)[NT][4]) const {
    constexpr int R = NT * 8, KU = Fmt<WT>::CB * 32, P = kF16 ? 1 : 2;
    const int o = g * 32 + w * 8 + (lane >> 2);
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const int n = t * 8 + (lane & 3) * 2;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float v = silu(acc[t][e]) * acc[t][e + 2];
        if constexpr (kF16) {
          static_cast<__half*>(h)[xchunk_index(o, n + e, 0, R, KU, P)] = __float2half_rn(v);
        } else {
          __nv_bfloat16* hp = static_cast<__nv_bfloat16*>(h);
          const __nv_bfloat16 hi = __float2bfloat16_rn(v);
          hp[xchunk_index(o, n + e, 0, R, KU, P)] = hi;
          hp[xchunk_index(o, n + e, 1, R, KU, P)] = __float2bfloat16_rn(v - __bfloat162float(hi));
        }
      }
    }
  }
  __device__ void after_group(const GemvArgs&, int, int, int*) const {}
  template <int NT>
  __device__ void finish(const GemvArgs&, Local&, int, int, int, unsigned long long*, int*) const {}
};

// Per-attention-head epilogue.  Group results are stored raw; the CTA that
// completes the last 64-row group of a head (atomic counter, no waiting)
// applies the per-head RMSNorm, the NeoX rotation and the FP16 rounding and
// writes the results: queries to q_ready, keys and values into the
// position-addressed state cells.
//   mode 0 (draft QKV): heads [0, n_q) are queries, then n_kv key heads, then
//     n_kv value heads; activation row n is block row n % 8 of slot n / 8 at
//     position anchor_pos[slot] + n % 8.
//   mode 1 (fusion K/V): per layer l, n_kv key heads then n_kv value heads;
//     activation row n is committed position positions[n].
struct EpiHeads {
  static constexpr bool kAfterGroup = true, kFinish = false, kPreload = false, kCluster = true;
  // cluster finishing of an 8-row pass: what a thread needs for its rows
  // (w, w + 4) and rotation pairs (lane + 32 j), prepared at kernel start
  // Thread t of the first warpgroup writes row t / 16, head columns
  // 64 gl + 4 (t % 16) + k (k < 4) of its group gl: each output is
  // rs * (y_i * A[k] + y_p * B[k]) with p the column paired with i by the
  // rotation, A = w_i cos * scale, B = -+ w_p sin * scale.
  struct Local {
    float A[4], B[4];
    int pos;
    int use;  // the row is written
  };
  int mode;
  float* raw;       // [R, ldr]
  int ldr;
  int d, n_q, n_kv, gph;
  int* head_cnt;
  const float* q_norm;   // mode 0: this layer's [d]
  const float* k_norm;   // mode 0: this layer's [d]; mode 1: all layers [L, d]
  const uint64_t* turns; // [d/2]
  float eps, q_scale;
  __half* q_ready;       // [slots, n_kv, n_q / n_kv * 8, d]
  __half* Kst;
  __half* Vst;
  int layer, n_slots, cap;
  int ring;              // cells form a ring (attention window): position pos in cell pos mod cap
  int n_seq;             // mode 0: slots in this pass
  int window;            // attention window (ring), else 0
  int prefetch_kv;       // mode 0: prefetch the layer's context K/V into L2 for the attention
  const int32_t* anchor_pos;
  const int32_t* block_len;
  int slot;              // mode 1
  const int32_t* positions;  // mode 1: [n_valid] of this tile
  int n_valid;               // mode 1
  // mode 0 with extra heads (n_heads0 > 0): heads hh >= n_heads0 are this
  // layer's key heads then value heads again, over the committed rows
  // (vpositions[vn_valid] of slot vslot), written like mode 1 (cluster
  // finishing only)
  int n_heads0;
  const int32_t* vpositions;
  int vn_valid;
  int vslot;
  int32_t* status;

  __device__ bool extra(int hh) const { return mode == 0 && n_heads0 > 0 && hh >= n_heads0; }

  __device__ void init(Local&) const {}
  __device__ void prologue(const GemvArgs&, int, const float*) const {}

  // Draft QKV (mode 0), producer lane after the dependent-launch wait: CTA
  // cta of G asks L2 for its share of this layer's context K and V cells
  // (positions [lo, p) of every slot and kv head, the cells the attention
  // reads next; evict-last, so the weight stream does not displace them).
  __device__ void producer_start(const GemvArgs&, int cta, int G) const {
    if (mode != 0 || !prefetch_kv) return;
    const uint64_t pol = l2_policy_evict_last();
    const long long row_bytes = static_cast<long long>(d) * 2;
    {
      // only a layer's K/V that L2 holds comfortably beside the weight
      // stream (longer contexts stream their K/V in the attention itself)
      long long total = 0;
      for (int s = 0; s < n_seq; ++s) {
        const int p = anchor_pos[s];
        int lo = 0;
        if (ring) lo = p - (window - DFLASH_MAX_BLOCK) > 0 ? p - (window - DFLASH_MAX_BLOCK) : 0;
        if (p > lo) total += static_cast<long long>(p - lo) * n_kv * 2 * row_bytes;
      }
      if (total > (32ll << 20)) return;
    }
    // total bytes over (slot, K/V, kv head) ranges, in cells
    for (int s = 0; s < n_seq; ++s) {
      const int p = anchor_pos[s];
      int lo = 0;
      if (ring) lo = p - (window - DFLASH_MAX_BLOCK) > 0 ? p - (window - DFLASH_MAX_BLOCK) : 0;
      if (p <= lo) continue;
      const long long n_pos = p - lo;
      const long long per_cta = (n_pos + G - 1) / G;
      const long long a0 = lo + per_cta * cta, a1 = a0 + per_cta < p ? a0 + per_cta : p;
      if (a0 >= a1) continue;
      for (int kvh = 0; kvh < n_kv; ++kvh)
        for (int kv = 0; kv < 2; ++kv) {
          const __half* base = (kv ? Vst : Kst) + static_cast<size_t>((layer * n_slots + s) * n_kv + kvh) * cap * d;
          // a ring wraps at cap: at most two runs of cells
          long long c0 = ring ? a0 % cap : a0;
          long long left = a1 - a0;
          while (left > 0) {
            const long long run = (c0 + left <= cap) ? left : cap - c0;
            const char* src = reinterpret_cast<const char*>(base + c0 * d);
            long long bytes = run * row_bytes;
            while (bytes > 0) {
              const uint32_t b = static_cast<uint32_t>(bytes < (1 << 20) ? bytes : (1 << 20));
              bulk_prefetch_l2(src, b, pol);
              src += b;
              bytes -= b;
            }
            left -= run;
            c0 = 0;
          }
        }
    }
  }

  // Row metadata of activation row n: position, whether its K/V cells are
  // written, whether it is used at all (queries always are).
  __device__ void row_info(int n, int kind, bool xh, int& pos, bool& write_state, bool& use) const {
    pos = 0;
    write_state = false;
    use = true;
    if (mode == 0 && !xh) {
      const int sl = n >> 3, i = n & 7;
      if (sl < n_seq) {
        int B = block_len[sl];
        B = B < DFLASH_MIN_BLOCK ? DFLASH_MIN_BLOCK : (B > DFLASH_MAX_BLOCK ? DFLASH_MAX_BLOCK : B);
        pos = anchor_pos[sl] + i;
        write_state = (i < B) && pos >= 0 && (ring || pos < cap);
      }
    } else {
      if (n >= (xh ? vn_valid : n_valid)) {
        use = false;
      } else {
        pos = (xh ? vpositions : positions)[n];
        // a negative position is a row to skip (no cell, no error)
        write_state = pos >= 0 && (ring || pos < cap);
      }
    }
    if (kind != 0 && !write_state) use = false;
  }

  // Cluster finishing, kernel start (8-row pass, this CTA = local group gl
  // of head g / gph): this thread's row metadata and, for query and key
  // heads, its columns' norm weights folded with their rotations at the
  // row's position, so the finishing step after the weight stream has no
  // global loads and no sin / cos left.
  __device__ void prepare_cluster(const GemvArgs&, Local& L, int g, int w, int lane) const {
    const int hh = g / gph, gl = g - hh * gph;
    const int kind = head_kind(hh);
    const bool xh = extra(hh);
    const int half = d / 2;
    const int t = w * 32 + lane, n = t >> 4;
    bool ws, use;
    row_info(n, kind, xh, L.pos, ws, use);
    if ((mode == 1 || xh) && L.pos >= 0 && !ws && n < (xh ? vn_valid : n_valid) && (t & 15) == 0 &&
        hh == (xh ? n_heads0 : 0))
      set_status(status, DFLASH_DEV_CAPACITY);
    L.use = use;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      L.A[k] = 1.f;
      L.B[k] = 0.f;
    }
    if (kind == 2) return;
    const float* wn = (mode == 0) ? (kind == 0 ? q_norm : k_norm) : k_norm + static_cast<size_t>(hh / (2 * n_kv)) * d;
    const float scale = kind == 0 ? q_scale : 1.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int i = gl * 64 + (t & 15) * 4 + k;
      const bool lo = i < half;
      const int f = lo ? i : i - half, p = lo ? i + half : i - half;
      float sn, cs;
      rope_sincos(__ldg(turns + f), L.pos, sn, cs);
      L.A[k] = __ldg(wn + i) * cs * scale;
      L.B[k] = (lo ? -1.f : 1.f) * __ldg(wn + p) * sn * scale;
    }
  }

  template <int WT, int NT>
  __device__ void group(const GemvArgs&, Local&, int g, int w, int lane, float (&acc)[NT][4]) const {
    if (extra(g / gph)) return;  // extra heads finish in clusters only
    const int m0 = g * 64 + frag_row<WT>(w, lane >> 2), m1 = g * 64 + frag_row<WT>(w, (lane >> 2) + 8);
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const int n = t * 8 + (lane & 3) * 2;
      __stcg(raw + static_cast<size_t>(n) * ldr + m0, acc[t][0]);
      __stcg(raw + static_cast<size_t>(n + 1) * ldr + m0, acc[t][1]);
      __stcg(raw + static_cast<size_t>(n) * ldr + m1, acc[t][2]);
      __stcg(raw + static_cast<size_t>(n + 1) * ldr + m1, acc[t][3]);
    }
  }

  __device__ void after_group(const GemvArgs& a, int g, int tid, int* sflag) const {
    const int head = g / gph;
    if (extra(head)) return;
    if (gph > 1) {
      if (tid == 0) {
        const int old = atomic_add_acq_rel(&head_cnt[head], 1);
        sflag[1] = (old == gph - 1);
        if (sflag[1]) head_cnt[head] = 0;
      }
      named_bar_sync(1, 128);
      if (!sflag[1]) return;
    }
    process_head(head, tid);
  }

  // 0: query head, 1: key head, 2: value head
  __device__ int head_kind(int hh) const {
    if (extra(hh)) return hh - n_heads0 < n_kv ? 1 : 2;
    if (mode == 0) return hh < n_q ? 0 : (hh < n_q + n_kv ? 1 : 2);
    return (hh % (2 * n_kv)) < n_kv ? 1 : 2;
  }

  __device__ void process_head(int hh, int tid) const {
    if (extra(hh)) return;  // extra heads finish in clusters only
    const float* base = raw + static_cast<size_t>(hh) * d;
    const int ld = ldr;
    process_head_src(hh, tid, [base, ld](int n, int i) { return __ldcg(base + static_cast<size_t>(n) * ld + i); },
                     0, d);
  }

  // Cluster finishing of the 8-row pass: this CTA holds the complete sums of
  // local group gl of head g / gph.  Key and query heads need every group of
  // the head (RMS over d, RoPE pairs (i, i + d/2)): each group's per-warp sums
  // of squares go to slot gl of every group CTA's buffer and its values to
  // slot gl of its RoPE partner's ([gph][8 rows][64] floats, in distributed
  // shared memory), and each CTA then writes its own 64 columns.
  // Value heads write their columns straight away.
  template <int WT>
  __device__ bool group_cluster(const GemvArgs& ga, const Local& L, int g, int gl, int parts, int w, int lane,
                                int tid, float (&acc)[1][4], float* hbuf, uint64_t* head_bar, bool ok) const {
#ifdef DFLASH_TRACE
    unsigned long long* a_trace = ga.trace;
#else
    (void)ga;
#endif
    constexpr int SLOT = 512 + 32;
    const int hh = g / gph;
    const int kind = head_kind(hh);
    const bool exch = gph > 1 && kind != 2;
    // this group's values in mma fragment order (thread t at 4 t) and, for
    // the norm, each warp's sums of squares of rows 0..7 over its 16 columns
    float* mine = hbuf + gl * SLOT;
    const int t4 = tid * 4;
    *reinterpret_cast<float4*>(mine + t4) = make_float4(acc[0][0], acc[0][1], acc[0][2], acc[0][3]);
    float s0 = 0.f, s1 = 0.f;
    if (kind != 2) {
      s0 = acc[0][0] * acc[0][0] + acc[0][2] * acc[0][2];  // row 2 (lane % 4)
      s1 = acc[0][1] * acc[0][1] + acc[0][3] * acc[0][3];  // row 2 (lane % 4) + 1
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        s0 += __shfl_xor_sync(0xffffffffu, s0, o);
        s1 += __shfl_xor_sync(0xffffffffu, s1, o);
      }
      if (lane < 4) *reinterpret_cast<float2*>(mine + 512 + w * 8 + lane * 2) = make_float2(s0, s1);
    }
    if (exch) {
      // every peer needs this group's sums of squares (the head's RMS); only
      // the RoPE partner (the group half a head away) needs its values
      const int partner = gl ^ (gph >> 1);
      for (int l2 = 0; l2 < gph; ++l2) {
        if (l2 == gl) continue;
        const uint32_t r = static_cast<uint32_t>(l2 * parts);
        if (l2 == partner)
          st_cluster_v4(mapa_shared(smem_u32(mine + t4), r), acc[0][0], acc[0][1], acc[0][2], acc[0][3]);
        if (lane < 4) {
          st_cluster_f32(mapa_shared(smem_u32(mine + 512 + w * 8 + lane * 2), r), s0);
          st_cluster_f32(mapa_shared(smem_u32(mine + 512 + w * 8 + lane * 2 + 1), r), s1);
        }
      }
    }
    named_bar_sync(1, 128);
#ifdef DFLASH_TRACE
    if (tid == 0 && a_trace) a_trace[static_cast<size_t>(blockIdx.x) * kTraceSlots + 9] = globaltimer_ns();
#endif
    if (exch) {
      if (tid == 0)
        for (int l2 = 0; l2 < gph; ++l2)
          if (l2 != gl) mbar_remote_arrive(mapa_shared(smem_u32(head_bar), static_cast<uint32_t>(l2 * parts)));
      if (ok && !mbar_wait_cluster(head_bar, 0)) {
        set_status(status, DFLASH_DEV_TIMEOUT);
        ok = false;
      }
    }
#ifdef DFLASH_TRACE
    if (tid == 0 && a_trace) a_trace[static_cast<size_t>(blockIdx.x) * kTraceSlots + 2] = globaltimer_ns();
#endif
    // ---- this thread's four outputs: row n, columns i0 .. i0 + 3
    if (!L.use) return ok;
    const int n = tid >> 4, c = (tid & 15) * 4, i0 = gl * 64 + c;
    const int half = d / 2;
    int kvh, l;
    const bool xh = extra(hh);
    if (xh) {
      l = layer;
      const int rem = hh - n_heads0;
      kvh = rem < n_kv ? rem : rem - n_kv;
    } else if (mode == 0) {
      l = layer;
      kvh = kind == 0 ? 0 : (kind == 1 ? hh - n_q : hh - n_q - n_kv);
    } else {
      l = hh / (2 * n_kv);
      const int rem = hh - l * 2 * n_kv;
      kvh = rem < n_kv ? rem : rem - n_kv;
    }
    float out[4];
    if (kind == 2) {
#pragma unroll
      for (int k = 0; k < 4; ++k) out[k] = mine[frag_index(c + k, n)];
    } else {
      float ss = 0.f;
      for (int g2 = 0; g2 < gph; ++g2)
#pragma unroll
        for (int w2 = 0; w2 < 4; ++w2) ss += hbuf[g2 * SLOT + 512 + w2 * 8 + n];
      const float rs = rsqrtf(ss / d + eps);
      const int ip0 = i0 < half ? i0 + half : i0 - half;  // partner columns ip0 .. ip0 + 3
      const float* ps = hbuf + (ip0 >> 6) * SLOT;
      const int cp = ip0 & 63;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float yi = mine[frag_index(c + k, n)];
        const float yp = ps[frag_index(cp + k, n)];
        out[k] = rs * (yi * L.A[k] + yp * L.B[k]);
      }
    }
    const int pos = L.pos;
    __half* dst;
    if (kind == 0) {
      const int gq = n_q / n_kv;
      dst = q_ready + ((static_cast<size_t>((n >> 3) * n_kv + hh / gq) * gq + hh % gq) * 8 + (n & 7)) * d + i0;
    } else {
      const int sl = xh ? vslot : (mode == 0 ? (n >> 3) : slot);
      const size_t cell = ((static_cast<size_t>((l * n_slots + sl) * n_kv + kvh) * cap) +
                           (ring ? pos % cap : pos)) * d;
      dst = (kind == 1 ? Kst : Vst) + cell + i0;
    }
    const __half2 h01 = __floats2half2_rn(out[0], out[1]), h23 = __floats2half2_rn(out[2], out[3]);
    *reinterpret_cast<uint2*>(dst) =
        make_uint2(*reinterpret_cast<const uint32_t*>(&h01), *reinterpret_cast<const uint32_t*>(&h23));
    return ok;
  }

  // Element (row n, column c) of one group's values in mma fragment order
  // (column c = 16 w' + r sits at thread w' * 32 + (r % 8) * 4 + n / 2,
  // value (r / 8) * 2 + n % 2).
  __device__ static int frag_index(int c, int n) {
    const int r = c & 15;
    return ((c >> 4) * 32 + (r & 7) * 4 + (n >> 1)) * 4 + (r >> 3) * 2 + (n & 1);
  }

  // Norm, rotation, FP16 rounding and cell / query writes of head hh for all
  // rows; src(n, i) gives element i of row n's raw head values.  Only the
  // outputs of columns [c_lo, c_hi) are written (their inputs may be read
  // from any column of the head).
  template <class Src>
  __device__ void process_head_src(int hh, int tid, Src src, int c_lo, int c_hi) const {
    const int w = tid >> 5, lane = tid & 31;
    const int half = d / 2;
    const int R = n_rows();
    int kind, kvh, l;
    const float* wn;
    const bool full = c_lo == 0 && c_hi >= d;  // every column written (no filtering)
    if (mode == 0) {
      l = layer;
      if (hh < n_q) { kind = 0; kvh = 0; wn = q_norm; }
      else if (hh < n_q + n_kv) { kind = 1; kvh = hh - n_q; wn = k_norm; }
      else { kind = 2; kvh = hh - n_q - n_kv; wn = nullptr; }
    } else {
      l = hh / (2 * n_kv);
      const int rem = hh - l * 2 * n_kv;
      kind = rem < n_kv ? 1 : 2;
      kvh = rem < n_kv ? rem : rem - n_kv;
      wn = kind == 1 ? k_norm + static_cast<size_t>(l) * d : nullptr;
    }
    // the head's per-column constants, loaded once and independent of the rows
    const int hj = d / 64;  // pairs per lane; element i + d/2 sits at yv[j + hj]
    float wa[4], wb[4];
    uint64_t tn[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      wa[j] = wb[j] = 0.f;
      tn[j] = 0;
      if (kind != 2 && j < hj) {
        const int i = lane + 32 * j;
        wa[j] = __ldg(wn + i);
        wb[j] = __ldg(wn + i + half);
        tn[j] = __ldg(turns + i);
      }
    }
    // warp w takes rows w, w + 4, w + 8, ... two at a time, both rows' loads in flight together
    for (int n0 = w; n0 < R; n0 += 8) {
      int pos[2], sl[2];
      bool use[2], write_state[2];
      float yv[2][8];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int n = n0 + 4 * q;
        pos[q] = 0;
        sl[q] = 0;
        write_state[q] = false;
        use[q] = n < R;
        if (use[q]) {
          if (mode == 0) {
            sl[q] = n >> 3;
            const int i = n & 7;
            if (sl[q] < n_seq) {
              int B = block_len[sl[q]];
              B = B < DFLASH_MIN_BLOCK ? DFLASH_MIN_BLOCK : (B > DFLASH_MAX_BLOCK ? DFLASH_MAX_BLOCK : B);
              pos[q] = anchor_pos[sl[q]] + i;
              write_state[q] = (i < B) && pos[q] >= 0 && (ring || pos[q] < cap);
            }
          } else {
            sl[q] = slot;
            if (n >= n_valid) {
              use[q] = false;
            } else {
              pos[q] = positions[n];
              // a negative position is a row to skip (no cell, no error)
              write_state[q] = pos[q] >= 0 && (ring || pos[q] < cap);
              if (pos[q] >= 0 && !write_state[q] && lane == 0 && hh == 0) set_status(status, DFLASH_DEV_CAPACITY);
            }
          }
          if (kind != 0 && !write_state[q]) use[q] = false;
        }
        // the row's d values, lane-strided: element lane + 32 j (d <= 256);
        // value heads read only the columns they write
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int i = lane + 32 * j;
          const bool need = i < d && (kind != 2 || full || (i >= c_lo && i < c_hi));
          yv[q][j] = (use[q] && need) ? src(n, i) : 0.f;
        }
      }
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        if (!use[q]) continue;
        const int n = n0 + 4 * q;
        const size_t cell =
            ((static_cast<size_t>((l * n_slots + sl[q]) * n_kv + kvh) * cap) + (ring ? pos[q] % cap : pos[q])) * d;
        if (kind == 2) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int i = lane + 32 * j;
            if (i < d && (full || (i >= c_lo && i < c_hi))) Vst[cell + i] = __float2half_rn(yv[q][j]);
          }
          continue;
        }
        float ss = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) ss += yv[q][j] * yv[q][j];
#pragma unroll
        for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        const float rs = rsqrtf(ss / d + eps);
        // queries: [slot][kv head][m = local head * 8 + block row][d] (contiguous per slot and kv head)
        const int gq = n_q / n_kv;
        __half* dst = kind == 0
                          ? q_ready + ((static_cast<size_t>(sl[q] * n_kv + hh / gq) * gq + hh % gq) * 8 + (n & 7)) * d
                          : Kst + cell;
        const float scale = kind == 0 ? q_scale : 1.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (j < hj) {
            const int i = lane + 32 * j;
            const float a = yv[q][j] * rs * wa[j];
            // element i + d/2 (d = 64, 128 or 256), picked without a runtime register index
            const float yb = hj == 4 ? yv[q][(j + 4) & 7] : (hj == 2 ? yv[q][(j + 2) & 7] : yv[q][(j + 1) & 7]);
            const float b = yb * rs * wb[j];
            const bool w_lo = full || (i >= c_lo && i < c_hi);
            const bool w_hi = full || (i + half >= c_lo && i + half < c_hi);
            if (w_lo || w_hi) {
              float sn, cs;
              rope_sincos(tn[j], pos[q], sn, cs);
              if (w_lo) dst[i] = __float2half_rn((a * cs - b * sn) * scale);
              if (w_hi) dst[i + half] = __float2half_rn((b * cs + a * sn) * scale);
            }
          }
        }
      }
    }
  }
  __device__ int n_rows() const { return rows_; }
  int rows_;
  template <int NT>
  __device__ void finish(const GemvArgs&, Local&, int, int, int, unsigned long long*, int*) const {}
};

// LM head + argmax.  Every thread keeps the best (value, vocab id) of its two
// activation rows per n-tile across all groups of the CTA's range; at the
// end the CTA reduces them, publishes one packed key per activation row, and
// the CTA that arrives last reduces all CTAs' keys into the drafts.  Keys are
// (order-preserving float bits << 32) | (0xffffffff - id), so the maximum is
// the largest logit with ties going to the lowest id.
template <int NT_>
struct EpiArgmax {
  static constexpr bool kAfterGroup = false, kFinish = true, kPreload = false, kCluster = false;
  struct Local {
    float v[NT_][2];
    int id[NT_][2];
    float s[NT_][2];  // sum of exp(logit - v) over the logits this thread saw
    int bad;
  };
  int vocab;
  int n_seq;
  const int32_t* block_len;
  int32_t* drafts;               // [n_seq, 7]
  unsigned long long* slots;     // [gridDim.x, R]
  float2* ms;                    // [gridDim.x, R]: each CTA's (max logit, sum of exp(logit - max))
  float* probs;                  // [n_seq, 7] out: softmax probability of each draft (-1 where none)
  float min_p;                   // confidence floor: drafts from the first one below it are not offered;
                                 // 0: no confidences are computed (probs are -1) and every draft is offered
  int* grid_cnt;
  float* final_hidden;           // optional [n_seq, 8, H] (X_NORM prologue)
  const float* x;                // residual rows for final_hidden
  const float* norm_w;
  int H;
  int32_t* status;

  __device__ void init(Local& L) const {
#pragma unroll
    for (int t = 0; t < NT_; ++t)
      for (int h = 0; h < 2; ++h) {
        L.v[t][h] = -INFINITY;
        L.id[t][h] = 0x7fffffff;
        L.s[t][h] = 0.f;
      }
    L.bad = 0;
  }
  __device__ void producer_start(const GemvArgs&, int, int) const {}
  __device__ void prologue(const GemvArgs&, int tid, const float* srs) const {
    if (final_hidden == nullptr || blockIdx.x != 0 || srs == nullptr) return;
    for (int i = tid; i < n_seq * 8 * H; i += 128) {
      const int n = i / H, k = i - n * H;
      final_hidden[i] = __ldcg(x + static_cast<size_t>(n) * H + k) * srs[n] * norm_w[k];
    }
  }
  template <int WT, int NT>
  __device__ void group(const GemvArgs&, Local& L, int g, int w, int lane, float (&acc)[NT][4]) const {
    const int m0 = g * 64 + frag_row<WT>(w, lane >> 2), m1 = g * 64 + frag_row<WT>(w, (lane >> 2) + 8);
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int m = e < 2 ? m0 : m1;
        const float v = acc[t][e];
        if (m < vocab) {
          constexpr float LOG2E = 1.4426950408889634f;
          const int h = e & 1;
          if (!isfinite(v)) {
            // only rows of the pass's sequences count (tile t holds sequence
            // t's 8 rows; the rows of a tile's unused slots carry no data)
            if (t < n_seq) L.bad = 1;
          } else if (min_p > 0.f) {
            if (v > L.v[t][h]) {
              // a new maximum: rescale the running sum to it (0 from -inf)
              L.s[t][h] = L.s[t][h] * ex2_approx((L.v[t][h] - v) * LOG2E) + 1.f;
              L.v[t][h] = v;
              L.id[t][h] = m;
            } else {
              L.s[t][h] += ex2_approx((v - L.v[t][h]) * LOG2E);
              if (v == L.v[t][h] && m < L.id[t][h]) L.id[t][h] = m;
            }
          } else if (v > L.v[t][h] || (v == L.v[t][h] && m < L.id[t][h])) {
            L.v[t][h] = v;
            L.id[t][h] = m;
          }
        }
      }
  }
  __device__ void after_group(const GemvArgs&, int, int, int*) const {}

  __device__ static unsigned long long pack(float v, int id) {
    if (id == 0x7fffffff) return 0ull;
    return (static_cast<unsigned long long>(float_order_key(v)) << 32) |
           static_cast<unsigned long long>(0xffffffffu - static_cast<uint32_t>(id));
  }

  // In the last CTA: the largest key of each of the R rows over every CTA's
  // slot (exact, order-free).  All 128 threads take part: thread t scans row
  // t % R over CTAs t / R, t / R + 128 / R, ... with 8 loads in flight, then
  // the stripes of a row are combined.  The result is valid in threads t < R.
  template <int R>
  __device__ unsigned long long grid_max(int tid, int w, int lane, unsigned long long* sstage) const {
    constexpr int NS = 128 / R;
    const int G = static_cast<int>(gridDim.x);
    const int r = tid % R, st = tid / R;
    unsigned long long k = 0ull;
    for (int c0 = st; c0 < G; c0 += 8 * NS) {
      unsigned long long v[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int c = c0 + q * NS;
        v[q] = c < G ? __ldcg(slots + static_cast<size_t>(c) * R + r) : 0ull;
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) k = v[q] > k ? v[q] : k;
    }
    if constexpr (R < 32) {
      // lanes r, r + R, ... of a warp hold row r
#pragma unroll
      for (int o = R; o < 32; o <<= 1) {
        const unsigned long long k2 = __shfl_xor_sync(0xffffffffu, k, o);
        k = k2 > k ? k2 : k;
      }
      if (lane < R) sstage[w * R + lane] = k;
    } else {
      sstage[tid] = k;  // stripe st of row r at st * R + r (at most 4 stripes)
    }
    named_bar_sync(1, 128);
    k = 0ull;
    if (tid < R) {
      constexpr int E = R < 32 ? 4 : 128 / R;  // partial maxima per row
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const unsigned long long k2 = sstage[e * R + tid];
        k = k2 > k ? k2 : k;
      }
    }
    return k;
  }

  template <int NT>
  __device__ void finish(const GemvArgs& a, Local& L, int w, int lane, int tid, unsigned long long* sstage,
                         int* sflag) const {
    constexpr int R = NT * 8;
    const bool any_bad = __any_sync(0xffffffffu, L.bad);
    if (any_bad && lane == 0) set_status(status, DFLASH_DEV_NONFINITE);
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        unsigned long long k = pack(L.v[t][h], L.id[t][h]);
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
          const unsigned long long k2 = __shfl_xor_sync(0xffffffffu, k, o);
          k = k2 > k ? k2 : k;
        }
        if (lane < 4) sstage[w * R + t * 8 + lane * 2 + h] = k;
      }
    named_bar_sync(1, 128);
    // the CTA's largest key per row; then, rescaled to the row's largest
    // logit, the CTA's sum of exp(logit - max) (float scratch over sstage:
    // [0, R) row maxima, [R, 5R) per-warp sums, [5R, 6R) probabilities)
    constexpr float LOG2E = 1.4426950408889634f;
    float* sf = reinterpret_cast<float*>(sstage);
    unsigned long long kc = 0ull;
    if (tid < R) {
      kc = sstage[tid];
      for (int ww = 1; ww < 4; ++ww) {
        const unsigned long long k2 = sstage[ww * R + tid];
        kc = k2 > kc ? k2 : kc;
      }
    }
    const bool sums = min_p > 0.f;  // uniform: confidences wanted
    named_bar_sync(1, 128);
    if (sums) {
      if (tid < R) sf[tid] = kc ? float_from_order_key(static_cast<uint32_t>(kc >> 32)) : -INFINITY;
      named_bar_sync(1, 128);
#pragma unroll
      for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const float mrow = sf[t * 8 + (lane & 3) * 2 + h];
          float c = L.s[t][h] > 0.f ? L.s[t][h] * ex2_approx((L.v[t][h] - mrow) * LOG2E) : 0.f;
#pragma unroll
          for (int o = 4; o < 32; o <<= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
          if (lane < 4) sf[R + w * R + t * 8 + lane * 2 + h] = c;
        }
      named_bar_sync(1, 128);
      if (tid < R) {
        const float S = (sf[R + tid] + sf[2 * R + tid]) + (sf[3 * R + tid] + sf[4 * R + tid]);
        __stcg(ms + static_cast<size_t>(blockIdx.x) * R + tid, make_float2(sf[tid], S));
      }
    }
    if (tid < R) __stcg(slots + static_cast<size_t>(blockIdx.x) * R + tid, kc);
    named_bar_sync(1, 128);
    if (tid == 0) {
      const int old = atomic_add_acq_rel(grid_cnt, 1);
      sflag[2] = (old == static_cast<int>(gridDim.x) - 1);
    }
    named_bar_sync(1, 128);
    if (!sflag[2]) return;
    const unsigned long long k = grid_max<R>(tid, w, lane, sstage);
    named_bar_sync(1, 128);
    if (sums) {
      if (tid < R) sf[tid] = k ? float_from_order_key(static_cast<uint32_t>(k >> 32)) : -INFINITY;
      named_bar_sync(1, 128);
      {
        // sum over every CTA of its sum rescaled to the row's overall maximum:
        // thread t takes row t % R over CTAs t / R, t / R + 128 / R, ...
        constexpr int NS = 128 / R;
        const int G = static_cast<int>(gridDim.x);
        const int r = tid % R, st = tid / R;
        const float mg = sf[r];
        float acc = 0.f;
        for (int c0 = st; c0 < G; c0 += 8 * NS) {
          float2 v[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const int c = c0 + q * NS;
            v[q] = c < G ? __ldcg(ms + static_cast<size_t>(c) * R + r) : make_float2(-INFINITY, 0.f);
          }
#pragma unroll
          for (int q = 0; q < 8; ++q)
            if (v[q].y > 0.f) acc += v[q].y * ex2_approx((v[q].x - mg) * LOG2E);
        }
        if constexpr (R < 32) {
#pragma unroll
          for (int o = R; o < 32; o <<= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
          if (lane < R) sf[R + w * R + lane] = acc;
        } else {
          sf[R + tid] = acc;  // stripe st of row r at R + st * R + r
        }
      }
      named_bar_sync(1, 128);
      if (tid < R) {
        constexpr int E = R < 32 ? 4 : 128 / R;
        float S = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) S += sf[R + e * R + tid];
        sf[5 * R + tid] = S > 0.f ? 1.f / S : 0.f;
      }
      named_bar_sync(1, 128);
    }
    if (tid < R) {
      const int s = tid >> 3, i = tid & 7;
      if (s < n_seq && i >= 1) {
        int B = block_len[s];
        B = B < DFLASH_MIN_BLOCK ? DFLASH_MIN_BLOCK : (B > DFLASH_MAX_BLOCK ? DFLASH_MAX_BLOCK : B);
        int out = -1;
        float prob = -1.f;
        if (i < B) {
          if (k == 0ull) {
            set_status(status, DFLASH_DEV_NONFINITE);
          } else {
            out = static_cast<int>(0xffffffffu - static_cast<uint32_t>(k & 0xffffffffull));
            if (sums) {
              prob = sf[5 * R + tid];
              // offered only if no draft of the block up to this one is below the floor
              for (int i2 = 1; i2 <= i; ++i2)
                if (sf[5 * R + s * 8 + i2] < min_p) out = -1;
            }
          }
        }
        drafts[s * (DFLASH_MAX_BLOCK - 1) + (i - 1)] = out;
        if (probs) probs[s * (DFLASH_MAX_BLOCK - 1) + (i - 1)] = prob;
      }
    }
    if (tid == 0) *grid_cnt = 0;
  }
};

}  // namespace dflash

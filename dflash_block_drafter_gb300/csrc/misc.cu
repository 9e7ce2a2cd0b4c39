// Small kernels of libdflash: weight repacking and its bit-exact check,
// block embedding, row RMSNorm for streamed-X GEMVs, greedy acceptance and
// K/V cell import / export.
#include "kernels.h"
#include "layout.cuh"

namespace dflash {

// ---------------------------------------------------------------- repack
// Destination row of source row `row` of a matrix placed into a packed
// matrix: rows are offset by `row_off`; with `interleave` = 0 / 1 the source
// is the gate / up matrix of a SwiGLU pair and its rows go to the first /
// second 8 rows of every 16-row m-tile.
__device__ __forceinline__ int repack_dst_row(int row, int row_off, int interleave) {
  if (interleave < 0) return row + row_off;
  return (row >> 3) * 16 + interleave * 8 + (row & 7) + row_off;
}

// Byte offset of the sub-chunk holding (packed row P, 32-block b) for m-tile
// and lane bookkeeping, per layout.cuh.
template <int WT>
__device__ __forceinline__ size_t chunk_offset(int P, int b, int UPG) {
  using F = Fmt<WT>;
  const int g = P >> 6, w = (P >> 4) & 3;
  const int j = b / F::CB, bl = b - j * F::CB;
  const int sc = bl / F::SUBB;
  return (static_cast<size_t>(g) * UPG + j) * F::UNIT + static_cast<size_t>(sc * 4 + w) * F::CHUNK;
}

// One thread per (source row, 32-block).
template <int WT>
__global__ void repack_kernel(const uint8_t* __restrict__ src, int rows, int K, uint8_t* __restrict__ dst,
                              int row_off, int interleave) {
  using F = Fmt<WT>;
  const int nb = K / 32;
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<long long>(rows) * nb) return;
  const int row = static_cast<int>(idx / nb), b = static_cast<int>(idx % nb);
  const int P = repack_dst_row(row, row_off, interleave);
  const int UPG = K / (32 * F::CB);
  uint8_t* chunk = dst + chunk_offset<WT>(P, b, UPG);
  const int r16 = P & 15, r = r16 & 7, half = r16 >> 3;
  if constexpr (WT == WT_BF16) {
    const uint16_t* s = reinterpret_cast<const uint16_t*>(src) + static_cast<size_t>(row) * K + b * 32;
    for (int c = 0; c < 4; ++c) {
      uint16_t* d = reinterpret_cast<uint16_t*>(chunk + half * 512 + (r * 4 + c) * 16);
      for (int t = 0; t < 8; ++t) d[t] = s[c * 8 + t];
    }
  } else {
    constexpr int BS = (WT == WT_Q8_0) ? 34 : (WT == WT_Q4_0 ? 18 : 22);
    const uint8_t* blk = src + (static_cast<size_t>(row) * nb + b) * BS;
    const uint16_t dbits = static_cast<uint16_t>(blk[0] | (blk[1] << 8));
    int q[32];
    if constexpr (WT == WT_Q8_0) {
      for (int e = 0; e < 32; ++e) q[e] = static_cast<int>(static_cast<int8_t>(blk[2 + e])) + 128;
    } else if constexpr (WT == WT_Q4_0) {
      for (int e = 0; e < 16; ++e) {
        q[e] = blk[2 + e] & 0xF;
        q[e + 16] = blk[2 + e] >> 4;
      }
    } else {
      const uint32_t qh = blk[2] | (blk[3] << 8) | (blk[4] << 16) | (static_cast<uint32_t>(blk[5]) << 24);
      for (int e = 0; e < 16; ++e) {
        q[e] = (blk[6 + e] & 0xF) | (((qh >> e) & 1) << 4);
        q[e + 16] = (blk[6 + e] >> 4) | (((qh >> (e + 16)) & 1) << 4);
      }
    }
    if constexpr (WT == WT_Q8_0) {
      for (int c = 0; c < 4; ++c)
        for (int t = 0; t < 8; ++t) chunk[(r * 4 + c) * 16 + half * 8 + t] = static_cast<uint8_t>(q[c * 8 + t]);
      reinterpret_cast<uint16_t*>(chunk + 512)[r * 2 + half] = dbits;
    } else {
      const int bp = (b % F::CB) & 1;  // block within the sub-chunk pair
      for (int c = 0; c < 4; ++c) {
        uint32_t word = 0;
        for (int t = 0; t < 8; ++t) {
          const int nib = (t & 1) ? (t >> 1) + 4 : (t >> 1);  // e0 e2 e4 e6 e1 e3 e5 e7
          word |= static_cast<uint32_t>(q[c * 8 + t] & 0xF) << (4 * nib);
        }
        reinterpret_cast<uint32_t*>(chunk + (r * 4 + c) * 16)[half * 2 + bp] = word;
        if constexpr (WT == WT_Q5_0) {
          uint32_t hb = 0;
          const int off = (half * 2 + bp) * 4;
          for (int t = 0; t < 8; ++t) {
            const uint32_t bit = (q[c * 8 + t] >> 4) & 1;
            hb |= bit << ((t & 1) ? off + (t >> 1) + 16 : off + (t >> 1));
          }
          atomicOr(reinterpret_cast<unsigned int*>(chunk + 512 + (r * 4 + c) * 4), hb);
        }
      }
      constexpr int SC_OFF = (WT == WT_Q4_0) ? 512 : 640;
      reinterpret_cast<uint16_t*>(chunk + SC_OFF)[r * 4 + bp * 2 + half] = dbits;
    }
  }
}

cudaError_t launch_repack(int wtype, const void* src, int rows, int K, uint8_t* dst, int row_off, int interleave,
                          cudaStream_t st) {
  const long long n = static_cast<long long>(rows) * (K / 32);
  const int threads = 256;
  const unsigned blocks = static_cast<unsigned>((n + threads - 1) / threads);
  const uint8_t* s = static_cast<const uint8_t*>(src);
  switch (wtype) {
    case WT_BF16: repack_kernel<WT_BF16><<<blocks, threads, 0, st>>>(s, rows, K, dst, row_off, interleave); break;
    case WT_Q8_0: repack_kernel<WT_Q8_0><<<blocks, threads, 0, st>>>(s, rows, K, dst, row_off, interleave); break;
    case WT_Q4_0: repack_kernel<WT_Q4_0><<<blocks, threads, 0, st>>>(s, rows, K, dst, row_off, interleave); break;
    case WT_Q5_0: repack_kernel<WT_Q5_0><<<blocks, threads, 0, st>>>(s, rows, K, dst, row_off, interleave); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

// ------------------------------------------------------- dequant check
// One CTA per unit: the unit is staged in shared memory and each warp decodes
// its m-tile with the GEMV's decode_block, writing w = d * code as float at
// the source row/column (undoing the gate/up interleave when `interleave`).
template <int WT>
__global__ void dequant_kernel(const uint8_t* __restrict__ packed, int N, int K, float* __restrict__ out,
                               int row_off, int rows_out, int interleave) {
  using F = Fmt<WT>;
  __shared__ __align__(16) uint8_t su[F::UNIT];
  const int UPG = K / (32 * F::CB);
  const int u = blockIdx.x;
  const int g = u / UPG, j = u - g * UPG;
  const uint4* src = reinterpret_cast<const uint4*>(packed + static_cast<size_t>(u) * F::UNIT);
  for (int i = threadIdx.x; i < F::UNIT / 16; i += blockDim.x) reinterpret_cast<uint4*>(su)[i] = src[i];
  __syncthreads();
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = lane >> 2, c = lane & 3;
  for (int bl = 0; bl < F::CB; ++bl) {
    const BlockFrag f = decode_block<WT>(smem_u32(su), w, lane, bl);  // the layer GEMVs' decode
    for (int s = 0; s < 2; ++s)
      for (int reg = 0; reg < 4; ++reg) {
        const uint32_t v = f.a[s][reg];
        float lo, hi;
        if constexpr (F::kF16) {
          const __half2 h = *reinterpret_cast<const __half2*>(&v);
          lo = __low2float(h);
          hi = __high2float(h);
        } else {
          lo = __uint_as_float(v << 16);
          hi = __uint_as_float(v & 0xffff0000u);
        }
        const int m = r + ((reg & 1) ? 8 : 0);
        const float d = (reg & 1) ? f.d_r8 : f.d_r;
        const int kk = j * F::CB * 32 + bl * 32 + 8 * c + 4 * s + ((reg & 2) ? 2 : 0);
        int P = g * 64 + w * 16 + m;  // packed row
        int row;
        if (interleave < 0) {
          row = P - row_off;
        } else {
          const int r16 = P & 15;
          if ((r16 >> 3) != interleave) continue;
          row = (P >> 4) * 8 + (r16 & 7);
        }
        if (row < 0 || row >= rows_out) continue;
        out[static_cast<size_t>(row) * K + kk] = lo * d;
        out[static_cast<size_t>(row) * K + kk + 1] = hi * d;
      }
  }
}

cudaError_t launch_dequant(int wtype, const uint8_t* packed, int N, int K, float* out, int row_off, int rows_out,
                           int interleave, cudaStream_t st) {
  int UPG = 0;
  switch (wtype) {
    case WT_BF16: UPG = K / (32 * Fmt<WT_BF16>::CB); break;
    default: UPG = K / (32 * Fmt<WT_Q8_0>::CB); break;
  }
  const unsigned blocks = static_cast<unsigned>((N / 64) * UPG);
  switch (wtype) {
    case WT_BF16: dequant_kernel<WT_BF16><<<blocks, 128, 0, st>>>(packed, N, K, out, row_off, rows_out, interleave); break;
    case WT_Q8_0: dequant_kernel<WT_Q8_0><<<blocks, 128, 0, st>>>(packed, N, K, out, row_off, rows_out, interleave); break;
    case WT_Q4_0: dequant_kernel<WT_Q4_0><<<blocks, 128, 0, st>>>(packed, N, K, out, row_off, rows_out, interleave); break;
    case WT_Q5_0: dequant_kernel<WT_Q5_0><<<blocks, 128, 0, st>>>(packed, N, K, out, row_off, rows_out, interleave); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

// ------------------------------------------------------------- embedding
// x[slot*8 + i] = E[token_i] (anchor for i = 0, the mask token otherwise),
// widened to fp32; slots >= n_seq are zero.  Also validates the pass's
// device-side scalars.

constexpr int kEmbedThreads = 128;  // one 16-byte piece (4 columns) of a row per thread

__global__ void __launch_bounds__(kEmbedThreads) embed_kernel(const __grid_constant__ EmbedArgs a) {
  const int s = blockIdx.x, i = blockIdx.y;
  const int c = blockIdx.z * kEmbedThreads + static_cast<int>(threadIdx.x);  // 4-column piece of the row
  const int H4 = a.H / 4;
  const bool live = s < a.n_seq, in_row = c < H4;
  // Before the dependent-launch wait only reads of what no kernel of this
  // stream is still writing: the token id (written by the caller or by an
  // earlier acceptance, complete before the previous kernel could release
  // this one), the embedding row and the norm weights (constants).
  int tok = a.mask_id;
  bool bad_tok = false;
  if (live && i == 0) {
    tok = a.anchor_tok[s];
    if (tok < 0 || tok >= a.vocab) {
      bad_tok = true;
      tok = 0;
    }
  }
  uint2 e = make_uint2(0u, 0u);
  float4 wv = make_float4(0.f, 0.f, 0.f, 0.f);
  if (live && in_row) {
    e = __ldg(reinterpret_cast<const uint2*>(a.embed + static_cast<size_t>(tok) * a.H) + c);
    if (a.xn) wv = __ldg(reinterpret_cast<const float4*>(a.w_next) + c);
  }
  pdl_wait();
  pdl_launch_dependents();
  if (live && i == 0 && blockIdx.z == 0 && threadIdx.x == 0) {
    if (bad_tok) set_status(a.status, DFLASH_DEV_BAD_TOKEN);
    const int B = a.block_len[s];
    if (B < DFLASH_MIN_BLOCK || B > DFLASH_MAX_BLOCK) set_status(a.status, DFLASH_DEV_BAD_BLOCK);
    const int Bc = B < DFLASH_MIN_BLOCK ? DFLASH_MIN_BLOCK : (B > DFLASH_MAX_BLOCK ? DFLASH_MAX_BLOCK : B);
    const int p = a.anchor_pos[s];
    if (p < 0 || (!a.ring && static_cast<long long>(p) + Bc > a.cap)) set_status(a.status, DFLASH_DEV_CAPACITY);
  }
  const int n = s * 8 + i;
  float4* xr = reinterpret_cast<float4*>(a.x + static_cast<size_t>(n) * a.H);
  // the BF16 row widened to fp32 (zeros for slots >= n_seq)
  const float4 v = make_float4(__uint_as_float(e.x << 16), __uint_as_float(e.x & 0xffff0000u),
                               __uint_as_float(e.y << 16), __uint_as_float(e.y & 0xffff0000u));
  if (in_row) xr[c] = v;
  if (!live || a.xn == nullptr) return;
  // one slot: the BF16 hi/lo planes (or the FP16 plane) of x * w_next and the
  // sum of squares of each 64-column group (16 consecutive lanes, fixed order)
  if (in_row) {
    if (a.f16) {
      *reinterpret_cast<uint2*>(static_cast<__half*>(a.xn) + xchunk_index(4 * c, n, 0, 8, a.ku, 1)) =
          make_uint2(pack_f16x2(v.x * wv.x, v.y * wv.y), pack_f16x2(v.z * wv.z, v.w * wv.w));
    } else {
      uint2 hi, lo;
      split_bf16x2(v.x * wv.x, v.y * wv.y, hi.x, lo.x);
      split_bf16x2(v.z * wv.z, v.w * wv.w, hi.y, lo.y);
      __nv_bfloat16* xb = static_cast<__nv_bfloat16*>(a.xn);
      *reinterpret_cast<uint2*>(xb + xchunk_index(4 * c, n, 0, 8, a.ku, 2)) = hi;
      *reinterpret_cast<uint2*>(xb + xchunk_index(4 * c, n, 1, 8, a.ku, 2)) = lo;
    }
  }
  float ss = v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
#pragma unroll
  for (int off = 8; off; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  if ((threadIdx.x & 15) == 0 && in_row) a.ssq[(c / 16) * 8 + n] = ss;
}

cudaError_t launch_embed(const EmbedArgs& a, int nt, cudaStream_t st) {
  if (a.H % 64 != 0) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(nt, 8, (a.H / 4 + kEmbedThreads - 1) / kEmbedThreads);
  cfg.blockDim = dim3(kEmbedThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, embed_kernel, a);
}

// ---------------------------------------------------------- row RMSNorm
// out[r] = act(x[r] / sqrt(mean(x[r]^2) + eps) * w) for the streamed-X
// GEMVs, and optionally the same rows in fp32 (final hidden state output).
// One CTA per row: the row is read once, as 16-byte loads all issued
// together (up to kNormV per thread), and normalised from registers.

constexpr int kNormThreads = 128, kNormV = 16;  // rows of up to 8192 floats

__global__ void __launch_bounds__(kNormThreads) rmsnorm_rows_kernel(const __grid_constant__ NormArgs a) {
  const int r = blockIdx.x;
  const int H4 = a.H >> 2;
  // the norm weights (constants) before the dependent-launch wait
  float4 w[kNormV];
#pragma unroll
  for (int i = 0; i < kNormV; ++i) {
    const int k4 = static_cast<int>(threadIdx.x) + i * kNormThreads;
    w[i] = k4 < H4 ? __ldg(reinterpret_cast<const float4*>(a.w) + k4) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  pdl_wait();
  pdl_launch_dependents();
  __shared__ float red[kNormThreads / 32];
  const bool valid = r < a.rows_valid;
  const float4* xr = reinterpret_cast<const float4*>(a.x + static_cast<size_t>(r) * a.H);
  float4 v[kNormV];
#pragma unroll
  for (int i = 0; i < kNormV; ++i) {
    const int k4 = static_cast<int>(threadIdx.x) + i * kNormThreads;
    v[i] = (valid && k4 < H4) ? __ldcg(xr + k4) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < kNormV; ++i) ss += v[i].x * v[i].x + v[i].y * v[i].y + v[i].z * v[i].z + v[i].w * v[i].w;
  for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int i = 0; i < kNormThreads / 32; ++i) tot += red[i];
  const float rs = valid ? rsqrtf(tot / a.H + a.eps) : 0.f;
  const int R = gridDim.x;
#pragma unroll
  for (int i = 0; i < kNormV; ++i) {
    const int k4 = static_cast<int>(threadIdx.x) + i * kNormThreads;
    if (k4 >= H4) break;
    const int k = 4 * k4;
    const float4 w4 = w[i];
    const float y0 = v[i].x * rs * w4.x, y1 = v[i].y * rs * w4.y, y2 = v[i].z * rs * w4.z, y3 = v[i].w * rs * w4.w;
    // four consecutive inputs of one chunk row (KU is a multiple of 4)
    if (a.out_f16) {
      *reinterpret_cast<uint2*>(static_cast<__half*>(a.out) + xchunk_index(k, r, 0, R, a.ku, 1)) =
          make_uint2(pack_f16x2(y0, y1), pack_f16x2(y2, y3));
    } else {
      uint32_t h01, l01, h23, l23;
      split_bf16x2(y0, y1, h01, l01);
      split_bf16x2(y2, y3, h23, l23);
      __nv_bfloat16* o = static_cast<__nv_bfloat16*>(a.out);
      *reinterpret_cast<uint2*>(o + xchunk_index(k, r, 0, R, a.ku, 2)) = make_uint2(h01, h23);
      *reinterpret_cast<uint2*>(o + xchunk_index(k, r, 1, R, a.ku, 2)) = make_uint2(l01, l23);
    }
    if (a.f32_out && r < a.rows_f32)
      reinterpret_cast<float4*>(a.f32_out + static_cast<size_t>(r) * a.H)[k4] = make_float4(y0, y1, y2, y3);
  }
}

cudaError_t launch_rmsnorm_rows(const NormArgs& a, int rows, cudaStream_t st) {
  if (a.H % 4 != 0 || a.H > 4 * kNormThreads * kNormV || a.ku % 4 != 0) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(rows);
  cfg.blockDim = dim3(kNormThreads);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, rmsnorm_rows_kernel, a);
}

// ------------------------------------------------------------- accept
// Greedy acceptance ("#366 [RFC] ...", "Verification and state management"):
// n = leading candidates equal to the verifier's argmax, bonus = target[n].
__global__ void accept_kernel(const int32_t* __restrict__ drafts, const int32_t* __restrict__ tgt,
                              const int32_t* __restrict__ block_len, int n_seq, int maxB,
                              int32_t* __restrict__ accept_len, int32_t* __restrict__ next_anchor,
                              int32_t* __restrict__ anchor_pos) {
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= n_seq) return;
  int B = block_len[s];
  B = B < DFLASH_MIN_BLOCK ? DFLASH_MIN_BLOCK : (B > maxB ? maxB : B);
  const int32_t* d = drafts + static_cast<size_t>(s) * (maxB - 1);
  const int32_t* t = tgt + static_cast<size_t>(s) * maxB;
  int n = 0;
  while (n < B - 1 && d[n] == t[n]) ++n;
  const int bonus = t[n];
  accept_len[s] = n;
  next_anchor[s] = bonus;
  if (anchor_pos) anchor_pos[s] += n + 1;
}

// Positions committed by the last acceptance, for the next fusion: with the
// anchor already advanced to p + n + 1, the committed rows are p .. p + n
// (the anchor and the n accepted candidates); the rest of the 8 are -1.
__global__ void commit_positions_kernel(const int32_t* __restrict__ anchor_pos, const int32_t* __restrict__ accept_len,
                                        int n_seq, int32_t* __restrict__ out) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n_seq * DFLASH_MAX_BLOCK) return;
  const int s = i / DFLASH_MAX_BLOCK, j = i - s * DFLASH_MAX_BLOCK;
  const int n = accept_len[s];
  out[i] = j <= n ? anchor_pos[s] - n - 1 + j : -1;
}

cudaError_t launch_commit_positions(const int32_t* anchor_pos, const int32_t* accept_len, int n_seq, int32_t* out,
                                    cudaStream_t st) {
  const int total = n_seq * DFLASH_MAX_BLOCK;
  commit_positions_kernel<<<(total + 127) / 128, 128, 0, st>>>(anchor_pos, accept_len, n_seq, out);
  return cudaGetLastError();
}

cudaError_t launch_accept(const int32_t* drafts, const int32_t* tgt, const int32_t* block_len, int n_seq, int maxB,
                          int32_t* accept_len, int32_t* next_anchor, int32_t* anchor_pos, cudaStream_t st) {
  const int threads = 128;
  accept_kernel<<<(n_seq + threads - 1) / threads, threads, 0, st>>>(drafts, tgt, block_len, n_seq, maxB,
                                                                      accept_len, next_anchor, anchor_pos);
  return cudaGetLastError();
}

// ------------------------------------------------------- K/V import/export
// Cell of position pos: pos itself, or pos mod cap in a ring of cells.
__device__ __forceinline__ size_t kv_cell(int pos, int cap, int ring) {
  return static_cast<size_t>(ring ? pos % cap : pos);
}

__global__ void kv_read_kernel(const __half* __restrict__ cells, int cap, int ring, int d, int n_kv, int pos0, int n,
                               float* __restrict__ out) {
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long total = static_cast<long long>(n_kv) * n * d;
  if (idx >= total) return;
  const int h = static_cast<int>(idx / (static_cast<long long>(n) * d));
  const long long rem = idx - static_cast<long long>(h) * n * d;
  const int i = static_cast<int>(rem / d), k = static_cast<int>(rem % d);
  out[idx] = __half2float(cells[(static_cast<size_t>(h) * cap + kv_cell(pos0 + i, cap, ring)) * d + k]);
}

__global__ void kv_write_kernel(__half* __restrict__ cells, int cap, int ring, int d, int n_kv, int pos0, int n,
                                const uint16_t* __restrict__ in) {
  const long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const long long total = static_cast<long long>(n_kv) * n * d;
  if (idx >= total) return;
  const int h = static_cast<int>(idx / (static_cast<long long>(n) * d));
  const long long rem = idx - static_cast<long long>(h) * n * d;
  const int i = static_cast<int>(rem / d), k = static_cast<int>(rem % d);
  cells[(static_cast<size_t>(h) * cap + kv_cell(pos0 + i, cap, ring)) * d + k] = __ushort_as_half(in[idx]);
}

cudaError_t launch_kv_copy(bool write, __half* cells, int cap, bool ring, int d, int n_kv, int pos0, int n, float* out,
                           const uint16_t* in, cudaStream_t st) {
  const long long total = static_cast<long long>(n_kv) * n * d;
  if (total == 0) return cudaSuccess;
  const int threads = 256;
  const unsigned blocks = static_cast<unsigned>((total + threads - 1) / threads);
  if (write) kv_write_kernel<<<blocks, threads, 0, st>>>(cells, cap, ring, d, n_kv, pos0, n, in);
  else kv_read_kernel<<<blocks, threads, 0, st>>>(cells, cap, ring, d, n_kv, pos0, n, out);
  return cudaGetLastError();
}

}  // namespace dflash

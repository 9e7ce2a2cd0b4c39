"""CPU oracle for the DFlash block-draft pass.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or
executes this module: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline / reference legs of ``bench.py`` use it, to check and to time the CUDA
path.  It shares no code with the CUDA library (``libdflash``) and does not
import it.

Plain NumPy, float64 throughout.  The only non-float64 values are the ones the
method itself stores at lower precision: the per-layer context K/V state is
FP16 ("#1426 dflash: experimental standalone DeepSpec DFlash block drafter",
section "Owned DFlash K/V state": FP16 K/V), BF16 weights and norm vectors are
read from their BF16 bit patterns, and GGUF-style blocks are dequantised from
their bytes.  Every function is the plain definition of one step, in the
order the pages give, with no blocking, fusion or reordering.

Citations name the page (by its title) and the section:
  [#1426] "#1426 dflash: experimental standalone DeepSpec DFlash block drafter
          for Qwen3.8-Flash-Next (greedy, correctness-first)"
  [#366]  "#366 [RFC] EXPERIMENTAL Investigate DFlash2 support for
          Qwen3.8-Flash-Next"
  [#3322] "#3322 [Engine] support the official Flash-Next DFlash2 checkpoint"

Readings where the pages are silent (the library header states the same ones):
  * RMSNorm is x / sqrt(mean(x^2) + eps) * w with eps = 1e-6.
  * per-head RMSNorm over head_dim on q and k ("q raw / q normed / q" stage
    names, [#1426] "Parity validation"), before RoPE, also on context k.
  * NeoX RoPE pairs (i, i + d/2), inv_freq_i = theta^(-2i/d), full head.
  * q head h reads kv head floor(h / (n_q / n_kv)).
  * The draft pass writes the block rows' K/V into the position-addressed
    cells [p, p + B) of each layer's state before attending over [0, p + B);
    fusing a committed position later overwrites its cell ([#1426]
    "Speculative decode integration": rejected cells need no rollback).
  * Drafts are the argmax of rows 1..B-1 (lowest id on ties).
  * Attention window W > 0 ([#1426] "Additional constraints": the drafter
    attention window defaults to 32768 cells; [#3322] keeps 32768 resident
    cells for a 262144-token context in physical rings): the block at p
    attends over positions [max(0, p + B - W), p + B), and the state keeps
    position pos in cell pos mod capacity.
  * Accept length n = longest prefix with draft_j == target_j; the bonus
    token is target_n.
  * Confidence gate (--spec-min-p floor, [#3322] "Long-prompt diagnosis and
    fix": floor 0.5 by default, 0.7 in the 256K run): a draft's confidence
    is the drafter's softmax probability of the drafted token, and the block
    offers the drafts before the first one whose confidence is below the
    floor (floor 0 offers all).

parity status: every function below is pinned by tests/test_oracle_pins.py
(closed forms, hand-packed blocks, invariants, brute force, the pages' own
geometry and acceptance cases).  The per-layer composition of the pass is
pinned as well: the per-head q / k norms (scale invariance of W_q, W_k; the
q_norm x k_norm product), which norm feeds which sub-layer (zero mlp_norm
removes the MLP; zero attn_norm gives uniform attention over the values),
the roles of gate and up (a one-unit SwiGLU closed form) and the value path
(an identity W_v stores the unnormed, unrotated input).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional

import numpy as np

GGUF_BLOCK_BYTES = {"q8_0": 34, "q5_0": 22, "q4_0": 18}


# ----------------------------------------------------------------------------
# storage formats
# ----------------------------------------------------------------------------

def decode_bf16(bits) -> np.ndarray:
    """BF16 bit patterns -> float64 (exact): the 16 bits are the top half of
    an IEEE float32."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def round_f16(x) -> np.ndarray:
    """Round to IEEE half precision (round to nearest, ties to even)."""
    return np.asarray(x, dtype=np.float64).astype(np.float16)


def dequantize(raw, wtype: str, n: int, k: int) -> np.ndarray:
    """GGUF-style 32-weight blocks -> float64 [n, k].

    Each block holds an FP16 scale d and 32 integer codes q; the weight is
    w = d * (q - offset) with offset 0 (Q8_0, signed 8-bit q), 8 (Q4_0,
    4-bit q) or 16 (Q5_0, 5-bit q) ([#3322] "Approach": Q8_0 / Q5_0 / Q4_0
    backbone quantisations of the 36 backbone matrices).  Byte layout (public
    GGUF block formats):
      Q8_0: d (2 B), q[32] int8
      Q4_0: d (2 B), qs[16]: element j in the low nibble of qs[j], element
            j + 16 in its high nibble
      Q5_0: d (2 B), qh (4 B little-endian, bit j = fifth bit of element j),
            qs[16] as Q4_0
    The product of an 11-bit FP16 mantissa and a code of at most 8 bits is
    exact in float64 (and in float32).
    """
    bs = GGUF_BLOCK_BYTES[wtype]
    nb = k // 32
    blk = np.asarray(raw, dtype=np.uint8).reshape(n, nb, bs)
    d = blk[..., 0:2].copy().view("<f2")[..., 0].astype(np.float64)
    if wtype == "q8_0":
        q = blk[..., 2:34].copy().view(np.int8).astype(np.float64)
    elif wtype == "q4_0":
        qs = blk[..., 2:18].astype(np.int64)
        q = np.concatenate([qs & 0xF, qs >> 4], axis=-1).astype(np.float64) - 8.0
    elif wtype == "q5_0":
        qh = blk[..., 2:6].copy().view("<u4")[..., 0].astype(np.int64)
        qs = blk[..., 6:22].astype(np.int64)
        low = np.concatenate([qs & 0xF, qs >> 4], axis=-1)
        fifth = np.stack([(qh >> j) & 1 for j in range(32)], axis=-1)
        q = (low | (fifth << 4)).astype(np.float64) - 16.0
    else:
        raise ValueError(wtype)
    return (d[..., None] * q).reshape(n, k)


# ----------------------------------------------------------------------------
# the steps of the pass
# ----------------------------------------------------------------------------

def rmsnorm(x, w, eps: float) -> np.ndarray:
    """RMSNorm over the last axis: x / sqrt(mean(x^2) + eps) * w."""
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(w, dtype=np.float64)


def rope_neox(x, pos, theta: float) -> np.ndarray:
    """Full-head NeoX rotary embedding ([#1426] "Drafter runtime": full-head
    NeoX RoPE, theta 1e7).

    x: [..., d]; pos broadcasts against x.shape[:-1].  Element i < d/2 is
    rotated together with element i + d/2 by the angle pos * theta^(-2i/d).
    """
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    half = d // 2
    inv_freq = float(theta) ** (-(2.0 * np.arange(half, dtype=np.float64)) / d)
    ang = np.asarray(pos, dtype=np.float64)[..., None] * inv_freq
    c, s = np.cos(ang), np.sin(ang)
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)


def silu(x) -> np.ndarray:
    x = np.asarray(x, dtype=np.float64)
    return x / (1.0 + np.exp(-x))


def attention(q, k, v, scale: float) -> np.ndarray:
    """Non-causal GQA attention of every query row over every key
    ([#1426] "Target feature taps": non-causal block attention, scale 1/16).

    q: [R, n_q, d]; k, v: [T, n_kv, d] -> [R, n_q, d].  Query head h reads
    kv head floor(h / (n_q / n_kv)).  Softmax in float64.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    R, nq, d = q.shape
    nkv = k.shape[1]
    grp = nq // nkv
    out = np.empty_like(q)
    for g in range(nkv):
        heads = slice(g * grp, (g + 1) * grp)
        qg = q[:, heads, :].reshape(R * grp, d)
        s = (qg @ k[:, g, :].T) * scale
        s = s - s.max(axis=-1, keepdims=True)
        p = np.exp(s)
        p = p / p.sum(axis=-1, keepdims=True)
        out[:, heads, :] = (p @ v[:, g, :]).reshape(R, grp, d)
    return out


# ----------------------------------------------------------------------------
# model and state
# ----------------------------------------------------------------------------

class Model:
    """The drafter's weights decoded to float64, from a checkpoint dict of
    BF16 bits / GGUF bytes (see dflash_synth.make_checkpoint).  The embedding
    and LM head are the target's ([#1426] "Drafter runtime": target embedding
    and LM head reused directly)."""

    def __init__(self, cfg, ckpt: Dict[str, np.ndarray]):
        self.cfg = cfg
        self.ckpt = ckpt
        self._cache: Dict[str, np.ndarray] = {}

    def mat(self, name: str) -> np.ndarray:
        if name not in self._cache:
            n, k = self.cfg.matrix_shapes()[name]
            raw = self.ckpt[name]
            if self.cfg.weight_type == "bf16":
                self._cache[name] = decode_bf16(raw).reshape(n, k)
            else:
                self._cache[name] = dequantize(raw, self.cfg.weight_type, n, k)
        return self._cache[name]

    def vec(self, name: str) -> np.ndarray:
        if name not in self._cache:
            self._cache[name] = decode_bf16(self.ckpt[name])
        return self._cache[name]

    def embed_rows(self, ids) -> np.ndarray:
        return decode_bf16(self.ckpt["embed"][np.asarray(ids, dtype=np.int64)])

    def head(self) -> np.ndarray:
        if "head" not in self._cache:
            self._cache["head"] = decode_bf16(self.ckpt["head"])
        return self._cache["head"]


class State:
    """Per-layer, position-addressed FP16 context K/V of one sequence
    ([#1426] "Owned DFlash K/V state": five independent per-layer states,
    FP16 K/V).  K[l], V[l]: float16 [n_kv, capacity, d].  ``held[l][c]`` is
    the position cell c holds (-1: never written); attention refuses to read
    a position whose cell does not hold it (the pages' parity harness fails
    hard on invalid cells, [#1426] "Parity validation").  Without an
    attention window position pos is cell pos (pos < capacity); with one
    (cfg.attn_window > 0) the cells are a ring and pos is cell pos mod
    capacity, so a later position overwrites the cell of an earlier one."""

    def __init__(self, cfg, capacity: int):
        self.cfg = cfg
        self.capacity = capacity
        self.window = int(getattr(cfg, "attn_window", 0) or 0)
        if self.window > capacity:
            raise ValueError("the attention window does not fit the state's cells")
        shape = (cfg.n_kv_heads, capacity, cfg.head_dim)
        self.K = [np.zeros(shape, dtype=np.float16) for _ in range(cfg.n_layers)]
        self.V = [np.zeros(shape, dtype=np.float16) for _ in range(cfg.n_layers)]
        self.held = [np.full(capacity, -1, dtype=np.int64) for _ in range(cfg.n_layers)]

    def cells(self, pos) -> np.ndarray:
        """Cell index of each position."""
        pos = np.asarray(pos, dtype=np.int64)
        if pos.size and pos.min() < 0:
            raise IndexError("negative position")
        if self.window > 0:
            return pos % self.capacity
        if pos.size and pos.max() >= self.capacity:
            raise IndexError("position outside the state's capacity")
        return pos

    def fill(self, kv_pairs, n_pos: int) -> None:
        """Set positions [0, n_pos) from float16 arrays [n_kv, n_pos, d]."""
        if n_pos > self.capacity:
            raise IndexError("more positions than cells")
        for l, (k, v) in enumerate(kv_pairs):
            self.K[l][:, :n_pos, :] = k
            self.V[l][:, :n_pos, :] = v
            self.held[l][:n_pos] = np.arange(n_pos)

    def write(self, l: int, pos, k, v) -> None:
        """Round k, v ([n, n_kv, d]) to FP16 and store them at positions pos."""
        pos = np.asarray(pos, dtype=np.int64)
        c = self.cells(pos)
        self.K[l][:, c, :] = round_f16(k).transpose(1, 0, 2)
        self.V[l][:, c, :] = round_f16(v).transpose(1, 0, 2)
        self.held[l][c] = pos

    def keys(self, l: int, hi: int, lo: int = 0):
        """float64 K, V of positions [lo, hi), as [hi - lo, n_kv, d]."""
        pos = np.arange(lo, hi, dtype=np.int64)
        c = self.cells(pos)
        held = self.held[l][c]
        if not np.array_equal(held, pos):
            bad = int(pos[np.argmax(held != pos)])
            raise ValueError(f"layer {l}: K/V of position {bad} read before it was written")
        k = self.K[l][:, c, :].astype(np.float64).transpose(1, 0, 2)
        v = self.V[l][:, c, :].astype(np.float64).transpose(1, 0, 2)
        return k, v


# ----------------------------------------------------------------------------
# step (1): feature fusion into the context K/V
# ----------------------------------------------------------------------------

def project_kv(model: Model, l: int, h: np.ndarray, pos) -> tuple:
    """Layer l's K/V of hidden rows h [n, H] at positions pos: k = RoPE(per-head
    RMSNorm(W_k h)), v = W_v h."""
    cfg = model.cfg
    n = h.shape[0]
    k = (h @ model.mat(f"layers.{l}.wk").T).reshape(n, cfg.n_kv_heads, cfg.head_dim)
    v = (h @ model.mat(f"layers.{l}.wv").T).reshape(n, cfg.n_kv_heads, cfg.head_dim)
    k = rmsnorm(k, model.vec(f"layers.{l}.k_norm"), cfg.norm_eps)
    k = rope_neox(k, np.asarray(pos)[:, None], cfg.rope_theta)
    return k, v


def fuse_hidden(model: Model, taps_bits) -> np.ndarray:
    """h_ctx = rmsnorm(fc(concat(taps))) ([#1426] "Drafter runtime").
    taps_bits: BF16 bits [n, n_taps * H], taps concatenated in boundary order."""
    cfg = model.cfg
    taps = decode_bf16(taps_bits).reshape(-1, cfg.tap_width)
    return rmsnorm(taps @ model.mat("fc").T, model.vec("hidden_norm"), cfg.norm_eps)


def fuse_context(model: Model, state: State, taps_bits, positions) -> np.ndarray:
    """Fuse newly committed positions: project h_ctx into every layer's own
    K/V and write it by position, overwriting the cell ([#1426] "Drafter
    runtime" and "Speculative decode integration").  A negative position
    marks a row that is not committed: it is skipped.  Returns h_ctx."""
    pos = np.asarray(positions, dtype=np.int64)
    h = fuse_hidden(model, taps_bits)
    keep = pos >= 0
    for l in range(model.cfg.n_layers):
        k, v = project_kv(model, l, h[keep], pos[keep])
        state.write(l, pos[keep], k, v)
    return h


def commit_positions(anchor_pos_after: int, n: int, rows: int = 8) -> np.ndarray:
    """The positions a cycle commits for the next fusion, given the anchor
    position after acceptance (p + n + 1) and the accept length n: the
    window's anchor at p and its n accepted candidates, p .. p + n; the
    remaining rows are -1 ([#1426] "Speculative decode integration")."""
    p = int(anchor_pos_after) - int(n) - 1
    return np.array([p + j if j <= n else -1 for j in range(rows)], dtype=np.int32)


# ----------------------------------------------------------------------------
# steps (2)-(4): the draft pass
# ----------------------------------------------------------------------------

@dataclasses.dataclass
class DraftResult:
    drafts: np.ndarray        # int32 [B-1]: argmax of rows 1..B-1
    final_hidden: np.ndarray  # float64 [B, H]: rmsnorm(x, final_norm) of every row
    logits: np.ndarray        # float64 [B-1, V]
    top2_gap: np.ndarray      # float64 [B-1]: top-1 minus top-2 logit
    stages: Optional[Dict[str, np.ndarray]] = None
    probs: Optional[np.ndarray] = None  # float64 [B-1]: softmax probability of each draft


def draft_block(model: Model, state: State, anchor_tok: int, anchor_pos: int,
                block_len: int, trace: bool = False) -> DraftResult:
    """One parallel draft pass over the block [anchor at p, mask x (B-1) at
    p+1 ..] ([#1426] "Target feature taps": anchor = bonus token at p,
    remaining rows the mask token; "Drafter runtime": 5 dense layers, GQA,
    full-head NeoX RoPE, non-causal block attention, SwiGLU MLP, target LM
    head, greedy proposal).

    Per layer, in the stage order of [#1426] "Parity validation":
      xn = rmsnorm(x); q, k, v = W xn; q, k per-head normed; RoPE at p + i;
      block K/V written to positions [p, p+B); attention over positions
      [lo, p+B), lo = 0 or, with an attention window W, max(0, p + B - W);
      x += W_o attn; x += W_down(silu(W_gate xn2) * W_up xn2).
    Then the final norm, the LM head on rows 1..B-1 and their argmax.
    """
    cfg = model.cfg
    B, p = int(block_len), int(anchor_pos)
    if not (2 <= B):
        raise ValueError("block_len must be >= 2")
    if state.window == 0 and p + B > state.capacity:
        raise IndexError("anchor_pos + block_len exceeds the state's capacity")
    lo = max(0, p + B - state.window) if state.window > 0 else 0
    d, nq, nkv = cfg.head_dim, cfg.n_q_heads, cfg.n_kv_heads
    toks = np.full(B, cfg.mask_token_id, dtype=np.int64)
    toks[0] = anchor_tok
    pos = p + np.arange(B, dtype=np.int64)
    x = model.embed_rows(toks)
    stages: Dict[str, np.ndarray] = {}
    for l in range(cfg.n_layers):
        pre = f"layers.{l}."
        xn = rmsnorm(x, model.vec(pre + "attn_norm"), cfg.norm_eps)
        q = (xn @ model.mat(pre + "wq").T).reshape(B, nq, d)
        q = rmsnorm(q, model.vec(pre + "q_norm"), cfg.norm_eps)
        q = rope_neox(q, pos[:, None], cfg.rope_theta)
        k, v = project_kv(model, l, xn, pos)
        state.write(l, pos, k, v)
        kc, vc = state.keys(l, p + B, lo)
        a = attention(q, kc, vc, 1.0 / math.sqrt(d))
        x = x + a.reshape(B, nq * d) @ model.mat(pre + "wo").T
        if trace:
            stages[pre + "q"] = q
            stages[pre + "attn"] = a
            stages[pre + "x_attn"] = x.copy()
        xn2 = rmsnorm(x, model.vec(pre + "mlp_norm"), cfg.norm_eps)
        g = xn2 @ model.mat(pre + "w_gate").T
        u = xn2 @ model.mat(pre + "w_up").T
        x = x + (silu(g) * u) @ model.mat(pre + "w_down").T
        if trace:
            stages[pre + "x_mlp"] = x.copy()
    hf = rmsnorm(x, model.vec("final_norm"), cfg.norm_eps)
    logits = hf[1:] @ model.head().T
    if not np.all(np.isfinite(logits)):
        raise FloatingPointError("non-finite logits")
    drafts = np.argmax(logits, axis=-1).astype(np.int32)
    part = np.partition(logits, -2, axis=-1)
    gap = part[:, -1] - part[:, -2]
    return DraftResult(drafts, hf, logits, gap, stages if trace else None, draft_probs(logits))


def draft_probs(logits) -> np.ndarray:
    """Softmax probability of each row's argmax: exp(max) / sum_v exp(l_v)
    = 1 / sum_v exp(l_v - max), float64."""
    logits = np.asarray(logits, dtype=np.float64)
    mx = logits.max(axis=-1, keepdims=True)
    return 1.0 / np.exp(logits - mx).sum(axis=-1)


def gate(drafts, probs, floor: float) -> np.ndarray:
    """The drafts a block offers under the confidence floor: the prefix
    before the first draft with probability < floor; the rest become -1
    (not offered, so acceptance stops there)."""
    out = np.array(drafts, dtype=np.int32, copy=True)
    low = np.nonzero(np.asarray(probs) < floor)[0]
    if low.size:
        out[low[0]:] = -1
    return out


# ----------------------------------------------------------------------------
# step (5): greedy acceptance
# ----------------------------------------------------------------------------

def accept(drafts, target_ids, block_len: int):
    """Greedy acceptance of one verify window [anchor, B-1 candidates]
    ([#1426] "Speculative decode integration"; [#366] "Verification and state
    management": full, partial and first-candidate rejection).

    target_ids[j] is the verifier's argmax after window row j (B entries).
    Returns (n, bonus): n = the number of leading candidates with
    drafts[j] == target_ids[j]; bonus = target_ids[n], the verifier's own
    continuation token, committed after the n accepted candidates.
    """
    n = 0
    while n < block_len - 1 and int(drafts[n]) == int(target_ids[n]):
        n += 1
    return n, int(target_ids[n])

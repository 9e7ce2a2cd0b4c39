"""Seeded synthetic inputs for the DFlash block-draft pass.

This module produces *inputs only*: a random drafter checkpoint in the storage
formats the drafter consumes (BF16 bit patterns and GGUF-style 32-weight
quantised blocks), target feature taps, pre-filled FP16 context K/V, token ids
and synthetic verifier ids.  It holds none of the draft pass's arithmetic:
no normalisation, projection, rotary embedding, attention, dequantisation or
argmax lives here.  Both the CPU oracle (tests) and the CUDA path (through
the C ABI) are fed from these generators.

The geometry is the one the DeepSpec DFlash drafter is described with on
"#1426 dflash: experimental standalone DeepSpec DFlash block drafter",
section "Drafter runtime": 5 dense layers, hidden 2560, 24 Q / 2 KV heads,
head dim 256, MLP 7680, NeoX RoPE theta 1e7, five 2560-wide target taps.
There are no trained weights here; every tensor is drawn from a seeded RNG
with the distributions stated per workload (weights N(0, 0.02), norm weights
1 + N(0, 0.1), taps N(0, 1)).
"""
from __future__ import annotations

import concurrent.futures as _cf
import dataclasses
import os
from typing import Dict, List, Optional, Tuple

import numpy as np

WEIGHT_TYPES = ("bf16", "q8_0", "q5_0", "q4_0")
# Bytes per 32-weight block of each GGUF-style type: FP16 scale + codes
# (+ 4 bytes of fifth bits for Q5_0).
BLOCK_BYTES = {"q8_0": 34, "q5_0": 22, "q4_0": 18}


@dataclasses.dataclass(frozen=True)
class DraftConfig:
    name: str
    n_layers: int
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    intermediate: int
    vocab: int
    n_taps: int = 5
    rope_theta: float = 1e7
    norm_eps: float = 1e-6
    weight_type: str = "bf16"
    ctx: int = 64          # anchor position p = number of context positions
    block: int = 4         # block rows B (anchor + B-1 mask rows)
    n_seq: int = 1
    fuse_per_cycle: int = 0  # positions fused each cycle (long-context workload)
    attn_window: int = 0     # drafter attention window in positions (0: the whole context)

    @property
    def mask_token_id(self) -> int:
        return self.vocab - 1

    @property
    def tap_width(self) -> int:
        return self.n_taps * self.hidden

    def matrix_shapes(self) -> Dict[str, Tuple[int, int]]:
        """Name -> (out_features, in_features) of the 36 backbone matrices
        (fc + per layer q, k, v, o, gate, up, down)."""
        H, d = self.hidden, self.head_dim
        s = {"fc": (H, self.tap_width)}
        for l in range(self.n_layers):
            s[f"layers.{l}.wq"] = (self.n_q_heads * d, H)
            s[f"layers.{l}.wk"] = (self.n_kv_heads * d, H)
            s[f"layers.{l}.wv"] = (self.n_kv_heads * d, H)
            s[f"layers.{l}.wo"] = (H, self.n_q_heads * d)
            s[f"layers.{l}.w_gate"] = (self.intermediate, H)
            s[f"layers.{l}.w_up"] = (self.intermediate, H)
            s[f"layers.{l}.w_down"] = (H, self.intermediate)
        return s

    def norm_shapes(self) -> Dict[str, int]:
        H, d = self.hidden, self.head_dim
        s = {"hidden_norm": H}
        for l in range(self.n_layers):
            s[f"layers.{l}.attn_norm"] = H
            s[f"layers.{l}.q_norm"] = d
            s[f"layers.{l}.k_norm"] = d
            s[f"layers.{l}.mlp_norm"] = H
        s["final_norm"] = H
        return s

    def tensor_names(self) -> List[str]:
        """The drafter's own tensors (no embedding / LM head), in a fixed order."""
        names = ["fc", "hidden_norm"]
        for l in range(self.n_layers):
            names += [f"layers.{l}.{t}" for t in
                      ("attn_norm", "wq", "wk", "wv", "q_norm", "k_norm", "wo",
                       "mlp_norm", "w_gate", "w_up", "w_down")]
        names.append("final_norm")
        return names

    def with_(self, **kw) -> "DraftConfig":
        return dataclasses.replace(self, **kw)


_FULL = dict(n_layers=5, hidden=2560, n_q_heads=24, n_kv_heads=2, head_dim=256,
             intermediate=7680, vocab=151936)

CONFIGS: Dict[str, DraftConfig] = {
    # tiny DFlash pass: 2 layers, hidden 256, 4Q/1KV x 64, MLP 768, vocab 1024,
    # context 64, block 4.
    "tiny": DraftConfig("tiny", n_layers=2, hidden=256, n_q_heads=4, n_kv_heads=1,
                        head_dim=64, intermediate=768, vocab=1024, ctx=64, block=4),
    # full DFlash shape, BF16 backbone, 8K context, block 8.
    "full_bf16": DraftConfig("full_bf16", **_FULL, ctx=8192, block=8),
    "full_q8_0": DraftConfig("full_q8_0", **_FULL, weight_type="q8_0", ctx=8192, block=8),
    "full_q5_0": DraftConfig("full_q5_0", **_FULL, weight_type="q5_0", ctx=8192, block=8),
    "full_q4_0": DraftConfig("full_q4_0", **_FULL, weight_type="q4_0", ctx=8192, block=8),
    # long context: 262144 resident positions, fuse 8 new positions per cycle.
    "long_q8_0": DraftConfig("long_q8_0", **_FULL, weight_type="q8_0", ctx=262144,
                             block=8, fuse_per_cycle=8),
    # batched serving mix: 16 sequences, ctx U[2048, 32768], block U{2..8}.
    "batched_q4_0": DraftConfig("batched_q4_0", **_FULL, weight_type="q4_0",
                                ctx=32768, block=8, n_seq=16),
}


# ----------------------------------------------------------------------------
# storage formats
# ----------------------------------------------------------------------------

def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest BF16 (ties to even); return uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    bias = ((u >> 16) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> 16).astype(np.uint16)


def bf16_bits_as_f32(bits: np.ndarray) -> np.ndarray:
    """Widen BF16 bit patterns to float32 (exact)."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _signed_absmax(b: np.ndarray) -> np.ndarray:
    idx = np.argmax(np.abs(b), axis=-1)
    return np.take_along_axis(b, idx[..., None], axis=-1)[..., 0]


def quantize_gguf(w: np.ndarray, wtype: str) -> np.ndarray:
    """Pack a float matrix [N, K] (K % 32 == 0) into GGUF-style blocks.

    Byte layout per 32-weight block (the public GGUF block formats):
      q8_0: f16 d, int8 q[32]                          value = d * q
      q4_0: f16 d, u8 qs[16]   (low nibble j, high j+16) value = d * (q - 8)
      q5_0: f16 d, u8 qh[4] (bit j = fifth bit of j), u8 qs[16]
                                                        value = d * (q - 16)
    Blocks run along K inside each row; rows are consecutive.  This is the
    synthetic quantiser that turns the seeded BF16 weights into the quantised
    checkpoint; it is input production, not part of the draft pass.
    """
    w = np.asarray(w, dtype=np.float32)
    n, k = w.shape
    assert k % 32 == 0
    b = w.reshape(n, k // 32, 32)
    if wtype == "q8_0":
        amax = np.abs(b).max(axis=-1)
        d = amax / 127.0
        inv = np.where(d > 0, 1.0 / np.where(d > 0, d, 1.0), 0.0).astype(np.float32)
        q = np.clip(np.rint(b * inv[..., None]), -127, 127).astype(np.int8)
        out = np.empty((n, k // 32, 34), dtype=np.uint8)
        out[..., 0:2] = d.astype(np.float16)[..., None].view(np.uint8)
        out[..., 2:34] = q.view(np.uint8)
    elif wtype in ("q4_0", "q5_0"):
        levels, off = (16, 8) if wtype == "q4_0" else (32, 16)
        m = _signed_absmax(b)
        d = m / -float(off)
        inv = np.where(d != 0, 1.0 / np.where(d != 0, d, 1.0), 0.0).astype(np.float32)
        q = np.clip(np.floor(b * inv[..., None] + (off + 0.5)), 0, levels - 1).astype(np.uint8)
        lo = q[..., :16] & 0xF
        hi = q[..., 16:] & 0xF
        qs = (lo | (hi << 4)).astype(np.uint8)
        d16 = d.astype(np.float16)[..., None].view(np.uint8)
        if wtype == "q4_0":
            out = np.empty((n, k // 32, 18), dtype=np.uint8)
            out[..., 0:2] = d16
            out[..., 2:18] = qs
        else:
            fifth = (q >> 4).astype(np.uint32) & 1
            qh = np.zeros((n, k // 32), dtype=np.uint32)
            for j in range(32):
                qh |= fifth[..., j] << np.uint32(j)
            out = np.empty((n, k // 32, 22), dtype=np.uint8)
            out[..., 0:2] = d16
            out[..., 2:6] = qh.astype("<u4")[..., None].view(np.uint8)
            out[..., 6:22] = qs
    else:
        raise ValueError(wtype)
    return out.reshape(n, (k // 32) * out.shape[-1])


# ----------------------------------------------------------------------------
# seeded generators
# ----------------------------------------------------------------------------

def _rng(seed: int, stream: int) -> np.random.Generator:
    return np.random.default_rng([int(seed), int(stream)])


def _normal_bf16(seed: int, stream: int, shape, std: float, mean: float = 0.0) -> np.ndarray:
    x = _rng(seed, stream).standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    if mean != 0.0:
        x += np.float32(mean)
    return to_bf16_bits(x)


def _threads() -> int:
    try:
        return max(1, min(16, len(os.sched_getaffinity(0))))
    except AttributeError:  # pragma: no cover
        return max(1, min(16, os.cpu_count() or 1))


def make_checkpoint(cfg: DraftConfig, seed: int = 0, with_target_tensors: bool = True,
                    threads: Optional[int] = None) -> Dict[str, np.ndarray]:
    """Seeded random drafter checkpoint.

    Returns name -> array.  Matrices are uint16 BF16 bits [out, in] when
    cfg.weight_type == "bf16", else uint8 GGUF block bytes [out, in/32*block].
    Norm vectors are uint16 BF16 bits.  With ``with_target_tensors`` the
    target's embedding and LM head (``embed``, ``head``: BF16 [vocab, hidden])
    are included too; the drafter borrows them and never owns them.

    The quantised checkpoints are the BF16 checkpoint of the same seed passed
    through :func:`quantize_gguf`, so all four weight types share one set of
    underlying values.
    """
    shapes = cfg.matrix_shapes()
    norms = cfg.norm_shapes()
    names = cfg.tensor_names()
    jobs = []
    for idx, name in enumerate(names):
        if name in shapes:
            jobs.append((name, idx, shapes[name], 0.02, 0.0))
        else:
            jobs.append((name, idx, (norms[name],), 0.1, 1.0))
    if with_target_tensors:
        jobs.append(("embed", 1000, (cfg.vocab, cfg.hidden), 0.02, 0.0))
        jobs.append(("head", 1001, (cfg.vocab, cfg.hidden), 0.02, 0.0))

    def run(job):
        name, idx, shape, std, mean = job
        bits = _normal_bf16(seed, idx, shape, std, mean)
        if cfg.weight_type != "bf16" and name in shapes:
            return name, quantize_gguf(bf16_bits_as_f32(bits), cfg.weight_type)
        return name, bits

    out: Dict[str, np.ndarray] = {}
    nthreads = threads or _threads()
    # big tensors first so the pool stays busy
    jobs.sort(key=lambda j: -int(np.prod(j[2])))
    with _cf.ThreadPoolExecutor(max_workers=nthreads) as ex:
        for name, arr in ex.map(run, jobs):
            out[name] = arr
    return out


def make_taps(cfg: DraftConfig, n: int, seed: int = 0, stream: int = 0) -> np.ndarray:
    """Target feature taps for n positions: BF16 bits [n, n_taps * hidden],
    values N(0, 1); the five taps of one position are concatenated in tap
    (boundary) order."""
    return _normal_bf16(seed, 5000 + stream, (n, cfg.tap_width), 1.0)


def make_kv_fill(cfg: DraftConfig, n_pos: int, seed: int = 0, slot: int = 0,
                 threads: Optional[int] = None) -> List[Tuple[np.ndarray, np.ndarray]]:
    """Pre-filled context K/V for positions [0, n_pos): per layer (K, V), each
    float16 [n_kv_heads, n_pos, head_dim] with values N(0, 1).  Stands in for
    a context too long to build by fusion in the oracle."""
    shape = (cfg.n_kv_heads, n_pos, cfg.head_dim)

    def run(j):
        x = _rng(seed, 7000 + 1000 * slot + j).standard_normal(size=shape, dtype=np.float32)
        return x.astype(np.float16)

    with _cf.ThreadPoolExecutor(max_workers=threads or _threads()) as ex:
        arrs = list(ex.map(run, range(2 * cfg.n_layers)))
    return [(arrs[2 * l], arrs[2 * l + 1]) for l in range(cfg.n_layers)]


def make_token_ids(cfg: DraftConfig, n: int, seed: int = 0, stream: int = 0) -> np.ndarray:
    """Uniform token ids in [0, vocab - 1) (the last id is the mask token)."""
    return _rng(seed, 9000 + stream).integers(0, cfg.vocab - 1, size=n, dtype=np.int64).astype(np.int32)


def make_target_ids(drafts: np.ndarray, vocab: int, seed: int = 0, p_agree: float = 0.7,
                    agree_prefix: Optional[int] = None, stream: int = 0) -> np.ndarray:
    """Synthetic verifier argmax ids for one window of B = len(drafts) + 1 rows.

    ``drafts`` are the B-1 candidate ids being verified (any source).  With
    ``agree_prefix = m`` the first m ids copy the drafts, id m differs from
    draft m (when m < B-1) and the rest are uniform; otherwise each id copies
    its draft with probability ``p_agree`` and is a different uniform id
    otherwise.  The last id (the verifier's continuation after the final
    candidate) is always uniform.
    """
    drafts = np.asarray(drafts, dtype=np.int64)
    rng = _rng(seed, 11000 + stream)
    nb = drafts.shape[0] + 1
    tgt = rng.integers(0, vocab, size=nb, dtype=np.int64)
    for j in range(nb - 1):
        if agree_prefix is not None:
            agree = j < agree_prefix
            force_diff = j == agree_prefix
        else:
            agree = rng.random() < p_agree
            force_diff = not agree
        if agree:
            tgt[j] = drafts[j]
        elif force_diff and tgt[j] == drafts[j]:
            tgt[j] = (drafts[j] + 1 + rng.integers(0, vocab - 1)) % vocab
    return tgt.astype(np.int32)


def batched_mix(cfg: DraftConfig, seed: int = 0) -> Tuple[np.ndarray, np.ndarray]:
    """Per-sequence context lengths U[2048, 32768] and block sizes U{2..8}
    for the batched serving mix."""
    rng = _rng(seed, 13000)
    ctx = rng.integers(2048, 32768 + 1, size=cfg.n_seq).astype(np.int32)
    blk = rng.integers(2, 8 + 1, size=cfg.n_seq).astype(np.int32)
    return ctx, blk

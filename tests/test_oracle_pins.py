"""Pins for the CPU oracle: each check ties the oracle to something other than
itself -- the pages' printed geometry and acceptance cases, closed forms,
hand-packed GGUF blocks, textbook special cases, invariants and brute force
on tiny inputs -- so that a dropped term, a wrong sign or index, or a
transposed operand in the oracle fails at least one of them.  CPU only."""
import json
import math
import os

import numpy as np
import pytest

import dflash_synth as synth
from oracle import dflash_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------------------
# geometry printed on the pages
# ---------------------------------------------------------------------------

def test_geometry_matches_pages():
    g = _golden("geometry.json")
    cfg = synth.CONFIGS["full_bf16"]
    assert (cfg.n_layers, cfg.hidden, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim,
            cfg.intermediate) == (g["n_layers"], g["hidden"], g["n_q_heads"],
                                  g["n_kv_heads"], g["head_dim"], g["intermediate"])
    assert cfg.rope_theta == g["rope_theta"]
    assert 1.0 / math.sqrt(cfg.head_dim) == g["attention_scale"]
    assert len(g["tap_boundaries"]) == cfg.n_taps
    assert [b - 1 for b in g["tap_boundaries"]] == g["trained_tap_layers"]
    assert cfg.tap_width == cfg.n_taps * g["tap_width"]
    # the pages' parameter count of the drafter (about 498M, embedding and LM
    # head excluded): the 36 backbone matrices.
    n_params = sum(a * b for a, b in cfg.matrix_shapes().values())
    assert n_params == 498_073_600
    assert round(n_params / 1e6) == g["params_millions"]
    n_norm = sum(cfg.norm_shapes().values())
    assert round((n_params + n_norm) / 1e6) == g["params_millions"]
    # "validates all 58 expected tensors": fc, hidden norm, 5 x 11, final norm.
    assert len(cfg.tensor_names()) == g["n_tensors"]
    assert len(cfg.matrix_shapes()) == 36
    assert g["spec_max"] - 1 == g["max_candidates"]


# ---------------------------------------------------------------------------
# formats: BF16, FP16, GGUF blocks
# ---------------------------------------------------------------------------

def test_decode_bf16_known_bits():
    bits = np.array([0x3F80, 0xBF80, 0x4049, 0x0000, 0x8000, 0x3E00, 0x7F7F], np.uint16)
    want = [1.0, -1.0, 3.140625, 0.0, -0.0, 0.125, 3.3895313892515355e38]
    got = O.decode_bf16(bits)
    assert got.dtype == np.float64
    assert list(got) == want


def test_round_f16_ties_to_even():
    # 1 + 2^-11 is halfway between 1 and 1 + 2^-10: ties to even -> 1.
    # 1 + 3*2^-11 is halfway between 1 + 2^-10 and 1 + 2^-9: -> 1 + 2^-9.
    x = np.array([1 + 2 ** -11, 1 + 3 * 2 ** -11, 65504.0, 2 ** -24])
    got = O.round_f16(x).astype(np.float64)
    assert list(got) == [1.0, 1 + 2 ** -9, 65504.0, 2 ** -24]


def _blk(d_bits, payload):
    return np.array([d_bits & 0xFF, d_bits >> 8] + list(payload), np.uint8)


def test_dequant_q8_0_hand_packed():
    # d = 0.5 (fp16 0x3800), q[j] = j - 16  ->  w[j] = 0.5 * (j - 16)
    b0 = _blk(0x3800, [(j - 16) & 0xFF for j in range(32)])
    # d = 0.125 (0x3000), q = 127, -127, -128, 1, then zeros
    q1 = [127, -127, -128, 1] + [0] * 28
    b1 = _blk(0x3000, [q & 0xFF for q in q1])
    w = O.dequantize(np.concatenate([b0, b1])[None, :], "q8_0", 1, 64)[0]
    assert list(w[:32]) == [0.5 * (j - 16) for j in range(32)]
    assert list(w[32:36]) == [15.875, -15.875, -16.0, 0.125]
    assert np.all(w[36:] == 0)


def test_dequant_q4_0_hand_packed():
    # d = 0.25 (0x3400); qs[j] = j | (15 - j) << 4:
    # element j has code j, element j + 16 has code 15 - j; offset 8.
    blk = _blk(0x3400, [j | ((15 - j) << 4) for j in range(16)])
    w = O.dequantize(blk[None, :], "q4_0", 1, 32)[0]
    assert list(w[:16]) == [0.25 * (j - 8) for j in range(16)]
    assert list(w[16:]) == [0.25 * (7 - j) for j in range(16)]


def test_dequant_q5_0_hand_packed():
    # d = 2.0 (0x4000); qh = 0x0000FFFF: fifth bit set for elements 0..15;
    # qs[j] = j | j << 4  ->  element j: 16 + j, element j + 16: j; offset 16.
    b0 = _blk(0x4000, [0xFF, 0xFF, 0x00, 0x00] + [j | (j << 4) for j in range(16)])
    # d = 1.0 (0x3C00); qh = 0x80000001 (little endian bytes 01 00 00 80):
    # only elements 0 and 31 have the fifth bit; all nibbles 0.
    b1 = _blk(0x3C00, [0x01, 0x00, 0x00, 0x80] + [0] * 16)
    w = O.dequantize(np.concatenate([b0, b1])[None, :], "q5_0", 1, 64)[0]
    assert list(w[:16]) == [2.0 * j for j in range(16)]
    assert list(w[16:32]) == [2.0 * (j - 16) for j in range(16)]
    assert w[32] == 0.0 and w[63] == 0.0
    assert np.all(w[33:63] == -16.0)


@pytest.mark.parametrize("wtype", ["q8_0", "q5_0", "q4_0"])
def test_dequant_round_trip_on_grid(wtype):
    """Values already on a block's grid survive the (independent) synthetic
    quantiser and the oracle's dequantiser unchanged, row by row and block by
    block -- a swapped nibble, a shifted bit or a misplaced scale breaks it."""
    rng = np.random.default_rng(3)
    n, k = 6, 128
    lo, hi, off = {"q8_0": (-127, 127, 0), "q4_0": (0, 15, 8), "q5_0": (0, 31, 16)}[wtype]
    q = rng.integers(lo, hi + 1, size=(n, k // 32, 32))
    # put the block's extreme on the grid so the quantiser recovers this d:
    # code 127 for Q8_0 (amax / 127), code 0 (value -offset * d) otherwise
    q[..., 5] = 127 if wtype == "q8_0" else 0
    d = (2.0 ** rng.integers(-8, -2, size=(n, k // 32))).astype(np.float64)
    if wtype == "q8_0":
        w = d[..., None] * q
    else:
        w = d[..., None] * (q - off)
    w = w.reshape(n, k).astype(np.float32)
    raw = synth.quantize_gguf(w, wtype)
    back = O.dequantize(raw, wtype, n, k)
    assert np.array_equal(back, w.astype(np.float64))


# ---------------------------------------------------------------------------
# RMSNorm
# ---------------------------------------------------------------------------

def test_rmsnorm_hand_case():
    x = np.array([3.0, 4.0])
    got = O.rmsnorm(x, np.ones(2), 0.0)
    r = math.sqrt((9 + 16) / 2)
    assert np.allclose(got, [3 / r, 4 / r], rtol=0, atol=1e-15)
    w = np.array([2.0, -0.5])
    assert np.allclose(O.rmsnorm(x, w, 0.0), [6 / r, -2 / r], atol=1e-15)


def test_rmsnorm_unit_rms_and_scale_invariance():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((5, 64)) * 7
    y = O.rmsnorm(x, np.ones(64), 1e-6)
    assert np.allclose(np.sqrt(np.mean(y * y, -1)), 1.0, atol=1e-7)
    assert np.allclose(O.rmsnorm(3.5 * x, np.ones(64), 0.0), O.rmsnorm(x, np.ones(64), 0.0), atol=1e-14)
    # eps enters under the root: a zero row stays zero, tiny rows are damped
    assert np.all(O.rmsnorm(np.zeros(8), np.ones(8), 1e-6) == 0)
    t = O.rmsnorm(np.full(4, 1e-3), np.ones(4), 1e-6)
    assert np.allclose(t, 1e-3 / math.sqrt(1e-6 + 1e-6))


# ---------------------------------------------------------------------------
# NeoX RoPE
# ---------------------------------------------------------------------------

def test_rope_hand_case_neox_pairs():
    # d = 4, theta = 100: inv_freq = [100^0, 100^-0.5] = [1, 0.1]; pairs
    # (x0, x2) rotated by pos * 1 and (x1, x3) by pos * 0.1.
    x = np.array([1.0, 2.0, 3.0, 4.0])
    pos = 2.0
    a0, a1 = 2.0, 0.2
    want = [1 * math.cos(a0) - 3 * math.sin(a0),
            2 * math.cos(a1) - 4 * math.sin(a1),
            3 * math.cos(a0) + 1 * math.sin(a0),
            4 * math.cos(a1) + 2 * math.sin(a1)]
    assert np.allclose(O.rope_neox(x, pos, 100.0), want, rtol=0, atol=1e-14)


def test_rope_identity_norm_and_relative():
    rng = np.random.default_rng(1)
    d = 64
    q = rng.standard_normal(d)
    k = rng.standard_normal(d)
    assert np.array_equal(O.rope_neox(q, 0, 1e7), q)
    r = O.rope_neox(q, 12345, 1e7)
    pair_norm = lambda v: v[: d // 2] ** 2 + v[d // 2:] ** 2
    assert np.allclose(pair_norm(r), pair_norm(q), atol=1e-12)
    # <R(m) q, R(n) k> depends only on m - n
    dots = [O.rope_neox(q, m, 1e7) @ O.rope_neox(k, m - 37, 1e7) for m in (37, 500, 262143)]
    assert np.allclose(dots, dots[0], atol=1e-9)
    assert not np.isclose(O.rope_neox(q, 40, 1e7) @ O.rope_neox(k, 0, 1e7), dots[0])


def test_rope_full_head_frequencies():
    # The last pair (i = d/2 - 1) turns at theta^(-(d-2)/d); position 1.
    d, theta = 8, 1e7
    x = np.zeros(d)
    x[d // 2 - 1] = 1.0
    y = O.rope_neox(x, 1, theta)
    ang = theta ** (-(d - 2) / d)
    assert np.isclose(y[d // 2 - 1], math.cos(ang)) and np.isclose(y[d - 1], math.sin(ang))


# ---------------------------------------------------------------------------
# attention
# ---------------------------------------------------------------------------

def test_attention_one_key_returns_v():
    rng = np.random.default_rng(2)
    q = rng.standard_normal((3, 4, 16))
    k = rng.standard_normal((1, 2, 16))
    v = rng.standard_normal((1, 2, 16))
    out = O.attention(q, k, v, 0.25)
    for h in range(4):
        assert np.allclose(out[:, h, :], v[0, h // 2, :], atol=1e-15)


def test_attention_two_keys_closed_form_and_scale():
    q = np.zeros((1, 1, 4)); q[0, 0, 0] = 2.0
    k = np.zeros((2, 1, 4)); k[0, 0, 0] = 1.0; k[1, 0, 0] = -1.0
    v = np.zeros((2, 1, 4)); v[0, 0, 1] = 1.0; v[1, 0, 2] = 1.0
    s = 0.5
    e0, e1 = math.exp(2.0 * s), math.exp(-2.0 * s)
    out = O.attention(q, k, v, s)[0, 0]
    assert np.allclose(out, [0, e0 / (e0 + e1), e1 / (e0 + e1), 0], atol=1e-15)


def test_attention_rows_sum_to_one():
    rng = np.random.default_rng(4)
    q = rng.standard_normal((5, 6, 8)) * 3
    k = rng.standard_normal((11, 3, 8))
    v = np.ones((11, 3, 8))
    assert np.allclose(O.attention(q, k, v, 0.3), 1.0, atol=1e-14)


def test_attention_gqa_equals_repeated_mha():
    rng = np.random.default_rng(5)
    nq, nkv, d, T = 12, 2, 16, 9
    q = rng.standard_normal((4, nq, d))
    k = rng.standard_normal((T, nkv, d))
    v = rng.standard_normal((T, nkv, d))
    rep = nq // nkv
    k_mha = np.repeat(k, rep, axis=1)  # head h gets kv head h // rep
    v_mha = np.repeat(v, rep, axis=1)
    assert np.allclose(O.attention(q, k, v, 0.25), O.attention(q, k_mha, v_mha, 0.25), atol=1e-14)


def test_attention_brute_force_tiny():
    rng = np.random.default_rng(6)
    R, nq, nkv, d, T = 3, 4, 2, 5, 7
    q = rng.standard_normal((R, nq, d))
    k = rng.standard_normal((T, nkv, d))
    v = rng.standard_normal((T, nkv, d))
    s = 1 / math.sqrt(d)
    got = O.attention(q, k, v, s)
    for r in range(R):
        for h in range(nq):
            g = h // (nq // nkv)
            sc = [sum(q[r, h, i] * k[t, g, i] for i in range(d)) * s for t in range(T)]
            m = max(sc)
            e = [math.exp(x - m) for x in sc]
            z = sum(e)
            for i in range(d):
                want = sum(e[t] * v[t, g, i] for t in range(T)) / z
                assert abs(got[r, h, i] - want) < 1e-12


def test_attention_split_keys_lse_merge():
    """Attention over [A | B] equals the log-sum-exp merge of the two halves
    (the identity a split-context kernel relies on)."""
    rng = np.random.default_rng(7)
    q = rng.standard_normal((2, 2, 8))
    k = rng.standard_normal((10, 1, 8))
    v = rng.standard_normal((10, 1, 8))
    s = 0.35
    full = O.attention(q, k, v, s)
    parts = []
    for lo, hi in ((0, 6), (6, 10)):
        sc = np.einsum("rhd,td->rht", q, k[lo:hi, 0]) * s
        m = sc.max(-1)
        e = np.exp(sc - m[..., None])
        parts.append((m, e.sum(-1), np.einsum("rht,td->rhd", e, v[lo:hi, 0])))
    M = np.maximum(parts[0][0], parts[1][0])
    L = sum(l * np.exp(m - M) for m, l, _ in parts)
    Ov = sum(o * np.exp(m - M)[..., None] for m, _, o in parts)
    assert np.allclose(Ov / L[..., None], full, atol=1e-14)


def test_attention_is_non_causal():
    rng = np.random.default_rng(8)
    q = rng.standard_normal((4, 2, 8))
    k = rng.standard_normal((4, 1, 8))
    v = rng.standard_normal((4, 1, 8))
    a = O.attention(q, k, v, 0.3)
    k2 = k.copy(); k2[3] += 1.0  # change the LAST key only
    b = O.attention(q, k2, v, 0.3)
    assert not np.allclose(a[0], b[0])  # row 0 sees key 3


# ---------------------------------------------------------------------------
# SwiGLU
# ---------------------------------------------------------------------------

def test_silu_closed_form():
    for x in (-3.0, -0.5, 0.0, 0.7, 4.0):
        assert abs(float(O.silu(x)) - x / (1 + math.exp(-x))) < 1e-15
    assert float(O.silu(0.0)) == 0.0


# ---------------------------------------------------------------------------
# acceptance
# ---------------------------------------------------------------------------

def test_accept_pages_three_cases():
    g = _golden("accept_cases.json")
    tgt = g["reference_continuation"]
    for c in g["cases"]:
        n, bonus = O.accept(c["drafts"], tgt, len(c["drafts"]) + 1)
        assert (n, bonus) == (c["accept_len"], c["bonus"]), c["name"]


def test_accept_brute_force():
    rng = np.random.default_rng(9)
    for _ in range(500):
        B = int(rng.integers(2, 9))
        drafts = rng.integers(0, 4, size=B - 1)
        tgt = rng.integers(0, 4, size=B)
        n, bonus = O.accept(drafts, tgt, B)
        # longest m with all(drafts[:m] == tgt[:m])
        best = max(m for m in range(B) if all(drafts[j] == tgt[j] for j in range(m)))
        assert n == best and bonus == tgt[n]


# ---------------------------------------------------------------------------
# whole-pass special cases and invariants (tiny shapes)
# ---------------------------------------------------------------------------

def _tiny(**kw):
    return synth.CONFIGS["tiny"].with_(**kw)


def _zero_matrix(ckpt, name, cfg):
    n, k = cfg.matrix_shapes()[name]
    if cfg.weight_type == "bf16":
        ckpt[name] = np.zeros((n, k), np.uint16)
    else:
        ckpt[name] = synth.quantize_gguf(np.zeros((n, k), np.float32), cfg.weight_type)


@pytest.mark.parametrize("wtype", ["bf16", "q4_0"])
def test_pass_without_sublayers_reduces_to_head_argmax(wtype):
    """With every W_o and W_down zero the residual stream stays the embedding,
    so the final hidden is rmsnorm(E[token]) * final_norm and each draft is
    the brute-force argmax of the LM head over it."""
    cfg = _tiny(weight_type=wtype)
    ck = synth.make_checkpoint(cfg, seed=11)
    for l in range(cfg.n_layers):
        _zero_matrix(ck, f"layers.{l}.wo", cfg)
        _zero_matrix(ck, f"layers.{l}.w_down", cfg)
    m = O.Model(cfg, ck)
    st = O.State(cfg, 128)
    taps = synth.make_taps(cfg, cfg.ctx, seed=11)
    O.fuse_context(m, st, taps, np.arange(cfg.ctx))
    res = O.draft_block(m, st, anchor_tok=17, anchor_pos=cfg.ctx, block_len=4)
    e = O.decode_bf16(ck["embed"][[17, cfg.mask_token_id]])
    fw = O.decode_bf16(ck["final_norm"])
    for row, tok in ((0, 0), (1, 1), (3, 1)):
        x = e[tok]
        want = x / math.sqrt(float(np.mean(x * x)) + cfg.norm_eps) * fw
        assert np.allclose(res.final_hidden[row], want, atol=1e-12)
    head = O.decode_bf16(ck["head"])
    for j in range(3):
        scores = [float(head[v] @ res.final_hidden[j + 1]) for v in range(cfg.vocab)]
        best = max(range(cfg.vocab), key=lambda v: (scores[v], -v))
        assert res.drafts[j] == best


def test_fusion_selects_taps_in_order():
    """With W_fc = [0 .. I .. 0] selecting tap t, h_ctx is rmsnorm(tap_t)."""
    cfg = _tiny()
    ck = synth.make_checkpoint(cfg, seed=12, with_target_tensors=False)
    H = cfg.hidden
    m_taps = synth.make_taps(cfg, 3, seed=12)
    for t in (0, 3):
        fc = np.zeros((H, cfg.tap_width), np.float32)
        fc[:, t * H:(t + 1) * H] = np.eye(H, dtype=np.float32)
        ck["fc"] = synth.to_bf16_bits(fc)
        m = O.Model(cfg, ck)
        h = O.fuse_hidden(m, m_taps)
        tap = O.decode_bf16(m_taps)[:, t * H:(t + 1) * H]
        hn = O.decode_bf16(ck["hidden_norm"])
        want = tap / np.sqrt(np.mean(tap * tap, -1, keepdims=True) + cfg.norm_eps) * hn
        assert np.allclose(h, want, atol=1e-12)


def test_pass_block_rows_see_later_rows():
    """Non-causal block: row 1's final hidden depends on whether row 3 exists."""
    cfg = _tiny()
    ck = synth.make_checkpoint(cfg, seed=13)
    m = O.Model(cfg, ck)
    taps = synth.make_taps(cfg, cfg.ctx, seed=13)
    outs = {}
    for B in (3, 4):
        st = O.State(cfg, 128)
        O.fuse_context(m, st, taps, np.arange(cfg.ctx))
        outs[B] = O.draft_block(m, st, 5, cfg.ctx, B).final_hidden
    assert not np.allclose(outs[3][1], outs[4][1], atol=1e-6)


def test_context_keys_rotated_at_their_position():
    """Fusing the same taps at positions [0, n) and [S, S + n): un-rotating
    each stored key by its own position gives the same vector (to FP16
    rounding), so context keys carry absolute-position rotations."""
    cfg = _tiny()
    ck = synth.make_checkpoint(cfg, seed=14, with_target_tensors=False)
    m = O.Model(cfg, ck)
    n, S = 32, 1000
    taps = synth.make_taps(cfg, n, seed=14)
    st0 = O.State(cfg, n)
    st1 = O.State(cfg, S + n)
    O.fuse_context(m, st0, taps, np.arange(n))
    O.fuse_context(m, st1, taps, S + np.arange(n))
    p = np.arange(n)
    for l in range(cfg.n_layers):
        u0 = O.rope_neox(st0.K[l].astype(np.float64), -p[None, :], cfg.rope_theta)
        u1 = O.rope_neox(st1.K[l][:, S:].astype(np.float64), -(S + p)[None, :], cfg.rope_theta)
        assert np.allclose(u0, u1, atol=4e-3)
        assert np.array_equal(st0.V[l], st1.V[l][:, S:])
        assert np.array_equal(st1.held[l][S:], S + p) and (st1.held[l][:S] == -1).all()


def test_pass_position_shift_invariance():
    """The whole pass with every position (context cells and block rows)
    shifted by S agrees with the unshifted pass up to the FP16 rounding of
    the stored keys: q and k are both rotated at absolute positions, so only
    relative positions matter.  The shifted run sees the cells [S, S+n+B)
    through a state view whose cell i holds position S + i."""
    cfg = _tiny()
    ck = synth.make_checkpoint(cfg, seed=15)
    m = O.Model(cfg, ck)
    n, B, S = 24, 5, 4096
    taps = synth.make_taps(cfg, n, seed=15)
    st0 = O.State(cfg, n + 8)
    O.fuse_context(m, st0, taps, np.arange(n))
    r0 = O.draft_block(m, st0, 9, n, B)

    st1 = O.State(cfg, S + n + 8)
    O.fuse_context(m, st1, taps, S + np.arange(n))
    view = O.State(cfg, n + 8)
    view.K = [k[:, S:] for k in st1.K]
    view.V = [v[:, S:] for v in st1.V]
    view.held = [hh[S:] - S for hh in st1.held]
    orig = O.rope_neox
    O.rope_neox = lambda x, pos, theta: orig(x, np.asarray(pos) + S, theta)
    try:
        r1 = O.draft_block(m, view, 9, n, B)
    finally:
        O.rope_neox = orig
    rms = float(np.sqrt(np.mean(r0.final_hidden ** 2)))
    assert np.allclose(r0.final_hidden, r1.final_hidden, atol=1e-2 * rms)
    sure = r0.top2_gap > 1e-2
    assert sure.any()
    assert np.array_equal(r0.drafts[sure], r1.drafts[sure])


# ---------------------------------------------------------------------------
# attention window and ring-addressed cells
# ---------------------------------------------------------------------------

def _window_setup(seed, n, W, capacity, positions=None):
    cfg = _tiny(attn_window=W)
    ck = synth.make_checkpoint(cfg, seed=seed)
    m = O.Model(cfg, ck)
    taps = synth.make_taps(cfg, n, seed=seed)
    st = O.State(cfg, capacity)
    O.fuse_context(m, st, taps, np.arange(n) if positions is None else positions)
    return cfg, m, st, taps


def test_window_that_covers_the_context_changes_nothing():
    """A window at least as long as p + B attends to exactly the positions of
    the plain pass: results bit-identical to no window."""
    n, B = 40, 4
    cfg0 = _tiny()
    ck = synth.make_checkpoint(cfg0, seed=31)
    taps = synth.make_taps(cfg0, n, seed=31)
    res = []
    for W in (0, n + B, 128):
        cfg = cfg0.with_(attn_window=W)
        m = O.Model(cfg, ck)
        st = O.State(cfg, 128)
        O.fuse_context(m, st, taps, np.arange(n))
        res.append(O.draft_block(m, st, 5, n, B))
    for r in res[1:]:
        assert np.array_equal(r.final_hidden, res[0].final_hidden)
        assert np.array_equal(r.drafts, res[0].drafts)


def test_window_reads_exactly_the_last_w_positions():
    """With W < p + B the pass depends on positions [p + B - W, p + B) only:
    replacing every K/V cell of an older position by large noise leaves the
    result bit-identical, while replacing the one position just inside the
    window changes it (so the boundary is exact, not off by one)."""
    n, B, W = 48, 4, 20
    cfg, m, st, _ = _window_setup(32, n, W, 64)
    ref = O.draft_block(m, st, 5, n, B)
    lo = n + B - W
    rng = np.random.default_rng(32)
    noisy = O.State(cfg, 64)
    noisy.K = [k.copy() for k in st.K]
    noisy.V = [v.copy() for v in st.V]
    noisy.held = [h.copy() for h in st.held]
    for l in range(cfg.n_layers):
        noisy.K[l][:, :lo, :] = rng.normal(0, 50, noisy.K[l][:, :lo, :].shape).astype(np.float16)
        noisy.V[l][:, :lo, :] = rng.normal(0, 50, noisy.V[l][:, :lo, :].shape).astype(np.float16)
    out = O.draft_block(m, noisy, 5, n, B)
    assert np.array_equal(out.final_hidden, ref.final_hidden)
    inside = O.State(cfg, 64)
    inside.K = [k.copy() for k in st.K]
    inside.V = [v.copy() for v in st.V]
    inside.held = [h.copy() for h in st.held]
    for l in range(cfg.n_layers):
        inside.V[l][:, lo, :] = rng.normal(0, 50, inside.V[l][:, lo, :].shape).astype(np.float16)
    assert not np.array_equal(O.draft_block(m, inside, 5, n, B).final_hidden, ref.final_hidden)


def test_ring_cells_match_position_addressed_cells():
    """Fusing positions past the capacity of a ring state overwrites the
    cells of older positions (pos mod capacity); as long as the window fits
    the ring, the pass equals the same windowed pass over a state large
    enough to keep every position in its own cell."""
    n, B, W, C = 200, 4, 96, 128
    cfg, m, ring, taps = _window_setup(33, n, W, C)
    big = O.State(cfg.with_(attn_window=0), 256)
    big.window = W  # the same window over position-addressed cells
    O.fuse_context(m, big, taps, np.arange(n))
    r_ring = O.draft_block(m, ring, 7, n, B)
    r_big = O.draft_block(m, big, 7, n, B)
    assert np.array_equal(r_ring.final_hidden, r_big.final_hidden)
    assert np.array_equal(r_ring.drafts, r_big.drafts)
    # position 0 was evicted by position C: reading it fails hard
    with pytest.raises(ValueError):
        ring.keys(0, 1, 0)
    # cell n % C - 1 holds the last fused position, cell n % C the block's
    # anchor position written by the pass, cell (n + B) % C an older position
    assert ring.held[0][n % C - 1] == n - 1 and ring.held[0][n % C] == n
    assert ring.held[0][(n + B) % C] == n + B - C


# ---------------------------------------------------------------------------
# confidence gate (spec-min-p)
# ---------------------------------------------------------------------------

def test_draft_probs_closed_forms():
    """Uniform logits give 1/V; one logit ahead of V - 1 equal ones by delta
    gives 1 / (1 + (V - 1) e^-delta); a shift of every logit changes nothing;
    large logits (1e4) do not overflow."""
    V = 1000
    assert np.allclose(O.draft_probs(np.zeros((1, V))), 1.0 / V)
    for delta in (0.0, 0.5, 3.0, 40.0):
        row = np.zeros(V)
        row[17] = delta
        want = 1.0 / (1.0 + (V - 1) * math.exp(-delta))
        assert math.isclose(O.draft_probs(row[None])[0], want, rel_tol=1e-12)
    rng = np.random.default_rng(51)
    lg = rng.normal(0, 3, (4, V))
    assert np.allclose(O.draft_probs(lg), O.draft_probs(lg + 1e4), rtol=1e-9)


def test_draft_probs_brute_force():
    """Against exp(max) / sum of exp over a tiny vocabulary, element by element
    with math.exp, and in (0, 1] always."""
    rng = np.random.default_rng(52)
    lg = rng.normal(0, 2, (6, 7))
    for r in range(6):
        tot = sum(math.exp(v) for v in lg[r])
        assert math.isclose(O.draft_probs(lg[r:r + 1])[0], math.exp(lg[r].max()) / tot, rel_tol=1e-12)
    p = O.draft_probs(rng.normal(0, 5, (50, 64)))
    assert np.all(p > 0) and np.all(p <= 1)


def test_gate_prefix_rule():
    d = np.array([5, 9, 2, 7])
    p = np.array([0.9, 0.6, 0.4, 0.95])
    assert np.array_equal(O.gate(d, p, 0.0), d)          # floor 0 offers every draft
    assert np.array_equal(O.gate(d, p, 0.5), [5, 9, -1, -1])  # cut at the first low one, later ones too
    assert np.array_equal(O.gate(d, p, 0.6), [5, 9, -1, -1])  # equal to the floor is offered
    assert np.array_equal(O.gate(d, p, 0.95), [-1, -1, -1, -1])
    assert np.array_equal(O.gate(d, p, 1.5), [-1, -1, -1, -1])
    # an offered prefix of length n accepts at most n proposals
    n, _ = O.accept(O.gate(d, p, 0.5), [5, 9, 2, 7, 1], 5)
    assert n == 2


# ---------------------------------------------------------------------------
# the device-chained cycle: committed positions, skipped fusion rows
# ---------------------------------------------------------------------------

def test_commit_positions_rule():
    """Anchor at p, n accepted: rows p .. p + n are committed, the bonus
    token's position p + n + 1 is the next anchor (the pages' acceptance
    cases: full, partial and first-candidate rejection)."""
    p = 100
    for n in (0, 3, 7):
        after = p + n + 1
        got = O.commit_positions(after, n)
        assert list(got[: n + 1]) == list(range(p, p + n + 1))
        assert (got[n + 1:] == -1).all() and len(got) == 8


def test_fusion_skips_negative_positions():
    """Fusing rows with some positions -1 writes exactly the other rows,
    bit-identical to fusing only those rows."""
    cfg = _tiny()
    ck = synth.make_checkpoint(cfg, seed=71, with_target_tensors=False)
    m = O.Model(cfg, ck)
    taps = synth.make_taps(cfg, 8, seed=71)
    pos = np.array([10, 11, 12, -1, -1, -1, -1, -1])
    a = O.State(cfg, 32)
    O.fuse_context(m, a, taps, pos)
    b = O.State(cfg, 32)
    O.fuse_context(m, b, taps[:3], pos[:3])
    for l in range(cfg.n_layers):
        assert np.array_equal(a.K[l], b.K[l]) and np.array_equal(a.V[l], b.V[l])
        assert np.array_equal(a.held[l], b.held[l])


# ---------------------------------------------------------------------------
# per-layer composition of the pass: which norm feeds which projection, the
# per-head q / k norms, the roles of gate and up, the value path
# ---------------------------------------------------------------------------

def _scaled(ck, name, c):
    """A BF16 tensor of the checkpoint times c (a power of two: exact)."""
    return synth.to_bf16_bits((O.decode_bf16(ck[name]) * c).astype(np.float32))


def _run_pass(cfg, ck, seed, B=4, trace=False):
    m = O.Model(cfg, ck)
    st = O.State(cfg, 128)
    O.fuse_context(m, st, synth.make_taps(cfg, cfg.ctx, seed=seed), np.arange(cfg.ctx))
    return O.draft_block(m, st, 21, cfg.ctx, B, trace=trace), st


@pytest.mark.parametrize("mat", ["wq", "wk"])
def test_per_head_qk_norm_makes_projection_scale_irrelevant(mat):
    """With eps = 0 the per-head RMSNorm of q (and of every k, context and
    block) removes any positive scale of W_q (W_k): the whole pass is
    unchanged.  Without the norm the attention logits would scale by 4."""
    cfg = _tiny(norm_eps=0.0)
    ck = synth.make_checkpoint(cfg, seed=31)
    r0, _ = _run_pass(cfg, ck, 31)
    ck2 = dict(ck)
    for l in range(cfg.n_layers):
        ck2[f"layers.{l}.{mat}"] = _scaled(ck, f"layers.{l}.{mat}", 4.0)
    r1, _ = _run_pass(cfg, ck2, 31)
    rms = float(np.sqrt(np.mean(r0.final_hidden ** 2)))
    assert np.allclose(r0.final_hidden, r1.final_hidden, rtol=0, atol=1e-12 * rms)
    assert np.array_equal(r0.drafts, r1.drafts)


def test_qk_norm_weights_enter_the_logits_as_a_product():
    """q_norm x 2 with k_norm x 1/2 leaves every logit q.k (hence the pass)
    unchanged; q_norm x 2 alone sharpens the softmax and changes it.  This
    separates the two weights: using k_norm for q, or ignoring q_norm, fails."""
    cfg = _tiny()
    ck = synth.make_checkpoint(cfg, seed=32)
    r0, _ = _run_pass(cfg, ck, 32)
    both, qonly = dict(ck), dict(ck)
    for l in range(cfg.n_layers):
        both[f"layers.{l}.q_norm"] = _scaled(ck, f"layers.{l}.q_norm", 2.0)
        both[f"layers.{l}.k_norm"] = _scaled(ck, f"layers.{l}.k_norm", 0.5)
        qonly[f"layers.{l}.q_norm"] = _scaled(ck, f"layers.{l}.q_norm", 2.0)
    r1, _ = _run_pass(cfg, both, 32)
    r2, _ = _run_pass(cfg, qonly, 32)
    rms = float(np.sqrt(np.mean(r0.final_hidden ** 2)))
    # k / 2 is stored in FP16 exactly (a power of two)
    assert np.allclose(r0.final_hidden, r1.final_hidden, rtol=0, atol=1e-12 * rms)
    assert not np.allclose(r0.final_hidden, r2.final_hidden, rtol=0, atol=1e-4 * rms)


def test_zero_mlp_norm_makes_the_mlp_vanish():
    """mlp_norm = 0 zeroes the MLP input, so silu(0) * 0 = 0 and every layer's
    residual leaves the MLP unchanged (x_mlp == x_attn); the attention
    sub-layers are untouched (its input norm is attn_norm, not mlp_norm)."""
    cfg = _tiny()
    ck = synth.make_checkpoint(cfg, seed=33)
    r0, _ = _run_pass(cfg, ck, 33, trace=True)
    ck2 = dict(ck)
    for l in range(cfg.n_layers):
        ck2[f"layers.{l}.mlp_norm"] = np.zeros_like(ck[f"layers.{l}.mlp_norm"])
    r1, _ = _run_pass(cfg, ck2, 33, trace=True)
    for l in range(cfg.n_layers):
        assert np.array_equal(r1.stages[f"layers.{l}.x_mlp"], r1.stages[f"layers.{l}.x_attn"])
        assert not np.allclose(r0.stages[f"layers.{l}.x_mlp"], r0.stages[f"layers.{l}.x_attn"])
    # layer 0's attention sub-layer does not see mlp_norm at all
    assert np.array_equal(r0.stages["layers.0.x_attn"], r1.stages["layers.0.x_attn"])


def test_zero_attn_norm_gives_uniform_attention_over_values():
    """attn_norm = 0 makes q = k = v = 0 for the block rows, so every score is
    0 and each head's attention output is the plain mean of its kv head's
    values over the context cells [0, p) and the B zero block rows."""
    cfg = _tiny()
    ck = synth.make_checkpoint(cfg, seed=34)
    ck2 = dict(ck)
    for l in range(cfg.n_layers):
        ck2[f"layers.{l}.attn_norm"] = np.zeros_like(ck[f"layers.{l}.attn_norm"])
    B = 4
    r, st = _run_pass(cfg, ck2, 34, B=B, trace=True)
    grp = cfg.n_q_heads // cfg.n_kv_heads
    for l in range(cfg.n_layers):
        v_ctx = st.V[l][:, :cfg.ctx, :].astype(np.float64)   # [n_kv, ctx, d]
        mean = v_ctx.sum(axis=1) / (cfg.ctx + B)
        a = r.stages[f"layers.{l}.attn"]                     # [B, n_q, d]
        for h in range(cfg.n_q_heads):
            assert np.allclose(a[:, h, :], mean[h // grp][None, :], rtol=0, atol=1e-12)
        assert not np.any(st.V[l][:, cfg.ctx:cfg.ctx + B, :])


def test_swiglu_gate_and_up_roles_closed_form():
    """One MLP unit: W_gate = a e_i^T, W_up = b e_j^T (row 0), W_down = e_k e_0^T
    gives x_mlp - x_attn = silu(a xn_i) * (b xn_j) at element k and 0
    elsewhere, xn = rmsnorm(x_attn, mlp_norm).  With a != b and xn_i != xn_j,
    silu on the up projection instead of the gate fails."""
    cfg = _tiny(n_layers=1)
    ck = synth.make_checkpoint(cfg, seed=35)
    H, I = cfg.hidden, cfg.intermediate
    i, j, k, a, b = 3, 17, 40, 1.5, -0.75
    g = np.zeros((I, H), np.float32); g[0, i] = a
    u = np.zeros((I, H), np.float32); u[0, j] = b
    dn = np.zeros((H, I), np.float32); dn[k, 0] = 1.0
    ck["layers.0.w_gate"] = synth.to_bf16_bits(g)
    ck["layers.0.w_up"] = synth.to_bf16_bits(u)
    ck["layers.0.w_down"] = synth.to_bf16_bits(dn)
    r, _ = _run_pass(cfg, ck, 35, trace=True)
    xa = r.stages["layers.0.x_attn"]
    xn = xa / np.sqrt(np.mean(xa * xa, -1, keepdims=True) + cfg.norm_eps) * O.decode_bf16(ck["layers.0.mlp_norm"])
    z = a * xn[:, i]
    want = (z / (1.0 + np.exp(-z))) * (b * xn[:, j])
    delta = r.stages["layers.0.x_mlp"] - xa
    assert np.allclose(delta[:, k], want, rtol=0, atol=1e-13)
    assert not np.any(np.delete(delta, k, axis=1))
    swapped = ((b * xn[:, j]) / (1.0 + np.exp(-b * xn[:, j]))) * (a * xn[:, i])
    assert not np.allclose(delta[:, k], swapped, rtol=0, atol=1e-6)


def test_values_are_the_unnormed_unrotated_projection():
    """W_v = [I 0] (selecting the first n_kv * d hidden elements): the fused
    context's V cells are FP16(h_ctx[:, :n_kv d]) and the block's own V cells
    are FP16(rmsnorm(embed, attn_norm)[:, :n_kv d]) -- no norm and no
    rotation on values, and the value input of the draft pass is the
    attn_norm output."""
    cfg = _tiny(n_layers=1)
    ck = synth.make_checkpoint(cfg, seed=36)
    H, nv = cfg.hidden, cfg.n_kv_heads * cfg.head_dim
    wv = np.zeros((nv, H), np.float32); wv[:, :nv] = np.eye(nv, dtype=np.float32)
    ck["layers.0.wv"] = synth.to_bf16_bits(wv)
    m = O.Model(cfg, ck)
    st = O.State(cfg, 128)
    taps = synth.make_taps(cfg, cfg.ctx, seed=36)
    h = O.fuse_context(m, st, taps, np.arange(cfg.ctx))
    want_ctx = O.round_f16(h[:, :nv]).reshape(cfg.ctx, cfg.n_kv_heads, cfg.head_dim).transpose(1, 0, 2)
    assert np.array_equal(st.V[0][:, :cfg.ctx, :], want_ctx)
    B = 4
    O.draft_block(m, st, 21, cfg.ctx, B)
    toks = [21] + [cfg.mask_token_id] * (B - 1)
    e = O.decode_bf16(ck["embed"][toks])
    xn = e / np.sqrt(np.mean(e * e, -1, keepdims=True) + cfg.norm_eps) * O.decode_bf16(ck["layers.0.attn_norm"])
    want_blk = O.round_f16(xn[:, :nv]).reshape(B, cfg.n_kv_heads, cfg.head_dim).transpose(1, 0, 2)
    assert np.array_equal(st.V[0][:, cfg.ctx:cfg.ctx + B, :], want_blk)

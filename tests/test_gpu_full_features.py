"""GPU parity of the draft cycle's features at the full DFlash geometry
(hidden 2560, 24Q/2KV x 256, vocab 151936) against the CPU oracle:

  * the drafter attention window over a ring of K/V cells ("#1426 dflash",
    "Additional constraints": a window of resident cells), with windows that
    start inside a 128-position attention tile, at head dim 256;
  * the confidence gate (spec-min-p, "#3322", "Long-prompt diagnosis and
    fix"): every draft's softmax probability over all 151936 logits, reduced
    across the LM head's CTAs, and the offered prefix under a floor;
  * two device-chained draft cycles (draft, accept, commit positions, an
    8-row fusion that skips rows, draft) with no host round trip.
"""
import numpy as np
import pytest

from gpu_helpers import O, build_lib, check_cells, check_drafts, check_hidden, device_ids, need_gpu, synth, torch

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

PROB_REL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _setup():
    need_gpu()
    build_lib()


def _prefill_range(st, ost, cfg, slot, pos0, n, seed):
    """Seeded FP16 K/V for positions [pos0, pos0 + n) on both sides (through
    the ring when the state has an attention window)."""
    kv = synth.make_kv_fill(cfg, n, seed=seed, slot=slot)
    pos = np.arange(pos0, pos0 + n)
    for l, (k, v) in enumerate(kv):
        st.write_kv(slot, l, pos0, torch.as_tensor(k.view(np.int16), device="cuda"),
                    torch.as_tensor(v.view(np.int16), device="cuda"))
        ost.write(l, pos, k.astype(np.float64).transpose(1, 0, 2), v.astype(np.float64).transpose(1, 0, 2))


def _fuse(st, ost, om, cfg, slot, pos, seed, stream):
    taps = synth.make_taps(cfg, len(pos), seed=seed, stream=stream)
    st.fuse(slot, torch.as_tensor(taps.view(np.int16), device="cuda"), device_ids(pos))
    O.fuse_context(om, ost, taps, pos)


def _setup_context(wtype, ctx, cap, window, seed):
    from dflash_block_drafter_gb300.runtime import DraftModel, DraftState
    cfg = synth.CONFIGS["full_bf16"].with_(weight_type=wtype, ctx=ctx, attn_window=window)
    ck = synth.make_checkpoint(cfg, seed=seed)
    om = O.Model(cfg, ck)
    model = DraftModel(cfg, ck)
    st = DraftState(model, 1, cap)
    ost = O.State(cfg, cap)
    lo = max(0, ctx + 8 - window) if window else 0
    _prefill_range(st, ost, cfg, 0, lo, ctx - 8 - lo, seed)
    _fuse(st, ost, om, cfg, 0, np.arange(ctx - 8, ctx), seed, 0)
    return cfg, om, model, st, ost


@pytest.mark.parametrize("wtype,window", [("q8_0", 4096), ("bf16", 4000)])
def test_full_window_ring(wtype, window):
    """p = 10000, block 8, a ring of 4096 cells: the window starts at
    10008 - W (position 5912 or 6008, inside an attention tile); the ring has
    wrapped twice by then."""
    ctx, B = 10000, 8
    cfg, om, model, st, ost = _setup_context(wtype, ctx, 4096, window, seed=91)
    assert (ctx + B - window) % 128 != 0
    anchor = int(synth.make_token_ids(cfg, 1, seed=91)[0])
    st.anchor_tok[0], st.anchor_pos[0], st.block_len[0] = anchor, ctx, B
    st.draft(1)
    res = O.draft_block(om, ost, anchor, ctx, B)
    torch.cuda.synchronize()
    what = f"{wtype} W={window}"
    check_hidden(st.final_hidden[0, :B].cpu().numpy(), res.final_hidden, what)
    check_drafts(st.drafts[0].cpu().numpy(), res, B, what)
    lo = ctx + B - window
    for l in range(cfg.n_layers):
        k, v = st.read_kv(0, l, lo, ctx + B - lo)
        ok, ov = ost.keys(l, ctx + B, lo)
        check_cells(k.cpu().numpy(), ok.transpose(1, 0, 2), f"{what} K l{l}")
        check_cells(v.cpu().numpy(), ov.transpose(1, 0, 2), f"{what} V l{l}")
    assert st.take_status() == 0


def _floor_between(probs):
    p = np.sort(np.asarray(probs))
    gaps = [(p[i + 1] / p[i], i) for i in range(len(p) - 1) if p[i] > 0]
    ratio, i = max(gaps)
    assert ratio > 1.04, "confidences too close to split with a margin"
    return float(np.sqrt(p[i] * p[i + 1]))


def test_full_gate():
    """Draft confidences at vocabulary 151936 (152 LM-head CTAs) within 1 %
    of the oracle's float64 softmax, the gated prefix under a floor between
    two of them, and floor 0 offering every draft."""
    ctx, B = 8192, 8
    cfg, om, model, st, ost = _setup_context("bf16", ctx, ctx + B, 0, seed=92)
    anchor = int(synth.make_token_ids(cfg, 1, seed=92)[0])
    st.anchor_tok[0], st.anchor_pos[0], st.block_len[0] = anchor, ctx, B
    res = O.draft_block(om, ost, anchor, ctx, B)
    st.set_spec_min_p(1e-12)
    st.draft(1)
    probs = st.draft_probs().cpu().numpy()[0]
    check_drafts(st.drafts[0].cpu().numpy(), res, B, "gate, every draft offered")
    assert np.allclose(probs, res.probs, rtol=PROB_REL, atol=0), f"{probs} vs {res.probs}"
    floor = _floor_between(res.probs)
    st.set_spec_min_p(floor)
    st.draft(1)
    torch.cuda.synchronize()
    want = O.gate(res.drafts, res.probs, floor)
    got = st.drafts[0, :B - 1].cpu().numpy()
    clear = np.abs(np.log(res.probs / floor)) > 1.5 * PROB_REL
    upto = len(want) if clear.all() else int(np.argmin(clear))
    assert np.array_equal(got[:upto] == -1, want[:upto] == -1), f"{got} vs {want} (floor {floor})"
    sure = (want[:upto] != -1) & (res.top2_gap[:upto] > 1e-2)
    assert np.array_equal(got[:upto][sure], want[:upto][sure])
    st.set_spec_min_p(0.0)
    st.draft(1)
    torch.cuda.synchronize()
    assert np.all(st.draft_probs().cpu().numpy() == -1)
    check_drafts(st.drafts[0].cpu().numpy(), res, B, "gate, floor 0")
    assert st.take_status() == 0


@pytest.mark.parametrize("defer", [False, True], ids=["kv_separate", "kv_in_next_qkv"])
def test_full_two_chained_cycles(defer):
    """Cycle 1 drafts at p = 8192; the verifier agrees with its first two
    drafts; acceptance advances the anchor on the device, the committed rows
    p .. p + 2 are fused (the other five rows skipped) and cycle 2 drafts at
    p + 3 from the device-resident anchor.  defer: the committed rows' K/V
    are projected inside cycle 2's QKV GEMVs."""
    from dflash_block_drafter_gb300.runtime import accept, commit_positions
    ctx, B = 8192, 8
    cfg, om, model, st, ost = _setup_context("bf16", ctx, ctx + 64, 0, seed=93)
    # an anchor whose first three drafts are clear of ties in the oracle
    for k in range(8):
        anchor = int(synth.make_token_ids(cfg, 1, seed=93, stream=k)[0])
        ost_try = O.State(cfg, ctx + 64)
        ost_try.K, ost_try.V, ost_try.held = [x.copy() for x in ost.K], [x.copy() for x in ost.V], \
            [x.copy() for x in ost.held]
        r1 = O.draft_block(om, ost_try, anchor, ctx, B)
        if np.all(r1.top2_gap[:3] > 1e-2):
            break
    assert np.all(r1.top2_gap[:3] > 1e-2)
    ost = ost_try
    tgt = np.array(list(r1.drafts[:2]) + [int(r1.drafts[2] + 1) % cfg.vocab] + [5] * (B - 3), np.int32)
    n1, bonus = O.accept(r1.drafts, tgt, B)
    assert n1 == 2
    new_taps = synth.make_taps(cfg, 8, seed=93, stream=1)

    st.anchor_tok[0], st.anchor_pos[0], st.block_len[0] = anchor, ctx, B
    st.set_defer_kv(defer)
    acc = torch.zeros(1, dtype=torch.int32, device="cuda")
    pos8 = torch.zeros((1, 8), dtype=torch.int32, device="cuda")
    st.draft(1)
    accept(st.drafts, device_ids(tgt[None]), st.block_len, acc, st.anchor_tok, st.anchor_pos)
    commit_positions(st.anchor_pos, acc, pos8)
    st.fuse(0, torch.as_tensor(new_taps.view(np.int16), device="cuda"), pos8[0])
    st.draft(1)
    torch.cuda.synchronize()

    committed = O.commit_positions(ctx + n1 + 1, n1)
    O.fuse_context(om, ost, new_taps, committed)
    r2 = O.draft_block(om, ost, bonus, ctx + n1 + 1, B)
    assert int(acc[0]) == n1 and int(st.anchor_tok[0]) == bonus and int(st.anchor_pos[0]) == ctx + n1 + 1
    assert np.array_equal(pos8[0].cpu().numpy(), committed)
    check_hidden(st.final_hidden[0, :B].cpu().numpy(), r2.final_hidden, "cycle 2")
    check_drafts(st.drafts[0].cpu().numpy(), r2, B, "cycle 2")
    hi = ctx + n1 + 1 + B
    for l in range(cfg.n_layers):
        k, v = st.read_kv(0, l, ctx - 8, hi - (ctx - 8))
        check_cells(k.cpu().numpy(), ost.K[l][:, ctx - 8:hi], f"K l{l}")
        check_cells(v.cpu().numpy(), ost.V[l][:, ctx - 8:hi], f"V l{l}")
    assert st.take_status() == 0

"""GPU parity of the CUDA path (through the C ABI) against the CPU oracle on
the tiny DFlash workload: 2 layers, hidden 256, 4Q/1KV x 64, MLP 768, vocab
1024, context 64, block 4 -- plus its quantised variants, other block sizes,
several slots, an empty context, a full state, a ragged vocabulary and the
device-detected errors.  The small shapes still span many GEMV units, split
groups and several attention tiles."""
import numpy as np
import pytest

from gpu_helpers import (O, build_lib, check_cells, check_drafts, check_hidden, compare_state, device_ids,
                         need_gpu, synth, torch)

pytestmark = pytest.mark.gpu

WTYPES = ["bf16", "q8_0", "q5_0", "q4_0"]


@pytest.fixture(scope="module", autouse=True)
def _setup():
    need_gpu()
    build_lib()


def _model(cfg, seed):
    from dflash_block_drafter_gb300.runtime import DraftModel
    ck = synth.make_checkpoint(cfg, seed=seed)
    return ck, DraftModel(cfg, ck), O.Model(cfg, ck)


def _state(model, n_slots, cap):
    from dflash_block_drafter_gb300.runtime import DraftState
    return DraftState(model, n_slots, cap)


def _fuse_both(st, ost, slot, cfg, taps, pos):
    st.fuse(slot, torch.as_tensor(taps.view(np.int16), device="cuda"), device_ids(pos))
    O.fuse_context(ost.om, ost, taps, pos)


def _ostate(om, cfg, cap):
    s = O.State(cfg, cap)
    s.om = om
    return s


def _draft_both(st, osts, toks, ps, Bs):
    n = len(toks)
    st.anchor_tok[:n] = device_ids(toks)
    st.anchor_pos[:n] = device_ids(ps)
    st.block_len[:n] = device_ids(Bs)
    st.draft(n)
    res = [O.draft_block(osts[s].om, osts[s], int(toks[s]), int(ps[s]), int(Bs[s])) for s in range(n)]
    torch.cuda.synchronize()
    return res


@pytest.mark.parametrize("wtype", WTYPES)
def test_dequant_bit_exact(wtype):
    cfg = synth.CONFIGS["tiny"].with_(weight_type=wtype)
    ck, model, om = _model(cfg, seed=21)
    names = ["fc"] + [f"layers.{l}.{t}" for l in range(cfg.n_layers)
                      for t in ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down")]
    for which, name in enumerate(names):
        got = model.dequantize(which).cpu().numpy().astype(np.float64)
        assert np.array_equal(got, om.mat(name)), f"{wtype} {name}: dequantised weights differ"


@pytest.mark.parametrize("wtype", WTYPES)
def test_fuse_context_cells(wtype):
    cfg = synth.CONFIGS["tiny"].with_(weight_type=wtype)
    ck, model, om = _model(cfg, seed=22)
    cap = 96
    st = _state(model, 1, cap)
    ost = _ostate(om, cfg, cap)
    # a 64-position fusion (128-row tile path), then 5 more positions out of
    # order (8-row tile path), then an overwrite of 3 cells
    taps = synth.make_taps(cfg, 64, seed=22)
    _fuse_both(st, ost, 0, cfg, taps, np.arange(64))
    taps2 = synth.make_taps(cfg, 5, seed=22, stream=1)
    _fuse_both(st, ost, 0, cfg, taps2, np.array([70, 66, 64, 65, 69]))
    taps3 = synth.make_taps(cfg, 3, seed=22, stream=2)
    _fuse_both(st, ost, 0, cfg, taps3, np.array([1, 30, 63]))
    torch.cuda.synchronize()
    for l in range(cfg.n_layers):
        for lo, hi in ((0, 64), (64, 67), (69, 71)):
            k, v = st.read_kv(0, l, lo, hi - lo)
            check_cells(k.cpu().numpy(), ost.K[l][:, lo:hi], f"K l{l} [{lo},{hi})")
            check_cells(v.cpu().numpy(), ost.V[l][:, lo:hi], f"V l{l} [{lo},{hi})")
    assert st.take_status() == 0


@pytest.mark.parametrize("wtype,B", [("bf16", 4), ("bf16", 2), ("bf16", 8), ("q8_0", 4), ("q5_0", 7),
                                     ("q4_0", 4)])
def test_draft_pass(wtype, B):
    cfg = synth.CONFIGS["tiny"].with_(weight_type=wtype)
    ck, model, om = _model(cfg, seed=23)
    cap = 128
    st = _state(model, 1, cap)
    ost = _ostate(om, cfg, cap)
    taps = synth.make_taps(cfg, cfg.ctx, seed=23)
    _fuse_both(st, ost, 0, cfg, taps, np.arange(cfg.ctx))
    anchor = int(synth.make_token_ids(cfg, 1, seed=23)[0])
    (res,) = _draft_both(st, [ost], [anchor], [cfg.ctx], [B])
    check_hidden(st.final_hidden[0, :B].cpu().numpy(), res.final_hidden)
    check_drafts(st.drafts[0].cpu().numpy(), res, B)
    # the block's own K/V cells [p, p + B) written by every layer
    compare_state(st, ost, 0, cfg.ctx + B, "after draft")
    assert st.take_status() == 0


def test_draft_repeat_is_deterministic():
    cfg = synth.CONFIGS["tiny"]
    ck, model, om = _model(cfg, seed=24)
    st = _state(model, 1, 128)
    taps = synth.make_taps(cfg, cfg.ctx, seed=24)
    st.fuse(0, torch.as_tensor(taps.view(np.int16), device="cuda"), device_ids(np.arange(cfg.ctx)))
    st.anchor_tok[0] = 5
    st.anchor_pos[0] = cfg.ctx
    st.block_len[0] = 4
    outs = []
    for _ in range(3):
        st.draft(1)
        torch.cuda.synchronize()
        outs.append((st.drafts.clone(), st.final_hidden.clone()))
    for d, h in outs[1:]:
        assert torch.equal(d, outs[0][0]) and torch.equal(h, outs[0][1])


@pytest.mark.parametrize("wtype", ["bf16", "q4_0"])
def test_batched_slots(wtype):
    """Three sequences with their own contexts, anchors and block sizes in one
    pass; each must match the oracle run on that sequence alone."""
    cfg = synth.CONFIGS["tiny"].with_(weight_type=wtype)
    ck, model, om = _model(cfg, seed=25)
    cap = 160
    st = _state(model, 3, cap)
    ctxs, Bs = [40, 97, 5], [3, 8, 2]
    osts = []
    for s, n in enumerate(ctxs):
        ost = _ostate(om, cfg, cap)
        _fuse_both(st, ost, s, cfg, synth.make_taps(cfg, n, seed=25, stream=s), np.arange(n))
        osts.append(ost)
    toks = synth.make_token_ids(cfg, 3, seed=25)
    res = _draft_both(st, osts, toks, ctxs, Bs)
    for s in range(3):
        check_hidden(st.final_hidden[s, :Bs[s]].cpu().numpy(), res[s].final_hidden, f"slot {s}")
        check_drafts(st.drafts[s].cpu().numpy(), res[s], Bs[s], f"slot {s}")
        compare_state(st, osts[s], s, ctxs[s] + Bs[s], f"slot {s}")
    assert st.take_status() == 0


@pytest.mark.parametrize("wtype", WTYPES)
def test_twelve_slots(wtype):
    """A 128-row pass (12 sequences of their own contexts and block sizes):
    the layer GEMMs and the LM head on the tcgen05 tensor cores, every slot
    against the oracle run on that sequence alone, with its K/V cells."""
    cfg = synth.CONFIGS["tiny"].with_(weight_type=wtype)
    ck, model, om = _model(cfg, seed=26)
    cap = 160
    n = 12
    st = _state(model, n, cap)
    ctxs = [40, 97, 5, 64, 130, 18, 77, 2, 150, 33, 88, 120]
    Bs = [3, 8, 2, 5, 8, 4, 7, 6, 2, 8, 3, 5]
    osts = []
    for s_, c in enumerate(ctxs):
        ost = _ostate(om, cfg, cap)
        _fuse_both(st, ost, s_, cfg, synth.make_taps(cfg, c, seed=26, stream=s_), np.arange(c))
        osts.append(ost)
    toks = synth.make_token_ids(cfg, n, seed=26)
    res = _draft_both(st, osts, toks, ctxs, Bs)
    for s_ in range(n):
        check_hidden(st.final_hidden[s_, :Bs[s_]].cpu().numpy(), res[s_].final_hidden, f"slot {s_}")
        check_drafts(st.drafts[s_].cpu().numpy(), res[s_], Bs[s_], f"slot {s_}")
        compare_state(st, osts[s_], s_, ctxs[s_] + Bs[s_], f"slot {s_}")
    assert st.take_status() == 0


def test_empty_context_and_full_state():
    cfg = synth.CONFIGS["tiny"]
    ck, model, om = _model(cfg, seed=26)
    # p = 0: the block attends only to itself
    st = _state(model, 1, 8)
    ost = _ostate(om, cfg, 8)
    (res,) = _draft_both(st, [ost], [3], [0], [8])
    check_hidden(st.final_hidden[0].cpu().numpy(), res.final_hidden, "p = 0")
    check_drafts(st.drafts[0].cpu().numpy(), res, 8)
    assert st.take_status() == 0
    # p + B == capacity exactly
    cap = 70
    st2 = _state(model, 1, cap)
    ost2 = _ostate(om, cfg, cap)
    _fuse_both(st2, ost2, 0, cfg, synth.make_taps(cfg, 66, seed=26), np.arange(66))
    (res2,) = _draft_both(st2, [ost2], [9], [66], [4])
    check_hidden(st2.final_hidden[0, :4].cpu().numpy(), res2.final_hidden, "full state")
    check_drafts(st2.drafts[0].cpu().numpy(), res2, 4)
    assert st2.take_status() == 0


@pytest.mark.parametrize("n_slots", [1, 12])
def test_ragged_vocab(n_slots):
    """A vocabulary that is not a multiple of the LM head's row tiles (64 for
    the GEMV head, 256 for the tcgen05 head of 9..16 slots)."""
    cfg = synth.CONFIGS["tiny"].with_(vocab=1000)
    ck, model, om = _model(cfg, seed=27)
    st = _state(model, n_slots, 128)
    osts = []
    for s in range(n_slots):
        ost = _ostate(om, cfg, 128)
        _fuse_both(st, ost, s, cfg, synth.make_taps(cfg, 50 + s, seed=27, stream=s), np.arange(50 + s))
        osts.append(ost)
    toks = [999] + list(synth.make_token_ids(cfg, n_slots - 1, seed=27))
    res = _draft_both(st, osts, toks, [50 + s for s in range(n_slots)], [6] * n_slots)
    for s in range(n_slots):
        check_hidden(st.final_hidden[s, :6].cpu().numpy(), res[s].final_hidden, f"slot {s}")
        check_drafts(st.drafts[s].cpu().numpy(), res[s], 6, f"slot {s}")
    assert (st.drafts[:n_slots, :5] < 1000).all()


def test_device_detected_errors():
    from dflash_block_drafter_gb300 import (DFLASH_DEV_BAD_BLOCK, DFLASH_DEV_BAD_TOKEN, DFLASH_DEV_CAPACITY,
                                            DFLASH_DEV_NONFINITE)
    cfg = synth.CONFIGS["tiny"]
    ck, model, om = _model(cfg, seed=28)
    st = _state(model, 1, 64)
    taps = synth.make_taps(cfg, 40, seed=28)
    st.fuse(0, torch.as_tensor(taps.view(np.int16), device="cuda"), device_ids(np.arange(40)))
    assert st.take_status() == 0
    # anchor id out of range
    st.anchor_tok[0], st.anchor_pos[0], st.block_len[0] = cfg.vocab + 5, 40, 4
    st.draft(1)
    assert st.take_status() & DFLASH_DEV_BAD_TOKEN
    # block beyond the capacity (the pass must not write outside the state)
    st.anchor_tok[0], st.anchor_pos[0], st.block_len[0] = 1, 62, 4
    st.draft(1)
    assert st.take_status() & DFLASH_DEV_CAPACITY
    # block length out of [2, 8]
    st.anchor_tok[0], st.anchor_pos[0], st.block_len[0] = 1, 40, 11
    st.draft(1)
    assert st.take_status() & DFLASH_DEV_BAD_BLOCK
    # a fusion position outside the state
    st.fuse(0, torch.as_tensor(taps[:2].view(np.int16), device="cuda"), device_ids([3, 64]))
    assert st.take_status() & DFLASH_DEV_CAPACITY
    # non-finite taps propagate to the logits and are refused
    bad = taps[:1].copy()
    bad[0, 7] = 0x7FC0  # BF16 NaN
    st.fuse(0, torch.as_tensor(bad.view(np.int16), device="cuda"), device_ids([10]))
    st.anchor_tok[0], st.anchor_pos[0], st.block_len[0] = 1, 40, 4
    st.draft(1)
    assert st.take_status() & DFLASH_DEV_NONFINITE


def test_attention_chunks_sixteen_slots():
    """16 slots of a 1300-position context (11 super-tiles) in 9 and in 10
    chunks per slot (144 and 160 CTAs, below and above the SM count), every
    slot against the oracle."""
    import dflash_block_drafter_gb300 as D
    cfg = synth.CONFIGS["tiny"]
    ck, model, om = _model(cfg, seed=31)
    cap, n_ctx, n = 1408, 1300, 16
    st = _state(model, n, cap)
    osts = [_ostate(om, cfg, cap) for _ in range(n)]
    taps = synth.make_taps(cfg, n_ctx, seed=31)
    for s in range(n):
        _fuse_both(st, osts[s], s, cfg, taps, np.arange(n_ctx))
    toks = synth.make_token_ids(cfg, n, seed=31)
    Bs = [2 + s % 7 for s in range(n)]
    assert D.dflash_state_set_attn_chunks(st.handle, 0) >= 10
    for chunks in (9, 10):
        D.dflash_state_set_attn_chunks(st.handle, chunks)
        res = _draft_both(st, osts, toks, [n_ctx] * n, Bs)
        for s in range(n):
            check_hidden(st.final_hidden[s, :Bs[s]].cpu().numpy(), res[s].final_hidden, f"chunks {chunks} slot {s}")
            check_drafts(st.drafts[s].cpu().numpy(), res[s], Bs[s], f"chunks {chunks} slot {s}")
        assert st.take_status() == 0


def test_accept_matches_oracle():
    from dflash_block_drafter_gb300.runtime import accept
    rng = np.random.default_rng(29)
    n_seq = 300
    maxb = 8
    Bs = rng.integers(2, maxb + 1, size=n_seq).astype(np.int32)
    drafts = rng.integers(0, 5, size=(n_seq, maxb - 1)).astype(np.int32)
    tgt = np.zeros((n_seq, maxb), np.int32)
    for s in range(n_seq):
        tgt[s] = synth.make_target_ids(drafts[s], 5, seed=29, stream=s)
    pos = rng.integers(0, 1000, size=n_seq).astype(np.int32)
    d_acc = torch.zeros(n_seq, dtype=torch.int32, device="cuda")
    d_next = torch.zeros(n_seq, dtype=torch.int32, device="cuda")
    d_pos = device_ids(pos)
    accept(device_ids(drafts), device_ids(tgt), device_ids(Bs), d_acc, d_next, d_pos)
    torch.cuda.synchronize()
    for s in range(n_seq):
        n, bonus = O.accept(drafts[s], tgt[s], int(Bs[s]))
        assert int(d_acc[s]) == n and int(d_next[s]) == bonus and int(d_pos[s]) == pos[s] + n + 1, s


def test_attention_chunks_two_long_slots():
    """Two slots of 3000 and 1100 positions (24 and 9 super-tiles) at 12
    chunks per slot: the plan gives the first sequence 12 chunks and the
    second 5, so the several-sequence merge folds more chunks than one batch
    of loads holds; both slots against the oracle."""
    import dflash_block_drafter_gb300 as D
    cfg = synth.CONFIGS["tiny"]
    ck, model, om = _model(cfg, seed=32)
    cap = 3072
    ctxs, Bs = [3000, 1100], [7, 4]
    st = _state(model, 2, cap)
    osts = []
    for s, n_ctx in enumerate(ctxs):
        ost = _ostate(om, cfg, cap)
        _fuse_both(st, ost, s, cfg, synth.make_taps(cfg, n_ctx, seed=32, stream=s), np.arange(n_ctx))
        osts.append(ost)
    assert D.dflash_state_set_attn_chunks(st.handle, 0) >= 12
    D.dflash_state_set_attn_chunks(st.handle, 12)
    res = _draft_both(st, osts, synth.make_token_ids(cfg, 2, seed=32), ctxs, Bs)
    for s in range(2):
        check_hidden(st.final_hidden[s, :Bs[s]].cpu().numpy(), res[s].final_hidden, f"slot {s}")
        check_drafts(st.drafts[s].cpu().numpy(), res[s], Bs[s], f"slot {s}")
    assert st.take_status() == 0


@pytest.mark.parametrize("chunks", [1, 2, 4, 5])
def test_attention_context_chunks(chunks):
    """The split-context attention and its log-sum-exp merge: a 600-position
    context (5 super-tiles of 128 keys) split into 1..5 chunks gives the
    oracle's pass.  1 chunk runs all 5 super-tiles through one CTA's
    pipeline; 4 chunks of 2 super-tiles leave the last chunk empty."""
    import dflash_block_drafter_gb300 as D
    cfg = synth.CONFIGS["tiny"]
    ck, model, om = _model(cfg, seed=30)
    cap = 640
    st = _state(model, 1, cap)
    assert D.dflash_state_set_attn_chunks(st.handle, 0) >= 5
    D.dflash_state_set_attn_chunks(st.handle, chunks)
    ost = _ostate(om, cfg, cap)
    _fuse_both(st, ost, 0, cfg, synth.make_taps(cfg, 600, seed=30), np.arange(600))
    (res,) = _draft_both(st, [ost], [77], [600], [6])
    check_hidden(st.final_hidden[0, :6].cpu().numpy(), res.final_hidden)
    check_drafts(st.drafts[0].cpu().numpy(), res, 6)
    assert st.take_status() == 0

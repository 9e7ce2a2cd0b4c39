"""GPU parity of the drafter attention window over ring-addressed K/V cells
against the CPU oracle (tiny DFlash workload): the block at p attends over
positions [max(0, p + B - W), p + B) and position pos lives in cell
pos mod capacity, so a context longer than the state's cells can be fused
and drafted from.  Windows that cut the context inside and at the edge of a
128-position attention tile, several CTA chunks of the window, a window that
covers the whole context, and K/V read-back through the ring."""
import numpy as np
import pytest

from gpu_helpers import O, build_lib, check_cells, check_drafts, check_hidden, device_ids, need_gpu, synth, torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    need_gpu()
    build_lib()


def _run(wtype, W, cap, n, B, seed, chunks=None):
    from dflash_block_drafter_gb300 import dflash_state_set_attn_chunks
    from dflash_block_drafter_gb300.runtime import DraftModel, DraftState
    cfg = synth.CONFIGS["tiny"].with_(weight_type=wtype, attn_window=W)
    ck = synth.make_checkpoint(cfg, seed=seed)
    model, om = DraftModel(cfg, ck), O.Model(cfg, ck)
    st = DraftState(model, 1, cap)
    if chunks is not None:
        dflash_state_set_attn_chunks(st.handle, chunks)
    ost = O.State(cfg, cap)
    # fuse positions [0, n) in tiles of up to 100, so the ring wraps part-way through a call
    for lo in range(0, n, 100):
        hi = min(n, lo + 100)
        taps = synth.make_taps(cfg, hi - lo, seed=seed, stream=lo)
        pos = np.arange(lo, hi)
        st.fuse(0, torch.as_tensor(taps.view(np.int16), device="cuda"), device_ids(pos))
        O.fuse_context(om, ost, taps, pos)
    anchor = int(synth.make_token_ids(cfg, 1, seed=seed)[0])
    st.anchor_tok[0], st.anchor_pos[0], st.block_len[0] = anchor, n, B
    st.draft(1)
    res = O.draft_block(om, ost, anchor, n, B)
    torch.cuda.synchronize()
    check_hidden(st.final_hidden[0, :B].cpu().numpy(), res.final_hidden, f"W={W} cap={cap} p={n}")
    check_drafts(st.drafts[0].cpu().numpy(), res, B, f"W={W} cap={cap} p={n}")
    # the window's cells (fused context and the block's own rows), read through the ring
    lo = max(0, n + B - W) if W else 0
    for l in range(cfg.n_layers):
        k, v = st.read_kv(0, l, lo, n + B - lo)
        ok, ov = ost.keys(l, n + B, lo)
        check_cells(k.cpu().numpy(), ok.transpose(1, 0, 2), f"K l{l}")
        check_cells(v.cpu().numpy(), ov.transpose(1, 0, 2), f"V l{l}")
    assert st.take_status() == 0


@pytest.mark.parametrize("wtype,W,cap,n,B", [
    ("bf16", 96, 128, 200, 4),    # ring wrapped once, window starts inside a tile
    ("bf16", 128, 128, 300, 8),   # window = capacity, starts on a tile boundary
    ("q4_0", 100, 256, 520, 5),   # ring wrapped twice
    ("bf16", 256, 256, 60, 4),    # window longer than the context: every position
])
def test_window_ring_parity(wtype, W, cap, n, B):
    _run(wtype, W, cap, n, B, seed=41)


def test_window_split_over_chunks():
    """A 384-position window over 4 attention tiles split across 3 CTA chunks."""
    _run("bf16", 384, 512, 900, 6, seed=42, chunks=3)


def test_ring_state_capacity_checks():
    """A ring state must hold the window and be a whole number of 128-cell
    attention tiles."""
    from dflash_block_drafter_gb300 import DFLASH_ERR_UNSUPPORTED, DflashError
    from dflash_block_drafter_gb300.runtime import DraftModel, DraftState
    cfg = synth.CONFIGS["tiny"].with_(attn_window=96)
    model = DraftModel(cfg, synth.make_checkpoint(cfg, seed=43))
    for cap in (64, 200):
        with pytest.raises(DflashError) as e:
            DraftState(model, 1, cap)
        assert e.value.status == DFLASH_ERR_UNSUPPORTED
    DraftState(model, 1, 128).close()


def test_window_several_slots():
    """Three slots with ring states of their own and contexts of different
    lengths in one pass (the pass's attention chunks are shared out among
    them by window length), each against the oracle."""
    from dflash_block_drafter_gb300.runtime import DraftModel, DraftState
    W, cap = 200, 256
    cfg = synth.CONFIGS["tiny"].with_(weight_type="bf16", attn_window=W)
    ck = synth.make_checkpoint(cfg, seed=43)
    model, om = DraftModel(cfg, ck), O.Model(cfg, ck)
    ctxs, Bs = [450, 90, 700], [6, 3, 8]
    st = DraftState(model, 3, cap)
    osts = []
    for s, n in enumerate(ctxs):
        ost = O.State(cfg, cap)
        for lo in range(0, n, 128):
            hi = min(n, lo + 128)
            taps = synth.make_taps(cfg, hi - lo, seed=43, stream=100 * s + lo)
            pos = np.arange(lo, hi)
            st.fuse(s, torch.as_tensor(taps.view(np.int16), device="cuda"), device_ids(pos))
            O.fuse_context(om, ost, taps, pos)
        osts.append(ost)
    toks = synth.make_token_ids(cfg, 3, seed=43)
    st.anchor_tok[:3] = device_ids(toks)
    st.anchor_pos[:3] = device_ids(ctxs)
    st.block_len[:3] = device_ids(Bs)
    st.draft(3)
    torch.cuda.synchronize()
    for s in range(3):
        res = O.draft_block(om, osts[s], int(toks[s]), ctxs[s], Bs[s])
        check_hidden(st.final_hidden[s, :Bs[s]].cpu().numpy(), res.final_hidden, f"slot {s}")
        check_drafts(st.drafts[s].cpu().numpy(), res, Bs[s], f"slot {s}")
    assert st.take_status() == 0

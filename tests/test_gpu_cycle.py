"""GPU parity of two device-chained draft cycles against the oracle: draft,
accept (anchor advanced on the device), commit positions (the accepted
prefix's rows, -1 for the rest), a fixed 8-row fusion that skips the -1 rows,
and the next draft from the device-resident anchor -- no host round trip
between the steps."""
import numpy as np
import pytest

from gpu_helpers import (O, build_lib, check_cells, check_drafts, check_hidden, device_ids, need_gpu, synth,
                         torch)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _setup():
    need_gpu()
    build_lib()


@pytest.mark.parametrize("wtype", ["bf16", "q4_0"])
@pytest.mark.parametrize("defer", [False, True], ids=["kv_separate", "kv_in_next_qkv"])
def test_two_chained_cycles(defer, wtype):
    """defer: the 8-row fusion leaves its K/V projection to the next draft
    pass, whose per-layer QKV GEMVs carry the committed rows."""
    from dflash_block_drafter_gb300.runtime import DraftModel, DraftState, accept, commit_positions
    cfg = synth.CONFIGS["tiny"].with_(weight_type=wtype)
    seed, n_ctx, B = 81, 64, 8
    ck = synth.make_checkpoint(cfg, seed=seed)
    model, om = DraftModel(cfg, ck), O.Model(cfg, ck)
    st = DraftState(model, 1, 128)
    ost = O.State(cfg, 128)
    taps = synth.make_taps(cfg, n_ctx, seed=seed)
    st.fuse(0, torch.as_tensor(taps.view(np.int16), device="cuda"), device_ids(np.arange(n_ctx)))
    O.fuse_context(om, ost, taps, np.arange(n_ctx))
    # cycle 1: the verifier agrees with the first two drafts; an anchor whose
    # first three drafts are clear of ties in the oracle
    for k in range(8):
        anchor = int(synth.make_token_ids(cfg, 1, seed=seed, stream=k)[0])
        ost_try = O.State(cfg, 128)
        ost_try.K, ost_try.V, ost_try.held = [x.copy() for x in ost.K], [x.copy() for x in ost.V], \
            [x.copy() for x in ost.held]
        r1 = O.draft_block(om, ost_try, anchor, n_ctx, B)
        if np.all(r1.top2_gap[:3] > 1e-2):
            break
    assert np.all(r1.top2_gap[:3] > 1e-2)
    ost = ost_try
    st.anchor_tok[0], st.anchor_pos[0], st.block_len[0] = anchor, n_ctx, B
    st.set_defer_kv(defer)
    tgt = np.array(list(r1.drafts[:2]) + [int(r1.drafts[2] + 1) % cfg.vocab] + [5] * (B - 3), np.int32)
    n1, bonus = O.accept(r1.drafts, tgt, B)
    assert n1 == 2
    new_taps = synth.make_taps(cfg, 8, seed=seed, stream=1)

    acc = torch.zeros(1, dtype=torch.int32, device="cuda")
    pos8 = torch.zeros((1, 8), dtype=torch.int32, device="cuda")
    st.draft(1)
    accept(st.drafts, device_ids(tgt[None]), st.block_len, acc, st.anchor_tok, st.anchor_pos)
    commit_positions(st.anchor_pos, acc, pos8)
    st.fuse(0, torch.as_tensor(new_taps.view(np.int16), device="cuda"), pos8[0])
    st.draft(1)
    torch.cuda.synchronize()

    # the oracle's cycle: the committed rows p .. p + n, then the next block at p + n + 1
    committed = O.commit_positions(n_ctx + n1 + 1, n1)
    assert list(committed[:3]) == [n_ctx, n_ctx + 1, n_ctx + 2] and (committed[3:] == -1).all()
    O.fuse_context(om, ost, new_taps, committed)
    r2 = O.draft_block(om, ost, bonus, n_ctx + n1 + 1, B)

    assert int(acc[0]) == n1 and int(st.anchor_tok[0]) == bonus and int(st.anchor_pos[0]) == n_ctx + n1 + 1
    assert np.array_equal(pos8[0].cpu().numpy(), committed)
    check_hidden(st.final_hidden[0, :B].cpu().numpy(), r2.final_hidden, "cycle 2")
    check_drafts(st.drafts[0].cpu().numpy(), r2, B, "cycle 2")
    for l in range(cfg.n_layers):
        k, v = st.read_kv(0, l, 0, n_ctx + n1 + 1 + B)
        check_cells(k.cpu().numpy(), ost.K[l][:, : n_ctx + n1 + 1 + B], f"K l{l}")
        check_cells(v.cpu().numpy(), ost.V[l][:, : n_ctx + n1 + 1 + B], f"V l{l}")
    assert st.take_status() == 0  # the skipped (-1) fusion rows raise no error


def test_deferred_fusion_flushed_by_reads():
    """Rows kept by a deferring fusion reach their cells before any call that
    needs them: dflash_state_read_kv, a later fusion, a multi-slot draft pass
    and dflash_state_flush; switching deferral off is refused while rows are
    kept."""
    from dflash_block_drafter_gb300 import DflashError
    from dflash_block_drafter_gb300.runtime import DraftModel, DraftState
    cfg = synth.CONFIGS["tiny"]
    seed, n_ctx = 82, 40
    ck = synth.make_checkpoint(cfg, seed=seed)
    model, om = DraftModel(cfg, ck), O.Model(cfg, ck)
    st = DraftState(model, 2, 128)
    ost = [O.State(cfg, 128), O.State(cfg, 128)]
    st.set_defer_kv(True)
    taps = synth.make_taps(cfg, 24, seed=seed)
    # 8 positions of slot 1, one of them skipped: kept, then read back
    # (a kept fusion's positions array must stay alive until its rows are projected)
    pos_a = np.array([3, 4, 5, -1, 7, 8, 9, 10], np.int32)
    dpos_a = device_ids(pos_a)
    st.fuse(1, torch.as_tensor(taps[:8].view(np.int16), device="cuda"), dpos_a)
    O.fuse_context(om, ost[1], taps[:8], pos_a)
    with pytest.raises(DflashError):
        st.set_defer_kv(False)
    for l in range(cfg.n_layers):
        k, v = st.read_kv(1, l, 0, 16)
        check_cells(k.cpu().numpy(), ost[1].K[l][:, :16], f"K l{l} (read)")
        check_cells(v.cpu().numpy(), ost[1].V[l][:, :16], f"V l{l} (read)")
    # kept rows of slot 0, then a second fusion (which projects them first)
    pos_b = np.arange(0, 8, dtype=np.int32)
    pos_c = np.arange(8, 14, dtype=np.int32)
    dpos_b, dpos_c = device_ids(pos_b), device_ids(pos_c)
    st.fuse(0, torch.as_tensor(taps[8:16].view(np.int16), device="cuda"), dpos_b)
    st.fuse(0, torch.as_tensor(taps[16:22].view(np.int16), device="cuda"), dpos_c)
    O.fuse_context(om, ost[0], taps[8:16], pos_b)
    O.fuse_context(om, ost[0], taps[16:22], pos_c)
    st.flush()
    st.set_defer_kv(False)
    # kept rows of slot 1 and a two-slot draft pass, which projects them before its layers
    st.set_defer_kv(True)
    pos_d = np.arange(20, 28, dtype=np.int32)
    dpos_d = device_ids(pos_d)
    st.fuse(1, torch.as_tensor(taps[:8].view(np.int16), device="cuda"), dpos_d)
    O.fuse_context(om, ost[1], taps[:8], pos_d)
    st.anchor_tok[:2] = 1
    st.anchor_pos[:2] = 64
    st.block_len[:2] = 4
    st.draft(2, want_hidden=False)
    st.set_defer_kv(False)  # nothing kept any more
    torch.cuda.synchronize()
    for l in range(cfg.n_layers):
        k, v = st.read_kv(1, l, 20, 8)
        check_cells(k.cpu().numpy(), ost[1].K[l][:, 20:28], f"K l{l} (two-slot pass)")
        check_cells(v.cpu().numpy(), ost[1].V[l][:, 20:28], f"V l{l} (two-slot pass)")
    for l in range(cfg.n_layers):
        k, v = st.read_kv(0, l, 0, 14)
        check_cells(k.cpu().numpy(), ost[0].K[l][:, :14], f"K l{l} (slot 0)")
        check_cells(v.cpu().numpy(), ost[0].V[l][:, :14], f"V l{l} (slot 0)")
    assert st.take_status() == 0

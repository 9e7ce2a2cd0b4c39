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


def test_two_chained_cycles():
    from dflash_block_drafter_gb300.runtime import DraftModel, DraftState, accept, commit_positions
    cfg = synth.CONFIGS["tiny"]
    seed, n_ctx, B = 81, 64, 8
    ck = synth.make_checkpoint(cfg, seed=seed)
    model, om = DraftModel(cfg, ck), O.Model(cfg, ck)
    st = DraftState(model, 1, 128)
    ost = O.State(cfg, 128)
    taps = synth.make_taps(cfg, n_ctx, seed=seed)
    st.fuse(0, torch.as_tensor(taps.view(np.int16), device="cuda"), device_ids(np.arange(n_ctx)))
    O.fuse_context(om, ost, taps, np.arange(n_ctx))
    anchor = int(synth.make_token_ids(cfg, 1, seed=seed)[0])
    st.anchor_tok[0], st.anchor_pos[0], st.block_len[0] = anchor, n_ctx, B

    # cycle 1: the verifier agrees with the first two drafts (both clear of ties)
    r1 = O.draft_block(om, ost, anchor, n_ctx, B)
    assert np.all(r1.top2_gap[:3] > 1e-2)
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

"""The allocation-free LM-head argmax entry point (dflash_head_argmax_static).

Some callers cannot allocate device memory -- code running inside CUDA graph
capture, engines that reserve all device memory up front as their own arena,
loops that must never enter the allocator -- so they cannot create a
dflash_state.  dflash_head_argmax_static serves them from a fixed scratch
array inside the library.  This test calls it through the C ABI twice in a
row, on two different sets of final hidden rows, and checks each result
against the drafts the regular entry point (dflash_draft_block) produced for
the same rows.  It lives in its own file so that it is collected last."""
import ctypes

import numpy as np
import pytest

from gpu_helpers import build_lib, device_ids, need_gpu, synth, torch

pytestmark = pytest.mark.gpu


def test_head_argmax_static_matches_draft_block_twice():
    need_gpu()
    build_lib()
    import dflash_block_drafter_gb300 as D
    from dflash_block_drafter_gb300.runtime import DraftModel, DraftState

    lib = D.load_library()
    cfg = synth.CONFIGS["tiny"]
    ck = synth.make_checkpoint(cfg, seed=41)
    model = DraftModel(cfg, ck)
    st = DraftState(model, 1, 128)
    taps = synth.make_taps(cfg, cfg.ctx, seed=41)
    st.fuse(0, torch.as_tensor(taps.view(np.int16), device="cuda"), device_ids(np.arange(cfg.ctx)))
    ids = torch.full((8,), -5, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    for call, anchor in enumerate((7, 900)):
        # the regular path: a draft pass that also returns its final hidden rows
        st.anchor_tok[0], st.anchor_pos[0], st.block_len[0] = anchor, cfg.ctx, 8
        st.draft(1)
        torch.cuda.synchronize()
        hidden = st.final_hidden[0].clone()
        want = st.drafts[0].cpu().numpy()
        # the allocation-free path on the same rows, through the C ABI
        rc = lib.dflash_head_argmax_static(ctypes.c_void_p(model.handle), ctypes.c_void_p(hidden.data_ptr()), 8,
                                           ctypes.c_void_p(ids.data_ptr()), ctypes.c_void_p(status.data_ptr()),
                                           ctypes.c_void_p(stream))
        assert rc == D.DFLASH_OK, D.status_string(rc)
        torch.cuda.synchronize()
        got = ids.cpu().numpy()
        assert int(status.item()) == 0
        assert np.array_equal(got[1:], want), f"call {call}: {got[1:]} vs draft pass {want}"
        assert 0 <= got[0] < cfg.vocab
    # sizes beyond the fixed scratch are refused
    rc = lib.dflash_head_argmax_static(ctypes.c_void_p(model.handle), ctypes.c_void_p(hidden.data_ptr()), 9,
                                       ctypes.c_void_p(ids.data_ptr()), None, ctypes.c_void_p(stream))
    assert rc == D.DFLASH_ERR_CAPACITY
    st.close()
    model.close()

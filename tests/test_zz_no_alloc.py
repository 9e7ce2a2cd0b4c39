"""The allocation-free LM-head argmax entry point (dflash_head_argmax_static).

Some callers cannot allocate device memory -- code running inside CUDA graph
capture, engines that reserve all device memory up front as their own arena,
loops that must never enter the allocator -- so they cannot create a
dflash_state.  dflash_head_argmax_static serves them from a fixed scratch
array inside the library.  These tests call it through the C ABI: twice in a
row on two sets of final hidden rows, on fewer than 8 rows, inside a captured
CUDA graph and at the full vocabulary, and check each result against the
drafts the regular entry point (dflash_draft_block) produced for the same
rows and against a brute-force argmax of head . row in the CPU oracle's
float64 (wherever its top-2 gap exceeds 1e-2).  The file is collected last."""
import ctypes

import numpy as np
import pytest

from gpu_helpers import GAP, O, build_lib, device_ids, need_gpu, synth, torch

pytestmark = pytest.mark.gpu


def _static(lib, model, hidden, n_rows, ids, status, stream):
    return lib.dflash_head_argmax_static(ctypes.c_void_p(model.handle), ctypes.c_void_p(hidden.data_ptr()), n_rows,
                                         ctypes.c_void_p(ids.data_ptr()),
                                         ctypes.c_void_p(status.data_ptr()) if status is not None else None,
                                         ctypes.c_void_p(stream))


def _oracle_ids(head_bits, rows):
    """Brute-force argmax (lowest id on ties) of head . row in float64, and
    each row's top-1 / top-2 gap."""
    head = O.decode_bf16(head_bits)
    logits = np.asarray(rows, np.float64) @ head.T
    ids = np.argmax(logits, axis=-1)
    part = np.partition(logits, -2, axis=-1)
    return ids, part[:, -1] - part[:, -2]


def _check_vs_oracle(got, head_bits, rows, what):
    want, gap = _oracle_ids(head_bits, rows)
    sure = gap > GAP
    assert sure.any(), what
    assert np.array_equal(np.asarray(got)[sure], want[sure]), f"{what}: {got} vs oracle {want} (gaps {gap})"


def _drafted(st, cfg, anchor):
    st.anchor_tok[0], st.anchor_pos[0], st.block_len[0] = anchor, cfg.ctx, 8
    st.draft(1)
    torch.cuda.synchronize()
    return st.final_hidden[0].clone(), st.drafts[0].cpu().numpy()


def test_head_argmax_static_tiny():
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
    # two calls in a row on different rows: the draft pass's drafts and the oracle
    for call, anchor in enumerate((7, 900)):
        hidden, want = _drafted(st, cfg, anchor)
        rc = _static(lib, model, hidden, 8, ids, status, stream)
        assert rc == D.DFLASH_OK, D.status_string(rc)
        torch.cuda.synchronize()
        got = ids.cpu().numpy()
        assert int(status.item()) == 0
        assert np.array_equal(got[1:], want), f"call {call}: {got[1:]} vs draft pass {want}"
        _check_vs_oracle(got, ck["head"], hidden.cpu().numpy(), f"call {call}")
    # fewer rows: rows 3..7 of the scratch are zero and ids[3..7] are not written
    ids.fill_(-5)
    rc = _static(lib, model, hidden, 3, ids, status, stream)
    assert rc == D.DFLASH_OK
    torch.cuda.synchronize()
    got = ids.cpu().numpy()
    assert np.all(got[3:] == -5), got
    _check_vs_oracle(got[:3], ck["head"], hidden[:3].cpu().numpy(), "3 rows")
    # inside a captured CUDA graph (the device's first call above did the set-up)
    ids.fill_(-5)
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.graph(g, stream=s):
        rc = _static(lib, model, hidden, 8, ids, status, s.cuda_stream)
    assert rc == D.DFLASH_OK
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(ids.cpu().numpy()[1:], want), "graph replay"
    # sizes beyond the fixed scratch are refused
    rc = _static(lib, model, hidden, 9, ids, None, stream)
    assert rc == D.DFLASH_ERR_CAPACITY
    assert int(status.item()) == 0
    st.close()
    model.close()


def test_head_argmax_static_full_vocab():
    """The LM head at vocabulary 151936 over the GEMV grid of every SM."""
    need_gpu()
    build_lib()
    import dflash_block_drafter_gb300 as D
    from dflash_block_drafter_gb300.runtime import DraftModel, DraftState

    lib = D.load_library()
    cfg = synth.CONFIGS["full_bf16"].with_(ctx=64)
    ck = synth.make_checkpoint(cfg, seed=44)
    model = DraftModel(cfg, ck)
    st = DraftState(model, 1, 128)
    taps = synth.make_taps(cfg, cfg.ctx, seed=44)
    st.fuse(0, torch.as_tensor(taps.view(np.int16), device="cuda"), device_ids(np.arange(cfg.ctx)))
    ids = torch.full((8,), -5, dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    for call, anchor in enumerate((11, 123456)):
        hidden, want = _drafted(st, cfg, anchor)
        rc = _static(lib, model, hidden, 8, ids, status, stream)
        assert rc == D.DFLASH_OK, D.status_string(rc)
        torch.cuda.synchronize()
        got = ids.cpu().numpy()
        assert int(status.item()) == 0
        assert np.array_equal(got[1:], want), f"call {call}: {got[1:]} vs draft pass {want}"
        _check_vs_oracle(got, ck["head"], hidden.cpu().numpy(), f"full vocab call {call}")
    st.close()
    model.close()

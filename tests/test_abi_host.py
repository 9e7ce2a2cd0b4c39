"""Host-side checks of the C ABI: the library builds and loads, exports every
entry point include/dflash.h declares, and rejects bad arguments
synchronously.  No GPU is used (no compute call is made)."""
import ctypes
import os
import shutil

import pytest

import dflash_block_drafter_gb300 as D
import dflash_synth as synth


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(D.LIB_PATH):
        if not shutil.which("nvcc") and not os.path.exists("/usr/local/cuda/bin/nvcc"):
            pytest.skip("nvcc unavailable and libdflash not built")
        from dflash_block_drafter_gb300 import build
        build.build()
    return D.load_library()


def _cfg(name="tiny", **kw):
    c = synth.CONFIGS[name].with_(**kw) if kw else synth.CONFIGS[name]
    return D.make_config(c.n_layers, c.hidden, c.n_q_heads, c.n_kv_heads, c.head_dim, c.intermediate, c.vocab,
                         c.n_taps, c.rope_theta, c.norm_eps, c.mask_token_id, c.weight_type)


def test_exports_every_declared_entry_point(lib):
    names = D.header_functions()
    assert "dflash_fuse_context" in names and "dflash_draft_block" in names and "dflash_accept" in names
    for n in names:
        assert hasattr(lib, n), n
        assert n in D._SIGS, f"binding lacks {n}"


def test_status_strings(lib):
    assert D.status_string(D.DFLASH_OK) == "ok"
    assert "invalid" in D.status_string(D.DFLASH_ERR_INVALID_ARG)
    assert D.status_string(12345) == "unknown status"


@pytest.mark.parametrize("name", list(synth.CONFIGS))
def test_config_check_accepts_workloads(lib, name):
    assert D.dflash_config_check(_cfg(name)) == D.DFLASH_OK


def test_config_check_rejects(lib):
    bad = [
        (dict(head_dim=96), D.DFLASH_ERR_UNSUPPORTED),
        (dict(n_q_heads=5, n_kv_heads=2), D.DFLASH_ERR_UNSUPPORTED),
        (dict(hidden=300), D.DFLASH_ERR_UNSUPPORTED),
        (dict(hidden=8448), D.DFLASH_ERR_UNSUPPORTED),
        (dict(intermediate=100), D.DFLASH_ERR_UNSUPPORTED),
        (dict(n_layers=0), D.DFLASH_ERR_UNSUPPORTED),
        (dict(n_layers=9), D.DFLASH_ERR_UNSUPPORTED),
        (dict(vocab=1), D.DFLASH_ERR_UNSUPPORTED),
    ]
    for kw, want in bad:
        assert D.dflash_config_check(_cfg(**kw)) == want, kw
    c = _cfg()
    c.mask_token_id = c.vocab
    assert D.dflash_config_check(c) == D.DFLASH_ERR_INVALID_ARG
    c = _cfg()
    c.rope_theta = 0.0
    assert D.dflash_config_check(c) == D.DFLASH_ERR_INVALID_ARG
    c = _cfg()
    c.weight_type = 7
    assert D.dflash_config_check(c) == D.DFLASH_ERR_UNSUPPORTED
    c = _cfg()
    c.attn_window = -1
    assert D.dflash_config_check(c) == D.DFLASH_ERR_INVALID_ARG
    c = _cfg()
    c.attn_window = 32768  # the pages' default drafter window is a valid model setting
    assert D.dflash_config_check(c) == D.DFLASH_OK
    assert lib.dflash_config_check(None) == D.DFLASH_ERR_INVALID_ARG


def test_null_and_range_arguments_rejected(lib):
    P = ctypes.c_void_p
    out = P()
    assert lib.dflash_model_create(None, None, ctypes.byref(out)) == D.DFLASH_ERR_INVALID_ARG
    cfg = _cfg()
    assert lib.dflash_model_create(ctypes.byref(cfg), ctypes.byref(D.DflashWeights()),
                                   ctypes.byref(out)) == D.DFLASH_ERR_INVALID_ARG
    assert lib.dflash_model_destroy(None) == D.DFLASH_ERR_INVALID_ARG
    assert lib.dflash_state_create(None, 1, 64, ctypes.byref(out)) == D.DFLASH_ERR_INVALID_ARG
    assert lib.dflash_state_destroy(None) == D.DFLASH_ERR_INVALID_ARG
    assert lib.dflash_fuse_context(None, None, 0, None, None, 1, None, None) == D.DFLASH_ERR_INVALID_ARG
    assert lib.dflash_draft_block(None, None, 1, None, None, None, None, None, None, None) == D.DFLASH_ERR_INVALID_ARG
    # accept: sizes are validated before anything touches the device
    fake = P(16)
    for n_seq, maxb in ((0, 8), (1, 1), (1, 9)):
        assert lib.dflash_accept(fake, fake, fake, n_seq, maxb, fake, fake, None, None) == D.DFLASH_ERR_INVALID_ARG
    assert lib.dflash_accept(None, fake, fake, 1, 8, fake, fake, None, None) == D.DFLASH_ERR_INVALID_ARG
    assert lib.dflash_commit_positions(None, fake, 1, fake, None) == D.DFLASH_ERR_INVALID_ARG
    assert lib.dflash_commit_positions(fake, fake, 0, fake, None) == D.DFLASH_ERR_INVALID_ARG
    assert lib.dflash_state_set_spec_min_p(None, 0.5) == D.DFLASH_ERR_INVALID_ARG
    assert lib.dflash_state_read_draft_probs(None, fake, None) == D.DFLASH_ERR_INVALID_ARG
    assert lib.dflash_state_read_kv(None, 0, 0, 0, 1, None, None, None) == D.DFLASH_ERR_INVALID_ARG
    assert lib.dflash_state_write_kv(None, 0, 0, 0, 1, None, None, None) == D.DFLASH_ERR_INVALID_ARG
    st = ctypes.c_int32()
    assert lib.dflash_state_status(None, ctypes.byref(st), None) == D.DFLASH_ERR_INVALID_ARG
    assert lib.dflash_model_dequantize(None, 0, fake, None) == D.DFLASH_ERR_INVALID_ARG


def test_binding_raises_on_error(lib):
    with pytest.raises(D.DflashError) as e:
        D.dflash_state_destroy(0)
    assert e.value.status == D.DFLASH_ERR_INVALID_ARG

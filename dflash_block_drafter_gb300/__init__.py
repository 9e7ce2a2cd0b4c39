"""Python binding of libdflash, the GB300 (sm_103a) DFlash block-draft pass.

Argument marshalling only: every function here forwards to the C ABI of the
same name (include/dflash.h) through ctypes; all computation happens in the
library's CUDA kernels.  Device buffers are passed as integer addresses (for
example ``torch.Tensor.data_ptr()``) and streams as ``cudaStream_t`` integers
(``torch.cuda.current_stream().cuda_stream``).  There is no CPU fallback:
loading fails loudly when the library has not been built.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Dict, Optional

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "lib", "libdflash.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG), "include", "dflash.h")

# ------------------------------------------------------------------ constants
DFLASH_OK = 0
DFLASH_ERR_INVALID_ARG = 1
DFLASH_ERR_UNSUPPORTED = 2
DFLASH_ERR_CAPACITY = 3
DFLASH_ERR_CUDA = 4
DFLASH_ERR_NO_DEVICE = 5
DFLASH_ERR_OUT_OF_MEMORY = 6

DFLASH_DEV_NONFINITE = 1
DFLASH_DEV_BAD_TOKEN = 2
DFLASH_DEV_CAPACITY = 4
DFLASH_DEV_BAD_BLOCK = 8
DFLASH_DEV_TIMEOUT = 16

DFLASH_WT_BF16 = 0
DFLASH_WT_Q8_0 = 1
DFLASH_WT_Q5_0 = 2
DFLASH_WT_Q4_0 = 3
WEIGHT_TYPE_IDS = {"bf16": DFLASH_WT_BF16, "q8_0": DFLASH_WT_Q8_0, "q5_0": DFLASH_WT_Q5_0, "q4_0": DFLASH_WT_Q4_0}

DFLASH_MAX_LAYERS = 8
DFLASH_MAX_BLOCK = 8
DFLASH_MIN_BLOCK = 2
DFLASH_MAX_SLOTS = 16


class DflashError(RuntimeError):
    def __init__(self, status: int, what: str):
        detail = ""
        if status == DFLASH_ERR_CUDA and _lib is not None:
            detail = " (" + _lib.dflash_last_cuda_error().decode() + ")"
        super().__init__(f"{what}: {status_string(status)}{detail}")
        self.status = status


# ------------------------------------------------------------------ structs
class DflashConfig(ctypes.Structure):
    _fields_ = [
        ("n_layers", ctypes.c_int32), ("hidden", ctypes.c_int32), ("n_q_heads", ctypes.c_int32),
        ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("intermediate", ctypes.c_int32),
        ("vocab", ctypes.c_int32), ("n_taps", ctypes.c_int32), ("rope_theta", ctypes.c_float),
        ("norm_eps", ctypes.c_float), ("mask_token_id", ctypes.c_int32), ("weight_type", ctypes.c_int32),
        ("attn_window", ctypes.c_int32),
    ]


_LAYER_FIELDS = ("attn_norm", "wq", "wk", "wv", "q_norm", "k_norm", "wo", "mlp_norm", "w_gate", "w_up", "w_down")


class DflashLayerWeights(ctypes.Structure):
    _fields_ = [(f, ctypes.c_void_p) for f in _LAYER_FIELDS]


class DflashWeights(ctypes.Structure):
    _fields_ = [
        ("fc", ctypes.c_void_p), ("hidden_norm", ctypes.c_void_p),
        ("layers", DflashLayerWeights * DFLASH_MAX_LAYERS),
        ("final_norm", ctypes.c_void_p), ("embed", ctypes.c_void_p), ("head", ctypes.c_void_p),
    ]


# ------------------------------------------------------------------ loading
_lib: Optional[ctypes.CDLL] = None

_P = ctypes.c_void_p
_I = ctypes.c_int32
_SIGS = {
    "dflash_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "dflash_last_cuda_error": (ctypes.c_char_p, []),
    "dflash_config_check": (ctypes.c_int, [ctypes.POINTER(DflashConfig)]),
    "dflash_model_create": (ctypes.c_int, [ctypes.POINTER(DflashConfig), ctypes.POINTER(DflashWeights),
                                           ctypes.POINTER(_P)]),
    "dflash_model_destroy": (ctypes.c_int, [_P]),
    "dflash_model_device_bytes": (ctypes.c_size_t, [_P]),
    "dflash_state_create": (ctypes.c_int, [_P, _I, _I, ctypes.POINTER(_P)]),
    "dflash_state_destroy": (ctypes.c_int, [_P]),
    "dflash_state_device_bytes": (ctypes.c_size_t, [_P]),
    "dflash_fuse_context": (ctypes.c_int, [_P, _P, _I, _P, _P, _I, _P, _P]),
    "dflash_draft_block": (ctypes.c_int, [_P, _P, _I, _P, _P, _P, _P, _P, _P, _P]),
    "dflash_accept": (ctypes.c_int, [_P, _P, _P, _I, _I, _P, _P, _P, _P]),
    "dflash_commit_positions": (ctypes.c_int, [_P, _P, _I, _P, _P]),
    "dflash_state_read_kv": (ctypes.c_int, [_P, _I, _I, _I, _I, _P, _P, _P]),
    "dflash_state_write_kv": (ctypes.c_int, [_P, _I, _I, _I, _I, _P, _P, _P]),
    "dflash_state_status": (ctypes.c_int, [_P, ctypes.POINTER(_I), _P]),
    "dflash_model_dequantize": (ctypes.c_int, [_P, _I, _P, _P]),
    "dflash_draft_launches": (ctypes.c_int32, [_P, _I]),
    "dflash_fuse_launches": (ctypes.c_int32, [_P, _I]),
    "dflash_state_set_head_events": (ctypes.c_int, [_P, _P, _P]),
    "dflash_state_set_profile_events": (ctypes.c_int, [_P, ctypes.POINTER(_P), _I]),
    "dflash_state_set_attn_chunks": (ctypes.c_int, [_P, _I, ctypes.POINTER(_I)]),
    "dflash_state_set_spec_min_p": (ctypes.c_int, [_P, ctypes.c_float]),
    "dflash_state_set_defer_kv": (ctypes.c_int, [_P, _I]),
    "dflash_state_flush": (ctypes.c_int, [_P, _P]),
    "dflash_state_read_draft_probs": (ctypes.c_int, [_P, _P, _P]),
    "dflash_head_argmax_static": (ctypes.c_int, [_P, _P, _I, _P, _P, _P]),
}


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libdflash (built by ``dflash_block_drafter_gb300.build``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"libdflash is not built ({path} missing); run "
                          "`python -m dflash_block_drafter_gb300.build`")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def header_functions(path: str = HEADER_PATH):
    """Names of the entry points include/dflash.h declares."""
    with open(path) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dflash_[a-z_0-9]+)\s*\(", text)))


def _check(status: int, what: str) -> None:
    if status != DFLASH_OK:
        raise DflashError(status, what)


def status_string(status: int) -> str:
    lib = load_library()
    return lib.dflash_status_string(int(status)).decode()


# ------------------------------------------------------------- C entry points
def dflash_status_string(status: int) -> str:
    return status_string(status)


def dflash_last_cuda_error() -> str:
    return load_library().dflash_last_cuda_error().decode()


def dflash_config_check(cfg: DflashConfig) -> int:
    return load_library().dflash_config_check(ctypes.byref(cfg))


def dflash_model_create(cfg: DflashConfig, weights: DflashWeights) -> int:
    h = _P()
    _check(load_library().dflash_model_create(ctypes.byref(cfg), ctypes.byref(weights), ctypes.byref(h)),
           "dflash_model_create")
    return h.value


def dflash_model_destroy(model: int) -> None:
    _check(load_library().dflash_model_destroy(model), "dflash_model_destroy")


def dflash_model_device_bytes(model: int) -> int:
    return load_library().dflash_model_device_bytes(model)


def dflash_state_create(model: int, n_slots: int, capacity: int) -> int:
    h = _P()
    _check(load_library().dflash_state_create(model, n_slots, capacity, ctypes.byref(h)), "dflash_state_create")
    return h.value


def dflash_state_destroy(state: int) -> None:
    _check(load_library().dflash_state_destroy(state), "dflash_state_destroy")


def dflash_state_device_bytes(state: int) -> int:
    return load_library().dflash_state_device_bytes(state)


def dflash_fuse_context(model: int, state: int, slot: int, taps: int, positions: int, n: int,
                        dev_status: int = 0, stream: int = 0) -> None:
    _check(load_library().dflash_fuse_context(model, state, slot, taps, positions, n, dev_status or None,
                                              stream or None), "dflash_fuse_context")


def dflash_draft_block(model: int, state: int, n_seq: int, anchor_tok: int, anchor_pos: int, block_len: int,
                       drafts: int, final_hidden: int = 0, dev_status: int = 0, stream: int = 0) -> None:
    _check(load_library().dflash_draft_block(model, state, n_seq, anchor_tok, anchor_pos, block_len, drafts,
                                             final_hidden or None, dev_status or None, stream or None),
           "dflash_draft_block")


def dflash_accept(drafts: int, target_ids: int, block_len: int, n_seq: int, max_block_len: int,
                  accept_len: int, next_anchor: int, anchor_pos_inout: int = 0, stream: int = 0) -> None:
    _check(load_library().dflash_accept(drafts, target_ids, block_len, n_seq, max_block_len, accept_len,
                                        next_anchor, anchor_pos_inout or None, stream or None), "dflash_accept")


def dflash_commit_positions(anchor_pos: int, accept_len: int, n_seq: int, positions: int, stream: int = 0) -> None:
    _check(load_library().dflash_commit_positions(anchor_pos, accept_len, n_seq, positions, stream or None),
           "dflash_commit_positions")


def dflash_state_read_kv(state: int, slot: int, layer: int, pos0: int, n: int, k_out: int, v_out: int,
                         stream: int = 0) -> None:
    _check(load_library().dflash_state_read_kv(state, slot, layer, pos0, n, k_out or None, v_out or None,
                                               stream or None), "dflash_state_read_kv")


def dflash_state_write_kv(state: int, slot: int, layer: int, pos0: int, n: int, k_in: int, v_in: int,
                          stream: int = 0) -> None:
    _check(load_library().dflash_state_write_kv(state, slot, layer, pos0, n, k_in or None, v_in or None,
                                                stream or None), "dflash_state_write_kv")


def dflash_state_status(state: int, stream: int = 0) -> int:
    out = _I()
    _check(load_library().dflash_state_status(state, ctypes.byref(out), stream or None), "dflash_state_status")
    return out.value


def dflash_model_dequantize(model: int, which: int, out: int, stream: int = 0) -> None:
    _check(load_library().dflash_model_dequantize(model, which, out, stream or None), "dflash_model_dequantize")


# ------------------------------------------------------------ marshalling aid
def make_config(n_layers, hidden, n_q_heads, n_kv_heads, head_dim, intermediate, vocab, n_taps=5,
                rope_theta=1e7, norm_eps=1e-6, mask_token_id=None, weight_type="bf16",
                attn_window=0) -> DflashConfig:
    wt = WEIGHT_TYPE_IDS[weight_type] if isinstance(weight_type, str) else int(weight_type)
    return DflashConfig(n_layers, hidden, n_q_heads, n_kv_heads, head_dim, intermediate, vocab, n_taps,
                        rope_theta, norm_eps, vocab - 1 if mask_token_id is None else mask_token_id, wt,
                        attn_window)


def make_weights(ptrs: Dict[str, int], n_layers: int) -> DflashWeights:
    """DflashWeights from a name -> device address dict using the tensor
    names fc, hidden_norm, layers.{l}.{attn_norm,wq,...}, final_norm, embed,
    head."""
    w = DflashWeights()
    w.fc = ptrs["fc"]
    w.hidden_norm = ptrs["hidden_norm"]
    w.final_norm = ptrs["final_norm"]
    w.embed = ptrs["embed"]
    w.head = ptrs["head"]
    for l in range(n_layers):
        lw = w.layers[l]
        for f in _LAYER_FIELDS:
            setattr(lw, f, ptrs[f"layers.{l}.{f}"])
    return w


def dflash_draft_launches(state: int, n_seq: int) -> int:
    return load_library().dflash_draft_launches(state, n_seq)


def dflash_fuse_launches(state: int, n: int) -> int:
    return load_library().dflash_fuse_launches(state, n)


def dflash_state_set_head_events(state: int, ev_begin: int, ev_end: int) -> None:
    _check(load_library().dflash_state_set_head_events(state, ev_begin or None, ev_end or None),
           "dflash_state_set_head_events")


def dflash_head_argmax_static(model: int, hidden: int, n_rows: int, ids: int, dev_status: int = 0,
                              stream: int = 0) -> None:
    """LM-head argmax of up to 8 final-hidden rows using only the library's
    fixed scratch array (no device allocation); see include/dflash.h."""
    _check(load_library().dflash_head_argmax_static(model, hidden, n_rows, ids, dev_status or None,
                                                    stream or None), "dflash_head_argmax_static")


def dflash_state_set_profile_events(state: int, events) -> None:
    """events: list of cudaEvent_t integers (empty list switches profiling off)."""
    arr = (_P * max(1, len(events)))(*events) if events else None
    _check(load_library().dflash_state_set_profile_events(state, arr, len(events)),
           "dflash_state_set_profile_events")


def dflash_state_set_spec_min_p(state: int, floor: float) -> None:
    _check(load_library().dflash_state_set_spec_min_p(state, floor), "dflash_state_set_spec_min_p")


def dflash_state_set_defer_kv(state: int, on: bool) -> None:
    _check(load_library().dflash_state_set_defer_kv(state, 1 if on else 0), "dflash_state_set_defer_kv")


def dflash_state_flush(state: int, stream: int = 0) -> None:
    _check(load_library().dflash_state_flush(state, stream or None), "dflash_state_flush")


def dflash_state_read_draft_probs(state: int, out: int, stream: int = 0) -> None:
    """Copy the last pass's [n_slots, 7] float draft confidences to out (device)."""
    _check(load_library().dflash_state_read_draft_probs(state, out, stream or None), "dflash_state_read_draft_probs")


def dflash_state_set_attn_chunks(state: int, chunks: int = 0) -> int:
    """Set the attention's context chunks per (sequence, kv head) (0: query
    only); returns the maximum the state supports."""
    mx = _I()
    _check(load_library().dflash_state_set_attn_chunks(state, chunks, ctypes.byref(mx)),
           "dflash_state_set_attn_chunks")
    return mx.value

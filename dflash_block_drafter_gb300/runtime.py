"""Device-memory plumbing around the libdflash C ABI, using PyTorch tensors.

PyTorch only allocates device memory and provides streams here; every step of
the draft pass runs in libdflash's CUDA kernels through the ctypes binding.
"""
from __future__ import annotations

from typing import Dict, Optional

import numpy as np
import torch

from . import (DFLASH_MAX_BLOCK, dflash_accept, dflash_commit_positions, dflash_draft_block, dflash_fuse_context,
               dflash_model_create, dflash_model_dequantize, dflash_model_destroy, dflash_model_device_bytes, dflash_state_create,
               dflash_state_destroy, dflash_state_device_bytes, dflash_state_read_kv, dflash_state_status,
               dflash_state_read_draft_probs, dflash_state_set_spec_min_p, dflash_state_write_kv, load_library,
               dflash_state_set_defer_kv, dflash_state_flush,
               make_config, make_weights)


def _stream(stream: Optional[torch.cuda.Stream] = None) -> int:
    return (stream or torch.cuda.current_stream()).cuda_stream


def to_device(arr: np.ndarray, device) -> torch.Tensor:
    """Copy a numpy array's bytes to the device (uint16 travels as int16)."""
    a = np.ascontiguousarray(arr)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).to(device)


class DraftModel:
    """A libdflash model built from a checkpoint dict (numpy arrays of BF16
    bits / GGUF bytes, names as in include/dflash.h).  Keeps the borrowed
    embedding and LM head alive for the model's lifetime."""

    def __init__(self, cfg, ckpt: Dict[str, np.ndarray], device="cuda:0", keep_sources: bool = False):
        load_library()
        self.cfg = cfg
        self.device = torch.device(device)
        self.ccfg = make_config(cfg.n_layers, cfg.hidden, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim,
                                cfg.intermediate, cfg.vocab, cfg.n_taps, cfg.rope_theta, cfg.norm_eps,
                                cfg.mask_token_id, cfg.weight_type, getattr(cfg, "attn_window", 0))
        with torch.cuda.device(self.device):
            src = {k: to_device(v, self.device) for k, v in ckpt.items()}
            ptrs = {k: t.data_ptr() for k, t in src.items()}
            w = make_weights(ptrs, cfg.n_layers)
            self.handle = dflash_model_create(self.ccfg, w)
        # the target's embedding and LM head are borrowed, the rest was copied
        self.embed = src["embed"]
        self.head = src["head"]
        self.sources = src if keep_sources else None
        del src

    @property
    def device_bytes(self) -> int:
        return dflash_model_device_bytes(self.handle)

    def dequantize(self, which: int) -> torch.Tensor:
        cfg = self.cfg
        shapes = list(cfg.matrix_shapes().values())
        names = ["fc"] + [f"layers.{l}.{t}" for l in range(cfg.n_layers)
                          for t in ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down")]
        n, k = cfg.matrix_shapes()[names[which]]
        out = torch.empty((n, k), dtype=torch.float32, device=self.device)
        dflash_model_dequantize(self.handle, which, out.data_ptr(), _stream())
        return out

    def close(self):
        if getattr(self, "handle", None):
            dflash_model_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class DraftState:
    """A libdflash state (per-slot FP16 K/V + pass workspace) with
    preallocated device I/O buffers."""

    def __init__(self, model: DraftModel, n_slots: int, capacity: int):
        self.model = model
        self.n_slots = n_slots
        self.capacity = capacity
        dev = model.device
        with torch.cuda.device(dev):
            self.handle = dflash_state_create(model.handle, n_slots, capacity)
        cfg = model.cfg
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.drafts = torch.full((n_slots, DFLASH_MAX_BLOCK - 1), -7, dtype=torch.int32, device=dev)
        self.final_hidden = torch.zeros((n_slots, 8, cfg.hidden), dtype=torch.float32, device=dev)
        self.anchor_tok = torch.zeros(n_slots, dtype=torch.int32, device=dev)
        self.anchor_pos = torch.zeros(n_slots, dtype=torch.int32, device=dev)
        self.block_len = torch.zeros(n_slots, dtype=torch.int32, device=dev)

    @property
    def device_bytes(self) -> int:
        return dflash_state_device_bytes(self.handle)

    def fuse(self, slot: int, taps: torch.Tensor, positions: torch.Tensor, stream=None) -> None:
        assert taps.is_cuda and positions.is_cuda and positions.dtype == torch.int32
        n = positions.numel()
        dflash_fuse_context(self.model.handle, self.handle, slot, taps.data_ptr(), positions.data_ptr(), n,
                            self.status.data_ptr(), _stream(stream))
        # a deferring state reads the positions again in a later call: keep them alive
        self._kept_positions = positions if getattr(self, "_defer_kv", False) and n <= 8 else None

    def draft(self, n_seq: int, want_hidden: bool = True, stream=None) -> None:
        """Draft with the anchor_tok / anchor_pos / block_len buffers as set."""
        dflash_draft_block(self.model.handle, self.handle, n_seq, self.anchor_tok.data_ptr(),
                           self.anchor_pos.data_ptr(), self.block_len.data_ptr(), self.drafts.data_ptr(),
                           self.final_hidden.data_ptr() if want_hidden else 0, self.status.data_ptr(),
                           _stream(stream))

    def read_kv(self, slot: int, layer: int, pos0: int, n: int):
        cfg = self.model.cfg
        k = torch.empty((cfg.n_kv_heads, n, cfg.head_dim), dtype=torch.float32, device=self.model.device)
        v = torch.empty_like(k)
        dflash_state_read_kv(self.handle, slot, layer, pos0, n, k.data_ptr(), v.data_ptr(), _stream())
        return k, v

    def write_kv(self, slot: int, layer: int, pos0: int, k16: torch.Tensor, v16: torch.Tensor) -> None:
        """k16, v16: float16 / int16 tensors [n_kv, n, d] on the device."""
        n = k16.shape[1]
        dflash_state_write_kv(self.handle, slot, layer, pos0, n, k16.data_ptr(), v16.data_ptr(), _stream())

    def set_defer_kv(self, on: bool) -> None:
        """Leave the K/V of 8-position fusions to the next one-slot draft pass."""
        dflash_state_set_defer_kv(self.handle, on)
        self._defer_kv = bool(on)

    def flush(self, stream=None) -> None:
        """Project the K/V of rows a deferring fusion kept, now."""
        dflash_state_flush(self.handle, _stream(stream))

    def set_spec_min_p(self, floor: float) -> None:
        """Confidence floor of the offered drafts (0: all)."""
        dflash_state_set_spec_min_p(self.handle, floor)

    def draft_probs(self) -> torch.Tensor:
        """[n_slots, 7] float confidences of the last pass's drafts (-1: none)."""
        out = torch.empty((self.n_slots, DFLASH_MAX_BLOCK - 1), dtype=torch.float32, device=self.model.device)
        dflash_state_read_draft_probs(self.handle, out.data_ptr(), _stream())
        return out

    def take_status(self) -> int:
        torch.cuda.synchronize(self.model.device)
        v = int(self.status.item())
        self.status.zero_()
        return v

    def close(self):
        if getattr(self, "handle", None):
            dflash_state_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def accept(drafts: torch.Tensor, target_ids: torch.Tensor, block_len: torch.Tensor, accept_len: torch.Tensor,
           next_anchor: torch.Tensor, anchor_pos: Optional[torch.Tensor] = None, stream=None) -> None:
    n_seq, max_b = target_ids.shape
    dflash_accept(drafts.data_ptr(), target_ids.data_ptr(), block_len.data_ptr(), n_seq, max_b,
                  accept_len.data_ptr(), next_anchor.data_ptr(), anchor_pos.data_ptr() if anchor_pos is not None
                  else 0, _stream(stream))


def commit_positions(anchor_pos: torch.Tensor, accept_len: torch.Tensor, positions: torch.Tensor,
                     stream=None) -> None:
    """positions [n_seq, 8] <- the rows the next fusion commits (-1: none)."""
    dflash_commit_positions(anchor_pos.data_ptr(), accept_len.data_ptr(), accept_len.numel(),
                            positions.data_ptr(), _stream(stream))

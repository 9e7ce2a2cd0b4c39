"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI
and the CPU oracle on the same seeded inputs, and the tolerances they are
compared with."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import dflash_synth as synth  # noqa: E402
from oracle import dflash_oracle as O  # noqa: E402

# Tolerances of the GPU-vs-oracle comparisons:
#  * final hidden states: max |err| <= 3e-2 x row RMS (the pass's stated bar);
#  * K/V cells (FP16 on both sides): max |err| <= 2e-2 x RMS of the cells and
#    mean |err| <= 2e-3 x RMS (one FP16 rounding, 2^-11 relative, of values
#    that pass through fp32 sums of up to 12800 terms, with margin for the
#    BF16 / FP16 rounding of the projections' operands);
#  * drafts: identical wherever the oracle's top-1/top-2 logit gap > 1e-2;
#  * dequantised weights, accept lengths and bonus tokens: bit-exact.
HIDDEN_REL = 3e-2
KV_MAX_REL = 2e-2
KV_MEAN_REL = 2e-3
GAP = 1e-2


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def build_lib():
    from dflash_block_drafter_gb300 import build
    build.build()


def device_ids(ids) -> "torch.Tensor":
    return torch.as_tensor(np.asarray(ids, dtype=np.int32), device="cuda")


def check_hidden(gpu_rows: np.ndarray, ref_rows: np.ndarray, what: str = "final hidden"):
    rms = np.sqrt(np.mean(ref_rows ** 2, axis=-1, keepdims=True))
    err = np.abs(gpu_rows - ref_rows)
    worst = float(np.max(err / rms))
    assert np.all(np.isfinite(gpu_rows)), f"{what}: non-finite values"
    assert worst <= HIDDEN_REL, f"{what}: max |err| / row RMS = {worst:.3e} > {HIDDEN_REL}"
    return worst


def check_cells(gpu: np.ndarray, ref: np.ndarray, what: str):
    ref = ref.astype(np.float64)
    rms = float(np.sqrt(np.mean(ref ** 2))) + 1e-30
    err = np.abs(gpu.astype(np.float64) - ref)
    assert float(err.max()) <= KV_MAX_REL * rms, f"{what}: max err {err.max():.3e} vs rms {rms:.3e}"
    assert float(err.mean()) <= KV_MEAN_REL * rms, f"{what}: mean err {err.mean():.3e} vs rms {rms:.3e}"


def check_drafts(gpu_drafts: np.ndarray, res: "O.DraftResult", B: int, what: str = "drafts"):
    sure = res.top2_gap > GAP
    got = gpu_drafts[: B - 1]
    assert np.array_equal(got[sure], res.drafts[sure]), f"{what}: {got} vs oracle {res.drafts} (gaps {res.top2_gap})"
    assert np.all(gpu_drafts[B - 1:] == -1), f"{what}: unused entries must be -1: {gpu_drafts}"
    # where the gap is small the GPU's id must still be a near-maximal logit
    for j in np.nonzero(~sure)[0]:
        assert res.logits[j, got[j]] >= res.logits[j].max() - 5 * GAP


def compare_state(state, ostate: "O.State", slot: int, upto: int, what: str):
    cfg = ostate.cfg
    for l in range(cfg.n_layers):
        k, v = state.read_kv(slot, l, 0, upto)
        check_cells(k.cpu().numpy(), ostate.K[l][:, :upto], f"{what} K layer {l}")
        check_cells(v.cpu().numpy(), ostate.V[l][:, :upto], f"{what} V layer {l}")

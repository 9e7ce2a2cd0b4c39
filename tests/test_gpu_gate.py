"""GPU parity of the confidence gate (spec-min-p) against the CPU oracle: the
LM-head kernel's per-draft softmax probability (an online sum of exp over the
whole vocabulary, reduced across CTAs) and the offered prefix under a floor,
for one slot and for two slots in one pass."""
import numpy as np
import pytest

from gpu_helpers import O, build_lib, check_drafts, device_ids, need_gpu, synth, torch

pytestmark = pytest.mark.gpu

# The drafts' logits carry the pass's rounding (final hidden rows within a
# few 1e-3 of their RMS): a confidence p = 1 / sum exp(l - l_max) moves by
# about the logits' absolute error, well under 1e-2 relative here.
PROB_REL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _setup():
    need_gpu()
    build_lib()


def _floor_between(probs):
    """A floor that splits the block's confidences with a clear margin."""
    p = np.sort(np.asarray(probs))
    gaps = [(p[i + 1] / p[i], i) for i in range(len(p) - 1) if p[i] > 0]
    ratio, i = max(gaps)
    assert ratio > 1.04, "confidences too close to split with a margin"
    return float(np.sqrt(p[i] * p[i + 1]))


def _setup_slots(wtype, ctxs, Bs, seed):
    from dflash_block_drafter_gb300.runtime import DraftModel, DraftState
    cfg = synth.CONFIGS["tiny"].with_(weight_type=wtype)
    ck = synth.make_checkpoint(cfg, seed=seed)
    model, om = DraftModel(cfg, ck), O.Model(cfg, ck)
    st = DraftState(model, len(ctxs), 128)
    osts = []
    for s, n in enumerate(ctxs):
        ost = O.State(cfg, 128)
        taps = synth.make_taps(cfg, n, seed=seed, stream=s)
        st.fuse(s, torch.as_tensor(taps.view(np.int16), device="cuda"), device_ids(np.arange(n)))
        O.fuse_context(om, ost, taps, np.arange(n))
        osts.append(ost)
    toks = synth.make_token_ids(cfg, len(ctxs), seed=seed)
    st.anchor_tok[:len(ctxs)] = device_ids(toks)
    st.anchor_pos[:len(ctxs)] = device_ids(ctxs)
    st.block_len[:len(ctxs)] = device_ids(Bs)
    return st, om, osts, toks


CTX12 = [64, 40, 61, 20, 33, 50, 12, 64, 9, 27, 44, 58]
B12 = [8, 6, 2, 7, 3, 8, 4, 5, 8, 2, 6, 7]


# twelve slots: a 128-row pass, whose LM head runs on the tcgen05 tensor cores
@pytest.mark.parametrize("wtype,ctxs,Bs", [("bf16", [64], [8]), ("q4_0", [40, 61], [8, 6]),
                                           ("bf16", CTX12, B12), ("q4_0", CTX12[::-1], B12[::-1])],
                         ids=["bf16-1", "q4_0-2", "bf16-12", "q4_0-12"])
def test_gate_parity(wtype, ctxs, Bs):
    st, om, osts, toks = _setup_slots(wtype, ctxs, Bs, seed=61)
    res = [O.draft_block(om, osts[s], int(toks[s]), ctxs[s], Bs[s]) for s in range(len(ctxs))]
    # confidences under a floor no draft is below: every draft offered
    st.set_spec_min_p(1e-12)
    st.draft(len(ctxs))
    probs = st.draft_probs().cpu().numpy()
    for s, r in enumerate(res):
        B = Bs[s]
        check_drafts(st.drafts[s].cpu().numpy(), r, B, f"slot {s}")
        got = probs[s, :B - 1]
        assert np.all(probs[s, B - 1:] == -1)
        assert np.allclose(got, r.probs, rtol=PROB_REL, atol=0), f"slot {s}: {got} vs {r.probs}"
    # a floor between two confidences of slot 0: the offered prefix follows the oracle's
    floor = _floor_between(res[0].probs)
    st.set_spec_min_p(floor)
    st.draft(len(ctxs))
    torch.cuda.synchronize()
    for s, r in enumerate(res):
        want = O.gate(r.drafts, r.probs, floor)
        got = st.drafts[s, :Bs[s] - 1].cpu().numpy()
        # compare only where the oracle's confidences are clear of the floor
        clear = np.abs(np.log(r.probs / floor)) > 1.5 * PROB_REL
        upto = len(want) if clear.all() else int(np.argmin(clear))
        assert np.array_equal(got[:upto] == -1, want[:upto] == -1), f"slot {s}: {got} vs {want} (floor {floor})"
        sure = (want[:upto] != -1) & (r.top2_gap[:upto] > 1e-2)
        assert np.array_equal(got[:upto][sure], want[:upto][sure]), f"slot {s}: {got} vs {want}"
    # floor 0 (the default) skips the confidences and offers every draft
    st.set_spec_min_p(0.0)
    st.draft(len(ctxs))
    torch.cuda.synchronize()
    assert np.all(st.draft_probs().cpu().numpy() == -1)
    for s, r in enumerate(res):
        check_drafts(st.drafts[s].cpu().numpy(), r, Bs[s], f"slot {s}, floor 0")
    assert st.take_status() == 0


def test_gate_floor_validation():
    from dflash_block_drafter_gb300 import DFLASH_ERR_INVALID_ARG, DflashError
    st, _, _, _ = _setup_slots("bf16", [16], [4], seed=62)
    for bad in (-0.1, 1.5, float("nan")):
        with pytest.raises(DflashError) as e:
            st.set_spec_min_p(bad)
        assert e.value.status == DFLASH_ERR_INVALID_ARG
    st.set_spec_min_p(1.0)  # offers nothing unless a draft is certain
    st.draft(1)
    torch.cuda.synchronize()
    probs = st.draft_probs().cpu().numpy()[0, :3]
    got = st.drafts[0, :3].cpu().numpy()
    assert np.all(probs < 1.0) and np.all(got == -1)

"""GPU parity at the full DFlash geometry (5 layers, hidden 2560, 24Q/2KV x
256, MLP 7680, vocab 151936), in the launch configuration bench.py times:
one sequence, 8-row block, the LM head over the whole vocabulary.

  * BF16, context 8192 built by fusion on both sides (the bench workload);
  * Q8_0 / Q5_0 / Q4_0 backbones, context 8192 pre-filled + 8 fused positions;
  * long context: Q8_0, 262144 pre-filled positions + 8 fused positions;
  * batched mix: 16 sequences, Q4_0, contexts U[2048, 32768], blocks U{2..8}.

The oracle runs the same seeded inputs in float64 (seconds to a minute per
case); outputs are compared element by element (final hidden rows of every
block row, every draft, the K/V cells the pass wrote and sampled context
cells)."""
import numpy as np
import pytest

from gpu_helpers import O, build_lib, check_cells, check_drafts, check_hidden, device_ids, need_gpu, synth, torch

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module", autouse=True)
def _setup():
    need_gpu()
    build_lib()


def _prefill(st, ost, cfg, slot, n, seed):
    kv = synth.make_kv_fill(cfg, n, seed=seed, slot=slot)
    ost.fill(kv, n)
    for l, (k, v) in enumerate(kv):
        st.write_kv(slot, l, 0, torch.as_tensor(k.view(np.int16), device="cuda"),
                    torch.as_tensor(v.view(np.int16), device="cuda"))


def _fuse(st, ost, om, cfg, slot, pos, seed, stream):
    taps = synth.make_taps(cfg, len(pos), seed=seed, stream=stream)
    st.fuse(slot, torch.as_tensor(taps.view(np.int16), device="cuda"), device_ids(pos))
    O.fuse_context(om, ost, taps, pos)


def _check_pass(st, ost, res, slot, p, B, what):
    torch.cuda.synchronize()
    check_hidden(st.final_hidden[slot, :B].cpu().numpy(), res.final_hidden, what)
    check_drafts(st.drafts[slot].cpu().numpy(), res, B, what)
    cfg = ost.cfg
    for l in range(cfg.n_layers):
        lo = max(0, p - 8)
        k, v = st.read_kv(slot, l, lo, p + B - lo)
        check_cells(k.cpu().numpy(), ost.K[l][:, lo:p + B], f"{what} K l{l}")
        check_cells(v.cpu().numpy(), ost.V[l][:, lo:p + B], f"{what} V l{l}")


def test_full_bf16_context_by_fusion():
    from dflash_block_drafter_gb300.runtime import DraftModel, DraftState
    cfg = synth.CONFIGS["full_bf16"]
    ck = synth.make_checkpoint(cfg, seed=0)
    om = O.Model(cfg, ck)
    model = DraftModel(cfg, ck)
    ctx, B = cfg.ctx, cfg.block
    st = DraftState(model, 1, ctx + B)
    ost = O.State(cfg, ctx + B)
    for i, base in enumerate(range(0, ctx, 2048)):
        _fuse(st, ost, om, cfg, 0, np.arange(base, base + 2048), 31, i)
    torch.cuda.synchronize()
    for l in range(cfg.n_layers):  # every context cell of every layer
        k, v = st.read_kv(0, l, 0, ctx)
        check_cells(k.cpu().numpy(), ost.K[l][:, :ctx], f"context K l{l}")
        check_cells(v.cpu().numpy(), ost.V[l][:, :ctx], f"context V l{l}")
    anchor = int(synth.make_token_ids(cfg, 1, seed=31)[0])
    st.anchor_tok[0], st.anchor_pos[0], st.block_len[0] = anchor, ctx, B
    st.draft(1)
    res = O.draft_block(om, ost, anchor, ctx, B)
    _check_pass(st, ost, res, 0, ctx, B, "full bf16")
    assert st.take_status() == 0


@pytest.mark.parametrize("wtype", ["q8_0", "q5_0", "q4_0"])
def test_full_quantised(wtype):
    from dflash_block_drafter_gb300.runtime import DraftModel, DraftState
    cfg = synth.CONFIGS[f"full_{wtype}"]
    ck = synth.make_checkpoint(cfg, seed=0)
    om = O.Model(cfg, ck)
    model = DraftModel(cfg, ck)
    ctx, B = cfg.ctx, cfg.block
    st = DraftState(model, 1, ctx + B)
    ost = O.State(cfg, ctx + B)
    _prefill(st, ost, cfg, 0, ctx - 8, seed=32)
    _fuse(st, ost, om, cfg, 0, np.arange(ctx - 8, ctx), 32, 0)
    anchor = int(synth.make_token_ids(cfg, 1, seed=32)[0])
    st.anchor_tok[0], st.anchor_pos[0], st.block_len[0] = anchor, ctx, B
    st.draft(1)
    res = O.draft_block(om, ost, anchor, ctx, B)
    _check_pass(st, ost, res, 0, ctx, B, f"full {wtype}")
    for which, name in ((0, "fc"), (4, "layers.0.wo"), (35, "layers.4.w_down")):
        got = model.dequantize(which).cpu().numpy().astype(np.float64)
        assert np.array_equal(got, om.mat(name)), name
    assert st.take_status() == 0


def test_long_context_q8_0():
    from dflash_block_drafter_gb300.runtime import DraftModel, DraftState
    cfg = synth.CONFIGS["long_q8_0"]
    ck = synth.make_checkpoint(cfg, seed=0)
    om = O.Model(cfg, ck)
    model = DraftModel(cfg, ck)
    ctx, B = cfg.ctx, cfg.block
    st = DraftState(model, 1, ctx + B)
    ost = O.State(cfg, ctx + B)
    _prefill(st, ost, cfg, 0, ctx - 8, seed=33)
    _fuse(st, ost, om, cfg, 0, np.arange(ctx - 8, ctx), 33, 0)
    anchor = int(synth.make_token_ids(cfg, 1, seed=33)[0])
    st.anchor_tok[0], st.anchor_pos[0], st.block_len[0] = anchor, ctx, B
    st.draft(1)
    res = O.draft_block(om, ost, anchor, ctx, B)
    _check_pass(st, ost, res, 0, ctx, B, "long q8_0")
    assert st.take_status() == 0


def test_batched_mix_q4_0():
    from dflash_block_drafter_gb300.runtime import DraftModel, DraftState, accept
    cfg = synth.CONFIGS["batched_q4_0"]
    ck = synth.make_checkpoint(cfg, seed=0)
    om = O.Model(cfg, ck)
    model = DraftModel(cfg, ck)
    ctxs, Bs = synth.batched_mix(cfg, seed=34)
    cap = int(ctxs.max()) + 8
    st = DraftState(model, cfg.n_seq, cap)
    osts = []
    for s in range(cfg.n_seq):
        ost = O.State(cfg, cap)
        _prefill(st, ost, cfg, s, int(ctxs[s]) - 4, seed=34)
        _fuse(st, ost, om, cfg, s, np.arange(ctxs[s] - 4, ctxs[s]), 34, s)
        osts.append(ost)
    toks = synth.make_token_ids(cfg, cfg.n_seq, seed=34)
    st.anchor_tok[:] = device_ids(toks)
    st.anchor_pos[:] = device_ids(ctxs)
    st.block_len[:] = device_ids(Bs)
    st.draft(cfg.n_seq)
    res = [O.draft_block(om, osts[s], int(toks[s]), int(ctxs[s]), int(Bs[s])) for s in range(cfg.n_seq)]
    for s in range(cfg.n_seq):
        _check_pass(st, osts[s], res[s], s, int(ctxs[s]), int(Bs[s]), f"slot {s}")
    # acceptance against verifier ids that agree per token with probability 0.7,
    # fed the oracle's drafts so both sides see the same candidates
    tgt = np.zeros((cfg.n_seq, 8), np.int32)
    drafts = np.full((cfg.n_seq, 7), -1, np.int32)
    for s in range(cfg.n_seq):
        drafts[s, :Bs[s] - 1] = res[s].drafts
        tgt[s, :Bs[s]] = synth.make_target_ids(res[s].drafts, cfg.vocab, seed=34, stream=s)
    acc = torch.zeros(cfg.n_seq, dtype=torch.int32, device="cuda")
    nxt = torch.zeros(cfg.n_seq, dtype=torch.int32, device="cuda")
    accept(device_ids(drafts), device_ids(tgt), device_ids(Bs), acc, nxt)
    torch.cuda.synchronize()
    for s in range(cfg.n_seq):
        n, bonus = O.accept(drafts[s], tgt[s], int(Bs[s]))
        assert (int(acc[s]), int(nxt[s])) == (n, bonus)
    assert st.take_status() == 0

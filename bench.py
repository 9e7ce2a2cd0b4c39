"""Benchmark of the DFlash block-draft cycle on GB300.

One step = one pass of the whole hot path over one batch of synthetic input,
on the full DFlash geometry (5 layers, hidden 2560, 24Q/2KV x 256, MLP 7680,
vocab 151936) with an 8192-position context and an 8-row block:
  fuse the taps of 8 committed positions [p-8, p) into every layer's FP16
  K/V  ->  draft the block at p (5 layers + final norm + LM head + argmax)
  ->  greedy acceptance against synthetic verifier ids.
All of it runs in libdflash's CUDA kernels through the C ABI.  The anchor
position stays at p = 8192 so every step does identical work.

The cycle is captured once in a CUDA graph (the C ABI reads positions, block
lengths and ids from device memory, so a captured cycle stays valid) and the
timed region replays it.

Printed (rank 0): one JSON line with the metric, device-timed passes/s, the
end-to-end number through the C ABI with host buffers, the dominant kernel's
roofline, the CPU oracle timed on the host cores as a baseline, SM clocks
sampled during the timed region and the kernel-launch count.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
  (N > 1: launched by torch.distributed.run; every rank runs an independent
  replica on its own GPU -- the sequences are independent, there is no
  data-path collective.)
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import dflash_synth as synth  # noqa: E402

METRIC = "draft passes/s and drafted tok/s at 8K ctx, block 8; HBM GB/s vs roofline"
UNIT = "draft passes/s"
WORKLOAD = "full_bf16"
FUSE_PER_STEP = 8
# DRAM bytes (read + write) of one LM-head launch at this workload, from one
# ncu capture of that kernel (dram__bytes_read.sum 778135552 +
# dram__bytes_write.sum 3333888).  Reset to None whenever the head kernel
# changes.
HEAD_TRAFFIC_BYTES = 781469440
HEAD_TRAFFIC_SOURCE = ("ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum on one LM-head launch "
                       "(head_tc8_kernel) of `bench.py --steps 3 --warmup 3 --no-cpu-baseline --no-extras`, "
                       "library as of commit f3b1c08")


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def algorithmic_bytes(cfg, ctx: int, B: int, n_fuse: int) -> dict:
    """Bytes the cycle must move (each weight byte and each context K/V cell
    read once, outputs written once)."""
    H, d, nkv, L = cfg.hidden, cfg.head_dim, cfg.n_kv_heads, cfg.n_layers
    shapes = cfg.matrix_shapes()
    bpw = {"bf16": 2.0, "q8_0": 34 / 32, "q5_0": 22 / 32, "q4_0": 18 / 32}[cfg.weight_type]
    layer_params = sum(a * b for n, (a, b) in shapes.items() if n != "fc")
    kv_params = sum(a * b for n, (a, b) in shapes.items() if n.endswith((".wk", ".wv")))
    head = cfg.vocab * H * 2
    window = getattr(cfg, "attn_window", 0)
    attended = min(ctx + B, window) if window > 0 else ctx + B
    kv_read = L * 2 * nkv * attended * d * 2
    kv_write_block = L * 2 * nkv * B * d * 2
    draft = layer_params * bpw + head + kv_read + kv_write_block + B * H * 2
    fuse = (shapes["fc"][0] * shapes["fc"][1] + kv_params) * bpw + n_fuse * cfg.tap_width * 2 \
        + L * 2 * nkv * n_fuse * d * 2
    return {"draft": int(draft), "fuse": int(fuse), "head": int(head), "step": int(draft + fuse)}


def draft_bytes(cfg, ctx: int, B: int) -> int:
    """Algorithmic bytes of one draft pass of one sequence (weights, LM head,
    context K/V read, block K/V written, embedding rows)."""
    return algorithmic_bytes(cfg, ctx, B, 0)["draft"]


def cpu_model() -> str:
    """The host CPU's name as the kernel reports it (x86 'model name', or the
    Arm implementer / part codes)."""
    try:
        with open("/proc/cpuinfo") as f:
            info = f.read()
    except OSError:
        return "unknown"
    for key in ("model name", "Model", "Hardware"):
        for line in info.splitlines():
            if line.startswith(key) and ":" in line:
                return line.split(":", 1)[1].strip()
    fields = {}
    for line in info.splitlines():
        if ":" in line:
            k, v = line.split(":", 1)
            fields.setdefault(k.strip(), v.strip())
    if "CPU implementer" in fields:
        return f"Arm implementer {fields['CPU implementer']} part {fields.get('CPU part', '?')}"
    return "unknown"


def replay_stats(event_pairs, per_replay: int) -> dict:
    """Median / min / max per step from (start, end) CUDA-event pairs around
    graph replays of `per_replay` steps each."""
    ms = sorted(a.elapsed_time(b) / per_replay for a, b in event_pairs)
    return {"median_ms": statistics.median(ms), "min_ms": ms[0], "max_ms": ms[-1], "replays": len(ms),
            "steps_per_replay": per_replay}


class ClockSampler:
    """nvidia-smi clock / throttle-reason sampling during the timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------------------
# replicas: timing reduction over ranks
# --------------------------------------------------------------------------
def max_over_ranks(values, device=None):
    """Element-wise maximum of this rank's timings over all ranks.  Every
    rank runs an independent replica (sequences are independent and the
    weights are replicated), so this timing reduction is the only collective;
    none touches the data path."""
    import torch
    import torch.distributed as dist
    t = torch.tensor(values, dtype=torch.float64, device=device)
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t]


def replica_throughput(world: int, steps: int, elapsed_ms: float) -> float:
    """Whole-job cycles/s: every rank ran `steps` cycles; the job took the
    slowest rank's time."""
    return world * steps / (elapsed_ms / 1000.0)


# --------------------------------------------------------------------------
# CPU oracle baseline (also the reference arm)
# --------------------------------------------------------------------------
def oracle_baseline(ckpt, cfg, budget_s: float = 12.0, max_steps: int = 1000):
    """The CPU oracle, as it stands, timed on this host's cores over a bounded
    sample of the same cycle (fuse 8 positions + draft + accept) at the same
    shapes.  Its 8192-position context is pre-filled with seeded FP16 values
    (fusing 8192 positions in float64 is not part of the timed cycle)."""
    from oracle import dflash_oracle as O
    cores = len(os.sched_getaffinity(0))
    ctx, B = cfg.ctx, cfg.block
    om = O.Model(cfg, ckpt)
    st = O.State(cfg, ctx + B)
    st.fill(synth.make_kv_fill(cfg, ctx, seed=1), ctx)
    taps = synth.make_taps(cfg, FUSE_PER_STEP, seed=2)
    fpos = np.arange(ctx - FUSE_PER_STEP, ctx)
    anchor = int(synth.make_token_ids(cfg, 1, seed=3)[0])
    tgt = synth.make_target_ids(np.zeros(B - 1, np.int32), cfg.vocab, seed=4, p_agree=0.0)

    def step():
        O.fuse_context(om, st, taps, fpos)
        r = O.draft_block(om, st, anchor, ctx, B)
        O.accept(r.drafts, tgt, B)

    t0 = time.perf_counter()
    step()  # first call decodes the weights to float64 (a one-time load)
    load_s = time.perf_counter() - t0
    n, t0 = 0, time.perf_counter()
    while n < max_steps:
        step()
        n += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return {"value": n / dt, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{n} oracle cycles (fuse 8 + draft + accept) at the full shape after one warm-up cycle "
                      f"({load_s:.1f} s incl. weight decode); context K/V pre-filled",
            "seconds": dt}


def oracle_one_thread(budget_s: float = 10.0) -> dict:
    """The same oracle cycle with every BLAS / OpenMP pool limited to one
    thread, in a child process (the pools size themselves at import)."""
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
        env[k] = "1"
    code = ("import json, sys; sys.path.insert(0, %r); import bench, dflash_synth as synth; "
            "cfg = synth.CONFIGS[bench.WORKLOAD]; ck = synth.make_checkpoint(cfg, seed=0, threads=1); "
            "r = bench.oracle_baseline(ck, cfg, budget_s=%r, max_steps=1000); r['cores'] = 1; "
            "print(json.dumps(r))") % (ROOT, budget_s)
    try:
        out = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                             timeout=budget_s * 6 + 120)
        return json.loads(out.stdout.strip().splitlines()[-1])
    except Exception as e:  # reported, never fatal
        return {"error": str(e)[:200]}


def run_reference(args, rank: int):
    if rank != 0:
        return
    cfg = synth.CONFIGS[WORKLOAD]
    ckpt = synth.make_checkpoint(cfg, seed=0)
    budget = max(5.0, min(120.0, 0.5 * (args.steps + args.warmup)))
    base = oracle_baseline(ckpt, cfg, budget_s=budget, max_steps=args.steps + args.warmup)
    v = base["value"]
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 / v if v else None,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_block(cfg),
            "drafted_tok_per_s": v * (cfg.block - 1),
            "cpu_baseline": {"value": v, "unit": UNIT, "cores": base["cores"], "kind": "oracle",
                             "sample": base["sample"]},
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def config_block(cfg):
    window = getattr(cfg, "attn_window", 0)
    win = (f", attention window {window} over a ring of {state_capacity(cfg)} cells" if window > 0 else "")
    block = {"workload": f"DFlash draft cycle: fuse 8 committed positions + draft an 8-row block at p = {cfg.ctx} "
                         "+ greedy accept; 5 layers, hidden 2560, 24Q/2KV x 256, MLP 7680, vocab 151936, "
                         f"{cfg.weight_type.upper()} backbone{win}",
             "ctx": cfg.ctx, "block": cfg.block, "fuse_per_step": FUSE_PER_STEP, "weight_type": cfg.weight_type,
             "sequences_per_gpu": 1,
             "l2": "inputs larger than L2: every step streams over 1 GB of weights and K/V (L2 is 129 MB)"}
    if window > 0:
        block["attn_window"] = window
    return block


def workload_config(args):
    cfg = synth.CONFIGS[WORKLOAD]
    if args.weight_type:
        cfg = cfg.with_(weight_type=args.weight_type)
    if args.ctx:
        cfg = cfg.with_(ctx=args.ctx)
    if args.window:
        cfg = cfg.with_(attn_window=args.window)
    return cfg


def state_capacity(cfg) -> int:
    """Cells of the bench's state: the context and one block, or with an
    attention window a ring of the window rounded up to 128 cells."""
    window = getattr(cfg, "attn_window", 0)
    if window > 0:
        return (window + 127) // 128 * 128
    return cfg.ctx + cfg.block


# --------------------------------------------------------------------------
# GPU arm
# --------------------------------------------------------------------------
def _fill_context_random(st, cfg, slot, n, dev, seed):
    """Seeded N(0, 1) FP16 K/V for positions [0, n) of one slot (the draft
    pass's work does not depend on the values)."""
    import torch
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    for l in range(cfg.n_layers):
        k = torch.randn(cfg.n_kv_heads, n, cfg.head_dim, device=dev, generator=g).half()
        v = torch.randn(cfg.n_kv_heads, n, cfg.head_dim, device=dev, generator=g).half()
        st.write_kv(slot, l, 0, k, v)


def _time_graph(fn, stream, G: int, n_rep: int) -> dict:
    """Capture G calls of fn in one CUDA graph and time n_rep replays with an
    event pair around each (median / min / max per call)."""
    import torch
    with torch.cuda.stream(stream):
        for _ in range(3):
            fn()
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for _ in range(G):
            fn()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_rep)]
    with torch.cuda.stream(stream):
        graph.replay()
        for a, b in ev:
            a.record(stream)
            graph.replay()
            b.record(stream)
    stream.synchronize()
    r = replay_stats(ev, G)
    r["mean_ms"] = ev[0][0].elapsed_time(ev[-1][1]) / (G * n_rep)
    return r


def time_weight_type(wt: str, dev, peak: float, n_rep: int = 20, cfg_name: str = "full_bf16") -> dict:
    """Device-timed draft pass and draft cycle of the full geometry (the
    8192-position context, or the workload cfg_name names) with the given
    backbone type (graph replays)."""
    import torch
    from dflash_block_drafter_gb300.runtime import DraftModel, DraftState, accept
    cfg = synth.CONFIGS[cfg_name].with_(weight_type=wt)
    ctx, B = cfg.ctx, cfg.block
    ck = synth.make_checkpoint(cfg, seed=0)
    model = DraftModel(cfg, ck, device=dev)
    del ck
    st = DraftState(model, 1, ctx + B)
    _fill_context_random(st, cfg, 0, ctx, dev, seed=1)
    st.set_defer_kv(True)  # the committed rows' K/V ride in the next pass's QKV GEMVs
    st.anchor_tok[0], st.anchor_pos[0], st.block_len[0] = 17, ctx, B
    taps = torch.as_tensor(synth.make_taps(cfg, FUSE_PER_STEP, seed=2).view(np.int16), device=dev)
    fpos = torch.arange(ctx - FUSE_PER_STEP, ctx, dtype=torch.int32, device=dev)
    tgt = torch.zeros((1, B), dtype=torch.int32, device=dev)
    acc = torch.zeros(1, dtype=torch.int32, device=dev)
    nxt = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(dev)

    def draft():
        st.draft(1, want_hidden=False, stream=stream)

    def cycle():
        st.fuse(0, taps, fpos, stream=stream)
        draft()
        accept(st.drafts, tgt, st.block_len, acc, nxt, stream=stream)

    d = _time_graph(draft, stream, 10, n_rep)
    c = _time_graph(cycle, stream, 10, n_rep)
    status = st.take_status()
    ab = algorithmic_bytes(cfg, ctx, B, FUSE_PER_STEP)
    gbs = ab["draft"] / (d["median_ms"] * 1e-3) / 1e9
    out = {"draft_passes_per_s": 1e3 / d["median_ms"], "draft_us": d["median_ms"] * 1e3,
           "draft_us_min_max": [d["min_ms"] * 1e3, d["max_ms"] * 1e3],
           "drafted_tok_per_s": (B - 1) * 1e3 / d["median_ms"],
           "draft_bytes": ab["draft"], "achieved_gbs": gbs, "frac": gbs / peak,
           "cycles_per_s": 1e3 / c["median_ms"], "cycle_us": c["median_ms"] * 1e3,
           "cycle_frac": ab["step"] / (c["median_ms"] * 1e-3) / 1e9 / peak, "device_status": status,
           "timing": f"median of {n_rep} CUDA-graph replays of 10 calls"}
    st.close()
    model.close()
    del st, model
    torch.cuda.empty_cache()
    return out


def time_batched_mix(dev, peak: float, n_rep: int = 10) -> dict:
    """The batched serving mix: 16 sequences, Q4_0 backbone, contexts
    U[2048, 32768], blocks U{2..8} (seeded), one dflash_draft_block call per
    step over all 16 slots."""
    import torch
    from dflash_block_drafter_gb300.runtime import DraftModel, DraftState
    cfg = synth.CONFIGS["batched_q4_0"]
    ctxs, Bs = synth.batched_mix(cfg, seed=34)
    ck = synth.make_checkpoint(cfg, seed=0)
    model = DraftModel(cfg, ck, device=dev)
    del ck
    cap = int(ctxs.max()) + 8
    st = DraftState(model, cfg.n_seq, cap)
    for s in range(cfg.n_seq):
        _fill_context_random(st, cfg, s, int(ctxs[s]), dev, seed=100 + s)
    st.anchor_tok[:] = torch.as_tensor(synth.make_token_ids(cfg, cfg.n_seq, seed=34), device=dev)
    st.anchor_pos[:] = torch.as_tensor(ctxs, device=dev)
    st.block_len[:] = torch.as_tensor(Bs, device=dev)
    stream = torch.cuda.Stream(dev)
    d = _time_graph(lambda: st.draft(cfg.n_seq, want_hidden=False, stream=stream), stream, 5, n_rep)
    status = st.take_status()
    one = algorithmic_bytes(cfg, 0, 0, 0)  # weights and head once per pass
    kv = sum(cfg.n_layers * 2 * cfg.n_kv_heads * (int(c) + int(b)) * cfg.head_dim * 2 for c, b in zip(ctxs, Bs))
    byts = one["draft"] + kv
    gbs = byts / (d["median_ms"] * 1e-3) / 1e9
    out = {"workload": "16 sequences, Q4_0 backbone, contexts U[2048, 32768], blocks U{2..8} (seed 34), "
                       "context K/V pre-filled", "pass_us": d["median_ms"] * 1e3,
           "sequence_passes_per_s": cfg.n_seq * 1e3 / d["median_ms"],
           "drafted_tok_per_s": float(np.sum(Bs - 1)) * 1e3 / d["median_ms"],
           "bytes_per_pass": int(byts), "achieved_gbs": gbs, "frac": gbs / peak, "device_status": status,
           "timing": f"median of {n_rep} CUDA-graph replays of 5 passes"}
    st.close()
    model.close()
    del st, model
    torch.cuda.empty_cache()
    return out

def run_gpu(args, rank: int, world: int, local_rank: int):
    import torch
    import torch.distributed as dist

    import dflash_block_drafter_gb300 as D
    from dflash_block_drafter_gb300.runtime import DraftModel, DraftState, accept

    D.load_library()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    cfg = workload_config(args)
    ctx, B = cfg.ctx, cfg.block
    t_setup = time.perf_counter()
    ckpt = synth.make_checkpoint(cfg, seed=0)
    model = DraftModel(cfg, ckpt, device=dev)
    st = DraftState(model, n_slots=1, capacity=state_capacity(cfg))
    # build the context by fusion (128-position tiles); long contexts reuse one
    # block of taps (its values do not change the work)
    shared = None
    for base in range(0, ctx, 1024):
        n = min(1024, ctx - base)
        if ctx <= 16384:
            taps = torch.as_tensor(synth.make_taps(cfg, n, seed=5, stream=base).view(np.int16), device=dev)
        else:
            if shared is None:
                shared = torch.as_tensor(synth.make_taps(cfg, 1024, seed=5).view(np.int16), device=dev)
            taps = shared[:n]
        st.fuse(0, taps, torch.arange(base, base + n, dtype=torch.int32, device=dev))
    torch.cuda.synchronize(dev)
    setup_s = time.perf_counter() - t_setup

    fuse_taps = torch.as_tensor(synth.make_taps(cfg, FUSE_PER_STEP, seed=2).view(np.int16), device=dev)
    fuse_pos = torch.arange(ctx - FUSE_PER_STEP, ctx, dtype=torch.int32, device=dev)
    # each cycle's 8 committed rows: the fc projection in the fusion call, their
    # K/V inside the next draft pass's QKV GEMVs (dflash_state_set_defer_kv)
    st.set_defer_kv(not args.no_defer_kv)
    anchor = int(synth.make_token_ids(cfg, 1, seed=3)[0])
    st.anchor_tok[0], st.anchor_pos[0], st.block_len[0] = anchor, ctx, B
    tgt_np = synth.make_target_ids(np.zeros(B - 1, np.int32), cfg.vocab, seed=4, p_agree=0.0)[None]
    tgt = torch.as_tensor(tgt_np, device=dev)
    acc_len = torch.zeros(1, dtype=torch.int32, device=dev)
    next_anchor = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(dev)

    def step():
        st.fuse(0, fuse_taps, fuse_pos, stream=stream)
        st.draft(1, want_hidden=False, stream=stream)
        accept(st.drafts, tgt, st.block_len, acc_len, next_anchor, stream=stream)

    launches = D.dflash_fuse_launches(st.handle, FUSE_PER_STEP) + D.dflash_draft_launches(st.handle, 1) + 1

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
    stream.synchronize()
    status = st.take_status()
    if status:
        raise RuntimeError(f"device status {status} during warm-up")

    # ---- the cycle as a CUDA graph: G cycles per graph, each with its own
    # pair of events around the LM-head launch (event-record nodes), so the
    # head's duration is read from the last replay inside the timed region
    G = 10 if args.steps % 10 == 0 else 1
    head_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(G)]
    with torch.cuda.stream(stream):
        for a, b in head_ev:  # CUDA events are created lazily on first record
            a.record(stream)
            b.record(stream)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(G):
            D.dflash_state_set_head_events(st.handle, head_ev[i][0].cuda_event, head_ev[i][1].cuda_event)
            step()
    D.dflash_state_set_head_events(st.handle, 0, 0)
    with torch.cuda.stream(stream):
        graph.replay()
    stream.synchronize()
    t_beg = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    n_rep = args.steps // G
    rep_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_rep)]
    with ClockSampler(local_rank) as clocks:
        time.sleep(0.15)
        with torch.cuda.stream(stream):
            t_beg.record(stream)
            for a, b in rep_ev:
                a.record(stream)
                graph.replay()
                b.record(stream)
            t_end.record(stream)
        torch.cuda.synchronize(dev)
        time.sleep(0.15)
    if world > 1:
        dist.barrier()
    elapsed_ms = t_beg.elapsed_time(t_end)
    head_ms = [a.elapsed_time(b) for a, b in head_ev]
    status = st.take_status()
    if status:
        raise RuntimeError(f"device status {status} during the timed region")

    # ---- draft-only device timing (context for the reader), also as a graph
    dgraph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(dgraph, stream=stream):
        st.draft(1, want_hidden=False, stream=stream)
    with torch.cuda.stream(stream):
        n_draft = max(20, args.steps // 4)
        dgraph.replay()
        d_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_draft)]
        for a, b in d_ev:
            a.record(stream)
            dgraph.replay()
            b.record(stream)
    torch.cuda.synchronize(dev)
    draft_stats = replay_stats(d_ev, 1)
    draft_only_ms = d_ev[0][0].elapsed_time(d_ev[-1][1]) / n_draft
    # ---- end to end through the C ABI with host buffers: every step copies
    # its inputs (the fusion taps and positions, the anchor token / position /
    # block length, the verifier's targets) from one pinned host buffer in one
    # transfer, replays the cycle -- whose graph starts by unpacking that
    # staging buffer into the library's inputs and ends by gathering the
    # results -- and reads the results (7 drafts, accepted count, next
    # anchor) back in one transfer, then waits for them
    parts = [fuse_taps.view(torch.uint8).reshape(-1), fuse_pos.view(torch.uint8).reshape(-1),
             torch.tensor([anchor, ctx, B], dtype=torch.int32).view(torch.uint8), tgt.view(torch.uint8).reshape(-1)]
    offs = [0]
    for t_ in parts:
        offs.append(offs[-1] + ((t_.numel() + 15) // 16) * 16)
    h_stage = torch.zeros(offs[-1], dtype=torch.uint8).pin_memory()
    for t_, o_ in zip(parts, offs):
        h_stage[o_:o_ + t_.numel()].copy_(t_.cpu())
    d_stage = torch.zeros(offs[-1], dtype=torch.uint8, device=dev)
    d_out = torch.zeros(7 + 2, dtype=torch.int32, device=dev)
    h_out = torch.zeros(7 + 2, dtype=torch.int32).pin_memory()
    scal = d_stage[offs[2]:offs[2] + 12].view(torch.int32)

    def e2e_step():
        fuse_taps.view(torch.uint8).reshape(-1).copy_(d_stage[offs[0]:offs[0] + parts[0].numel()])
        fuse_pos.view(torch.uint8).reshape(-1).copy_(d_stage[offs[1]:offs[1] + parts[1].numel()])
        st.anchor_tok[:1].copy_(scal[0:1])
        st.anchor_pos[:1].copy_(scal[1:2])
        st.block_len[:1].copy_(scal[2:3])
        tgt.view(torch.uint8).reshape(-1).copy_(d_stage[offs[3]:offs[3] + parts[3].numel()])
        step()
        d_out[:7].copy_(st.drafts[0])
        d_out[7:8].copy_(acc_len)
        d_out[8:9].copy_(next_anchor)

    one = torch.cuda.CUDAGraph()
    with torch.cuda.graph(one, stream=stream):
        e2e_step()
    n_e2e = max(20, min(args.steps, 500))
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for _ in range(n_e2e):
            d_stage.copy_(h_stage, non_blocking=True)
            one.replay()
            h_out.copy_(d_out, non_blocking=True)
            stream.synchronize()
    e2e_s = time.perf_counter() - t0
    h2d = offs[-1]
    d2h = h_out.numel() * 4

    # ---- gather over ranks (max time), replicas only
    elapsed_ms, e2e_s = max_over_ranks([elapsed_ms, e2e_s], device=dev)
    if rank != 0:
        return
    ms_per_step = elapsed_ms / args.steps
    value = replica_throughput(world, args.steps, elapsed_ms)
    ab = algorithmic_bytes(cfg, ctx, B, FUSE_PER_STEP)
    peak, peak_kind = load_peaks()
    head_avg_ms = statistics.mean(head_ms)
    head_gbs = ab["head"] / (head_avg_ms * 1e-3) / 1e9
    step_gbs = ab["step"] / (ms_per_step * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": cfg.weight_type, "data": "synthetic (seeded; random-init weights of the "
        "DFlash geometry, N(0,1) taps)",
        "config": dict(config_block(cfg), committed_kv=("separate launch in the fusion call" if args.no_defer_kv else
                                                         "projected inside the next draft pass's QKV GEMVs")),
        "drafted_tok_per_s": value * (B - 1),
        "draft_passes_per_s": 1e3 / draft_stats["median_ms"],
        "draft_only_ms": draft_only_ms,
        "draft_stats": draft_stats,
        "step_stats": replay_stats(rep_ev, G),
        "achieved_gbs_step": step_gbs,
        "algorithmic_bytes_per_step": ab["step"],
        "roofline": {"bound": "hbm", "kernel": "lm_head_argmax (head_tc8_kernel, tcgen05)",
                     "achieved": head_gbs, "peak": peak, "unit": "GB/s", "frac": head_gbs / peak,
                     "peak_kind": peak_kind, "traffic": HEAD_TRAFFIC_BYTES, "traffic_source": HEAD_TRAFFIC_SOURCE,
                     "bytes_per_launch": ab["head"], "avg_launch_ms": head_avg_ms},
        "step_roofline": {"achieved": step_gbs, "peak": peak, "frac": step_gbs / peak, "unit": "GB/s"},
        "e2e": {"value": replica_throughput(world, n_e2e, e2e_s * 1000.0), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": n_e2e},
        "gpu_launches": launches * args.steps,
        "cuda_graph": f"{G} cycles per graph, replayed {args.steps // G} times",
        "launches_per_step": launches,
        "clocks": clocks.summary(),
        "setup_s": setup_s,
    }
    if not args.no_extras:
        draft_ab = algorithmic_bytes(cfg, ctx, B, FUSE_PER_STEP)
        per = {cfg.weight_type: {
            "draft_passes_per_s": 1e3 / draft_stats["median_ms"], "draft_us": draft_stats["median_ms"] * 1e3,
            "draft_us_min_max": [draft_stats["min_ms"] * 1e3, draft_stats["max_ms"] * 1e3],
            "drafted_tok_per_s": (B - 1) * 1e3 / draft_stats["median_ms"], "draft_bytes": draft_ab["draft"],
            "achieved_gbs": draft_ab["draft"] / (draft_stats["median_ms"] * 1e-3) / 1e9,
            "frac": draft_ab["draft"] / (draft_stats["median_ms"] * 1e-3) / 1e9 / peak,
            "cycles_per_s": value, "cycle_us": ms_per_step * 1e3, "cycle_frac": step_gbs / peak,
            "timing": "the headline run above"}}
        del graph, dgraph, one
        st.close()
        model.close()
        torch.cuda.empty_cache()
        if cfg.ctx == 8192 and getattr(cfg, "attn_window", 0) == 0:
            for wt in ("q8_0", "q5_0", "q4_0"):
                if wt != cfg.weight_type:
                    per[wt] = time_weight_type(wt, dev, peak)
        line["per_weight_type"] = per
        line["batched_mix"] = time_batched_mix(dev, peak)
        lc = time_weight_type("q8_0", dev, peak, n_rep=10, cfg_name="long_q8_0")
        lc["workload"] = ("long context: 262144 positions of pre-filled K/V (2.7 GB), Q8_0 backbone, "
                          "block 8, fuse 8 per cycle")
        line["long_context"] = lc
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = {k: v for k, v in oracle_baseline(ckpt, cfg).items() if k != "seconds"}
        line["cpu_baseline"]["cpu_model"] = cpu_model()
        one_t = oracle_one_thread()
        line["cpu_baseline"]["one_thread"] = {k: v for k, v in one_t.items() if k in ("value", "unit", "cores",
                                                                                     "sample", "error")}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--weight-type", default=None, choices=[None, "bf16", "q8_0", "q5_0", "q4_0"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extras", action="store_true",
                    help="skip the per-weight-type and batched-mix timings that follow the headline run")
    ap.add_argument("--no-defer-kv", action="store_true",
                    help="project each cycle's committed rows' K/V in a separate launch of the fusion call")
    ap.add_argument("--batched-mix-only", action="store_true",
                    help="time only the 16-sequence batched mix and print its figures as one JSON line")
    ap.add_argument("--ctx", type=int, default=0, help="anchor position p (default: the workload's 8192)")
    ap.add_argument("--window", type=int, default=0, help="drafter attention window over a ring of cells (0: none)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank)
        return
    if args.batched_mix_only:
        import torch
        import dflash_block_drafter_gb300 as D
        D.load_library()
        dev = torch.device("cuda", local_rank)
        torch.cuda.set_device(dev)
        print(json.dumps({"batched_mix": time_batched_mix(dev, load_peaks()[0])}), flush=True)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    try:
        run_gpu(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()

#!/usr/bin/env python
"""Benchmark of the EAGLE-3 drafter draft round on GB300.

One step = one speculative round of the whole hot path over one batch: a gamma-step
draft chain (embed, norms, q/k/v + RoPE + KV append, split-KV attention, o_proj,
SwiGLU MLP, lm_head + argmax + d2t), rewind, the greedy accept walk against synthetic
target predictions, and rebuild_after_verify (fc encode of the verify features + k/v
teacher forcing + new boundary).  Metric: draft tokens/s (B * gamma per round) and
microseconds per draft step, plus the HBM roofline fraction.

  python bench.py [--gpus N --steps K --warmup W] [--config c2] [--impl reference]

Under torchrun every rank runs an independent replica on its own GPU (the drafter's
sequences are independent: no collective on the data path; weak scaling); rank 0 prints
one JSON line with the whole-job throughput.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "draft tokens/sec & µs/draft step at 1×GB300; % of HBM roofline per step"

CONFIGS = {
    "c1": dict(workload="tiny drafter n_embd 256, B=1, prompt 32, gamma 3", geom="tiny", B=1,
               prompt=(32, 32), gamma=3, p_accept=0.6, page_size=16),
    "c2": dict(workload="drafter n_embd 4096 (fc 4096x12288, q 4096x8192, k/v 1024x8192, "
                        "o 4096x4096, ff 12288, 16:4 GQA d256, RoPE 64/256, V_d 32000 -> V_t 248320) "
                        "bf16, B=1, prompt 512, gamma 3",
               geom="full", B=1, prompt=(512, 512), gamma=3, p_accept=0.6, page_size=64),
    "c3": dict(workload="drafter n_embd 4096 bf16, B=8 ragged prompts U[512, 8192], gamma 5, "
                        "accept length uniform 0..gamma",
               geom="full", B=8, prompt=(512, 8192), gamma=5, p_accept=None, page_size=64),
    "c4": dict(workload="drafter n_embd 4096 bf16, B=64, context 2048, gamma 3, "
                        "per-token accept probability 0.6",
               geom="full", B=64, prompt=(2048, 2048), gamma=3, p_accept=0.6, page_size=64),
    "c5": dict(workload="drafter n_embd 4096 bf16, B=4, context 32768, gamma 7, paged KV "
                        "(page 64)",
               geom="full", B=4, prompt=(32768, 32768), gamma=7, p_accept=0.6, page_size=64),
}


# DRAM traffic (ncu dram__bytes_read.sum + dram__bytes_write.sum, bytes per launch) of the
# kernels profiled on these workloads, valid only while the kernel's sources are byte for
# byte the profiled ones (sha256 over the listed csrc files); the summaries under
# profiles/ give the commands.  Keyed by (config, dominant projection or "attn").
PROFILED_TRAFFIC = {
    ('c2', 'lmhead'): {"bytes": 262222080 + 2776064,
                      "sources": ('gemv.cu', 'gemv_kernel.cuh', 'epilogue.cuh', 'common.cuh'),
                      "sha256": "83f4692564160a301bfc11f44cc6e27fce044bc69a5d134f643af10fc0533de1"},
    ('c4', 'attn'): {"bytes": 539141376 + 3132160,
                    "sources": ('attention.cu', 'attn_sched.cuh', 'common.cuh'),
                    "sha256": "f1c15ad2a3315885ac9c99241d4de4ae3d67abc8c143441bff022c8afb18017e"},
    ('c4', 'lmhead'): {"bytes": 265026560 + 5626880,
                      "sources": ('gemm_tc.cuh', 'gemm_tc.cu', 'epilogue.cuh', 'common.cuh'),
                      "sha256": "9a91526e826f19bab67fb100a50526ab97a65ddf8646787cb860a78f4feeb383"},
    ('c5', 'attn', 'q8_0/q5_1'): {"bytes": 243893760 + 2939904,
                                 "sources": ('attention.cu', 'attn_sched.cuh', 'common.cuh'),
                                 "sha256": "f1c15ad2a3315885ac9c99241d4de4ae3d67abc8c143441bff022c8afb18017e"},
}


def profiled_traffic(config: str, kind: str, kv_format: str = "bf16", weights: str = "bf16"):
    import hashlib
    if weights != "bf16":
        key = (config, kind, kv_format, weights)
    else:
        key = (config, kind) if kv_format == "bf16" else (config, kind, kv_format)
    e = PROFILED_TRAFFIC.get(key)
    if e is None:
        return None
    csrc = os.path.join(os.path.dirname(os.path.abspath(__file__)), "eagle_speculative_decode_gb300", "csrc")
    h = hashlib.sha256()
    for f in e["sources"]:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return e["bytes"] if h.hexdigest() == e["sha256"] else None


def kernel_label(kind: str, batch: int, weights: str = "bf16") -> str:
    """Name of the kernel that runs a phase at this batch on the bench's drafter geometry
    (projections of three or more items run on the tcgen05 GEMM -- INT4 codes decoded into
    tensor memory -- smaller ones on the CUDA-core GEMV; single-item INT4 projections with
    K <= 8192 on the mma.sync tensor-core GEMV)."""
    if kind == "attn":
        return "attention"
    if weights == "int4":
        if batch >= 3:
            return f"{kind} INT4 tcgen05 GEMM"
        return f"{kind} INT4 mma.sync GEMV" if batch == 1 and kind != "down" else f"{kind} INT4 GEMV"
    return f"{kind} tcgen05 GEMM" if batch >= 3 else f"{kind} GEMV"


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


# ------------------------------------------------------------------ clocks sampler
class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.samples = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for s in self.samples:
            f = [x.strip() for x in s.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for name, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": float(max(smax)) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ algorithmic bytes
def kv_bytes_per_position(geo, kv_format):
    """Bytes of the K and V rows of one position, all kv heads: 2 x 2 bytes per value for
    bf16; 34 + 24 bytes per 32 values for q8_0 keys and q5_1 values."""
    if kv_format == "bf16":
        return 2 * geo.kv_rows * 2
    return geo.kv_rows // 32 * (34 + 24)


def matrix_bytes(rows, K, weights="bf16"):
    """Bytes of a [rows, K] projection: bf16, or INT4 codes plus the (scale, zero) rows
    (one bf16 pair per 128 inputs, rows padded to a multiple of 4 pairs)."""
    if weights == "bf16":
        return rows * K * 2
    return rows * (K // 2 + ((K // 128 + 3) // 4 * 4) * 4)


def phase_bytes(geo, B, ctx_len, kv_format="bf16", weights="bf16"):
    """Bytes each kernel of one draft step must move (weights once per step for all B
    sequences, plus per-sequence activations and KV)."""
    n, F, qr, kr = geo.n_embd, geo.n_ff, geo.q_rows, geo.kv_rows
    act = 4 * B
    kvp = kv_bytes_per_position(geo, kv_format)
    mb = lambda rows, K: matrix_bytes(rows, K, weights)  # noqa: E731
    return {
        "qkv": mb(qr + 2 * kr, 2 * n) + B * (2 * n + 4 * n) + 3 * n * 2 + B * kvp + act * qr,
        "attn": B * (ctx_len * kvp + 2 * qr * 4),
        "o": mb(n, qr) + act * (qr + 2 * n),
        "gateup": mb(2 * F, n) + act * (n + F) + n * 2,
        "down": mb(n, F) + act * (F + 2 * n),
        "lmhead": mb(geo.draft_vocab, n) + act * n + n * 2 + B * 8,
    }


def round_bytes(geo, B, gamma, ctx_len, kv_format="bf16", weights="bf16"):
    ph = phase_bytes(geo, B, ctx_len, kv_format, weights)
    chain = gamma * sum(ph.values())
    rebuild = 3 * geo.n_embd * geo.n_embd * 2 + matrix_bytes(2 * geo.kv_rows, 2 * geo.n_embd, weights) \
        + B * (gamma + 1) * (3 * geo.n_embd * 2 + geo.n_embd * 4)
    return chain + rebuild


NOMINAL_HBM_GBS = 8000.0  # HBM3e bandwidth of the part's datasheet (≈8 TB/s)


def static_config(args, cfg, world=1):
    """The `config` object both arms print: the workload and the storage formats."""
    lo, hi = cfg["prompt"]
    return {"workload": cfg["workload"], "name": args.config, "batch": cfg["B"], "gamma": cfg["gamma"],
            "prompt": [lo, hi], "page_size": cfg["page_size"],
            "kv_format": args.kv_format, "weights": args.weights,
            "storage": ("bf16 weights" if args.weights == "bf16" else
                        "INT4 projections (128-wide groups, bf16 scale and zero), bf16 fc / norms / embedding")
                       + (", bf16 KV" if args.kv_format == "bf16" else ", q8_0 K / q5_1 V cache")
                       + ", float32 activations and accumulation",
            "l2": "inputs larger than L2: 0.8 GB of weights streamed per draft step",
            "step": "chain of gamma draft steps + rewind + accept + rebuild (encode of "
                    "gamma+1 verify features, k/v teacher forcing)",
            "parallelism": f"replicas x{world}"}


def make_bench_weights(geo, weights):
    from eagle_speculative_decode_gb300 import synth
    return synth.make_int4_weights(geo, seed=0) if weights == "int4" else synth.make_weights(geo, seed=0)


# ------------------------------------------------------------------ oracle timing
def oracle_round_rate(geo_name, gamma, rounds, seed=0, kv_format="bf16", weights="bf16",
                      prompt=32, seconds=0.0):
    """Times the CPU oracle on one sequence: chains of gamma draft steps from a prefilled
    state of `prompt` tokens at the benchmark's geometry, at least `rounds` chains and
    until `seconds` have passed (a bounded sample of the workload).  Returns (draft tok/s,
    seconds, sample description)."""
    from eagle_speculative_decode_gb300 import synth
    from oracle import eagle3_oracle as O
    geo = synth.GEOMETRIES[geo_name]
    wts = make_bench_weights(geo, weights)
    dr = O.Drafter(geo, wts.bits, wts.d2t, kv_format=kv_format, int4=wts.int4)
    P = int(prompt)
    toks = synth.make_tokens((P + 1,), geo, seed + 1)
    aux = synth.make_aux((P,), geo, seed + 1)
    st = O.prefill(dr, toks[:P], int(toks[P]), aux)
    t0 = time.perf_counter()
    n = 0
    while n < max(1, rounds) or (time.perf_counter() - t0 < seconds and n < 10000):
        O.draft_chain(dr, st, gamma)
        n += 1
    dt = time.perf_counter() - t0
    desc = (f"{n} chain(s) of {gamma} draft steps of one sequence from a {P}-token prefilled "
            f"state (prefill not timed), {geo_name} geometry, {weights} weights, {kv_format} KV, "
            "float64 numpy oracle")
    return n * gamma / dt, dt, desc


# ------------------------------------------------------------------ distributed
def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def _all_reduce(x: float, op) -> float:
    """All-reduce of one float over the ranks: on the GPU with NCCL, on the host with gloo
    (the CPU tests of the replica bookkeeping)."""
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=op)
    return float(t.item())


def max_over_ranks(world, x: float) -> float:
    if world <= 1:
        return x
    import torch.distributed as dist
    return _all_reduce(x, dist.ReduceOp.MAX)


def sum_over_ranks(world, x: float) -> float:
    if world <= 1:
        return x
    import torch.distributed as dist
    return _all_reduce(x, dist.ReduceOp.SUM)


def replica_throughput(world, tokens_local: float, elapsed_ms_local: float):
    """Whole-job throughput of N independent replicas (weak scaling): the tokens of every
    rank over the slowest rank's time.  Returns (tokens/s, max elapsed ms)."""
    elapsed = max_over_ranks(world, elapsed_ms_local)
    tokens = sum_over_ranks(world, tokens_local)
    return tokens / (elapsed / 1e3), elapsed


# ------------------------------------------------------------------ reference arm
def run_reference(args, cfg):
    """The reference arm is the float64 CPU oracle, timed as it stands on the host cores on
    the unit `cpu_baseline` times: one step = one chain of gamma draft steps of one sequence
    from a prefilled state of the config's prompt length (at most 512 tokens, so that a
    step stays a bounded sample; prefill not timed)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from eagle_speculative_decode_gb300 import synth  # noqa: F401  (generators only)
    from oracle import eagle3_oracle as O
    geo = synth.GEOMETRIES[cfg["geom"]]
    wts = make_bench_weights(geo, args.weights)
    dr = O.Drafter(geo, wts.bits, wts.d2t, kv_format=args.kv_format, int4=wts.int4)
    del wts
    P = min(int(cfg["prompt"][0]), 512)
    toks = synth.make_tokens((P + 1,), geo, 1)
    aux = synth.make_aux((P,), geo, 1)
    st = O.prefill(dr, toks[:P], int(toks[P]), aux)
    gamma = cfg["gamma"]
    for _ in range(args.warmup):
        O.draft_chain(dr, st, gamma)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        O.draft_chain(dr, st, gamma)
    dt = time.perf_counter() - t0
    value = args.steps * gamma / dt
    sample = (f"each step = one chain of {gamma} float64 oracle draft steps of one sequence from a "
              f"{P}-token prefilled state ({cfg['geom']} geometry, prefill not timed); the benchmark's "
              f"batch of {cfg['B']} is not reproduced on the CPU")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "draft tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": static_config(args, cfg, int(os.environ.get("WORLD_SIZE", "1"))),
            "cpu_baseline": {"value": value, "unit": "draft tokens/s", "cores": os.cpu_count(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "draft tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ main arm
def run_mine(args, cfg):
    import torch

    from eagle_speculative_decode_gb300 import binding as Bd
    from eagle_speculative_decode_gb300 import build as _build
    from eagle_speculative_decode_gb300 import synth
    from eagle_speculative_decode_gb300.runtime import DraftModel

    world, rank, local = dist_setup(args.gpus)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if rank == 0:
        _build.build()
    barrier(world)
    Bd.load()

    geo = synth.GEOMETRIES[cfg["geom"]]
    B, gamma, ps = cfg["B"], cfg["gamma"], cfg["page_size"]
    seed = 1000 * rank
    wts = make_bench_weights(geo, args.weights)
    lo, hi = cfg["prompt"]
    lens = synth.ragged_lengths(B, lo, hi, seed=seed + 1) if lo != hi else np.full(B, lo, np.int32)
    rounds = args.warmup + args.steps + args.e2e_steps + args.phase_rounds + 2
    max_cache = int(lens.max()) + (gamma + 1) * rounds + 64
    max_cache = (max_cache + ps - 1) // ps * ps
    model = DraftModel(wts, max_batch=B, max_gamma=gamma, max_cache_len=max_cache, page_size=ps,
                       device=dev, kv_format=args.kv_format)
    del wts
    if args.tc_min_items:
        model.set_tc_min_items(args.tc_min_items)
    if args.tc_schedule:
        model.set_tc_schedule(args.tc_schedule)
    seq = model.new_state(B)

    # prompt: tokens, aux features, the target's next token
    P_max = int(lens.max())
    toks = synth.make_tokens((B, P_max + 1), geo, seed + 2)
    aux = torch.from_numpy(synth.make_aux((B, P_max), geo, seed + 3).view(np.int16)).to(dev)
    t_tok = torch.from_numpy(toks[:, :P_max].copy()).to(dev)
    t_next = torch.from_numpy(toks[np.arange(B), lens].astype(np.int32)).to(dev)
    torch.cuda.synchronize()
    pf0, pf1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    pf0.record()
    seq.prefill(t_tok, t_next, lens, aux)
    pf1.record()
    del aux
    torch.cuda.synchronize()
    prefill_ms = pf0.elapsed_time(pf1)
    prefill_positions = int(lens.sum())

    # per-round synthetic verifier inputs: verify features and imposed accept lengths
    n_rounds_max = rounds
    vaux_host = synth.make_aux((n_rounds_max, B, gamma + 1), geo, seed + 4)
    vaux = torch.from_numpy(vaux_host.view(np.int16)).to(dev)
    n_imp_host = np.stack([synth.imposed_accept_lengths(B, gamma, seed + 5, stream=r,
                                                        p_accept=cfg["p_accept"])
                           for r in range(n_rounds_max)]).astype(np.int32)
    n_imp = torch.from_numpy(n_imp_host).to(dev)
    ar = torch.arange(gamma + 1, device=dev, dtype=torch.int32)
    # The synthetic target's predictions y[b, :gamma] = draft XOR flip: flip is 0 on the
    # first n_imp drafts and 1 after, so exactly n_imp drafts are accepted; the bonus
    # column y[b, gamma] is a fixed token.  One launch per round (the target vocabulary is
    # even, so a flipped id stays in range).
    assert geo.target_vocab % 2 == 0
    flip = (ar[None, None, :gamma] >= n_imp[:, :, None]).to(torch.int32)  # [round, B, gamma]
    out = {"draft_tok": torch.empty(B, gamma, dtype=torch.int32, device=dev),
           "gamma_eff": torch.empty(B, dtype=torch.int32, device=dev)}
    y = torch.full((B, gamma + 1), 7, dtype=torch.int32, device=dev)

    def verify(r, d):
        torch.bitwise_xor(d, flip[r], out=y[:, :gamma])
    n_acc = torch.empty(B, dtype=torch.int32, device=dev)
    bonus = torch.empty(B, dtype=torch.int32, device=dev)
    ctx_sum = [0.0]

    def one_round(r, chain_events=None):
        if chain_events is not None:
            chain_events[0].record()
        seq.draft_chain(gamma, out=out)
        if chain_events is not None:
            chain_events[1].record()
        ctx_sum[0] += float(np.mean(seq._round_start_host)) + (gamma + 1) / 2.0
        seq.rewind()
        # synthetic target: accepts exactly n_imp[r] drafts, then disagrees
        d = out["draft_tok"]
        verify(r, d)
        seq.accept(d, y, out["gamma_eff"], n_acc=n_acc, bonus=bonus)
        seq.rebuild_after_verify(n_acc, d, bonus, vaux[r], n_acc_host=n_imp_host[r])

    r = 0
    for _ in range(args.warmup):
        one_round(r)
        r += 1
    torch.cuda.synchronize()

    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    launches0 = Bd.eagle3_launch_count(model.ctx)
    chain_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(args.steps)]
    ctx_sum[0] = 0.0
    barrier(world)
    torch.cuda.synchronize()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    for i in range(args.steps):
        one_round(r, chain_ev[i])
        r += 1
    stop.record()
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    launches = Bd.eagle3_launch_count(model.ctx) - launches0
    elapsed_ms = start.elapsed_time(stop)
    chain_ms = sum(a.elapsed_time(b) for a, b in chain_ev)
    mean_ctx = ctx_sum[0] / args.steps
    assert model.status() == 0, "device status word set during the benchmark"

    value, elapsed_max = replica_throughput(world, float(B * gamma * args.steps), elapsed_ms)
    ms_per_step = elapsed_max / args.steps

    # ---- per-kernel durations (direct launches with events between kernels)
    model.set_graph_mode(False)
    n_ev = 4 * (2 + 8 * gamma * max(1, (B + 1) // 2) + 16)
    per_label = {}
    for _ in range(args.phase_rounds):
        Bd.eagle3_profile_begin(model.ctx, n_ev)
        seq.draft_chain(gamma, out=out)
        seq.rewind()
        d = out["draft_tok"]
        verify(r, d)
        seq.accept(d, y, out["gamma_eff"], n_acc=n_acc, bonus=bonus)
        seq.rebuild_after_verify(n_acc, d, bonus, vaux[r], n_acc_host=n_imp_host[r])
        for lab, ms in Bd.eagle3_profile_end(model.ctx):
            per_label.setdefault(lab, []).append(ms * 1e3)
        r += 1
    torch.cuda.synchronize()
    model.set_graph_mode(True)
    names = {1: "qkv", 2: "attn", 3: "o", 4: "gateup", 5: "down", 6: "lmhead"}
    # per launch, per kind: average microseconds (one launch per kind per step when B fits)
    kern_us = {names[k]: float(np.mean(v)) for k, v in per_label.items() if k in names}
    # the rebuild's two projections, once per round: encode of the gamma + 1 verify
    # features (fc) and the k/v-only teacher forcing; bytes = weights + activations
    rb_names = {7: "encode", 8: "kv"}
    rb_bytes = {"encode": 3 * geo.n_embd * geo.n_embd * 2 + B * (gamma + 1) * (3 * geo.n_embd * 2 + geo.n_embd * 4),
                "kv": matrix_bytes(2 * geo.kv_rows, 2 * geo.n_embd, args.weights)
                + B * (gamma + 1) * (geo.n_embd * 2 + geo.n_embd * 4 + kv_bytes_per_position(geo, args.kv_format))}
    rebuild_us = {}
    for k, v in per_label.items():
        if k in rb_names:
            us = float(np.sum(v)) / max(1, args.phase_rounds)
            nm = rb_names[k]
            rebuild_us[nm] = {"us_per_round": us, "gbs": rb_bytes[nm] / (us * 1e-6) / 1e9}
    pb = phase_bytes(geo, B, int(mean_ctx), args.kv_format, args.weights)
    hbm_peak, tf_peak, peak_src = load_peaks()
    launches_per_kind = {k: max(1, len(per_label.get(kk, [])) // max(1, args.phase_rounds * gamma))
                         for kk, k in names.items()}
    dominant = max(kern_us, key=lambda k: kern_us[k] * launches_per_kind[k]) if kern_us else "lmhead"
    dom_bytes = pb[dominant] / launches_per_kind[dominant]
    achieved = dom_bytes / (kern_us[dominant] * 1e-6) / 1e9 if kern_us else None
    rb = round_bytes(geo, B, gamma, int(mean_ctx), args.kv_format, args.weights)
    step_frac = (rb / (ms_per_step * 1e-3) / 1e9) / hbm_peak
    chain_bytes = gamma * sum(pb.values())
    chain_frac = (chain_bytes / (chain_ms * 1e-3 / args.steps) / 1e9) / hbm_peak

    # ---- end to end through the C ABI with host buffers
    pin_vaux = torch.from_numpy(vaux_host.view(np.int16)).pin_memory()
    host_tok = torch.empty(B, gamma, dtype=torch.int32).pin_memory()
    host_acc = torch.empty(2, B, dtype=torch.int32).pin_memory()
    acc_pair = torch.empty(2, B, dtype=torch.int32, device=dev)
    vbuf = torch.empty_like(vaux[0])
    torch.cuda.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    for i in range(args.e2e_steps):
        # the chain first (it needs nothing from the host); the round's verify features
        # (the target's, which exist only after it has seen the drafts) are copied in while
        # the chain runs, before the rebuild that reads them
        seq.draft_chain(gamma, out=out)
        vbuf.copy_(pin_vaux[r], non_blocking=True)
        seq.rewind()
        d = out["draft_tok"]
        verify(r, d)
        seq.accept(d, y, out["gamma_eff"], n_acc=acc_pair[0], bonus=acc_pair[1])
        seq.rebuild_after_verify(acc_pair[0], d, acc_pair[1], vbuf, n_acc_host=n_imp_host[r])
        host_tok.copy_(d, non_blocking=True)
        host_acc.copy_(acc_pair, non_blocking=True)
        torch.cuda.synchronize()
        r += 1
    e2e_s = time.perf_counter() - t0
    e2e_s = max_over_ranks(world, e2e_s)
    e2e_val = sum_over_ranks(world, float(B * gamma * args.e2e_steps)) / e2e_s

    # ---- target-side greedy verify of the window (eagle3_verify_greedy): the target head
    # is the tied embedding [V_t, n]; synthetic last hidden states of the B x (gamma + 1)
    # window rows; timed apart from the round (the round's verifier is synthetic)
    verify = None
    if args.verify_steps > 0:
        hid_v = torch.from_numpy(synth.make_hidden((B, gamma + 1), geo, seed + 6)).to(dev)
        t_pred = torch.empty(B, gamma + 1, dtype=torch.int32, device=dev)
        head, tnorm = model.w["embed"], model.w["final_norm"]
        d = out["draft_tok"]
        for _ in range(3):
            seq.verify_greedy(head, tnorm, hid_v, d, out["gamma_eff"], target_pred=t_pred,
                              n_acc=n_acc, bonus=bonus)
        torch.cuda.synchronize()
        v0, v1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        v0.record()
        for _ in range(args.verify_steps):
            seq.verify_greedy(head, tnorm, hid_v, d, out["gamma_eff"], target_pred=t_pred,
                              n_acc=n_acc, bonus=bonus)
        v1.record()
        torch.cuda.synchronize()
        v_us = v0.elapsed_time(v1) * 1e3 / args.verify_steps
        rows = B * (gamma + 1)
        v_bytes = geo.target_vocab * geo.n_embd * 2 + rows * geo.n_embd * 4 + geo.n_embd * 2 + rows * 4
        verify = {"us_per_call": v_us, "rows": rows, "target_vocab": geo.target_vocab,
                  "bytes_per_call": v_bytes, "achieved_gbs": v_bytes / (v_us * 1e-6) / 1e9,
                  "frac": v_bytes / (v_us * 1e-6) / 1e9 / hbm_peak,
                  "kernel": ("target lm_head tcgen05 GEMM" if rows >= 3 else "target lm_head GEMV")
                  + " + argmax, then the accept walk",
                  "note": "target head = the tied embedding bf16 [V_t, n]; float32 synthetic hidden states"}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        try:
            rate, secs, desc = oracle_round_rate(cfg["geom"], gamma, args.cpu_rounds,
                                                 kv_format=args.kv_format, weights=args.weights,
                                                 prompt=min(int(lens.min()), 512),
                                                 seconds=args.cpu_seconds)
            cpu = {"value": rate, "unit": "draft tokens/s", "cores": os.cpu_count(),
                   "kind": "oracle", "sample": desc, "seconds": secs}
        except Exception as e:  # reported, not fatal
            cpu = {"value": None, "unit": "draft tokens/s", "cores": os.cpu_count(),
                   "kind": "oracle", "sample": f"failed: {e}"}

    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": "draft tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if args.weights == "bf16" else "int4", "data": "synthetic",
        "config": dict(static_config(args, cfg, world), prompt=[int(lens.min()), int(lens.max())],
                       mean_context=round(mean_ctx, 1)),
        "us_per_draft_step": ms_per_step * 1e3 / gamma,
        "chain_us_per_draft_step": chain_ms * 1e3 / (args.steps * gamma),
        "step_roofline": {"bytes_per_step": rb, "achieved_gbs": rb / (ms_per_step * 1e-3) / 1e9,
                          "peak_gbs": hbm_peak, "frac": step_frac,
                          "frac_of_nominal": step_frac * hbm_peak / NOMINAL_HBM_GBS,
                          "chain_frac": chain_frac, "chain_frac_of_nominal": chain_frac * hbm_peak / NOMINAL_HBM_GBS,
                          "note": f"algorithmic bytes of the whole round (chain: of the gamma draft steps) / "
                                  f"its time, of {peak_src} hbm_gbs; *_of_nominal: of the 8 TB/s datasheet peak"},
        "roofline": {"bound": "hbm", "kernel": kernel_label(dominant, B, args.weights),
                     "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                     "frac": (achieved / hbm_peak) if achieved else None,
                     "frac_of_nominal": (achieved / NOMINAL_HBM_GBS) if achieved else None,
                     "traffic": profiled_traffic(args.config, dominant, args.kv_format, args.weights)
                     if args.weights == "bf16" else None,
                     "peak_source": f"{peak_src} hbm_gbs (copy, burst)",
                     "bytes_per_launch": dom_bytes, "us_per_launch": kern_us.get(dominant)},
        "kernel_us": kern_us,
        "rebuild_kernel_us": rebuild_us,
        "prefill": {"positions": prefill_positions, "ms": prefill_ms,
                    "positions_per_s": prefill_positions / (prefill_ms * 1e-3),
                    "note": "eagle3_prefill of the prompts (encode + k/v teacher forcing), timed once"},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_val, "unit": "draft tokens/s",
                "h2d_bytes_per_step": int(vaux[0].numel() * 2),
                "d2h_bytes_per_step": int(host_tok.numel() * 4 + host_acc.numel() * 4),
                "steps": args.e2e_steps},
        "verify": verify,
        "gpu_launches": int(launches),
        "clocks": clk,
    }
    print(json.dumps(line), flush=True)
    model.close()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="mine", choices=["mine", "reference"])
    ap.add_argument("--config", default="c2", choices=sorted(CONFIGS))
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--phase-rounds", type=int, default=3)
    ap.add_argument("--cpu-rounds", type=int, default=1,
                    help="chains the CPU baseline times at least")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="CPU baseline sample length: chains are timed until this many seconds")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--verify-steps", type=int, default=10,
                    help="timed calls of the target-side greedy verify (0: skip)")
    ap.add_argument("--weights", default="bf16", choices=["bf16", "int4"],
                    help="drafter projection weights: bf16, or INT4 codes with bf16 group scale / zero")
    ap.add_argument("--kv-format", default="bf16", choices=["bf16", "q8_0/q5_1"],
                    help="drafter KV cache storage: bf16, or q8_0 keys / q5_1 values")
    ap.add_argument("--tc-min-items", type=int, default=0,
                    help="activation rows from which projections use the tensor cores (0: library default)")
    ap.add_argument("--tc-schedule", type=int, default=0, choices=[0, 1, 2],
                    help="tensor-core tile schedule: 0 library default, 1 stream-K, 2 cluster split-K where it fits")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    cfg = CONFIGS[args.config]
    if args.impl == "reference":
        run_reference(args, cfg)
    else:
        run_mine(args, cfg)


if __name__ == "__main__":
    main()

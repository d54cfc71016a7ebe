#!/usr/bin/env python
"""Benchmark of the KDA recurrent-state hot path on one GB300 per rank.

Main line: speculative-decode verify + ReplaySSM commit, 16 sequences x 32
heads x d=128, bf16 inputs, fp32 state in 64 shuffled slots, T = 8 drafts,
accepted_len ~ U{0..8}, ring depth 8.  One step = one decode step of the
model's KDA layers: kda_verify on each of NL layers (each also applies that
layer's pending commit from the previous step), then one kda_commit_layers
recording the step's accepted lengths in every layer's ring.  NL layers have their own state
pools, so the state touched per step is NL x 32 MiB, at least 4x the L2.  The
value is drafted tokens verified through one KDA layer per second,
B * T * NL * steps / time.  Each step is one CUDA graph captured from the
public API calls, with a timing event pair around its NL verify launches
(the verify launch duration is that block's time / NL).

Extra keys: `roofline` (verify kernel vs HBM), `cpu_baseline` (the fp64
oracle on the host cores, bounded sample), `e2e` (same metric through the
public calls issued eagerly every step -- kda_verify per layer and
kda_commit_layers through the binding -- with every step's inputs copied from
pinned host memory and its outputs copied back inside the timed region, the
copies of neighbouring steps overlapping the compute on their own streams),
`e2e_graph` (the same loop replaying CUDA graphs captured from those calls), `prefill` (chunked prefill with in-pass checkpoints,
1 x 8192 tokens, chunk 64, checkpoint every 1024, own timed region: the
two-pass path through the workspace, and the single pass beside it),
`clocks` (nvidia-smi samples during the timed region),
`mixed` (the mixed-batch workload: 64 rows, 8 speculative + 56 ordinary, in
256 shuffled slots, own timed region with its HBM roofline; and the same
batch with a 2048-token prefill segment in front through kda_forward_mixed,
one stream and with a side stream),
`serving` (16 sequences x 8192-token prefill with checkpoints every 1024,
then T = 8 verify + commit with capped-geometric acceptance until 1024 tokens
are committed per sequence, on the same NL layers: prefill, verified and
committed tokens/s and the KDA-layer time),
`tiny` (latency of the tiny correctness workload: 1 sequence, 2 heads,
d = 16, fp32, a 64-token prefill then 8 verify + commit steps with T = 4),
`ablation_direct_snapshots` (the design ReplaySSM replaces -- the state
stored at every drafted position, the accepted one copied at commit -- on the
same workload, its own timed region; with both designs' algorithmic bytes
per step and state-cache bytes per sequence at a 46.48 GiB budget).

`--impl reference` times the oracle itself on the host cores on the same
workload (rank 0 only).
"""
import argparse
import hashlib
import json
import math
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import kda_inputs as ki  # noqa: E402

METRIC = "KDA verify+commit tokens/s, % of HBM roofline; chunked-prefill tokens/s"
B, H, D, P, T, DEPTH = 16, 32, 128, 64, 8, 8
FALLBACK_HBM_GBS = 6800.0


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1024)
    ap.add_argument("--warmup", type=int, default=16)
    ap.add_argument("--impl", choices=["kda", "reference"], default="kda")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="budget of the oracle CPU-baseline sample")
    return ap.parse_args()


# ------------------------------------------------------------------ helpers
def unit_bytes(a_prev, d=D, t=T):
    """Algorithmic HBM bytes of one (sequence, head) unit of one verify launch:
    state read, state write when the pending commit is non-empty, the T drafted
    tokens' inputs (q, k, v, alpha bf16 + beta), their fp32 outputs, ring write
    of (k, v, alpha, beta) for T tokens, ring read of a_prev entries, slot and
    ctrl words."""
    ring_tok = 3 * d * 2 + 2
    return (d * d * 4 + d * d * 4 * (a_prev > 0) + t * (4 * d * 2 + 2)
            + t * d * 4 + t * ring_tok + a_prev * ring_tok + 8)


def load_tensor_peak():
    """Measured dense bf16 tensor peak (burst) in TFLOP/s, and its source."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                pk = json.load(f)
            if pk.get("bf16_tflops"):
                return float(pk["bf16_tflops"]), "measured"
        except Exception:
            pass
    return 1900.0, "fallback"


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                pk = json.load(f)
            if pk.get("hbm_gbs"):
                return float(pk["hbm_gbs"]), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


def source_hash(unit, extra=()):
    """First 16 hex digits of the SHA-256 of a kernel's translation unit and
    the headers it includes: a committed profile is used only when it was
    taken on the same source."""
    h = hashlib.sha256()
    for name in (unit,) + tuple(extra) + ("kda_umma.cuh", "kda_internal.cuh"):
        with open(os.path.join(ROOT, "recurrent_kda_state_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def verify_source_hash():
    """The pipelined verify kernel (the spec-decode and mixed workloads' shape)
    and the single-token step it shares with the per-unit kernel."""
    return source_hash("kda_verify_pipe.cu", ("kda_step.cuh",))


def ncu_traffic():
    """Per-launch DRAM bytes of the verify kernel from the committed ncu
    summary, if it was taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "verify_spec_traffic.json")
    if not os.path.exists(path):
        return None
    try:
        with open(path) as f:
            rec = json.load(f)
        if rec.get("kernel_source_sha256_16") == verify_source_hash():
            return float(rec["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while running."""
    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index),
                 "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)

    def summary(self, t0, t1):
        rows = [s for (t, s) in self.samples if t0 <= t <= t1] or \
               [s for (_, s) in self.samples]
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for r in rows:
            parts = [p.strip() for p in r.split(",")]
            if len(parts) < 6:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for n, v in zip(names, parts[2:6]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                    "samples": 0}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------ oracle timing
def oracle_spec_rate(seconds, heads_sampled=2, seed=ki.SEED_SPEC):
    """Oracle verify+commit on the spec workload, restricted to a sample of
    heads, until `seconds` of CPU work are spent.  Returns (tokens/s scaled to
    all heads, cores, sample description, steps)."""
    import oracle
    rng = np.random.default_rng(seed)
    slots = ki.slot_table(rng, B, P)
    sess = oracle.OracleSession(P, heads_sampled, D, D)
    toks = [ki.round_to(ki.gen_tokens(rng, [T] * B, heads_sampled, D), "bf16")
            for _ in range(8)]
    accs = [ki.accepted_uniform(rng, B, T) for _ in range(8)]
    steps, t0 = 0, time.perf_counter()
    while steps < 1 or time.perf_counter() - t0 < seconds:
        sess.verify(toks[steps % 8], slots)
        sess.commit(accs[steps % 8], slots)
        steps += 1
    el = time.perf_counter() - t0
    rate = B * T * steps * heads_sampled / H / el
    desc = ("%d spec steps (16 seqs x T=8, commit a~U{0..8}) on %d of 32 heads, "
            "d=128, fp64; scaled to 32 heads" % (steps, heads_sampled))
    return rate, oracle.num_threads(), desc, steps


# ----------------------------------------------------------- reference arm
# ---------------------------------------------------------- replicas (N > 1)
# The path has no exchange step: every rank runs an independent replica of
# the workload (weak scaling).  These are the host-side pieces of that.
def replica_rng(rank, seed=None):
    """Each replica draws its own inputs from its own seeded stream."""
    return np.random.default_rng((ki.SEED_SPEC if seed is None else seed) + 7919 * rank)


def max_over_ranks(x, dist, device="cpu"):
    """The largest value of x over the ranks (x itself without a group)."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(tokens_per_rank, world, ms):
    """Whole-job tokens/s: all ranks' tokens over the slowest rank's time."""
    return tokens_per_rank * world / (ms * 1e-3)


def run_reference(args, rank, world):
    if rank != 0:
        return
    import oracle
    rng = np.random.default_rng(ki.SEED_SPEC)
    hs = 1  # each step: one layer x 16 seqs x 1 head (bounded sample)
    slots = ki.slot_table(rng, B, P)
    sess = oracle.OracleSession(P, hs, D, D)
    toks = [ki.round_to(ki.gen_tokens(rng, [T] * B, hs, D), "bf16")
            for _ in range(8)]
    accs = [ki.accepted_uniform(rng, B, T) for _ in range(8)]

    def step(s):
        sess.verify(toks[s % 8], slots)
        sess.commit(accs[s % 8], slots)
    for s in range(args.warmup):
        step(s)
    t0 = time.perf_counter()
    for s in range(args.steps):
        step(s)
    el = time.perf_counter() - t0
    value = B * T * args.steps * hs / H / el
    line = {
        "impl": "reference", "metric": METRIC, "value": value,
        "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": el * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic",
        "config": {"workload": ki.SPEC.name, "sample": "1 of 32 heads per step"},
        "cpu_baseline": {"value": value, "unit": "tokens/s",
                         "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": "each step: verify T=8 + commit for 16 seqs "
                                   "on 1 of 32 heads (fp64), scaled to 32 heads"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------ kda arm
def build_inputs(torch, rng, NL, dev):
    """One input set: NL layers of packed tokens in one contiguous arena."""
    N = B * T
    per = N * H * D * 4 + N * H          # q, k, v, alpha + beta (bf16 elems)
    arena = torch.empty(NL * per, dtype=torch.bfloat16, device=dev)
    views = []
    for l in range(NL):
        tok = ki.gen_tokens(rng, [T] * B, H, D)
        base = l * per
        vs = {}
        off = base
        for n in ("q", "k", "v", "alpha"):
            vs[n] = arena[off:off + N * H * D].view(N, H, D)
            vs[n].copy_(torch.from_numpy(tok[n]).to(torch.bfloat16))
            off += N * H * D
        vs["beta"] = arena[off:off + N * H].view(N, H)
        vs["beta"].copy_(torch.from_numpy(tok["beta"]).to(torch.bfloat16))
        views.append(vs)
    return arena, views


def prefill_tensor_profile():
    """Tensor-pipe utilisation of the two prefill passes from the committed ncu
    summary, when it was taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", "prefill_tc_tensor.json")
    try:
        with open(path) as f:
            prof = json.load(f)
        sha = source_hash("kda_prefill_tc.cu")
    except OSError:
        return None
    if prof.get("kernel_source_sha256_16") != sha:
        return None
    return {k: prof[k] for k in ("sm__pipe_tensor_cycles_active_pct",
                                 "dram_bytes_per_call", "kernels", "source")
            if k in prof}


def run_prefill(torch, K, dev):
    w = ki.PREFILL
    rng = np.random.default_rng(w.seed)
    L, C, E = 8192, 64, 1024
    tok = ki.gen_tokens(rng, [L], H, D)
    t = {n: torch.from_numpy(tok[n]).to(device=dev, dtype=torch.bfloat16)
         for n in ("q", "k", "v", "alpha", "beta")}
    cu = torch.tensor([0, L], dtype=torch.int32, device=dev)
    tb = K.TokenBatch(t["q"], t["k"], t["v"], t["alpha"], t["beta"], cu)
    init = ki.initial_states(rng, 1, H, D, D, 0.02)
    pool = K.StatePool.zeros(1 + L // E, H, D, device=dev)
    pool.data[0].copy_(torch.from_numpy(np.swapaxes(init[0], -1, -2).copy()))
    slots = torch.tensor([0], dtype=torch.int32, device=dev)
    ck = torch.arange(1, 1 + L // E, dtype=torch.int32, device=dev).view(1, -1)
    ws_bytes = K.kda_prefill_workspace_size(L, 1, H, D, D, C, K.KDA_BF16)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev) if ws_bytes else None
    stream = torch.cuda.current_stream()
    reps = 10

    def timed(single):
        for _ in range(3):
            K.kda_prefill_chunked(tb, pool, slots, C, E, ck, workspace=ws,
                                  single_pass=single)
        evs = [(torch.cuda.Event(enable_timing=True),
                torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
        torch.cuda.synchronize()
        for e0, e1 in evs:
            e0.record(stream)
            K.kda_prefill_chunked(tb, pool, slots, C, E, ck, workspace=ws,
                                  single_pass=single)
            e1.record(stream)
        torch.cuda.synchronize()
        return float(np.mean([a.elapsed_time(b) for a, b in evs]))

    ms = timed(False)
    ms_single = timed(True)
    # the same prefill on projection-space inputs, prep fused into the kernels
    rtok = ki.gen_raw_tokens(rng, [L], H, D)
    rt = {n: torch.from_numpy(rtok[n]).to(device=dev, dtype=torch.bfloat16)
          for n in ("q", "k", "v", "alpha", "beta")}
    rtb = K.TokenBatch(rt["q"], rt["k"], rt["v"], rt["alpha"], rt["beta"], cu)
    for _ in range(3):
        K.kda_prefill_chunked(rtb, pool, slots, C, E, ck, workspace=ws, raw=True)
    revs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(reps)]
    torch.cuda.synchronize()
    for e0, e1 in revs:
        e0.record(stream)
        K.kda_prefill_chunked(rtb, pool, slots, C, E, ck, workspace=ws, raw=True)
        e1.record(stream)
    torch.cuda.synchronize()
    ms_raw = float(np.mean([a.elapsed_time(b) for a, b in revs]))
    # a separate prep pass would read the raw k, alpha, beta and write them back
    prep_bytes = 2 * (L * H * (2 * D) * 2 + L * H * 2)
    del ws, rt, rtb
    torch.cuda.empty_cache()
    alg_bytes = (L * H * (4 * D * 2 + 2) + L * H * D * 4
                 + (2 + L // E) * H * D * D * 4)
    flops = 11.6e6 * (L // C) * H
    # every tensor-core product of a non-input operand is taken as three bf16
    # products (hi*hi, lo*hi, hi*lo): the MMAs issue about 3x the chunk form
    issued = 3.0 * flops
    hbm_peak, hbm_kind = load_peaks()
    tc_peak, tc_kind = load_tensor_peak()
    prof = prefill_tensor_profile()
    achieved_gbs = alg_bytes / (ms * 1e-3) / 1e9
    roofline = {
        "bound": "hbm", "achieved": achieved_gbs, "peak": hbm_peak, "unit": "GB/s",
        "frac": achieved_gbs / hbm_peak, "peak_source": hbm_kind,
        "traffic": prof.get("dram_bytes_per_call") if prof else None,
        "alg_bytes": alg_bytes,
        "tensor": {"chunk_tflops": flops / (ms * 1e-3) / 1e12,
                   "issued_tflops": issued / (ms * 1e-3) / 1e12,
                   "peak_tflops": tc_peak, "peak_source": tc_kind,
                   "frac_chunk": flops / (ms * 1e-3) / 1e12 / tc_peak,
                   "frac_issued": issued / (ms * 1e-3) / 1e12 / tc_peak,
                   "pipe_active_pct": prof.get("sm__pipe_tensor_cycles_active_pct")
                   if prof else None,
                   "chunk_flops": flops},
    }
    return {
        "workload": w.name, "tokens_per_s": L / (ms * 1e-3), "ms": ms,
        "roofline": roofline,
        "workspace_bytes": ws_bytes,
        "single_pass_ms": ms_single,
        "raw_inputs_fused_prep_ms": ms_raw,
        "raw_prep_pass_bytes_avoided": prep_bytes,
        "reps": reps,
    }


def decode_unit_bytes(d=D):
    """Algorithmic bytes of an ordinary (one-token, committed at once) row's
    (sequence, head) unit: state read and write, the token's inputs and
    output, ctrl word and slot."""
    return 2 * d * d * 4 + (4 * d * 2 + 2) + d * 4 + 8 + 4


def run_mixed(torch, K, dev, steps=32, warmup=4, NL=4, prefill_len=2048):
    """The mixed-batch workload: 64 sequences in 256 shuffled slots, 8
    speculative (T = 8, accepted ~ U{0..8}) at seeded random positions among
    56 ordinary one-token rows, one packed batch per step (kda_verify over all
    64, then the commit); NL layer pools rotate so the state touched per step
    (NL x 128 MiB) exceeds the L2; one CUDA graph per step, an event pair
    around its NL verify launches.  Then the same batch with a 2048-token
    prefill segment in front (checkpoint every 1024), one layer, through
    kda_forward_mixed on one stream and with the prefill on a side stream."""
    w = ki.MIXED
    rng = np.random.default_rng(w.seed)
    Bm, Pm, nspec, Tm = w.num_seqs, w.extra["num_slots"], w.extra["num_spec"], w.extra["T"]
    slots_np = ki.slot_table(rng, Bm, Pm)
    is_spec_np = np.zeros(Bm, np.int32)
    is_spec_np[rng.choice(Bm, nspec, replace=False)] = 1
    lens = [Tm if x else 1 for x in is_spec_np]
    N = sum(lens)
    slots = torch.as_tensor(slots_np, device=dev)
    is_spec = torch.as_tensor(is_spec_np, device=dev)
    pools = [K.StatePool.zeros(Pm + 3, H, D, device=dev) for _ in range(NL)]
    rings = [K.ReplayRing(Pm + 3, H, D, Tm, torch.bfloat16, device=dev) for _ in range(NL)]

    def batch(lengths):
        tok = ki.gen_tokens(rng, lengths, H, D)
        t = {n: torch.from_numpy(tok[n]).to(device=dev, dtype=torch.bfloat16)
             for n in ("q", "k", "v", "alpha", "beta")}
        cu = torch.as_tensor(tok["cu_seqlens"], device=dev)
        return K.TokenBatch(t["q"], t["k"], t["v"], t["alpha"], t["beta"], cu)

    G = 4
    sets = [[batch(lens) for _ in range(NL)] for _ in range(G)]
    A = 64
    acc_np = np.where(is_spec_np[None, :] == 1,
                      ki.accepted_uniform(rng, A * Bm, Tm).reshape(A, Bm), 0).astype(np.int32)
    acc = torch.as_tensor(acc_np, device=dev)
    # one CUDA graph per step (NL verify launches between one event pair,
    # then the commit), as in the main line
    gstream = torch.cuda.Stream(device=dev)
    graphs = []
    with torch.cuda.stream(gstream):
        for s in range(warmup + steps):
            g = torch.cuda.CUDAGraph()
            ev = (torch.cuda.Event(enable_timing=True, external=True),
                  torch.cuda.Event(enable_timing=True, external=True)) \
                if s >= warmup else None
            g.capture_begin()
            if ev:
                ev[0].record(gstream)
            for l in range(NL):
                K.kda_verify(sets[s % G][l], Tm, pools[l], slots, rings[l],
                             is_spec=is_spec, stream=gstream)
            if ev:
                ev[1].record(gstream)
            K.kda_commit_layers(acc[s % A], slots, pools[0], rings, stream=gstream)
            g.capture_end()
            graphs.append((g, ev))
    torch.cuda.synchronize()
    with torch.cuda.stream(gstream):
        for g, _ in graphs[:warmup]:
            g.replay()
        torch.cuda.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(gstream)
        for g, _ in graphs[warmup:]:
            g.replay()
        t1.record(gstream)
    torch.cuda.synchronize()
    ms = t0.elapsed_time(t1)
    durs, byts = [], []
    for s in range(warmup, warmup + steps):
        ev = graphs[s][1]
        durs.append(ev[0].elapsed_time(ev[1]) / NL)
        prev = acc_np[(s - 1) % A]
        byts.append(float(sum(unit_bytes(int(prev[i])) if is_spec_np[i] else decode_unit_bytes()
                              for i in range(Bm)) * H))
    del graphs
    stream = torch.cuda.current_stream()
    mean_us = float(np.mean(durs)) * 1e3
    achieved = float(np.mean(byts)) / (mean_us * 1e-6) / 1e9
    peak, _ = load_peaks()
    bits = K.kda_get_device_error()

    # the same decode batch with a prefill segment in front, one layer
    mixed = batch([prefill_len] + lens)
    pslots = torch.as_tensor(np.concatenate([[Pm], slots_np]).astype(np.int32), device=dev)
    pspec = torch.as_tensor(np.concatenate([[0], is_spec_np]).astype(np.int32), device=dev)
    ck = torch.tensor([[Pm + 1, Pm + 2]], dtype=torch.int32, device=dev)
    sp = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = None
    side = torch.cuda.Stream(device=dev)
    acc_m = torch.as_tensor(np.concatenate([np.zeros((A, 1), np.int32), acc_np], 1), device=dev)

    def mixed_ms(use_side, n=16):
        nonlocal ws
        out = []
        for s in range(3 + n):
            e0, e1 = (torch.cuda.Event(enable_timing=True),
                      torch.cuda.Event(enable_timing=True))
            e0.record(stream)
            ws = K.kda_forward_mixed(mixed, 1, prefill_len, pools[0], pslots, 64, Tm, rings[0],
                                     ckpt_every=1024, ckpt_slots=ck, start_pos=sp,
                                     is_spec=pspec, workspace=ws,
                                     side_stream=side if use_side else None)
            K.kda_commit(acc_m[s % A], pslots, pools[0], rings[0])
            e1.record(stream)
            if s >= 3:
                out.append((e0, e1))
        torch.cuda.synchronize()
        return float(np.mean([a.elapsed_time(b) for a, b in out]))

    one = mixed_ms(False)
    two = mixed_ms(True)
    bits |= K.kda_get_device_error()
    del pools, rings, sets, ws
    torch.cuda.empty_cache()
    return {
        "workload": w.name, "kda_layers": NL, "steps": steps,
        "tokens_per_step": N, "value": N * steps * NL / (ms * 1e-3), "unit": "tokens/s",
        "ms_per_step": ms / steps,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "kernel": "verify_pipe_kernel (d=128, bf16; 64 rows)",
                     "mean_launch_us": mean_us, "alg_bytes_per_launch": float(np.mean(byts))},
        "with_prefill_segment": {
            "prefill_tokens": prefill_len, "decode_tokens": N,
            "ms_one_stream": one, "ms_side_stream": two,
            "note": "kda_forward_mixed + commit, one layer: the prefill segment "
                    "(two passes through the workspace) and the 64 decode rows "
                    "of one packed batch, serial on one stream or with the "
                    "prefill part forked onto a side stream"},
        "device_error_bits": bits,
    }


CACHE_BUDGET_GIB = 46.48   # the pages' KV/state cache budget for the comparison


def state_cache_bytes(d=D, h=H, t=T, depth=DEPTH):
    """Per-sequence state-cache bytes of one KDA layer in each design: the
    committed state plus, for ReplaySSM, the ring (k, alpha, v bf16 + beta
    per entry, and the control pair), for direct snapshots, T more states."""
    state = h * d * d * 4
    ring = h * depth * (3 * d * 2 + 2) + h * 2 * 4
    return {"replay_ssm": state + ring, "direct_snapshots": state * (1 + t)}


def snapshot_unit_bytes(a, d=D, t=T):
    """Algorithmic HBM bytes of one (sequence, head) unit of one step of the
    direct design: verify reads the state and the T drafted tokens' inputs,
    writes T outputs and T state snapshots; the commit copies snapshot a - 1
    into the pool when a > 0; slot and accepted-length words."""
    verify = d * d * 4 + t * (4 * d * 2 + 2) + t * d * 4 + t * d * d * 4 + 4
    commit = 2 * d * d * 4 * (a > 0) + 8
    return verify, commit


def run_snapshot_ablation(torch, K, dev, NL, slots, batches, acc, acc_np, G, A,
                          steps=64, warmup=4):
    """The direct per-position snapshot design on the same workload: per step
    kda_verify_snapshot on each of NL layers, then kda_commit_snapshot of the
    step's accepted lengths on each layer.  Own pools (zero), own timed
    region, one CUDA event pair around each step's NL verify launches and
    one around its NL commits (launch durations = block time / NL)."""
    pools = [K.StatePool.zeros(P, H, D, device=dev) for _ in range(NL)]
    snaps = [K.snapshot_buffer(B, T, pools[l]) for l in range(NL)]
    stream = torch.cuda.Stream(device=dev)
    graphs, events = [], []
    with torch.cuda.stream(stream):
        for s in range(warmup + steps):
            g = torch.cuda.CUDAGraph()
            # event pairs around the NL verify launches and the NL commits
            ev = [torch.cuda.Event(enable_timing=True, external=True)
                  for _ in range(4)] if s >= warmup else None
            g.capture_begin()
            if ev:
                ev[0].record(stream)
            for l in range(NL):
                K.kda_verify_snapshot(batches[s % G][l], T, pools[l], slots,
                                      snaps[l], stream=stream)
            if ev:
                ev[1].record(stream)
                ev[2].record(stream)
            for l in range(NL):
                K.kda_commit_snapshot(acc[s % A], slots, pools[l], snaps[l],
                                      stream=stream)
            if ev:
                ev[3].record(stream)
            g.capture_end()
            graphs.append(g)
            events.append(ev)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for s in range(warmup):
            graphs[s].replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for s in range(warmup, warmup + steps):
            graphs[s].replay()
        e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    bits = K.kda_get_device_error()
    v_us, c_us, v_bytes, c_bytes = [], [], [], []
    for s in range(warmup, warmup + steps):
        per = [snapshot_unit_bytes(int(x)) for x in acc_np[s % A]]
        v_bytes.append(float(sum(p[0] for p in per) * H))
        c_bytes.append(float(sum(p[1] for p in per) * H))
        ev = events[s]
        v_us.append(ev[0].elapsed_time(ev[1]) * 1e3 / NL)
        c_us.append(ev[2].elapsed_time(ev[3]) * 1e3 / NL)
    del graphs, snaps, pools
    torch.cuda.empty_cache()
    v_mean, c_mean = float(np.mean(v_us)), float(np.mean(c_us))
    return {
        "value": B * T * steps * NL / (ms * 1e-3), "unit": "tokens/s",
        "ms_per_step": ms / steps, "steps": steps, "warmup": warmup,
        "kda_layers": NL,
        "verify_launch_us": v_mean, "commit_launch_us": c_mean,
        "alg_bytes_per_layer_step": float(np.mean(v_bytes) + np.mean(c_bytes)),
        "verify_achieved_gbs": float(np.mean(v_bytes)) / (v_mean * 1e-6) / 1e9,
        "commit_achieved_gbs": float(np.mean(c_bytes)) / (c_mean * 1e-6) / 1e9,
        "device_error_bits": bits,
        "note": "direct design: T state snapshots written per (sequence, head) "
                "per step, the accepted one copied into the pool; same inputs, "
                "slots and accepted lengths as the main line",
    }


def serving_schedule(rng, n, decode_tokens, rho, t=T):
    """Decode steps of the serving-shaped load: each step every live sequence
    verifies t drafts and commits a capped-geometric accepted count, the last
    one clipped so that a sequence stops at exactly ``decode_tokens``
    committed.  Returns [(live sequence indices, accepted counts)]."""
    committed = np.zeros(n, dtype=np.int64)
    steps = []
    while committed.min() < decode_tokens:
        live = np.nonzero(committed < decode_tokens)[0].astype(np.int32)
        a = ki.accepted_capped_geometric(rng, len(live), rho, t)
        a = np.minimum(a, decode_tokens - committed[live]).astype(np.int32)
        committed[live] += a
        steps.append((live, a))
    return steps


def serving_verify_bytes(steps, h=H):
    """Algorithmic bytes of the decode phase's verify launches (one layer):
    per live (sequence, head) unit the spec-verify bytes, with the replay of
    that sequence's previous accepted count."""
    prev = {}
    total = 0
    for live, a in steps:
        total += sum(unit_bytes(prev.get(int(i), 0)) for i in live) * h
        prev.update({int(i): int(x) for i, x in zip(live, a)})
    return total


def run_verify_raw(torch, K, dev, NL, slots, acc, A, G=4, steps=64, warmup=4):
    """The spec-decode step on projection-space inputs: kda_verify_raw (key
    L2 norm, alpha = exp(-softplus(z)), beta = sigmoid(b) fused into the
    verify kernel) on each of NL layers, then kda_commit_layers, with the
    main line's slots and accepted lengths.  Own pools and rings, own timed
    region, one CUDA event pair around each step's NL verify launches."""
    rng = np.random.default_rng(ki.SPEC.seed + 7)
    pools = [K.StatePool.zeros(P, H, D, device=dev) for _ in range(NL)]
    rings = [K.ReplayRing(P, H, D, DEPTH, torch.bfloat16, device=dev) for _ in range(NL)]
    cu = torch.tensor(np.arange(0, (B + 1) * T, T, dtype=np.int32), device=dev)
    batches = []
    for _ in range(G):
        tok = ki.gen_raw_tokens(rng, [T] * B, H, D)
        t = {n: torch.from_numpy(tok[n]).to(device=dev, dtype=torch.bfloat16)
             for n in ("q", "k", "v", "alpha", "beta")}
        batches.append(K.TokenBatch(t["q"], t["k"], t["v"], t["alpha"], t["beta"], cu))
    stream = torch.cuda.Stream(device=dev)
    graphs, events = [], []
    with torch.cuda.stream(stream):
        for s in range(warmup + steps):
            g = torch.cuda.CUDAGraph()
            ev = [torch.cuda.Event(enable_timing=True, external=True)
                  for _ in range(2)] if s >= warmup else None
            g.capture_begin()
            if ev:
                ev[0].record(stream)
            for l in range(NL):
                K.kda_verify(batches[s % G], T, pools[l], slots, rings[l], stream=stream,
                             raw=True)
            if ev:
                ev[1].record(stream)
            K.kda_commit_layers(acc[s % A], slots, pools[0], rings, stream=stream)
            g.capture_end()
            graphs.append(g)
            events.append(ev)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for s in range(warmup + steps):
            graphs[s].replay()
    torch.cuda.synchronize()
    bits = K.kda_get_device_error()
    us = float(np.mean([events[s][0].elapsed_time(events[s][1]) * 1e3 / NL
                        for s in range(warmup, warmup + steps)]))
    del graphs, rings, pools
    torch.cuda.empty_cache()
    return {"verify_launch_us": us, "tokens_per_s": B * T / (us * 1e-6),
            "device_error_bits": bits,
            "note": "kda_verify_raw x NL + kda_commit_layers per step, CUDA graphs, "
                    "event pair around the NL verify launches; raw keys, decay and "
                    "beta logits prepared in the kernel"}


def run_serving(torch, K, dev, NL, G=4):
    """Serving-shaped load on NL KDA layers (own pools and rings per layer):
    16 sequences prefilled in passes of at most 16384 tokens (chunk 64, a
    checkpoint every 1024 tokens into its own slot), their rings reset, then
    T = 8 verify + ReplaySSM commit steps with capped-geometric accepted
    counts until every sequence has 1024 tokens committed, and a final
    materialize.  The decode steps are CUDA graphs captured from the public
    calls (their live slot tables and accepted counts on the device before
    timing); one warm run, then one timed run, events at the phase
    boundaries."""
    w = ki.SERVING
    x = w.extra
    Bs, L, C, E = w.num_seqs, x["prefill_len"], x["chunk"], x["ckpt_every"]
    rng = np.random.default_rng(w.seed)
    per_pass = max(1, 16384 // L)
    n_ck = L // E
    Ps = Bs * (1 + n_ck)
    perm = rng.permutation(Ps).astype(np.int32)
    seq_slot = perm[:Bs]
    ck_np = perm[Bs:].reshape(Bs, n_ck)
    pools = [K.StatePool.zeros(Ps, H, D, device=dev) for _ in range(NL)]
    rings = [K.ReplayRing(Ps, H, D, x["depth"], torch.bfloat16, device=dev)
             for _ in range(NL)]
    tok = ki.gen_tokens(rng, [L] * per_pass, H, D)
    pt = {n: torch.from_numpy(tok[n]).to(device=dev, dtype=torch.bfloat16)
          for n in ("q", "k", "v", "alpha", "beta")}
    del tok
    cu_p = torch.arange(0, (per_pass + 1) * L, L, dtype=torch.int32, device=dev)
    ptb = K.TokenBatch(pt["q"], pt["k"], pt["v"], pt["alpha"], pt["beta"], cu_p)
    ws_bytes = K.kda_prefill_workspace_size(per_pass * L, per_pass, H, D, D, C,
                                            K.KDA_BF16)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev) if ws_bytes else None
    passes = [(torch.as_tensor(seq_slot[i:i + per_pass], device=dev),
               torch.as_tensor(ck_np[i:i + per_pass].copy(), device=dev))
              for i in range(0, Bs, per_pass)]
    all_slots = torch.as_tensor(seq_slot, device=dev)

    steps = serving_schedule(rng, Bs, x["decode_tokens"], x["rho"], x["T"])
    sets = [build_inputs(torch, rng, NL, dev) for _ in range(G)]
    cu_d = torch.arange(0, (Bs + 1) * T, T, dtype=torch.int32, device=dev)
    outs = torch.empty(G, NL, Bs * T, H, D, dtype=torch.float32, device=dev)
    live_slots = [torch.as_tensor(seq_slot[live], device=dev) for live, _ in steps]
    accs = [torch.as_tensor(a, device=dev) for _, a in steps]
    stream = torch.cuda.Stream(device=dev)
    graphs = []
    with torch.cuda.stream(stream):
        for s, (live, _) in enumerate(steps):
            n = len(live)
            g = torch.cuda.CUDAGraph()
            g.capture_begin()
            for l in range(NL):
                v = sets[s % G][1][l]
                tb = K.TokenBatch(v["q"][:n * T], v["k"][:n * T], v["v"][:n * T],
                                  v["alpha"][:n * T], v["beta"][:n * T],
                                  cu_d[:n + 1], o=outs[s % G, l, :n * T])
                K.kda_verify(tb, T, pools[l], live_slots[s], rings[l],
                             stream=stream)
            K.kda_commit_layers(accs[s], live_slots[s], pools[0], rings,
                                stream=stream)
            g.capture_end()
            graphs.append(g)
    torch.cuda.synchronize()

    def flow():
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        with torch.cuda.stream(stream):
            ev[0].record(stream)
            for l in range(NL):
                for slots_p, ck_p in passes:
                    K.kda_prefill_chunked(ptb, pools[l], slots_p, C, E, ck_p,
                                          workspace=ws, stream=stream)
                K.kda_ring_reset(all_slots, pools[l], rings[l], stream=stream)
            ev[1].record(stream)
            for g in graphs:
                g.replay()
            for l in range(NL):
                K.kda_materialize(all_slots, pools[l], rings[l], stream=stream)
            ev[2].record(stream)
        torch.cuda.synchronize()
        return ev[0].elapsed_time(ev[1]), ev[1].elapsed_time(ev[2])

    K.kda_get_device_error()
    flow()
    prefill_ms, decode_ms = flow()
    bits = K.kda_get_device_error()
    del graphs, ws, pools, rings, sets, outs, pt, ptb
    torch.cuda.empty_cache()
    verified = sum(len(live) for live, _ in steps) * T
    committed = sum(int(a.sum()) for _, a in steps)
    vbytes = serving_verify_bytes(steps) * NL
    return {
        "workload": w.name, "kda_layers": NL,
        "prefill_passes_per_layer": len(passes),
        "prefill_tokens_per_s": Bs * L * NL / (prefill_ms * 1e-3),
        "prefill_ms_per_layer": prefill_ms / NL,
        "decode_steps": len(steps),
        "verified_tokens_per_s": verified * NL / (decode_ms * 1e-3),
        "committed_tokens_per_s": committed * NL / (decode_ms * 1e-3),
        "mean_accepted": committed / sum(len(live) for live, _ in steps),
        "decode_ms_per_layer": decode_ms / NL,
        "kda_layer_ms": (prefill_ms + decode_ms) / NL,
        "decode_verify_alg_gbs": vbytes / (decode_ms * 1e-3) / 1e9,
        "device_error_bits": bits,
        "note": "per-layer figures = totals over the NL layers / NL; the "
                "decode phase's GB/s counts the verify launches' algorithmic "
                "bytes over the whole phase (commit and materialize launches "
                "included in the time)",
    }


def run_tiny(torch, K, dev, reps=50, warmup=5):
    """Latency of the tiny workload (a correctness workload: no roofline).
    One sequence, 2 heads, d = 16, fp32 inputs, state from zero: a 64-token
    prefill (chunk 16, checkpoints after tokens 32 and 64), the ring reset,
    then 8 steps of verify T = 4 + commit with accepted ~ U{0..4}.  Eager
    calls on one stream; CUDA events at the phase boundaries and the host
    wall time of a whole flow (synchronized at its end), over ``reps`` flows
    after ``warmup``."""
    w = ki.TINY
    x = w.extra
    rng = np.random.default_rng(w.seed)
    Hn, d, L, Tn, n = w.num_heads, w.d, x["prefill_len"], x["T"], x["steps"]
    C, E = x["chunk"], x["ckpt_every"]

    def batch(tok):
        t = {k: torch.from_numpy(tok[k]).to(device=dev, dtype=torch.float32)
             for k in ("q", "k", "v", "alpha", "beta")}
        cu = torch.as_tensor(np.asarray(tok["cu_seqlens"], dtype=np.int32),
                             device=dev)
        return K.TokenBatch(t["q"], t["k"], t["v"], t["alpha"], t["beta"], cu)

    prompt = batch(ki.gen_tokens(rng, [L], Hn, d))
    drafts = [batch(ki.gen_tokens(rng, [Tn], Hn, d)) for _ in range(n)]
    acc = [torch.as_tensor(ki.accepted_uniform(rng, 1, Tn), device=dev)
           for _ in range(n)]
    n_ck = L // E
    pool = K.StatePool.zeros(1 + n_ck, Hn, d, device=dev)
    ring = K.ReplayRing(1 + n_ck, Hn, d, Tn, torch.float32, device=dev)
    slots = torch.zeros(1, dtype=torch.int32, device=dev)
    ck = torch.arange(1, 1 + n_ck, dtype=torch.int32, device=dev).view(1, -1)
    ws_bytes = K.kda_prefill_workspace_size(L, 1, Hn, d, d, C, K.KDA_F32)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev) if ws_bytes else None
    stream = torch.cuda.current_stream()

    def flow(ev=None):
        if ev:
            ev[0].record(stream)
        K.kda_prefill_chunked(prompt, pool, slots, C, E, ck, workspace=ws)
        K.kda_ring_reset(slots, pool, ring)
        if ev:
            ev[1].record(stream)
        for s in range(n):
            K.kda_verify(drafts[s], Tn, pool, slots, ring)
            K.kda_commit(acc[s], slots, pool, ring)
        if ev:
            ev[2].record(stream)

    K.kda_get_device_error()
    pre, dec, wall = [], [], []
    for r in range(warmup + reps):
        pool.data.zero_()
        torch.cuda.synchronize()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        t0 = time.perf_counter()
        flow(ev)
        torch.cuda.synchronize()
        if r >= warmup:
            wall.append(time.perf_counter() - t0)
            pre.append(ev[0].elapsed_time(ev[1]))
            dec.append(ev[1].elapsed_time(ev[2]))
    bits = K.kda_get_device_error()
    return {
        "workload": w.name, "reps": reps,
        "prefill_us": float(np.median(pre)) * 1e3,
        "verify_commit_us_per_step": float(np.median(dec)) * 1e3 / n,
        "flow_wall_us": float(np.median(wall)) * 1e6,
        "device_error_bits": bits,
        "note": "medians; device times from CUDA events around the eager "
                "calls (prefill + ring reset; the 8 verify + commit steps), "
                "wall time of the whole flow on the host including the "
                "binding's call overhead; launch-bound at this size",
    }


def run_kda(args, rank, world, local_rank):
    import torch
    from recurrent_kda_state_gb300 import kda as K
    from recurrent_kda_state_gb300._build import build_library
    build_library()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 126 * 2 ** 20))
    touched = B * H * D * D * 4
    NL = max(1, math.ceil(4 * l2 / touched))
    rng = replica_rng(rank)
    slots_np = ki.slot_table(rng, B, P)
    slots = torch.as_tensor(slots_np, device=dev)
    pools = [K.StatePool.zeros(P, H, D, device=dev) for _ in range(NL)]
    rings = [K.ReplayRing(P, H, D, DEPTH, torch.bfloat16, device=dev)
             for _ in range(NL)]
    G = 4
    sets = [build_inputs(torch, rng, NL, dev) for _ in range(G)]
    N = B * T
    cu = torch.arange(0, (B + 1) * T, T, dtype=torch.int32, device=dev)
    outs = torch.empty(G, NL, N, H, D, dtype=torch.float32, device=dev)
    batches = [[K.TokenBatch(v["q"], v["k"], v["v"], v["alpha"], v["beta"], cu,
                             o=outs[g, l]) for l, v in enumerate(sets[g][1])]
               for g in range(G)]
    A = 256
    acc_np = ki.accepted_uniform(rng, A * B, T).reshape(A, B)
    acc = torch.as_tensor(acc_np, device=dev)

    stream = torch.cuda.Stream(device=dev)
    total_steps = args.warmup + args.steps
    graphs, events = [], []
    K.kda_get_device_error()
    with torch.cuda.stream(stream):
        for s in range(total_steps):
            g = torch.cuda.CUDAGraph()
            # one event pair around the step's NL verify launches: a pair
            # around every launch delays each launch by several microseconds
            evs = (torch.cuda.Event(enable_timing=True, external=True),
                   torch.cuda.Event(enable_timing=True, external=True)) \
                if s >= args.warmup else None
            g.capture_begin()
            if evs:
                evs[0].record(stream)
            for l in range(NL):
                K.kda_verify(batches[s % G][l], T, pools[l], slots, rings[l],
                             stream=stream)
            if evs:
                evs[1].record(stream)
            # the sampler's accepted lengths, recorded in every layer's ring
            K.kda_commit_layers(acc[s % A], slots, pools[0], rings, stream=stream)
            g.capture_end()
            graphs.append(g)
            events.append(evs)
    torch.cuda.synchronize()
    dist = None
    if world > 1:
        import torch.distributed as dist

    def barrier():
        if dist is not None:
            dist.barrier()

    # warm-up
    with torch.cuda.stream(stream):
        for s in range(args.warmup):
            graphs[s].replay()
    torch.cuda.synchronize()
    clocks = ClockSampler(local_rank)
    clocks.start()
    time.sleep(0.3)
    barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    w0 = time.time()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for s in range(args.warmup, total_steps):
            graphs[s].replay()
        e1.record(stream)
    torch.cuda.synchronize()
    w1 = time.time()
    barrier()
    clocks.stop()
    ms = max_over_ranks(e0.elapsed_time(e1), dist, dev)
    bits = K.kda_get_device_error()
    # average verify launch duration over the timed region: each step's block
    # of NL back-to-back launches / NL (the gaps between launches included)
    durs, abytes = [], []
    for s in range(args.warmup, total_steps):
        a_prev = acc_np[(s - 1) % A]
        abytes.append(float(sum(unit_bytes(int(x)) for x in a_prev) * H))
        ev0, ev1 = events[s]
        durs.append(ev0.elapsed_time(ev1) / NL)
    mean_dur_s = float(np.mean(durs)) * 1e-3
    achieved = float(np.mean(abytes)) / mean_dur_s / 1e9
    peak, peak_kind = load_peaks()
    tokens_rank = B * T * args.steps * NL
    value = job_rate(tokens_rank, world, ms)

    # end to end: inputs from pinned host memory, outputs back, same graphs
    host_in = [sets[g][0].cpu().pin_memory() for g in range(G)]
    host_acc = acc.cpu().pin_memory()
    host_out = torch.empty(outs.shape[1:], dtype=torch.float32).pin_memory()
    h2d = sets[0][0].numel() * 2 + B * 4
    d2h = host_out.numel() * 4
    # Pipelined as a serving loop would run it: one stream copies step s+1's
    # inputs in while step s computes, another reads step s's outputs back;
    # events keep each of the G input sets and output buffers from being
    # overwritten while in use.  Every step's copies are in the timed region.
    h2d_s = torch.cuda.Stream(device=dev)
    d2h_s = torch.cuda.Stream(device=dev)
    first = args.warmup
    ev_in, ev_cmp, ev_out = {}, {}, {}

    def issue_h2d(s):
        with torch.cuda.stream(h2d_s):
            if s - G >= first:
                h2d_s.wait_event(ev_cmp[s - G])   # input set s % G is free
            sets[s % G][0].copy_(host_in[s % G], non_blocking=True)
            acc[s % A].copy_(host_acc[s % A], non_blocking=True)
            ev_in[s] = torch.cuda.Event()
            ev_in[s].record(h2d_s)

    barrier()
    torch.cuda.synchronize()
    f0 = torch.cuda.Event(enable_timing=True)
    f1 = torch.cuda.Event(enable_timing=True)
    f0.record(h2d_s)
    issue_h2d(first)
    for s in range(first, total_steps):
        if s + 1 < total_steps:
            issue_h2d(s + 1)
        stream.wait_event(ev_in[s])
        if s - G >= first:
            stream.wait_event(ev_out[s - G])      # output buffer s % G read back
        with torch.cuda.stream(stream):
            graphs[s].replay()
        ev_cmp[s] = torch.cuda.Event()
        ev_cmp[s].record(stream)
        with torch.cuda.stream(d2h_s):
            d2h_s.wait_event(ev_cmp[s])
            host_out.copy_(outs[s % G], non_blocking=True)
            ev_out[s] = torch.cuda.Event()
            ev_out[s].record(d2h_s)
    f1.record(d2h_s)
    torch.cuda.synchronize()
    ms_e2e = max_over_ranks(f0.elapsed_time(f1), dist, dev)
    # the graphs' timing events were recorded again by this pass: the verify
    # launches' duration while the copies ran beside them
    e2e_launch_us = float(np.mean([events[s][0].elapsed_time(events[s][1]) / NL
                                   for s in range(args.warmup, total_steps)])) * 1e3

    # The same end-to-end loop through the public calls themselves: every step
    # issues kda_verify for each layer and kda_commit_layers eagerly through
    # the binding (argument marshalling, host validation and the launch on
    # every call), with the same pipelined host copies.
    ev_in, ev_cmp, ev_out = {}, {}, {}
    barrier()
    torch.cuda.synchronize()
    a0 = torch.cuda.Event(enable_timing=True)
    a1 = torch.cuda.Event(enable_timing=True)
    aw0 = time.time()
    a0.record(h2d_s)
    issue_h2d(first)
    for s in range(first, total_steps):
        if s + 1 < total_steps:
            issue_h2d(s + 1)
        stream.wait_event(ev_in[s])
        if s - G >= first:
            stream.wait_event(ev_out[s - G])
        for l in range(NL):
            K.kda_verify(batches[s % G][l], T, pools[l], slots, rings[l], stream=stream)
        K.kda_commit_layers(acc[s % A], slots, pools[0], rings, stream=stream)
        ev_cmp[s] = torch.cuda.Event()
        ev_cmp[s].record(stream)
        with torch.cuda.stream(d2h_s):
            d2h_s.wait_event(ev_cmp[s])
            host_out.copy_(outs[s % G], non_blocking=True)
            ev_out[s] = torch.cuda.Event()
            ev_out[s].record(d2h_s)
    a1.record(d2h_s)
    torch.cuda.synchronize()
    aw1 = time.time()
    ms_api = max_over_ranks(a0.elapsed_time(a1), dist, dev)

    prefill = run_prefill(torch, K, dev)
    mixed = run_mixed(torch, K, dev)
    direct = run_snapshot_ablation(torch, K, dev, NL, slots, batches, acc, acc_np,
                                   G, A)
    raw_verify = run_verify_raw(torch, K, dev, NL, slots, acc, A)
    serving = run_serving(torch, K, dev, NL)
    tiny = run_tiny(torch, K, dev)
    cache = state_cache_bytes()
    budget = CACHE_BUDGET_GIB * 2 ** 30
    replay_step_bytes = float(np.mean(abytes)) + B * H * 8
    direct.update({
        "replay_alg_bytes_per_layer_step": replay_step_bytes,
        "replay_ms_per_step": ms / args.steps,
        "replay_speedup": direct["ms_per_step"] / (ms / args.steps),
        "state_cache_bytes_per_seq_layer": cache,
        "seqs_per_layer_at_budget": {k: int(budget // v) for k, v in cache.items()},
        "cache_budget_gib": CACHE_BUDGET_GIB,
    })
    cpu = None
    if rank == 0:
        rate, cores, desc, _ = oracle_spec_rate(args.cpu_seconds)
        cpu = {"value": rate, "unit": "tokens/s", "cores": cores,
               "kind": "oracle", "sample": desc}
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {
            "workload": ki.SPEC.name, "num_seqs": B, "heads": H, "d": D,
            "T": T, "ring_depth": DEPTH, "slots": P, "kda_layers": NL,
            "inputs": "bf16 q/k/v/alpha/beta, fp32 state and outputs",
            "value_def": "verified draft tokens per second per KDA layer "
                         "(B*T*layers*steps/time)",
            "l2": "inputs larger than L2: %d layer state pools touched per "
                  "step = %.0f MiB vs L2 %.0f MiB" % (
                      NL, NL * touched / 2 ** 20, l2 / 2 ** 20),
            "parallelism": "replicas" if world > 1 else "single GPU",
        },
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak,
                     "unit": "GB/s", "frac": achieved / peak,
                     "traffic": ncu_traffic(), "kernel": "verify_pipe_kernel (d=128, bf16)",
                     "peak_source": peak_kind,
                     "mean_launch_us": mean_dur_s * 1e6,
                     "launch_timing": "one CUDA event pair around each step's "
                                      "%d back-to-back verify launches, / %d" % (NL, NL),
                     "alg_bytes_per_launch": float(np.mean(abytes))},
        "cpu_baseline": cpu,
        "e2e": {"value": job_rate(tokens_rank, world, ms_api), "unit": "tokens/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "ms_per_step": ms_api / args.steps,
                "host_wall_ms_per_step": (aw1 - aw0) * 1e3 / args.steps,
                "calls": "eager kda_verify x %d + kda_commit_layers per step "
                         "through the binding, host copies in the timed region" % NL},
        "gpu_launches": (NL + 1) * args.steps,
        "clocks": clocks.summary(w0, w1),
        "device_error_bits": bits,
        "prefill": prefill,
        "e2e_graph": {"value": job_rate(tokens_rank, world, ms_e2e), "unit": "tokens/s",
                      "ms_per_step": ms_e2e / args.steps,
                      "verify_launch_us_during_copies": e2e_launch_us,
                      "calls": "the same steps replayed as CUDA graphs captured from the calls"},
        "mixed": mixed,
        "serving": serving,
        "tiny": tiny,
        "ablation_direct_snapshots": direct,
        "verify_raw_inputs": raw_verify,
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    run_kda(args, rank, world, local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

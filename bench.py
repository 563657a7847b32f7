#!/usr/bin/env python3
"""Benchmark of the GDN state-scan hot path on GB300.

One step = one pass of the whole path over one batch of the 8 x 16-head,
N = 8192, bf16 prefill workload:
  1. gdn_prefill_ckpt     : scan with bf16 readout and 16 equally spaced fp32
                            checkpoints per sequence (index plan on the host);
  2. gdn_resume_from_ckpt : 16 resume probes (sequence ~ U, depth ~ U[1, N])
                            recomputing c_j+1..d with readout;
  3. gdn_tail_replay      : Tail-Replay at m = N with r = 5 % (k = 410) from
                            a zero state.
value = whole-job tok*head per second over all ranks, device-timed with
inputs resident in HBM; e2e = the same step through the Python/C API with
pinned host inputs copied in and every result copied out each step.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

For N > 1 run under torchrun: every rank scans its own batch (weak scaling,
no collective on the data path; the barrier and a max-reduction of the
elapsed time are the only cross-rank calls).
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time
from typing import Optional

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import synth  # noqa: E402

METRIC = "GDN scan Mtok·head/s (prefill+ckpt, resume, tail replay)"
UNIT = "Mtok·head/s"
WORKLOAD = "prefill"
N_PROBES = 16
REPLAY_R = (1, 20)
FP32_LANES_PER_SM = 128
SM_COUNT = 152
SM_MAX_MHZ = 2070.0
PEAK_ALU_TFLOPS = SM_COUNT * FP32_LANES_PER_SM * 2 * SM_MAX_MHZ * 1e6 / 1e12  # 80.54
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "gdn_chunk_tc_kernel_step_8x16x8192.md")
# the kernel and the host code that splits the step into its launches: the committed DRAM traffic holds for both
KERNEL_SRC = [os.path.join(ROOT, "hybrid_model_recurrent_gb300", "csrc", n) for n in ("gdn_chunk_tc.cuh", "gdn_api.cu")]
# tcgen05.mma MACs per 64-token chunk and head in the chunked kernel: 76 MMAs of 128x64x16
# ([K;Q] K^T 8, W^T and U~^T 16, S_0 (-W)^T and S_0 Q^T 40, U''^T P''^T 12) and 8 of 128x128x16
# (the state update)
CHUNK_MACS = 76 * 128 * 64 * 16 + 8 * 128 * 128 * 16
# without a readout the S_0 Q^T and U''^T P^T products (16 + 12 of 128x64x16) are not issued
CHUNK_MACS_NO_READOUT = CHUNK_MACS - 28 * 128 * 64 * 16


def measured_peaks():
    """(hbm GB/s, bf16 TFLOP/s burst, source) from MEASURED_PEAKS.json, else the fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


# -------------------------------------------------------------------------------------------
# distributed plumbing
# -------------------------------------------------------------------------------------------
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(ws, backend):
    if ws > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group(backend=backend)


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, ws: int, device) -> float:
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, ws: int, device) -> float:
    if ws == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def aggregate(units_per_rank: float, elapsed_s: float, ws: int, device):
    """Whole-job throughput: all ranks' units over the slowest rank's time."""
    total = sum_over_ranks(units_per_rank, ws, device)
    slowest = max_over_ranks(elapsed_s, ws, device)
    return total, slowest, total / slowest


# -------------------------------------------------------------------------------------------
# clocks during the timed region
# -------------------------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = os.path.join("/tmp", f"gdn_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 7:
                    continue
                try:
                    sm.append(float(parts[0]))
                    mx.append(float(parts[1]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[3:7]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# -------------------------------------------------------------------------------------------
# the step
# -------------------------------------------------------------------------------------------
class Step:
    def __init__(self, w: synth.Workload, device, algo: str = "auto"):
        import hybrid_model_recurrent_gb300 as gdn
        self.gdn = gdn
        self.algo = algo
        self.w = w
        self.dev = device
        self.cu = w.cu_seqlens
        self.ck = w.ckpt_positions()
        self.probes = dataclasses.replace(w, n_probes=N_PROBES).probes()
        self.m = list(w.seq_lens)
        T, H, dk, dv, B = w.T, w.H, w.dk, w.dv, w.B
        f32 = torch.float32
        self.inp = synth.make_inputs(w, device=device)
        self.o = torch.empty((T, H, dv), dtype=w.out_dtype, device=device)
        self.S_final = torch.empty((B, H, dv, dk), dtype=f32, device=device)
        n_ck = sum(len(c) for c in self.ck)
        # The checkpoint store, two buffers: a step's prefill writes one while its resumes read the other,
        # written by the step before (as a serving step resumes requests from checkpoints stored earlier;
        # every step processes the same batch, so both buffers end up holding the same states).
        self.ck_store = [torch.empty((n_ck, H, dv, dk), dtype=f32, device=device) for _ in range(2)]
        self.n_runs = 0
        self.ckpt = self.ck_store[0]
        self.chosen = []
        self.resume_lens = []
        for s, d in self.probes:
            j = gdn.gdn_select_ckpt(self.ck[s], d)
            self.resume_lens.append(d - (0 if j < 0 else self.ck[s][j]))
        rows = sum(self.resume_lens)
        self.resume_rows = rows
        self.o_res = torch.empty((max(rows, 1), H, dv), dtype=w.out_dtype, device=device)
        self.S_out = torch.empty((len(self.probes), H, dv, dk), dtype=f32, device=device)
        self.S_hat = torch.empty((B, H, dv, dk), dtype=f32, device=device)
        self.replay_tokens = sum(gdn.gdn_replay_plan(m, *REPLAY_R)[1] for m in self.m)
        self.tok_head = {"prefill": T * H, "resume": rows * H, "replay": self.replay_tokens * H}
        self.ws = gdn.workspace(device)
        # gdn_step splits the step into two launches side by side: the prefill jobs (128 CTAs) and the resume and
        # replay jobs (at most a quarter of their length) on the remaining SMs
        self.launches_per_step = 2
        self.ev = None
        # the store the first step's resumes read (untimed)
        gdn.gdn_prefill_ckpt(self.inp.q, self.inp.k, self.inp.v, self.inp.alpha, self.inp.beta, self.cu,
                             ckpt_pos=self.ck, o=self.o, S_final=self.S_final, ckpt_states=self.ck_store[1],
                             ws=self.ws, algo=algo)

    def units(self) -> int:
        return sum(self.tok_head.values())

    def run(self, inp=None, record=None):
        """The step: the batch's prefill (readout + checkpoints), the resume probes (from the checkpoint
        store of the step before) and the tail replays: one gdn_step call (two launches side by side)."""
        g = self.gdn
        inp = inp or self.inp
        s = torch.cuda.current_stream(self.dev)
        write, read = self.ck_store[self.n_runs & 1], self.ck_store[(self.n_runs + 1) & 1]
        self.n_runs += 1
        self.ckpt = write
        if record is not None:
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(s)
        g.gdn_step(inp.q, inp.k, inp.v, inp.alpha, inp.beta, self.cu, ws=self.ws,
                   prefill=dict(ckpt_pos=self.ck, o=self.o, S_final=self.S_final, ckpt_states=write),
                   resume=dict(ckpt_states=read, ckpt_pos=self.ck, probes=self.probes, o_out=self.o_res,
                               S_out=self.S_out),
                   replay=dict(m=self.m, r_num=REPLAY_R[0], r_den=REPLAY_R[1], S_hat=self.S_hat), algo=self.algo)
        if record is not None:
            e1.record(s)
            record.append((e0, e1))

    def run_three_calls(self, inp=None):
        """The same step as three launches, one per entry point, each resume reading the checkpoints its own
        step's prefill has just written."""
        g = self.gdn
        inp = inp or self.inp
        g.gdn_prefill_ckpt(inp.q, inp.k, inp.v, inp.alpha, inp.beta, self.cu, ckpt_pos=self.ck, o=self.o,
                           S_final=self.S_final, ckpt_states=self.ckpt, ws=self.ws, algo=self.algo)
        g.gdn_resume_from_ckpt(inp.q, inp.k, inp.v, inp.alpha, inp.beta, self.cu, self.ckpt, self.ck, self.probes,
                               o_out=self.o_res, S_out=self.S_out, ws=self.ws, algo=self.algo)
        g.gdn_tail_replay(None, inp.k, inp.v, inp.alpha, inp.beta, self.cu, self.m, *REPLAY_R, S_hat=self.S_hat,
                          ws=self.ws, algo=self.algo)

    def outputs(self):
        return [self.o, self.S_final, self.ckpt, self.S_out, self.o_res[:self.resume_rows], self.S_hat]


def source_sha256() -> str:
    """sha256 over the kernel source and the launch-splitting host source, in that order."""
    h = hashlib.sha256()
    for path in KERNEL_SRC:
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def profile_traffic():
    """DRAM bytes of the step's launches from the committed ncu summary, only if it was taken on the current
    kernel and launch-splitting source."""
    try:
        with open(PROFILE_SUMMARY) as f:
            text = f.read()
        sha = source_sha256()
    except OSError:
        return None
    vals = {}
    for line in text.splitlines():
        if ":" in line:
            k, v = line.split(":", 1)
            vals[k.strip().strip("`- ")] = v.strip().strip("`")
    if vals.get("kernel_source_sha256") != sha:
        return None
    try:
        return int(vals["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# -------------------------------------------------------------------------------------------
# oracle timing (CPU baseline and the reference arm)
# -------------------------------------------------------------------------------------------
def oracle_jobs(w: synth.Workload, pairs, tokens: int):
    """Oracle jobs for `pairs` (seq, head) streams of `tokens` tokens each: prefill
    with readout and the workload's checkpoints (inputs generated here, untimed)."""
    import oracle
    oracle.build()
    jobs = []
    for b, h in pairs:
        t0 = w.cu_seqlens[b]
        inp = synth.make_inputs(w, t_range=(t0, t0 + tokens), heads=range(h, h + 1))
        ck = [c for c in w.ckpt_positions()[b] if c <= tokens]
        jobs.append(lambda i=inp, ck=ck: oracle.prefill(i.q[:, 0], i.k[:, 0], i.v[:, 0], i.alpha[:, 0],
                                                        i.beta[:, 0], ckpt_pos=ck))
    return jobs


def time_oracle(jobs, threads: int) -> float:
    import oracle
    t = time.perf_counter()
    oracle.run_many(jobs, threads)
    return time.perf_counter() - t


def placement_report(N: int = 8192, M: int = 16, n_requests: int = 10000):
    """Checkpoint placement ("Sparse prefix caching ...", sections 3-5) on the seeded depth
    distributions: expected recompute per request and tokens saved per checkpoint for every
    strategy at the prefill workload's N and M, and the host time of the O(N M) programme at the
    long-prefill size (N = 131072, M = 32)."""
    import hybrid_model_recurrent_gb300 as gdn
    out = {"N": N, "M": M, "requests": n_requests, "unit": "tokens", "distributions": {}}
    for kind in synth.DEPTH_KINDS:
        w = synth.depth_weights(kind, N, n_requests, seed=0)
        tot = sum(w)
        none = gdn.gdn_expected_recompute(w, [])
        row = {"no_cache_per_request": none / tot}
        for strat in ("balanced", "block", "random", "greedy", "dp"):
            _, cost = gdn.gdn_ckpt_placement(w, M, strat, seed=0)
            row[strat] = {"recompute_per_request": cost / tot, "saved_per_checkpoint": (none - cost) / tot / M}
        out["distributions"][kind] = row
    wl = synth.depth_weights("prompts", 131072, 20000, seed=0)
    gdn.gdn_ckpt_placement(wl, 32, "dp")
    reps = 5
    t0 = time.perf_counter()
    for _ in range(reps):
        gdn.gdn_ckpt_placement(wl, 32, "dp")
    out["dp_ms_N131072_M32"] = (time.perf_counter() - t0) / reps * 1e3
    return out


def two_pass_report(step, reps: int = 20):
    """The prefill call of the timed step in both chunked variants, on the step's own inputs: the fused
    tcgen05 scan (the default, 256-byte workspace) and the two-pass scan (chunk schedule and T of every chunk
    first, then the scan; it needs gdn_workspace_size_two_pass bytes).  CUDA events around `reps` back-to-back
    calls, per call."""
    import hybrid_model_recurrent_gb300 as gdn
    w, inp, dev = step.w, step.inp, step.dev
    big = torch.zeros(int(gdn.lib().gdn_workspace_size_two_pass(w.T, w.H, w.B)), dtype=torch.uint8, device=dev)
    out = {}
    for name, algo, ws in (("fused_ms", "chunked", step.ws), ("two_pass_ms", "two_pass", big)):
        def call():
            gdn.gdn_prefill_ckpt(inp.q, inp.k, inp.v, inp.alpha, inp.beta, step.cu, ckpt_pos=step.ck, o=step.o,
                                 S_final=step.S_final, ckpt_states=step.ckpt, ws=ws, algo=algo)
        for _ in range(2):
            call()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            call()
        e1.record()
        torch.cuda.synchronize(dev)
        out[name] = e0.elapsed_time(e1) / reps
    out["two_pass_workspace_bytes"] = int(big.numel())
    out["workload"] = "the timed step's prefill call (8 x 16 heads, N = 8192, 16 checkpoints)"
    return out


def step_forms_report(step, reps: int = 50):
    """The timed step as one gdn_step call against the three entry points one after another: CUDA events around
    `reps` back-to-back steps (the device stays busy, so host time between calls is hidden), per step."""
    dev = step.dev
    out = {}
    for name, fn in (("gdn_step_ms", step.run), ("three_calls_ms", step.run_three_calls)):
        for _ in range(3):
            fn()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize(dev)
        out[name] = e0.elapsed_time(e1) / reps
    out["note"] = ("gdn_step: the prefill's 128 (sequence, head) jobs in one launch on a high-priority stream, the "
                   "resume and replay jobs in a second launch beside it on the other 24 SMs")
    return out


def overlap_report(dev, reps: int = 5):
    """Transfer / replay overlap ("Tail-Replay" notes page, section 2.5) on the 5 % replay workload:
    768 (layer, head) scans, tail k = 1639 of m = 32768, replayed from zero.  The transfer is the
    matched prefix's attention KV of an assumed 3:1 hybrid (8 attention layers, 8 KV heads x 128,
    bf16): 32768 tokens x 8 x 2 x 8 x 128 x 2 B = 1 GiB from pinned host memory.  Times are medians of
    CUDA-event spans on the compute stream."""
    import hybrid_model_recurrent_gb300 as gdn
    k_tail, H = 1639, 768
    w = synth.Workload("replay5-tail", [k_tail], H, 128, 128, torch.bfloat16, torch.bfloat16, 0.97, 1.0,
                       "uniform", seed=0)
    inp = synth.make_inputs(w, device=dev)
    cu, m = w.cu_seqlens, [k_tail]
    kv_bytes = 32768 * 8 * 2 * 8 * 128 * 2
    kv_h = torch.empty(kv_bytes, dtype=torch.uint8).pin_memory()
    kv_d = torch.empty(kv_bytes, dtype=torch.uint8, device=dev)
    comp = torch.cuda.current_stream(dev)
    copy = torch.cuda.Stream(dev)
    S_hat = torch.empty((1, H, 128, 128), dtype=torch.float32, device=dev)
    ws = gdn.workspace(dev)

    def replay():
        gdn.gdn_tail_replay(None, inp.k, inp.v, inp.alpha, inp.beta, cu, m, 1, 1, S_hat=S_hat, ws=ws)

    def transfer():
        kv_d.copy_(kv_h, non_blocking=True)

    def serial():
        transfer()
        replay()

    def overlapped():
        gdn.gdn_tail_replay_overlap(None, inp.k, inp.v, inp.alpha, inp.beta, cu, m, 1, 1, kv_h, kv_d,
                                    copy_stream=copy, S_hat=S_hat, ws=ws)

    def timed(fn):
        fn()
        torch.cuda.synchronize(dev)
        ts = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(comp)
            fn()
            e1.record(comp)
            torch.cuda.synchronize(dev)
            ts.append(e0.elapsed_time(e1))
        return float(np.median(ts))

    t_rep, t_kv, t_ser, t_ovl = timed(replay), timed(transfer), timed(serial), timed(overlapped)
    return {"workload": "768 scans x tail 1639 (5 % of 32768), state only; KV 1 GiB pinned H2D",
            "unit": "ms", "T_replay": t_rep, "T_KV": t_kv, "T_serial": t_ser, "T_overlap": t_ovl,
            "model_max": max(t_rep, t_kv), "model_sum": t_rep + t_kv,
            "kv_GBps": kv_bytes / (t_kv * 1e-3) / 1e9,
            "replay_Mtok_head_per_s": k_tail * H / (t_rep * 1e-3) / 1e6}


def workloads_report(dev, hbm_peak: float, reps: int = 5, only: Optional[str] = None):
    """Every synthetic workload on its own (CUDA events around `reps` back-to-back calls, per call); with `only`,
    that one tail-replay workload alone.
    Throughput in tok*head/s and, against the HBM peak, the algorithmic bytes of the call: per tok*head
    q, k, v + gates + o (1,032 B at bf16 d = 128) with a readout, k, v + gates (520 B) without; 64 KiB per
    state read or written.  The replay workloads are given as their tails alone (the rows the kernel reads:
    a sequence of k_b rows replayed whole), which is the same scan over the same tokens as ceil(r m_b) of a
    prefix of m_b."""
    import hybrid_model_recurrent_gb300 as gdn
    ws = gdn.workspace(dev)
    out = {}

    def timed(fn):
        fn()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / reps

    def row(ms, tok_head, nbytes, states=None):
        r = {"ms": ms, "tok_head": tok_head, "Mtok_head_per_s": tok_head / (ms * 1e-3) / 1e6,
             "algorithmic_bytes": nbytes, "achieved_GBps": nbytes / (ms * 1e-3) / 1e9,
             "hbm_frac": nbytes / (ms * 1e-3) / 1e9 / hbm_peak}
        if states is not None:
            r["states_per_s"] = states / (ms * 1e-3)
        return r

    def per_tok(w, readout):
        es = 2 if w.qkv_dtype == torch.bfloat16 else 4
        eo = 2 if w.out_dtype == torch.bfloat16 else 4
        return (w.dk + w.dv + (w.dk if readout else 0)) * es + 8 + (w.dv * eo if readout else 0)

    if only:
        return {only: replay_rows(gdn, dev, only, ws, timed, row, per_tok)}

    # tiny: prefill (readout, checkpoints every 64), 4 resume probes, tail replay r = 1/20 at m = 256 with twin
    w = synth.workload("tiny")
    x = synth.make_inputs(w, device=dev)
    cu, ck, D = w.cu_seqlens, w.ckpt_positions(), w.dv * w.dk * 4
    r = gdn.gdn_prefill_ckpt(x.q, x.k, x.v, x.alpha, x.beta, cu, ckpt_pos=ck, ws=ws)
    probes = [(0, 100), (0, 191), (0, 200), (0, 256)]
    S_a = torch.zeros((1, w.H, w.dv, w.dk), dtype=torch.float32, device=dev)
    t_pf = timed(lambda: gdn.gdn_prefill_ckpt(x.q, x.k, x.v, x.alpha, x.beta, cu, ckpt_pos=ck, ws=ws))
    t_rs = timed(lambda: gdn.gdn_resume_from_ckpt(x.q, x.k, x.v, x.alpha, x.beta, cu, r["ckpt_states"], ck, probes,
                                                  ws=ws))
    t_rp = timed(lambda: gdn.gdn_tail_replay(None, x.k, x.v, x.alpha, x.beta, cu, [256], 1, 20, S_a=S_a, ws=ws))
    n_rs = sum(d - max([c for c in ck[0] if c <= d], default=0) for _, d in probes)
    out["tiny"] = {"prefill": row(t_pf, 256 * w.H, 256 * w.H * per_tok(w, True) + w.H * 5 * D, 4 * w.H),
                   "resume": row(t_rs, n_rs * w.H, n_rs * w.H * per_tok(w, True) + len(probes) * w.H * 2 * D),
                   "replay_with_twin": row(t_rp, 13 * w.H, 13 * w.H * per_tok(w, False) + w.H * 3 * D),
                   "note": "d = 32 fp32 (per-token kernel); launch-bound"}
    del x, r

    # long prefill: 4 x 32 heads, N = 131072, 32 checkpoints; then the 64 resume probes
    w = synth.workload("long")
    x = synth.make_inputs(w, device=dev)
    cu, ck, D = w.cu_seqlens, w.ckpt_positions(), w.dv * w.dk * 4
    o = torch.empty((w.T, w.H, w.dv), dtype=w.out_dtype, device=dev)
    S_f = torch.empty((w.B, w.H, w.dv, w.dk), dtype=torch.float32, device=dev)
    cks = torch.empty((sum(len(c) for c in ck), w.H, w.dv, w.dk), dtype=torch.float32, device=dev)
    t_pf = timed(lambda: gdn.gdn_prefill_ckpt(x.q, x.k, x.v, x.alpha, x.beta, cu, ckpt_pos=ck, o=o, S_final=S_f,
                                              ckpt_states=cks, ws=ws))
    probes = w.probes()
    n_rs = sum(d - max([c for c in ck[s] if c <= d], default=0) for s, d in probes)
    o_r = torch.empty((max(n_rs, 1), w.H, w.dv), dtype=w.out_dtype, device=dev)
    S_o = torch.empty((len(probes), w.H, w.dv, w.dk), dtype=torch.float32, device=dev)
    t_rs = timed(lambda: gdn.gdn_resume_from_ckpt(x.q, x.k, x.v, x.alpha, x.beta, cu, cks, ck, probes, o_out=o_r,
                                                  S_out=S_o, ws=ws))
    n_ck = cks.shape[0] * w.H
    out["long"] = {"prefill": row(t_pf, w.T * w.H, w.T * w.H * per_tok(w, True) + (n_ck + w.B * w.H) * D, n_ck),
                   "resume": row(t_rs, n_rs * w.H, n_rs * w.H * per_tok(w, True) + len(probes) * w.H * 2 * D),
                   "note": "prefill: 128 (sequence, head) scans of 131072 tokens; resume: 64 probes x 32 heads"}
    del x, o, S_f, cks, o_r, S_o
    torch.cuda.empty_cache()

    # tail replays: replay5 and ragged10, each given as its tails alone
    for name in ("replay5", "ragged10"):
        out[name] = replay_rows(gdn, dev, name, ws, timed, row, per_tok)
    return out


def replay_rows(gdn, dev, name, ws, timed, row, per_tok):
    """Tail replays of one workload: replay5 (768 scans x 1639, 5 % of 32768, with and without the exact twin) or
    ragged10 (32 ragged requests x 16 heads, k_b = ceil(m_b / 10)), given as their tails alone."""
    wf = synth.workload(name)
    rn, rd = wf.replay_r
    tails = [gdn.gdn_replay_plan(m, rn, rd)[1] for m in wf.seq_lens]
    w = synth.Workload(name + "-tails", tails, wf.H, wf.dk, wf.dv, wf.qkv_dtype, wf.out_dtype, wf.alpha_lo,
                       wf.alpha_hi, wf.beta_kind, seed=wf.seed)
    x = synth.make_inputs(w, device=dev, with_q=False)
    cu, D = w.cu_seqlens, w.dv * w.dk * 4
    S_h = torch.empty((w.B, w.H, w.dv, w.dk), dtype=torch.float32, device=dev)
    t = timed(lambda: gdn.gdn_tail_replay(None, x.k, x.v, x.alpha, x.beta, cu, tails, 1, 1, S_hat=S_h, ws=ws))
    rows = {"replay": row(t, w.T * w.H, w.T * w.H * per_tok(w, False) + w.B * w.H * D)}
    if name == "replay5":
        S_a = synth.state(101, w.B * w.H, w.dv, w.dk, 1.0, device=dev).view(w.B, w.H, w.dv, w.dk)
        S_e = torch.empty_like(S_h)
        t2 = timed(lambda: gdn.gdn_tail_replay(None, x.k, x.v, x.alpha, x.beta, cu, tails, 1, 1, S_a=S_a,
                                               S_hat=S_h, S_exact=S_e, ws=ws))
        rows["replay_with_twin"] = row(t2, 2 * w.T * w.H, w.T * w.H * per_tok(w, False) + w.B * w.H * 3 * D)
    rows["note"] = f"{w.B * w.H} scans, {w.T * w.H} tail tok*head"
    del x, S_h
    torch.cuda.empty_cache()
    return rows


def cpu_baseline(w: synth.Workload):
    threads = os.cpu_count() or 1
    pairs = [(b, h) for b in range(w.B) for h in range(w.H)][: 2 * threads]
    dt = time_oracle(oracle_jobs(w, pairs, w.seq_lens[0]), threads)
    units = len(pairs) * w.seq_lens[0]
    return {"value": units / dt / 1e6, "unit": UNIT, "cores": min(threads, len(pairs)), "kind": "oracle",
            "sample": f"fp64 oracle prefill (readout + 16 checkpoints) of {len(pairs)} of the "
                      f"{w.B * w.H} (sequence, head) streams, {w.seq_lens[0]} tokens each "
                      f"({units} tok*head, {dt:.1f} s on {min(threads, len(pairs))} threads)"}


def config_dict(w, ws):
    return {"workload": "prefill+ckpt 8x16 heads, N=8192, dk=dv=128, bf16 q/k/v/o, fp32 state, M=16 ckpts; "
                        f"+{N_PROBES} resume probes; +tail replay r=5% at m=N",
            "seqs_per_rank": w.B, "heads": w.H, "seq_len": w.seq_lens[0], "d_k": w.dk, "d_v": w.dv,
            "ckpts_per_seq": len(w.ckpt_positions()[0]), "resume_probes": N_PROBES,
            "replay_r": f"{REPLAY_R[0]}/{REPLAY_R[1]}", "parallelism": f"dp{ws} (weak: one batch per rank)",
            "step": "one gdn_step call (two launches side by side); the resumes read the checkpoint store written "
                    "by the step before",
            "l2": "inputs larger than L2 (805 MB of bf16 q/k/v streamed per step)", "seed": 0}


def run_reference(args, ws, rank):
    """The reference arm: the fp64 oracle, as it stands, on the host cores."""
    if rank != 0:
        return
    w = synth.workload(WORKLOAD, seed=0)
    threads = os.cpu_count() or 1
    steps, warm = args.steps, args.warmup
    budget_s = 150.0
    rate = 256 / max(time_oracle(oracle_jobs(w, [(0, 0)], 256), 1), 1e-6)  # tok*head/s per thread
    per_step_s = budget_s / max(steps + warm, 1)
    tokens = int(max(32, min(w.seq_lens[0], rate * per_step_s)))
    pairs = [(b % w.B, (b // w.B) % w.H) for b in range(threads)]
    jobs = oracle_jobs(w, pairs, tokens)
    for _ in range(warm):
        time_oracle(jobs, threads)
    dt = sum(time_oracle(jobs, threads) for _ in range(steps))
    units = len(pairs) * tokens * steps
    val = units / dt / 1e6
    line = {"metric": METRIC, "value": val, "unit": UNIT, "n_gpus": args.gpus, "steps": steps, "warmup": warm,
            "ms_per_step": dt / steps * 1e3, "higher_is_better": True, "impl": "reference",
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded generator)",
            "config": config_dict(w, args.gpus),
            "cpu_baseline": {"value": val, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": f"per step: fp64 oracle prefill (readout + checkpoints) of {len(pairs)} "
                                       f"(sequence, head) streams x {tokens} tokens, one per host thread"},
            "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# -------------------------------------------------------------------------------------------
# our arm
# -------------------------------------------------------------------------------------------
def run_ours(args, ws, rank, local):
    import hybrid_model_recurrent_gb300 as gdn
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    init_dist(ws, "nccl")
    gdn.build()
    w = synth.workload(WORKLOAD, seed=rank)
    step = Step(w, dev, args.algo)
    gdn.clear_status(dev)
    for _ in range(max(args.warmup, 3)):
        step.run()
    torch.cuda.synchronize(dev)

    # ---- device-timed region ----
    sampler = ClockSampler(local) if rank == 0 else None
    barrier(ws)
    torch.cuda.synchronize(dev)
    if sampler:
        sampler.start()
        time.sleep(0.3)
    rec = []
    e_start = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)
    e_start.record()
    for _ in range(args.steps):
        step.run(record=rec)
    e_end.record()
    torch.cuda.synchronize(dev)
    barrier(ws)
    clocks = sampler.stop() if sampler else None
    elapsed = e_start.elapsed_time(e_end) / 1e3
    status = gdn.read_status(dev)
    if status != gdn.GDN_OK:
        raise RuntimeError(f"device status {gdn.status_string(status)} during the timed region")
    units = step.units() * args.steps
    total, slowest, thr = aggregate(units, elapsed, ws, dev)
    launch_ms = statistics.mean(a.elapsed_time(b) for a, b in rec)

    # ---- end to end: pinned host inputs in, every result out, each step ----
    host_in = [t.cpu().pin_memory() for t in (step.inp.q, step.inp.k, step.inp.v, step.inp.alpha, step.inp.beta)]
    dev_in = synth.Inputs(*[torch.empty_like(t) for t in (step.inp.q, step.inp.k, step.inp.v, step.inp.alpha,
                                                           step.inp.beta)])
    host_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in step.outputs()]
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out)
    e2e_steps = max(3, min(args.steps, 30))

    def e2e_step():
        for d_, h_ in zip((dev_in.q, dev_in.k, dev_in.v, dev_in.alpha, dev_in.beta), host_in):
            d_.copy_(h_, non_blocking=True)
        step.run(inp=dev_in)
        for h_, d_ in zip(host_out, step.outputs()):
            h_.copy_(d_, non_blocking=True)
        torch.cuda.current_stream(dev).synchronize()

    e2e_step()
    barrier(ws)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    e2e_el = time.perf_counter() - t0
    barrier(ws)
    _, _, e2e_serial_thr = aggregate(step.units() * e2e_steps, e2e_el, ws, dev)

    # The same steps as a serving loop runs them: step i's inputs go in on one stream while step i-1 computes
    # and step i-2's results come out on a third (two sets of device inputs and outputs, one pinned host set
    # each way); every step still copies all of its inputs in and all of its results out.
    step2 = Step(w, dev, args.algo)
    steps = (step, step2)
    fields = lambda x: (x.q, x.k, x.v, x.alpha, x.beta)
    dev_ins = (dev_in, synth.Inputs(*[torch.empty_like(t) for t in fields(dev_in)]))
    s_in, s_cmp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def e2e_pipelined(n):
        in_free, out_free = [None, None], [None, None]
        for i in range(n):
            b = i & 1
            with torch.cuda.stream(s_in):
                if in_free[b] is not None:
                    s_in.wait_event(in_free[b])
                for d_, h_ in zip(fields(dev_ins[b]), host_in):
                    d_.copy_(h_, non_blocking=True)
                ev_in = torch.cuda.Event()
                ev_in.record(s_in)
            with torch.cuda.stream(s_cmp):
                s_cmp.wait_event(ev_in)
                if out_free[b] is not None:
                    s_cmp.wait_event(out_free[b])
                steps[b].run(inp=dev_ins[b])
                ev_c = torch.cuda.Event()
                ev_c.record(s_cmp)
                in_free[b] = ev_c
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_c)
                for h_, d_ in zip(host_out, steps[b].outputs()):
                    h_.copy_(d_, non_blocking=True)
                ev_o = torch.cuda.Event()
                ev_o.record(s_out)
                out_free[b] = ev_o
        for st in (s_in, s_cmp, s_out):
            st.synchronize()

    e2e_pipelined(2)
    # three timed passes, the median reported (a transient on the host link in one pass does not set the figure)
    e2e_runs = []
    for _ in range(3):
        barrier(ws)
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        e2e_pipelined(e2e_steps)
        e2e_el = time.perf_counter() - t0
        barrier(ws)
        e2e_runs.append(aggregate(step.units() * e2e_steps, e2e_el, ws, dev)[2])
    e2e_thr = statistics.median(e2e_runs)

    # The step's one launch: algorithmic bytes and the method's flops of its three kinds of jobs
    # (per tok*head: q, k, v bf16 768 B + alpha, beta 8 B + o bf16 256 B with a readout, k, v and gates 520 B
    # without; states read or written once each, 64 KiB per (range, head)).
    D = w.dv * w.dk
    es = 2
    n_ck = len(step.ck[0])
    pf_th, rs_th, rp_th = step.tok_head["prefill"], step.tok_head["resume"], step.tok_head["replay"]
    bytes_pf = pf_th * ((2 * w.dk + w.dv) * es + 8 + w.dv * es) + w.B * w.H * (n_ck + 1) * D * 4
    bytes_rs = rs_th * ((2 * w.dk + w.dv) * es + 8 + w.dv * es) + len(step.probes) * w.H * 2 * D * 4
    bytes_rp = rp_th * ((w.dk + w.dv) * es + 8) + w.B * w.H * D * 4
    bytes_per_launch = bytes_pf + bytes_rs + bytes_rp
    flops_per_launch = 6 * D * (pf_th + rs_th) + 4 * D * rp_th   # 3 (2 without a readout) FMAs per element
    launch_s = launch_ms * 1e-3
    achieved_gbs = bytes_per_launch / launch_s / 1e9
    hbm_peak, bf16_peak, peak_src = measured_peaks()
    ch = lambda n: (n + 63) // 64
    chunks_rd = w.B * w.H * ch(w.seq_lens[0]) + w.H * sum(ch(n) for n in step.resume_lens)
    chunks_nr = w.H * sum(ch(gdn.gdn_replay_plan(m, *REPLAY_R)[1]) for m in step.m)
    mma_flops = 2 * (chunks_rd * CHUNK_MACS + chunks_nr * CHUNK_MACS_NO_READOUT)
    base = cpu_baseline(w) if (rank == 0 and ws == 1 and not args.no_cpu_baseline) else None
    if rank == 0:
        line = {
            "metric": METRIC, "value": thr / 1e6, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": max(args.warmup, 3), "ms_per_step": slowest / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32 (bf16 q/k/v/o)",
            "data": "synthetic (seeded counter-based generator)",
            "config": dict(config_dict(w, ws), **({} if args.algo == "auto" else {"algo": args.algo})),
            "e2e": {"value": e2e_thr / 1e6, "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "pipelined": "step i+1's inputs in and step i-1's results out overlap step i (3 streams)",
                    "serial_value": e2e_serial_thr / 1e6,
                    "passes": [v / 1e6 for v in e2e_runs], "value_is": "median of the three timed passes",
                    "steps": e2e_steps},
            "gpu_launches": step.launches_per_step * args.steps,
            "roofline": {"bound": "hbm",
                         "kernel": ("gdn_chunk_tc_kernel<bf16 out, readout>" if args.algo in ("auto", "chunked")
                                    else f"the {args.algo} path") +
                                   ": the step's two launches side by side (the prefill jobs; the resume and "
                                   "tail-replay jobs), bytes of both over the step's span",
                         "achieved": achieved_gbs, "peak": hbm_peak, "unit": "GB/s",
                         "frac": achieved_gbs / hbm_peak,
                         "traffic": profile_traffic() if args.algo in ("auto", "chunked") else None,
                         "launch_ms": launch_ms, "algorithmic_bytes_per_launch": bytes_per_launch,
                         "launch_ms_is": "CUDA-event span of the gdn_step call on the step's stream (both launches)",
                         "algorithmic_bytes": {"prefill": bytes_pf, "resume": bytes_rs, "replay": bytes_rp,
                                               "per_tok_head": "1032 with a readout, 520 without; + 64 KiB per "
                                                               "state read or written"},
                         "peak_source": f"hbm_gbs of MEASURED_PEAKS.json ({peak_src})",
                         "tensor_view": {"executed_mma_tflops": mma_flops / launch_s / 1e12,
                                         "peak_bf16_tflops": bf16_peak,
                                         "frac": mma_flops / launch_s / 1e12 / bf16_peak},
                         "fp32_alu_equivalent": {
                             "algorithmic_tflops": flops_per_launch / launch_s / 1e12,
                             "peak_tflops": PEAK_ALU_TFLOPS,
                             "frac": flops_per_launch / launch_s / 1e12 / PEAK_ALU_TFLOPS,
                             "peak_source": "152 SMs x 128 FP32 lanes x 2 flop x 2070 MHz"}},
            "phases": {k: v for k, v in step.tok_head.items()},
            "states_per_s": sum(len(c) for c in step.ck) * w.H * args.steps / slowest,
            "cpu_baseline": base,
            "placement": None if args.step_only else placement_report(),
            "replay_overlap": None if args.step_only else overlap_report(dev),
            "chunked_variants": None if args.step_only else two_pass_report(step),
            "step_forms": step_forms_report(step),
            "workloads": None if args.step_only else workloads_report(dev, hbm_peak),
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--algo", choices=["auto", "chunked", "two_pass", "per_token"], default="auto",
                    help="kernel the step's calls ask for (default: the library's choice, the tcgen05 chunked scan); "
                         "the others are for profiling those kernels on the same step")
    ap.add_argument("--step-only", action="store_true",
                    help="time the step (and its three-call form) only: no placement, overlap, chunked-variant or "
                         "other-workload reports (a few GB on the device, for profiler captures)")
    ap.add_argument("--only-workload", choices=["replay5", "ragged10"],
                    help="time that tail-replay workload alone and print its figures (for profiler captures)")
    args = ap.parse_args()
    if args.only_workload:
        import hybrid_model_recurrent_gb300 as gdn
        dev = torch.device("cuda", 0)
        gdn.build()
        print(json.dumps(workloads_report(dev, measured_peaks()[0], only=args.only_workload)), flush=True)
        return
    ws, rank, local = dist_env()
    if args.impl == "reference":
        run_reference(args, ws, rank)
        return
    run_ours(args, ws, rank, local)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

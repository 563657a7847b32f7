"""Seeded synthetic inputs for the Gated DeltaNet scan workloads.

Harness code shared by the oracle tests and by the CUDA path's tests and
benchmarks.  It draws inputs only and holds none of the recurrence's
arithmetic.  Every value is a pure function of (seed, stream, element index)
(see ``synth_gen.h``), so any slice of a stream -- one head, the tail of a
prefix, one probe -- regenerates bit-identically on the host or on the GPU.

Workload presets mirror the five shapes of the pages' settings: a tiny case,
prefill with sparse checkpoints (8K prefixes), Tail-Replay at 5 % of a 32K
matched prefix, ragged Tail-Replay at 10 %, and a 128K long prefill with
resume probes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from dataclasses import dataclass, field
from typing import List, Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libsynth.so")
_lock = threading.Lock()
_lib = None

STREAM_Q, STREAM_K, STREAM_V, STREAM_ALPHA, STREAM_BETA, STREAM_STATE, STREAM_AUX = 1, 2, 3, 4, 5, 6, 7
F32, BF16 = 0, 1


def build(force: bool = False) -> str:
    """Compile libsynth.so (host + sm_103a) next to this file."""
    src = os.path.join(_HERE, "synth_lib.cu")
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= max(os.path.getmtime(src),
                                                   os.path.getmtime(os.path.join(_HERE, "synth_gen.h")))):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
           "-Xcompiler", "-fPIC,-ffp-contract=off", "-fmad=false", "-shared", "-o", tmp, src]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            i32, i64, u32, u64, vp, dbl = (ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32,
                                           ctypes.c_uint64, ctypes.c_void_p, ctypes.c_double)
            lib.syn_fill_rows_host.argtypes = [vp, ctypes.c_int, u64, u32, i64, i64, i32, i32, i32, i32, ctypes.c_int]
            lib.syn_fill_rows_dev.argtypes = [vp, ctypes.c_int, u64, u32, i64, i64, i32, i32, i32, i32, ctypes.c_int, vp]
            lib.syn_fill_normal_host.argtypes = [vp, u64, u32, u64, i64, dbl]
            lib.syn_fill_normal_dev.argtypes = [vp, u64, u32, u64, i64, dbl, vp]
            lib.syn_fill_gates_host.argtypes = [vp, vp, u64, i64, i64, i32, i32, i32, dbl, dbl, ctypes.c_int]
            lib.syn_fill_int_host.argtypes = [vp, u64, u32, u64, i64, i64, i64]
            for f in ("syn_fill_rows_host", "syn_fill_rows_dev", "syn_fill_normal_host", "syn_fill_normal_dev",
                      "syn_fill_gates_host", "syn_fill_int_host"):
                getattr(lib, f).restype = ctypes.c_int
            _lib = lib
    return _lib


def _stream_ptr(device: torch.device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def rows(seed: int, stream: int, t0: int, t1: int, H: int, d: int, dtype: torch.dtype,
         normalize: bool, device="cpu", heads: Optional[range] = None) -> torch.Tensor:
    """Rows of a [T, H, d] stream for t in [t0, t1) and the given head range.

    ``normalize`` draws unit-norm rows (q, k: L2-normalised in fp64, rounded
    once to fp32 then to bf16); otherwise raw unit-variance draws (v)."""
    lib = _load()
    h0, h1 = (0, H) if heads is None else (heads.start, heads.stop)
    device = torch.device(device)
    code = F32 if dtype == torch.float32 else BF16
    if dtype not in (torch.float32, torch.bfloat16):
        raise ValueError("dtype must be float32 or bfloat16")
    out = torch.empty((t1 - t0, h1 - h0, d), dtype=dtype, device=device)
    if device.type == "cuda":
        rc = lib.syn_fill_rows_dev(ctypes.c_void_p(out.data_ptr()), code, seed, stream, t0, t1, H, h0, h1, d,
                                   int(normalize), _stream_ptr(device))
    else:
        rc = lib.syn_fill_rows_host(ctypes.c_void_p(out.data_ptr()), code, seed, stream, t0, t1, H, h0, h1, d,
                                    int(normalize))
    if rc != 0:
        raise RuntimeError(f"synth rows failed rc={rc}")
    return out


def rows_into(out: torch.Tensor, seed: int, stream: int, t0: int, t1: int, H: int, d: int,
              normalize: bool) -> None:
    """Fill ``out`` (a contiguous [t1-t0, H, d] view, any device) in place."""
    lib = _load()
    assert out.is_contiguous() and tuple(out.shape) == (t1 - t0, H, d)
    code = F32 if out.dtype == torch.float32 else BF16
    if out.device.type == "cuda":
        rc = lib.syn_fill_rows_dev(ctypes.c_void_p(out.data_ptr()), code, seed, stream, t0, t1, H, 0, H, d,
                                   int(normalize), _stream_ptr(out.device))
    else:
        rc = lib.syn_fill_rows_host(ctypes.c_void_p(out.data_ptr()), code, seed, stream, t0, t1, H, 0, H, d,
                                    int(normalize))
    if rc != 0:
        raise RuntimeError(f"synth rows_into failed rc={rc}")


def normal(seed: int, stream: int, idx0: int, shape, scale: float = 1.0, device="cpu") -> torch.Tensor:
    """fp32 tensor of ``scale`` * unit-variance draws, element i has index idx0 + i."""
    lib = _load()
    device = torch.device(device)
    out = torch.empty(shape, dtype=torch.float32, device=device)
    n = out.numel()
    if device.type == "cuda":
        rc = lib.syn_fill_normal_dev(ctypes.c_void_p(out.data_ptr()), seed, stream, idx0, n, scale,
                                     _stream_ptr(device))
    else:
        rc = lib.syn_fill_normal_host(ctypes.c_void_p(out.data_ptr()), seed, stream, idx0, n, scale)
    if rc != 0:
        raise RuntimeError(f"synth normal failed rc={rc}")
    return out


def gates(seed: int, t0: int, t1: int, H: int, alpha_lo: float, alpha_hi: float, beta_kind: str,
          heads: Optional[range] = None):
    """(alpha, beta) fp32 [t1-t0, nheads] on the host.

    alpha ~ U[alpha_lo, alpha_hi]; beta_kind 'uniform' -> U[0,1),
    'sigmoid' -> sigmoid of a unit-variance draw."""
    lib = _load()
    h0, h1 = (0, H) if heads is None else (heads.start, heads.stop)
    a = torch.empty((t1 - t0, h1 - h0), dtype=torch.float32)
    b = torch.empty((t1 - t0, h1 - h0), dtype=torch.float32)
    kind = {"uniform": 0, "sigmoid": 1}[beta_kind]
    rc = lib.syn_fill_gates_host(ctypes.c_void_p(a.data_ptr()), ctypes.c_void_p(b.data_ptr()), seed, t0, t1, H,
                                 h0, h1, alpha_lo, alpha_hi, kind)
    if rc != 0:
        raise RuntimeError(f"synth gates failed rc={rc}")
    return a, b


def integers(seed: int, stream: int, idx0: int, n: int, lo: int, hi: int) -> List[int]:
    """n integers uniform on [lo, hi] (inclusive)."""
    lib = _load()
    out = torch.empty((n,), dtype=torch.int64)
    rc = lib.syn_fill_int_host(ctypes.c_void_p(out.data_ptr()), seed, stream, idx0, n, lo, hi)
    if rc != 0:
        raise RuntimeError(f"synth integers failed rc={rc}")
    return [int(x) for x in out.tolist()]


# --------------------------------------------------------------------------------------------
# workload presets
# --------------------------------------------------------------------------------------------

@dataclass
class Workload:
    """Shape and distribution recipe of one synthetic workload."""
    name: str
    seq_lens: List[int]            # N_b (prefill) or matched prefix m_b (replay)
    H: int
    dk: int
    dv: int
    qkv_dtype: torch.dtype
    out_dtype: torch.dtype
    alpha_lo: float
    alpha_hi: float
    beta_kind: str
    ckpt_every: Optional[int] = None       # equally spaced checkpoints c_i = i * every
    replay_r: Optional[tuple] = None       # (r_num, r_den)
    n_probes: int = 0                      # resume probes (seq ~ U, depth ~ U[1, N])
    seed: int = 0

    @property
    def B(self) -> int:
        return len(self.seq_lens)

    @property
    def cu_seqlens(self) -> List[int]:
        cu = [0]
        for n in self.seq_lens:
            cu.append(cu[-1] + n)
        return cu

    @property
    def T(self) -> int:
        return sum(self.seq_lens)

    def ckpt_positions(self) -> List[List[int]]:
        if not self.ckpt_every:
            return [[] for _ in self.seq_lens]
        return [list(range(self.ckpt_every, n + 1, self.ckpt_every)) for n in self.seq_lens]

    def probes(self):
        """(seq, depth) pairs for resume probes: seq ~ U{0..B-1}, depth ~ U{1..N_seq}."""
        if self.n_probes == 0:
            return []
        seqs = integers(self.seed, STREAM_AUX, 1 << 20, self.n_probes, 0, self.B - 1)
        out = []
        for i, s in enumerate(seqs):
            d = integers(self.seed, STREAM_AUX, (1 << 21) + i, 1, 1, self.seq_lens[s])[0]
            out.append((s, d))
        return out


def _ragged_lengths(seed: int, n: int, lo: int, hi: int) -> List[int]:
    return integers(seed, STREAM_AUX, 0, n, lo, hi)


def workload(name: str, seed: int = 0) -> Workload:
    """The five synthetic workloads, by name: tiny, prefill, replay5, ragged10, long."""
    if name == "tiny":
        return Workload("tiny", [256], 2, 32, 32, torch.float32, torch.float32, 0.9, 1.0, "uniform",
                        ckpt_every=64, replay_r=(1, 20), seed=seed)
    if name == "prefill":
        return Workload("prefill", [8192] * 8, 16, 128, 128, torch.bfloat16, torch.bfloat16, 0.95, 1.0,
                        "sigmoid", ckpt_every=512, seed=seed)
    if name == "replay5":
        return Workload("replay5", [32768], 24 * 32, 128, 128, torch.bfloat16, torch.bfloat16, 0.97, 1.0,
                        "uniform", replay_r=(1, 20), seed=seed)
    if name == "ragged10":
        return Workload("ragged10", _ragged_lengths(seed, 32, 4096, 32768), 16, 128, 128, torch.bfloat16,
                        torch.bfloat16, 0.97, 1.0, "uniform", replay_r=(1, 10), seed=seed)
    if name == "long":
        return Workload("long", [131072] * 4, 32, 128, 128, torch.bfloat16, torch.bfloat16, 0.98, 1.0,
                        "uniform", ckpt_every=4096, n_probes=64, seed=seed)
    raise KeyError(name)


WORKLOADS = ("tiny", "prefill", "replay5", "ragged10", "long")


@dataclass
class Inputs:
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    alpha: torch.Tensor
    beta: torch.Tensor


def make_inputs(w: Workload, device="cpu", t_range: Optional[tuple] = None,
                heads: Optional[range] = None, with_q: bool = True) -> Inputs:
    """Streams [T, H, d] for the token rows t_range=(t0, t1) (default: all)."""
    t0, t1 = t_range if t_range is not None else (0, w.T)
    device = torch.device(device)
    q = rows(w.seed, STREAM_Q, t0, t1, w.H, w.dk, w.qkv_dtype, True, device, heads) if with_q else None
    k = rows(w.seed, STREAM_K, t0, t1, w.H, w.dk, w.qkv_dtype, True, device, heads)
    v = rows(w.seed, STREAM_V, t0, t1, w.H, w.dv, w.qkv_dtype, False, device, heads)
    a, b = gates(w.seed, t0, t1, w.H, w.alpha_lo, w.alpha_hi, w.beta_kind, heads)
    return Inputs(q, k, v, a.to(device), b.to(device))


def state(seed: int, n: int, dv: int, dk: int, scale: float = 1.0, device="cpu", salt: int = 0) -> torch.Tensor:
    """Seeded fp32 states [n, dv, dk] (an arbitrary initial / cached state)."""
    return normal(seed, STREAM_STATE, salt * (1 << 40), (n, dv, dk), scale, device)


# --------------------------------------------------------------------------------------------
# overlap-depth distributions for checkpoint placement
# --------------------------------------------------------------------------------------------
DEPTH_KINDS = ("uniform", "prompts", "documents")


def depth_weights(kind: str, N: int, n_requests: int, seed: int = 0) -> List[int]:
    """Integer weights w[0..N]: counts of `n_requests` seeded overlap depths d in [0, N].

    Stand-ins for the pages' measured overlap distributions (document QA and shared system
    prompts, whose data is not available here):
      uniform   - d ~ U{1..N};
      prompts   - three requests in four reuse one of 8 shared prompt lengths (lengths ~ U{1..N},
                  request's prompt ~ U{0..7}); the rest d ~ U{0..N} (0: no overlap at all);
      documents - d = floor((u1 + u2) / 2) with u1, u2 ~ U{1..N} (overlaps cluster mid-document),
                  and one request in ten has no overlap (d = 0)."""
    if kind not in DEPTH_KINDS:
        raise ValueError(kind)
    w = [0] * (N + 1)
    if kind == "uniform":
        for d in integers(seed, 101, 0, n_requests, 1, N):
            w[d] += 1
    elif kind == "prompts":
        spikes = integers(seed, 102, 0, 8, 1, N)
        pick = integers(seed, 103, 0, n_requests, 0, 7)
        coin = integers(seed, 104, 0, n_requests, 0, 3)
        other = integers(seed, 105, 0, n_requests, 0, N)
        for i in range(n_requests):
            w[spikes[pick[i]] if coin[i] < 3 else other[i]] += 1
    else:
        u1 = integers(seed, 106, 0, n_requests, 1, N)
        u2 = integers(seed, 107, 0, n_requests, 1, N)
        coin = integers(seed, 108, 0, n_requests, 0, 9)
        for i in range(n_requests):
            w[0 if coin[i] == 0 else (u1[i] + u2[i]) // 2] += 1
    return w


# --------------------------------------------------------------------------------------------
# synthetic linear-attention group for chained replay (its weights are inputs of the method)
# --------------------------------------------------------------------------------------------
def group_weights(seed: int, layers: int, heads: int, d_model: int, d_head: int, device="cpu") -> torch.Tensor:
    """Flat fp32 weights, layer after layer: W_q, W_k, W_v [heads d_head, d_model] and w_a, w_b
    [heads, d_model] with N(0, 1/d_model) entries, W_o [d_model, heads d_head] with N(0, 1/(4 heads d_head))."""
    Hd = heads * d_head
    parts = []
    for l in range(layers):
        base = 300 + 8 * l
        for j, (n, sc) in enumerate(((Hd * d_model, d_model ** -0.5), (Hd * d_model, d_model ** -0.5),
                                     (Hd * d_model, d_model ** -0.5), (heads * d_model, d_model ** -0.5),
                                     (heads * d_model, d_model ** -0.5), (d_model * Hd, 0.5 * Hd ** -0.5))):
            parts.append(normal(seed, base + j, 0, (n,), sc, device=device))
    return torch.cat(parts)


def group_inputs(seed: int, rows: int, d_model: int, device="cpu") -> torch.Tensor:
    """The group's cached input hidden states h [rows, d_model], N(0, 1) fp32."""
    return normal(seed, 299, 0, (rows, d_model), 1.0, device=device)

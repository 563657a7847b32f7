"""The seeded generator (CPU): slices regenerate bit-identically, shapes and
distributions follow the workload recipes."""
import torch

import synth


def test_slices_are_consistent():
    full = synth.rows(0, synth.STREAM_K, 0, 40, 6, 32, torch.bfloat16, True)
    tail = synth.rows(0, synth.STREAM_K, 25, 40, 6, 32, torch.bfloat16, True)
    head = synth.rows(0, synth.STREAM_K, 0, 40, 6, 32, torch.bfloat16, True, heads=range(2, 4))
    assert torch.equal(full[25:], tail)
    assert torch.equal(full[:, 2:4], head)
    a, b = synth.gates(0, 0, 40, 6, 0.9, 1.0, "uniform")
    a2, b2 = synth.gates(0, 25, 40, 6, 0.9, 1.0, "uniform", heads=range(1, 3))
    assert torch.equal(a[25:, 1:3], a2) and torch.equal(b[25:, 1:3], b2)


def test_unit_rows_and_moments():
    q = synth.rows(3, synth.STREAM_Q, 0, 512, 4, 128, torch.float32, True)
    n = q.double().norm(dim=-1)
    assert torch.allclose(n, torch.ones_like(n), atol=1e-6)
    v = synth.rows(3, synth.STREAM_V, 0, 512, 4, 128, torch.float32, False).double()
    assert abs(v.mean().item()) < 0.02 and abs(v.var().item() - 1.0) < 0.03
    assert v.abs().max().item() <= 2 * 3 ** 0.5
    qb = synth.rows(3, synth.STREAM_Q, 0, 512, 4, 128, torch.bfloat16, True)
    assert torch.equal(qb, q.to(torch.bfloat16))  # fp64 -> fp32 -> bf16, each RNE


def test_gate_ranges_and_seeds():
    a, b = synth.gates(0, 0, 1000, 16, 0.95, 1.0, "sigmoid")
    assert a.min() >= 0.95 and a.max() <= 1.0 and 0 < b.min() and b.max() < 1
    a1, _ = synth.gates(1, 0, 1000, 16, 0.95, 1.0, "sigmoid")
    assert not torch.equal(a, a1)
    streams = {s: synth.rows(0, s, 0, 8, 2, 32, torch.float32, False) for s in (1, 2, 3)}
    assert not torch.equal(streams[1], streams[2]) and not torch.equal(streams[2], streams[3])


def test_workload_recipes():
    w = synth.workload("tiny")
    assert (w.B, w.H, w.dk, w.T) == (1, 2, 32, 256) and w.ckpt_positions() == [[64, 128, 192, 256]]
    w = synth.workload("prefill")
    assert w.ckpt_positions()[0] == [512 * i for i in range(1, 17)]
    w = synth.workload("ragged10")
    assert w.B == 32 and all(4096 <= m <= 32768 for m in w.seq_lens)
    w = synth.workload("long")
    pr = w.probes()
    assert len(pr) == 64 and all(0 <= s < 4 and 1 <= d <= 131072 for s, d in pr)

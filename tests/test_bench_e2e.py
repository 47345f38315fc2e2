"""The end-to-end measurement overlaps host copies and kernels on three streams;
its results must be exactly those of the same steps run one after another on
one stream (same inputs, same step counters, the same error-feedback state
carried from step to step).  A missing event between the streams would show
here as a stale or half-written buffer."""
from __future__ import annotations

import types

import numpy as np
import pytest
import torch

import bench

pytestmark = pytest.mark.gpu


def _components():
    rx = bench.Receiver("rx_u8", 0, 8, n=1 << 20, M=4)
    return [bench.Fp8Rowwise(rows=20_000),
            bench.UniformEF("sr4_ef", 3_000_000, 4, 512, True, 2, "bucket"),
            bench.SignVote(n=1_000_000, M=4),
            rx, bench.Receiver("rx_ternary", 2, 2, n=1 << 20, M=4, shared=rx)]


def test_pipelined_e2e_matches_sequential_steps():
    import embedding_communication_codecs_gb300 as q
    steps = 3
    seq, pipe = _components(), _components()
    for c in seq + pipe:
        c.setup(q, torch)
    for c in seq:   # as in the end-to-end run: each step reads the buffer the host refills
        if hasattr(c, "fixed_input"):
            c.fixed_input = True
    timer = bench.KernelTimer(torch, enabled=False)
    for t in range(steps):
        for c in seq:
            c.run(q, 1000 + t, timer)
    torch.cuda.synchronize()
    want = [d.cpu() for c in seq for d in c.host_outputs()]
    got = []
    args = types.SimpleNamespace(steps=steps, e2e_steps=steps)
    units = sum(c.units for c in pipe)
    line = bench.run_e2e(args, pipe, q, torch, 1, units, results=got)
    assert line["value"] > 0 and line["streams"] == 3
    assert len(got) == len(want)
    for k, (g, w) in enumerate(zip(got, want)):
        a = g.numpy().view(np.uint8)
        b = w.numpy().view(np.uint8)
        assert np.array_equal(a, b), f"output {k} differs"

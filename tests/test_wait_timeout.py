"""The pipelines' failure path on the GPU, without a fault: a block waits on a
barrier that nothing completes, its bounded wait runs out, it records the
timeout flag and returns.  The host reads the flag, the flag clears, and the
context is still usable for a normal encode afterwards."""
from __future__ import annotations

import time

import numpy as np
import pytest
import torch

import oracle as orc
import workloads as wl
from tests._gpu import assert_bits_equal, host, u32

pytestmark = pytest.mark.gpu


def test_wait_runs_out_and_is_reported():
    import embedding_communication_codecs_gb300 as q
    assert q.qc_take_device_errors() == 0
    t0 = time.perf_counter()
    q.qc_selftest_wait_timeout(4096)
    flags = q.qc_take_device_errors()
    took = time.perf_counter() - t0
    assert flags & 1, flags
    assert took < 30.0
    print(f"4096 bounded tries ran out in {took * 1e3:.2f} ms (launch and read-back included)")
    assert q.qc_take_device_errors() == 0          # read and cleared
    # the context still works: a normal encode matches the oracle
    n, bits, bucket = 10_000 + 3, 8, 1024
    g = wl.std_normal(5, 1, n)
    gd = torch.from_numpy(g).cuda()
    codes, scale, offset = q.encode_ef(gd, None, bits=bits, bucket=bucket)
    assert q.qc_take_device_errors() == 0
    c_or, s_or, o_or = orc.encode_uniform(g, None, bits=bits, bucket=bucket)
    assert_bits_equal(u32(codes), c_or, "codes")
    assert_bits_equal(host(scale), s_or, "scale")
    assert_bits_equal(host(offset), o_or, "offset")

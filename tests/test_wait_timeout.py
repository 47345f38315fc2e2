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
    limit_ms = 20.0
    t0 = time.perf_counter()
    q.qc_selftest_wait_timeout(int(limit_ms * 1000))
    flags = q.qc_take_device_errors()
    took = (time.perf_counter() - t0) * 1e3
    assert flags & 1, flags
    # the wait is bounded by the GPU's global timer: it gives up after the
    # limit, not before, and not much later (launch and read-back included)
    assert limit_ms <= took < limit_ms + 2000.0, took
    print(f"a {limit_ms:.0f} ms bounded wait ran out after {took:.2f} ms (launch and read-back included)")
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


def test_status_word_reports_in_stream_order():
    """A caller-supplied status word learns, in stream order and without a
    device synchronisation, which launches timed out: the self-test's wait runs
    out and sets bit 0 of the word that was current at its launch; a normal
    encode launched with a second word leaves that word at zero."""
    import embedding_communication_codecs_gb300 as q
    assert q.qc_take_device_errors() == 0
    s = torch.cuda.Stream()
    words = torch.zeros(2, dtype=torch.int32, device="cuda")
    n, bits, bucket = 1 << 16, 4, 512
    g = torch.from_numpy(wl.std_normal(6, 1, n)).cuda()
    err = torch.zeros(n, device="cuda")
    codes, scale, offset = q.alloc_payload(n, bits, bucket, q.QC_SCHEME_UNIFORM)
    torch.cuda.synchronize()
    try:
        with torch.cuda.stream(s):
            q.qc_set_status_word(words[0:1])
            q.qc_selftest_wait_timeout(5000)
            q.qc_set_status_word(words[1:2])
            q.qc_encode_ef(g, err, n, bits, bucket, q.QC_SCHEME_UNIFORM, q.QC_ROUND_STOCHASTIC, 1,
                           0, codes, scale, offset)
            seen = words.to("cpu", non_blocking=True)
            done = torch.cuda.Event()
            done.record(s)
        done.synchronize()
    finally:
        q.qc_set_status_word(None)
    assert int(seen[0]) & 1 and int(seen[1]) == 0, seen
    assert q.qc_take_device_errors() & 1           # the global flag saw it too
    assert q.qc_take_device_errors() == 0

"""Every binary32 value with |x| <= 448 (the E4M3 range), converted by the row-wise
FP8 kernel and by the oracle's conversion written from the OCP 8-bit floating
point specification (round to nearest even, saturation to +-448).

The kernel divides each element by its row's scale absmax / 448; a row whose
first element is 448 has scale exactly 1, so x / scale = x and the code is the
plain conversion of x.  Each row carries 127 test values after that element.
The hardware conversion and the oracle's spec-written one must agree on all
~2.28e9 values; NaN inputs must give a NaN code.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle as orc

pytestmark = pytest.mark.gpu

TOP = 0x43E00000          # bit pattern of 448.0f
CHUNK = 127 * (1 << 19)   # test values per launch


def _patterns():
    """Bit-pattern ranges: [0, 448] for both signs."""
    return [(0x00000000, TOP + 1), (0x80000000, 0x80000000 + TOP + 1)]


def test_e4m3_all_values_in_range():
    import embedding_communication_codecs_gb300 as q
    dim = 128
    rows_max = CHUNK // 127
    xd = torch.empty((rows_max, dim), dtype=torch.float32, device="cuda")
    codes = torch.empty((rows_max, dim), dtype=torch.uint8, device="cuda")
    sc = torch.empty(rows_max, device="cuda")
    checked = 0
    for lo, hi in _patterns():
        for start in range(lo, hi, CHUNK):
            cnt = min(CHUNK, hi - start)
            vals = np.arange(start, start + cnt, dtype=np.uint64).astype(np.uint32).view(np.float32)
            rows = -(-cnt // 127)
            body = np.zeros(rows * 127, dtype=np.float32)
            body[:cnt] = vals
            x = np.empty((rows, dim), dtype=np.float32)
            x[:, 0] = 448.0
            x[:, 1:] = body.reshape(rows, 127)
            xd[:rows].copy_(torch.from_numpy(x))
            q.qc_rowwise_fp8(xd[:rows], rows, dim, codes[:rows], sc[:rows])
            assert bool((sc[:rows] == 1.0).all())
            got = codes[:rows].cpu().numpy()[:, 1:].reshape(-1)[:cnt]
            want = orc.e4m3_from_f32_array(vals)
            bad = np.flatnonzero(got != want)
            assert bad.size == 0, [(hex(int(vals[i].view(np.uint32))), int(got[i]), int(want[i]))
                                   for i in bad[:8]]
            checked += cnt
    assert checked == 2 * (TOP + 1)


def test_e4m3_nan_inputs():
    import embedding_communication_codecs_gb300 as q
    dim = 128
    rng = np.random.default_rng(0)
    mant = rng.integers(1, 1 << 23, size=127 * 64, dtype=np.uint64).astype(np.uint32)
    sign = (rng.integers(0, 2, size=mant.size, dtype=np.uint64).astype(np.uint32) << 31)
    nan = (sign | 0x7F800000 | mant).view(np.float32)
    x = np.zeros((64, dim), dtype=np.float32)
    x[:, 0] = 448.0
    x[:, 1:] = nan.reshape(64, 127)
    codes = torch.empty((64, dim), dtype=torch.uint8, device="cuda")
    sc = torch.empty(64, device="cuda")
    q.qc_rowwise_fp8(torch.from_numpy(x).cuda(), 64, dim, codes, sc)
    got = codes.cpu().numpy()[:, 1:]
    assert np.all((got & 0x7F) == 0x7F)
    assert np.all((orc.e4m3_from_f32_array(nan) & 0x7F) == 0x7F)

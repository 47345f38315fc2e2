"""GPU <-> oracle parity for top-k sparsification with 8-bit codes and error
feedback, and for its receiver.

Indices, codes, scales, offsets, residuals and decoded sums must match the
oracle bit for bit.  Cases: keep from 1 to the whole bucket, buckets that take
one warp and teams of 2..8 warps, short last buckets (fewer elements than
keep), ties at the threshold (resolved by index), zero buckets, bf16 inputs,
stochastic rounding, and decode of M workers with sentinel and out-of-bucket
slots.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle as orc
import workloads as wl
from tests._gpu import assert_bits_equal, dev, host

pytestmark = pytest.mark.gpu

SEED = 0x70C4_0000_0000_0003
STEP = 9


@pytest.fixture(scope="module")
def q():
    import embedding_communication_codecs_gb300 as q
    assert torch.cuda.is_available()
    return q


@pytest.fixture(autouse=True)
def no_device_errors(q):
    q.qc_take_device_errors()
    yield
    assert q.qc_take_device_errors() == 0


def _run(q, g, err0, n, bucket, keep, mode):
    nb = q.qc_num_buckets(n, bucket)
    idx = torch.full((nb * keep,), -7, dtype=torch.int32, device="cuda")
    codes = torch.full((nb * keep,), 77, dtype=torch.uint8, device="cuda")
    scale = torch.full((nb,), -7.0, device="cuda")
    offset = torch.full((nb,), -7.0, device="cuda")
    err = torch.from_numpy(err0.copy()).cuda() if err0 is not None else None
    dtype = q.QC_DTYPE_BF16 if g.dtype == np.uint16 else q.QC_DTYPE_F32
    q.qc_topk_encode_ef(dev(g), err, n, bucket, keep, mode, SEED, STEP, idx, codes, scale, offset,
                        dtype=dtype)
    torch.cuda.synchronize()
    return (host(idx, np.uint32), host(codes), host(scale), host(offset),
            host(err) if err is not None else None)


def _check(q, g, err0, n, bucket, keep, mode, tag):
    i, c, s, o, e = _run(q, g, err0, n, bucket, keep, mode)
    e_or = err0.copy() if err0 is not None else None
    i_or, c_or, s_or, o_or = orc.topk_encode(g, e_or, bucket=bucket, keep=keep, mode=mode,
                                             seed=SEED, step=STEP)
    assert_bits_equal(i, i_or, tag + " idx")
    assert_bits_equal(c, c_or, tag + " codes")
    assert_bits_equal(s, s_or, tag + " scale")
    assert_bits_equal(o, o_or, tag + " offset")
    if err0 is not None:
        assert_bits_equal(e, e_or, tag + " err")


@pytest.mark.parametrize("ef", [False, True])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("mode", [0, 1], ids=["nearest", "stochastic"])
def test_topk_encode(q, mode, dtype, ef):
    for bucket in (32, 96, 512, 1024, 2048, 4096):
        for keep in sorted({1, 5, max(1, bucket // 100), bucket // 4, bucket}):
            n = 5 * bucket + max(1, keep // 2)       # the last bucket is shorter than keep
            gf = wl.outlier_gradient(n, seed=bucket + keep)
            g = wl.to_bf16_bits(gf) if dtype == "bf16" else gf
            err0 = (wl.std_normal(91, 1, n) * np.float32(1e-4)) if ef else None
            _check(q, g, err0, n, bucket, keep, mode, f"topk {dtype} ef={ef} m={mode} B={bucket} K={keep}")


@pytest.mark.parametrize("keep", [1, 7, 100])
def test_topk_ties_and_degenerate(q, keep):
    """Equal magnitudes of both signs (ties decided by index), an all-zero
    bucket, a constant bucket, few distinct values, one huge outlier."""
    bucket = 1024
    n = 6 * bucket
    rng = np.random.default_rng(keep)
    g = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    g[0:bucket] = np.where(np.arange(bucket) % 3 == 0, -1.0, 1.0).astype(np.float32)
    g[bucket:2 * bucket] = 0.0
    g[2 * bucket:3 * bucket] = np.float32(0.5)
    g[3 * bucket:4 * bucket] = rng.choice(np.float32([-2.0, -1.0, 0.0, 1.0, 2.0]), bucket)
    g[4 * bucket + 77] = np.float32(1e6)
    for mode in (0, 1):
        _check(q, g, np.zeros(n, np.float32), n, bucket, keep, mode, f"topk ties K={keep} m={mode}")


@pytest.mark.parametrize("M,bucket,keep,tail,shift", [(1, 512, 12, 100, 0), (3, 512, 12, 101, 0),
                                                      (16, 512, 12, 100, 0), (8, 1024, 32, 101, 1),
                                                      (5, 992, 45, 101, 1), (9, 4096, 300, 100, 0)])
def test_topk_decode(q, M, bucket, keep, tail, shift):
    """keep <= 32 (a lane per pair, workers batched) and above; an output that
    starts one float past a 16-byte boundary, and a ragged last bucket, take the
    scalar output path."""
    n = 40 * bucket + tail                       # short last bucket
    idxs, codes, scales, offsets = [], [], [], []
    for w in range(M):
        i, c, s, o = orc.topk_encode(wl.outlier_gradient(n, seed=200 + w), bucket=bucket, keep=keep)
        idxs.append(i)
        codes.append(c)
        scales.append(s)
        offsets.append(o)
    idx = np.stack(idxs)
    cod = np.stack(codes)
    sc = np.stack(scales)
    of = np.stack(offsets)
    idx[0, 3] = 10 ** 6                           # out of its bucket: skipped
    idx[-1, keep + 1] = 5                         # belongs to bucket 0, sits in bucket 1: skipped
    prior = np.random.default_rng(M).standard_normal(n).astype(np.float32)
    for flags in (0, 1, 3):
        buf = torch.zeros(n + shift, dtype=torch.float32, device="cuda")
        out = buf[shift:]
        out.copy_(torch.from_numpy(prior))
        q.qc_topk_decode_accumulate(dev(idx), dev(cod), idx.shape[1], dev(sc), dev(of), sc.shape[1],
                                    M, n, bucket, keep, out, flags)
        want = orc.topk_decode(idx, cod, sc, of, M=M, n=n, bucket=bucket, keep=keep, flags=flags,
                               out=prior.copy())
        assert_bits_equal(host(out), want, f"topk decode M={M} flags={flags}")


def test_topk_full_size_sampled(q):
    """2^26 fp32 elements, buckets of 1024, keep 10 (1 %), with EF: a sample of
    whole buckets checked one by one by the oracle."""
    n, bucket, keep = 1 << 26, 1024, 10
    g = wl.outlier_gradient(n, seed=9)
    i, c, s, o, e = _run(q, g, np.zeros(n, np.float32), n, bucket, keep, 1)
    rng = np.random.default_rng(2)
    for k in list(rng.choice(n // bucket, 24, replace=False)) + [0, n // bucket - 1]:
        k = int(k)
        sl = slice(k * bucket, (k + 1) * bucket)
        e_or = np.zeros(bucket, np.float32)
        i_or, c_or, s_or, o_or = orc.topk_encode(g[sl], e_or, bucket=bucket, keep=keep, mode=1,
                                                 seed=SEED, step=STEP, index_base=k * bucket)
        ks = slice(k * keep, (k + 1) * keep)
        assert_bits_equal(i[ks], i_or, f"bucket {k} idx")
        assert_bits_equal(c[ks], c_or, f"bucket {k} codes")
        assert_bits_equal(s[k:k + 1], s_or, f"bucket {k} scale")
        assert_bits_equal(o[k:k + 1], o_or, f"bucket {k} offset")
        assert_bits_equal(e[sl], e_or, f"bucket {k} err")

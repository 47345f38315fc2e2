"""GPU <-> oracle parity for uniform quantization over the percentile-clipped
range (1st..99th percentile, nearest rank, per bucket).

Codes, scales, offsets and residuals must match the oracle bit for bit: the
bounds are elements of the bucket (an exact selection), the clamp is exact and
the rest is the uniform scheme's arithmetic.  Cases cover one warp per bucket
and teams of 2..8 warps, ragged tails (partial last buckets of 1, 37, 100 and
101 elements), heavy ties, constant and signed-zero buckets and outliers.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle as orc
import workloads as wl
from tests._gpu import assert_bits_equal, dev, host, u32

pytestmark = pytest.mark.gpu

SEED = 0x0C11_9000_0000_0001
STEP = 5


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


def _run(q, g, err0, n, bits, bucket, mode):
    words, nb = q.qc_code_words(n, bits), q.qc_num_buckets(n, bucket)
    codes = torch.full((words,), -7, dtype=torch.int32, device="cuda")
    scale = torch.full((nb,), -7.0, device="cuda")
    offset = torch.full((nb,), -7.0, device="cuda")
    err = torch.from_numpy(err0.copy()).cuda() if err0 is not None else None
    dtype = q.QC_DTYPE_BF16 if g.dtype == np.uint16 else q.QC_DTYPE_F32
    q.qc_encode_ef(dev(g), err, n, bits, bucket, q.QC_SCHEME_UNIFORM_CLIP, mode, SEED, STEP,
                   codes, scale, offset, dtype=dtype)
    torch.cuda.synchronize()
    return u32(codes), host(scale), host(offset), (host(err) if err is not None else None)


def _check(q, g, err0, n, bits, bucket, mode, tag):
    c, s, o, e = _run(q, g, err0, n, bits, bucket, mode)
    e_or = err0.copy() if err0 is not None else None
    c_or, s_or, o_or = orc.encode_uniform_clip(g, e_or, bits=bits, bucket=bucket, mode=mode,
                                               seed=SEED, step=STEP)
    assert_bits_equal(o, o_or, tag + " offset")
    assert_bits_equal(s, s_or, tag + " scale")
    assert_bits_equal(c, c_or, tag + " codes")
    if err0 is not None:
        assert_bits_equal(e, e_or, tag + " err")


@pytest.mark.parametrize("ef", [False, True])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("mode", [0, 1], ids=["nearest", "stochastic"])
@pytest.mark.parametrize("bits", [1, 2, 4, 8])
def test_encode_clip(q, bits, mode, dtype, ef):
    for bucket, tail in ((32, 1), (96, 37), (512, 100), (1024, 101), (2048, 37), (4096, 1)):
        n = 6 * bucket + tail
        gf = wl.outlier_gradient(n, seed=bucket + 3 * bits)
        g = wl.to_bf16_bits(gf) if dtype == "bf16" else gf
        err0 = (wl.std_normal(93, 1, n) * np.float32(1e-4)) if ef else None
        _check(q, g, err0, n, bits, bucket, mode, f"clip b={bits} m={mode} {dtype} ef={ef} B={bucket}")


@pytest.mark.parametrize("bits", [2, 8])
def test_encode_clip_degenerate(q, bits):
    """Constant, +-0, few distinct values (the percentiles fall inside runs of
    equal keys), all negative, tiny and huge magnitudes, and one outlier per
    bucket on either side."""
    bucket = 1024
    n = 9 * bucket
    rng = np.random.default_rng(bits)
    g = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    g[0:bucket] = np.float32(0.25)
    g[bucket:2 * bucket] = np.where(np.arange(bucket) % 2, 0.0, -0.0).astype(np.float32)
    g[2 * bucket:3 * bucket] = rng.choice(np.float32([-2.0, -1.0, 0.0, 1.0, 3.0]), bucket)
    g[3 * bucket:4 * bucket] = -np.abs(g[3 * bucket:4 * bucket]) - np.float32(1.0)
    g[4 * bucket:5 * bucket] *= np.float32(1e-36)
    g[5 * bucket:6 * bucket] *= np.float32(1e33)
    g[6 * bucket + 5] = np.float32(50.0)
    g[6 * bucket + 9] = np.float32(-70.0)
    g[7 * bucket:8 * bucket] = rng.choice(np.float32([-0.0, 0.0, 1e-3]), bucket)
    for mode in (0, 1):
        _check(q, g, np.zeros(n, np.float32), n, bits, bucket, mode, f"clip degenerate b={bits} m={mode}")


def test_clip_payload_decodes_as_uniform(q):
    n, bits, bucket, M = 20_000 + 7, 4, 512, 3
    payloads = [orc.encode_uniform_clip(wl.outlier_gradient(n, seed=60 + w), bits=bits, bucket=bucket)
                for w in range(M)]
    codes = np.stack([c for c, _, _ in payloads])
    scale = np.stack([s for _, s, _ in payloads])
    offset = np.stack([o for _, _, o in payloads])
    words, nb = codes.shape[1], scale.shape[1]
    out_clip = torch.empty(n, device="cuda")
    out_uni = torch.empty(n, device="cuda")
    for sch, out in ((q.QC_SCHEME_UNIFORM_CLIP, out_clip), (q.QC_SCHEME_UNIFORM, out_uni)):
        q.qc_decode_accumulate(dev(codes), words, dev(scale), dev(offset), nb, M, n, bits, bucket,
                               sch, out, q.QC_OUT_MEAN)
    want = orc.decode_accumulate(codes, scale, offset, M=M, n=n, bits=bits, bucket=bucket,
                                 scheme=orc.SCHEME_UNIFORM_CLIP, flags=orc.OUT_MEAN)
    assert_bits_equal(host(out_clip), want, "decode clip")
    assert_bits_equal(host(out_uni), want, "decode as uniform")


def test_clip_full_size_sampled(q):
    """The 2^20-element outlier workload with 2048-element buckets (the small
    configuration), whole-array comparison, then 2^26 elements with a sample of
    buckets checked by the oracle one by one."""
    n, bucket = 1 << 20, 2048
    g = wl.outlier_gradient(n, seed=0)
    _check(q, g, np.zeros(n, np.float32), n, 8, bucket, 0, "clip 2^20")
    n = 1 << 26
    g = wl.outlier_gradient(n, seed=7)
    c, s, o, e = _run(q, g, np.zeros(n, np.float32), n, 8, bucket, 1)
    rng = np.random.default_rng(1)
    wpb = bucket // 4
    for k in list(rng.choice(n // bucket, 24, replace=False)) + [0, n // bucket - 1]:
        k = int(k)
        sl = slice(k * bucket, (k + 1) * bucket)
        e_or = np.zeros(bucket, np.float32)
        c_or, s_or, o_or = orc.encode_uniform_clip(g[sl], e_or, bits=8, bucket=bucket, mode=1,
                                                   seed=SEED, step=STEP, index_base=k * bucket)
        assert_bits_equal(c[k * wpb:(k + 1) * wpb], c_or, f"bucket {k} codes")
        assert_bits_equal(s[k:k + 1], s_or, f"bucket {k} scale")
        assert_bits_equal(o[k:k + 1], o_or, f"bucket {k} offset")
        assert_bits_equal(e[sl], e_or, f"bucket {k} err")

"""GPU <-> oracle parity for the logarithmic-level scheme (a sign bit over the
index j of the level s * 2^(j - J), s = max |p| of the bucket).

Every output is bit-exact: the scale is a maximum, the level a decision taken
on the correctly rounded quotient |p| / s on both sides, and the dequantized
value one binary32 product.  The cases cover the encode kernels (f32 and bf16,
with and without error feedback, both rounding modes, one warp to whole-block
buckets, ragged tails), values placed on every decision boundary of the level
rule and one ulp either side, degenerate buckets, quotients below the smallest
normal number, the two decode kernels and the fused re-encode.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle as orc
import workloads as wl
from tests._gpu import assert_bits_equal, dev, host, u32

pytestmark = pytest.mark.gpu

SEED = 0x1357_9BDF_2468_ACE0
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


def _unpack(words, n, bits):
    per = 32 // bits
    sh = (np.arange(per, dtype=np.uint32) * bits).astype(np.uint32)
    return ((words.reshape(-1)[:, None] >> sh[None, :]) & np.uint32((1 << bits) - 1)).reshape(-1)[:n]


def _encode(q, g, err0, n, bits, bucket, mode):
    words, nb = q.qc_code_words(n, bits), q.qc_num_buckets(n, bucket)
    codes = torch.full((words,), -7, dtype=torch.int32, device="cuda")
    scale = torch.full((nb,), -7.0, device="cuda")
    err = torch.from_numpy(err0.copy()).cuda() if err0 is not None else None
    dtype = q.QC_DTYPE_BF16 if g.dtype == np.uint16 else q.QC_DTYPE_F32
    q.qc_encode_ef(dev(g), err, n, bits, bucket, q.QC_SCHEME_LOG, mode, SEED, STEP, codes, scale,
                   None, dtype=dtype)
    torch.cuda.synchronize()
    return u32(codes), host(scale), (host(err) if err is not None else None)


def _check(q, g, err0, n, bits, bucket, mode, tag):
    c, s, e = _encode(q, g, err0, n, bits, bucket, mode)
    e_or = err0.copy() if err0 is not None else None
    c_or, s_or = orc.encode_log(g, e_or, bits=bits, bucket=bucket, mode=mode, seed=SEED, step=STEP)
    assert_bits_equal(s, s_or, tag + " scale")
    assert_bits_equal(c, c_or, tag + " codes")
    if err0 is not None:
        assert_bits_equal(e, e_or, tag + " err")
    return c, s


@pytest.mark.parametrize("ef", [False, True])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("mode", [0, 1], ids=["nearest", "stochastic"])
@pytest.mark.parametrize("bits", [2, 4, 8])
def test_encode_log(q, bits, mode, dtype, ef):
    buckets = [32, 96, 512, 1024, 2048, 4096] + ([8192] if dtype == "bf16" and not ef else [])
    for bucket in buckets:
        n = max(5 * bucket, 6000) + 37
        gf = wl.outlier_gradient(n, seed=11 * bucket + bits)
        if dtype == "f32":
            gf[bucket:2 * bucket] = 0.0           # an all-zero bucket: scale 0, codes 0
        g = wl.to_bf16_bits(gf) if dtype == "bf16" else gf
        err0 = (wl.std_normal(97, 1, n) * np.float32(1e-4)) if ef else None
        _check(q, g, err0, n, bits, bucket, mode, f"log b={bits} m={mode} {dtype} ef={ef} B={bucket}")


def _boundary_gradient(bits, s_val, bucket=256):
    """Buckets whose largest magnitude is s_val (its first element) and whose
    other elements sit at fl(s_val * x) for x on every decision boundary of the
    level rule -- the levels 2^(j-J), the midpoints 1.5 * 2^e between two of
    them, 2^-J (half the smallest level) -- and one ulp either side, with
    alternating signs."""
    J = (1 << (bits - 1)) - 1
    xs = [2.0 ** e for e in range(-J, 1)] + [1.5 * 2.0 ** e for e in range(1 - J, 0)]
    xs += [0.75 * 2.0 ** (1 - J), 0.25 * 2.0 ** (1 - J)]
    v = (np.array(xs, dtype=np.float64) * s_val).astype(np.float32)
    v = np.concatenate([v, np.nextafter(v, np.float32(np.inf)), np.nextafter(v, np.float32(0))])
    v = v[(v > 0) & (v <= np.float32(s_val))]
    per = bucket - 1
    nb = (v.size + per - 1) // per
    g = np.zeros(nb * bucket, dtype=np.float32)
    for k in range(nb):
        chunk = v[k * per:(k + 1) * per]
        sign = np.where(np.arange(chunk.size) % 2, -1.0, 1.0).astype(np.float32)
        g[k * bucket] = np.float32(s_val) * (1 if k % 2 == 0 else -1)
        g[k * bucket + 1:k * bucket + 1 + chunk.size] = chunk * sign
    return g, bucket


@pytest.mark.parametrize("s_val", [1.0, 3.0, 0.7, 2.0 ** -100, 1.0e30])
@pytest.mark.parametrize("bits", [2, 4, 8])
def test_encode_log_decision_boundaries(q, bits, s_val):
    """Every level, every midpoint and the lower edge of the smallest level, on
    the boundary and one ulp either side (with s a power of two the quotient is
    exactly the boundary; otherwise its rounding decides)."""
    g, bucket = _boundary_gradient(bits, s_val)
    n = g.size
    for mode in (0, 1):
        err0 = np.zeros(n, dtype=np.float32)
        c, s = _check(q, g, err0, n, bits, bucket, mode, f"log boundaries b={bits} s={s_val} m={mode}")
        assert np.all(s == np.float32(s_val))


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_encode_log_degenerate(q, bits):
    """Zero and +-0 buckets (scale 0, every code 0), one non-zero element (the
    top level, its sign), a constant bucket (every element at the top level),
    and buckets spanning more than 2^126 so that quotients fall below the
    smallest normal number."""
    bucket = 512
    n = 8 * bucket + 5
    J = (1 << (bits - 1)) - 1
    g = wl.std_normal(9, 1, n) * np.float32(1e-3)
    g[0:bucket] = 0.0
    g[bucket:2 * bucket] = np.where(np.arange(bucket) % 2, 0.0, -0.0).astype(np.float32)
    g[2 * bucket:3 * bucket] = 0.0
    g[2 * bucket + 17] = np.float32(-30.0)
    g[3 * bucket:4 * bucket] = np.float32(0.25)
    g[4 * bucket:5 * bucket] *= np.float32(1e-30)              # subnormal and tiny inputs
    g[5 * bucket] = np.float32(1e30)                            # quotients down to ~1e-66
    g[6 * bucket:7 * bucket] *= np.float32(1e35)
    g[6 * bucket + 3] = np.float32(2.0 ** -149)                 # the smallest subnormal
    for mode in (0, 1):
        err0 = np.zeros(n, dtype=np.float32)
        c, s = _check(q, g, err0, n, bits, bucket, mode, f"log degenerate b={bits} m={mode}")
        codes = _unpack(c, n, bits)
        assert s[0] == 0 and s[1] == 0
        assert np.all(codes[:2 * bucket] == 0)
        assert codes[2 * bucket + 17] == (1 << (bits - 1)) | J
        assert np.all(codes[3 * bucket:4 * bucket] == J)


@pytest.mark.parametrize("mode", [0, 1], ids=["nearest", "stochastic"])
@pytest.mark.parametrize("bits", [2, 4, 8])
def test_encode_log_direct_kernel(q, bits, mode):
    """The direct kernel: buckets above the pipelined team window (two passes,
    f32 with and without error feedback) and a bf16 gradient whose base is 8- but
    not 16-byte aligned."""
    for bucket in (8192, 16384):
        n = 3 * bucket + 77
        g = wl.outlier_gradient(n, seed=bucket + bits)
        for ef in (False, True):
            err0 = (wl.std_normal(98, 1, n) * np.float32(1e-4)) if ef else None
            _check(q, g, err0, n, bits, bucket, mode, f"log direct b={bits} m={mode} B={bucket} ef={ef}")
    bucket, n = 1024, 1024 * 9 + 20
    gb = wl.to_bf16_bits(wl.outlier_gradient(n + 4, seed=bits))
    base = torch.from_numpy(gb.view(np.int16).copy()).cuda()
    g_dev = base[4:]                       # 8 bytes past a 16-byte aligned allocation
    assert g_dev.data_ptr() % 16 == 8
    words, nb = q.qc_code_words(n, bits), q.qc_num_buckets(n, bucket)
    codes = torch.full((words,), -7, dtype=torch.int32, device="cuda")
    scale = torch.full((nb,), -7.0, device="cuda")
    q.qc_encode_ef(g_dev, None, n, bits, bucket, q.QC_SCHEME_LOG, mode, SEED, STEP, codes, scale,
                   None, dtype=q.QC_DTYPE_BF16)
    torch.cuda.synchronize()
    c_or, s_or = orc.encode_log(gb[4:], None, bits=bits, bucket=bucket, mode=mode, seed=SEED,
                                step=STEP)
    assert_bits_equal(host(scale), s_or, "log bf16 unaligned scale")
    assert_bits_equal(u32(codes), c_or, "log bf16 unaligned codes")


def test_encode_log_large(q):
    """n = 2^22 + 3 f32 elements, 4 bits, stochastic rounding, error feedback,
    B = 512, compared whole."""
    n, bits, bucket = (1 << 22) + 3, 4, 512
    g = wl.outlier_gradient(n, seed=31)
    err0 = wl.std_normal(32, 1, n) * np.float32(1e-4)
    _check(q, g, err0, n, bits, bucket, 1, "log large")


def _payload(rng, M, n, bits, bucket, zero_scale=True):
    words, nb = orc.code_words(n, bits), orc.num_buckets(n, bucket)
    cstride = words + (-words) % 4 + 4
    mstride = nb + 3
    codes = rng.integers(0, 1 << 32, size=(M, cstride), dtype=np.uint64).astype(np.uint32)
    scale = (rng.random((M, mstride)) * 1e-2).astype(np.float32)
    if zero_scale:
        scale[:, 1] = 0.0
    return codes, cstride, scale, mstride


@pytest.mark.parametrize("bits", [2, 4, 8])
@pytest.mark.parametrize("M", [1, 3, 8, 16])
def test_decode_log(q, bits, M):
    """Random code words (every word is a valid payload: the sign bit over any
    level index) from M workers, fixed-order fp32 accumulation; M < 4 takes the
    direct decode kernel, M >= 4 the pipelined one."""
    rng = np.random.default_rng(100 * M + bits)
    for bucket, flags in ((32, orc.OUT_SUM), (512, orc.OUT_MEAN),
                          (2048, orc.OUT_MEAN | orc.ACCUMULATE_INTO_OUT)):
        n = 3 * bucket + 4099
        codes, cstride, scale, mstride = _payload(rng, M, n, bits, bucket)
        out0 = wl.std_normal(M + bits, 2, n)
        out = torch.from_numpy(out0.copy()).cuda()
        q.qc_decode_accumulate(dev(codes), cstride, dev(scale), None, mstride, M, n, bits, bucket,
                               q.QC_SCHEME_LOG, out, flags)
        torch.cuda.synchronize()
        want = orc.decode_accumulate(codes, scale, None, M=M, n=n, bits=bits, bucket=bucket,
                                     scheme=orc.SCHEME_LOG, flags=flags,
                                     codes_stride_words=cstride, meta_stride=mstride,
                                     out=out0.copy())
        assert_bits_equal(host(out), want, f"log decode b={bits} M={M} B={bucket} f={flags}")


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_decode_inverts_encode(q, bits):
    """Decoding one worker's payload gives back p - err exactly: the residual
    of the encode is the dequantization error of the payload it wrote.  With
    nearest rounding every non-zero level lies within a factor of two of its
    element, so p - deq and p - (p - deq) are exact (Sterbenz); stochastic
    rounding may lift a tiny element to the smallest level, where they are not."""
    n, bucket = 40_000 + 7, 1024
    g = wl.outlier_gradient(n, seed=bits)
    err0 = np.zeros(n, dtype=np.float32)
    c, s, e = _encode(q, g, err0, n, bits, bucket, 0)
    out = torch.empty(n, device="cuda")
    q.qc_decode_accumulate(dev(c), 0, dev(s), None, 0, 1, n, bits, bucket, q.QC_SCHEME_LOG, out,
                           q.QC_OUT_SUM)
    torch.cuda.synchronize()
    d = host(out)
    assert_bits_equal((g - e).astype(np.float32), d + np.float32(0.0), f"b={bits} deq")


@pytest.mark.parametrize("mode", [0, 1], ids=["nearest", "stochastic"])
@pytest.mark.parametrize("bits", [2, 4, 8])
@pytest.mark.parametrize("M", [1, 5, 16])
def test_reencode_log(q, bits, mode, M):
    """Decode, accumulate and re-encode with the receiver's residual, fused;
    r, the new payload and the residual bit-exact."""
    rng = np.random.default_rng(7 * M + bits + 100 * mode)
    for i, bucket in enumerate((32, 1024, 4096)):
        n = max(3 * bucket, 3000) + 13
        flags = orc.OUT_MEAN if i % 2 == 0 else orc.OUT_SUM
        ef = i != 1
        codes, cstride, scale, mstride = _payload(rng, M, n, bits, bucket, zero_scale=False)
        words, nb = orc.code_words(n, bits), orc.num_buckets(n, bucket)
        err0 = (wl.std_normal(int(rng.integers(1 << 30)), 1, n) * np.float32(1e-4)) if ef else None
        err_d = torch.from_numpy(err0.copy()).cuda() if ef else None
        co = torch.full((words,), -7, dtype=torch.int32, device="cuda")
        so = torch.full((nb,), -7.0, device="cuda")
        out = torch.full((n,), -7.0, device="cuda")
        q.qc_reencode(dev(codes), cstride, dev(scale), None, mstride, M, n, bits, bucket,
                      q.QC_SCHEME_LOG, flags, err_d, mode, SEED, STEP, co, so, None, out)
        torch.cuda.synchronize()
        e_or = err0.copy() if ef else None
        r, c_or, s_or, _ = orc.reencode(codes, scale, None, M=M, n=n, bits=bits, bucket=bucket,
                                        scheme=orc.SCHEME_LOG, flags=flags, err=e_or, mode=mode,
                                        seed=SEED, step=STEP, codes_stride_words=cstride,
                                        meta_stride=mstride)
        tag = f"log reencode b={bits} m={mode} M={M} B={bucket}"
        assert_bits_equal(host(out), r, tag + " r")
        assert_bits_equal(u32(co), c_or, tag + " codes")
        assert_bits_equal(host(so), s_or, tag + " scale")
        if ef:
            assert_bits_equal(host(err_d), e_or, tag + " err")

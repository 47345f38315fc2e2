"""GPU <-> oracle parity on small inputs: every scheme x bits x rounding x dtype x
error feedback, bucket sizes that take every launch shape (one warp per bucket,
teams of 2..8 warps, two-pass buckets), ragged tails, and the degenerate cases.

Codes, packed words, votes and FP8 bytes must match bit for bit.  Uniform and
ternary floats (scales, offsets, residuals) and every decoded sum are expected
bit-exact too; the sign scheme's mean |p| is compared within 1e-6 * max|p| of
its bucket, its only freedom being the order of the sum.  Every output sits
between canary guard regions that must survive the launch.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle as orc
import workloads as wl
from tests._gpu import assert_bits_equal, assert_close_per_bucket, dev, host, u32

pytestmark = pytest.mark.gpu

SEED = 0x1234_5678_9ABC_DEF0
STEP = 7


@pytest.fixture(scope="module")
def q():
    import embedding_communication_codecs_gb300 as q
    assert torch.cuda.is_available()
    return q


@pytest.fixture(autouse=True)
def no_device_errors(q):
    """No pipelined kernel may report a timed-out wait."""
    q.qc_take_device_errors()
    yield
    assert q.qc_take_device_errors() == 0


class Guarded:
    """A device tensor between canary regions."""

    def __init__(self, n, dtype, init=None, guard=64, fill=-7):
        self.base = torch.full((n + 2 * guard,), fill, dtype=dtype, device="cuda")
        self.t = self.base[guard:guard + n]
        if init is not None:
            self.t.copy_(init)
        self.guard, self.fill, self.n = guard, fill, n

    def check(self):
        b = self.base.cpu()
        assert bool((b[:self.guard] == self.fill).all()), "canary before the buffer was overwritten"
        assert bool((b[self.guard + self.n:] == self.fill).all()), "canary after the buffer was overwritten"


def _grad(n, dtype, seed):
    g = wl.outlier_gradient(n, seed=seed)
    if dtype == "bf16":
        return wl.to_bf16_bits(g)
    return g


def _grad_dev(g):
    return dev(g)


def _run_encode(q, g, err0, n, bits, bucket, scheme, mode):
    words, nb = q.qc_code_words(n, bits), q.qc_num_buckets(n, bucket)
    codes = Guarded(words, torch.int32)
    scale = Guarded(nb, torch.float32)
    offset = Guarded(nb, torch.float32) if scheme == q.QC_SCHEME_UNIFORM else None
    err = Guarded(n, torch.float32, init=torch.from_numpy(err0).cuda()) if err0 is not None else None
    dtype = q.QC_DTYPE_BF16 if g.dtype == np.uint16 else q.QC_DTYPE_F32
    q.qc_encode_ef(_grad_dev(g), err.t if err else None, n, bits, bucket, scheme, mode, SEED, STEP,
                   codes.t, scale.t, offset.t if offset else None, dtype=dtype)
    torch.cuda.synchronize()
    for b in (codes, scale, offset, err):
        if b is not None:
            b.check()
    return (u32(codes.t), host(scale.t), host(offset.t) if offset else None,
            host(err.t) if err else None)


def _p_of(g, err0):
    gf = wl.bf16_bits_to_f32(g) if g.dtype == np.uint16 else g
    return gf if err0 is None else (err0 + gf).astype(np.float32)


BUCKETS = [32, 96, 512, 1024, 2048, 4096, 8192]


def _n_for(bucket):
    return max(5 * bucket, 6000) + 37        # partial last bucket, n % 4 != 0


@pytest.mark.parametrize("ef", [False, True])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("mode", [0, 1], ids=["nearest", "stochastic"])
@pytest.mark.parametrize("bits", [1, 2, 4, 8])
def test_encode_uniform(q, bits, mode, dtype, ef):
    for bucket in BUCKETS:
        n = _n_for(bucket)
        g = _grad(n, dtype, seed=bucket + bits)
        err0 = (wl.std_normal(99, 1, n) * np.float32(1e-4)) if ef else None
        codes, scale, offset, err = _run_encode(q, g, err0, n, bits, bucket,
                                                q.QC_SCHEME_UNIFORM, mode)
        e_or = err0.copy() if ef else None
        c_or, s_or, o_or = orc.encode_uniform(g, e_or, bits=bits, bucket=bucket, mode=mode,
                                              seed=SEED, step=STEP)
        tag = f"uniform b={bits} mode={mode} {dtype} ef={ef} B={bucket}"
        assert_bits_equal(codes, c_or, tag + " codes")
        assert_bits_equal(scale, s_or, tag + " scale")
        assert_bits_equal(offset, o_or, tag + " offset")
        if ef:
            assert_bits_equal(err, e_or, tag + " err")


@pytest.mark.parametrize("ef", [False, True])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_encode_sign(q, dtype, ef):
    for bucket in [32, 96, 512, 2048, 4096, 8192]:
        n = _n_for(bucket)
        g = _grad(n, dtype, seed=3 + bucket)
        err0 = (wl.std_normal(98, 1, n) * np.float32(5e-4)) if ef else None
        codes, scale, _, err = _run_encode(q, g, err0, n, 1, bucket, q.QC_SCHEME_SIGN, 0)
        e_or = err0.copy() if ef else None
        c_or, s_or = orc.encode_sign(g, e_or, bucket=bucket)
        tag = f"sign {dtype} ef={ef} B={bucket}"
        assert_bits_equal(codes, c_or, tag + " bits")
        p = _p_of(g, err0)
        nb = s_or.size
        pmax = np.array([np.abs(p[k * bucket:(k + 1) * bucket]).max() for k in range(nb)])
        assert np.all(np.abs(scale.astype(np.float64) - s_or) <= 1e-6 * pmax), tag + " scale"
        if ef:
            assert_close_per_bucket(err, e_or, p, bucket, 1e-6, tag + " err")


@pytest.mark.parametrize("ef", [False, True])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("mode", [0, 1], ids=["nearest", "stochastic"])
def test_encode_ternary(q, mode, dtype, ef):
    for bucket in [32, 512, 1024, 4096, 8192]:
        n = _n_for(bucket)
        g = _grad(n, dtype, seed=5 + bucket)
        if dtype == "f32":
            g[bucket:2 * bucket] = 0.0          # an all-zero bucket
        err0 = (wl.std_normal(97, 1, n) * np.float32(1e-4)) if ef else None
        codes, scale, _, err = _run_encode(q, g, err0, n, 2, bucket, q.QC_SCHEME_TERNARY, mode)
        e_or = err0.copy() if ef else None
        c_or, s_or = orc.encode_ternary(g, e_or, bucket=bucket, mode=mode, seed=SEED, step=STEP)
        tag = f"ternary mode={mode} {dtype} ef={ef} B={bucket}"
        assert_bits_equal(codes, c_or, tag + " codes")
        assert_bits_equal(scale, s_or, tag + " scale")
        if ef:
            assert_bits_equal(err, e_or, tag + " err")


@pytest.mark.parametrize("bits", [1, 2, 4, 8])
def test_encode_degenerate_buckets(q, bits):
    """Constant buckets, +-0, a single outlier, tiny (subnormal) ranges, huge values."""
    bucket = 512
    n = 8 * bucket + 5
    g = wl.std_normal(5, 1, n) * np.float32(1e-3)
    g[0:bucket] = np.float32(0.25)                              # constant
    g[bucket:2 * bucket] = np.where(np.arange(bucket) % 2, 0.0, -0.0).astype(np.float32)
    g[2 * bucket + 17] = np.float32(30.0)                       # one outlier
    g[3 * bucket:4 * bucket] = (np.arange(bucket) % 7).astype(np.float32) * np.float32(1e-44)
    g[4 * bucket:5 * bucket] *= np.float32(1e36)                # near the top of the range
    g[5 * bucket:6 * bucket] = np.float32(-3.0)
    g[5 * bucket + 9] = np.float32(-3.0000002)
    for mode in (0, 1):
        err0 = np.zeros(n, dtype=np.float32)
        codes, scale, offset, err = _run_encode(q, g, err0, n, bits, bucket,
                                                q.QC_SCHEME_UNIFORM, mode)
        e_or = err0.copy()
        c_or, s_or, o_or = orc.encode_uniform(g, e_or, bits=bits, bucket=bucket, mode=mode,
                                              seed=SEED, step=STEP)
        tag = f"degenerate b={bits} mode={mode}"
        assert_bits_equal(codes, c_or, tag + " codes")
        assert_bits_equal(scale, s_or, tag + " scale")
        assert_bits_equal(offset, o_or, tag + " offset")
        assert_bits_equal(err, e_or, tag + " err")


@pytest.mark.parametrize("bits", [1, 2, 4, 8])
def test_encode_decision_boundaries(q, bits):
    """Elements exactly on, and one ulp either side of, every rounding decision:
    half-integer levels (ties to even), integer levels (the floor of stochastic
    rounding), and for the ternary scheme |p| / s = 1/2 and |p| = s."""
    L = (1 << bits) - 1
    bucket = 512
    c = np.float32(2.0 ** -6)
    vals = []
    for k in range(L + 1):
        for frac in (0.0, 0.5):
            v = np.float32((k + frac) * c)
            vals += [v, np.nextafter(v, np.float32(1e9)), np.nextafter(v, np.float32(-1e9))]
    vals = np.array(vals, dtype=np.float32)
    vals = vals[(vals >= 0) & (vals <= np.float32(L * c))]
    reps = -(-bucket // vals.size)
    g = np.tile(vals, reps * 6)[:6 * bucket].astype(np.float32)
    for k in range(6):                         # pin min 0 and max L*c in every bucket
        g[k * bucket] = 0.0
        g[k * bucket + 1] = np.float32(L * c)
    for mode in (0, 1):
        for scheme, b in ((0, bits), (2, 2)):
            if scheme == 2 and bits != 2:
                continue
            gg = g.copy()
            if scheme == 2:
                gg = np.where(np.arange(gg.size) % 3 == 0, np.float32(0.5), gg).astype(np.float32)
                gg[::bucket] = 1.0
            codes, scale, offset, err = _run_encode(q, gg, np.zeros_like(gg), gg.size, b, bucket,
                                                    scheme, mode)
            e_or = np.zeros_like(gg)
            if scheme == 0:
                c_or, s_or, o_or = orc.encode_uniform(gg, e_or, bits=b, bucket=bucket, mode=mode,
                                                      seed=SEED, step=STEP)
                assert s_or[0] == c
            else:
                c_or, s_or = orc.encode_ternary(gg, e_or, bucket=bucket, mode=mode, seed=SEED,
                                                step=STEP)
            tag = f"boundaries scheme={scheme} b={b} mode={mode}"
            assert_bits_equal(codes, c_or, tag + " codes")
            assert_bits_equal(scale, s_or, tag + " scale")
            assert_bits_equal(err, e_or, tag + " err")


@pytest.mark.parametrize("scheme,bits,mode", [(0, 8, 0), (0, 4, 1), (1, 1, 0), (2, 2, 1)])
def test_encode_bf16_unaligned_base(q, scheme, bits, mode):
    """A bf16 gradient that is 8- but not 16-byte aligned takes the direct kernel;
    results are the same as the oracle's (and so as the pipelined kernel's)."""
    bucket, n = 1024, 1024 * 9 + 20
    g = wl.to_bf16_bits(wl.outlier_gradient(n, seed=21))
    base = torch.zeros(n + 8, dtype=torch.int16, device="cuda")
    view = base[4:4 + n]
    view.copy_(torch.from_numpy(g.view(np.int16)).cuda())
    assert view.data_ptr() % 16 == 8
    words, nb = q.qc_code_words(n, bits), q.qc_num_buckets(n, bucket)
    codes = torch.empty(words, dtype=torch.int32, device="cuda")
    scale = torch.empty(nb, device="cuda")
    offset = torch.empty(nb, device="cuda") if scheme == 0 else None
    err = torch.zeros(n, device="cuda")
    q.qc_encode_ef(view, err, n, bits, bucket, scheme, mode, SEED, STEP, codes, scale, offset,
                   dtype=q.QC_DTYPE_BF16)
    e_or = np.zeros(n, dtype=np.float32)
    if scheme == 0:
        c_or, s_or, o_or = orc.encode_uniform(g, e_or, bits=bits, bucket=bucket, mode=mode,
                                              seed=SEED, step=STEP)
        assert_bits_equal(host(offset), o_or)
    elif scheme == 1:
        c_or, s_or = orc.encode_sign(g, e_or, bucket=bucket)
    else:
        c_or, s_or = orc.encode_ternary(g, e_or, bucket=bucket, mode=mode, seed=SEED, step=STEP)
    assert_bits_equal(u32(codes), c_or, "codes")
    if scheme != 1:
        assert_bits_equal(host(scale), s_or, "scale")
        assert_bits_equal(host(err), e_or, "err")


@pytest.mark.parametrize("n", [1, 3, 31, 32, 33, 100, 511, 513])
def test_encode_tiny_sizes(q, n):
    g = wl.std_normal(11, 1, n) * np.float32(1e-3)
    for scheme, bits in ((0, 8), (0, 1), (1, 1), (2, 2)):
        err0 = np.zeros(n, dtype=np.float32)
        codes, scale, offset, err = _run_encode(q, g, err0, n, bits, 64, scheme, 0)
        e_or = err0.copy()
        if scheme == 0:
            c_or, s_or, o_or = orc.encode_uniform(g, e_or, bits=bits, bucket=64)
            assert_bits_equal(offset, o_or)
        elif scheme == 1:
            c_or, s_or = orc.encode_sign(g, e_or, bucket=64)
        else:
            c_or, s_or = orc.encode_ternary(g, e_or, bucket=64, mode=0)
        assert_bits_equal(codes, c_or, f"n={n} scheme={scheme} codes")
        if scheme != 1:
            assert_bits_equal(scale, s_or)
            assert_bits_equal(err, e_or)


def test_encode_n_zero_is_noop(q):
    x = torch.zeros(4, device="cuda")
    q.qc_encode_ef(x, None, 0, 8, 512, 0, 0, 0, 0, x, x, x)


# ------------------------------------------------------------------ decode

DEC_CASES = [(0, 1), (0, 2), (0, 4), (0, 8), (1, 1), (2, 2)]


@pytest.mark.parametrize("scheme,bits", DEC_CASES)
@pytest.mark.parametrize("M", [1, 3, 16])
def test_decode_accumulate(q, scheme, bits, M):
    rng = np.random.default_rng(100 * M + bits)
    for bucket, aligned in ((32, True), (96, True), (512, True), (1024, True), (4096, True),
                            (512, False), (1024, False)):
        n = max(3 * bucket, 3000) + 13
        words, nb = orc.code_words(n, bits), orc.num_buckets(n, bucket)
        # padded worker strides: a multiple of 4 words takes the pipelined
        # kernel, an odd stride the direct one
        cstride = words + (-words) % 4 + 4 if aligned else words + 5
        mstride = nb + 3
        codes = rng.integers(0, 1 << 32, size=(M, cstride), dtype=np.uint64).astype(np.uint32)
        scale = (rng.random((M, mstride)) * 1e-3).astype(np.float32)
        offset = (rng.standard_normal((M, mstride)) * 1e-2).astype(np.float32)
        prior = rng.standard_normal(n).astype(np.float32)
        for flags in (0, 1, 3):
            out = torch.from_numpy(prior.copy()).cuda()
            q.qc_decode_accumulate(dev(codes), cstride, dev(scale),
                                   dev(offset) if scheme == 0 else None, mstride, M, n, bits,
                                   bucket, scheme, out, flags)
            want = orc.decode_accumulate(codes, scale, offset if scheme == 0 else None, M=M, n=n,
                                         bits=bits, bucket=bucket, scheme=scheme, flags=flags,
                                         codes_stride_words=cstride, meta_stride=mstride,
                                         out=prior.copy())
            assert_bits_equal(host(out), want,
                              f"decode s={scheme} b={bits} M={M} B={bucket} f={flags} al={aligned}")


def test_decode_guards(q):
    n, bucket, M = 4096 + 7, 512, 4
    rng = np.random.default_rng(3)
    words, nb = orc.code_words(n, 8), orc.num_buckets(n, bucket)
    codes = rng.integers(0, 1 << 32, size=(M, words), dtype=np.uint64).astype(np.uint32)
    scale = rng.random((M, nb)).astype(np.float32)
    offset = rng.random((M, nb)).astype(np.float32)
    out = Guarded(n, torch.float32, guard=256)
    q.qc_decode_accumulate(dev(codes), words, dev(scale), dev(offset), nb, M, n, 8, bucket, 0,
                           out.t, 1)
    torch.cuda.synchronize()
    out.check()
    want = orc.decode_accumulate(codes, scale, offset, M=M, n=n, bits=8, bucket=bucket,
                                 scheme=0, flags=1)
    assert_bits_equal(host(out.t), want)


# -------------------------------------------------------------------- vote

@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 7, 8, 9, 16, 33, 128])
def test_sign_vote(q, M):
    rng = np.random.default_rng(M)
    for n in (1, 31, 32, 100, 4096, 4096 * 5 + 17):
        words = orc.code_words(n, 1)
        for stride in (words + (-words) % 4, words + 1 if M > 1 else words):
            signs = rng.integers(0, 1 << 32, size=(M, stride), dtype=np.uint64).astype(np.uint32)
            out = Guarded(words, torch.int32)
            q.qc_sign_vote(dev(signs), stride, M, n, out.t)
            torch.cuda.synchronize()
            out.check()
            want = orc.sign_vote(signs, M=M, n=n, stride_words=stride)
            assert_bits_equal(u32(out.t), want, f"vote M={M} n={n} stride={stride}")


# --------------------------------------------------------------------- FP8

@pytest.mark.parametrize("dim", [4, 36, 64, 128, 132, 512, 1000, 2052, 4096])
def test_rowwise_fp8(q, dim):
    for rows in (1, 5, 1031):
        x = wl.embedding_rows(rows=rows, dim=dim, seed=dim + rows).copy()
        if rows > 4:
            x[1] = 0.0                                        # zero row
            x[2, dim // 2] = np.float32(1e30)                 # one huge value
            x[3] *= np.float32(1e-38)                         # subnormal scale
            x[4] = -np.abs(x[4])                              # all negative
        if rows > 6:
            x[5] = np.float32(np.nan)                         # NaN row: its maximum is +0
            x[6, : (dim + 1) // 2] = np.float32(np.nan)       # NaN elements are left out of the maximum
        codes = Guarded(rows * dim, torch.uint8, fill=0xA5)
        sc = Guarded(rows, torch.float32)
        q.qc_rowwise_fp8(dev(x), rows, dim, codes.t, sc.t)
        torch.cuda.synchronize()
        codes.check()
        sc.check()
        c_or, s_or = orc.rowwise_fp8(x)
        assert_bits_equal(host(codes.t), c_or.reshape(-1), f"fp8 codes dim={dim} rows={rows}")
        assert_bits_equal(host(sc.t), s_or, f"fp8 scale dim={dim} rows={rows}")
        out = Guarded(rows * dim, torch.float32)
        q.qc_rowwise_fp8_dequant(dev(c_or), dev(s_or), rows, dim, out.t)
        torch.cuda.synchronize()
        out.check()
        want = orc.rowwise_fp8_dequant(c_or, s_or).reshape(-1)
        got = host(out.t)
        nan = np.isnan(want)                                  # NaN codes: any NaN pattern
        assert np.array_equal(np.isnan(got), nan), f"fp8 dequant NaNs dim={dim} rows={rows}"
        assert_bits_equal(got[~nan], want[~nan], f"fp8 dequant dim={dim} rows={rows}")


def test_fp8_dequant_all_codes(q):
    """Every byte value, including both NaN encodings, decodes as the spec says."""
    rows, dim = 4, 64
    c = np.arange(256, dtype=np.uint8).reshape(rows, dim)
    s = np.array([1.0, 0.5, 3.0, 1e-3], dtype=np.float32)
    out = torch.empty(rows * dim, dtype=torch.float32, device="cuda")
    q.qc_rowwise_fp8_dequant(dev(c), dev(s), rows, dim, out)
    got = host(out).reshape(rows, dim)
    want = orc.rowwise_fp8_dequant(c, s)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert_bits_equal(got[~nan], want[~nan])


def test_encode_largest_bucket(q):
    """bucket = 2^24, the largest accepted: one two-pass bucket plus a ragged one."""
    bucket = 1 << 24
    n = bucket + 4099
    g = wl.outlier_gradient(n, seed=13)
    err0 = np.zeros(n, dtype=np.float32)
    codes, scale, offset, err = _run_encode(q, g, err0, n, 8, bucket, q.QC_SCHEME_UNIFORM, 1)
    e_or = err0.copy()
    c_or, s_or, o_or = orc.encode_uniform(g, e_or, bits=8, bucket=bucket, mode=1, seed=SEED,
                                          step=STEP)
    assert_bits_equal(codes, c_or, "codes")
    assert_bits_equal(scale, s_or, "scale")
    assert_bits_equal(offset, o_or, "offset")
    assert_bits_equal(err, e_or, "err")


def test_most_workers(q):
    """M = 1024 (the largest accepted) for decode and vote."""
    M, n, bucket = q.QC_MAX_WORKERS, 4096 + 32, 1024
    rng = np.random.default_rng(5)
    words, nb = orc.code_words(n, 8), orc.num_buckets(n, bucket)
    codes = rng.integers(0, 1 << 32, size=(M, words), dtype=np.uint64).astype(np.uint32)
    scale = (rng.random((M, nb)) * 1e-3).astype(np.float32)
    offset = (rng.standard_normal((M, nb)) * 1e-3).astype(np.float32)
    out = torch.empty(n, device="cuda")
    q.qc_decode_accumulate(dev(codes), words, dev(scale), dev(offset), nb, M, n, 8, bucket, 0,
                           out, 1)
    want = orc.decode_accumulate(codes, scale, offset, M=M, n=n, bits=8, bucket=bucket,
                                 scheme=0, flags=1)
    assert_bits_equal(host(out), want, "decode M=1024")
    sw = orc.code_words(n, 1)
    signs = rng.integers(0, 1 << 32, size=(M, sw), dtype=np.uint64).astype(np.uint32)
    vote = torch.empty(sw, dtype=torch.int32, device="cuda")
    q.qc_sign_vote(dev(signs), sw, M, n, vote)
    assert_bits_equal(u32(vote), orc.sign_vote(signs, M=M, n=n), "vote M=1024")


def test_encode_ternary_bf16_near_draws(q):
    """The bf16 ternary kernel decides keep = [u < |p| / s] division-free and
    falls back to the exact path when u and |p| / s are within 2^-21.  Buckets
    with s = 1 make |p| / s = |p|; every element whose draw u is below 2^-12 gets
    |p| = u rounded to bf16 (or one bf16 step either side), which lands within
    reach of the fallback and sometimes exactly on u."""
    bucket, nb = 1024, 256
    n = bucket * nb
    g = (wl.std_normal(41, 1, n) * np.float32(0.2)).astype(np.float32)
    g = np.clip(g, -0.9, 0.9)
    g[::bucket] = 1.0                                   # s = max|p| = 1 in every bucket
    u = np.array([orc.uniform(SEED, STEP, i) for i in range(n)], dtype=np.float32)
    small = np.flatnonzero((u < 2.0 ** -12) & (np.arange(n) % bucket != 0))
    assert small.size > 20
    gb = wl.to_bf16_bits(g)
    ub = wl.to_bf16_bits(u[small])
    side = (np.arange(small.size) % 3).astype(np.int32) - 1   # -1, 0, +1 bf16 steps
    gb[small] = (ub.astype(np.int32) + side).astype(np.uint16)
    exact_hits = int((wl.bf16_bits_to_f32(gb[small]) == u[small]).sum())
    codes, scale, _, _ = _run_encode(q, gb, None, n, 2, bucket, q.QC_SCHEME_TERNARY, 1)
    c_or, s_or = orc.encode_ternary(gb, None, bucket=bucket, mode=orc.ROUND_STOCHASTIC,
                                    seed=SEED, step=STEP)
    assert np.all(s_or == 1.0)
    assert_bits_equal(codes, c_or, f"ternary bf16 near draws ({small.size} planted, "
                                   f"{exact_hits} exactly on u)")


def test_decode_after_a_worker_drops_out(q):
    """A worker that fails before sending: the receiver decodes the M - 1
    payloads that arrived (gathered contiguously on the host), and the result is
    the oracle's over the same M - 1 workers in their order."""
    M, n, bits, bucket = 6, 20_000 + 9, 8, 1024
    payloads = [orc.encode_uniform(wl.outlier_gradient(n, seed=300 + w), bits=bits, bucket=bucket)
                for w in range(M)]
    dropped = 2
    kept = [payloads[w] for w in range(M) if w != dropped]
    codes = np.stack([c for c, _, _ in kept])
    scale = np.stack([s for _, s, _ in kept])
    offset = np.stack([o for _, _, o in kept])
    out = torch.empty(n, device="cuda")
    q.qc_decode_accumulate(dev(codes), codes.shape[1], dev(scale), dev(offset), scale.shape[1],
                           M - 1, n, bits, bucket, 0, out, q.QC_OUT_MEAN)
    want = orc.decode_accumulate(codes, scale, offset, M=M - 1, n=n, bits=bits, bucket=bucket,
                                 scheme=0, flags=orc.OUT_MEAN)
    assert_bits_equal(host(out), want, "decode without worker 2")


def _unpack_codes(words, n, bits):
    per = 32 // bits
    sh = (np.arange(per, dtype=np.uint32) * bits).astype(np.uint32)
    return ((words[:, None] >> sh[None, :]) & np.uint32((1 << bits) - 1)).reshape(-1)[:n]


_NAN_CASES = [("uniform", 1), ("uniform", 2), ("uniform", 4), ("uniform", 8), ("ternary", 2),
              ("qsgd", 2), ("qsgd", 4), ("qsgd", 8), ("log", 2), ("log", 4), ("log", 8)]


@pytest.mark.parametrize("scheme,bits", _NAN_CASES)
@pytest.mark.parametrize("dtype,ef,bucket", [("f32", True, 512), ("f32", False, 4096),
                                             ("bf16", False, 1024), ("f32", True, 8192)])
@pytest.mark.parametrize("mode", [0, 1], ids=["nearest", "stochastic"])
def test_nan_element_keeps_to_its_own_field(q, scheme, bits, dtype, ef, bucket, mode):
    """A NaN inside a packed word (never a bucket's first element, whose value the
    oracle's running min/max starts from) gives an unspecified code for that
    element only: every other element's code, every bucket's metadata and every
    other residual match the oracle bit for bit, in the pipelined fp32 kernel,
    the bf16 kernel and the two-pass direct kernel."""
    sch = {"uniform": q.QC_SCHEME_UNIFORM, "ternary": q.QC_SCHEME_TERNARY,
           "qsgd": q.QC_SCHEME_QSGD, "log": q.QC_SCHEME_LOG}[scheme]
    n = 3 * bucket + 100
    gf = wl.outlier_gradient(n, seed=4242 + bits)
    nan_at = np.array([5, bucket + 33, 2 * bucket + bucket // 2 + 1])
    gf[nan_at] = np.float32(np.nan)
    g = wl.to_bf16_bits(gf) if dtype == "bf16" else gf
    err0 = (wl.std_normal(17, 1, n) * np.float32(1e-4)) if ef else None
    codes, scale, offset, err = _run_encode(q, g, err0, n, bits, bucket, sch, mode)
    e_or = err0.copy() if ef else None
    kw = dict(bucket=bucket, mode=mode, seed=SEED, step=STEP)
    if scheme == "uniform":
        c_or, s_or, o_or = orc.encode_uniform(g, e_or, bits=bits, **kw)
        assert_bits_equal(offset, o_or, "offset")
    elif scheme == "ternary":
        c_or, s_or = orc.encode_ternary(g, e_or, **kw)
    elif scheme == "qsgd":
        c_or, s_or = orc.encode_qsgd(g, e_or, bits=bits, **kw)
    else:
        c_or, s_or = orc.encode_log(g, e_or, bits=bits, **kw)
    assert_bits_equal(scale, s_or, "scale")
    keep = np.ones(n, dtype=bool)
    keep[nan_at] = False
    cg, co = _unpack_codes(codes, n, bits), _unpack_codes(c_or, n, bits)
    bad = np.flatnonzero(keep & (cg != co))
    assert bad.size == 0, [(int(i), int(cg[i]), int(co[i])) for i in bad[:8]]
    if ef:
        assert_bits_equal(err[keep], e_or[keep], "residual")


@pytest.mark.parametrize("scheme,bits,mode", [("uniform", 8, 0), ("uniform", 4, 1), ("ternary", 2, 1),
                                              ("uniform", 2, 0), ("uniform", 1, 0)])
@pytest.mark.parametrize("bucket", [1024, 2048])
def test_bf16_tails_of_every_length(q, scheme, bits, mode, bucket):
    """bf16 gradients whose last bucket holds 1 .. 9 elements past a multiple of
    8 (and a word offset of the code buffer that is 4- but not 8-byte aligned):
    codes, metadata and the canaries after the last code word match the
    oracle, in the receiver kernels for buckets of 1024 and the general bf16
    kernel for 2048."""
    sch = q.QC_SCHEME_UNIFORM if scheme == "uniform" else q.QC_SCHEME_TERNARY
    for r in range(1, 10):
        n = 2 * bucket + 8 * 5 + r
        g = wl.to_bf16_bits(wl.outlier_gradient(n, seed=300 + r))
        codes, scale, offset, _ = _run_encode(q, g, None, n, bits, bucket, sch, mode)
        if scheme == "uniform":
            c_or, s_or, o_or = orc.encode_uniform(g, None, bits=bits, bucket=bucket, mode=mode,
                                                  seed=SEED, step=STEP)
            assert_bits_equal(offset, o_or, f"offset r={r}")
        else:
            c_or, s_or = orc.encode_ternary(g, None, bucket=bucket, mode=mode, seed=SEED, step=STEP)
        assert_bits_equal(codes, c_or, f"codes r={r}")
        assert_bits_equal(scale, s_or, f"scale r={r}")
    # a code buffer one word into an 8-byte aligned allocation
    n = 3 * bucket + 13
    g = wl.to_bf16_bits(wl.outlier_gradient(n, seed=399))
    words, nb = q.qc_code_words(n, bits), q.qc_num_buckets(n, bucket)
    base = torch.full((words + 2,), -7, dtype=torch.int32, device="cuda")
    codes = base[1:1 + words]
    assert codes.data_ptr() % 8 == 4
    scale = torch.empty(nb, device="cuda")
    offset = torch.empty(nb, device="cuda") if scheme == "uniform" else None
    q.qc_encode_ef(dev(g), None, n, bits, bucket, sch, mode, SEED, STEP, codes, scale, offset,
                   dtype=q.QC_DTYPE_BF16)
    torch.cuda.synchronize()
    if scheme == "uniform":
        c_or, _, _ = orc.encode_uniform(g, None, bits=bits, bucket=bucket, mode=mode, seed=SEED,
                                        step=STEP)
    else:
        c_or, _ = orc.encode_ternary(g, None, bucket=bucket, mode=mode, seed=SEED, step=STEP)
    assert_bits_equal(u32(codes), c_or, "codes at a 4-byte offset")
    b = host(base)
    assert b[0] == -7 and b[-1] == -7

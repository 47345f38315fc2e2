"""GPU <-> oracle parity for the QSGD scheme (per-bucket L2 norm, s = 2^(b-1) - 1
levels under a sign bit).

The norm is the binary32 rounding of the square root of the exact sum of
squares on both sides: the oracle computes it with a wide integer, the kernels
from a double-word sum with a proven error bound, falling back to an exact
wide-integer path for buckets within that bound of a rounding boundary.  Units,
codes and residuals must therefore be bit-identical in every bucket.  The
tests plant buckets whose exact norm lies within 2^-90 of a rounding boundary,
on either side and exactly on it, so that the exact path runs, and buckets
whose squares leave the binary32 range of the fast path.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle as orc
import workloads as wl
from tests._gpu import assert_bits_equal, dev, host, u32
from tests._norm_cases import midpoint_bucket

pytestmark = pytest.mark.gpu

SEED = 0x0FED_CBA9_8765_4321
STEP = 11


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
    return ((words[:, None] >> sh[None, :]) & np.uint32((1 << bits) - 1)).reshape(-1)[:n]


def _p_of(g, err0):
    gf = wl.bf16_bits_to_f32(g) if g.dtype == np.uint16 else g
    return gf.astype(np.float32) if err0 is None else (err0 + gf).astype(np.float32)


def _encode(q, g, err0, n, bits, bucket, mode, grad_t=None):
    words, nb = q.qc_code_words(n, bits), q.qc_num_buckets(n, bucket)
    codes = torch.full((words,), -7, dtype=torch.int32, device="cuda")
    unit = torch.full((nb,), -7.0, device="cuda")
    err = torch.from_numpy(err0.copy()).cuda() if err0 is not None else None
    dtype = q.QC_DTYPE_BF16 if g.dtype == np.uint16 else q.QC_DTYPE_F32
    gt = dev(g) if grad_t is None else grad_t
    q.qc_encode_ef(gt, err, n, bits, bucket, q.QC_SCHEME_QSGD, mode, SEED, STEP, codes, unit,
                   None, dtype=dtype)
    torch.cuda.synchronize()
    return u32(codes), host(unit), (host(err) if err is not None else None)


def check_qsgd(got, want, p, n, bits, bucket, tag):
    """Units, codes and residuals bit-identical to the oracle's; level range and
    sign bit checked on their own as well."""
    codes, unit, err = got
    c_or, u_or, e_or = want
    s = (1 << (bits - 1)) - 1
    assert_bits_equal(unit, u_or, tag + " unit")
    cg, co = _unpack(codes, n, bits), _unpack(c_or, n, bits)
    bad = np.flatnonzero(cg != co)
    assert bad.size == 0, (tag, "codes", [(int(i), int(cg[i]), int(co[i])) for i in bad[:5]])
    assert_bits_equal(codes, c_or, tag + " code words")
    lvl = cg & np.uint32(s)
    neg = cg >> np.uint32(bits - 1)
    assert np.all(lvl <= s), tag
    assert np.array_equal(neg.astype(bool), p < 0), (tag, "sign bit")
    if err is not None:
        assert_bits_equal(err, e_or, tag + " err")


BUCKETS = [32, 96, 512, 1024, 2048, 4096, 8192]


@pytest.mark.parametrize("ef", [False, True])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("mode", [0, 1], ids=["nearest", "stochastic"])
@pytest.mark.parametrize("bits", [2, 4, 8])
def test_encode_qsgd(q, bits, mode, dtype, ef):
    for bucket in BUCKETS:
        n = max(5 * bucket, 6000) + 37
        gf = wl.outlier_gradient(n, seed=7 * bucket + bits)
        if dtype == "f32":
            gf[bucket:2 * bucket] = 0.0           # an all-zero bucket: unit 0, codes 0
        g = wl.to_bf16_bits(gf) if dtype == "bf16" else gf
        err0 = (wl.std_normal(96, 1, n) * np.float32(1e-4)) if ef else None
        got = _encode(q, g, err0, n, bits, bucket, mode)
        e_or = err0.copy() if ef else None
        c_or, u_or = orc.encode_qsgd(g, e_or, bits=bits, bucket=bucket, mode=mode, seed=SEED,
                                     step=STEP)
        check_qsgd(got, (c_or, u_or, e_or), _p_of(g, err0), n, bits, bucket,
                   f"qsgd b={bits} mode={mode} {dtype} ef={ef} B={bucket}")


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_encode_qsgd_degenerate(q, bits):
    """Zero and +-0 buckets, one non-zero element (it takes the top level), a
    constant bucket, tiny and huge magnitudes."""
    bucket = 512
    n = 8 * bucket + 5
    g = wl.std_normal(8, 1, n) * np.float32(1e-3)
    g[0:bucket] = 0.0
    g[bucket:2 * bucket] = np.where(np.arange(bucket) % 2, 0.0, -0.0).astype(np.float32)
    g[2 * bucket:3 * bucket] = 0.0
    g[2 * bucket + 17] = np.float32(-30.0)
    g[3 * bucket:4 * bucket] = np.float32(0.25)
    g[4 * bucket:5 * bucket] *= np.float32(1e-8)     # norm ~ 2e-11
    g[5 * bucket:6 * bucket] *= np.float32(1e17)     # norm ~ 2e15
    for mode in (0, 1):
        err0 = np.zeros(n, dtype=np.float32)
        got = _encode(q, g, err0, n, bits, bucket, mode)
        e_or = err0.copy()
        c_or, u_or = orc.encode_qsgd(g, e_or, bits=bits, bucket=bucket, mode=mode, seed=SEED,
                                     step=STEP)
        assert u_or[0] == 0 and u_or[1] == 0
        check_qsgd(got, (c_or, u_or, e_or), _p_of(g, err0), n, bits, bucket,
                   f"qsgd degenerate b={bits} m={mode}")
        codes = _unpack(got[0], n, bits)
        s = (1 << (bits - 1)) - 1
        assert np.all(codes[:2 * bucket] == 0)
        assert codes[2 * bucket + 17] == (1 << (bits - 1)) | s   # -|v| = -||v||: top level


def _boundary_gradient(bits, bucket):
    """One bucket per boundary value: t = k and t = k + 1/2 (k = 0 .. s-1) and one
    ulp either side, each in its own bucket over small random elements (the
    squares of a bucket's t values cannot exceed s^2).  Each boundary element
    depends on its bucket's unit and the unit on the element, so the values are
    re-derived from the oracle's units until they stop changing."""
    s = (1 << (bits - 1)) - 1
    targets = [k + f for k in range(s) for f in (0.0, 0.5) if k + f > 0]
    nb = 3 * len(targets)
    rng = np.random.default_rng(bits)
    g = (rng.standard_normal(nb * bucket) * 0.01).astype(np.float32)
    slot = np.arange(nb) * bucket + 37
    sign = np.where(np.arange(nb) % 2, -1.0, 1.0).astype(np.float32)
    t = np.repeat(np.array(targets), 3)
    side = np.tile(np.array([0, 1, -1]), len(targets))
    for _ in range(80):
        _, unit = orc.encode_qsgd(g, None, bits=bits, bucket=bucket, mode=0)
        v = (t * unit.astype(np.float64)).astype(np.float32)
        v = np.where(side > 0, np.nextafter(v, np.float32(np.inf)),
                     np.where(side < 0, np.nextafter(v, np.float32(-np.inf)), v))
        new = g.copy()
        new[slot] = v.astype(np.float32) * sign
        if np.array_equal(new, g):
            break
        g = new
    _, unit = orc.encode_qsgd(g, None, bits=bits, bucket=bucket, mode=0)
    on = np.abs(g[slot]) == (t * unit.astype(np.float64)).astype(np.float32)
    return g, on, side


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_encode_qsgd_decision_boundaries(q, bits):
    """Elements exactly on every decision boundary of the level (ties of rint,
    integer t for the floor of stochastic rounding) and one ulp either side."""
    bucket = 256
    g, on, side = _boundary_gradient(bits, bucket)
    assert on[side == 0].mean() >= 0.9, "the boundary construction did not settle"
    n = g.size
    for mode in (0, 1):
        err0 = np.zeros(n, dtype=np.float32)
        got = _encode(q, g, err0, n, bits, bucket, mode)
        e_or = err0.copy()
        c_or, u_or = orc.encode_qsgd(g, e_or, bits=bits, bucket=bucket, mode=mode, seed=SEED,
                                     step=STEP)
        check_qsgd(got, (c_or, u_or, e_or), _p_of(g, err0), n, bits, bucket,
                   f"qsgd boundaries b={bits} m={mode}")


def _planted_norm_buckets(bucket, rng, bf16=False):
    """Buckets whose exact norm sits within 2^-90 (relative) below, above, or
    (where the construction closes exactly) on a midpoint between two binary32
    values, over several magnitudes, each padded with zeros; plus (fp32) one
    bucket of the exact tie 1 + 2^-24 and one with a subnormal element more."""
    out = []
    for f in (1.0, 3.7, 0.1, 1e-20, 2.5e15, 7.0e-30, 6.0e18, 1.0e-3, 12345.678):
        for side in ("below", "above"):
            vals, _ = midpoint_bucket(f, steps=14 if bf16 else 4, side=side, bf16=bf16)
            b = np.zeros(bucket, dtype=np.float32)
            pos = rng.permutation(bucket)[:len(vals)]
            b[pos] = vals * np.where(rng.random(len(vals)) < 0.5, -1, 1).astype(np.float32)
            out.append(b)
    if not bf16:
        b = np.zeros(bucket, dtype=np.float32)
        b[[3, 40, 41, bucket - 1]] = [1.0, 2.0 ** -12, -(2.0 ** -12), 2.0 ** -24]  # norm 1 + 2^-24
        out.append(b)
        b = b.copy()
        b[7] = np.float32(2.0 ** -149)                                            # just above it
        out.append(b)
    return np.concatenate(out)


@pytest.mark.parametrize("bits", [2, 4, 8])
@pytest.mark.parametrize("path", ["tma", "direct", "bf16"])
def test_encode_qsgd_norm_on_rounding_boundaries(q, bits, path):
    """Buckets planted on the rounding boundaries of the norm take the exact
    path; every unit, code and residual matches the oracle bit for bit: the
    pipelined fp32 kernel with error feedback (buckets of 512, one warp, and
    4096, eight warps), the two-pass direct kernel (buckets of 8192) and the bf16
    kernel without error feedback (buckets of 1024 and 2048, planted with bf16
    values)."""
    rng = np.random.default_rng(77 + bits)
    buckets = {"tma": (512, 4096), "direct": (8192,), "bf16": (1024, 2048)}[path]
    for bucket in buckets:
        g = _planted_norm_buckets(bucket, rng, bf16=path == "bf16")
        if path == "bf16":
            g = wl.to_bf16_bits(g)
        n = g.size
        for mode in (0, 1):
            err0 = np.zeros(n, dtype=np.float32) if path != "bf16" else None
            got = _encode(q, g, err0, n, bits, bucket, mode)
            e_or = err0.copy() if err0 is not None else None
            c_or, u_or = orc.encode_qsgd(g, e_or, bits=bits, bucket=bucket, mode=mode,
                                         seed=SEED, step=STEP)
            check_qsgd(got, (c_or, u_or, e_or), _p_of(g, err0), n, bits, bucket,
                       f"planted norms b={bits} {path} B={bucket} m={mode}")


@pytest.mark.parametrize("bits", [4, 8])
def test_encode_qsgd_norm_outside_the_fast_range(q, bits):
    """Buckets whose sum of squares lies below 2^-60 or above 2^124 (subnormal
    elements, norms near 2^-70 and 2^63, and their mix) go through the exact
    path: bit-identical to the oracle."""
    bucket = 512
    rng = np.random.default_rng(5 + bits)
    parts = []
    for scale in (2.0 ** -140, 2.0 ** -100, 2.0 ** -75, 2.0 ** 55, 2.0 ** 60):
        parts.append((rng.standard_normal(bucket) * scale).astype(np.float32))
    mix = (rng.standard_normal(bucket) * 2.0 ** -80).astype(np.float32)
    mix[rng.integers(0, bucket, 16)] = np.float32(2.0 ** -149) * rng.integers(1, 50, 16)
    parts.append(mix)
    g = np.concatenate(parts)
    n = g.size
    for mode in (0, 1):
        err0 = np.zeros(n, dtype=np.float32)
        got = _encode(q, g, err0, n, bits, bucket, mode)
        e_or = err0.copy()
        c_or, u_or = orc.encode_qsgd(g, e_or, bits=bits, bucket=bucket, mode=mode, seed=SEED,
                                     step=STEP)
        check_qsgd(got, (c_or, u_or, e_or), _p_of(g, err0), n, bits, bucket,
                   f"extreme norms b={bits} m={mode}")


@pytest.mark.parametrize("bits", [4, 8])
def test_encode_qsgd_bf16_unaligned_and_two_pass(q, bits):
    """An 8- but not 16-byte aligned bf16 gradient (direct kernel) and a bucket
    too large for one pass over registers (two-pass direct kernel)."""
    bucket, n = 1024, 1024 * 9 + 20
    g = wl.to_bf16_bits(wl.outlier_gradient(n, seed=23))
    base = torch.zeros(n + 8, dtype=torch.int16, device="cuda")
    view = base[4:4 + n]
    view.copy_(torch.from_numpy(g.view(np.int16)).cuda())
    assert view.data_ptr() % 16 == 8
    err0 = np.zeros(n, dtype=np.float32)
    got = _encode(q, g, err0, n, bits, bucket, 1, grad_t=view)
    e_or = err0.copy()
    c_or, u_or = orc.encode_qsgd(g, e_or, bits=bits, bucket=bucket, mode=1, seed=SEED, step=STEP)
    check_qsgd(got, (c_or, u_or, e_or), wl.bf16_bits_to_f32(g), n, bits, bucket, "bf16 unaligned")

    bucket = 1 << 16
    n = 3 * bucket + 1001
    gf = wl.outlier_gradient(n, seed=29)
    err0 = (wl.std_normal(95, 1, n) * np.float32(1e-4))
    got = _encode(q, gf, err0, n, bits, bucket, 1)
    e_or = err0.copy()
    c_or, u_or = orc.encode_qsgd(gf, e_or, bits=bits, bucket=bucket, mode=1, seed=SEED, step=STEP)
    check_qsgd(got, (c_or, u_or, e_or), _p_of(gf, err0), n, bits, bucket, "two-pass")


@pytest.mark.parametrize("bits", [2, 4, 8])
@pytest.mark.parametrize("M", [1, 4, 16])
def test_decode_qsgd(q, bits, M):
    """Random code words (every code is a valid QSGD code) and random units,
    pipelined (stride a multiple of 4 words) and direct (odd stride)."""
    rng = np.random.default_rng(1000 * M + bits)
    for bucket, aligned in ((32, True), (512, True), (4096, True), (512, False)):
        n = max(3 * bucket, 3000) + 13
        words, nb = orc.code_words(n, bits), orc.num_buckets(n, bucket)
        cstride = words + (-words) % 4 + 4 if aligned else words + 5
        mstride = nb + 3
        codes = rng.integers(0, 1 << 32, size=(M, cstride), dtype=np.uint64).astype(np.uint32)
        unit = (rng.random((M, mstride)) * 1e-3).astype(np.float32)
        prior = rng.standard_normal(n).astype(np.float32)
        for flags in (0, 1, 3):
            out = torch.from_numpy(prior.copy()).cuda()
            q.qc_decode_accumulate(dev(codes), cstride, dev(unit), None, mstride, M, n, bits,
                                   bucket, q.QC_SCHEME_QSGD, out, flags)
            want = orc.decode_accumulate(codes, unit, None, M=M, n=n, bits=bits, bucket=bucket,
                                         scheme=orc.SCHEME_QSGD, flags=flags,
                                         codes_stride_words=cstride, meta_stride=mstride,
                                         out=prior.copy())
            assert_bits_equal(host(out), want, f"decode qsgd b={bits} M={M} B={bucket} f={flags}")


def test_qsgd_round_trip_unbiased_on_gpu(q):
    """Stochastic QSGD is unbiased: over many steps the mean decoded value of
    each element converges to the element (checked with a 6-sigma bound from
    the per-element variance unit^2 / 4)."""
    bits, bucket, n, steps = 4, 256, 4096, 400
    g = wl.std_normal(31, 1, n).astype(np.float32)
    gd = dev(g)
    words, nb = q.qc_code_words(n, bits), q.qc_num_buckets(n, bucket)
    codes = torch.empty((steps, words), dtype=torch.int32, device="cuda")
    unit = torch.empty((steps, nb), device="cuda")
    for t in range(steps):
        q.qc_encode_ef(gd, None, n, bits, bucket, q.QC_SCHEME_QSGD, q.QC_ROUND_STOCHASTIC, SEED,
                       t, codes[t], unit[t], None)
    out = torch.empty(n, device="cuda")
    q.qc_decode_accumulate(codes, words, unit, None, nb, steps, n, bits, bucket,
                           q.QC_SCHEME_QSGD, out, q.QC_OUT_MEAN)
    u = host(unit)[0]
    sd = np.repeat(u, bucket)[:n] / 2 / np.sqrt(steps)
    assert np.all(np.abs(host(out) - g) <= 6 * sd + 1e-7)

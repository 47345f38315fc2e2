"""GPU <-> oracle parity for the QSGD scheme (per-bucket L2 norm, s = 2^(b-1) - 1
levels under a sign bit).

The norm is the one float the two sides may round differently: the oracle sums
the squares in fp64, the kernels in a double word, so a bucket whose norm lies
within about 2^-40 of a binary32 rounding boundary may come out one ulp apart.
The tests therefore require every unit within one ulp of the oracle's, at most
one bucket in a hundred (in practice none) not bit-identical, and, in every
bucket whose unit is bit-identical, codes and residuals bit-identical too.  In
every bucket the residual must equal p - deq(code, unit) for the kernel's own
code and unit, the level must not exceed s and the sign bit must be [p < 0].
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle as orc
import workloads as wl
from tests._gpu import assert_bits_equal, dev, host, u32

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
    codes, unit, err = got
    c_or, u_or, e_or = want
    s = (1 << (bits - 1)) - 1
    nb = u_or.size
    ui = unit.view(np.int32).astype(np.int64)
    uo = u_or.view(np.int32).astype(np.int64)
    assert np.all(np.abs(ui - uo) <= 1), (tag, "unit more than one ulp off",
                                          np.flatnonzero(np.abs(ui - uo) > 1)[:5])
    same_b = ui == uo
    assert (~same_b).sum() <= max(1, nb // 100), (tag, "too many units differ", (~same_b).sum())
    same = np.repeat(same_b, bucket)[:n]
    cg, co = _unpack(codes, n, bits), _unpack(c_or, n, bits)
    bad = np.flatnonzero(same & (cg != co))
    assert bad.size == 0, (tag, "codes", [(int(i), int(cg[i]), int(co[i])) for i in bad[:5]])
    # validity everywhere: level range, sign bit, and the residual from the
    # kernel's own code and unit
    lvl = cg & np.uint32(s)
    neg = cg >> np.uint32(bits - 1)
    assert np.all(lvl <= s), tag
    assert np.array_equal(neg.astype(bool), p < 0), (tag, "sign bit")
    if err is not None:
        u_el = np.repeat(unit, bucket)[:n]
        mag = (lvl.astype(np.float32) * u_el).astype(np.float32)
        deq = np.where(neg.astype(bool), -mag, mag).astype(np.float32)
        assert_bits_equal(err, (p - deq).astype(np.float32), tag + " err vs own code")
        assert_bits_equal(err[same], e_or[same], tag + " err")


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
    constant bucket, tiny and huge magnitudes inside the supported norm range."""
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

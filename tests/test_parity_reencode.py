"""GPU <-> oracle parity for the receiver re-encode (decode and accumulate M
payloads, then encode the result with the receiver's own residual).

The decoded result r must match the oracle bit for bit.  The new payload and
residual must match bit for bit for the uniform and ternary schemes; the sign
scheme's mean |p| is compared within 1e-6 * max|p| of its bucket (its only
freedom is the order of the sum); QSGD's unit, codes and residuals are
bit-identical (its norm is the exactly rounded one on both sides).
Worker counts cover one chunk per stage and several; buckets cover one warp,
teams and the largest supported bucket; every n leaves a ragged tail.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle as orc
import workloads as wl
from tests._gpu import assert_bits_equal, assert_close_per_bucket, dev, host, u32
from tests.test_parity_qsgd import check_qsgd

pytestmark = pytest.mark.gpu

SEED = 0x5EED_0000_1111_2222
STEP = 3


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


def _payloads(rng, scheme, bits, M, n, bucket):
    """Random code words (any word is a valid payload) and metadata, worker
    strides padded to a multiple of 4 words."""
    words, nb = orc.code_words(n, bits), orc.num_buckets(n, bucket)
    cstride = words + (-words) % 4 + 4
    mstride = nb + 3
    codes = rng.integers(0, 1 << 32, size=(M, cstride), dtype=np.uint64).astype(np.uint32)
    if scheme == orc.SCHEME_TERNARY:
        # a ternary field is 0, 1 or 2; 3 is not a code
        f = _unpack(codes, M * cstride * 16, 2)
        f = np.where(f == 3, 1, f).astype(np.uint32)
        codes = _pack(f, 2).reshape(M, cstride)
    scale = (rng.random((M, mstride)) * 1e-2).astype(np.float32)
    offset = (rng.standard_normal((M, mstride)) * 1e-2).astype(np.float32)
    return codes, cstride, scale, offset, mstride


def _unpack(words, n, bits):
    per = 32 // bits
    sh = (np.arange(per, dtype=np.uint32) * bits).astype(np.uint32)
    return ((words.reshape(-1)[:, None] >> sh[None, :]) & np.uint32((1 << bits) - 1)).reshape(-1)[:n]


def _pack(vals, bits):
    per = 32 // bits
    v = vals.reshape(-1, per).astype(np.uint32)
    out = np.zeros(v.shape[0], dtype=np.uint32)
    for j in range(per):
        out |= v[:, j] << np.uint32(j * bits)
    return out


def _run(q, scheme, bits, M, n, bucket, flags, ef, mode, want_out, rng):
    codes, cstride, scale, offset, mstride = _payloads(rng, scheme, bits, M, n, bucket)
    uni = scheme == orc.SCHEME_UNIFORM
    words, nb = orc.code_words(n, bits), orc.num_buckets(n, bucket)
    err0 = (wl.std_normal(int(rng.integers(1 << 30)), 1, n) * np.float32(1e-4)) if ef else None
    err_d = torch.from_numpy(err0.copy()).cuda() if ef else None
    co = torch.full((words,), -7, dtype=torch.int32, device="cuda")
    so = torch.full((nb,), -7.0, device="cuda")
    oo = torch.full((nb,), -7.0, device="cuda") if uni else None
    out = torch.full((n,), -7.0, device="cuda") if want_out else None
    q.qc_reencode(dev(codes), cstride, dev(scale), dev(offset) if uni else None, mstride, M, n,
                  bits, bucket, scheme, flags, err_d, mode, SEED, STEP, co, so, oo, out)
    torch.cuda.synchronize()
    e_or = err0.copy() if ef else None
    r, c_or, s_or, o_or = orc.reencode(codes, scale, offset if uni else None, M=M, n=n, bits=bits,
                                       bucket=bucket, scheme=scheme, flags=flags, err=e_or,
                                       mode=mode, seed=SEED, step=STEP,
                                       codes_stride_words=cstride, meta_stride=mstride)
    tag = f"reencode s={scheme} b={bits} M={M} B={bucket} f={flags} ef={ef} m={mode}"
    if want_out:
        assert_bits_equal(host(out), r, tag + " r")
    got_c, got_s = u32(co), host(so)
    got_e = host(err_d) if ef else None
    p = r if err0 is None else (err0 + r).astype(np.float32)
    if scheme == orc.SCHEME_QSGD:
        check_qsgd((got_c, got_s, got_e), (c_or, s_or, e_or), p, n, bits, bucket, tag)
    elif scheme == orc.SCHEME_SIGN:
        assert_bits_equal(got_c, c_or, tag + " bits")
        pm = np.array([np.abs(p[k * bucket:(k + 1) * bucket]).max() for k in range(nb)])
        assert np.all(np.abs(got_s.astype(np.float64) - s_or) <= 1e-6 * pm), tag + " scale"
        if ef:
            assert_close_per_bucket(got_e, e_or, p, bucket, 1e-6, tag + " err")
    else:
        assert_bits_equal(got_c, c_or, tag + " codes")
        assert_bits_equal(got_s, s_or, tag + " scale")
        if uni:
            assert_bits_equal(host(oo), o_or, tag + " offset")
        if ef:
            assert_bits_equal(got_e, e_or, tag + " err")


CASES = [(orc.SCHEME_UNIFORM, 8), (orc.SCHEME_UNIFORM, 4), (orc.SCHEME_UNIFORM, 2),
         (orc.SCHEME_UNIFORM, 1), (orc.SCHEME_SIGN, 1), (orc.SCHEME_TERNARY, 2),
         (orc.SCHEME_QSGD, 2), (orc.SCHEME_QSGD, 4), (orc.SCHEME_QSGD, 8)]


@pytest.mark.parametrize("scheme,bits", CASES)
@pytest.mark.parametrize("M", [1, 3, 16, 100])
def test_reencode(q, scheme, bits, M):
    rng = np.random.default_rng(1000 * M + 10 * scheme + bits)
    for i, bucket in enumerate((32, 96, 1024, 8192)):
        n = max(3 * bucket, 3000) + 13
        flags = orc.OUT_MEAN if i % 2 == 0 else orc.OUT_SUM
        ef = i != 1
        mode = orc.ROUND_NEAREST if (scheme == orc.SCHEME_SIGN or i % 2) else orc.ROUND_STOCHASTIC
        _run(q, scheme, bits, M, n, bucket, flags, ef, mode, want_out=i != 2, rng=rng)


@pytest.mark.parametrize("M", [2, 5])
def test_reencode_matches_two_calls(q, M):
    """The fused call equals qc_decode_accumulate into a buffer followed by
    qc_encode_ef of that buffer, both on the GPU."""
    rng = np.random.default_rng(M)
    n, bits, bucket = 50_000 + 3, 4, 512
    codes, cstride, scale, offset, mstride = _payloads(rng, orc.SCHEME_UNIFORM, bits, M, n, bucket)
    words, nb = orc.code_words(n, bits), orc.num_buckets(n, bucket)
    err0 = wl.std_normal(4, 1, n) * np.float32(1e-4)
    cd, sd, od = dev(codes), dev(scale), dev(offset)
    e1 = torch.from_numpy(err0.copy()).cuda()
    e2 = torch.from_numpy(err0.copy()).cuda()
    c1 = torch.empty(words, dtype=torch.int32, device="cuda")
    c2 = torch.empty_like(c1)
    s1, s2, o1, o2 = (torch.empty(nb, device="cuda") for _ in range(4))
    r1 = torch.empty(n, device="cuda")
    r2 = torch.empty(n, device="cuda")
    q.qc_reencode(cd, cstride, sd, od, mstride, M, n, bits, bucket, 0, q.QC_OUT_MEAN, e1,
                  q.QC_ROUND_STOCHASTIC, SEED, STEP, c1, s1, o1, r1)
    q.qc_decode_accumulate(cd, cstride, sd, od, mstride, M, n, bits, bucket, 0, r2, q.QC_OUT_MEAN)
    q.qc_encode_ef(r2, e2, n, bits, bucket, 0, q.QC_ROUND_STOCHASTIC, SEED, STEP, c2, s2, o2)
    torch.cuda.synchronize()
    for a, b, what in ((r1, r2, "r"), (c1, c2, "codes"), (s1, s2, "scale"), (o1, o2, "offset"),
                       (e1, e2, "err")):
        assert_bits_equal(host(a), host(b), what)


def test_reencode_large_sampled(q):
    """n = 2^24 elements from M = 16 workers, 8-bit uniform, B = 1024: the
    oracle checks a sample of whole buckets spread over the vector (each bucket
    depends only on its own elements)."""
    M, n, bits, bucket = 16, 1 << 24, 8, 1024
    rng = np.random.default_rng(12)
    words, nb = orc.code_words(n, bits), orc.num_buckets(n, bucket)
    codes = torch.randint(-(1 << 31), (1 << 31) - 1, (M, words), dtype=torch.int32, device="cuda",
                          generator=torch.Generator(device="cuda").manual_seed(5))
    scale = (rng.random((M, nb)) * 1e-2).astype(np.float32)
    offset = (rng.standard_normal((M, nb)) * 1e-2).astype(np.float32)
    err0 = wl.std_normal(6, 1, n) * np.float32(1e-4)
    err = torch.from_numpy(err0.copy()).cuda()
    co = torch.empty(words, dtype=torch.int32, device="cuda")
    so, oo = torch.empty(nb, device="cuda"), torch.empty(nb, device="cuda")
    q.qc_reencode(codes, words, dev(scale), dev(offset), nb, M, n, bits, bucket, 0,
                  q.QC_OUT_MEAN, err, q.QC_ROUND_NEAREST, SEED, STEP, co, so, oo, None)
    torch.cuda.synchronize()
    ch = u32(codes)
    cw, eh = u32(co), host(err)
    sh, oh = host(so), host(oo)
    wpb = bucket * bits // 32
    for k in list(rng.choice(nb, 24, replace=False)) + [0, nb - 1]:
        k = int(k)
        sl = slice(k * bucket, (k + 1) * bucket)
        e = err0[sl].copy()
        _, c_or, s_or, o_or = orc.reencode(ch[:, k * wpb:(k + 1) * wpb], scale[:, k:k + 1],
                                           offset[:, k:k + 1], M=M, n=bucket, bits=bits,
                                           bucket=bucket, scheme=0, flags=orc.OUT_MEAN, err=e)
        assert_bits_equal(cw[k * wpb:(k + 1) * wpb], c_or, f"bucket {k} codes")
        assert_bits_equal(sh[k:k + 1], s_or, f"bucket {k} scale")
        assert_bits_equal(oh[k:k + 1], o_or, f"bucket {k} offset")
        assert_bits_equal(eh[sl], e, f"bucket {k} err")

"""GPU <-> oracle parity at the full sizes of the five workloads, through the same
calls and launch configuration as the benchmark, every element of every
output compared.  The oracle runs over bucket-aligned slices on every host
core (tests/_par_oracle.py: its global-index slicing reproduces a whole-array
call exactly).  Properties that hold at any size are checked on the GPU over
the full arrays as well: the error-feedback identity over 10 steps, and the
vote being the majority of the GPU's own sign vectors.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle as orc
import workloads as wl
from tests import _par_oracle as par
from tests._gpu import assert_bits_equal, host, u32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    import embedding_communication_codecs_gb300 as q
    assert torch.cuda.is_available()
    yield q
    assert q.qc_take_device_errors() == 0


# ------------------------------------------------------- uniform 8-bit, n = 2^20

def test_u8_ef_outliers_full(q):
    """2^20 elements ~ N(0, 1e-3) with 0.1% outliers, buckets of 2048, 8-bit
    round to nearest with error feedback: every output compared in full."""
    n, bucket, bits = 1 << 20, 2048, 8
    g = wl.outlier_gradient(n, seed=0)
    gd = torch.from_numpy(g).cuda()
    err = torch.zeros(n, device="cuda")
    codes, scale, offset = q.alloc_payload(n, bits, bucket, 0)
    out = torch.empty(n, device="cuda")
    q.qc_encode_ef(gd, err, n, bits, bucket, 0, 0, 0, 0, codes, scale, offset)
    q.qc_decode_accumulate(codes, 0, scale, offset, 0, 1, n, bits, bucket, 0, out, 0)
    e_or = np.zeros(n, dtype=np.float32)
    c_or, s_or, o_or = orc.encode_uniform(g, e_or, bits=bits, bucket=bucket)
    d_or = orc.decode_accumulate(c_or, s_or, o_or, M=1, n=n, bits=bits, bucket=bucket,
                                 scheme=orc.SCHEME_UNIFORM)
    assert_bits_equal(u32(codes), c_or, "codes")
    assert_bits_equal(host(scale), s_or, "scale")
    assert_bits_equal(host(offset), o_or, "offset")
    assert_bits_equal(host(err), e_or, "residual")
    assert_bits_equal(host(out), d_or, "decoded")


# ----------------------------------------------------- FP8 row-wise 1,000,000 x 128

def test_fp8_rowwise_full(q):
    rows, dim = 1_000_000, 128
    x = wl.embedding_rows(rows, dim, seed=1)
    xd = torch.from_numpy(x).cuda()
    codes = torch.empty((rows, dim), dtype=torch.uint8, device="cuda")
    sc = torch.empty(rows, device="cuda")
    q.qc_rowwise_fp8(xd, rows, dim, codes, sc)
    xh = torch.empty_like(xd)
    q.qc_rowwise_fp8_dequant(codes, sc, rows, dim, xh)
    c_or, s_or = orc.rowwise_fp8(x)
    assert codes.numel() == 128_000_000 and sc.numel() * 4 == 4_000_000
    assert np.array_equal(codes.cpu().numpy(), c_or)
    assert_bits_equal(host(sc), s_or, "row scale")
    assert_bits_equal(host(xh), orc.rowwise_fp8_dequant(c_or, s_or), "dequant")


# ------------------------------------- stochastic 4-bit with error feedback, 10 steps

@pytest.mark.slow
def test_sr4_ef_ten_steps_full(q):
    """250,000,000 elements (1 GB), buckets of 512, per-bucket std log-uniform in
    [1e-5, 1e-2], a fresh draw each step, Philox (seed 2, step, index).  The
    oracle runs all 10 steps over the whole array with its own residual; codes,
    scales and offsets are compared in full at every step, the residual and the
    decoded gradient in full at steps 0, 4 and 9."""
    n, bucket, bits, seed, steps = 250_000_000, 512, 4, 2, 10
    sig = wl.bucket_sigmas(n, bucket, seed)
    e_or = np.zeros(n, dtype=np.float32)
    err = torch.zeros(n, device="cuda")
    codes, scale, offset = q.alloc_payload(n, bits, bucket, 0)
    out = torch.empty(n, device="cuda")
    sent = torch.zeros(n, dtype=torch.float64, device="cuda")
    gsum = torch.zeros(n, dtype=torch.float64, device="cuda")
    bound = torch.zeros(n, dtype=torch.float64, device="cuda")
    for t in range(steps):
        g = wl.bucket_sigma_gradient(n, bucket, t, seed, sigmas=sig)
        gd = torch.from_numpy(g).cuda()
        e_prev = err.abs()
        q.qc_encode_ef(gd, err, n, bits, bucket, 0, 1, seed, t, codes, scale, offset)
        q.qc_decode_accumulate(codes, 0, scale, offset, 0, 1, n, bits, bucket, 0, out, 0)
        c, s_, o = par.encode(orc.encode_uniform, g, e_or, bucket=bucket, bits=bits, mode=1,
                              seed=seed, step=t)
        tag = f"step {t}"
        assert_bits_equal(u32(codes), c, tag + " codes")
        assert_bits_equal(host(scale), s_, tag + " scale")
        assert_bits_equal(host(offset), o, tag + " offset")
        if t in (0, 4, steps - 1):
            d = par.decode(c, s_, o, M=1, n=n, bits=bits, bucket=bucket,
                           scheme=orc.SCHEME_UNIFORM)
            assert_bits_equal(host(err), e_or, tag + " residual")
            assert_bits_equal(host(out), d, tag + " decoded")
        sent += out.double()
        gsum += gd.double()
        # each step rounds p = e + g once and e_new = p - deq once
        bound += 2.0 ** -23 * (gd.double().abs() + e_prev.double() + out.double().abs()
                               + err.double().abs())
    resid = (sent + err.double() - gsum).abs()
    assert bool((resid <= bound + 1e-30).all()), float((resid - bound).max())


def test_ef_resume_is_bit_identical(q):
    """Copying the residual to the host after 5 steps and back, then running 5 more,
    gives exactly the 10-step result (the only state is err and (seed, step))."""
    n, bucket = (1 << 22) + 100, 512
    sig = wl.bucket_sigmas(n, bucket, 7)
    grads = [torch.from_numpy(wl.bucket_sigma_gradient(n, bucket, t, 7, sigmas=sig)).cuda()
             for t in range(10)]

    def run(err, ts):
        outs = []
        for t in ts:
            codes, scale, offset = q.alloc_payload(n, 4, bucket, 0)
            q.qc_encode_ef(grads[t], err, n, 4, bucket, 0, 1, 7, t, codes, scale, offset)
            outs.append(u32(codes))
        return outs

    e1 = torch.zeros(n, device="cuda")
    a = run(e1, range(10))
    e2 = torch.zeros(n, device="cuda")
    b = run(e2, range(5))
    e2 = torch.from_numpy(e2.cpu().numpy().copy()).cuda()
    b += run(e2, range(5, 10))
    for t in range(10):
        assert_bits_equal(a[t], b[t], f"codes step {t}")
    assert_bits_equal(host(e1), host(e2), "residual")


# ------------------------------------------ sign with error feedback + majority vote

def test_sign_ef_vote_full(q):
    """8 workers x 25,600,000 elements ~ N(mu, 1e-3), shared mu ~ N(0, 5e-4),
    buckets of 4096, scaled sign with error feedback (one multi-segment launch),
    then the vote."""
    n, M, bucket = 25_600_000, 8, 4096
    nb = n // bucket
    gw = wl.shared_mean_gradients(n, M, seed=3)
    g = torch.from_numpy(gw).cuda()
    err = torch.zeros((M, n), device="cuda")
    words = q.qc_code_words(n, 1)
    signs = torch.empty((M, words), dtype=torch.int32, device="cuda")
    scale = torch.empty((M, nb), device="cuda")
    vote = torch.empty(words, dtype=torch.int32, device="cuda")
    # the benchmark's call: the 8 workers as the segments of one launch
    q.qc_encode_ef_segments([(g[w], err[w], n, signs[w], scale[w], None) for w in range(M)],
                            q.QC_DTYPE_F32, 1, bucket, 1, 0, 0, 0)
    q.qc_sign_vote(signs, words, M, n, vote)
    sh, vh, eh = u32(signs).reshape(M, words), u32(vote), host(err)
    sc = host(scale)
    bits_or = np.empty((M, words), dtype=np.uint32)
    for w in range(M):
        e_or = np.zeros(n, dtype=np.float32)
        c, s = par.encode(orc.encode_sign, gw[w], e_or, bucket=bucket, index=False)
        bits_or[w] = c
        assert_bits_equal(sh[w], c, f"worker {w} bits")
        # the mean |p| may differ in the order of its sum only: within 1e-6 max|p|
        pmax = np.abs(gw[w]).reshape(nb, bucket).max(axis=1).astype(np.float64)
        assert np.all(np.abs(sc[w].astype(np.float64) - s) <= 1e-6 * pmax), f"worker {w} scale"
        de = np.abs(eh[w].astype(np.float64) - e_or).reshape(nb, bucket).max(axis=1)
        assert np.all(de <= 1e-6 * pmax), f"worker {w} residual"
    assert_bits_equal(vh, par.sign_vote(bits_or, M=M, n=n), "vote")
    # the whole vote is the majority of the GPU's own sign vectors
    bitsum = torch.zeros((words, 32), dtype=torch.int32, device="cuda")
    shifts = torch.arange(32, device="cuda", dtype=torch.int64)
    for w in range(M):
        bitsum += ((signs[w].to(torch.int64).unsqueeze(1) >> shifts) & 1).to(torch.int32)
    want = ((2 * bitsum >= M).to(torch.int64) << shifts).sum(dim=1)
    assert torch.equal(want, vote.to(torch.int64) & 0xFFFFFFFF)


# --------------------------------- quantized all-reduce receiver, 16 x 2^26 bf16

@pytest.mark.parametrize("scheme", ["u8", "ternary"])
def test_allreduce_receiver_full(q, scheme):
    n, M, bucket, seed = 1 << 26, 16, 1024, 4
    nb = n // bucket
    gb = wl.bf16_gradients(n, M, seed=seed)
    g = torch.from_numpy(gb.view(np.int16)).cuda()
    sch, bits, mode = (0, 8, 0) if scheme == "u8" else (2, 2, 1)
    codes, scale, offset = q.alloc_payload(n, bits, bucket, sch, workers=M)
    out = torch.empty(n, device="cuda")
    # the benchmark's call: the 16 workers as the segments of one launch, worker
    # w's draws indexed w * n + i under the one seed
    q.qc_encode_ef_segments([(g[w], None, n, codes[w], scale[w],
                              offset[w] if offset is not None else None) for w in range(M)],
                            q.QC_DTYPE_BF16, bits, bucket, sch, mode, seed, 0)
    q.qc_decode_accumulate(codes, codes.stride(0), scale, offset, scale.stride(0), M, n, bits,
                           bucket, sch, out, q.QC_OUT_MEAN)
    ch = u32(codes).reshape(M, -1)
    sh = host(scale)
    oh = host(offset) if offset is not None else None
    cs, ss, os_ = [], [], []
    for w in range(M):
        if sch == 0:
            c, s, o = par.encode(orc.encode_uniform, gb[w], None, bucket=bucket, bits=8,
                                 base=w * n)
            assert_bits_equal(oh[w], o, f"{scheme} worker {w} offset")
            os_.append(o)
        else:
            c, s = par.encode(orc.encode_ternary, gb[w], None, bucket=bucket, mode=1, seed=seed,
                              step=0, base=w * n)
        assert_bits_equal(ch[w], c, f"{scheme} worker {w} codes")
        assert_bits_equal(sh[w], s, f"{scheme} worker {w} scale")
        cs.append(c)
        ss.append(s)
    d = par.decode(np.stack(cs), np.stack(ss), np.stack(os_) if os_ else None, M=M, n=n,
                   bits=bits, bucket=bucket, scheme=sch, flags=orc.OUT_MEAN)
    assert_bits_equal(host(out), d, f"{scheme} mean")

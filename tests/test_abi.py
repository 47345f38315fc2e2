"""The C ABI without a GPU: the library builds and loads, exports every symbol
include/qcodec.h declares, and rejects bad arguments on the host.

Every call here fails validation (or is an n == 0 no-op) before any CUDA API is
touched, so nothing is launched; the pointers are fake addresses never
dereferenced.
"""
from __future__ import annotations

import os
import re
import subprocess

import pytest

import __graft_entry__

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
qbuild = __graft_entry__._build_module()


@pytest.fixture(scope="module")
def q():
    qbuild.build_library()
    import embedding_communication_codecs_gb300 as q
    return q


def _declared():
    text = open(os.path.join(ROOT, "include", "qcodec.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qc_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(q):
    declared = _declared()
    assert set(declared) == set(q.EXPORTS)
    out = subprocess.run(["nm", "-D", "--defined-only", qbuild.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (qc_[a-z0-9_]+)$", out, flags=re.M))
    for name in declared:
        assert name in exported, name
        assert hasattr(q.lib, name)


def test_size_helpers(q):
    assert q.qc_code_words(0, 8) == 0
    assert q.qc_code_words(1, 1) == 1
    assert q.qc_code_words(250_000_000, 4) == 31_250_000
    assert q.qc_code_words(25_600_000, 1) == 800_000
    assert q.qc_num_buckets(250_000_000, 512) == 488_282
    assert q.qc_num_buckets(10, 0) == 0
    assert "sm_103a" in q.qc_version()


A = 0x10000          # fake, 256-byte aligned device addresses (never dereferenced)
B = 0x20000000
C = 0x30000000
D = 0x40000000


def _enc(q, **kw):
    args = dict(grad=A, dtype=q.QC_DTYPE_F32, err=B, n=4096, bits=8, bucket=2048,
                scheme=q.QC_SCHEME_UNIFORM, mode=q.QC_ROUND_NEAREST, seed=0, step=0, codes=C,
                scale=D, offset=D + 0x100000, stream=0)
    args.update(kw)
    return q.lib.qc_encode_ef(args["grad"], args["dtype"], args["err"], args["n"], args["bits"],
                              args["bucket"], args["scheme"], args["mode"], args["seed"],
                              args["step"], args["codes"], args["scale"], args["offset"],
                              args["stream"])


def test_encode_rejects(q):
    assert _enc(q, bits=3) == q.QC_ERR_INVALID_ARG
    assert b"bits" in q.lib.qc_last_error()
    assert _enc(q, scheme=q.QC_SCHEME_SIGN, bits=8) == q.QC_ERR_INVALID_ARG
    assert _enc(q, scheme=q.QC_SCHEME_SIGN, bits=1, mode=q.QC_ROUND_STOCHASTIC) == q.QC_ERR_INVALID_ARG
    assert _enc(q, scheme=q.QC_SCHEME_TERNARY, bits=1) == q.QC_ERR_INVALID_ARG
    assert _enc(q, scheme=7) == q.QC_ERR_INVALID_ARG
    assert _enc(q, mode=5) == q.QC_ERR_INVALID_ARG
    assert _enc(q, dtype=9) == q.QC_ERR_INVALID_ARG
    for bucket in (0, 16, 48, 2050, (1 << 24) + 32):
        assert _enc(q, bucket=bucket) == q.QC_ERR_INVALID_ARG
    assert _enc(q, grad=None) == q.QC_ERR_NULL
    assert _enc(q, codes=None) == q.QC_ERR_NULL
    assert _enc(q, offset=None) == q.QC_ERR_NULL
    assert _enc(q, grad=A + 4) == q.QC_ERR_ALIGNMENT
    assert _enc(q, dtype=q.QC_DTYPE_BF16, grad=A + 4) == q.QC_ERR_ALIGNMENT
    assert _enc(q, err=B + 8) == q.QC_ERR_ALIGNMENT
    assert _enc(q, codes=C + 2) == q.QC_ERR_ALIGNMENT
    # outputs overlapping inputs or each other
    assert _enc(q, codes=A + 64) == q.QC_ERR_INVALID_ARG
    assert _enc(q, scale=C) == q.QC_ERR_INVALID_ARG
    assert _enc(q, err=A) == q.QC_ERR_INVALID_ARG
    assert _enc(q, n=1 << 41) == q.QC_ERR_UNSUPPORTED


def test_encode_empty_is_noop(q):
    assert _enc(q, n=0, grad=None, codes=None, scale=None, offset=None) == q.QC_OK
    assert q.lib.qc_last_error() == b""


def test_decode_rejects(q):
    def dec(**kw):
        a = dict(codes=C, cs=1024, scale=D, offset=D + 0x100000, ms=2, M=2, n=4096, bits=8,
                 bucket=2048, scheme=q.QC_SCHEME_UNIFORM, out=A, flags=0)
        a.update(kw)
        return q.lib.qc_decode_accumulate(a["codes"], a["cs"], a["scale"], a["offset"], a["ms"],
                                          a["M"], a["n"], a["bits"], a["bucket"], a["scheme"],
                                          a["out"], a["flags"], 0)
    assert dec(M=0) == q.QC_ERR_INVALID_ARG
    assert dec(M=q.QC_MAX_WORKERS + 1) == q.QC_ERR_INVALID_ARG
    assert dec(flags=4) == q.QC_ERR_INVALID_ARG
    assert dec(cs=1023) == q.QC_ERR_INVALID_ARG
    assert dec(ms=1) == q.QC_ERR_INVALID_ARG
    assert dec(bits=3) == q.QC_ERR_INVALID_ARG
    assert dec(scheme=q.QC_SCHEME_TERNARY, bits=8) == q.QC_ERR_INVALID_ARG
    assert dec(out=None) == q.QC_ERR_NULL
    assert dec(offset=None) == q.QC_ERR_NULL
    assert dec(out=A + 4) == q.QC_ERR_ALIGNMENT
    assert dec(out=C) == q.QC_ERR_INVALID_ARG
    assert dec(n=0, codes=None, out=None) == q.QC_OK


def test_vote_and_fp8_reject(q):
    L = q.lib
    assert L.qc_sign_vote(C, 8, 0, 256, A, 0) == q.QC_ERR_INVALID_ARG
    assert L.qc_sign_vote(C, 7, 2, 256, A, 0) == q.QC_ERR_INVALID_ARG
    assert L.qc_sign_vote(None, 8, 2, 256, A, 0) == q.QC_ERR_NULL
    assert L.qc_sign_vote(C + 2, 8, 2, 256, A, 0) == q.QC_ERR_ALIGNMENT
    assert L.qc_sign_vote(C, 8, 2, 256, C + 4, 0) == q.QC_ERR_INVALID_ARG
    assert L.qc_sign_vote(C, 8, 2, 0, None, 0) == q.QC_OK
    assert L.qc_rowwise_fp8(A, 10, 6, C, D, 0) == q.QC_ERR_INVALID_ARG
    assert L.qc_rowwise_fp8(A, 10, 0, C, D, 0) == q.QC_ERR_INVALID_ARG
    assert L.qc_rowwise_fp8(A, 10, 8192, C, D, 0) == q.QC_ERR_UNSUPPORTED
    assert L.qc_rowwise_fp8(A + 8, 10, 128, C, D, 0) == q.QC_ERR_ALIGNMENT
    assert L.qc_rowwise_fp8(None, 10, 128, C, D, 0) == q.QC_ERR_NULL
    assert L.qc_rowwise_fp8(A, 10, 128, A + 256, D, 0) == q.QC_ERR_INVALID_ARG
    assert L.qc_rowwise_fp8(A, 0, 128, None, None, 0) == q.QC_OK
    assert L.qc_rowwise_fp8_dequant(C, D, 10, 128, A + 4, 0) == q.QC_ERR_ALIGNMENT
    assert L.qc_rowwise_fp8_dequant(C, D, 10, 128, C, 0) == q.QC_ERR_INVALID_ARG


def test_qsgd_bits_rejected(q):
    for bits in (1, 3, 16):
        assert _enc(q, scheme=q.QC_SCHEME_QSGD, bits=bits) == q.QC_ERR_INVALID_ARG
    assert _enc(q, scheme=q.QC_SCHEME_QSGD, bits=4, offset=None, n=0) == q.QC_OK


def test_reencode_rejects(q):
    E = 0x50000000
    F = 0x60000000

    def re_(**kw):
        a = dict(codes=C, cs=1024, scale=D, offset=D + 0x100000, ms=2, M=2, n=4096, bits=8,
                 bucket=2048, scheme=q.QC_SCHEME_UNIFORM, flags=q.QC_OUT_MEAN, err=B,
                 mode=q.QC_ROUND_NEAREST, codes_out=E, scale_out=F, offset_out=F + 0x1000,
                 out=A)
        a.update(kw)
        return q.lib.qc_reencode(a["codes"], a["cs"], a["scale"], a["offset"], a["ms"], a["M"],
                                 a["n"], a["bits"], a["bucket"], a["scheme"], a["flags"],
                                 a["err"], a["mode"], 0, 0, a["codes_out"], a["scale_out"],
                                 a["offset_out"], a["out"], 0)
    assert re_(M=0) == q.QC_ERR_INVALID_ARG
    assert re_(flags=q.QC_ACCUMULATE_INTO_OUT) == q.QC_ERR_INVALID_ARG
    assert re_(bits=3) == q.QC_ERR_INVALID_ARG
    assert re_(scheme=q.QC_SCHEME_SIGN, bits=1, mode=q.QC_ROUND_STOCHASTIC) == q.QC_ERR_INVALID_ARG
    assert re_(mode=4) == q.QC_ERR_INVALID_ARG
    assert re_(cs=1023) == q.QC_ERR_INVALID_ARG
    assert re_(codes_out=None) == q.QC_ERR_NULL
    assert re_(offset_out=None) == q.QC_ERR_NULL
    assert re_(err=B + 4) == q.QC_ERR_ALIGNMENT
    assert re_(out=A + 8) == q.QC_ERR_ALIGNMENT
    assert re_(codes_out=C + 64) == q.QC_ERR_INVALID_ARG     # output over the input payload
    assert re_(out=B) == q.QC_ERR_INVALID_ARG                # output over another output
    # layouts the fused kernel does not take
    assert re_(cs=1026) == q.QC_ERR_UNSUPPORTED
    assert re_(codes=C + 4) == q.QC_ERR_UNSUPPORTED
    assert re_(bucket=16384, n=1 << 15, cs=1 << 13, ms=2) == q.QC_ERR_UNSUPPORTED
    assert b"qc_decode_accumulate followed by qc_encode_ef" in q.lib.qc_last_error()
    assert re_(n=0, codes=None, codes_out=None) == q.QC_OK


def test_clip_rejects(q):
    C_ = q.QC_SCHEME_UNIFORM_CLIP
    assert _enc(q, scheme=C_, bits=3) == q.QC_ERR_INVALID_ARG
    assert _enc(q, scheme=C_, offset=None) == q.QC_ERR_NULL
    assert _enc(q, scheme=C_, bucket=8192, n=1 << 15) == q.QC_ERR_UNSUPPORTED
    assert b"percentile" in q.lib.qc_last_error()
    assert _enc(q, scheme=C_, grad=A + 8, dtype=q.QC_DTYPE_BF16) == q.QC_ERR_UNSUPPORTED
    assert q.lib.qc_reencode(C, 1024, D, D + 0x100000, 2, 2, 4096, 8, 2048, C_, 0, B, 0, 0, 0,
                             0x50000000, 0x60000000, 0x60001000, A, 0) == q.QC_ERR_UNSUPPORTED


def test_selftest_rejects(q):
    for us in (0, 10_000_001):
        assert q.lib.qc_selftest_wait_timeout(us, 0) == q.QC_ERR_INVALID_ARG
    assert b"timeout_us" in q.lib.qc_last_error()


def test_status_word_setting(q):
    """The status word is a host-side setting: it takes any 4-byte aligned
    address (or NULL) without touching the device."""
    assert q.lib.qc_set_status_word(0x1002) == q.QC_ERR_ALIGNMENT
    assert q.lib.qc_set_status_word(0x1000) == q.QC_OK
    assert q.lib.qc_set_status_word(None) == q.QC_OK


def test_log_rejects(q):
    L_ = q.QC_SCHEME_LOG
    for bits in (1, 3, 16):
        assert _enc(q, scheme=L_, bits=bits) == q.QC_ERR_INVALID_ARG
    assert b"logarithmic" in q.lib.qc_last_error()
    assert _enc(q, scheme=L_, bits=4, offset=None, n=0) == q.QC_OK


def test_topk_rejects(q):
    L = q.lib
    E = 0x50000000

    def enc(**kw):
        a = dict(grad=A, dtype=q.QC_DTYPE_F32, err=B, n=4096, bucket=1024, keep=10,
                 mode=q.QC_ROUND_NEAREST, idx=C, codes=E, scale=D, offset=D + 0x100000)
        a.update(kw)
        return L.qc_topk_encode_ef(a["grad"], a["dtype"], a["err"], a["n"], a["bucket"], a["keep"],
                                   a["mode"], 0, 0, a["idx"], a["codes"], a["scale"], a["offset"], 0)
    assert enc(keep=0) == q.QC_ERR_INVALID_ARG
    assert enc(keep=1025) == q.QC_ERR_INVALID_ARG
    assert enc(bucket=48) == q.QC_ERR_INVALID_ARG
    assert enc(bucket=8192, n=1 << 15) == q.QC_ERR_UNSUPPORTED
    assert enc(n=1 << 32) == q.QC_ERR_UNSUPPORTED
    assert enc(idx=None) == q.QC_ERR_NULL
    assert enc(grad=A + 4) == q.QC_ERR_UNSUPPORTED
    assert enc(err=B + 4) == q.QC_ERR_ALIGNMENT
    assert enc(idx=A + 64) == q.QC_ERR_INVALID_ARG
    assert enc(n=0, grad=None, idx=None) == q.QC_OK

    def dec(**kw):
        a = dict(idx=C, codes=E, ps=40, scale=D, offset=D + 0x100000, ms=4, M=2, n=4096,
                 bucket=1024, keep=10, out=A, flags=1)
        a.update(kw)
        return L.qc_topk_decode_accumulate(a["idx"], a["codes"], a["ps"], a["scale"], a["offset"],
                                           a["ms"], a["M"], a["n"], a["bucket"], a["keep"], a["out"],
                                           a["flags"], 0)
    assert dec(M=0) == q.QC_ERR_INVALID_ARG
    assert dec(ps=39) == q.QC_ERR_INVALID_ARG
    assert dec(flags=8) == q.QC_ERR_INVALID_ARG
    assert dec(out=None) == q.QC_ERR_NULL
    assert dec(out=C) == q.QC_ERR_INVALID_ARG
    assert dec(bucket=32768, n=1 << 16, ps=20, ms=2, keep=10) == q.QC_ERR_UNSUPPORTED
    assert dec(bucket=4096, keep=2000, ps=2000) == q.QC_ERR_UNSUPPORTED
    assert dec(n=0, idx=None, out=None) == q.QC_OK


def _segs(q, *rows):
    arr = (q.QcSegment * max(1, len(rows)))()
    for k, (grad, err, n, codes, scale, offset) in enumerate(rows):
        arr[k] = q.QcSegment(grad, err, n, codes, scale, offset)
    return arr


def _enc_segs(q, rows, dtype=None, bits=4, bucket=512, scheme=None, mode=None, nseg=None):
    dtype = q.QC_DTYPE_F32 if dtype is None else dtype
    scheme = q.QC_SCHEME_UNIFORM if scheme is None else scheme
    mode = q.QC_ROUND_STOCHASTIC if mode is None else mode
    return q.lib.qc_encode_ef_segments(_segs(q, *rows), len(rows) if nseg is None else nseg,
                                       dtype, bits, bucket, scheme, mode, 1, 0, 0)


MB = 0x100000


def _seg(k, n=4096):
    """Segment k's buffers, 16 MB apart from every other segment's."""
    base = 0x1000000 * (k + 1)
    return (base, base + 4 * MB, n, base + 8 * MB, base + 12 * MB, base + 14 * MB)


def test_segments_reject(q):
    assert _enc_segs(q, [], nseg=0) == q.QC_OK                      # nothing to do
    assert _enc_segs(q, [_seg(0)], nseg=-1) == q.QC_ERR_INVALID_ARG
    assert q.lib.qc_encode_ef_segments(None, 2, q.QC_DTYPE_F32, 4, 512, 0, 1, 1, 0, 0) == \
        q.QC_ERR_NULL
    assert _enc_segs(q, [_seg(0)], bits=3) == q.QC_ERR_INVALID_ARG   # arguments of the call
    # a bad segment is named
    g, e, n, c, s, o = _seg(1)
    assert _enc_segs(q, [_seg(0), (g, e, n, c, s, 0)]) == q.QC_ERR_NULL
    assert b"segment 1" in q.lib.qc_last_error()
    assert _enc_segs(q, [_seg(0), (g + 2, e, n, c, s, o)]) == q.QC_ERR_ALIGNMENT
    # residuals for every segment or for none
    assert _enc_segs(q, [_seg(0), (g, 0, n, c, s, o)]) == q.QC_ERR_INVALID_ARG
    assert b"every segment or for none" in q.lib.qc_last_error()
    # an output of one segment over a buffer of another
    g0, e0, n0, c0, s0, o0 = _seg(0)
    assert _enc_segs(q, [_seg(0), (g, e, n, c0 + 256, s, o)]) == q.QC_ERR_INVALID_ARG
    assert b"overlaps" in q.lib.qc_last_error()
    assert _enc_segs(q, [_seg(0), (g, g0, n, c, s, o)]) == q.QC_ERR_INVALID_ARG  # err over grad
    # empty segments take no buffers and are not checked
    assert _enc_segs(q, [(0, 0, 0, 0, 0, 0)]) == q.QC_OK
    assert q.QC_MAX_SEGMENTS_PER_LAUNCH == 60

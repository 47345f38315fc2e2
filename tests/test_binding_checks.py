"""The Python binding checks every torch tensor against what the C call will
read or write (dtype, dense layout, bytes, row stride, device) and raises
ValueError before anything is launched.  CPU only: the device check comes last,
so every other rejection is reached with host tensors, and a call whose tensors
are all right except for living on the host fails on the device check."""
from __future__ import annotations

import pytest
import torch

import embedding_communication_codecs_gb300 as q


def f32(n):
    return torch.zeros(n, dtype=torch.float32)


def words(n, bits):
    return torch.zeros(q.qc_code_words(n, bits), dtype=torch.int32)


N, B = 4096 + 37, 512
NB = q.qc_num_buckets(N, B)


def _enc(**kw):
    args = dict(grad=f32(N), err=f32(N), n=N, bits=4, bucket=B, scheme=q.QC_SCHEME_UNIFORM,
                mode=q.QC_ROUND_NEAREST, seed=0, step=0, codes=words(N, 4), scale=f32(NB),
                offset=f32(NB))
    args.update(kw)
    q.qc_encode_ef(**args)


def test_encode_all_right_but_on_the_host():
    with pytest.raises(ValueError, match="CUDA tensor"):
        _enc()


@pytest.mark.parametrize("kw,msg", [
    (dict(grad=f32(N - 1)), "grad spans"),
    (dict(grad=torch.zeros(2 * N)[::2]), "grad must be contiguous"),
    (dict(err=f32(N - 4)), "err spans"),
    (dict(err=torch.zeros(N, dtype=torch.bfloat16)), "err has dtype"),
    (dict(codes=words(N, 4)[:-1]), "codes spans"),
    (dict(codes=torch.zeros(q.qc_code_words(N, 4), dtype=torch.float32)), "codes has dtype"),
    (dict(scale=f32(NB - 1)), "scale spans"),
    (dict(offset=f32(NB - 1)), "offset spans"),
    (dict(codes=words(N, 2), bits=4), "codes spans"),
    (dict(grad=torch.zeros(N, dtype=torch.bfloat16)[:N - 8], dtype=q.QC_DTYPE_BF16), "grad spans"),
])
def test_encode_rejections(kw, msg):
    with pytest.raises(ValueError, match=msg):
        _enc(**kw)


def test_encode_gradient_of_another_dtype():
    with pytest.raises(TypeError, match="not float32 or bfloat16"):
        _enc(grad=torch.zeros(N, dtype=torch.float64))
    with pytest.raises(ValueError, match="grad has dtype"):
        _enc(grad=torch.zeros(N, dtype=torch.float64), dtype=q.QC_DTYPE_F32)


def test_decode_rejections():
    M, bits = 3, 8
    w = q.qc_code_words(N, bits)
    codes = torch.zeros((M, w + 4), dtype=torch.int32)
    scale = torch.zeros((M, NB + 3))
    offset = torch.zeros((M, NB + 3))
    out = f32(N)
    base = dict(codes=codes, codes_stride_words=w + 4, scale=scale, offset=offset,
                meta_stride=NB + 3, M=M, n=N, bits=bits, bucket=B, scheme=q.QC_SCHEME_UNIFORM,
                out=out)
    with pytest.raises(ValueError, match="CUDA tensor"):
        q.qc_decode_accumulate(**base)
    for kw, msg in [
        (dict(codes_stride_words=w + 5), "codes's row stride"),
        (dict(offset=torch.zeros((M, NB + 4))), "offset's row stride"),
        (dict(scale=torch.zeros((M, NB + 3))[:, :NB - 1]), "scale's row stride|scale spans"),
        (dict(codes=torch.zeros((M, w + 4), dtype=torch.int32)[:2]), "codes spans"),
        (dict(out=f32(N - 1)), "out spans"),
        (dict(codes=torch.zeros((w + 4, M), dtype=torch.int32).t()), "dense along its last"),
    ]:
        with pytest.raises(ValueError, match=msg):
            q.qc_decode_accumulate(**{**base, **kw})


def test_reencode_topk_vote_fp8_rejections():
    M, bits = 2, 2
    w = q.qc_code_words(N, bits)
    codes = torch.zeros((M, w), dtype=torch.int32)
    scale = torch.zeros((M, NB))
    with pytest.raises(ValueError, match="codes_out spans"):
        q.qc_reencode(codes, w, scale, None, NB, M, N, bits, B, q.QC_SCHEME_TERNARY,
                      q.QC_OUT_MEAN, f32(N), q.QC_ROUND_STOCHASTIC, 0, 0, words(N, bits)[:-1],
                      f32(NB), None)
    with pytest.raises(ValueError, match="err spans"):
        q.qc_reencode(codes, w, scale, None, NB, M, N, bits, B, q.QC_SCHEME_TERNARY,
                      q.QC_OUT_MEAN, f32(N - 1), q.QC_ROUND_STOCHASTIC, 0, 0, words(N, bits),
                      f32(NB), None)
    keep = 8
    with pytest.raises(ValueError, match="idx spans"):
        q.qc_topk_encode_ef(f32(N), None, N, B, keep, q.QC_ROUND_NEAREST, 0, 0,
                            torch.zeros(NB * keep - 1, dtype=torch.int32),
                            torch.zeros(NB * keep, dtype=torch.uint8), f32(NB), f32(NB))
    with pytest.raises(ValueError, match="codes has dtype"):
        q.qc_topk_decode_accumulate(torch.zeros(NB * keep, dtype=torch.int32),
                                    torch.zeros(NB * keep, dtype=torch.float32), NB * keep,
                                    f32(NB), f32(NB), NB, 1, N, B, keep, f32(N))
    sw = q.qc_code_words(N, 1)
    with pytest.raises(ValueError, match="signs's row stride"):
        q.qc_sign_vote(torch.zeros((3, sw + 1), dtype=torch.int32), sw, 3, N,
                       torch.zeros(sw, dtype=torch.int32))
    with pytest.raises(ValueError, match="out spans"):
        q.qc_sign_vote(torch.zeros((3, sw), dtype=torch.int32), sw, 3, N,
                       torch.zeros(sw - 1, dtype=torch.int32))
    rows, dim = 100, 128
    with pytest.raises(ValueError, match="codes spans"):
        q.qc_rowwise_fp8(f32(rows * dim), rows, dim, torch.zeros(rows * dim - 1, dtype=torch.uint8),
                         f32(rows))
    with pytest.raises(ValueError, match="row_scale spans"):
        q.qc_rowwise_fp8_dequant(torch.zeros(rows * dim, dtype=torch.uint8), f32(rows - 1), rows,
                                 dim, f32(rows * dim))
    with pytest.raises(ValueError, match="x must be contiguous"):
        q.qc_rowwise_fp8(torch.zeros((dim, rows)).t(), rows, dim,
                         torch.zeros(rows * dim, dtype=torch.uint8), f32(rows))

"""CPU oracle for the communication codec -- TEST INFRASTRUCTURE ONLY.

Plain scalar C (``qc_oracle.c``) behind a thin numpy/ctypes wrapper.  Only the
test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import this package; the product library never calls it and has no CPU
fallback.  It shares no code with the CUDA path.

Every function restates one step of the method from the pages on quantized
communication (see the header of ``qc_oracle.c`` for the sections followed).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qc_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

SCHEME_UNIFORM, SCHEME_SIGN, SCHEME_TERNARY, SCHEME_QSGD, SCHEME_UNIFORM_CLIP, SCHEME_LOG = 0, 1, 2, 3, 4, 5
ROUND_NEAREST, ROUND_STOCHASTIC = 0, 1
DTYPE_F32, DTYPE_BF16 = 0, 1
OUT_SUM, OUT_MEAN, ACCUMULATE_INTO_OUT = 0, 1, 2

# -ffp-contract=off: every a*b+c in the source is two roundings unless written
# as fmaf(); GCC contracts by default on aarch64 hosts.
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
          "-fvisibility=hidden"]


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` next to the source (gcc)."""
    with _lock:
        if (not force and os.path.exists(_LIB_PATH)
                and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
            return _LIB_PATH
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
        return _LIB_PATH


def _L():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        P = ctypes.c_void_p
        S = ctypes.c_size_t
        U64 = ctypes.c_uint64
        U32 = ctypes.c_uint32
        I = ctypes.c_int
        lib.oracle_philox4x32_10.argtypes = [P, P, P]
        lib.oracle_philox4x32_10.restype = None
        lib.oracle_uniform.argtypes = [U64, U32, U64]
        lib.oracle_uniform.restype = ctypes.c_float
        lib.oracle_code_words.argtypes = [S, I]
        lib.oracle_code_words.restype = S
        lib.oracle_num_buckets.argtypes = [S, S]
        lib.oracle_num_buckets.restype = S
        lib.oracle_encode_uniform.argtypes = [P, I, P, S, U64, I, S, I, U64, U32, P, P, P]
        lib.oracle_encode_uniform_clip.argtypes = [P, I, P, S, U64, I, S, I, U64, U32, P, P, P]
        lib.oracle_encode_sign.argtypes = [P, I, P, S, S, P, P]
        lib.oracle_encode_ternary.argtypes = [P, I, P, S, U64, S, I, U64, U32, P, P]
        lib.oracle_encode_qsgd.argtypes = [P, I, P, S, U64, I, S, I, U64, U32, P, P]
        lib.oracle_encode_log.argtypes = [P, I, P, S, U64, I, S, I, U64, U32, P, P]
        lib.oracle_decode_accumulate.argtypes = [P, S, P, P, S, I, S, I, S, I, P, I]
        lib.oracle_sign_vote.argtypes = [P, S, I, S, P]
        lib.oracle_topk_encode.argtypes = [P, I, P, S, U64, S, S, I, U64, U32, P, P, P, P]
        lib.oracle_topk_decode.argtypes = [P, P, S, P, P, S, I, S, S, S, P, I]
        lib.oracle_e4m3_to_f32.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_to_f32.restype = ctypes.c_float
        lib.oracle_e4m3_from_f32.argtypes = [ctypes.c_float]
        lib.oracle_e4m3_from_f32.restype = ctypes.c_uint8
        lib.oracle_e4m3_from_f32_array.argtypes = [P, S, P]
        lib.oracle_e4m3_from_f32_array.restype = None
        lib.oracle_rowwise_fp8.argtypes = [P, S, S, P, P]
        lib.oracle_rowwise_fp8_dequant.argtypes = [P, P, S, S, P]
        for name in ("oracle_encode_uniform", "oracle_encode_uniform_clip", "oracle_encode_sign",
                     "oracle_encode_ternary",
                     "oracle_encode_qsgd", "oracle_encode_log",
                     "oracle_decode_accumulate", "oracle_sign_vote", "oracle_rowwise_fp8",
                     "oracle_topk_encode", "oracle_topk_decode",
                     "oracle_rowwise_fp8_dequant"):
            getattr(lib, name).restype = I
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments (rc={rc})")


def _grad_dtype(g):
    if g.dtype == np.float32:
        return DTYPE_F32
    if g.dtype == np.uint16:  # bf16 bit patterns
        return DTYPE_BF16
    raise TypeError("gradient must be float32 or uint16 (bf16 bits)")


def code_words(n: int, bits: int) -> int:
    return int(_L().oracle_code_words(n, bits))


def num_buckets(n: int, bucket: int) -> int:
    return int(_L().oracle_num_buckets(n, bucket))


def philox4x32_10(counter, key):
    c = np.ascontiguousarray(counter, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    _L().oracle_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def uniform(seed: int, step: int, index: int) -> float:
    return float(_L().oracle_uniform(seed, step, index))


def encode_uniform(grad, err=None, *, bits, bucket, mode=ROUND_NEAREST, seed=0, step=0,
                   index_base=0):
    """Returns (codes uint32[], scale f32[], offset f32[]); ``err`` is updated in place."""
    g = np.ascontiguousarray(grad)
    n = g.size
    if err is not None:
        assert err.dtype == np.float32 and err.flags.c_contiguous and err.size == n
    codes = np.zeros(max(code_words(n, bits), 1), dtype=np.uint32)
    nb = max(num_buckets(n, bucket), 1)
    scale = np.zeros(nb, dtype=np.float32)
    offset = np.zeros(nb, dtype=np.float32)
    rc = _L().oracle_encode_uniform(_ptr(g), _grad_dtype(g), _ptr(err), n, index_base, bits,
                                    bucket, mode, seed, step, _ptr(codes), _ptr(scale),
                                    _ptr(offset))
    _check(rc, "encode_uniform")
    nw = code_words(n, bits)
    return codes[:nw], scale[:num_buckets(n, bucket)], offset[:num_buckets(n, bucket)]


def encode_uniform_clip(grad, err=None, *, bits, bucket, mode=ROUND_NEAREST, seed=0, step=0,
                        index_base=0):
    """Uniform quantization over the bucket's 1st..99th percentile range
    (nearest rank); returns (codes, scale, offset) and updates ``err``."""
    g = np.ascontiguousarray(grad)
    n = g.size
    if err is not None:
        assert err.dtype == np.float32 and err.flags.c_contiguous and err.size == n
    codes = np.zeros(max(code_words(n, bits), 1), dtype=np.uint32)
    nb = max(num_buckets(n, bucket), 1)
    scale = np.zeros(nb, dtype=np.float32)
    offset = np.zeros(nb, dtype=np.float32)
    rc = _L().oracle_encode_uniform_clip(_ptr(g), _grad_dtype(g), _ptr(err), n, index_base, bits,
                                         bucket, mode, seed, step, _ptr(codes), _ptr(scale),
                                         _ptr(offset))
    _check(rc, "encode_uniform_clip")
    return codes[:code_words(n, bits)], scale[:num_buckets(n, bucket)], offset[:num_buckets(n, bucket)]


def encode_sign(grad, err=None, *, bucket):
    g = np.ascontiguousarray(grad)
    n = g.size
    codes = np.zeros(max(code_words(n, 1), 1), dtype=np.uint32)
    scale = np.zeros(max(num_buckets(n, bucket), 1), dtype=np.float32)
    rc = _L().oracle_encode_sign(_ptr(g), _grad_dtype(g), _ptr(err), n, bucket, _ptr(codes),
                                 _ptr(scale))
    _check(rc, "encode_sign")
    return codes[:code_words(n, 1)], scale[:num_buckets(n, bucket)]


def encode_ternary(grad, err=None, *, bucket, mode=ROUND_STOCHASTIC, seed=0, step=0,
                   index_base=0):
    g = np.ascontiguousarray(grad)
    n = g.size
    codes = np.zeros(max(code_words(n, 2), 1), dtype=np.uint32)
    scale = np.zeros(max(num_buckets(n, bucket), 1), dtype=np.float32)
    rc = _L().oracle_encode_ternary(_ptr(g), _grad_dtype(g), _ptr(err), n, index_base, bucket,
                                    mode, seed, step, _ptr(codes), _ptr(scale))
    _check(rc, "encode_ternary")
    return codes[:code_words(n, 2)], scale[:num_buckets(n, bucket)]


def encode_qsgd(grad, err=None, *, bits, bucket, mode=ROUND_STOCHASTIC, seed=0, step=0,
                index_base=0):
    """Returns (codes uint32[], unit f32[]); ``err`` is updated in place."""
    g = np.ascontiguousarray(grad)
    n = g.size
    codes = np.zeros(max(code_words(n, bits), 1), dtype=np.uint32)
    scale = np.zeros(max(num_buckets(n, bucket), 1), dtype=np.float32)
    rc = _L().oracle_encode_qsgd(_ptr(g), _grad_dtype(g), _ptr(err), n, index_base, bits, bucket,
                                 mode, seed, step, _ptr(codes), _ptr(scale))
    _check(rc, "encode_qsgd")
    return codes[:code_words(n, bits)], scale[:num_buckets(n, bucket)]


def encode_log(grad, err=None, *, bits, bucket, mode=ROUND_NEAREST, seed=0, step=0, index_base=0):
    """Logarithmic levels s * 2^(j - J) under a sign bit; returns (codes, s) and
    updates ``err``."""
    g = np.ascontiguousarray(grad)
    n = g.size
    codes = np.zeros(max(code_words(n, bits), 1), dtype=np.uint32)
    scale = np.zeros(max(num_buckets(n, bucket), 1), dtype=np.float32)
    rc = _L().oracle_encode_log(_ptr(g), _grad_dtype(g), _ptr(err), n, index_base, bits, bucket,
                                mode, seed, step, _ptr(codes), _ptr(scale))
    _check(rc, "encode_log")
    return codes[:code_words(n, bits)], scale[:num_buckets(n, bucket)]


def decode_accumulate(codes, scale, offset, *, M, n, bits, bucket, scheme, flags=OUT_SUM,
                      codes_stride_words=None, meta_stride=None, out=None):
    """``codes`` is uint32 of shape [M, stride] (or flat with explicit strides)."""
    c = np.ascontiguousarray(codes, dtype=np.uint32)
    s = np.ascontiguousarray(scale, dtype=np.float32)
    o = None if offset is None else np.ascontiguousarray(offset, dtype=np.float32)
    if codes_stride_words is None:
        codes_stride_words = c.shape[-1] if c.ndim == 2 else code_words(n, bits)
    if meta_stride is None:
        meta_stride = s.shape[-1] if s.ndim == 2 else num_buckets(n, bucket)
    if out is None:
        out = np.zeros(n, dtype=np.float32)
    assert out.dtype == np.float32 and out.flags.c_contiguous
    rc = _L().oracle_decode_accumulate(_ptr(c), codes_stride_words, _ptr(s), _ptr(o),
                                       meta_stride, M, n, bits, bucket, scheme, _ptr(out),
                                       flags)
    _check(rc, "decode_accumulate")
    return out


def reencode(codes, scale, offset, *, M, n, bits, bucket, scheme, flags=OUT_SUM, err=None,
             mode=ROUND_NEAREST, seed=0, step=0, codes_stride_words=None, meta_stride=None):
    """Receiver re-encode ("Quantization-Aware All-Reduce": dequantize after the
    exchange, accumulate, quantize again for the all-gather): the decode of M
    payloads followed by the encode of the result, with the residual ``err``
    (updated in place), in the same scheme, bits and bucket.  Returns
    (r, codes, scale, offset-or-None)."""
    r = decode_accumulate(codes, scale, offset, M=M, n=n, bits=bits, bucket=bucket,
                          scheme=scheme, flags=flags, codes_stride_words=codes_stride_words,
                          meta_stride=meta_stride)
    if scheme == SCHEME_UNIFORM:
        c, s, o = encode_uniform(r, err, bits=bits, bucket=bucket, mode=mode, seed=seed, step=step)
        return r, c, s, o
    if scheme == SCHEME_UNIFORM_CLIP:
        c, s, o = encode_uniform_clip(r, err, bits=bits, bucket=bucket, mode=mode, seed=seed,
                                      step=step)
        return r, c, s, o
    if scheme == SCHEME_SIGN:
        c, s = encode_sign(r, err, bucket=bucket)
    elif scheme == SCHEME_LOG:
        c, s = encode_log(r, err, bits=bits, bucket=bucket, mode=mode, seed=seed, step=step)
    elif scheme == SCHEME_TERNARY:
        c, s = encode_ternary(r, err, bucket=bucket, mode=mode, seed=seed, step=step)
    else:
        c, s = encode_qsgd(r, err, bits=bits, bucket=bucket, mode=mode, seed=seed, step=step)
    return r, c, s, None


def topk_encode(grad, err=None, *, bucket, keep, mode=ROUND_NEAREST, seed=0, step=0,
                index_base=0):
    """Per-bucket top-k (largest |p|, ties to the lower index) with 8-bit codes of
    the kept values; returns (idx uint32[nb*keep], codes uint8[nb*keep], scale,
    offset) and updates ``err``."""
    g = np.ascontiguousarray(grad)
    n = g.size
    if err is not None:
        assert err.dtype == np.float32 and err.flags.c_contiguous and err.size == n
    nb = num_buckets(n, bucket)
    idx = np.zeros(max(nb * keep, 1), dtype=np.uint32)
    codes = np.zeros(max(nb * keep, 1), dtype=np.uint8)
    scale = np.zeros(max(nb, 1), dtype=np.float32)
    offset = np.zeros(max(nb, 1), dtype=np.float32)
    rc = _L().oracle_topk_encode(_ptr(g), _grad_dtype(g), _ptr(err), n, index_base, bucket, keep,
                                 mode, seed, step, _ptr(idx), _ptr(codes), _ptr(scale),
                                 _ptr(offset))
    _check(rc, "topk_encode")
    return idx[:nb * keep], codes[:nb * keep], scale[:nb], offset[:nb]


def topk_decode(idx, codes, scale, offset, *, M, n, bucket, keep, flags=OUT_SUM,
                pair_stride=None, meta_stride=None, out=None):
    i = np.ascontiguousarray(idx, dtype=np.uint32)
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    s = np.ascontiguousarray(scale, dtype=np.float32)
    o = np.ascontiguousarray(offset, dtype=np.float32)
    if pair_stride is None:
        pair_stride = i.shape[-1] if i.ndim == 2 else num_buckets(n, bucket) * keep
    if meta_stride is None:
        meta_stride = s.shape[-1] if s.ndim == 2 else num_buckets(n, bucket)
    if out is None:
        out = np.zeros(n, dtype=np.float32)
    rc = _L().oracle_topk_decode(_ptr(i), _ptr(c), pair_stride, _ptr(s), _ptr(o), meta_stride, M,
                                 n, bucket, keep, _ptr(out), flags)
    _check(rc, "topk_decode")
    return out


def sign_vote(signs, *, M, n, stride_words=None):
    s = np.ascontiguousarray(signs, dtype=np.uint32)
    if stride_words is None:
        stride_words = s.shape[-1] if s.ndim == 2 else code_words(n, 1)
    out = np.zeros(max(code_words(n, 1), 1), dtype=np.uint32)
    rc = _L().oracle_sign_vote(_ptr(s), stride_words, M, n, _ptr(out))
    _check(rc, "sign_vote")
    return out[:code_words(n, 1)]


def e4m3_to_f32(code: int) -> float:
    return float(_L().oracle_e4m3_to_f32(code))


def e4m3_from_f32(x: float) -> int:
    return int(_L().oracle_e4m3_from_f32(x))


def e4m3_from_f32_array(x):
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint8)
    _L().oracle_e4m3_from_f32_array(_ptr(x), x.size, _ptr(out))
    return out


def rowwise_fp8(x):
    x = np.ascontiguousarray(x, dtype=np.float32)
    rows, dim = x.shape
    codes = np.zeros((rows, dim), dtype=np.uint8)
    scale = np.zeros(rows, dtype=np.float32)
    _check(_L().oracle_rowwise_fp8(_ptr(x), rows, dim, _ptr(codes), _ptr(scale)),
           "rowwise_fp8")
    return codes, scale


def rowwise_fp8_dequant(codes, row_scale):
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    s = np.ascontiguousarray(row_scale, dtype=np.float32)
    rows, dim = c.shape
    out = np.zeros((rows, dim), dtype=np.float32)
    _check(_L().oracle_rowwise_fp8_dequant(_ptr(c), _ptr(s), rows, dim, _ptr(out)),
           "rowwise_fp8_dequant")
    return out

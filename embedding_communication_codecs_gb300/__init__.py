"""GB300-native communication codec (libqcodec) for data-parallel training.

The encode half compresses a gradient for the wire with error feedback. The
options are uniform min/max levels at 8/4/2/1 bits (round to nearest or Philox
stochastic rounding), TernGrad ternary and scaled sign. FP32 -> FP8 e4m3
row-wise quantization covers embedding payloads. The decode half dequantizes
and accumulates M workers' payloads in fp32 in a fixed worker order. It also
majority-votes signSGD sign vectors.

Every step runs in hand-written CUDA kernels for sm_103a inside ``libqcodec.so``.
The functions here only pass torch tensors' device pointers and the current
stream through the C ABI declared in ``include/qcodec.h``, under the same names.
There is no CPU fallback: importing this package fails if the library has not
been built (``python embedding_communication_codecs_gb300/build.py``).
"""
from __future__ import annotations

import ctypes
import os

from .build import LIB_PATH

QC_OK, QC_ERR_NULL, QC_ERR_INVALID_ARG, QC_ERR_ALIGNMENT, QC_ERR_UNSUPPORTED, QC_ERR_CUDA = range(6)
QC_SCHEME_UNIFORM, QC_SCHEME_SIGN, QC_SCHEME_TERNARY, QC_SCHEME_QSGD = 0, 1, 2, 3
QC_SCHEME_UNIFORM_CLIP = 4
QC_SCHEME_LOG = 5
QC_ROUND_NEAREST, QC_ROUND_STOCHASTIC = 0, 1
QC_DTYPE_F32, QC_DTYPE_BF16 = 0, 1
QC_OUT_SUM, QC_OUT_MEAN, QC_ACCUMULATE_INTO_OUT = 0, 1, 2
QC_MAX_WORKERS = 1024
QC_MAX_FP8_DIM = 4096
QC_MAX_SEGMENTS_PER_LAUNCH = 60

STATUS_NAMES = {0: "QC_OK", 1: "QC_ERR_NULL", 2: "QC_ERR_INVALID_ARG", 3: "QC_ERR_ALIGNMENT",
                4: "QC_ERR_UNSUPPORTED", 5: "QC_ERR_CUDA"}

# Every symbol the C ABI exports, in header order.
EXPORTS = ("qc_code_words", "qc_num_buckets", "qc_encode_ef", "qc_encode_ef_segments",
           "qc_decode_accumulate",
           "qc_reencode", "qc_topk_encode_ef", "qc_topk_decode_accumulate", "qc_sign_vote", "qc_rowwise_fp8", "qc_rowwise_fp8_dequant", "qc_take_device_errors",
           "qc_set_status_word", "qc_selftest_wait_timeout",
           "qc_last_error", "qc_version")


class QCodecError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class QcSegment(ctypes.Structure):
    """One flat gradient of qc_encode_ef_segments (the C struct qc_segment)."""
    _fields_ = [("grad", ctypes.c_void_p), ("err", ctypes.c_void_p), ("n", ctypes.c_size_t),
                ("codes", ctypes.c_void_p), ("scale", ctypes.c_void_p),
                ("offset", ctypes.c_void_p)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with "
                          "`python embedding_communication_codecs_gb300/build.py`")
    lib = ctypes.CDLL(LIB_PATH)
    P, S, I = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
    U64, U32 = ctypes.c_uint64, ctypes.c_uint32
    lib.qc_code_words.argtypes, lib.qc_code_words.restype = [S, I], S
    lib.qc_num_buckets.argtypes, lib.qc_num_buckets.restype = [S, S], S
    lib.qc_encode_ef.argtypes = [P, I, P, S, I, S, I, I, U64, U32, P, P, P, P]
    lib.qc_encode_ef_segments.argtypes = [ctypes.POINTER(QcSegment), I, I, I, S, I, I, U64, U32, P]
    lib.qc_decode_accumulate.argtypes = [P, S, P, P, S, I, S, I, S, I, P, I, P]
    lib.qc_reencode.argtypes = [P, S, P, P, S, I, S, I, S, I, I, P, I, U64, U32, P, P, P, P, P]
    lib.qc_topk_encode_ef.argtypes = [P, I, P, S, S, U32, I, U64, U32, P, P, P, P, P]
    lib.qc_topk_decode_accumulate.argtypes = [P, P, S, P, P, S, I, S, S, U32, P, I, P]
    lib.qc_sign_vote.argtypes = [P, S, I, S, P, P]
    lib.qc_rowwise_fp8.argtypes = [P, S, S, P, P, P]
    lib.qc_rowwise_fp8_dequant.argtypes = [P, P, S, S, P, P]
    for name in ("qc_encode_ef", "qc_encode_ef_segments", "qc_decode_accumulate", "qc_reencode", "qc_topk_encode_ef",
                 "qc_topk_decode_accumulate", "qc_sign_vote",
                 "qc_rowwise_fp8",
                 "qc_rowwise_fp8_dequant"):
        getattr(lib, name).restype = I
    lib.qc_take_device_errors.argtypes, lib.qc_take_device_errors.restype = [P], I
    lib.qc_selftest_wait_timeout.argtypes, lib.qc_selftest_wait_timeout.restype = [U32, P], I
    lib.qc_set_status_word.argtypes, lib.qc_set_status_word.restype = [P], I
    lib.qc_last_error.argtypes, lib.qc_last_error.restype = [], ctypes.c_char_p
    lib.qc_version.argtypes, lib.qc_version.restype = [], ctypes.c_char_p
    return lib


lib = _load()


def _check(status: int):
    if status != QC_OK:
        raise QCodecError(status, lib.qc_last_error().decode())


def _ptr(t):
    """Device address of a tensor (None -> NULL).  Integers pass through, so raw
    addresses can be given too."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


# ------------------------------------------------------- argument validation
#
# The C ABI takes raw addresses and sizes, so it cannot see a tensor's dtype,
# device, layout or length.  Before any call the wrappers check every torch
# tensor they are given against what the call will read or write: its dtype,
# that its rows are dense (flat buffers: contiguous), that it holds at least the
# bytes the call touches; and, only after every argument has passed those,
# that each lives on a CUDA device (so the other checks can be exercised
# without a GPU).  A mismatch raises ValueError and
# nothing is launched.  Raw integer addresses are passed through unchecked.

def _torch():
    import torch
    return torch


def _extent_bytes(t) -> int:
    """Bytes from t's first element to one past its last (non-negative strides)."""
    if t.numel() == 0:
        return 0
    return (sum((n - 1) * st for n, st in zip(t.shape, t.stride())) + 1) * t.element_size()


def _need(t, name, nbytes, dtypes=None, flat=True):
    """Check a tensor argument; `flat` asks for a contiguous buffer, otherwise
    only the innermost dimension must be dense (stacked payload rows)."""
    if t is None or isinstance(t, int):
        return
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise ValueError(f"{name} must be a torch tensor or an integer address")
    if dtypes is not None and t.dtype not in dtypes:
        raise ValueError(f"{name} has dtype {t.dtype}; expected one of {tuple(dtypes)}")
    if t.is_contiguous():   # the common case: a dense buffer, its extent is its size
        extent = t.numel() * t.element_size()
    else:
        if any(st < 0 for st in t.stride()):
            raise ValueError(f"{name} has a negative stride")
        if flat:
            raise ValueError(f"{name} must be contiguous")
        if t.dim() > 0 and t.shape[-1] > 1 and t.stride(-1) != 1:
            raise ValueError(f"{name} must be dense along its last dimension")
        extent = _extent_bytes(t)
    if extent < nbytes:
        raise ValueError(f"{name} spans {extent} bytes; the call needs {nbytes}")


def _on_device(**tensors):
    """The last check of every call: each tensor argument lives on a CUDA device."""
    for name, t in tensors.items():
        if t is not None and not isinstance(t, int) and not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")


def _row_stride(t, name, stride_elems, M):
    """With M > 1 a 2-D payload tensor's row stride must be the stride passed."""
    if M > 1 and t is not None and not isinstance(t, int) and t.dim() == 2:
        if t.stride(0) * t.element_size() != stride_elems * 4:
            raise ValueError(f"{name}'s row stride ({t.stride(0)} elements) differs from the "
                             f"stride passed ({stride_elems} 4-byte units)")


_DTYPES = {}


def _words32():
    if "w" not in _DTYPES:
        torch = _torch()
        _DTYPES["w"] = (torch.int32, torch.uint32) if hasattr(torch, "uint32") else (torch.int32,)
    return _DTYPES["w"]


def _f32():
    if "f" not in _DTYPES:
        _DTYPES["f"] = (_torch().float32,)
    return _DTYPES["f"]


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def qc_selftest_wait_timeout(timeout_us, stream=None):
    """One block whose bounded wait runs out after timeout_us microseconds."""
    _check(lib.qc_selftest_wait_timeout(timeout_us, _stream(stream)))


def qc_set_status_word(status):
    """Launches from this thread report failures into the device word `status`
    (a one-element int32 CUDA tensor or an address; None turns it off)."""
    if status is not None and not isinstance(status, int):
        _need(status, "status", 4, _words32())
        _on_device(status=status)
    _check(lib.qc_set_status_word(_ptr(status)))


def qc_take_device_errors() -> int:
    """Synchronise the device and return (and clear) the pipelined kernels'
    device-side error flags; 0 means no wait ever timed out."""
    flags = ctypes.c_uint32(0)
    _check(lib.qc_take_device_errors(ctypes.byref(flags)))
    return int(flags.value)


def qc_version() -> str:
    return lib.qc_version().decode()


def qc_code_words(n: int, bits: int) -> int:
    return int(lib.qc_code_words(n, bits))


def qc_num_buckets(n: int, bucket: int) -> int:
    return int(lib.qc_num_buckets(n, bucket))


def _dtype_code(grad, dtype):
    if dtype is not None:
        return dtype
    import torch
    if grad.dtype == torch.float32:
        return QC_DTYPE_F32
    if grad.dtype == torch.bfloat16:
        return QC_DTYPE_BF16
    raise TypeError(f"gradient dtype {grad.dtype} is not float32 or bfloat16")


def qc_encode_ef(grad, err, n, bits, bucket, scheme, mode, seed, step, codes, scale, offset,
                 stream=None, dtype=None):
    """Sender half: error-feedback encode of ``n`` gradient elements.

    ``err`` (fp32, in/out) may be None for no error feedback; ``offset`` may be
    None unless ``scheme`` is uniform.  Raises QCodecError on a non-OK status."""
    if n:   # n == 0 is a no-op that reads and writes nothing
        if not isinstance(grad, int):
            dt = _dtype_code(grad, dtype)
            torch = _torch()
            want = (torch.float32,) if dt == QC_DTYPE_F32 else (torch.bfloat16, torch.int16)
            _need(grad, "grad", n * (4 if dt == QC_DTYPE_F32 else 2), want)
        nb = qc_num_buckets(n, bucket) if bucket else 0
        _need(err, "err", 4 * n, _f32())
        _need(codes, "codes", 4 * qc_code_words(n, bits), _words32())
        _need(scale, "scale", 4 * nb, _f32())
        if scheme in (QC_SCHEME_UNIFORM, QC_SCHEME_UNIFORM_CLIP):
            _need(offset, "offset", 4 * nb, _f32())
        _on_device(grad=grad, err=err, codes=codes, scale=scale, offset=offset)
    _check(lib.qc_encode_ef(_ptr(grad), _dtype_code(grad, dtype), _ptr(err), n, bits, bucket,
                            scheme, mode, seed, step, _ptr(codes), _ptr(scale), _ptr(offset),
                            _stream(stream)))


def segment_draw_bases(sizes):
    """The draw index of element 0 of each segment of a qc_encode_ef_segments
    call: the segments laid end to end, each padded to a multiple of 4."""
    out, base = [], 0
    for n in sizes:
        out.append(base)
        base += (int(n) + 3) & ~3
    return out


def qc_encode_ef_segments(segments, dtype, bits, bucket, scheme, mode, seed, step, stream=None):
    """qc_encode_ef over a list of flat gradients in one launch.

    ``segments`` holds (grad, err, n, codes, scale, offset) tuples, each as for
    qc_encode_ef; element i of segment s draws with the index I_s + i, I_s the
    sum of the earlier segments' n, each rounded up to a multiple of 4
    (segment_draw_bases).  Every tensor is checked before anything runs."""
    torch = _torch()
    segs = []
    for k, (grad, err, n, codes, scale, offset) in enumerate(segments):
        if n:
            if not isinstance(grad, int):
                want = (torch.float32,) if dtype == QC_DTYPE_F32 else (torch.bfloat16, torch.int16)
                _need(grad, f"segment {k} grad", n * (4 if dtype == QC_DTYPE_F32 else 2), want)
            nb = qc_num_buckets(n, bucket) if bucket else 0
            _need(err, f"segment {k} err", 4 * n, _f32())
            _need(codes, f"segment {k} codes", 4 * qc_code_words(n, bits), _words32())
            _need(scale, f"segment {k} scale", 4 * nb, _f32())
            if scheme in (QC_SCHEME_UNIFORM, QC_SCHEME_UNIFORM_CLIP):
                _need(offset, f"segment {k} offset", 4 * nb, _f32())
        segs.append((grad, err, n, codes, scale, offset))
    for grad, err, n, codes, scale, offset in segs:
        if n:
            _on_device(grad=grad, err=err, codes=codes, scale=scale, offset=offset)
    arr = (QcSegment * max(1, len(segs)))()
    for k, (grad, err, n, codes, scale, offset) in enumerate(segs):
        arr[k] = QcSegment(_ptr(grad), _ptr(err), n, _ptr(codes), _ptr(scale), _ptr(offset))
    _check(lib.qc_encode_ef_segments(arr, len(segs), dtype, bits, bucket, scheme, mode, seed, step,
                                     _stream(stream)))


def _check_payloads(codes, codes_stride_words, scale, offset, meta_stride, M, n, bits, bucket,
                    scheme):
    """The M stacked payloads a decode or re-encode reads."""
    words = qc_code_words(n, bits)
    nb = qc_num_buckets(n, bucket) if bucket else 0
    cs, ms = (codes_stride_words, meta_stride) if M > 1 else (0, 0)
    _need(codes, "codes", 4 * ((M - 1) * cs + words), _words32(), flat=False)
    _need(scale, "scale", 4 * ((M - 1) * ms + nb), _f32(), flat=False)
    _row_stride(codes, "codes", codes_stride_words, M)
    _row_stride(scale, "scale", meta_stride, M)
    if scheme in (QC_SCHEME_UNIFORM, QC_SCHEME_UNIFORM_CLIP):
        _need(offset, "offset", 4 * ((M - 1) * ms + nb), _f32(), flat=False)
        _row_stride(offset, "offset", meta_stride, M)


def qc_decode_accumulate(codes, codes_stride_words, scale, offset, meta_stride, M, n, bits,
                         bucket, scheme, out, flags=QC_OUT_SUM, stream=None):
    """Receiver half: ``out`` = fixed-order fp32 sum (or mean) of M decoded payloads."""
    if n:   # an empty call reads and writes nothing
        _check_payloads(codes, codes_stride_words, scale, offset, meta_stride, M, n, bits, bucket,
                        scheme)
        _need(out, "out", 4 * n, _f32())
        _on_device(codes=codes, scale=scale, offset=offset, out=out)
    _check(lib.qc_decode_accumulate(_ptr(codes), codes_stride_words, _ptr(scale), _ptr(offset),
                                    meta_stride, M, n, bits, bucket, scheme, _ptr(out), flags,
                                    _stream(stream)))


def qc_reencode(codes, codes_stride_words, scale, offset, meta_stride, M, n, bits, bucket,
                scheme, flags, err, mode, seed, step, codes_out, scale_out, offset_out, out=None,
                stream=None):
    """Receiver re-encode: decode and accumulate M payloads (sum, or mean with
    QC_OUT_MEAN), then encode the result with the residual ``err`` (fp32,
    in/out, or None) in the same scheme, bits and bucket.  ``out`` (optional)
    receives the decoded result itself."""
    if n:   # an empty call reads and writes nothing
        _check_payloads(codes, codes_stride_words, scale, offset, meta_stride, M, n, bits, bucket,
                        scheme)
        nb = qc_num_buckets(n, bucket) if bucket else 0
        _need(err, "err", 4 * n, _f32())
        _need(out, "out", 4 * n, _f32())
        _need(codes_out, "codes_out", 4 * qc_code_words(n, bits), _words32())
        _need(scale_out, "scale_out", 4 * nb, _f32())
        if scheme == QC_SCHEME_UNIFORM:
            _need(offset_out, "offset_out", 4 * nb, _f32())
        _on_device(codes=codes, scale=scale, offset=offset, err=err, out=out, codes_out=codes_out,
                   scale_out=scale_out, offset_out=offset_out)
    _check(lib.qc_reencode(_ptr(codes), codes_stride_words, _ptr(scale), _ptr(offset),
                           meta_stride, M, n, bits, bucket, scheme, flags, _ptr(err), mode, seed,
                           step, _ptr(codes_out), _ptr(scale_out), _ptr(offset_out), _ptr(out),
                           _stream(stream)))


def qc_topk_encode_ef(grad, err, n, bucket, keep, mode, seed, step, idx, codes, scale, offset,
                      stream=None, dtype=None):
    """Top-k sparsification per bucket with 8-bit codes of the kept values and
    error feedback (``err`` may be None); outputs keep slots per bucket."""
    if n:   # an empty call reads and writes nothing
        torch = _torch()
        if not isinstance(grad, int):
            dt = _dtype_code(grad, dtype)
            want = (torch.float32,) if dt == QC_DTYPE_F32 else (torch.bfloat16, torch.int16)
            _need(grad, "grad", n * (4 if dt == QC_DTYPE_F32 else 2), want)
        nb = qc_num_buckets(n, bucket) if bucket else 0
        _need(err, "err", 4 * n, _f32())
        _need(idx, "idx", 4 * nb * keep, _words32())
        _need(codes, "codes", nb * keep, (torch.uint8, torch.int8))
        _need(scale, "scale", 4 * nb, _f32())
        _need(offset, "offset", 4 * nb, _f32())
        _on_device(grad=grad, err=err, idx=idx, codes=codes, scale=scale, offset=offset)
    _check(lib.qc_topk_encode_ef(_ptr(grad), _dtype_code(grad, dtype), _ptr(err), n, bucket, keep,
                                 mode, seed, step, _ptr(idx), _ptr(codes), _ptr(scale),
                                 _ptr(offset), _stream(stream)))


def qc_topk_decode_accumulate(idx, codes, pair_stride, scale, offset, meta_stride, M, n, bucket,
                              keep, out, flags=QC_OUT_SUM, stream=None):
    """Scatter M workers' top-k pairs into a dense fp32 vector in worker order."""
    if n:   # an empty call reads and writes nothing
        torch = _torch()
        nb = qc_num_buckets(n, bucket) if bucket else 0
        ps, ms = (pair_stride, meta_stride) if M > 1 else (0, 0)
        _need(idx, "idx", 4 * ((M - 1) * ps + nb * keep), _words32(), flat=False)
        _need(codes, "codes", (M - 1) * ps + nb * keep, (torch.uint8, torch.int8), flat=False)
        _need(scale, "scale", 4 * ((M - 1) * ms + nb), _f32(), flat=False)
        _need(offset, "offset", 4 * ((M - 1) * ms + nb), _f32(), flat=False)
        _need(out, "out", 4 * n, _f32())
        _on_device(idx=idx, codes=codes, scale=scale, offset=offset, out=out)
    _check(lib.qc_topk_decode_accumulate(_ptr(idx), _ptr(codes), pair_stride, _ptr(scale),
                                         _ptr(offset), meta_stride, M, n, bucket, keep, _ptr(out),
                                         flags, _stream(stream)))


def qc_sign_vote(signs, stride_words, M, n, out, stream=None):
    """Majority vote over M packed sign vectors."""
    if n:   # an empty call reads and writes nothing
        words = qc_code_words(n, 1)
        _need(signs, "signs", 4 * ((M - 1) * (stride_words if M > 1 else 0) + words), _words32(),
              flat=False)
        _row_stride(signs, "signs", stride_words, M)
        _need(out, "out", 4 * words, _words32())
        _on_device(signs=signs, out=out)
    _check(lib.qc_sign_vote(_ptr(signs), stride_words, M, n, _ptr(out), _stream(stream)))


def qc_rowwise_fp8(x, rows, dim, codes, row_scale, stream=None):
    """FP32 rows -> E4M3 codes + per-row fp32 scale."""
    if rows:   # an empty call reads and writes nothing
        torch = _torch()
        _need(x, "x", 4 * rows * dim, _f32())
        _need(codes, "codes", rows * dim, (torch.uint8, torch.int8))
        _need(row_scale, "row_scale", 4 * rows, _f32())
        _on_device(x=x, codes=codes, row_scale=row_scale)
    _check(lib.qc_rowwise_fp8(_ptr(x), rows, dim, _ptr(codes), _ptr(row_scale), _stream(stream)))


def qc_rowwise_fp8_dequant(codes, row_scale, rows, dim, out, stream=None):
    """E4M3 codes + per-row scale -> fp32 rows."""
    if rows:   # an empty call reads and writes nothing
        torch = _torch()
        _need(codes, "codes", rows * dim, (torch.uint8, torch.int8))
        _need(row_scale, "row_scale", 4 * rows, _f32())
        _need(out, "out", 4 * rows * dim, _f32())
        _on_device(codes=codes, row_scale=row_scale, out=out)
    _check(lib.qc_rowwise_fp8_dequant(_ptr(codes), _ptr(row_scale), rows, dim, _ptr(out),
                                      _stream(stream)))


# ---------------------------------------------------------------- conveniences

def alloc_payload(n: int, bits: int, bucket: int, scheme: int, device="cuda", workers: int = 0):
    """Empty (codes, scale, offset) device tensors for one payload, or for
    ``workers`` payloads stacked along a leading dimension when workers > 0.
    Offset is None except for the uniform scheme."""
    import torch
    words = qc_code_words(n, bits)
    nb = qc_num_buckets(n, bucket)
    lead = (workers,) if workers else ()
    codes = torch.empty(lead + (words,), dtype=torch.int32, device=device)
    scale = torch.empty(lead + (nb,), dtype=torch.float32, device=device)
    offset = (torch.empty(lead + (nb,), dtype=torch.float32, device=device)
              if scheme in (QC_SCHEME_UNIFORM, QC_SCHEME_UNIFORM_CLIP) else None)
    return codes, scale, offset


def encode_ef(grad, err, *, bits, bucket, scheme=QC_SCHEME_UNIFORM, mode=QC_ROUND_NEAREST,
              seed=0, step=0, out=None, stream=None):
    """Encode a flat device tensor; returns (codes int32[words], scale, offset)."""
    n = grad.numel()
    codes, scale, offset = out if out is not None else alloc_payload(n, bits, bucket, scheme,
                                                                     grad.device)
    qc_encode_ef(grad, err, n, bits, bucket, scheme, mode, seed, step, codes, scale, offset,
                 stream=stream)
    return codes, scale, offset


def decode_accumulate(codes, scale, offset, *, n, bits, bucket, scheme=QC_SCHEME_UNIFORM,
                      flags=QC_OUT_SUM, out=None, stream=None):
    """Decode stacked payloads ([M, words] codes, [M, nb] scale/offset) or a single
    payload (1-D) into a fresh or given fp32 tensor of n elements."""
    import torch
    M = codes.shape[0] if codes.dim() == 2 else 1
    cs = codes.stride(0) if codes.dim() == 2 else 0
    ms = scale.stride(0) if scale.dim() == 2 else 0
    if out is None:
        out = torch.empty(n, dtype=torch.float32, device=codes.device)
    qc_decode_accumulate(codes, cs, scale, offset, ms, M, n, bits, bucket, scheme, out, flags,
                         stream=stream)
    return out

"""The oracle over a whole workload, as it stands, on every host core: the
workload is cut into bucket-aligned slices, each slice is encoded by the
oracle with its global index base (so stochastic draws and outputs are exactly
those of one whole-array call) in its own thread (the ctypes calls release the
GIL), and the slices' outputs are concatenated.  Test infrastructure only."""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

import oracle as orc


def _cores() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def slices(n: int, align: int, parts: int | None = None):
    parts = parts or _cores()
    per = -(-(-(-n // parts)) // align) * align
    per = max(per, align)
    return [(lo, min(n, lo + per)) for lo in range(0, n, per)]


def _run(fn, parts):
    with ThreadPoolExecutor(len(parts)) as ex:
        return list(ex.map(fn, parts))


def encode(fn, g, err, *, bucket, index=True, base=0, **kw):
    """fn(g[lo:hi], err[lo:hi], bucket=bucket, index_base=base + lo, **kw) over
    every slice; returns the outputs concatenated (err is updated in place)."""
    def one(p):
        lo, hi = p
        args = dict(kw, bucket=bucket)
        if index:
            args["index_base"] = base + lo
        return fn(g[lo:hi], None if err is None else err[lo:hi], **args)
    res = _run(one, slices(g.shape[-1], bucket))
    return tuple(np.concatenate([r[i] for r in res]) for i in range(len(res[0])))


def decode(codes, scale, offset, *, M, n, bits, bucket, scheme, flags=orc.OUT_SUM):
    """decode_accumulate of M stacked payloads ([M, words], [M, buckets])."""
    codes = codes.reshape(M, -1)
    scale = scale.reshape(M, -1)
    offset = None if offset is None else offset.reshape(M, -1)
    out = np.empty(n, dtype=np.float32)

    def one(p):
        lo, hi = p
        w0, w1 = lo * bits // 32, (hi * bits + 31) // 32
        k0, k1 = lo // bucket, -(-hi // bucket)
        out[lo:hi] = orc.decode_accumulate(
            np.ascontiguousarray(codes[:, w0:w1]), np.ascontiguousarray(scale[:, k0:k1]),
            None if offset is None else np.ascontiguousarray(offset[:, k0:k1]), M=M, n=hi - lo,
            bits=bits, bucket=bucket, scheme=scheme, flags=flags)
    _run(one, slices(n, bucket))
    return out


def sign_vote(signs, *, M, n):
    words = (n + 31) // 32
    out = np.empty(words, dtype=np.uint32)

    def one(p):
        lo, hi = p
        w0, w1 = lo // 32, (hi + 31) // 32
        out[w0:w1] = orc.sign_vote(np.ascontiguousarray(signs[:, w0:w1]), M=M, n=hi - lo)
    _run(one, slices(n, 32 * 1024))
    return out

"""Seeded synthetic inputs for the codec, shared by the tests, the smoke check and
the benchmark.  This module holds no codec arithmetic: it only draws random
numbers (numpy PCG64) and lays them out like the pages' workloads.

Every stream is generated in independent chunks of ``CHUNK`` elements, each from
its own ``SeedSequence([seed, tag, chunk])``, so any slice can be regenerated on
its own and large arrays are drawn in parallel threads.

Workloads (sizes and distributions of the pages' examples):

* ``outlier_gradient``     -- fp32 gradient ~ N(0, 1e-3) with 0.1% outliers
  ~ N(0, 1e-1) (uniform 8-bit error-feedback encode, buckets of 2048).
* ``embedding_rows``       -- 1,000,000 x 128 fp32 ~ N(0, 0.05): the embedding
  lookup payload of the FP32 -> FP8 numeric example.
* ``bucket_sigma_gradient``-- flat fp32 gradient, per-bucket std drawn
  log-uniform in [1e-5, 1e-2], a fresh N(0, std) draw per step (4-bit
  stochastic rounding with error feedback over 10 steps).
* ``shared_mean_gradients``-- M workers' fp32 gradients N(mu, 1e-3) around a
  shared mean mu ~ N(0, 5e-4) (signSGD with majority vote, ResNet-50 size).
* ``bf16_gradients``       -- M workers' N(0, 1e-3) gradients rounded to bf16
  (receiver side of a quantized all-reduce).
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

CHUNK = 1 << 20

# Stream tags (any distinct integers).
TAG_NORMAL = 1
TAG_OUTLIER_NORMAL = 2
TAG_OUTLIER_MASK = 3
TAG_SIGMA = 4
TAG_STEP_BASE = 100      # + step
TAG_MEAN = 5
TAG_WORKER_BASE = 1000   # + worker


def _threads() -> int:
    try:
        return max(1, min(32, len(os.sched_getaffinity(0))))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def _gen(seed: int, tag: int, chunk: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tag, chunk])))


def _fill(n: int, dtype, fn) -> np.ndarray:
    out = np.empty(n, dtype=dtype)
    nchunks = (n + CHUNK - 1) // CHUNK

    def work(c):
        lo = c * CHUNK
        hi = min(n, lo + CHUNK)
        fn(c, out[lo:hi])

    if nchunks <= 1:
        for c in range(nchunks):
            work(c)
    else:
        with ThreadPoolExecutor(_threads()) as ex:
            list(ex.map(work, range(nchunks)))
    return out


def std_normal(seed: int, tag: int, n: int) -> np.ndarray:
    """float32 N(0, 1), chunk-seeded."""
    def fn(c, view):
        _gen(seed, tag, c).standard_normal(out=view, dtype=np.float32)
    return _fill(n, np.float32, fn)


def std_uniform(seed: int, tag: int, n: int) -> np.ndarray:
    """float64 U[0, 1), chunk-seeded."""
    def fn(c, view):
        _gen(seed, tag, c).random(out=view)
    return _fill(n, np.float64, fn)


def outlier_gradient(n: int = 1 << 20, seed: int = 0, sigma: float = 1e-3,
                     outlier_sigma: float = 1e-1, outlier_rate: float = 1e-3) -> np.ndarray:
    g = std_normal(seed, TAG_NORMAL, n)
    g *= np.float32(sigma)
    mask = std_uniform(seed, TAG_OUTLIER_MASK, n) < outlier_rate
    big = std_normal(seed, TAG_OUTLIER_NORMAL, n)
    g[mask] = big[mask] * np.float32(outlier_sigma)
    return g


def embedding_rows(rows: int = 1_000_000, dim: int = 128, seed: int = 1,
                   sigma: float = 0.05) -> np.ndarray:
    x = std_normal(seed, TAG_NORMAL, rows * dim)
    x *= np.float32(sigma)
    return x.reshape(rows, dim)


def bucket_sigmas(n: int, bucket: int, seed: int = 2, lo_exp: float = -5.0,
                  hi_exp: float = -2.0) -> np.ndarray:
    """Per-bucket std 10**U(lo_exp, hi_exp), drawn once and fixed across steps."""
    nb = (n + bucket - 1) // bucket
    u = std_uniform(seed, TAG_SIGMA, nb)
    return (10.0 ** (lo_exp + (hi_exp - lo_exp) * u)).astype(np.float32)


def bucket_sigma_gradient(n: int, bucket: int, step: int, seed: int = 2,
                          sigmas: np.ndarray | None = None) -> np.ndarray:
    """Step ``step``'s fresh draw g_t = sigma_k * z."""
    if sigmas is None:
        sigmas = bucket_sigmas(n, bucket, seed)
    z = std_normal(seed, TAG_STEP_BASE + step, n)
    nb = sigmas.size

    def scale(c):
        lo = c * CHUNK
        hi = min(n, lo + CHUNK)
        idx = np.arange(lo, hi, dtype=np.int64) // bucket
        z[lo:hi] *= sigmas[np.minimum(idx, nb - 1)]

    nchunks = (n + CHUNK - 1) // CHUNK
    with ThreadPoolExecutor(_threads()) as ex:
        list(ex.map(scale, range(nchunks)))
    return z


def shared_mean_gradients(n: int, M: int, seed: int = 3, mean_sigma: float = 5e-4,
                          sigma: float = 1e-3) -> np.ndarray:
    """[M, n] float32: worker w holds mu + sigma * z_w, mu = mean_sigma * z shared."""
    mu = std_normal(seed, TAG_MEAN, n)
    mu *= np.float32(mean_sigma)
    out = np.empty((M, n), dtype=np.float32)
    for w in range(M):
        z = std_normal(seed, TAG_WORKER_BASE + w, n)
        z *= np.float32(sigma)
        np.add(mu, z, out=out[w])
    return out


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest-even, via torch on the CPU); returns uint16 bits."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def bf16_gradients(n: int, M: int, seed: int = 4, sigma: float = 1e-3) -> np.ndarray:
    """[M, n] uint16 bf16 bit patterns of sigma * z_w, workers drawn in order."""
    out = np.empty((M, n), dtype=np.uint16)
    for w in range(M):
        z = std_normal(seed, TAG_WORKER_BASE + w, n)
        z *= np.float32(sigma)
        out[w] = to_bf16_bits(z)
    return out


# Full-size workloads of the five configurations (parameters only).
CONFIGS = {
    "u8_ef_outliers": dict(n=1 << 20, bits=8, bucket=2048, mode="nearest", seed=0, ef=True),
    "fp8_rowwise": dict(rows=1_000_000, dim=128, seed=1),
    "sr4_ef_10step": dict(n=250_000_000, bits=4, bucket=512, mode="stochastic", seed=2,
                          steps=10, ef=True),
    "sign_ef_vote": dict(n=25_600_000, M=8, bucket=4096, seed=3, ef=True),
    "allreduce_rx_bf16": dict(n=1 << 26, M=16, bits=8, bucket=1024, seed=4,
                              ternary_bucket=1024),
}

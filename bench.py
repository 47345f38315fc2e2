#!/usr/bin/env python
"""Benchmark of the communication codec's hot path on one GB300.

One step runs every row of the hot path once over its full-size synthetic
workload, with inputs resident in HBM:
  fp8_rowwise   FP32 -> E4M3 row-wise quantize, then dequantize, 1,000,000 x 128.
  sr4_ef        4-bit stochastic rounding with error feedback over 250,000,000
                elements (buckets of 512, Philox keyed (2, step, index)). The
                step counter advances each step. Then decode with M = 1.
  sign_ef_vote  scaled sign with error feedback for 8 workers x 25,600,000
                (buckets of 4096). Then the majority vote over the 8 sign vectors.
  rx_u8         16 workers x 2^26 bf16 -> 8-bit uniform (buckets of 1024, no
                error feedback). Then decode-accumulate MEAN over M = 16.
  rx_ternary    the same 16 workers -> TernGrad 2-bit stochastic. Then decode
                MEAN over M = 16.

The metric is codec GB/s of fp32 gradient: 4 bytes x the gradient elements the
step encodes or decodes (the payload elements for decode and vote, rows x dim
for FP8), divided by the device time of the step.  Alongside it: the
algorithmic HBM bytes per step, the dominant kernel's roofline against the
measured HBM copy peak, the oracle's CPU throughput on a bounded sample, and
the end-to-end rate through the public API with host buffers.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload suite|fp8_rowwise|sr4_ef|sign_ef_vote|rx_u8|rx_ternary|u8_ef_small|u8_ef_large]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time
from concurrent.futures import ThreadPoolExecutor

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import workloads as wl  # noqa: E402

METRIC = "codec GB/s of fp32 gradient (encode+EF, decode+accumulate) vs GB300 HBM peak"
UNIT = "GB/s"
PEAK_FALLBACK_GBS = 6800.0


# ----------------------------------------------------------------- workloads

class Component:
    """One row group of the hot path: buffers, launches, byte and unit counts."""

    name = ""
    # kernel name -> (launches per step, algorithmic bytes per launch)
    kernels: dict = {}
    units = 0            # fp32-equivalent elements per step
    h2d = 0              # bytes a step takes from the host in the end-to-end run
    d2h = 0              # bytes a step returns to the host

    def setup(self, q, torch):
        raise NotImplementedError

    def run(self, q, t, timer):
        raise NotImplementedError

    def host_inputs(self):
        """Device tensors refilled from pinned host memory every end-to-end step."""
        return []

    def reads(self):
        """Device tensors the step reads that come from the host (its own inputs
        and any it shares with another component)."""
        return self.host_inputs()

    def host_outputs(self):
        return []

    def oracle_sample(self, frac):
        """A closure running the oracle on about `frac` of this component, and the
        fp32-equivalent elements it processes."""
        raise NotImplementedError

    def kernel_units(self):
        """Elements each launch of each kernel processes (for scaling counters)."""
        return {}

    def quality(self, q, torch):
        """Compression ratio and the error of one more step's result against the
        exact value (torch, outside the timed region); None if not defined."""
        return None


def _rel_rms(torch, got, want):
    d = (got.double() - want.double()).pow(2).mean().sqrt()
    w = want.double().pow(2).mean().sqrt()
    return float(d / w) if float(w) > 0 else 0.0


def _rms_ratio(torch, a, b):
    w = b.double().pow(2).mean().sqrt()
    return float(a.double().pow(2).mean().sqrt() / w) if float(w) > 0 else 0.0


def _words(n, bits):
    return (n * bits + 31) // 32


def _nb(n, b):
    return (n + b - 1) // b


class Fp8Rowwise(Component):
    name = "fp8_rowwise"

    def __init__(self, rows=1_000_000, dim=128, seed=1):
        self.rows, self.dim, self.seed = rows, dim, seed
        nd = rows * dim
        b = 4 * nd + nd + 4 * rows
        self.kernels = {"fp8_quant": (1, b), "fp8_dequant": (1, b)}
        self.units = 2 * nd
        self.h2d = 4 * nd
        self.d2h = 4 * nd

    def setup(self, q, torch):
        x = wl.embedding_rows(self.rows, self.dim, self.seed)
        self.x = torch.from_numpy(x).cuda()
        self.codes = torch.empty((self.rows, self.dim), dtype=torch.uint8, device="cuda")
        self.sc = torch.empty(self.rows, device="cuda")
        self.out = torch.empty_like(self.x)

    def run(self, q, t, timer):
        with timer("fp8_quant"):
            q.qc_rowwise_fp8(self.x, self.rows, self.dim, self.codes, self.sc)
        with timer("fp8_dequant"):
            q.qc_rowwise_fp8_dequant(self.codes, self.sc, self.rows, self.dim, self.out)

    def host_inputs(self):
        return [self.x]

    def host_outputs(self):
        return [self.out]

    def kernel_units(self):
        return {"fp8_quant": self.rows * self.dim, "fp8_dequant": self.rows * self.dim}

    def quality(self, q, torch):
        self.run(q, 0, KernelTimer(torch, enabled=False))
        return {"compression": round(4 * self.dim / (self.dim + 4), 3),
                "rel_rms_error": _rel_rms(torch, self.out, self.x)}

    def oracle_sample(self, frac):
        import oracle as orc
        rows = max(64, int(self.rows * frac))
        x = wl.embedding_rows(rows, self.dim, self.seed)

        def go(lo, hi):
            c, s = orc.rowwise_fp8(x[lo:hi])
            orc.rowwise_fp8_dequant(c, s)
        return _split(go, rows, 1), 2 * rows * self.dim


class UniformEF(Component):
    """Encode with error feedback of one flat fp32 gradient (uniform, QSGD,
    clipped uniform or logarithmic-level scheme), then decode M = 1."""

    def __init__(self, name, n, bits, bucket, stochastic, seed, sigma_mode, scheme=0):
        self.name, self.n, self.bits, self.bucket = name, n, bits, bucket
        self.stochastic, self.seed, self.sigma_mode = stochastic, seed, sigma_mode
        self.scheme = scheme
        words, nb = _words(n, bits), _nb(n, bucket)
        meta = 8 if scheme in (0, 4) else 4
        enc = 12 * n + 4 * words + meta * nb
        dec = 4 * words + meta * nb + 4 * n
        tag = {0: f"u{bits}", 3: f"qsgd{bits}", 4: f"clip{bits}", 5: f"log{bits}"}[scheme]
        self.enc_name, self.dec_name = f"encode_{tag}_ef", f"decode_{tag}_m1"
        self.kernels = {self.enc_name: (1, enc), self.dec_name: (1, dec)}
        self.units = 2 * n
        self.h2d = 4 * n
        self.d2h = 4 * n

    def _grad(self, n, step=0):
        """The first n elements of the workload's gradient of `step` (the
        per-bucket-sigma recipe draws a fresh gradient every step)."""
        if self.sigma_mode == "bucket":
            sig = wl.bucket_sigmas(self.n, self.bucket, self.seed)
            return wl.bucket_sigma_gradient(n, self.bucket, step, self.seed,
                                            sigmas=sig[:(n + self.bucket - 1) // self.bucket])
        return wl.outlier_gradient(n, seed=self.seed)

    def setup(self, q, torch, shared=None):
        """`shared`: another component of the same recipe whose device gradients
        this one reads instead of drawing its own."""
        if shared is not None:
            self.gs = shared.gs
        else:
            self.gs = [torch.from_numpy(self._grad(self.n, 0)).cuda()]
            if self.sigma_mode == "bucket":
                # two independent step draws, alternated step by step, so the
                # residual evolves as under fresh gradients
                self.gs.append(torch.from_numpy(self._grad(self.n, 1)).cuda())
        self.g = self.gs[0]
        self.fixed_input = False
        self.err = torch.zeros(self.n, device="cuda")
        self.codes, self.scale, self.offset = q.alloc_payload(self.n, self.bits, self.bucket,
                                                              self.scheme)
        self.out = torch.empty(self.n, device="cuda")

    def run(self, q, t, timer):
        mode = q.QC_ROUND_STOCHASTIC if self.stochastic else q.QC_ROUND_NEAREST
        g = self.g if self.fixed_input else self.gs[t % len(self.gs)]
        with timer(self.enc_name):
            q.qc_encode_ef(g, self.err, self.n, self.bits, self.bucket, self.scheme, mode,
                           self.seed, t, self.codes, self.scale, self.offset)
        with timer(self.dec_name):
            q.qc_decode_accumulate(self.codes, 0, self.scale, self.offset, 0, 1, self.n, self.bits,
                                   self.bucket, self.scheme, self.out, 0)

    def host_inputs(self):
        return [self.g]

    def host_outputs(self):
        return [self.out]

    def kernel_units(self):
        return {k: self.n for k in self.kernels}

    def quality(self, q, torch):
        e_old = self.err.clone()
        self.run(q, 10_000, KernelTimer(torch, enabled=False))
        meta = 8 if self.scheme in (0, 4) else 4
        p = self.gs[10_000 % len(self.gs)] + e_old
        return {"compression": round(32 / (self.bits + 8 * meta / self.bucket), 3),
                "rel_rms_error_of_step": _rel_rms(torch, self.out, p),
                "residual_rms_over_gradient_rms": _rms_ratio(torch, self.err, self.g)}

    def oracle_sample(self, frac):
        import oracle as orc
        n = max(self.bucket, int(self.n * frac) // self.bucket * self.bucket)
        g = self._grad(n)
        err = np.zeros(n, dtype=np.float32)
        mode = orc.ROUND_STOCHASTIC if self.stochastic else orc.ROUND_NEAREST

        def go(lo, hi):
            if self.scheme in (0, 4):
                enc = orc.encode_uniform if self.scheme == 0 else orc.encode_uniform_clip
                c, s, o = enc(g[lo:hi], err[lo:hi], bits=self.bits, bucket=self.bucket, mode=mode,
                              seed=self.seed, step=0, index_base=lo)
            else:
                enc = orc.encode_qsgd if self.scheme == 3 else orc.encode_log
                (c, s), o = enc(g[lo:hi], err[lo:hi], bits=self.bits, bucket=self.bucket,
                                mode=mode, seed=self.seed, step=0, index_base=lo), None
            orc.decode_accumulate(c, s, o, M=1, n=hi - lo, bits=self.bits, bucket=self.bucket,
                                  scheme=self.scheme)
        return _split(go, n, self.bucket), 2 * n


class SignVote(Component):
    name = "sign_ef_vote"

    def __init__(self, n=25_600_000, M=8, bucket=4096, seed=3):
        self.n, self.M, self.bucket, self.seed = n, M, bucket, seed
        words, nb = _words(n, 1), _nb(n, bucket)
        self.kernels = {"encode_sign_ef": (1, M * (12 * n + 4 * words + 4 * nb)),
                        "sign_vote": (1, (M + 1) * 4 * words)}
        self.units = 2 * M * n
        self.h2d = 4 * M * n
        self.d2h = 4 * words

    def setup(self, q, torch):
        self.g = torch.from_numpy(wl.shared_mean_gradients(self.n, self.M, self.seed)).cuda()
        self.err = torch.zeros((self.M, self.n), device="cuda")
        words, nb = _words(self.n, 1), _nb(self.n, self.bucket)
        self.words = words
        self.signs = torch.empty((self.M, words), dtype=torch.int32, device="cuda")
        self.scale = torch.empty((self.M, nb), device="cuda")
        self.vote = torch.empty(words, dtype=torch.int32, device="cuda")

    def run(self, q, t, timer):
        # the M workers' encodes as the segments of one launch (each with its
        # own residual; the sign scheme draws nothing)
        with timer("encode_sign_ef"):
            q.qc_encode_ef_segments([(self.g[w], self.err[w], self.n, self.signs[w], self.scale[w],
                                      None) for w in range(self.M)],
                                    q.QC_DTYPE_F32, 1, self.bucket, q.QC_SCHEME_SIGN,
                                    q.QC_ROUND_NEAREST, 0, t)
        with timer("sign_vote"):
            q.qc_sign_vote(self.signs, self.words, self.M, self.n, self.vote)

    def host_inputs(self):
        return [self.g]

    def host_outputs(self):
        return [self.vote]

    def kernel_units(self):
        return {"encode_sign_ef": self.M * self.n, "sign_vote": self.M * self.n}

    def quality(self, q, torch):
        self.run(q, 10_000, KernelTimer(torch, enabled=False))
        mean = self.g.mean(dim=0)
        bits = ((self.vote.view(torch.int32).unsqueeze(1) >>
                 torch.arange(32, device="cuda", dtype=torch.int32)) & 1).reshape(-1)[:self.n]
        agree = float(((mean >= 0).to(torch.int32) == bits).float().mean())
        return {"compression": round(32 * self.bucket / (self.bucket + 32), 3),
                "vote_agrees_with_sign_of_mean": round(agree, 5)}

    def oracle_sample(self, frac):
        import oracle as orc
        n = max(self.bucket, int(self.n * frac) // self.bucket * self.bucket)
        gw = wl.shared_mean_gradients(n, self.M, self.seed)

        def go(lo, hi):
            signs = []
            for w in range(self.M):
                c, _ = orc.encode_sign(gw[w, lo:hi], np.zeros(hi - lo, np.float32),
                                       bucket=self.bucket)
                signs.append(c)
            orc.sign_vote(np.stack(signs), M=self.M, n=hi - lo)
        return _split(go, n, self.bucket), 2 * self.M * n


class Receiver(Component):
    """M workers' bf16 gradients encoded without error feedback, then decoded as
    the MEAN over M in fixed worker order."""

    def __init__(self, name, scheme, bits, n=1 << 26, M=16, bucket=1024, seed=4, shared=None):
        self.name, self.scheme, self.bits = name, scheme, bits
        self.n, self.M, self.bucket, self.seed, self.shared = n, M, bucket, seed, shared
        words, nb = _words(n, bits), _nb(n, bucket)
        meta = 8 if scheme == 0 else 4
        tag = "u8" if scheme == 0 else "ternary"
        self.enc_name, self.dec_name = f"encode_{tag}_bf16", f"decode_{tag}_m{M}"
        self.kernels = {self.enc_name: (1, M * (2 * n + 4 * words + meta * nb)),
                        self.dec_name: (1, M * (4 * words + meta * nb) + 4 * n)}
        self.units = 2 * M * n
        self.h2d = 2 * M * n if shared is None else 0
        self.d2h = 4 * n

    def setup(self, q, torch):
        if self.shared is not None and hasattr(self.shared, "g"):
            self.g = self.shared.g
        else:
            self.g = torch.from_numpy(wl.bf16_gradients(self.n, self.M, self.seed)
                                      .view(np.int16)).cuda()
        self.codes, self.scale, self.offset = q.alloc_payload(self.n, self.bits, self.bucket,
                                                              self.scheme, workers=self.M)
        self.out = torch.empty(self.n, device="cuda")

    def encode_all(self, q, t):
        """The M workers' encodes as one multi-segment call (one launch): worker
        w's draws are indexed w * n + i, the workers' gradients laid end to end
        under the one seed."""
        mode = q.QC_ROUND_NEAREST if self.scheme == 0 else q.QC_ROUND_STOCHASTIC
        segs = [(self.g[w], None, self.n, self.codes[w], self.scale[w],
                 self.offset[w] if self.offset is not None else None) for w in range(self.M)]
        q.qc_encode_ef_segments(segs, q.QC_DTYPE_BF16, self.bits, self.bucket, self.scheme, mode,
                                self.seed, t)

    def run(self, q, t, timer):
        with timer(self.enc_name):
            self.encode_all(q, t)
        with timer(self.dec_name):
            q.qc_decode_accumulate(self.codes, self.codes.stride(0), self.scale,
                                   self.offset, self.scale.stride(0), self.M, self.n, self.bits,
                                   self.bucket, self.scheme, self.out, q.QC_OUT_MEAN)

    def host_inputs(self):
        return [self.g] if self.h2d else []

    def reads(self):
        return [self.g]

    def kernel_units(self):
        return {self.enc_name: self.M * self.n, self.dec_name: self.M * self.n}

    def host_outputs(self):
        return [self.out]

    def quality(self, q, torch):
        self.run(q, 10_000, KernelTimer(torch, enabled=False))
        g = self.g.view(torch.bfloat16).float()
        meta = 8 if self.scheme == 0 else 4
        return {"compression_vs_bf16": round(16 / (self.bits + 8 * meta / self.bucket), 3),
                "rel_rms_error_of_mean": _rel_rms(torch, self.out, g.mean(dim=0))}

    def oracle_sample(self, frac):
        import oracle as orc
        n = max(self.bucket, int(self.n * frac) // self.bucket * self.bucket)
        gb = wl.bf16_gradients(n, self.M, self.seed)

        def go(lo, hi):
            cs, ss, os_ = [], [], []
            for w in range(self.M):
                if self.scheme == 0:
                    c, s, o = orc.encode_uniform(gb[w, lo:hi], None, bits=8, bucket=self.bucket,
                                                 index_base=w * self.n + lo)
                    os_.append(o)
                else:
                    c, s = orc.encode_ternary(gb[w, lo:hi], None, bucket=self.bucket,
                                              mode=orc.ROUND_STOCHASTIC, seed=self.seed,
                                              index_base=w * self.n + lo)
                cs.append(c)
                ss.append(s)
            orc.decode_accumulate(np.stack(cs), np.stack(ss), np.stack(os_) if os_ else None,
                                  M=self.M, n=hi - lo, bits=self.bits, bucket=self.bucket,
                                  scheme=self.scheme, flags=orc.OUT_MEAN)
        return _split(go, n, self.bucket), 2 * self.M * n


class TopkEF(Component):
    """M workers' fp32 gradients sparsified to the largest 1 % per bucket with
    8-bit codes and error feedback, then scattered and averaged by the receiver."""

    def __init__(self, name="topk_ef", n=25_600_000, M=8, bucket=1024, keep=10, seed=3):
        self.name, self.n, self.M, self.bucket, self.keep, self.seed = name, n, M, bucket, keep, seed
        nb = _nb(n, bucket)
        self.kernels = {"topk_encode_ef": (M, 12 * n + 5 * nb * keep + 8 * nb),
                        f"topk_decode_m{M}": (1, M * (5 * nb * keep + 8 * nb) + 4 * n)}
        self.units = 2 * M * n
        self.h2d = 4 * M * n
        self.d2h = 4 * n

    def setup(self, q, torch, shared=None):
        """`shared`: the sign workload, whose device gradients (the same recipe)
        this component reads instead of drawing its own."""
        if shared is not None:
            self.g = shared.g
        else:
            self.g = torch.from_numpy(wl.shared_mean_gradients(self.n, self.M, self.seed)).cuda()
        self.err = torch.zeros((self.M, self.n), device="cuda")
        nb = _nb(self.n, self.bucket)
        self.slots = nb * self.keep
        self.idx = torch.empty((self.M, self.slots), dtype=torch.int32, device="cuda")
        self.codes = torch.empty((self.M, self.slots), dtype=torch.uint8, device="cuda")
        self.scale = torch.empty((self.M, nb), device="cuda")
        self.offset = torch.empty((self.M, nb), device="cuda")
        self.out = torch.empty(self.n, device="cuda")

    def run(self, q, t, timer):
        for w in range(self.M):
            with timer("topk_encode_ef"):
                q.qc_topk_encode_ef(self.g[w], self.err[w], self.n, self.bucket, self.keep,
                                    q.QC_ROUND_NEAREST, 0, t, self.idx[w], self.codes[w],
                                    self.scale[w], self.offset[w])
        with timer(f"topk_decode_m{self.M}"):
            q.qc_topk_decode_accumulate(self.idx, self.codes, self.slots, self.scale, self.offset,
                                        self.scale.shape[1], self.M, self.n, self.bucket, self.keep,
                                        self.out, q.QC_OUT_MEAN)

    def host_inputs(self):
        return [self.g]

    def host_outputs(self):
        return [self.out]

    def kernel_units(self):
        return {"topk_encode_ef": self.n, f"topk_decode_m{self.M}": self.M * self.n}

    def quality(self, q, torch):
        self.run(q, 10_000, KernelTimer(torch, enabled=False))
        return {"compression": round(4 * self.bucket / (5 * self.keep + 8), 3),
                "kept_fraction": round(self.keep / self.bucket, 5),
                "rel_rms_error_of_mean": _rel_rms(torch, self.out, self.g.mean(dim=0))}

    def oracle_sample(self, frac):
        import oracle as orc
        n = max(self.bucket, int(self.n * frac) // self.bucket * self.bucket)
        gw = wl.shared_mean_gradients(n, self.M, self.seed)

        def go(lo, hi):
            parts = []
            for w in range(self.M):
                parts.append(orc.topk_encode(gw[w, lo:hi], np.zeros(hi - lo, np.float32),
                                             bucket=self.bucket, keep=self.keep, index_base=0))
            orc.topk_decode(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]),
                            np.stack([p[2] for p in parts]), np.stack([p[3] for p in parts]),
                            M=self.M, n=hi - lo, bucket=self.bucket, keep=self.keep,
                            flags=orc.OUT_MEAN)
        return _split(go, n, self.bucket), 2 * self.M * n


class Reencode(Receiver):
    """M workers' bf16 gradients encoded without error feedback, then the
    receiver's fused decode + MEAN + re-encode with its own residual (the
    reduce-scatter owner's step of a two-phase quantized all-reduce)."""

    def __init__(self, name, scheme, bits, n=1 << 26, M=16, bucket=1024, seed=4):
        super().__init__(name, scheme, bits, n=n, M=M, bucket=bucket, seed=seed)
        words, nb = _words(n, bits), _nb(n, bucket)
        meta = 8 if scheme == 0 else 4
        tag = "u8" if scheme == 0 else ("ternary" if scheme == 2 else f"s{scheme}b{bits}")
        self.dec_name = f"reencode_{tag}_m{M}"
        self.kernels = {self.enc_name: (1, M * (2 * n + 4 * words + meta * nb)),
                        self.dec_name: (1, M * (4 * words + meta * nb) + 8 * n + 4 * words +
                                        meta * nb)}
        self.units = 2 * M * n + n
        self.d2h = 4 * words

    def setup(self, q, torch):
        super().setup(q, torch)
        self.err = torch.zeros(self.n, device="cuda")
        self.codes2, self.scale2, self.offset2 = q.alloc_payload(self.n, self.bits, self.bucket,
                                                                 self.scheme)

    def run(self, q, t, timer):
        mode = q.QC_ROUND_NEAREST if self.scheme == 0 else q.QC_ROUND_STOCHASTIC
        with timer(self.enc_name):
            self.encode_all(q, t)
        with timer(self.dec_name):
            q.qc_reencode(self.codes, self.codes.stride(0), self.scale, self.offset,
                          self.scale.stride(0), self.M, self.n, self.bits, self.bucket,
                          self.scheme, q.QC_OUT_MEAN, self.err, mode, self.seed | (1 << 40), t,
                          self.codes2, self.scale2, self.offset2, None)

    def host_outputs(self):
        return [self.codes2]

    def quality(self, q, torch):
        meta = 8 if self.scheme == 0 else 4
        return {"compression_vs_fp32": round(32 / (self.bits + 8 * meta / self.bucket), 3)}

    def kernel_units(self):
        return {self.enc_name: self.M * self.n, self.dec_name: self.M * self.n}

    def oracle_sample(self, frac):
        import oracle as orc
        n = max(self.bucket, int(self.n * frac) // self.bucket * self.bucket)
        gb = wl.bf16_gradients(n, self.M, self.seed)
        err = np.zeros(n, dtype=np.float32)
        mode = orc.ROUND_NEAREST if self.scheme == 0 else orc.ROUND_STOCHASTIC

        def go(lo, hi):
            cs, ss, os_ = [], [], []
            for w in range(self.M):
                if self.scheme == 0:
                    c, s, o = orc.encode_uniform(gb[w, lo:hi], None, bits=8, bucket=self.bucket,
                                                 index_base=w * self.n + lo)
                    os_.append(o)
                else:
                    c, s = orc.encode_ternary(gb[w, lo:hi], None, bucket=self.bucket,
                                              mode=orc.ROUND_STOCHASTIC, seed=self.seed,
                                              index_base=w * self.n + lo)
                cs.append(c)
                ss.append(s)
            orc.reencode(np.stack(cs), np.stack(ss), np.stack(os_) if os_ else None, M=self.M,
                         n=hi - lo, bits=self.bits, bucket=self.bucket, scheme=self.scheme,
                         flags=orc.OUT_MEAN, err=err[lo:hi], mode=mode)
        return _split(go, n, self.bucket), self.units * n // self.n


class VoteOnly(Component):
    """The majority vote alone over M packed sign vectors of n bits (the vote's
    streaming rate, at a size far above L2).  The sign words are seeded random
    bits drawn on the device: the vote's work does not depend on their values."""

    def __init__(self, name="vote_2p30", n=1 << 30, M=8, seed=3):
        self.name, self.n, self.M, self.seed = name, n, M, seed
        words = _words(n, 1)
        self.kernels = {f"sign_vote_m{M}_{name.split('_')[-1]}": (1, (M + 1) * 4 * words)}
        self.units = M * n

    def setup(self, q, torch, shared=None):
        gen = torch.Generator(device="cuda").manual_seed(self.seed)
        words = _words(self.n, 1)
        self.signs = torch.randint(-2 ** 31, 2 ** 31 - 1, (self.M, words), dtype=torch.int32,
                                   device="cuda", generator=gen)
        self.out = torch.empty(words, dtype=torch.int32, device="cuda")

    def run(self, q, t, timer):
        with timer(next(iter(self.kernels))):
            q.qc_sign_vote(self.signs, self.signs.stride(0), self.M, self.n, self.out)

    def kernel_units(self):
        return {next(iter(self.kernels)): self.M * self.n}


class ReencodeOnly(Component):
    """The fused receiver re-encode alone, on the M payloads another component
    (the 8-bit receiver workload) has just encoded: decode, MEAN, re-encode
    with the receiver's own residual (seed 4 | 1 << 40)."""

    def __init__(self, name="rx_reencode_u8_m16", src=None):
        self.name, self.src = name, src
        n, M, b = src.n, src.M, src.bucket
        words, nb = _words(n, 8), _nb(n, b)
        self.kernels = {"reencode_u8_m16": (1, M * (4 * words + 8 * nb) + 8 * n + 4 * words + 8 * nb)}
        self.units = M * n

    def setup(self, q, torch, shared=None):
        r = self.src
        self.err = torch.zeros(r.n, device="cuda")
        self.codes2, self.scale2, self.offset2 = q.alloc_payload(r.n, 8, r.bucket, 0)

    def run(self, q, t, timer):
        r = self.src
        with timer("reencode_u8_m16"):
            q.qc_reencode(r.codes, r.codes.stride(0), r.scale, r.offset, r.scale.stride(0), r.M,
                          r.n, 8, r.bucket, 0, q.QC_OUT_MEAN, self.err, q.QC_ROUND_NEAREST,
                          r.seed | (1 << 40), t, self.codes2, self.scale2, self.offset2, None)

    def kernel_units(self):
        return {"reencode_u8_m16": self.src.M * self.src.n}


SUPPLEMENT_TEXT = {
    "u8_ef_2p20": "uniform 8-bit EF encode + M=1 decode, 2^20 fp32 (outlier recipe), B=2048, RN "
                  "(13.6 MB: L2-resident; per-launch times from events and from a CUDA graph)",
    "vote_2p30": "majority vote of 8 packed sign vectors of 2^30 bits",
    "qsgd4_ef": "QSGD 4-bit SR + EF encode, M=1 decode, 250M fp32 (per-bucket sigma), B=512",
    "log4_ef": "logarithmic levels 4-bit SR + EF encode, M=1 decode, 250M fp32, B=512",
    "clip8_ef_2p28": "percentile-clipped 8-bit RN + EF encode, M=1 decode, 2^28 fp32 (outliers), "
                     "B=2048",
    "topk_ef": "top-k (10 of every 1024) 8-bit + EF encode x8 workers of 25.6M, scatter decode "
               "MEAN M=8",
    "rx_reencode_u8_m16": "fused decode MEAN + 8-bit re-encode with EF of 16 bf16-encoded payloads "
                          "of 2^26",
}


def _kernel_stats(comp, timer, peak):
    out = {}
    per = timer.per_kernel_ms()
    units = comp.kernel_units()
    for name, (cnt, b) in comp.kernels.items():
        ts = per.get(name, [])
        if not ts:
            continue
        avg = sum(ts) / len(ts)
        e = {"launches": len(ts), "avg_us": round(avg * 1e3, 2), "bytes_per_launch": b,
             "gbs": round(b / (avg * 1e-3) / 1e9, 1), "frac_of_peak": round(b / (avg * 1e-3) / 1e9 / peak, 4)}
        if units.get(name):
            e["units_per_launch"] = units[name]
            e["elements_per_s"] = float(f"{units[name] / (avg * 1e-3):.4g}")
            e["fp32_equiv_gbs"] = round(4 * units[name] / (avg * 1e-3) / 1e9, 1)
            # DRAM bytes per launch from the kernel's committed ncu capture (None
            # when there is none or its sources changed since)
            e["traffic"] = ncu_traffic(name, units[name])
        out[name] = e
    return out


def _graph_us_per_launch(q, torch, comp, which, reps=64):
    """Per-launch device time of one kernel of `comp` replayed back to back from
    a CUDA graph (no host launch overhead between launches)."""
    timer = KernelTimer(torch, enabled=False)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        comp.run(q, 1, timer)                  # warm-up outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        for r in range(reps):
            which(r)
    graph.replay()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(5):
        graph.replay()
    b.record()
    torch.cuda.synchronize()
    return round(a.elapsed_time(b) * 1e3 / (5 * reps), 2)


def run_supplements(q, torch, suite, peak, reps=10):
    """The workloads outside the headline suite, each timed on its own after the
    suite (CUDA events around every launch on the launching stream, 2 untimed
    launches first): the 2^20 8-bit EF workload, the vote at 2^30, QSGD,
    logarithmic levels, percentile clipping, top-k and the fused re-encode.
    They reuse the suite's device data where the recipe is the same."""
    by_name = {c.name: c for c in suite}
    comps = [UniformEF("u8_ef_2p20", 1 << 20, 8, 2048, False, 0, "outlier"), VoteOnly()]
    shared = {}
    if "sr4_ef" in by_name:
        comps += [UniformEF("qsgd4_ef", 250_000_000, 4, 512, True, 2, "bucket", scheme=3),
                  UniformEF("log4_ef", 250_000_000, 4, 512, True, 2, "bucket", scheme=5)]
        shared["qsgd4_ef"] = shared["log4_ef"] = by_name["sr4_ef"]
    comps.append(UniformEF("clip8_ef_2p28", 1 << 28, 8, 2048, False, 0, "outlier", scheme=4))
    if "sign_ef_vote" in by_name:
        comps.append(TopkEF())
        shared["topk_ef"] = by_name["sign_ef_vote"]
    if "rx_u8" in by_name:
        comps.append(ReencodeOnly(src=by_name["rx_u8"]))
    out = {}
    for c in comps:
        c.setup(q, torch, shared=shared.get(c.name))
        warm = KernelTimer(torch, enabled=False)
        for t in range(2):
            c.run(q, t, warm)
        torch.cuda.synchronize()
        timer = KernelTimer(torch, enabled=True)
        for t in range(2, 2 + reps):
            c.run(q, t, timer)
        torch.cuda.synchronize()
        entry = {"workload": SUPPLEMENT_TEXT.get(c.name, c.name), "kernels": _kernel_stats(c, timer, peak)}
        if c.name == "u8_ef_2p20":
            mode = q.QC_ROUND_NEAREST
            enc = lambda r: q.qc_encode_ef(c.g, c.err, c.n, 8, c.bucket, 0, mode, 0, r, c.codes,
                                           c.scale, c.offset)
            dec = lambda r: q.qc_decode_accumulate(c.codes, 0, c.scale, c.offset, 0, 1, c.n, 8,
                                                   c.bucket, 0, c.out, 0)
            entry["graph_us_per_launch"] = {c.enc_name: _graph_us_per_launch(q, torch, c, enc),
                                            c.dec_name: _graph_us_per_launch(q, torch, c, dec)}
        out[c.name] = entry
        for attr in list(vars(c)):
            if attr not in ("src",) and hasattr(getattr(c, attr), "is_cuda"):
                setattr(c, attr, None)
        c.gs = None
        torch.cuda.empty_cache()
    return out


def _split(fn, n, align):
    """A closure running fn over n elements in bucket-aligned parts on every core."""
    cores = _cores()
    per = max(align, -(-(-(-n // cores)) // align) * align)
    parts = [(lo, min(n, lo + per)) for lo in range(0, n, per)]

    def run():
        with ThreadPoolExecutor(len(parts)) as ex:
            list(ex.map(lambda p: fn(*p), parts))
    run.threads = len(parts)
    return run


def _cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def make_workload(name):
    if name == "suite":
        rx = Receiver("rx_u8", 0, 8)
        return [Fp8Rowwise(), UniformEF("sr4_ef", 250_000_000, 4, 512, True, 2, "bucket"),
                SignVote(), rx, Receiver("rx_ternary", 2, 2, shared=rx)]
    table = {
        "fp8_rowwise": lambda: [Fp8Rowwise()],
        "sr4_ef": lambda: [UniformEF("sr4_ef", 250_000_000, 4, 512, True, 2, "bucket")],
        "sign_ef_vote": lambda: [SignVote()],
        "rx_u8": lambda: [Receiver("rx_u8", 0, 8)],
        "rx_ternary": lambda: [Receiver("rx_ternary", 2, 2)],
        "qsgd4_ef": lambda: [UniformEF("qsgd4_ef", 250_000_000, 4, 512, True, 2, "bucket",
                                       scheme=3)],
        "log4_ef": lambda: [UniformEF("log4_ef", 250_000_000, 4, 512, True, 2, "bucket",
                                      scheme=5)],
        "rx_reencode_u8": lambda: [Reencode("rx_reencode_u8", 0, 8)],
        "rx_reencode_ternary": lambda: [Reencode("rx_reencode_ternary", 2, 2)],
        "topk_ef": lambda: [TopkEF()],
        "probe_topk_ef": lambda: [TopkEF(n=1 << 24, M=2)],
        "u8_ef_small": lambda: [UniformEF("u8_ef_small", 1 << 20, 8, 2048, False, 0, "outlier")],
        "clip8_ef_small": lambda: [UniformEF("clip8_ef_small", 1 << 20, 8, 2048, False, 0,
                                             "outlier", scheme=4)],
        "clip8_ef_large": lambda: [UniformEF("clip8_ef_large", 1 << 28, 8, 2048, False, 0,
                                             "outlier", scheme=4)],
        "u8_ef_large": lambda: [UniformEF("u8_ef_large", 1 << 28, 8, 2048, False, 0, "outlier")],
        # smaller single-kernel cases (inputs still larger than L2) for profiler captures
        "probe_sr4_ef": lambda: [UniformEF("sr4_ef", 1 << 26, 4, 512, True, 2, "bucket")],
        "probe_qsgd4_ef": lambda: [UniformEF("qsgd4_ef", 1 << 26, 4, 512, True, 2, "bucket",
                                             scheme=3)],
        "probe_log4_ef": lambda: [UniformEF("log4_ef", 1 << 26, 4, 512, True, 2, "bucket",
                                            scheme=5)],
        "probe_clip8_ef": lambda: [UniformEF("clip8_ef", 1 << 26, 8, 2048, False, 0, "outlier",
                                             scheme=4)],
        "probe_sign": lambda: [SignVote(n=1 << 24, M=2)],
        "probe_u8_bf16": lambda: [Receiver("rx_u8", 0, 8, n=1 << 27, M=1)],
        "probe_ternary_bf16": lambda: [Receiver("rx_ternary", 2, 2, n=1 << 27, M=1)],
        "probe_decode_u8_m16": lambda: [Receiver("rx_u8", 0, 8, n=1 << 24, M=16)],
        "probe_decode_ternary_m16": lambda: [Receiver("rx_ternary", 2, 2, n=1 << 24, M=16)],
        "probe_decode_u8_m16_full": lambda: [Receiver("rx_u8", 0, 8, n=1 << 26, M=16)],
        "probe_decode_ternary_m16_full": lambda: [Receiver("rx_ternary", 2, 2, n=1 << 26, M=16)],
        "probe_vote": lambda: [VoteOnly("vote_2p28", n=1 << 28, M=8)],
        "vote_2p30": lambda: [VoteOnly()],
        "probe_reencode_u8_m16": lambda: [Reencode("rx_reencode_u8", 0, 8, n=1 << 24, M=16)],
        "probe_fp8": lambda: [Fp8Rowwise(rows=1 << 19)],
    }
    return table[name]()


WORKLOAD_TEXT = {
    "suite": "codec suite: fp8_rowwise 1,000,000x128 + sr4_ef 250M (B=512, 1 step) + "
             "sign_ef_vote 8x25.6M (B=4096) + rx_u8 and rx_ternary 16x2^26 bf16 (B=1024, MEAN)",
}


# ------------------------------------------------------------- timing helpers

class KernelTimer:
    """CUDA events around each launch on the launching (current) stream."""

    def __init__(self, torch, enabled=True):
        self.torch, self.enabled = torch, enabled
        self.events = []   # (name, start, end)
        self.launches = 0

    def __call__(self, name):
        timer = self

        class _Ctx:
            def __enter__(self):
                timer.launches += 1
                if timer.enabled:
                    self.s = timer.torch.cuda.Event(enable_timing=True)
                    self.e = timer.torch.cuda.Event(enable_timing=True)
                    self.s.record()

            def __exit__(self, *a):
                if timer.enabled:
                    self.e.record()
                    timer.events.append((name, self.s, self.e))
        return _Ctx()

    def per_kernel_ms(self):
        out = {}
        for name, s, e in self.events:
            out.setdefault(name, []).append(s.elapsed_time(e))
        return out


class ClockSampler:
    """nvidia-smi clock/throttle samples every 200 ms while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu, self.proc, self.path = gpu_index, None, None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.fh,
                stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[0]) for r in rows if num(r[0]) is not None]
        mx = [num(r[1]) for r in rows if num(r[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[4 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return PEAK_FALLBACK_GBS, "fallback"


def source_digest(files):
    """Short hash over the named kernel source files (in csrc/)."""
    h = hashlib.sha256()
    for name in files:
        with open(os.path.join(ROOT, "embedding_communication_codecs_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel, units_per_launch):
    """DRAM bytes per launch of `kernel` from the committed ncu summary, scaled
    from the captured launch to this launch by the units processed; None if
    the summary is missing or was taken on different kernel sources."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            ent = json.load(f).get(kernel)
        if not ent or source_digest(ent["sources"]) != ent["digest"]:
            return None
    except (OSError, ValueError, KeyError):
        return None
    return int(round(ent["dram_bytes"] * units_per_launch / ent["units"]))


# ------------------------------------------------------------- distributed

def dist_setup(backend=None):
    """Rank, world size and local rank from the launcher's environment; with
    more than one rank, a process group (NCCL on GPUs unless told otherwise)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        if backend is None:
            backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def max_over_ranks(x, world):
    """Maximum of a float over all ranks (a host-side reduction of timings)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ arms

def run_ours(args, world, rank, local):
    import torch
    import embedding_communication_codecs_gb300 as q

    torch.cuda.set_device(local)
    comps = make_workload(args.workload)
    for c in comps:
        c.setup(q, torch)
    torch.cuda.synchronize()

    def step(t, timer):
        for c in comps:
            c.run(q, t, timer)

    # warm-up (untimed)
    warm = KernelTimer(torch, enabled=False)
    for t in range(args.warmup):
        step(t, warm)
    torch.cuda.synchronize()

    sampler = ClockSampler(local)
    timer = KernelTimer(torch, enabled=True)
    barrier(world)
    torch.cuda.synchronize()
    sampler.start()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    for t in range(args.warmup, args.warmup + args.steps):
        step(t, timer)
    t1.record()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    barrier(world)
    elapsed_ms = max_over_ranks(t0.elapsed_time(t1), world)

    units = sum(c.units for c in comps)
    ms_per_step = elapsed_ms / args.steps
    value = world * units * 4 * args.steps / (elapsed_ms * 1e-3) / 1e9
    alg_bytes = sum(cnt * b for c in comps for cnt, b in c.kernels.values())
    per_kernel = timer.per_kernel_ms()
    kinfo = {}
    for c in comps:
        for name, (cnt, b) in c.kernels.items():
            ts = per_kernel.get(name, [])
            if not ts:
                continue
            avg = sum(ts) / len(ts)
            kinfo[name] = {"launches": len(ts), "avg_us": round(avg * 1e3, 2),
                           "total_ms": round(sum(ts), 3), "bytes_per_launch": b,
                           "gbs": round(b / (avg * 1e-3) / 1e9, 1)}
    peak, peak_src = measured_peak()
    dom = max(kinfo, key=lambda k: kinfo[k]["total_ms"])
    achieved = kinfo[dom]["gbs"]
    units_per_launch = {k: u for c in comps for k, u in c.kernel_units().items()}
    roofline = {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peak,
                "peak_source": peak_src, "unit": "GB/s", "frac": round(achieved / peak, 4),
                "traffic": ncu_traffic(dom, units_per_launch.get(dom, 0)),
                "bytes_per_launch": kinfo[dom]["bytes_per_launch"]}
    for k in kinfo:
        kinfo[k]["frac_of_peak"] = round(kinfo[k]["gbs"] / peak, 4)
        u = units_per_launch.get(k)
        if u:
            kinfo[k]["units_per_launch"] = u
            kinfo[k]["elements_per_s"] = float(f"{u / (kinfo[k]['avg_us'] * 1e-6):.4g}")
            # DRAM bytes per launch from the kernel's committed ncu capture (None
            # when there is none or its sources changed since)
            kinfo[k]["traffic"] = ncu_traffic(k, u)

    quality = {}
    for c in comps:
        qc = c.quality(q, torch)
        if qc is not None:
            quality[c.name] = {k: (round(v, 6) if isinstance(v, float) else v) for k, v in qc.items()}
    torch.cuda.synchronize()

    e2e = run_e2e(args, comps, q, torch, world, units)
    supplements = None
    if not args.no_supplements and args.workload == "suite":
        supplements = run_supplements(q, torch, comps, peak)

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded numpy PCG64 draws shaped like the pages' workloads)",
        "config": {"workload": WORKLOAD_TEXT.get(args.workload, args.workload),
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "inputs larger than L2 (the step streams ~15 GB; every kernel but the "
                         "vote reads > 129 MB)",
                   "fp32_equiv_elements_per_step": units},
        "hbm": {"algorithmic_bytes_per_step": alg_bytes,
                "gbs": round(alg_bytes / (ms_per_step * 1e-3) / 1e9, 1),
                "frac": round(alg_bytes / (ms_per_step * 1e-3) / 1e9 / peak, 4)},
        "roofline": roofline,
        "kernels": kinfo,
        "e2e": e2e,
        "gpu_launches": timer.launches,
        "clocks": clocks,
        "quality": quality,
    }
    if supplements is not None:
        line["supplements"] = supplements
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(comps, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_e2e(args, comps, q, torch, world, units, results=None):
    """The same steps through the public API with host buffers: each step copies
    its inputs in from pinned host memory and reads its results back.  As a user
    of the stream-ordered API would, the run keeps three streams busy at once:
    component k's inputs go in on the copy-in stream while earlier components
    run on the compute stream and their results come back on the copy-out
    stream.  Events keep every buffer safe: an input is refilled only after the
    previous step's last reader of it has run, and a component writes its
    outputs only after the previous step's copy of them has left.  `results`, if
    given, receives the pinned host copies of the last step's outputs."""
    ins = [[(d, torch.empty(d.shape, dtype=d.dtype, pin_memory=True).copy_(d))
            for d in c.host_inputs()] for c in comps]
    outs = [[(d, torch.empty(d.shape, dtype=d.dtype, pin_memory=True)) for d in c.host_outputs()]
            for c in comps]
    bi = sum(h.numel() * h.element_size() for pairs in ins for _, h in pairs)
    bo = sum(h.numel() * h.element_size() for pairs in outs for _, h in pairs)
    # the last component of the step that reads each component's inputs
    last_reader = []
    for k, c in enumerate(comps):
        ptrs = {d.data_ptr() for d in c.host_inputs()}
        last_reader.append(max([j for j, o in enumerate(comps)
                                if ptrs & {d.data_ptr() for d in o.reads()}], default=k))
    steps = max(1, min(args.steps, args.e2e_steps))
    timer = KernelTimer(torch, enabled=False)
    for c in comps:   # each step's gradient comes in from the host into the one buffer
        if hasattr(c, "fixed_input"):
            c.fixed_input = True
    s_in, s_cmp, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    cur = torch.cuda.current_stream()
    torch.cuda.synchronize()
    barrier(world)
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    s.record(cur)
    for st in (s_in, s_cmp, s_out):
        st.wait_event(s)
    prev_c, prev_o = None, None
    for t in range(steps):
        done_c, done_o = [], []
        for k, c in enumerate(comps):
            with torch.cuda.stream(s_in):
                if prev_c is not None:
                    s_in.wait_event(prev_c[last_reader[k]])
                for d, h in ins[k]:
                    d.copy_(h, non_blocking=True)
                ev_in = torch.cuda.Event()
                ev_in.record(s_in)
            s_cmp.wait_event(ev_in)
            if prev_o is not None:
                s_cmp.wait_event(prev_o[k])
            with torch.cuda.stream(s_cmp):
                c.run(q, 1000 + t, timer)
                ev_c = torch.cuda.Event()
                ev_c.record(s_cmp)
            done_c.append(ev_c)
            s_out.wait_event(ev_c)
            with torch.cuda.stream(s_out):
                for d, h in outs[k]:
                    h.copy_(d, non_blocking=True)
                ev_o = torch.cuda.Event()
                ev_o.record(s_out)
            done_o.append(ev_o)
        prev_c, prev_o = done_c, done_o
    for st in (s_in, s_cmp, s_out):
        cur.wait_stream(st)
    e.record(cur)
    torch.cuda.synchronize()
    for c in comps:
        if hasattr(c, "fixed_input"):
            c.fixed_input = False
    if results is not None:
        results.extend(h for pairs in outs for _, h in pairs)
    ms = max_over_ranks(s.elapsed_time(e), world)
    value = world * units * 4 * steps / (ms * 1e-3) / 1e9
    return {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": bi,
            "d2h_bytes_per_step": bo, "steps": steps, "streams": 3}


def oracle_rate(comps, budget_s):
    """Time the oracle (as it stands) on a bounded sample of every component,
    threads over all host cores; returns (GB/s fp32-equivalent, cores, sample text)."""
    import oracle
    oracle.build()

    def measure(frac, samples=None):
        """Runs each component's sample once (built here unless given; inputs are
        generated outside the timed calls)."""
        tt, uu, thr, parts = 0.0, 0, 1, []
        built = samples if samples is not None else [c.oracle_sample(frac) for c in comps]
        for c, (fn, u) in zip(comps, built):
            a = time.perf_counter()
            fn()
            dt = time.perf_counter() - a
            tt += dt
            uu += u
            thr = max(thr, fn.threads)
            parts.append(f"{c.name} {u:,} elements {dt:.2f}s")
        measure.last = built
        return tt, uu, thr, parts

    # calibrate on a small sample, size the sample to the budget (at most a
    # quarter of each component, which bounds the host memory of the inputs),
    # then repeat it until the budget of CPU time is spent
    frac = 1e-3
    total_t, total_u, threads, parts = measure(frac)
    for _ in range(3):
        if total_t >= budget_s / 3 or frac >= 0.25:
            break
        frac = min(0.25, frac * budget_s / max(total_t, 1e-3))
        total_t, total_u, threads, parts = measure(frac)
    reps, t_all, u_all, samples = 1, total_t, total_u, measure.last
    while t_all < budget_s and reps < 64:
        t, u, _, _ = measure(frac, samples)
        t_all, u_all, reps = t_all + t, u_all + u, reps + 1
    rate = u_all * 4 / t_all / 1e9
    return rate, threads, (f"{frac:.4%} of each component's full workload, {reps} passes, "
                           f"{t_all:.1f} s of oracle time; last pass: " + "; ".join(parts))


def cpu_baseline(comps, budget_s):
    rate, cores, sample = oracle_rate(comps, budget_s)
    return {"value": round(rate, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": sample}


def run_reference(args, world, rank):
    """The oracle arm: the CPU oracle timed on the host cores, on bounded samples
    of the same workload, rank 0 only."""
    if rank != 0:
        return
    comps = make_workload(args.workload)
    per_step = max(0.5, 150.0 / (args.steps + args.warmup))
    times, units = [], 0
    fns = []
    probe_rate, cores, _ = oracle_rate(comps, min(2.0, per_step))
    for c in comps:
        full = c.units * 4 / 1e9 / probe_rate        # seconds for the full component
        frac = min(1.0, per_step / max(full * len(comps), 1e-9))
        fn, u = c.oracle_sample(frac)
        fns.append(fn)
        units += u
    for i in range(args.warmup + args.steps):
        a = time.perf_counter()
        for fn in fns:
            fn()
        dt = time.perf_counter() - a
        if i >= args.warmup:
            times.append(dt)
    total = sum(times)
    value = units * 4 * len(times) / total / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total / len(times) * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded numpy PCG64 draws shaped like the pages' workloads)",
        "config": {"workload": WORKLOAD_TEXT.get(args.workload, args.workload),
                   "sample_fp32_equiv_elements_per_step": units},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": cores,
                         "kind": "oracle",
                         "sample": f"{units:,} fp32-equivalent elements per step across all "
                                   f"components (bucket-aligned slices of each workload)"},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="suite")
    ap.add_argument("--e2e-steps", type=int, default=5)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-supplements", action="store_true",
                    help="skip the workloads timed outside the headline suite")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

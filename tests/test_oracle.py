"""Pins of the CPU oracle against what the pages and the mathematics fix.

No GPU.  Every check here is independent of the oracle's own code: published
known-answer vectors, the pages' byte counts and ratios, closed forms on hand-built
buckets, exact rational arithmetic, brute force on tiny inputs, invariants and
statistical tests of unbiasedness.
"""
from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle as orc
import workloads as wl
from tests._exact import dist_to_half_integer, frac, round_half_even, to_f32, ulp32
from tests._norm_cases import exact_norm_f32, midpoint_bucket

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _read_golden(golden_dir, name):
    rows = []
    with open(os.path.join(golden_dir, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def _unpack(words, n, bits):
    per = 32 // bits
    out = []
    for i in range(n):
        out.append((int(words[i // per]) >> ((i % per) * bits)) & ((1 << bits) - 1))
    return out


def _pack(codes, bits):
    per = 32 // bits
    words = [0] * ((len(codes) * bits + 31) // 32)
    for i, c in enumerate(codes):
        words[i // per] |= int(c) << ((i % per) * bits)
    return np.array(words, dtype=np.uint32)


# --------------------------------------------------------------------------- Philox

def test_philox_known_answers(golden_dir):
    rows = _read_golden(golden_dir, "philox4x32_10_kat.txt")
    assert len(rows) == 3
    for r in rows:
        v = [int(x, 16) for x in r]
        got = orc.philox4x32_10(v[0:4], v[4:6])
        assert [int(x) for x in got] == v[6:10]


def test_uniform_draw_layout():
    # The reading: key = seed words, counter = (i/4 low, i/4 high, step, 0),
    # element i takes output word i mod 4, u = (word >> 8) * 2^-24.
    for seed, step, idx in [(0, 0, 0), (0, 0, 3), (7, 2, 5), (2 | (5 << 32), 9, (1 << 33) + 6)]:
        blk = idx >> 2
        r = orc.philox4x32_10([blk & 0xFFFFFFFF, blk >> 32, step, 0],
                              [seed & 0xFFFFFFFF, seed >> 32])
        want = float(int(r[idx & 3]) >> 8) * 2.0 ** -24
        assert orc.uniform(seed, step, idx) == want


def test_uniform_draw_statistics():
    n = 1 << 16
    u = np.array([orc.uniform(11, 3, i) for i in range(n)])
    assert u.min() >= 0.0 and u.max() < 1.0
    counts, _ = np.histogram(u, bins=64, range=(0.0, 1.0))
    expected = n / 64
    chi2 = float(((counts - expected) ** 2 / expected).sum())
    # 63 degrees of freedom: mean 63, sd ~11.2; 130 is beyond 6 sd.
    assert chi2 < 130.0
    # neighbouring draws are uncorrelated
    c = np.corrcoef(u[:-1], u[1:])[0, 1]
    assert abs(c) < 5.0 / math.sqrt(n)


# --------------------------------------------------------------- sizes and ratios

def test_compression_ratios_pages(golden_dir):
    rows = _read_golden(golden_dir, "compression_ratios.txt")
    ratios = {int(r[0]): int(r[1]) for r in rows if r[0].isdigit()}
    n = 1 << 16
    for bits, ratio in ratios.items():
        words = orc.code_words(n, bits)
        assert (n * 4) / (words * 4) == ratio
    per_word = [r for r in rows if r[0] == "codes_per_word_4bit"][0]
    assert 32 // 4 == int(per_word[1])
    # with one fp32 scale + one fp32 offset per bucket the ratio is slightly lower
    for bits, ratio in ratios.items():
        for bucket in (512, 1024, 2048):
            eff = 32.0 * bucket / (bits * bucket + 64)
            assert ratio * 0.85 < eff < ratio


def test_code_words_and_buckets():
    assert orc.code_words(0, 8) == 0
    assert orc.code_words(1, 1) == 1
    assert orc.code_words(33, 1) == 2
    assert orc.code_words(250_000_000, 4) == 125_000_000 // 4
    assert orc.num_buckets(250_000_000, 512) == 488_282
    assert orc.num_buckets(1 << 20, 2048) == 512


# ------------------------------------------------------------ uniform, nearest

@pytest.mark.parametrize("bits", [1, 2, 4, 8])
def test_uniform_ramp_closed_form(bits):
    L = (1 << bits) - 1
    bucket = max(32, L + 1)
    c = 2.0 ** -10
    base = -3.0
    levels = [j % (L + 1) for j in range(bucket)]
    g = np.array([base + lv * c for lv in levels], dtype=np.float32)
    err = np.zeros_like(g)
    codes, scale, offset = orc.encode_uniform(g, err, bits=bits, bucket=bucket)
    assert scale[0] == np.float32(c)
    assert offset[0] == np.float32(base)
    assert _unpack(codes, bucket, bits) == levels
    assert np.array_equal(codes, _pack(levels, bits))
    assert np.all(err == 0.0)


def test_uniform_ties_to_even():
    bucket = 32
    vals = [0.0, 255.0, 2.5, 3.5, 100.5, 101.5, 0.5, 254.5] + [7.0] * 24
    g = np.array(vals, dtype=np.float32)
    codes, scale, offset = orc.encode_uniform(g, None, bits=8, bucket=bucket)
    assert scale[0] == 1.0 and offset[0] == 0.0
    q = _unpack(codes, bucket, 8)
    assert q[:8] == [0, 255, 2, 4, 100, 102, 0, 254]


def test_uniform_constant_bucket():
    g = np.full(96, np.float32(0.125), dtype=np.float32)
    g[64:] = np.float32(-2.0)
    err = np.zeros_like(g)
    codes, scale, offset = orc.encode_uniform(g, err, bits=4, bucket=64)
    assert scale[0] == 0.0 and offset[0] == np.float32(0.125)
    assert scale[1] == 0.0 and offset[1] == np.float32(-2.0)
    assert not codes.any()
    assert np.all(err == 0.0)


def _tiny_buckets(seed, n, scale=1e-3):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal(n) * scale).astype(np.float32)


@pytest.mark.parametrize("bits", [1, 2, 4, 8])
def test_uniform_nearest_level_exact(bits):
    """Each code is the level nearest to the exact (p - min)/scale."""
    L = (1 << bits) - 1
    bucket = 64
    g = _tiny_buckets(bits, 4 * bucket + 40)   # ragged last bucket
    n = g.size
    codes, scale, offset = orc.encode_uniform(g, None, bits=bits, bucket=bucket)
    q = _unpack(codes, n, bits)
    for k in range(orc.num_buckets(n, bucket)):
        seg = g[k * bucket:(k + 1) * bucket]
        mn, mx = seg.min(), seg.max()
        assert offset[k] == mn
        # scale is the binary32 rounding of the binary32 range over L
        rng32 = to_f32(frac(mx) - frac(mn))
        assert scale[k] == to_f32(frac(rng32) / L)
        for j, p in enumerate(seg):
            t = (frac(p) - frac(mn)) / frac(scale[k])
            want = min(round_half_even(t), L)
            got = q[k * bucket + j]
            if got != want:
                # only allowed within two roundings of a half-integer
                assert dist_to_half_integer(t) <= t * Fraction(1, 1 << 22)
                assert abs(got - want) == 1


def test_uniform_invariants_outlier_workload():
    n, bucket, bits = 1 << 14, 2048, 8
    g = wl.outlier_gradient(n, seed=0)
    e0 = np.zeros(n, dtype=np.float32)
    err = e0.copy()
    codes, scale, offset = orc.encode_uniform(g, err, bits=bits, bucket=bucket)
    q = np.array(_unpack(codes, n, bits))
    for k in range(n // bucket):
        s = slice(k * bucket, (k + 1) * bucket)
        seg = g[s]
        assert q[s][np.argmin(seg)] == 0
        assert q[s][np.argmax(seg)] == 255
        deq = np.float32(offset[k]) + q[s].astype(np.float64) * np.float64(scale[k])
        # |p - deq| <= scale/2 up to rounding
        bound = 0.5 * float(scale[k]) * (1 + 2.0 ** -20) + 2 * ulp32(np.abs(seg).max())
        assert np.all(np.abs(seg.astype(np.float64) - deq) <= bound)
        # error feedback keeps exactly what was dropped (up to one rounding)
        assert np.all(np.abs(err[s].astype(np.float64) - (seg - deq)) <= bound)


def test_uniform_ef_identity_and_monotone():
    n, bucket = 3000, 512
    g = _tiny_buckets(5, n)
    e_old = _tiny_buckets(6, n, scale=1e-4)
    err = e_old.copy()
    codes, scale, offset = orc.encode_uniform(g, err, bits=4, bucket=bucket)
    q = np.array(_unpack(codes, n, 4))
    p = (e_old + g).astype(np.float32)         # one binary32 rounding of e + g
    for k in range(orc.num_buckets(n, bucket)):
        s = slice(k * bucket, min(n, (k + 1) * bucket))
        deq = np.array([float(np.float32(frac(qq) * frac(scale[k]) + frac(offset[k])))
                        for qq in q[s]])
        lhs = err[s].astype(np.float64) + deq
        tol = np.array([ulp32(max(abs(a), abs(b))) for a, b in zip(p[s], deq)])
        assert np.all(np.abs(lhs - p[s].astype(np.float64)) <= tol)
        order = np.argsort(p[s], kind="stable")
        assert np.all(np.diff(q[s][order]) >= 0)


# ------------------------------------------------------------- uniform, stochastic

def test_stochastic_floor_or_ceil_and_unbiased():
    bits, bucket = 4, 32
    L = 15
    fracs = [0.0, 0.1, 0.25, 0.5, 0.7, 0.9, 0.99]
    vals = [0.0, 15.0] + [3 + f for f in fracs] + [8 + f for f in fracs]
    vals += [1.0] * (bucket - len(vals))
    g = np.array(vals, dtype=np.float32) * np.float32(2.0 ** -7)
    K = 6000
    acc = np.zeros(bucket)
    ceil_count = np.zeros(bucket)
    t_exact = [(frac(v) - frac(g.min())) / frac(np.float32(2.0 ** -7)) for v in g]
    for step in range(K):
        codes, scale, offset = orc.encode_uniform(g, None, bits=bits, bucket=bucket,
                                                  mode=orc.ROUND_STOCHASTIC, seed=17,
                                                  step=step)
        assert scale[0] == np.float32(2.0 ** -7)
        q = np.array(_unpack(codes, bucket, bits))
        fl = np.array([math.floor(t) for t in t_exact])
        assert np.all((q == fl) | (q == np.minimum(fl + 1, L)))
        ceil_count += (q > fl)
        acc += offset[0] + q * float(scale[0])
    mean = acc / K
    for j in range(bucket):
        fr = float(t_exact[j] - math.floor(t_exact[j]))
        sd = math.sqrt(max(fr * (1 - fr), 1e-12) / K)
        assert abs(ceil_count[j] / K - fr) <= 5 * sd + 1e-12
        assert abs(mean[j] - float(g[j])) <= 5 * float(scale[0]) * sd + 1e-12


def test_stochastic_deterministic_and_global_index():
    n, bucket = 4096 + 96, 512
    g = _tiny_buckets(9, n)
    a = orc.encode_uniform(g, None, bits=2, bucket=bucket, mode=orc.ROUND_STOCHASTIC,
                           seed=5, step=4)
    b = orc.encode_uniform(g, None, bits=2, bucket=bucket, mode=orc.ROUND_STOCHASTIC,
                           seed=5, step=4)
    c = orc.encode_uniform(g, None, bits=2, bucket=bucket, mode=orc.ROUND_STOCHASTIC,
                           seed=5, step=5)
    assert all(np.array_equal(x, y) for x, y in zip(a, b))
    assert not np.array_equal(a[0], c[0])
    # a slice starting on a bucket boundary reproduces its part of the whole
    lo = 2 * bucket
    part = orc.encode_uniform(g[lo:], None, bits=2, bucket=bucket,
                              mode=orc.ROUND_STOCHASTIC, seed=5, step=4, index_base=lo)
    assert np.array_equal(part[0], a[0][lo * 2 // 32:])
    assert np.array_equal(part[1], a[1][2:])


def test_ef_chain_delays_not_loses():
    """Sum of transmitted values + final residual = sum of gradients (p4: the
    dropped signal is only delayed)."""
    n, bucket, steps = 2048 + 128, 512, 10
    sig = wl.bucket_sigmas(n, bucket, seed=2)
    err = np.zeros(n, dtype=np.float32)
    sent = np.zeros(n)
    gsum = np.zeros(n)
    bound = np.zeros(n)
    for t in range(steps):
        g = wl.bucket_sigma_gradient(n, bucket, t, seed=2, sigmas=sig)
        codes, scale, offset = orc.encode_uniform(g, err, bits=4, bucket=bucket,
                                                  mode=orc.ROUND_STOCHASTIC, seed=2, step=t)
        out = orc.decode_accumulate(codes, scale, offset, M=1, n=n, bits=4, bucket=bucket,
                                    scheme=orc.SCHEME_UNIFORM)
        sent += out
        gsum += g
        bound += 4 * np.spacing(np.abs(out).astype(np.float32) + np.abs(g) + 1e-30)
    assert np.all(np.abs(sent + err - gsum) <= bound)


# -------------------------------------------------------------------------- sign

def test_sign_bits_scale_and_partial_bucket():
    n, bucket = 64 * 3 + 16, 64
    g = _tiny_buckets(21, n)
    g[3] = np.float32(0.0)
    g[4] = np.float32(-0.0)
    g[-16:] = np.float32(1.0)                 # partial last bucket: mean over 16
    e_old = np.zeros(n, dtype=np.float32)
    err = e_old.copy()
    codes, scale = orc.encode_sign(g, err, bucket=bucket)
    bits = _unpack(codes, n, 1)
    assert bits == [1 if v >= 0 else 0 for v in g]   # sign(+-0) = +1
    assert scale[-1] == 1.0
    for k in range(orc.num_buckets(n, bucket)):
        seg = g[k * bucket:(k + 1) * bucket]
        exact = sum(abs(frac(v)) for v in seg) / len(seg)
        assert abs(frac(scale[k]) - exact) <= Fraction(ulp32(scale[k]))
        deq = np.where(np.array(bits[k * bucket:k * bucket + len(seg)]) == 1,
                       scale[k], -scale[k]).astype(np.float32)
        assert np.all(err[k * bucket:k * bucket + len(seg)] == (seg - deq))
        assert math.isclose(float(np.abs(deq.astype(np.float64)).sum()),
                            len(seg) * float(scale[k]), rel_tol=1e-12)


def test_sign_with_residual():
    n, bucket = 4096 * 2, 4096
    g = wl.shared_mean_gradients(n, 1, seed=3)[0]
    e_old = _tiny_buckets(4, n, scale=5e-4)
    err = e_old.copy()
    codes, scale = orc.encode_sign(g, err, bucket=bucket)
    p = (e_old + g).astype(np.float32)
    assert _unpack(codes, n, 1) == [int(v >= 0) for v in p]
    deq = np.where(p >= 0, np.repeat(scale, bucket), -np.repeat(scale, bucket))
    lhs = err.astype(np.float64) + deq
    assert np.all(np.abs(lhs - p) <= np.spacing(np.abs(p) + np.abs(deq).astype(np.float32)))


# ----------------------------------------------------------------------- ternary

def test_ternary_levels_and_nearest_rule():
    n, bucket = 256 + 32, 128
    g = _tiny_buckets(31, n)
    g[200:232] = 0.0                          # part of a bucket at zero
    codes, scale = orc.encode_ternary(g, None, bucket=bucket, mode=orc.ROUND_NEAREST)
    c = np.array(_unpack(codes, n, 2))
    assert set(np.unique(c)) <= {0, 1, 2}
    for k in range(orc.num_buckets(n, bucket)):
        seg = g[k * bucket:(k + 1) * bucket]
        cs = c[k * bucket:k * bucket + len(seg)]
        s = np.abs(seg).max()
        assert scale[k] == s
        am = np.argmax(np.abs(seg))
        assert cs[am] == (2 if seg[am] > 0 else 0)
        for v, code in zip(seg, cs):
            r = abs(frac(v)) / frac(s)
            if r > Fraction(1, 2) * (1 + Fraction(1, 1 << 22)):
                assert code == (2 if v > 0 else 0)
            elif r <= Fraction(1, 2):
                assert code == 1


def test_ternary_zero_bucket_and_unbiased():
    g = np.zeros(64, dtype=np.float32)
    codes, scale = orc.encode_ternary(g, None, bucket=32, mode=orc.ROUND_STOCHASTIC, seed=1)
    assert scale.tolist() == [0.0, 0.0]
    assert _unpack(codes, 64, 2) == [1] * 64

    vals = np.array([1.0, -1.0, 0.5, -0.25, 0.1, 0.9, -0.75, 0.0] * 4, dtype=np.float32)
    K = 5000
    acc = np.zeros(vals.size)
    for step in range(K):
        codes, scale = orc.encode_ternary(vals, None, bucket=32, mode=orc.ROUND_STOCHASTIC,
                                          seed=8, step=step)
        c = np.array(_unpack(codes, vals.size, 2))
        acc += (c - 1) * float(scale[0])
    mean = acc / K
    for j, v in enumerate(vals):
        pr = abs(float(v))
        sd = math.sqrt(max(pr * (1 - pr), 1e-12) / K)
        assert abs(mean[j] - float(v)) <= 5 * sd + 1e-12


# ------------------------------------------------------------------------ decode

def test_decode_hand_built_exact():
    """Three workers, two buckets, exact dyadic values: the sums are exact."""
    n, bucket, M = 64, 32, 3
    rng = np.random.default_rng(0)
    for bits in (1, 2, 4, 8):
        L = (1 << bits) - 1
        q = rng.integers(0, L + 1, size=(M, n))
        words = np.stack([_pack(q[w], bits) for w in range(M)])
        scale = np.array([[0.5, 0.25], [2.0, 0.125], [1.0, 4.0]], dtype=np.float32)
        off = np.array([[-1.0, 3.0], [0.0, -8.0], [16.0, 0.5]], dtype=np.float32)
        out = orc.decode_accumulate(words, scale, off, M=M, n=n, bits=bits, bucket=bucket,
                                    scheme=orc.SCHEME_UNIFORM)
        want = [sum(q[w, i] * float(scale[w, i // bucket]) + float(off[w, i // bucket])
                    for w in range(M)) for i in range(n)]
        assert out.tolist() == want
        # mean over M=4 (power of two: exact) and accumulate into out
        words4 = np.concatenate([words, words[:1]])
        sc4 = np.concatenate([scale, scale[:1]])
        of4 = np.concatenate([off, off[:1]])
        prior = np.full(n, 0.5, dtype=np.float32)
        out4 = orc.decode_accumulate(words4, sc4, of4, M=4, n=n, bits=bits, bucket=bucket,
                                     scheme=orc.SCHEME_UNIFORM,
                                     flags=orc.OUT_MEAN | orc.ACCUMULATE_INTO_OUT,
                                     out=prior.copy())
        want4 = [0.5 + (want[i] + q[0, i] * float(scale[0, i // bucket])
                        + float(off[0, i // bucket])) / 4 for i in range(n)]
        assert out4.tolist() == want4


def _one_vs_two_roundings(q, s, o):
    """(one rounding of q*s + o, two roundings) as binary32, from exact rationals."""
    one = to_f32(q * frac(s) + frac(o))
    two = to_f32(frac(to_f32(q * frac(s))) + frac(o))
    return one, two


def test_decode_dequantization_rounds_once():
    """'x ~ q * scale + min' is read as one rounding (fma).  With scales and
    offsets that are not powers of two, fl(q * s + o) and fl(fl(q * s) + o)
    differ on many codes; the decode (M = 1) must give the first on every one."""
    n, bucket, bits = 512, 256, 8
    q = np.arange(n) % 256
    words = _pack(q, bits)
    scale = np.array([np.float32(0.1), np.float32(1.0) / np.float32(3.0)], dtype=np.float32)
    off = np.array([np.float32(-12.7), np.float32(5.0e-3)], dtype=np.float32)
    out = orc.decode_accumulate(words[None], scale[None], off[None], M=1, n=n, bits=bits,
                                bucket=bucket, scheme=orc.SCHEME_UNIFORM)
    differ = 0
    for i in range(n):
        one, two = _one_vs_two_roundings(int(q[i]), scale[i // bucket], off[i // bucket])
        assert out[i] == one, i
        differ += one != two
    assert differ >= 20          # the pin tells the two readings apart


@pytest.mark.parametrize("mode", [orc.ROUND_NEAREST, orc.ROUND_STOCHASTIC])
def test_uniform_ef_residual_rounds_dequantization_once(mode):
    """The encode's residual e = fl(p - deq) with deq = fl(q * scale + min) (one
    rounding), checked bit for bit from exact rationals on every element, on
    buckets whose scale and min are not powers of two; the two-rounding deq
    differs on a good share of them."""
    n, bucket, bits = 1024, 256, 4
    rng = np.random.default_rng(31)
    g = (rng.standard_normal(n) * 0.37 + 0.011).astype(np.float32)
    e0 = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    err = e0.copy()
    codes, scale, off = orc.encode_uniform(g, err, bits=bits, bucket=bucket, mode=mode,
                                           seed=5, step=2)
    q = _unpack(codes, n, bits)
    differ = 0
    for i in range(n):
        k = i // bucket
        p = to_f32(frac(e0[i]) + frac(g[i]))
        one, two = _one_vs_two_roundings(q[i], scale[k], off[k])
        assert err[i] == to_f32(frac(p) - frac(one)), i
        differ += to_f32(frac(p) - frac(one)) != to_f32(frac(p) - frac(two))
    assert differ >= 20


def test_decode_sign_ternary_closed_form():
    n, bucket = 96, 32
    rng = np.random.default_rng(1)
    bitsv = rng.integers(0, 2, size=(2, n))
    s = np.array([[0.5, 1.0, 2.0], [0.25, 4.0, 8.0]], dtype=np.float32)
    out = orc.decode_accumulate(np.stack([_pack(b, 1) for b in bitsv]), s, None, M=2, n=n,
                                bits=1, bucket=bucket, scheme=orc.SCHEME_SIGN)
    want = [sum((1 if bitsv[w, i] else -1) * float(s[w, i // bucket]) for w in range(2))
            for i in range(n)]
    assert out.tolist() == want
    t = rng.integers(0, 3, size=(2, n))
    out = orc.decode_accumulate(np.stack([_pack(c, 2) for c in t]), s, None, M=2, n=n, bits=2,
                                bucket=bucket, scheme=orc.SCHEME_TERNARY)
    want = [sum((int(t[w, i]) - 1) * float(s[w, i // bucket]) for w in range(2))
            for i in range(n)]
    assert out.tolist() == want


def test_decode_fixed_worker_order():
    """Accumulation runs over workers 0..M-1 in order: 1 + 2^-24 + 2^-24 = 1 under
    round-to-nearest-even, while the reverse order would give 1 + 2^-23."""
    n, bucket = 32, 32
    codes = np.zeros((3, 1), dtype=np.uint32)
    scale = np.zeros((3, 1), dtype=np.float32)
    fwd = np.array([[1.0], [2.0 ** -24], [2.0 ** -24]], dtype=np.float32)
    out = orc.decode_accumulate(codes, scale, fwd, M=3, n=n, bits=1, bucket=bucket,
                                scheme=orc.SCHEME_UNIFORM)
    assert np.all(out == 1.0)
    out = orc.decode_accumulate(codes, scale, fwd[::-1].copy(), M=3, n=n, bits=1,
                                bucket=bucket, scheme=orc.SCHEME_UNIFORM)
    assert np.all(out == np.float32(1.0 + 2.0 ** -23))


def test_decode_single_worker_matches_encoder():
    n, bucket = 5000, 1024
    g = wl.outlier_gradient(n, seed=3)
    err = np.zeros(n, dtype=np.float32)
    codes, scale, offset = orc.encode_uniform(g, err, bits=8, bucket=bucket)
    out = orc.decode_accumulate(codes, scale, offset, M=1, n=n, bits=8, bucket=bucket,
                                scheme=orc.SCHEME_UNIFORM)
    # e = p - deq with one rounding, so deq + e recovers p to one ulp
    assert np.all(np.abs(out.astype(np.float64) + err - g) <= np.spacing(np.abs(g) + np.abs(out)))


# -------------------------------------------------------------------------- vote

@pytest.mark.parametrize("M", list(range(1, 10)))
def test_vote_brute_force(M):
    patterns = 1 << M
    reps = max(1, 96 // patterns)
    n = patterns * reps + 5                  # ragged last word
    bits = np.zeros((M, n), dtype=np.int64)
    for i in range(n):
        pat = i % patterns
        for w in range(M):
            bits[w, i] = (pat >> w) & 1
    words = np.stack([_pack(bits[w], 1) for w in range(M)])
    out = orc.sign_vote(words, M=M, n=n)
    want = [1 if 2 * bin(i % patterns).count("1") >= M else 0 for i in range(n)]
    assert _unpack(out, n, 1) == want
    tail = n % 32
    if tail:
        assert int(out[-1]) >> tail == 0
    if M % 2 == 1:                          # odd M: textbook strict majority
        assert want == [1 if bin(i % patterns).count("1") > M // 2 else 0 for i in range(n)]


# --------------------------------------------------------------------------- FP8

def test_e4m3_spec_points(golden_dir):
    for code, val in _read_golden(golden_dir, "e4m3_spec_points.txt"):
        got = orc.e4m3_to_f32(int(code, 16))
        if val == "nan":
            assert math.isnan(got)
        else:
            assert got == float(val) and math.copysign(1, got) == math.copysign(1, float(val))


def test_e4m3_order_round_trip_and_ties():
    vals = [orc.e4m3_to_f32(c) for c in range(0x7F)]
    assert all(a < b for a, b in zip(vals, vals[1:]))
    for c in range(256):
        if (c & 0x7F) == 0x7F:
            continue
        assert orc.e4m3_from_f32(orc.e4m3_to_f32(c)) == c
    for c in range(0x7E):
        lo, hi = vals[c], vals[c + 1]
        mid = (Fraction(lo) + Fraction(hi)) / 2
        even = c if c % 2 == 0 else c + 1
        assert orc.e4m3_from_f32(float(mid)) == even
        assert orc.e4m3_from_f32(-float(mid)) == 0x80 | even
        eps = (Fraction(hi) - Fraction(lo)) / 64
        assert orc.e4m3_from_f32(float(mid - eps)) == c
        assert orc.e4m3_from_f32(float(mid + eps)) == c + 1


def test_e4m3_saturation_and_nan():
    for x in (448.0, 449.0, 464.0, 479.0, 480.0, 1e6, 3.0e38, math.inf):
        assert orc.e4m3_from_f32(x) == 0x7E
        assert orc.e4m3_from_f32(-x) == 0xFE
    assert orc.e4m3_from_f32(math.nan) & 0x7F == 0x7F
    assert orc.e4m3_from_f32(2.0 ** -11) == 0x00      # below half the smallest subnormal
    assert orc.e4m3_from_f32(-(2.0 ** -11)) == 0x80
    assert orc.e4m3_from_f32(3 * 2.0 ** -11) == 0x01   # rounds up past the midpoint


def test_rowwise_fp8_rows():
    x = wl.embedding_rows(rows=257, dim=128, seed=1)
    x[5] = 0.0
    x[6, :] = np.float32(-1e-3)
    codes, sc = orc.rowwise_fp8(x)
    assert sc[5] == 0.0 and not codes[5].any()
    for r in range(x.shape[0]):
        if r == 5:
            continue
        a = np.abs(x[r]).max()
        assert sc[r] == to_f32(frac(a) / 448)
        j = int(np.argmax(np.abs(x[r])))
        assert codes[r, j] == (0x7E if x[r, j] > 0 else 0xFE)
    xh = orc.rowwise_fp8_dequant(codes, sc)
    scb = sc[:, None].astype(np.float64)
    t = np.abs(x / np.where(scb == 0, 1, scb))
    err = np.abs(xh.astype(np.float64) - x)
    normal = t >= 2.0 ** -6
    assert np.all(err[normal] <= (2.0 ** -4) * np.abs(x[normal]) * (1 + 2.0 ** -20))
    assert np.all(err[~normal] <= (2.0 ** -10) * np.broadcast_to(scb, x.shape)[~normal]
                  * (1 + 2.0 ** -20) + 1e-45)


@pytest.mark.slow
def test_rowwise_fp8_numeric_example(golden_dir):
    kv = {r[0]: int(r[1]) for r in _read_golden(golden_dir, "fp8_numeric_example.txt")}
    rows, dim = kv["lookups"], kv["dim"]
    x = wl.embedding_rows(rows=rows, dim=dim, seed=1)
    assert x.nbytes == kv["fp32_payload_bytes"]
    codes, sc = orc.rowwise_fp8(x)
    assert codes.nbytes == kv["fp8_payload_bytes"]
    assert sc.nbytes == 4 * rows
    shrink = 1 - (codes.nbytes + sc.nbytes) / x.nbytes
    assert 0.74 < shrink < 0.75


# ------------------------------------------------------------------ workloads

def test_workload_distributions():
    g = wl.outlier_gradient(1 << 20, seed=0)
    big = np.abs(g) > 0.01
    assert 0.0005 < big.mean() < 0.0015
    assert 0.9e-3 < g[~big].std() < 1.1e-3
    x = wl.embedding_rows(rows=1000, dim=128, seed=1)
    assert 0.048 < x.std() < 0.052
    sig = wl.bucket_sigmas(512 * 4000, 512, seed=2)
    lg = np.log10(sig)
    assert lg.min() >= -5 and lg.max() <= -2 and abs(lg.mean() + 3.5) < 0.05
    gw = wl.shared_mean_gradients(1 << 16, 2, seed=3)
    d = gw[0] - gw[1]
    assert abs(d.std() - math.sqrt(2) * 1e-3) < 5e-5
    b = wl.bf16_gradients(1 << 12, 2, seed=4)
    assert b.dtype == np.uint16 and b.shape == (2, 1 << 12)


# -------------------------------------------------------------------------- QSGD

@pytest.mark.parametrize("bits", [2, 4, 8])
def test_qsgd_unit_levels_and_signs(bits):
    s = (1 << (bits - 1)) - 1
    bucket, n = 64, 64 * 3 + 20
    g = _tiny_buckets(40 + bits, n)
    g[5] = -0.0
    codes, unit = orc.encode_qsgd(g, None, bits=bits, bucket=bucket, mode=orc.ROUND_STOCHASTIC,
                                  seed=3, step=1)
    c = np.array(_unpack(codes, n, bits))
    for k in range(orc.num_buckets(n, bucket)):
        seg = g[k * bucket:(k + 1) * bucket]
        want_unit = to_f32(frac(exact_norm_f32(seg)) / s)
        assert unit[k] == want_unit
        for j, v in enumerate(seg):
            code = int(c[k * bucket + j])
            assert (code >> (bits - 1)) == (1 if v < 0 else 0)
            lvl = code & s
            t = abs(frac(v)) / frac(unit[k])
            fl = t.numerator // t.denominator
            assert lvl in (min(fl, s), min(fl + 1, s))


def test_qsgd_norm_tie_and_tiny_tail():
    """sqrt(1 + 2^-23 + 2^-48) = 1 + 2^-24 exactly: the midpoint between 1 and
    its upper neighbour, so the norm rounds to even (1.0).  One element of 2^-100
    more puts the exact root just above the midpoint (1 + 2^-23); a sum of the
    squares in binary64 loses that element and would still give 1.0."""
    g = np.zeros(32, dtype=np.float32)
    g[:4] = [1.0, 2.0 ** -12, 2.0 ** -12, 2.0 ** -24]
    _, u = orc.encode_qsgd(g, None, bits=2, bucket=32)      # s = 1: unit = norm
    assert u[0] == np.float32(1.0)
    g[9] = np.float32(2.0 ** -100)
    _, u = orc.encode_qsgd(g, None, bits=2, bucket=32)
    assert u[0] == np.float32(1.0 + 2.0 ** -23)
    s64 = sum(float(v) * float(v) for v in g)
    assert np.float32(math.sqrt(s64)) == np.float32(1.0)    # the binary64 sum cannot see it


@pytest.mark.parametrize("f", [1.0, 3.7, 1e-20, 2.5e15, 0.1, 7.0e-30, 6.0e18])
@pytest.mark.parametrize("side", ["below", "above"])
def test_qsgd_norm_next_to_a_rounding_boundary(f, side):
    """Buckets whose exact sum of squares lies within 2^-90 (relative) of the
    square of a midpoint between two binary32 values: the unit is the exactly
    rounded norm divided by s (compared with Python's integer square root on
    the exact rational sum)."""
    vals, want = midpoint_bucket(f, side=side)
    bucket = 32
    g = np.zeros(bucket, dtype=np.float32)
    rng = np.random.default_rng(int(f * 1000) % 1000 + len(side))
    pos = rng.permutation(bucket)[:len(vals)]
    g[pos] = vals * np.where(rng.random(len(vals)) < 0.5, -1, 1).astype(np.float32)
    assert exact_norm_f32(g) == want
    for bits in (2, 4, 8):
        s = (1 << (bits - 1)) - 1
        _, u = orc.encode_qsgd(g, None, bits=bits, bucket=bucket, mode=orc.ROUND_NEAREST)
        assert u[0] == to_f32(frac(want) / s)


def test_qsgd_norm_random_buckets_every_magnitude():
    """Units of random buckets from 2^-140 to 2^60 in magnitude, with subnormal
    and zero elements mixed in, against the exact rational norm."""
    rng = np.random.default_rng(12)
    bucket = 64
    for t in range(60):
        g = (rng.standard_normal(bucket) * 2.0 ** rng.uniform(-140, 60)).astype(np.float32)
        g[rng.integers(0, bucket, 4)] = np.float32(2.0 ** -149) * rng.integers(1, 9)
        g[rng.integers(0, bucket, 2)] = 0.0
        _, u = orc.encode_qsgd(g, None, bits=8, bucket=bucket)
        assert u[0] == to_f32(frac(exact_norm_f32(g)) / 127), t


def test_qsgd_single_element_takes_top_level():
    g = np.zeros(32, dtype=np.float32)
    g[7] = np.float32(-0.37)
    codes, unit = orc.encode_qsgd(g, None, bits=4, bucket=32, mode=orc.ROUND_NEAREST)
    c = _unpack(codes, 32, 4)
    assert c[7] == (1 << 3) | 7
    assert all(v == 0 for i, v in enumerate(c) if i != 7)
    z, u0 = orc.encode_qsgd(np.zeros(32, dtype=np.float32), None, bits=8, bucket=32)
    assert u0[0] == 0.0 and not z.any()


def test_qsgd_unbiased_and_variance_bound():
    """E[Q(v)] = v, and E||Q(v) - v||^2 <= min(n / s^2, sqrt(n) / s) ||v||^2
    (the QSGD variance bound), over many independent steps."""
    bits, n = 4, 32
    s = (1 << (bits - 1)) - 1
    v = (np.random.default_rng(4).standard_normal(n)).astype(np.float32)
    K = 4000
    acc = np.zeros(n)
    sqerr = 0.0
    for step in range(K):
        codes, unit = orc.encode_qsgd(v, None, bits=bits, bucket=n, seed=9, step=step)
        c = np.array(_unpack(codes, n, bits))
        deq = np.where(c >> (bits - 1), -1.0, 1.0) * (c & s) * float(unit[0])
        acc += deq
        sqerr += float(((deq - v) ** 2).sum())
    mean = acc / K
    nrm2 = float((v.astype(np.float64) ** 2).sum())
    assert np.all(np.abs(mean - v) <= 6 * float(unit[0]) / math.sqrt(K))
    bound = min(n / s ** 2, math.sqrt(n) / s) * nrm2
    assert sqerr / K <= bound


def test_qsgd_decode_closed_form():
    n, bucket, bits = 64, 32, 4
    rng = np.random.default_rng(2)
    q = rng.integers(0, 16, size=(2, n))
    unit = np.array([[0.25, 2.0], [0.5, 0.125]], dtype=np.float32)
    words = np.stack([_pack(q[w], bits) for w in range(2)])
    out = orc.decode_accumulate(words, unit, None, M=2, n=n, bits=bits, bucket=bucket,
                                scheme=orc.SCHEME_QSGD)
    want = [sum((-1 if q[w, i] >> 3 else 1) * (q[w, i] & 7) * float(unit[w, i // bucket])
                for w in range(2)) for i in range(n)]
    assert out.tolist() == want


# ------------------------------------------------------------- re-encode

def _payloads(scheme, bits, M, n, bucket, seed):
    """M workers' payloads from the oracle's own encoder on seeded gradients."""
    cs, ss, os_ = [], [], []
    for w in range(M):
        g = wl.std_normal(seed + w, 1, n) * np.float32(1e-2)
        if scheme == orc.SCHEME_UNIFORM:
            c, s, o = orc.encode_uniform(g, bits=bits, bucket=bucket)
            os_.append(o)
        elif scheme == orc.SCHEME_SIGN:
            c, s = orc.encode_sign(g, bucket=bucket)
        elif scheme == orc.SCHEME_TERNARY:
            c, s = orc.encode_ternary(g, bucket=bucket, mode=orc.ROUND_NEAREST)
        else:
            c, s = orc.encode_qsgd(g, bits=bits, bucket=bucket, mode=orc.ROUND_NEAREST)
        cs.append(c)
        ss.append(s)
    return np.stack(cs), np.stack(ss), (np.stack(os_) if os_ else None)


def _unpack_codes(words, n, bits):
    per = 32 // bits
    sh = (np.arange(per, dtype=np.uint32) * bits).astype(np.uint32)
    return ((words[..., :, None] >> sh) & np.uint32((1 << bits) - 1)).reshape(*words.shape[:-1], -1)[..., :n]


def test_reencode_mean_and_quantizer_bound():
    """The decoded mean agrees with an fp64 evaluation of the dequantized
    payloads (so the sum runs over all M workers and divides by M once), and the
    re-encoded payload decodes to within half a step of err + r (round to
    nearest on the new bucket grid), with err' = (err + r) - deq' exactly."""
    M, n, bits, bucket = 5, 3000 + 17, 8, 512
    c, s, o = _payloads(orc.SCHEME_UNIFORM, bits, M, n, bucket, 40)
    q = _unpack_codes(c, n, bits).astype(np.float64)
    k = np.arange(n) // bucket
    d64 = q * s[:, k].astype(np.float64) + o[:, k].astype(np.float64)
    mean64 = d64.sum(axis=0) / M
    err0 = (wl.std_normal(9, 1, n) * np.float32(1e-5)).astype(np.float32)
    err = err0.copy()
    r, c2, s2, o2 = orc.reencode(c, s, o, M=M, n=n, bits=bits, bucket=bucket,
                                 scheme=orc.SCHEME_UNIFORM, flags=orc.OUT_MEAN, err=err)
    assert np.all(np.abs(r - mean64) <= 8 * np.finfo(np.float32).eps * np.abs(d64).sum(axis=0) / M + 1e-30)
    p = (err0 + r).astype(np.float32)
    q2 = _unpack_codes(c2, n, bits).astype(np.float64)
    deq2 = q2 * s2[k] + o2[k]
    assert np.all(np.abs(deq2 - p) <= 0.5 * s2[k] * (1 + 1e-5) + 1e-12)
    assert np.array_equal(err, (p - orc.decode_accumulate(c2, s2, o2, M=1, n=n, bits=bits,
                                                          bucket=bucket, scheme=orc.SCHEME_UNIFORM))
                          .astype(np.float32))


@pytest.mark.parametrize("scheme,bits", [(orc.SCHEME_UNIFORM, 8), (orc.SCHEME_UNIFORM, 2),
                                         (orc.SCHEME_SIGN, 1), (orc.SCHEME_TERNARY, 2)])
@pytest.mark.parametrize("mode", [orc.ROUND_NEAREST, orc.ROUND_STOCHASTIC])
def test_reencode_of_identical_payloads_is_idempotent(scheme, bits, mode):
    """Two identical payloads averaged give back each dequantized value exactly
    (x + x and the halving are exact), and those values already sit on the
    quantizer's grid: re-encoding them returns the payload's own codes.  For the
    uniform scheme every bucket holds code 0 and code L so that its min and max
    are the grid's ends; stochastic rounding of a value on the grid has nothing
    to round."""
    if scheme == orc.SCHEME_SIGN and mode == orc.ROUND_STOCHASTIC:
        pytest.skip("the sign scheme is deterministic")
    n, bucket = 4096 + 64, 512
    c, s, o = _payloads(scheme, bits, 1, n, bucket, 77)
    if scheme == orc.SCHEME_UNIFORM:
        codes = _unpack_codes(c[0], n, bits)
        L = (1 << bits) - 1
        codes[0::bucket] = 0
        codes[1::bucket] = L
        per = 32 // bits
        padded = np.zeros(-(-n // per) * per, dtype=np.uint32)
        padded[:n] = codes
        words = np.zeros(padded.size // per, dtype=np.uint32)
        for j in range(per):
            words |= padded[j::per] << np.uint32(j * bits)
        c = words[None, :]
    c2 = np.concatenate([c, c])
    s2 = np.concatenate([s, s])
    o2 = None if o is None else np.concatenate([o, o])
    r, cr, sr, orr = orc.reencode(c2, s2, o2, M=2, n=n, bits=bits, bucket=bucket, scheme=scheme,
                                  flags=orc.OUT_MEAN, mode=mode, seed=5, step=1)
    d1 = orc.decode_accumulate(c, s, o, M=1, n=n, bits=bits, bucket=bucket, scheme=scheme)
    assert np.array_equal(r.view(np.uint32), d1.view(np.uint32))
    assert np.array_equal(cr, c[0])
    if scheme == orc.SCHEME_TERNARY or scheme == orc.SCHEME_SIGN:
        assert np.array_equal(sr, s[0])


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("mode", [orc.ROUND_NEAREST, orc.ROUND_STOCHASTIC])
def test_reencode_of_identical_log_payloads_is_idempotent(bits, mode):
    """The logarithmic levels s * 2^(j - J) are exact products at these widths
    (no underflow), two identical payloads average back to them exactly, and
    every bucket keeps its top level, so the re-encode sees the same s and each
    value sits exactly on a level: the payload's own codes come back.  The one
    exception is a negative element rounded to level 0: the accumulation starts
    from +0, so it decodes to +0, which encodes with the sign bit clear."""
    n, bucket = 4096 + 64, 512
    J = (1 << (bits - 1)) - 1
    g = wl.std_normal(78, 1, n) * np.float32(1e-2)
    c, sc = orc.encode_log(g, bits=bits, bucket=bucket)
    r, cr, sr, _ = orc.reencode(np.stack([c, c]), np.stack([sc, sc]), None, M=2, n=n, bits=bits,
                                bucket=bucket, scheme=orc.SCHEME_LOG, flags=orc.OUT_MEAN,
                                mode=mode, seed=5, step=1)
    d1 = orc.decode_accumulate(c, sc, None, M=1, n=n, bits=bits, bucket=bucket,
                               scheme=orc.SCHEME_LOG)
    assert np.array_equal(r.view(np.uint32), d1.view(np.uint32))
    assert np.array_equal(sr, sc)
    codes = _unpack_codes(c, n, bits)
    want = np.where((codes & np.uint32(J)) == 0, np.uint32(0), codes)
    assert np.array_equal(_unpack_codes(cr, n, bits), want)
    assert np.any(codes != want)          # the -0 case does occur in this draw


# ------------------------------------------------------------- percentile clip

def _nearest_rank_index(cnt, pct):
    """0-based index of the nearest-rank percentile: rank ceil(pct/100 * cnt)."""
    return math.ceil(Fraction(pct, 100) * cnt) - 1


@pytest.mark.parametrize("cnt", [1, 2, 37, 99, 100, 101, 512, 1000, 2048, 4096])
def test_clip_bounds_are_nearest_rank_percentiles(cnt):
    """offset = the 1st-percentile element and scale = (p99 - p1) / L, with the
    order statistics taken from numpy's sort and the ranks from the definition."""
    rng = np.random.default_rng(cnt)
    bits, L = 8, 255
    p = (rng.standard_normal(cnt) * 1e-3).astype(np.float32)
    p[rng.integers(0, cnt, size=max(1, cnt // 50))] *= np.float32(100.0)   # outliers
    _, s, o = orc.encode_uniform_clip(p, bits=bits, bucket=max(32, -(-cnt // 32) * 32))
    srt = np.sort(p)
    lo, hi = srt[_nearest_rank_index(cnt, 1)], srt[_nearest_rank_index(cnt, 99)]
    assert o[0] == lo
    assert s[0] == np.float32(np.float32(hi - lo) / np.float32(L))


def test_clip_small_buckets_are_the_min_max_scheme():
    """Up to 99 elements the 1st and 99th percentiles are the extremes: the
    clipped encoder reproduces the min/max encoder bit for bit."""
    g = wl.outlier_gradient(99 * 7, seed=12)
    for bucket in (32, 64, 96):
        for mode in (orc.ROUND_NEAREST, orc.ROUND_STOCHASTIC):
            e1 = np.zeros(g.size, np.float32)
            e2 = np.zeros(g.size, np.float32)
            a = orc.encode_uniform(g, e1, bits=4, bucket=bucket, mode=mode, seed=3, step=1)
            b = orc.encode_uniform_clip(g, e2, bits=4, bucket=bucket, mode=mode, seed=3, step=1)
            for x, y in zip(a, b):
                assert np.array_equal(x, y)
            assert np.array_equal(e1, e2)


def test_clip_outliers_saturate_and_residual_keeps_them():
    """Elements beyond the clipped range take code 0 or L (nearest rounding); the
    residual is exactly p - deq, so an outlier's excess stays in the error
    feedback; inner elements are within half a step of their level."""
    bucket, bits, L = 2048, 8, 255
    g = wl.outlier_gradient(bucket * 4, seed=13)
    err = np.zeros(g.size, np.float32)
    c, s, o = orc.encode_uniform_clip(g, err, bits=bits, bucket=bucket)
    q = np.array([(int(c[i // 4]) >> (8 * (i % 4))) & 0xFF for i in range(g.size)])
    for k in range(4):
        sl = slice(k * bucket, (k + 1) * bucket)
        pk, qk = g[sl], q[sl]
        mx = np.sort(pk)[_nearest_rank_index(bucket, 99)]
        assert np.all(qk[pk < o[k]] == 0) and np.all(qk[pk > mx] == L)
        # one rounding of the exact q * scale + offset
        deq = np.array([to_f32(Fraction(int(a)) * Fraction(float(s[k])) + Fraction(float(o[k])))
                        for a in qk], dtype=np.float32)
        assert np.array_equal(err[sl], (pk - deq).astype(np.float32))
        inner = (pk >= o[k]) & (pk <= mx)
        assert np.all(np.abs(pk[inner].astype(np.float64) - deq[inner]) <= 0.5001 * float(s[k]))


def test_clip_shrinks_the_step_on_outlier_buckets():
    """On the outlier workload the clipped range is far narrower than min..max,
    so the quantization step of the inner elements shrinks accordingly."""
    g = wl.outlier_gradient(1 << 16, seed=14)
    _, s_mm, _ = orc.encode_uniform(g, bits=8, bucket=2048)
    _, s_cl, _ = orc.encode_uniform_clip(g, bits=8, bucket=2048)
    assert np.all(s_cl <= s_mm)
    assert np.median(s_mm / s_cl) > 3.0


def test_clip_payload_decodes_as_uniform():
    g = wl.outlier_gradient(5000, seed=15)
    c, s, o = orc.encode_uniform_clip(g, bits=4, bucket=512)
    a = orc.decode_accumulate(c, s, o, M=1, n=g.size, bits=4, bucket=512,
                              scheme=orc.SCHEME_UNIFORM_CLIP)
    b = orc.decode_accumulate(c, s, o, M=1, n=g.size, bits=4, bucket=512,
                              scheme=orc.SCHEME_UNIFORM)
    assert np.array_equal(a, b)


# ------------------------------------------------------------------ top-k

def _topk_expected(p, bucket, keep):
    """Kept indices per bucket from numpy's lexsort: |p| descending, then index."""
    out = []
    for lo in range(0, p.size, bucket):
        seg = p[lo:lo + bucket]
        order = np.lexsort((np.arange(seg.size), -np.abs(seg.astype(np.float64))))
        kept = np.sort(order[:min(keep, seg.size)]) + lo
        out.append(np.concatenate([kept, np.full(keep - kept.size, 0xFFFFFFFF)]).astype(np.uint32))
    return np.concatenate(out)


@pytest.mark.parametrize("bucket,keep,n", [(32, 1, 100), (512, 5, 3000), (1024, 10, 5000),
                                           (2048, 100, 2048 * 3 + 7), (64, 64, 200)])
def test_topk_kept_set_brute_force(bucket, keep, n):
    g = wl.outlier_gradient(n, seed=bucket + keep)
    idx, codes, s, o = orc.topk_encode(g, bucket=bucket, keep=keep)
    assert np.array_equal(idx, _topk_expected(g, bucket, keep))
    assert np.all(codes[idx == 0xFFFFFFFF] == 0)


@pytest.mark.parametrize("mode", [orc.ROUND_NEAREST, orc.ROUND_STOCHASTIC])
def test_topk_keep_all_is_the_uniform_8bit_scheme(mode):
    """Keeping every element of every bucket reduces to the uniform 8-bit encoder:
    same codes in index order, same scale, offset and residual."""
    bucket = 256
    g = wl.outlier_gradient(bucket * 5, seed=21)
    e1, e2 = np.zeros(g.size, np.float32), np.zeros(g.size, np.float32)
    idx, codes, s, o = orc.topk_encode(g, e1, bucket=bucket, keep=bucket, mode=mode, seed=4, step=2)
    c_u, s_u, o_u = orc.encode_uniform(g, e2, bits=8, bucket=bucket, mode=mode, seed=4, step=2)
    assert np.array_equal(idx, np.arange(g.size, dtype=np.uint32))
    assert np.array_equal(codes, c_u.view(np.uint8))
    assert np.array_equal(s, s_u) and np.array_equal(o, o_u) and np.array_equal(e1, e2)


def test_topk_ties_go_to_the_lower_index():
    bucket, keep = 128, 7
    g = np.where(np.arange(bucket * 2) % 2, 1.0, -1.0).astype(np.float32)
    g[bucket + 100] = 3.0
    idx, _, _, _ = orc.topk_encode(g, bucket=bucket, keep=keep)
    assert list(idx[:keep]) == list(range(keep))
    assert list(idx[keep:]) == sorted([bucket + 100] + list(range(bucket, bucket + keep - 1)))


def test_topk_residual_keeps_what_was_not_sent():
    """Dropped elements stay whole in the residual; kept ones leave p - deq, with
    deq the exact fma of code, scale and offset rounded once."""
    bucket, keep = 512, 9
    g = wl.outlier_gradient(bucket * 3, seed=22)
    e0 = (wl.std_normal(5, 1, g.size) * np.float32(1e-3)).astype(np.float32)
    err = e0.copy()
    idx, codes, s, o = orc.topk_encode(g, err, bucket=bucket, keep=keep)
    p = (e0 + g).astype(np.float32)
    sent = np.zeros(g.size, bool)
    sent[idx[idx != 0xFFFFFFFF]] = True
    assert np.array_equal(err[~sent], p[~sent])
    for t, i in enumerate(idx):
        k = int(i) // bucket
        deq = to_f32(Fraction(int(codes[t])) * Fraction(float(s[k])) + Fraction(float(o[k])))
        assert err[i] == np.float32(p[i] - deq)


def test_topk_error_feedback_delays_not_loses():
    """Over steps, everything sent plus the final residual adds up to the sum of
    the gradients (to fp32 rounding of the accumulations)."""
    bucket, keep, n, steps = 256, 4, 1024, 30
    err = np.zeros(n, np.float32)
    sent = np.zeros(n, np.float64)
    total = np.zeros(n, np.float64)
    for t in range(steps):
        g = wl.std_normal(100 + t, 1, n) * np.float32(1e-2)
        total += g
        idx, codes, s, o = orc.topk_encode(g, err, bucket=bucket, keep=keep)
        sent += orc.topk_decode(idx, codes, s, o, M=1, n=n, bucket=bucket, keep=keep)
    assert np.allclose(sent + err, total, atol=1e-5)


def test_topk_decode_scatter_order_and_skips():
    """Hand-built pairs: sentinel and out-of-bucket indices are skipped; two
    workers adding to the same element accumulate in worker order."""
    n, bucket, keep = 40, 32, 3
    idx = np.array([[5, 31, 0xFFFFFFFF, 32, 39, 3],            # worker 0: 3 is outside bucket 1
                    [5, 6, 40, 33, 0xFFFFFFFF, 0xFFFFFFFF]],   # worker 1: 40 is past n
                   dtype=np.uint32)
    codes = np.array([[2, 1, 9, 4, 1, 7], [1, 3, 5, 2, 0, 0]], dtype=np.uint8)
    scale = np.array([[1.0, 2.0], [0.5, 0.25]], dtype=np.float32)
    offset = np.array([[0.0, -1.0], [1.0, 0.0]], dtype=np.float32)
    out = orc.topk_decode(idx, codes, scale, offset, M=2, n=n, bucket=bucket, keep=keep)
    want = np.zeros(n, np.float32)
    want[5] = 2.0 + 1.5
    want[31] = 1.0
    want[6] = 2.5
    want[32] = 7.0
    want[39] = 1.0
    want[33] = 0.5
    assert np.array_equal(out, want)
    # fixed worker order: 1 + 2^-24 + 2^-24 rounds to 1 when added one by one
    idx2 = np.array([[0], [0], [0]], dtype=np.uint32)
    c2 = np.array([[1], [1], [1]], dtype=np.uint8)
    s2 = np.array([[1.0], [2.0 ** -24], [2.0 ** -24]], dtype=np.float32)
    o2 = np.zeros((3, 1), np.float32)
    r = orc.topk_decode(idx2, c2, s2, o2, M=3, n=1, bucket=32, keep=1)
    assert r[0] == np.float32(1.0)


# ------------------------------------------------------------------ log levels

def _unpack4(c, n, bits):
    per = 32 // bits
    return np.array([(int(c[i // per]) >> (bits * (i % per))) & ((1 << bits) - 1) for i in range(n)])


def test_log_levels_hand_worked():
    """4-bit codes (J = 7, levels 2^(j-7) of s = 1): exact levels, the midpoints
    (ties to the even level index), the region below the smallest level, signs."""
    g = np.array([1.0, 0.5, 0.25, 0.75, 0.375, 0.7, 0.8, -0.5, 0.0, 2.0 ** -6, 2.0 ** -7,
                  0.012, -0.3, 3 * 2.0 ** -8], np.float32)
    want = [7, 6, 5, 6, 6, 6, 7, 8 | 6, 0, 1, 0, 1, 8 | 5, 1]
    c, s = orc.encode_log(g, bits=4, bucket=32)
    assert s[0] == 1.0
    assert list(_unpack4(c, g.size, 4)) == want


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_log_nearest_is_the_nearest_level(bits):
    """Nearest rounding picks a level at least as close as either neighbour,
    measured exactly (fractions), on a random bucket of every width."""
    J = (1 << (bits - 1)) - 1
    g = (wl.std_normal(30 + bits, 1, 512) * np.float32(1e-2)).astype(np.float32)
    c, s = orc.encode_log(g, bits=bits, bucket=512)
    codes = _unpack4(c, g.size, bits)
    sv = Fraction(float(s[0]))
    levels = [Fraction(0)] + [sv * Fraction(2) ** (j - J) for j in range(1, J + 1)]
    for v, code in zip(g, codes):
        j = int(code) & ((1 << (bits - 1)) - 1)
        assert (int(code) >> (bits - 1)) == (1 if v < 0 else 0)
        x = abs(Fraction(float(v)))
        best = min(abs(x - L) for L in levels)
        # the oracle decides on fl(|p| / s), one rounding away from the exact ratio
        assert abs(x - levels[j]) <= best + sv * Fraction(2) ** -23


def test_log_stochastic_is_unbiased():
    bits, n, steps = 4, 64, 4000
    g = (wl.std_normal(33, 1, n) * np.float32(0.1)).astype(np.float32)
    acc = np.zeros(n)
    for t in range(steps):
        c, s = orc.encode_log(g, bits=bits, bucket=64, mode=orc.ROUND_STOCHASTIC, seed=9, step=t)
        acc += orc.decode_accumulate(c, s, None, M=1, n=n, bits=bits, bucket=64, scheme=orc.SCHEME_LOG)
    mean = acc / steps
    # the two levels around |p| are at most max(|p|, s * 2^(1-J)) apart (above the
    # smallest level the gap is the lower level, below it the smallest level):
    # one draw's sd is at most half the gap
    gap = np.maximum(np.abs(g), s[0] * 2.0 ** (1 - ((1 << (bits - 1)) - 1)))
    assert np.all(np.abs(mean - g) <= 6 * gap / 2 / np.sqrt(steps) + 1e-9)


def test_log_decode_closed_form_and_zero_bucket():
    bits, J = 8, 127
    g = np.zeros(64, np.float32)
    g[:32] = (wl.std_normal(34, 1, 32) * np.float32(1e-3)).astype(np.float32)
    err = np.zeros(64, np.float32)
    c, s = orc.encode_log(g, err, bits=bits, bucket=32)
    assert s[1] == 0.0 and np.all(_unpack4(c, 64, bits)[32:] == 0)
    d = orc.decode_accumulate(c, s, None, M=1, n=64, bits=bits, bucket=32, scheme=orc.SCHEME_LOG)
    codes = _unpack4(c, 64, bits)
    for i in range(32):
        j = int(codes[i]) & 0x7F
        mag = np.float32(0.0) if j == 0 else np.float32(s[0]) * np.float32(2.0 ** (j - J))
        want = -mag if codes[i] >> 7 else mag
        assert d[i] == want and err[i] == np.float32(g[i] - want)

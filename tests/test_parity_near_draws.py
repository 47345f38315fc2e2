"""Stochastic rounding exactly where the kernels' division-free decision hands
over to the division: elements whose position between two levels lies on, or
a few ulps either side of, their own Philox draw u.

The encode kernels decide u < position on a quotient taken through a rounded
reciprocal and recompute an element with the IEEE division when the two are
within reach of each other.  Random gradients almost never land there, so these
tests plant the elements: the draw u_i of every element index comes from the
oracle's generator, and the element is set so that its position equals u_i up
to a rounding or two (the planted value is rounded to binary32, then nudged by
-2..+2 ulps).  Each scheme's scale is pinned so that it is known beforehand
(QSGD's norm depends on the planted values, so those are re-planted until the
unit stops changing).  Every output must match the oracle bit for bit.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle as orc
import workloads as wl
from tests._gpu import assert_bits_equal, dev, host, u32

pytestmark = pytest.mark.gpu

SEED = 0x2468_ACE0_1357_9BDF
STEP = 9
BUCKET = 512
NB = 48


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


def _draws(n):
    return np.array([orc.uniform(SEED, STEP, i) for i in range(n)], dtype=np.float64)


def _nudge(v, k):
    """v moved by k ulps (binary32), k in -2..2."""
    v = np.asarray(v, dtype=np.float32).copy()
    for _ in range(abs(int(k))):
        v = np.nextafter(v, np.float32(np.inf) if k > 0 else np.float32(-np.inf))
    return v


def _planted(values, n):
    """values[i] rounded to binary32 and nudged by (i mod 5) - 2 ulps."""
    out = np.empty(n, dtype=np.float32)
    base = np.asarray(values, dtype=np.float64).astype(np.float32)
    for k in range(-2, 3):
        sel = (np.arange(n) % 5) == k + 2
        out[sel] = _nudge(base[sel], k)
    return out


def _encode(q, g, err0, bits, scheme):
    n = g.size
    words, nb = q.qc_code_words(n, bits), q.qc_num_buckets(n, BUCKET)
    codes = torch.full((words,), -7, dtype=torch.int32, device="cuda")
    scale = torch.full((nb,), -7.0, device="cuda")
    offset = torch.full((nb,), -7.0, device="cuda") if scheme == orc.SCHEME_UNIFORM else None
    err = torch.from_numpy(err0.copy()).cuda() if err0 is not None else None
    q.qc_encode_ef(dev(g), err, n, bits, BUCKET, scheme, q.QC_ROUND_STOCHASTIC, SEED, STEP, codes,
                   scale, offset)
    torch.cuda.synchronize()
    return (u32(codes), host(scale), host(offset) if offset is not None else None,
            host(err) if err is not None else None)


def _check(q, g, bits, scheme, oracle_fn, tag):
    for ef in (False, True):
        err0 = np.zeros(g.size, dtype=np.float32) if ef else None
        c, s, o, e = _encode(q, g, err0, bits, scheme)
        e_or = err0.copy() if ef else None
        want = oracle_fn(g, e_or)
        assert_bits_equal(c, want[0], f"{tag} ef={ef} codes")
        assert_bits_equal(s, want[1], f"{tag} ef={ef} scale")
        if o is not None:
            assert_bits_equal(o, want[2], f"{tag} ef={ef} offset")
        if ef:
            assert_bits_equal(e, e_or, f"{tag} ef={ef} err")


@pytest.mark.parametrize("bits", [1, 2, 4, 8])
def test_uniform_near_draws(q, bits):
    """Every bucket holds 0 and L*c (so min 0 and scale c exactly, c not a power
    of two); the other elements sit at (k + u_i) * c for random levels k."""
    L = (1 << bits) - 1
    n = NB * BUCKET
    c = 3.0 * 2.0 ** -7
    u = _draws(n)
    k = np.random.default_rng(bits).integers(0, max(L, 1), size=n)
    g = _planted((k + u) * c, n)
    g[::BUCKET] = 0.0
    g[1::BUCKET] = np.float32(L * c)
    g = np.clip(g, np.float32(0.0), np.float32(L * c)).astype(np.float32)
    _check(q, g, bits, orc.SCHEME_UNIFORM,
           lambda gg, e: orc.encode_uniform(gg, e, bits=bits, bucket=BUCKET,
                                            mode=orc.ROUND_STOCHASTIC, seed=SEED, step=STEP),
           f"uniform b={bits}")


def test_ternary_near_draws(q):
    """max |p| = 3 in every bucket; |p_i| = u_i * 3, random signs."""
    n = NB * BUCKET
    s = 3.0
    u = _draws(n)
    sign = np.where(np.random.default_rng(5).random(n) < 0.5, -1.0, 1.0).astype(np.float32)
    g = (_planted(u * s, n) * sign).astype(np.float32)
    g = np.clip(g, np.float32(-s), np.float32(s)).astype(np.float32)
    g[::BUCKET] = np.float32(s)
    _check(q, g, 2, orc.SCHEME_TERNARY,
           lambda gg, e: orc.encode_ternary(gg, e, bucket=BUCKET, mode=orc.ROUND_STOCHASTIC,
                                            seed=SEED, step=STEP),
           "ternary")


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_log_near_draws(q, bits):
    """max |p| = 3 in every bucket.  Between two levels the position is the
    mantissa fraction of |p| / s, so |p_i| = 3 * 2^e * (1 + u_i) for random level
    exponents e; below the smallest level it is |p| / s * 2^(J-1), so a quarter
    of the elements take |p_i| = 3 * u_i * 2^(1-J)."""
    J = (1 << (bits - 1)) - 1
    n = NB * BUCKET
    s = 3.0
    u = _draws(n)
    rng = np.random.default_rng(10 + bits)
    if J > 1:
        e = rng.integers(1 - J, 0, size=n).astype(np.float64)
        x = 2.0 ** e * (1.0 + u)
    else:
        x = u.copy()
    low = rng.random(n) < 0.25
    x[low] = u[low] * 2.0 ** (1 - J)
    sign = np.where(rng.random(n) < 0.5, -1.0, 1.0).astype(np.float32)
    g = (_planted(x * s, n) * sign).astype(np.float32)
    g = np.clip(g, np.float32(-s), np.float32(s)).astype(np.float32)
    g[::BUCKET] = np.float32(s)
    _check(q, g, bits, orc.SCHEME_LOG,
           lambda gg, e: orc.encode_log(gg, e, bits=bits, bucket=BUCKET,
                                        mode=orc.ROUND_STOCHASTIC, seed=SEED, step=STEP),
           f"log b={bits}")


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_qsgd_near_draws(q, bits):
    """Eight elements per bucket (one for 2 bits, whose single level is the
    norm itself) at (k + u_i) * unit among small random ones; the unit depends
    on them, so they are re-planted from the oracle's unit until it no longer
    changes."""
    S = (1 << (bits - 1)) - 1
    n = NB * BUCKET
    u = _draws(n)
    rng = np.random.default_rng(20 + bits)
    base = (rng.standard_normal(n) * 0.01).astype(np.float32)
    per = 1 if S == 1 else 8
    slots = []
    for b in range(NB):
        cand = np.arange(b * BUCKET + 2, (b + 1) * BUCKET)
        if S == 1:   # u_i * unit is most of the norm: keep the re-planting contracting
            cand = cand[u[cand] < 0.7]
        slots.append(rng.choice(cand, per, replace=False))
    slots = np.sort(np.concatenate(slots))
    k = rng.integers(0, max(1, (S + 3) // 4), size=slots.size).astype(np.float64)
    sign = np.where(rng.random(slots.size) < 0.5, -1.0, 1.0)
    g = base.copy()
    for _ in range(60):
        _, unit = orc.encode_qsgd(g, None, bits=bits, bucket=BUCKET, mode=orc.ROUND_STOCHASTIC,
                                  seed=SEED, step=STEP)
        ue = np.repeat(unit.astype(np.float64), BUCKET)[slots]
        new = g.copy()
        new[slots] = (_planted((k + u[slots]) * ue, slots.size) * sign).astype(np.float32)
        if np.array_equal(new, g):
            break
        g = new
    else:
        pytest.fail("the planted values did not settle")
    _check(q, g, bits, orc.SCHEME_QSGD,
           lambda gg, e: orc.encode_qsgd(gg, e, bits=bits, bucket=BUCKET,
                                         mode=orc.ROUND_STOCHASTIC, seed=SEED, step=STEP),
           f"qsgd b={bits}")


def _encode_bf16(q, g16, bits, scheme, mode, bucket):
    n = g16.size
    words, nb = q.qc_code_words(n, bits), q.qc_num_buckets(n, bucket)
    codes = torch.full((words,), -7, dtype=torch.int32, device="cuda")
    scale = torch.full((nb,), -7.0, device="cuda")
    offset = torch.full((nb,), -7.0, device="cuda") if scheme == orc.SCHEME_UNIFORM else None
    q.qc_encode_ef(dev(g16), None, n, bits, bucket, scheme, mode, SEED, STEP, codes, scale, offset,
                   dtype=q.QC_DTYPE_BF16)
    torch.cuda.synchronize()
    return u32(codes), host(scale), host(offset) if offset is not None else None


def test_ternary_bf16_draws_on_the_quotient(q):
    """bf16 gradients in buckets of 1024 with max |p| = 1, so |p| / s = |p|
    exactly: wherever an element's draw u has at most 8 significant bits it is
    a bf16 value, and the element is planted at u itself (u < |p| / s is false),
    one bf16 step above (true) or below (false), with random signs.  Every code
    and scale matches the oracle bit for bit."""
    bucket, n = 1024, 1 << 20
    u = _draws(n)
    k = np.round(u * 2.0 ** 24).astype(np.int64)
    nz = k > 0
    sig = np.zeros(n, dtype=np.int64)
    sig[nz] = np.floor(np.log2(k[nz])).astype(np.int64) - (
        np.log2(k[nz] & -k[nz]).astype(np.int64))          # span of significant bits - 1
    hits = np.flatnonzero(nz & (sig <= 7))
    assert hits.size >= 40, hits.size
    rng = np.random.default_rng(8)
    g = (rng.random(n) * 0.5).astype(np.float32) * np.where(rng.random(n) < 0.5, -1, 1).astype(np.float32)
    g16 = wl.to_bf16_bits(g)
    which = np.arange(hits.size) % 3
    vals = wl.to_bf16_bits(u[hits].astype(np.float32))
    vals = np.where(which == 1, vals + 1, np.where(which == 2, vals - 1, vals)).astype(np.uint16)
    sign = np.where(rng.random(hits.size) < 0.5, 0x8000, 0).astype(np.uint16)
    g16[hits] = vals | sign
    g16[::bucket] = wl.to_bf16_bits(np.array([1.0], dtype=np.float32))[0]
    assert np.array_equal(wl.bf16_bits_to_f32(g16[hits] & 0x7FFF)[which == 0], u[hits][which == 0])
    c, s, _ = _encode_bf16(q, g16, 2, orc.SCHEME_TERNARY, q.QC_ROUND_STOCHASTIC, bucket)
    c_or, s_or = orc.encode_ternary(g16, None, bucket=bucket, mode=orc.ROUND_STOCHASTIC,
                                    seed=SEED, step=STEP)
    assert_bits_equal(s, s_or, "ternary bf16 scale")
    assert_bits_equal(c, c_or, "ternary bf16 codes")


def test_uniform8_bf16_ties(q):
    """bf16 buckets of 1024 with min 0 and max 255 * 2^-10, so scale = 2^-10 and
    (p - min) / scale = p * 2^10 exactly: elements at k + 1/2 steps for every k
    are ties, rounded to the even level; one bf16 step either side is not."""
    bucket, nb = 1024, 64
    n = bucket * nb
    rng = np.random.default_rng(21)
    t = rng.integers(0, 127, size=n) + 0.5
    t = np.where(rng.random(n) < 0.2, rng.integers(0, 256, size=n), t)
    g16 = wl.to_bf16_bits((t * 2.0 ** -10).astype(np.float32))
    nudge = rng.integers(-1, 2, size=n)
    g16 = (g16.astype(np.int32) + np.where(g16 > 0, nudge, 0)).astype(np.uint16)
    g16[::bucket] = 0
    g16[1::bucket] = wl.to_bf16_bits(np.array([255 * 2.0 ** -10], dtype=np.float32))[0]
    g16 = np.minimum(g16, g16[1])                     # keep every bucket's max at 255 * 2^-10
    c, s, o = _encode_bf16(q, g16, 8, orc.SCHEME_UNIFORM, q.QC_ROUND_NEAREST, bucket)
    c_or, s_or, o_or = orc.encode_uniform(g16, None, bits=8, bucket=bucket)
    assert np.all(s_or == np.float32(2.0 ** -10))
    assert_bits_equal(s, s_or, "u8 bf16 scale")
    assert_bits_equal(o, o_or, "u8 bf16 offset")
    assert_bits_equal(c, c_or, "u8 bf16 codes")

"""GPU <-> oracle parity for qc_encode_ef_segments: a list of flat gradients
encoded in one launch (one per QC_MAX_SEGMENTS_PER_LAUNCH segments), each
segment bit-identical to the oracle's encode of that segment alone with its
draws indexed from the segment's place in the list, the segments laid end to
end and each padded to a multiple of 4 (the oracle's index_base).
Segments of every size, tiny and ragged, empty ones among them; the pipelined
kernel (fp32 and bf16, with and without error feedback, every scheme but the
clipped one), the receiver's bf16 kernel (8-bit nearest, ternary stochastic),
lists longer than one launch takes, and layouts that fall back to a launch per
segment (two-pass buckets, an unaligned bf16 gradient)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle as orc
import workloads as wl
from tests._gpu import assert_bits_equal, dev, host, u32

pytestmark = pytest.mark.gpu

SEED = 0x0BAD_5EED_0000_0007
STEP = 5


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


def _oracle(scheme, g, e, bits, bucket, mode, base):
    kw = dict(bucket=bucket)
    if scheme == orc.SCHEME_UNIFORM:
        c, s, o = orc.encode_uniform(g, e, bits=bits, mode=mode, seed=SEED, step=STEP,
                                     index_base=base, **kw)
        return c, s, o
    if scheme == orc.SCHEME_SIGN:
        c, s = orc.encode_sign(g, e, **kw)
    elif scheme == orc.SCHEME_TERNARY:
        c, s = orc.encode_ternary(g, e, mode=mode, seed=SEED, step=STEP, index_base=base, **kw)
    elif scheme == orc.SCHEME_QSGD:
        c, s = orc.encode_qsgd(g, e, bits=bits, mode=mode, seed=SEED, step=STEP, index_base=base,
                               **kw)
    else:
        c, s = orc.encode_log(g, e, bits=bits, mode=mode, seed=SEED, step=STEP, index_base=base,
                              **kw)
    return c, s, None


def _run(q, sizes, scheme, bits, bucket, mode, dtype, ef, unaligned=()):
    uni = scheme == orc.SCHEME_UNIFORM
    rng = np.random.default_rng(sum(sizes) + bits)
    host_g, host_e, dev_bufs, segs = [], [], [], []
    for k, n in enumerate(sizes):
        gf = (wl.std_normal(700 + k, 1, n) * np.float32(10.0 ** rng.uniform(-4, 0))) if n else \
            np.zeros(0, np.float32)
        g = wl.to_bf16_bits(gf) if dtype == "bf16" else gf
        e = (wl.std_normal(800 + k, 1, n) * np.float32(1e-5)) if ef else None
        if k in unaligned:       # a bf16 gradient 8 but not 16 bytes into its allocation
            base = torch.zeros(n + 8, dtype=torch.int16, device="cuda")
            gd = base[4:4 + n]
            gd.copy_(torch.from_numpy(g.view(np.int16)))
        else:
            gd = dev(g) if n else torch.zeros(4, device="cuda")
        ed = torch.from_numpy(e.copy()).cuda() if ef else None
        words, nb = q.qc_code_words(n, bits), q.qc_num_buckets(n, bucket)
        cd = torch.full((max(words, 1),), -7, dtype=torch.int32, device="cuda")
        sd = torch.full((max(nb, 1),), -7.0, device="cuda")
        od = torch.full((max(nb, 1),), -7.0, device="cuda") if uni else None
        host_g.append(g)
        host_e.append(e)
        dev_bufs.append((gd, ed, cd, sd, od))
        segs.append((gd, ed, n, cd, sd, od))
    dt = q.QC_DTYPE_BF16 if dtype == "bf16" else q.QC_DTYPE_F32
    q.qc_encode_ef_segments(segs, dt, bits, bucket, scheme, mode, SEED, STEP)
    torch.cuda.synchronize()
    base = 0
    for k, n in enumerate(sizes):
        gd, ed, cd, sd, od = dev_bufs[k]
        tag = f"segment {k} (n={n})"
        if n == 0:
            assert int(host(cd)[0]) == -7 and float(host(sd)[0]) == -7.0, tag + " written"
            continue
        e_or = host_e[k].copy() if ef else None
        c, s, o = _oracle(scheme, host_g[k], e_or, bits, bucket, mode, base)
        assert_bits_equal(u32(cd)[:c.size], c, tag + " codes")
        assert_bits_equal(host(sd)[:s.size], s, tag + " scale")
        if o is not None:
            assert_bits_equal(host(od)[:o.size], o, tag + " offset")
        if ef:
            assert_bits_equal(host(ed), e_or, tag + " residual")
        base += (n + 3) & ~3


SIZES = [1, 31, 32, 1000, 4096 + 17, 0, 65536, 7, 3 * 512 + 100]


@pytest.mark.parametrize("scheme,bits,mode", [(0, 8, 0), (0, 4, 1), (0, 2, 1), (0, 1, 0), (1, 1, 0),
                                              (2, 2, 1), (2, 2, 0), (3, 4, 1), (3, 8, 0), (5, 4, 1)])
@pytest.mark.parametrize("dtype,ef", [("f32", True), ("f32", False), ("bf16", False), ("bf16", True)])
def test_segments_pipelined(q, scheme, bits, mode, dtype, ef):
    """Buckets of 512: every segment on the pipelined kernel, one launch."""
    _run(q, SIZES, scheme, bits, 512, mode, dtype, ef)


@pytest.mark.parametrize("scheme,bits,mode", [(0, 8, 0), (2, 2, 1)])
def test_segments_receiver_kernel(q, scheme, bits, mode):
    """bf16, no error feedback, buckets of 1024: the receiver's kernel, with
    tiny, ragged and large segments, 16 workers' worth as one list."""
    _run(q, [1024 * 5 + 3, 17, 1024, 70_000, 0, 1] + [1 << 16] * 10, scheme, bits, 1024, mode,
         "bf16", False)


def test_segments_more_than_one_launch_holds(q):
    """150 small segments: three launches of at most 60 segments each."""
    rng = np.random.default_rng(3)
    sizes = [int(x) for x in rng.integers(1, 3000, size=150)]
    _run(q, sizes, orc.SCHEME_UNIFORM, 4, 512, 1, "f32", True)
    _run(q, sizes, orc.SCHEME_TERNARY, 2, 1024, 1, "bf16", False)


def test_segments_falling_back_to_one_launch_each(q):
    """Two-pass buckets (8192) and an unaligned bf16 gradient: each segment takes
    its own launch, with the same draw indexing."""
    _run(q, [9000, 30, 20_000], orc.SCHEME_UNIFORM, 4, 8192, 1, "f32", True)
    _run(q, [3000, 5000, 1000], orc.SCHEME_TERNARY, 2, 1024, 1, "bf16", False, unaligned=(1,))


def test_single_segment_is_encode_ef(q):
    """One segment gives qc_encode_ef's outputs (draws from index 0)."""
    n, bucket = 50_000, 512
    g = wl.std_normal(9, 1, n) * np.float32(1e-2)
    a = [torch.empty(q.qc_code_words(n, 4), dtype=torch.int32, device="cuda"),
         torch.empty(q.qc_num_buckets(n, bucket), device="cuda"),
         torch.empty(q.qc_num_buckets(n, bucket), device="cuda")]
    b = [torch.empty_like(x) for x in a]
    gd = dev(g)
    q.qc_encode_ef(gd, None, n, 4, bucket, 0, 1, SEED, STEP, *a)
    q.qc_encode_ef_segments([(gd, None, n, *b)], q.QC_DTYPE_F32, 4, bucket, 0, 1, SEED, STEP)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


@pytest.mark.parametrize("scheme,bits,mode,dtype,ef,bucket", [
    (0, 4, 1, "f32", True, 512), (2, 2, 1, "bf16", False, 1024), (0, 8, 0, "bf16", False, 1024),
    (3, 4, 1, "f32", True, 256), (5, 8, 1, "bf16", True, 512)])
def test_segments_of_one_array_are_one_call(q, scheme, bits, mode, dtype, ef, bucket):
    """Consecutive bucket-aligned slices of one array, passed as segments (each a
    view into the same buffers), give exactly one qc_encode_ef over the whole
    array: the statistics are per bucket and the draws run on end to end."""
    uni = scheme == orc.SCHEME_UNIFORM
    n = bucket * 37 + 90
    cuts = [0, bucket * 5, bucket * 6, bucket * 20, n]
    gf = wl.std_normal(31, 1, n) * np.float32(1e-2)
    g = dev(wl.to_bf16_bits(gf)) if dtype == "bf16" else dev(gf)
    e0 = wl.std_normal(32, 1, n) * np.float32(1e-5)
    dt = q.QC_DTYPE_BF16 if dtype == "bf16" else q.QC_DTYPE_F32
    per_word = 32 // bits
    outs = []
    for split in (False, True):
        err = torch.from_numpy(e0.copy()).cuda() if ef else None
        codes = torch.full((q.qc_code_words(n, bits),), -7, dtype=torch.int32, device="cuda")
        scale = torch.full((q.qc_num_buckets(n, bucket),), -7.0, device="cuda")
        offset = torch.full_like(scale, -7.0) if uni else None
        if split:
            segs = []
            for lo, hi in zip(cuts[:-1], cuts[1:]):
                bl, bh = lo // bucket, -(-hi // bucket)
                segs.append((g[lo:hi], err[lo:hi] if ef else None, hi - lo,
                             codes[lo // per_word:-(-hi // per_word)], scale[bl:bh],
                             offset[bl:bh] if uni else None))
            q.qc_encode_ef_segments(segs, dt, bits, bucket, scheme, mode, SEED, STEP)
        else:
            q.qc_encode_ef(g, err, n, bits, bucket, scheme, mode, SEED, STEP, codes, scale,
                           offset, dtype=dt)
        outs.append([x for x in (codes, scale, offset, err) if x is not None])
    for a, b in zip(*outs):
        assert torch.equal(a, b)

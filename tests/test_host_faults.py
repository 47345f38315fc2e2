"""Host-side fault injection (no GPU): an allocation that fails inside the
Python helpers must surface as the allocator's own error before anything is
launched, and leave the caller's error-feedback buffer untouched."""
from __future__ import annotations

import pytest
import torch


@pytest.fixture()
def q():
    import embedding_communication_codecs_gb300 as q
    return q


def _failing_empty(*args, **kwargs):
    raise torch.cuda.OutOfMemoryError("forced allocation failure")


def test_encode_helper_surfaces_allocation_failure(q, monkeypatch):
    calls = []
    monkeypatch.setattr(q, "qc_encode_ef", lambda *a, **k: calls.append(a))
    monkeypatch.setattr(torch, "empty", _failing_empty)
    grad = torch.ones(4096)
    err = torch.full((4096,), 0.25)
    with pytest.raises(torch.cuda.OutOfMemoryError, match="forced"):
        q.encode_ef(grad, err, bits=8, bucket=1024)
    assert calls == []
    assert bool((err == 0.25).all())


def test_decode_helper_surfaces_allocation_failure(q, monkeypatch):
    calls = []
    monkeypatch.setattr(q, "qc_decode_accumulate", lambda *a, **k: calls.append(a))
    codes = torch.zeros((2, 1024), dtype=torch.int32)
    scale = torch.zeros((2, 4))
    offset = torch.zeros((2, 4))
    monkeypatch.setattr(torch, "empty", _failing_empty)
    with pytest.raises(torch.cuda.OutOfMemoryError, match="forced"):
        q.decode_accumulate(codes, scale, offset, n=4096, bits=8, bucket=1024)
    assert calls == []


def test_library_failure_raises_with_its_message(q):
    """A non-OK status from the C ABI becomes a Python exception carrying the
    library's message (here: a bad bit width, rejected before any launch)."""
    with pytest.raises(q.QCodecError) as ei:
        q.qc_encode_ef(0x10000, None, 4096, 3, 1024, q.QC_SCHEME_UNIFORM, q.QC_ROUND_NEAREST, 0,
                       0, 0x20000, 0x30000, 0x40000, stream=0, dtype=q.QC_DTYPE_F32)
    assert ei.value.status == q.QC_ERR_INVALID_ARG
    assert "bits" in str(ei.value)

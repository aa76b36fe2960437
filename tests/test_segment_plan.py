"""Host-side segment plan of the state walks (gdr_segment_plan): a document
whose walk chain (about 7.7 us per chunk, forward and backward steps) would
outlast the rest of the step (about 50 us of SM time per chunk and value head,
spread over the SMs) is split into segments of max(64, chunks x heads / SMs)
chunks that are walked in parallel.  No device work: runs on CPU."""
import math

import numpy as np
import pytest

import gated_delta_rule_varlen_gb300 as gdr


@pytest.fixture(scope="module", autouse=True)
def lib():
    from gated_delta_rule_varlen_gb300 import build

    build.build()
    gdr.load()
    # the default slice and segment settings for every test here
    prev = gdr.gdr_set_slice_chunks(0), gdr.gdr_set_segment_chunks(0)
    yield
    gdr.gdr_set_slice_chunks(prev[0])
    gdr.gdr_set_segment_chunks(prev[1])


def _sms():
    """The SM count the library reads (152 when no device answers)."""
    import torch

    return torch.cuda.get_device_properties(0).multi_processor_count if torch.cuda.is_available() else 152


def _cu(lengths):
    return np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)


def _chunks(lengths):
    return [(n + 63) // 64 for n in lengths]


def test_one_long_document_splits_at_few_heads_only():
    # 32,768 tokens = 512 chunks: split at 16 heads and fewer, whole from 24 on
    # (measured on GB300: KDA H=16 3.47 ms split against 4.49 whole; H=24 and
    # GDN with 48 value heads faster whole).
    sms = _sms()
    for HV in (1, 4, 8, 16):
        lseg, nseg = gdr.gdr_segment_plan([0, 32768], HV)
        expect = max(64, math.ceil(512 * HV / sms))
        assert lseg == expect
        assert nseg == math.ceil(512 / expect)
    for HV in (24, 32, 48):
        assert gdr.gdr_segment_plan([0, 32768], HV) == (0, 1)


def test_four_document_pack_splits_only_at_four_heads():
    lengths = [42024, 57573, 73122, 88673]
    ch = _chunks(lengths)
    assert sum(ch) == 4086 and max(ch) == 1386
    lseg, nseg = gdr.gdr_segment_plan(_cu(lengths), 4)
    expect = max(64, math.ceil(4086 * 4 / _sms()))
    assert lseg == expect  # 108 chunks at 152 SMs
    assert nseg == sum(math.ceil(c / expect) for c in ch)
    for HV in (16, 64):
        assert gdr.gdr_segment_plan(_cu(lengths), HV) == (0, 4)


def test_many_short_documents_stay_whole():
    lengths = [2048] * 100
    assert gdr.gdr_segment_plan(_cu(lengths), 1) == (0, 100)


def test_forced_segment_length():
    prev = gdr.gdr_set_segment_chunks(100)
    try:
        # empty, 200-chunk and one-chunk documents: 1 + 2 + 1 segments
        assert gdr.gdr_segment_plan(_cu([0, 200 * 64, 64]), 16) == (100, 4)
        # a document of exactly one segment stays whole
        assert gdr.gdr_segment_plan(_cu([100 * 64]), 16) == (100, 1)
        assert gdr.gdr_segment_plan(_cu([100 * 64 + 1]), 16) == (100, 2)
    finally:
        gdr.gdr_set_segment_chunks(prev)


def test_no_documents():
    assert gdr.gdr_segment_plan([0], 16) == (0, 0)


def test_invalid_arguments():
    import ctypes

    lib = gdr.load()
    lseg, nseg = ctypes.c_int32(0), ctypes.c_int64(0)

    def plan(cu, HV, a=ctypes.byref(lseg), b=ctypes.byref(nseg)):
        arr = np.ascontiguousarray(np.asarray(cu, dtype=np.int32))
        return lib.gdr_segment_plan(len(cu) - 1, arr.ctypes.data_as(gdr.PI32), HV, a, b)

    assert plan([0, 10], 0) == gdr.GDR_INVALID_ARG
    assert plan([0, 10], 16, a=None) == gdr.GDR_INVALID_ARG
    assert plan([0, 10], 16, b=None) == gdr.GDR_INVALID_ARG
    assert plan([1, 10], 16) == gdr.GDR_BAD_CU_SEQLENS
    assert plan([0, 10, 5], 16) == gdr.GDR_BAD_CU_SEQLENS
    assert lib.gdr_segment_plan(-1, None, 16, ctypes.byref(lseg), ctypes.byref(nseg)) == gdr.GDR_INVALID_ARG
    with pytest.raises(ValueError):  # the binding maps argument errors to ValueError
        gdr.gdr_segment_plan([0, 10, 5], 16)

"""Host-side slice plan of a pipelined walk (gdr_walk_slices): the forward and
the backward walk cut a long document into slices whose end slices are
shorter, every slice starting at an even chunk.  No device work: runs on CPU."""
import pytest

import gated_delta_rule_varlen_gb300 as gdr


@pytest.fixture(scope="module", autouse=True)
def lib():
    from gated_delta_rule_varlen_gb300 import build

    build.build()
    gdr.load()


@pytest.fixture
def slice_len():
    """Sets the slice length for one test and restores the previous one."""
    prev = []

    def set_(n):
        prev.append(gdr.gdr_set_slice_chunks(n))

    yield set_
    if prev:
        gdr.gdr_set_slice_chunks(prev[0])


def _end(S, direction):
    return max(2, (S // (4 if direction else 2)) & ~1)


def _check(bounds, nch, S, direction):
    assert bounds[0] == 0 and bounds[-1] == nch
    assert all(a < b for a, b in zip(bounds, bounds[1:]))
    assert all(b % 2 == 0 for b in bounds[:-1])  # every slice starts at an even chunk
    lens = [b - a for a, b in zip(bounds, bounds[1:])]
    e = _end(S, direction)
    if nch >= 2 * e + 2:
        assert lens[0] == e
        assert lens[-1] in (e, e + 1)
        assert all(1 <= n <= S + 2 for n in lens[1:-1])
        # no more middle slices than equal slices of S need
        assert len(lens) - 2 <= -(-(nch - 2 * e) // S) + 1
    else:
        assert all(n == S for n in lens[:-1]) and 1 <= lens[-1] <= S


@pytest.mark.parametrize("direction", [0, 1])
def test_default_slices_of_a_long_document(slice_len, direction):
    slice_len(0)  # the default length, 128 chunks
    nch = 1386  # the longest document of the 4-document KDA pack, in chunks
    b = gdr.gdr_walk_slices(nch, direction)
    _check(b, nch, 128, direction)
    assert b[1] == (64 if direction == 0 else 32)


@pytest.mark.parametrize("S", [2, 4, 6, 8, 64, 128])
@pytest.mark.parametrize("direction", [0, 1])
def test_plans_over_lengths_and_slice_sizes(slice_len, S, direction):
    slice_len(S)
    for nch in list(range(1, 80)) + [127, 128, 129, 255, 256, 257, 1000, 1386, 4095]:
        _check(gdr.gdr_walk_slices(nch, direction), nch, S, direction)


def test_odd_slice_length_is_rounded_down(slice_len):
    slice_len(9)
    b = gdr.gdr_walk_slices(100, 0)
    _check(b, 100, 8, 0)


def test_empty_document_has_no_slice():
    assert gdr.gdr_walk_slices(0, 0) == [0]
    assert gdr.gdr_walk_slices(0, 1) == [0]


def test_invalid_arguments():
    import ctypes

    lib = gdr.load()
    bounds = (ctypes.c_int32 * 4)()
    n = ctypes.c_int32(0)
    assert lib.gdr_walk_slices(10, 2, bounds, 4, ctypes.byref(n)) == gdr.GDR_INVALID_ARG
    assert lib.gdr_walk_slices(-1, 0, bounds, 4, ctypes.byref(n)) == gdr.GDR_INVALID_ARG
    assert lib.gdr_walk_slices(10, 0, None, 4, ctypes.byref(n)) == gdr.GDR_INVALID_ARG
    assert lib.gdr_walk_slices(10, 0, bounds, 4, None) == gdr.GDR_INVALID_ARG
    # a plan with more slices than the array holds
    assert lib.gdr_walk_slices(1386, 0, bounds, 4, ctypes.byref(n)) == gdr.GDR_INVALID_ARG

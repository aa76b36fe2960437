"""Host-side plan of the backward's document groups (gdr_doc_groups): the
documents are ranked longest first, chunks are numbered in that order, and the
longest documents get streams of their own.  No device work: runs on CPU."""
import numpy as np
import pytest

import gated_delta_rule_varlen_gb300 as gdr


def _cu(lengths):
    return np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)


def _nch(n):
    return (n + 63) // 64


def _check_cover(groups, lengths):
    N = len(lengths)
    NC = sum(_nch(n) for n in lengths)
    assert groups[0][0] == 0 and groups[0][2] == 0
    assert groups[-1][1] == N and groups[-1][3] == NC
    for a, b in zip(groups, groups[1:]):
        assert a[1] == b[0] and a[3] == b[2]
    # chunk ranges follow the longest-first ranks
    order = sorted(range(N), key=lambda i: (-lengths[i], i))
    for r0, r1, c0, c1 in groups:
        assert c1 - c0 == sum(_nch(lengths[order[r]]) for r in range(r0, r1))


def test_four_document_pack():
    lengths = [42024, 57573, 73122, 88673]
    g = gdr.gdr_doc_groups(_cu(lengths))
    assert g == [(0, 1, 0, 1386), (1, 2, 1386, 2529), (2, 3, 2529, 3429), (3, 4, 3429, 4086)]
    _check_cover(g, lengths)


def test_single_document_and_many_short_ones_stay_one_group():
    assert gdr.gdr_doc_groups(_cu([32768])) == [(0, 1, 0, 512)]
    lengths = [256] * 100
    assert gdr.gdr_doc_groups(_cu(lengths)) == [(0, 100, 0, 400)]


def test_mixed_lengths_and_ties():
    lengths = [5000, 100, 200, 9000, 64, 0]
    g = gdr.gdr_doc_groups(_cu(lengths))
    # 9000 (141 chunks) and 5000 (79) are long enough to stand alone; the rest share one group.
    assert g == [(0, 1, 0, 141), (1, 2, 141, 220), (2, 6, 220, 227)]
    _check_cover(g, lengths)
    lengths = [8192, 8192, 8192, 8192, 8192]
    g = gdr.gdr_doc_groups(_cu(lengths))
    assert g == [(0, 1, 0, 128), (1, 2, 128, 256), (2, 3, 256, 384), (3, 5, 384, 640)]
    _check_cover(g, lengths)


def test_random_packs_cover_every_chunk_once():
    rng = np.random.default_rng(7)
    for _ in range(50):
        N = int(rng.integers(1, 40))
        lengths = [int(x) for x in rng.integers(0, 20000, N)]
        g = gdr.gdr_doc_groups(_cu(lengths))
        assert 1 <= len(g) <= 4
        _check_cover(g, lengths)


def test_bad_cu_seqlens():
    with pytest.raises(ValueError):
        gdr.gdr_doc_groups(np.array([1, 5], dtype=np.int32))
    with pytest.raises(ValueError):
        gdr.gdr_doc_groups(np.array([0, 5, 3], dtype=np.int32))
    assert gdr.gdr_doc_groups(np.array([0], dtype=np.int32)) == []


def test_above_the_ranking_limit_the_given_order_is_kept():
    # Above 4096 documents the plan keeps the given order (no ranking), on the device and here.
    lengths = [10] * 4097 + [10000]
    g = gdr.gdr_doc_groups(_cu(lengths))
    assert g == [(0, 4098, 0, 4097 + 157)]
    lengths = [10000] + [10] * 4097
    g = gdr.gdr_doc_groups(_cu(lengths))
    assert g == [(0, 1, 0, 157), (1, 4098, 157, 157 + 4097)]


def test_last_group_may_hold_only_empty_documents():
    lengths = [4200, 4096, 0, 4500]
    g = gdr.gdr_doc_groups(_cu(lengths))
    assert g == [(0, 1, 0, 71), (1, 2, 71, 137), (2, 3, 137, 201), (3, 4, 201, 201)]
    _check_cover(g, lengths)

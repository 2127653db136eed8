"""Pins of the oracle's KV index layouts ("Mini-SGLang 完整剖析" 4.6.4): the
FlashAttention / TRT-LLM dense page-id table (every page_size-th column of the
global token table divided by page_size) and the FlashInfer ragged list with
offsets.  A hand-worked example fixes the arithmetic; round trips over random
batches check that every form reads back the same slot for every token."""
import numpy as np
import pytest

import oracle
from paged_kv_gqa_store_gb300 import workload as wl

# Worked by hand, page_size 4.  Request 0 holds pages 2, 1, 5 (slots 8-11,
# 4-7, 20-23) and 10 tokens; request 1 holds pages 0, 3 and 5 tokens.
P = 4
TABLE = np.array([
    [8, 9, 10, 11, 4, 5, 6, 7, 20, 21, 22, 23],
    [0, 1, 2, 3, 12, 13, 14, 15, -1, -1, -1, -1],
], np.int32)
CACHED = np.array([7, 4], np.int32)
EXTEND = np.array([3, 1], np.int32)


def test_page_table_worked_example():
    pages, dense = oracle.build_kv_index(oracle.KV_PAGE_TABLE, P, TABLE, CACHED, EXTEND)
    assert pages == [[2, 1, 5], [0, 3]]
    assert dense.tolist() == [[2, 1, 5], [0, 3, -1]]


def test_ragged_worked_example():
    _, (indices, indptr) = oracle.build_kv_index(oracle.KV_RAGGED, P, TABLE, CACHED, EXTEND)
    assert indices.tolist() == [2, 1, 5, 0, 3]
    assert indptr.tolist() == [0, 3, 5]


def test_read_back_worked_example():
    kv_len = CACHED + EXTEND
    want = [[8, 9, 10, 11, 4, 5, 6, 7, 20, 21], [0, 1, 2, 3, 12]]
    _, dense = oracle.build_kv_index(oracle.KV_PAGE_TABLE, P, TABLE, CACHED, EXTEND)
    _, (idx, ptr) = oracle.build_kv_index(oracle.KV_RAGGED, P, TABLE, CACHED, EXTEND)
    for kind, tab, ptr_ in ((oracle.KV_TOKEN_TABLE, TABLE, None),
                            (oracle.KV_PAGE_TABLE, dense, None),
                            (oracle.KV_RAGGED, idx, ptr)):
        got = oracle.token_slots(kind, P, tab, kv_len, indptr=ptr_)
        for r in range(2):
            assert got[r, :kv_len[r]].tolist() == want[r], kind


def test_page_size_one_ragged_is_the_concatenated_rows():
    table = np.array([[5, 3, 9, 0], [7, 1, 2, 8]], np.int32)
    _, (idx, ptr) = oracle.build_kv_index(oracle.KV_RAGGED, 1, table, [2, 0], [1, 1])
    assert idx.tolist() == [5, 3, 9, 7] and ptr.tolist() == [0, 3, 4]


@pytest.mark.parametrize("page_size", [1, 16, 64])
def test_every_form_reads_back_the_token_table(page_size):
    rng = np.random.default_rng(page_size)
    cached = rng.integers(0, 300, size=9)
    ext = np.where(rng.random(9) < 0.5, 1, rng.integers(2, 90, size=9))
    need = int(((cached + ext + page_size - 1) // page_size).sum())
    spec = wl.make_batch("layouts", 77 + page_size, cached, ext, page_size, num_pages=need + 5,
                         shuffle_rows=True, extra_rows=4)
    kv_len = spec.cached_len + spec.extend_len
    ref = oracle.token_slots(oracle.KV_TOKEN_TABLE, page_size, spec.page_table, kv_len,
                             req_rows=spec.req_rows)
    _, dense = oracle.build_kv_index(oracle.KV_PAGE_TABLE, page_size, spec.page_table,
                                     spec.cached_len, spec.extend_len, spec.req_rows)
    _, (idx, ptr) = oracle.build_kv_index(oracle.KV_RAGGED, page_size, spec.page_table,
                                          spec.cached_len, spec.extend_len, spec.req_rows)
    assert np.array_equal(oracle.token_slots(oracle.KV_PAGE_TABLE, page_size, dense, kv_len), ref)
    assert np.array_equal(oracle.token_slots(oracle.KV_RAGGED, page_size, idx, kv_len,
                                             indptr=ptr), ref)
    # and the metadata of the batch read through the derived table is unchanged
    a = oracle.metadata(spec.page_table, spec.cached_len, spec.extend_len, spec.req_rows)
    b = oracle.metadata(ref, spec.cached_len, spec.extend_len)
    assert np.array_equal(a["out_loc"], b["out_loc"])

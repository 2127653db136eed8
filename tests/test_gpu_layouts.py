"""GPU parity of the KV index layouts ("Mini-SGLang 完整剖析" 4.6.4): the
FlashAttention / TRT-LLM dense page-id table and the FlashInfer ragged list,
built on the GPU from the global token table and consumed by the plan and
attention kernels.

Bars: the built indices and out_loc bit-exact against the oracle; attention
bit-identical across the three layouts (the kernels' arithmetic does not
depend on where the slots come from) and within the attention tolerance of the
oracle reading the same layout."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_gqa_store_gb300 as msg
from paged_kv_gqa_store_gb300 import workload as wl

from _harness import GpuBatch, assert_attn_close, i32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    msg.load_library()


def _spec(seed, page_size, n_dec=13, n_ext=4):
    rng = np.random.default_rng(seed)
    cached = np.concatenate([rng.integers(0, 900, size=n_dec), rng.integers(0, 300, size=n_ext)])
    ext = np.concatenate([np.ones(n_dec, np.int64), rng.integers(2, 200, size=n_ext)])
    order = rng.permutation(n_dec + n_ext)
    cached, ext = cached[order], ext[order]
    need = int(((cached + ext + page_size - 1) // page_size).sum())
    return wl.make_batch(f"layout{seed}_p{page_size}", seed, cached, ext, page_size,
                         num_pages=need + 9, shuffle_rows=True, extra_rows=3)


def _build(spec, kind, gb, status):
    kv_len = spec.cached_len.astype(np.int64) + spec.extend_len
    pages = (kv_len + spec.page_size - 1) // spec.page_size
    if kind == msg.MSG_KV_PAGE_TABLE:
        out = torch.full((spec.num_reqs, int(pages.max()) + 3), -7, dtype=torch.int32,
                         device="cuda")
        msg.msg_build_kv_index(kind, spec.page_size, gb.page_table, gb.cached, gb.extend, out,
                               req_rows=gb.rows, dev_status=status)
        return msg.KvIndex(kind, out, spec.page_size), out, None
    out = torch.full((int(pages.sum()) + 5,), -7, dtype=torch.int32, device="cuda")
    ptr = torch.zeros(spec.num_reqs + 1, dtype=torch.int32, device="cuda")
    msg.msg_build_kv_index(kind, spec.page_size, gb.page_table, gb.cached, gb.extend, out,
                           req_rows=gb.rows, out_indptr=ptr, dev_status=status)
    return msg.KvIndex(kind, out, spec.page_size, indptr=ptr), out, ptr


@pytest.mark.parametrize("page_size", [1, 16, 64])
def test_build_kv_index_matches_oracle(page_size):
    spec = _spec(500 + page_size, page_size)
    gb = GpuBatch(spec)
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    _, dense, _ = _build(spec, msg.MSG_KV_PAGE_TABLE, gb, status)
    _, flat, ptr = _build(spec, msg.MSG_KV_RAGGED, gb, status)
    torch.cuda.synchronize()
    assert msg.msg_read_device_status(status)[0] == msg.MSG_OK
    _, want_dense = oracle.build_kv_index(oracle.KV_PAGE_TABLE, page_size, spec.page_table,
                                          spec.cached_len, spec.extend_len, spec.req_rows)
    _, (want_idx, want_ptr) = oracle.build_kv_index(oracle.KV_RAGGED, page_size, spec.page_table,
                                                    spec.cached_len, spec.extend_len,
                                                    spec.req_rows)
    got = dense.cpu().numpy()
    w = want_dense.shape[1]
    # entries past a request's pages are left untouched
    valid = want_dense >= 0
    assert np.array_equal(got[:, :w][valid], want_dense[valid])
    assert (got[:, :w][~valid] == -7).all() and (got[:, w:] == -7).all()
    assert np.array_equal(ptr.cpu().numpy(), want_ptr)
    f = flat.cpu().numpy()
    assert np.array_equal(f[:len(want_idx)], want_idx) and (f[len(want_idx):] == -7).all()


@pytest.mark.parametrize("page_size", [1, 16])
def test_attention_layouts_identical_and_match_oracle(page_size):
    spec = _spec(600 + page_size, page_size)
    host = wl.host_tensors(spec)
    gb = GpuBatch(spec)
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    q = wl.bits_to_torch(host["q"], "cuda")
    kn, vn = wl.bits_to_torch(host["k_new"], "cuda"), wl.bits_to_torch(host["v_new"], "cuda")
    kp, vp = wl.bits_to_torch(host["k_pool"], "cuda"), wl.bits_to_torch(host["v_pool"], "cuda")
    loc = gb.plan()
    msg.msg_store_kv(kn, vn, kp, vp, loc, dev_status=gb.ws)
    outs = {"token": gb.attention(q, kp, vp)}
    kv_len = spec.cached_len.astype(np.int64) + spec.extend_len
    for name, kind in (("page", msg.MSG_KV_PAGE_TABLE), ("ragged", msg.MSG_KV_RAGGED)):
        kv, table, ptr = _build(spec, kind, gb, status)
        # the plan through this layout gives the same out_loc as the oracle reading it
        loc2 = torch.zeros_like(loc)
        msg.msg_plan_ex(kv, gb.cached, gb.extend, spec.total_q, spec.num_slots, gb.ws,
                        out_loc_out=loc2)
        out = torch.empty_like(q)
        msg.msg_paged_attention_ex(q, kp, vp, kv, gb.cached, gb.extend, gb.qo, out, gb.ws,
                                   max_kv_len=spec.max_kv_len)
        torch.cuda.synchronize()
        tab = table.cpu().numpy()
        slots = oracle.token_slots(kind, page_size, tab, kv_len,
                                   indptr=None if ptr is None else ptr.cpu().numpy())
        meta = oracle.metadata(slots, spec.cached_len, spec.extend_len)
        assert np.array_equal(loc2.cpu().numpy(), meta["out_loc"]), name
        outs[name] = out
        ref = oracle.paged_attention(host["q"], wl.torch_to_bits(kp), wl.torch_to_bits(vp), slots,
                                     spec.cached_len, meta["qo_indptr"], 16, 8, 128)
        assert_attn_close(wl.torch_to_bits(out), ref, name)
    assert msg.msg_read_device_status(gb.ws)[0] == msg.MSG_OK
    assert msg.msg_read_device_status(status)[0] == msg.MSG_OK
    for name in ("page", "ragged"):
        assert torch.equal(outs[name].view(torch.int16), outs["token"].view(torch.int16)), name


def test_ragged_range_shorter_than_the_request_is_reported():
    spec = _spec(700, 1, n_dec=3, n_ext=1)
    gb = GpuBatch(spec)
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    kv, flat, ptr = _build(spec, msg.MSG_KV_RAGGED, gb, status)
    bad = ptr.clone()
    need1 = int(spec.cached_len[1]) + int(spec.extend_len[1])
    bad[2] = bad[1] + need1 - 1                        # request 1's range one entry short
    kv_bad = msg.KvIndex(msg.MSG_KV_RAGGED, flat, 1, indptr=bad)
    msg.msg_plan_ex(kv_bad, gb.cached, gb.extend, spec.total_q, spec.num_slots, gb.ws)
    st, info = msg.msg_read_device_status(gb.ws)
    assert st == msg.MSG_ERR_DEVICE_CHECK and info[0] == msg.MSG_DEV_BAD_LENGTHS


def test_page_id_outside_the_pool_is_reported_and_read_as_slot_zero():
    spec = _spec(710, 16, n_dec=4, n_ext=0)
    host = wl.host_tensors(spec)
    gb = GpuBatch(spec)
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    kv, dense, _ = _build(spec, msg.MSG_KV_PAGE_TABLE, gb, status)
    dense[2, 0] = spec.num_slots // 16 + 3            # a page past the pool
    q = wl.bits_to_torch(host["q"], "cuda")
    kp, vp = wl.bits_to_torch(host["k_pool"], "cuda"), wl.bits_to_torch(host["v_pool"], "cuda")
    gb.plan()
    out = torch.empty_like(q)
    msg.msg_paged_attention_ex(q, kp, vp, kv, gb.cached, gb.extend, gb.qo, out, gb.ws)
    st, info = msg.msg_read_device_status(gb.ws)
    assert st == msg.MSG_ERR_DEVICE_CHECK and info[0] == msg.MSG_DEV_SLOT_OUT_OF_RANGE


def test_misaligned_page_start_is_reported_when_building():
    spec = _spec(720, 16, n_dec=3, n_ext=1)
    gb = GpuBatch(spec)
    pt = gb.page_table.clone()
    row = int(spec.req_rows[1])
    pt[row, 0] += 1                                    # page start no longer a multiple of 16
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    out = torch.full((spec.num_reqs, 64), -7, dtype=torch.int32, device="cuda")
    msg.msg_build_kv_index(msg.MSG_KV_PAGE_TABLE, 16, pt, gb.cached, gb.extend, out,
                           req_rows=gb.rows, dev_status=status)
    st, info = msg.msg_read_device_status(status)
    assert st == msg.MSG_ERR_DEVICE_CHECK and info[0] == msg.MSG_DEV_PAGE_MISALIGNED
    assert int(out[1, 0]) == -1

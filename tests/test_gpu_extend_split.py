"""Extend batches with few work items, whose key tiles the extend kernel
splits over all CTAs (each CTA an equal range of key tiles, a range boundary
inside an item leaving fp32 partials that the item's last piece merges):
a chunked-prefill step (one 128-token query tile over a long cached prefix:
"Mini-SGLang 源码解析（四）" chunked prefill; "第 0 步" causal attention
offset by cached_len) and a few ragged extends mixed with decodes.

Each batch is checked against the fp64 oracle with the workspace the library
asks for (key split) and with a workspace too small for the split (items
taken whole); a repeated call gives the same bits (the merge sums the
pieces in a fixed order)."""
import numpy as np
import pytest
import torch

import paged_kv_gqa_store_gb300 as msg
from paged_kv_gqa_store_gb300 import workload as wl

from _harness import GpuBatch, assert_attn_close, oracle_small

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    msg.load_library()


def _run(spec, host, ws_bytes=None):
    dev = "cuda"
    gb = GpuBatch(spec, dev)
    if ws_bytes is not None:
        gb.ws = gb.ws[:ws_bytes]
    q = wl.bits_to_torch(host["q"], dev)
    k_pool, v_pool = wl.bits_to_torch(host["k_pool"], dev), wl.bits_to_torch(host["v_pool"], dev)
    loc = gb.plan()
    msg.msg_store_kv(wl.bits_to_torch(host["k_new"], dev), wl.bits_to_torch(host["v_new"], dev),
                     k_pool, v_pool, loc, dev_status=gb.ws)
    out = gb.attention(q, k_pool, v_pool, flags=msg.MSG_ATTN_REUSE_PLAN)
    torch.cuda.synchronize()
    st, info = gb.status()
    assert st == msg.MSG_OK, info
    return wl.torch_to_bits(out)


def _check(spec):
    host = wl.host_tensors(spec)
    ref = oracle_small(spec, host)["out"]
    split = _run(spec, host)
    assert_attn_close(split, ref, f"{spec.name} (key split)")
    assert np.array_equal(_run(spec, host), split), "repeated call differs"
    # 16 MiB holds the plan and the decode partials of these batches but not
    # the split's partial slots: the kernel then takes items whole
    whole = _run(spec, host, ws_bytes=16 << 20)
    assert_attn_close(whole, ref, f"{spec.name} (whole items)")


@pytest.mark.parametrize("page_size", [1, 16])
def test_chunked_prefill_tile_over_long_prefix(page_size):
    """One request, 128 new tokens (8 work items) over a 20,000-token prefix:
    158 key tiles per item spread over every CTA."""
    cached, ext = np.array([20000]), np.array([128])
    pages = int(((cached + ext + page_size - 1) // page_size)[0]) + 9
    spec = wl.make_batch("split_chunk", 700 + page_size, cached, ext, page_size, num_pages=pages)
    _check(spec)


def test_ragged_extends_with_decodes():
    """Four extends (100, 300, 70 and 2 new tokens over prefixes of 6,000,
    15,000, 9,000 and 0) and five decodes in one call: 40 work items; pieces
    that start late hold rows none of whose keys they see."""
    cached = np.array([6000, 15000, 9000, 0, 40, 3000, 700, 12000, 1])
    ext = np.array([100, 300, 70, 2, 1, 1, 1, 1, 1])
    spec = wl.make_batch("split_ragged", 710, cached, ext, 1,
                         num_pages=int((cached + ext).sum()) + 16)
    _check(spec)


@pytest.mark.parametrize("hkv", [4, 2])
def test_chunked_prefill_on_a_head_slice(hkv):
    """The chunked-prefill step on a tensor-parallel rank's head slice (8q/4kv
    at tp = 2, 4q/2kv at tp = 4: "Mini-SGLang 完整剖析" 4.5): 256 new tokens
    over a 40,000-token prefix, 2 query tiles x hkv work items, split the same
    way."""
    cached, ext = np.array([40000]), np.array([256])
    spec = wl.make_batch("split_chunk_tp", 720 + hkv, cached, ext, 1, num_pages=40256 + 9,
                         num_qo_heads=2 * hkv, num_kv_heads=hkv)
    _check(spec)


def test_split_step_captured_in_a_graph():
    """A chunked-prefill step (plan, store_kv, the split extend kernel and the
    merge kernel, the counters zeroed between them) captured once in a CUDA
    graph and replayed: each replay equals the oracle and the eager call bit
    for bit."""
    cached, ext = np.array([20000]), np.array([128])
    spec = wl.make_batch("split_graph", 730, cached, ext, 1, num_pages=20128 + 9)
    host = wl.host_tensors(spec)
    ref = oracle_small(spec, host)["out"]
    eager = _run(spec, host)
    dev = "cuda"
    gb = GpuBatch(spec, dev)
    q = wl.bits_to_torch(host["q"], dev)
    kn, vn = wl.bits_to_torch(host["k_new"], dev), wl.bits_to_torch(host["v_new"], dev)
    kp, vp = wl.bits_to_torch(host["k_pool"], dev), wl.bits_to_torch(host["v_pool"], dev)
    out = torch.empty_like(q)

    def step():
        loc = gb.plan()
        msg.msg_store_kv(kn, vn, kp, vp, loc, dev_status=gb.ws)
        gb.attention(q, kp, vp, out=out, flags=msg.MSG_ATTN_REUSE_PLAN)

    step()                                           # warm-up (kernel attributes)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for rep in range(2):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert gb.status()[0] == msg.MSG_OK
        got = wl.torch_to_bits(out)
        assert np.array_equal(got, eager), f"replay {rep} differs from the eager call"
        assert_attn_close(got, ref, f"graph replay {rep}")

"""GPU parity at the full workload sizes, in the launch configuration the
benchmark times, on outputs the oracle computes one by one: a sample of
requests (and, for extend requests, of query rows incl. tile boundaries) is
relabelled into a compact pool and checked against the fp64 oracle; store_kv is
checked bit-exactly on the rows it wrote."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_gqa_store_gb300 as msg
from paged_kv_gqa_store_gb300 import workload as wl

from _harness import GpuBatch, assert_attn_close, sampled_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    msg.load_library()
    yield
    torch.cuda.empty_cache()


def _check_qo_and_loc(spec, gb):
    meta = oracle.metadata(spec.page_table, spec.cached_len, spec.extend_len, spec.req_rows)
    assert np.array_equal(gb.qo.cpu().numpy(), meta["qo_indptr"])
    assert np.array_equal(gb.out_loc.cpu().numpy(), meta["out_loc"])
    assert np.array_equal(gb.positions.cpu().numpy(), meta["positions"])
    return meta


def _check_store(t, loc):
    idx = loc if loc.dtype == torch.int64 else loc.long()
    assert torch.equal(t["k_pool"].index_select(0, idx).view(torch.int16),
                       t["k_new"].view(torch.int16))
    assert torch.equal(t["v_pool"].index_select(0, idx).view(torch.int16),
                       t["v_new"].view(torch.int16))


def test_decode_64_reqs_28_layers():
    spec = wl.config_decode_28_layers()
    gb = GpuBatch(spec)
    layers = [wl.device_tensors(spec, layer) for layer in range(spec.num_layers)]
    rng = np.random.default_rng(5)
    reqs = np.sort(rng.choice(spec.num_reqs, 8, replace=False))
    refs = {}
    for layer in (0, 13, 27):
        t = layers[layer]
        refs[layer] = sampled_oracle(spec, (t["k_pool"], t["v_pool"]), t["q"], t["k_new"],
                                     t["v_new"], reqs)
    loc = gb.plan()
    outs = []
    for t in layers:
        msg.msg_store_kv(t["k_new"], t["v_new"], t["k_pool"], t["v_pool"], loc)
        outs.append(gb.attention(t["q"], t["k_pool"], t["v_pool"],
                                 flags=msg.MSG_ATTN_REUSE_PLAN | msg.MSG_ATTN_DECODE_ONLY))
    torch.cuda.synchronize()
    assert gb.status()[0] == msg.MSG_OK
    _check_qo_and_loc(spec, gb)
    for layer, (rows, ref) in refs.items():
        _check_store(layers[layer], loc)
        got = wl.torch_to_bits(outs[layer][torch.from_numpy(rows).cuda()])
        assert_attn_close(got, ref, f"layer {layer}")
    for o in outs:
        assert torch.isfinite(o.float()).all()


def test_decode_64_reqs_28_layers_fused_store_as_benchmarked():
    """The benchmark's headline step exactly: one plan, then per layer one
    msg_paged_attention_store (the decode kernel stores the step's new K/V rows
    itself) with MSG_ATTN_REUSE_PLAN | MSG_ATTN_DECODE_ONLY and the host
    max_kv_len hint, 28 layers on one workspace.  Every layer: 6 sampled
    requests against the oracle, and the 64 stored rows bit-exactly."""
    spec = wl.config_decode_28_layers()
    gb = GpuBatch(spec)
    layers = [wl.device_tensors(spec, layer) for layer in range(spec.num_layers)]
    rng = np.random.default_rng(15)
    refs = {}
    for layer, t in enumerate(layers):
        reqs = np.sort(rng.choice(spec.num_reqs, 6, replace=False))
        refs[layer] = sampled_oracle(spec, (t["k_pool"], t["v_pool"]), t["q"], t["k_new"],
                                     t["v_new"], reqs)
    loc = gb.plan()
    outs = []
    flags = msg.MSG_ATTN_REUSE_PLAN | msg.MSG_ATTN_DECODE_ONLY
    for t in layers:
        o = torch.full_like(t["q"], float("nan"))
        msg.msg_paged_attention_store(t["q"], t["k_new"], t["v_new"], t["k_pool"], t["v_pool"],
                                      gb.page_table, gb.cached, gb.extend, gb.qo, o, gb.ws,
                                      page_size=spec.page_size, req_rows=gb.rows,
                                      max_kv_len=spec.max_kv_len, flags=flags)
        outs.append(o)
    torch.cuda.synchronize()
    assert gb.status()[0] == msg.MSG_OK
    _check_qo_and_loc(spec, gb)
    for layer, (rows, ref) in refs.items():
        _check_store(layers[layer], loc)
        got = wl.torch_to_bits(outs[layer][torch.from_numpy(rows).cuda()])
        assert_attn_close(got, ref, f"layer {layer}")
    for o in outs:
        assert torch.isfinite(o.float()).all()


def test_decode_256_reqs_page16_pool_90pct_of_free_hbm():
    torch.cuda.empty_cache()
    free, _ = torch.cuda.mem_get_info()
    pages = int(0.9 * free) // (2 * 16 * spec_row_bytes())
    spec = wl.config_large_decode(pages)
    t = wl.device_tensors(spec)
    gb = GpuBatch(spec)
    reqs = np.sort(np.random.default_rng(6).choice(spec.num_reqs, 8, replace=False))
    rows, ref = sampled_oracle(spec, (t["k_pool"], t["v_pool"]), t["q"], t["k_new"],
                               t["v_new"], reqs)
    loc = gb.plan()
    msg.msg_store_kv(t["k_new"], t["v_new"], t["k_pool"], t["v_pool"], loc)
    out = gb.attention(t["q"], t["k_pool"], t["v_pool"],
                       flags=msg.MSG_ATTN_REUSE_PLAN | msg.MSG_ATTN_DECODE_ONLY)
    torch.cuda.synchronize()
    assert gb.status()[0] == msg.MSG_OK
    _check_qo_and_loc(spec, gb)
    _check_store(t, loc)
    assert_attn_close(wl.torch_to_bits(out[torch.from_numpy(rows).cuda()]), ref, "config 3")
    assert torch.isfinite(out.float()).all()
    del t
    torch.cuda.empty_cache()


def spec_row_bytes():
    return wl.HKV * wl.HEAD_DIM * 2


def test_extend_8_reqs():
    spec = wl.config_extend()
    t = wl.device_tensors(spec)
    gb = GpuBatch(spec)
    rows, ref = sampled_oracle(spec, (t["k_pool"], t["v_pool"]), t["q"], t["k_new"], t["v_new"],
                               np.arange(spec.num_reqs), rows_per_req=48,
                               rng=np.random.default_rng(8))
    loc = gb.plan()
    msg.msg_store_kv(t["k_new"], t["v_new"], t["k_pool"], t["v_pool"], loc)
    out = gb.attention(t["q"], t["k_pool"], t["v_pool"],
                       flags=msg.MSG_ATTN_REUSE_PLAN | msg.MSG_ATTN_EXTEND_ONLY)
    torch.cuda.synchronize()
    assert gb.status()[0] == msg.MSG_OK
    _check_qo_and_loc(spec, gb)
    _check_store(t, loc)
    assert_attn_close(wl.torch_to_bits(out[torch.from_numpy(rows).cuda()]), ref, "config 4")
    assert torch.isfinite(out.float()).all()


def test_long_context_mixed_page64():
    spec = wl.config_long_mixed()
    t = wl.device_tensors(spec)
    gb = GpuBatch(spec)
    reqs = np.array([0, 17, 31, 32, 33])
    rows, ref = sampled_oracle(spec, (t["k_pool"], t["v_pool"]), t["q"], t["k_new"], t["v_new"],
                               reqs, rows_per_req=40, rng=np.random.default_rng(9))
    loc = gb.plan()
    msg.msg_store_kv(t["k_new"], t["v_new"], t["k_pool"], t["v_pool"], loc)
    out = gb.attention(t["q"], t["k_pool"], t["v_pool"], flags=msg.MSG_ATTN_REUSE_PLAN)
    torch.cuda.synchronize()
    assert gb.status()[0] == msg.MSG_OK
    _check_qo_and_loc(spec, gb)
    _check_store(t, loc)
    assert_attn_close(wl.torch_to_bits(out[torch.from_numpy(rows).cuda()]), ref, "config 5")
    assert torch.isfinite(out.float()).all()

"""CUDA-graph replay of the decode step, checked against the fp64 oracle.

The whole path runs from device-side metadata with no host synchronisation and
fixed launch shapes, so one captured graph serves every later step of a
fixed-size (padded) decode batch: the caller updates cached_len, the page-table
rows, q and the new k/v in place and replays.  Padding requests point at the
dummy slot, as in a CUDA-graph-padded engine batch ("Engine 与采样器", 初始化的
顺序: the extra dummy page and the dummy row; "Mini-SGLang 源码解析（四）"
10.6-10.7: the batch-size ladder and padding to the next captured size).

Every replayed step's outputs and the pools are compared with the oracle run
on the same inputs; replay and eager execution must also agree bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_gqa_store_gb300 as msg
from paged_kv_gqa_store_gb300 import graph as mgraph
from paged_kv_gqa_store_gb300 import workload as wl

from _harness import assert_attn_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    msg.load_library()


def test_ladder_and_padding_rule():
    # CPU logic, exercised here with its GPU users: the pages' ladder and
    # "the first captured size >= the batch"
    sizes = mgraph.graph_batch_sizes(256)
    assert sizes[:5] == [1, 2, 4, 8, 16] and sizes[-1] == 256 and len(sizes) == 35
    assert mgraph.padded_size(sizes, 10) == 16 and mgraph.padded_size(sizes, 3) == 4
    assert mgraph.padded_size(sizes, 256) == 256


class _Requests:
    """Decode requests with room for `steps` more tokens each, a dummy row
    (every entry the dummy slot, the last slot of the pool) and host copies
    of the pools that the oracle updates step by step."""

    def __init__(self, seed, n, ctx_lo, ctx_hi, steps, layers):
        rng = np.random.default_rng(seed)
        self.ctx = rng.integers(ctx_lo, ctx_hi, size=n)
        spec = wl.make_batch("graph", seed, cached_len=self.ctx - 1 + steps,
                             extend_len=np.ones(n, np.int32), page_size=1,
                             num_pages=int((self.ctx + steps).sum()) + 64)
        self.dummy_slot = spec.num_slots
        self.num_slots = spec.num_slots + 1
        width = spec.page_table.shape[1]
        self.pt = np.zeros((n + 1, width), np.int32)
        self.pt[:n] = spec.page_table
        self.pt[n, :] = self.dummy_slot
        self.dummy_row = n
        self.cached = (self.ctx - 1).astype(np.int32)        # advances one per step
        self.pools = [(wl.random_bf16(rng, (self.num_slots, 8, 128)),
                       wl.random_bf16(rng, (self.num_slots, 8, 128))) for _ in range(layers)]
        self.rng = rng

    def device_pools(self):
        return [(wl.bits_to_torch(k, "cuda"), wl.bits_to_torch(v, "cuda")) for k, v in self.pools]

    def oracle_step(self, live, q, kn, vn):
        """Store the live requests' new rows in the host pools and attend;
        returns one fp64 output per layer."""
        cached = self.cached[live]
        ext = np.ones(len(live), np.int32)
        meta = oracle.metadata(self.pt, cached, ext, live.astype(np.int32))
        outs = []
        for (kp, vp), qq, kk, vv in zip(self.pools, q, kn, vn):
            oracle.store_kv(kk, vv, meta["out_loc"], kp, vp)
            outs.append(oracle.paged_attention(qq, kp, vp, self.pt, cached, meta["qo_indptr"],
                                               16, 8, 128, req_rows=live.astype(np.int32)))
        self.cached[live] += 1                                # Req.complete_one
        return outs


def test_graph_ladder_replay_matches_oracle():
    """Graphs captured for the ladder up to 32 (1, 2, 4, 8, 16, 24, 32), live
    batches of 7 sizes padded to 7 different captured sizes, 2 layers of the
    fused store + decode step per replay; every step checked against the
    oracle, and the pools bit-exactly at the end."""
    layers, max_bs = 2, 32
    live_sizes = [3, 1, 13, 24, 2, 8, 30, 5]
    R = _Requests(21, max_bs, 20, 700, len(live_sizes), layers)
    pools = R.device_pools()
    runner = mgraph.DecodeGraphRunner(pools, torch.from_numpy(R.pt).cuda(), R.dummy_row, max_bs)
    runner.capture()
    seen = set()
    for step, n in enumerate(live_sizes):
        live = np.sort(R.rng.choice(max_bs, n, replace=False))
        q = [wl.random_bf16(R.rng, (n, 16, 128)) for _ in range(layers)]
        kn = [wl.random_bf16(R.rng, (n, 8, 128)) for _ in range(layers)]
        vn = [wl.random_bf16(R.rng, (n, 8, 128)) for _ in range(layers)]
        for i in range(layers):
            runner.q[i][:n].copy_(wl.bits_to_torch(q[i], "cuda"))
            runner.k_new[i][:n].copy_(wl.bits_to_torch(kn[i], "cuda"))
            runner.v_new[i][:n].copy_(wl.bits_to_torch(vn[i], "cuda"))
        bs = runner.replay(R.cached[live], live)
        seen.add(bs)
        assert bs == mgraph.padded_size(runner.sizes, n)
        torch.cuda.synchronize()
        refs = R.oracle_step(live, q, kn, vn)
        for i in range(layers):
            assert_attn_close(wl.torch_to_bits(runner.out[i][:n]), refs[i],
                              f"step {step} (live {n}, graph {bs}) layer {i}")
    assert len(seen) == len(live_sizes) - 1 >= 4
    real = np.arange(R.num_slots) != R.dummy_slot
    for (kd, vd), (kh, vh) in zip(pools, R.pools):
        assert np.array_equal(wl.torch_to_bits(kd)[real], kh[real])
        assert np.array_equal(wl.torch_to_bits(vd)[real], vh[real])
    assert msg.msg_read_device_status(runner.ws)[0] == msg.MSG_OK


def test_graph_replay_matches_eager_and_oracle_over_steps():
    """The same padded batch (6 live requests in a graph of 8) over 3 steps:
    replay equals eager execution bit for bit, and both equal the oracle."""
    layers, max_bs, n, steps = 2, 8, 6, 3
    R = _Requests(7, n, 200, 3000, steps, layers)
    pools_g, pools_e = R.device_pools(), R.device_pools()
    pt = torch.from_numpy(R.pt).cuda()
    graph_r = mgraph.DecodeGraphRunner(pools_g, pt, R.dummy_row, max_bs)
    eager_r = mgraph.DecodeGraphRunner(pools_e, pt, R.dummy_row, max_bs)
    graph_r.capture()
    live = np.arange(n)
    for s in range(steps):
        q = [wl.random_bf16(R.rng, (n, 16, 128)) for _ in range(layers)]
        kn = [wl.random_bf16(R.rng, (n, 8, 128)) for _ in range(layers)]
        vn = [wl.random_bf16(R.rng, (n, 8, 128)) for _ in range(layers)]
        for r in (graph_r, eager_r):
            for i in range(layers):
                r.q[i][:n].copy_(wl.bits_to_torch(q[i], "cuda"))
                r.k_new[i][:n].copy_(wl.bits_to_torch(kn[i], "cuda"))
                r.v_new[i][:n].copy_(wl.bits_to_torch(vn[i], "cuda"))
        assert graph_r.replay(R.cached[live], live) == 8
        assert eager_r.eager(R.cached[live], live) == 8
        torch.cuda.synchronize()
        refs = R.oracle_step(live, q, kn, vn)
        for i in range(layers):
            g = wl.torch_to_bits(graph_r.out[i][:n])
            assert np.array_equal(g, wl.torch_to_bits(eager_r.out[i][:n])), f"step {s}"
            assert_attn_close(g, refs[i], f"step {s} layer {i}")
    real = np.arange(R.num_slots) != R.dummy_slot
    for (kg, vg), (ke, ve), (kh, vh) in zip(pools_g, pools_e, R.pools):
        assert np.array_equal(wl.torch_to_bits(kg)[real], kh[real])
        assert np.array_equal(wl.torch_to_bits(ke)[real], kh[real])
        assert np.array_equal(wl.torch_to_bits(vg)[real], vh[real])
    assert msg.msg_read_device_status(graph_r.ws)[0] == msg.MSG_OK


def test_mixed_call_captured_in_a_graph():
    """A mixed batch's step (plan, store_kv, then the decode and the extend
    kernels) captured in a CUDA graph and replayed gives the oracle's result."""
    from _harness import GpuBatch, oracle_small
    rng = np.random.default_rng(33)
    cached = np.r_[rng.integers(100, 2000, size=20), rng.integers(0, 300, size=3)]
    ext = np.r_[np.ones(20, np.int64), rng.integers(100, 300, size=3)]
    spec = wl.make_batch("graph_mixed", 33, cached, ext, 1, num_pages=int((cached + ext).sum()) + 9)
    host = wl.host_tensors(spec)
    gb = GpuBatch(spec)
    q = wl.bits_to_torch(host["q"], "cuda")
    kn, vn = wl.bits_to_torch(host["k_new"], "cuda"), wl.bits_to_torch(host["v_new"], "cuda")
    kp, vp = wl.bits_to_torch(host["k_pool"], "cuda"), wl.bits_to_torch(host["v_pool"], "cuda")
    out = torch.empty_like(q)

    def step():
        loc = gb.plan()
        msg.msg_store_kv(kn, vn, kp, vp, loc)
        gb.attention(q, kp, vp, out=out, flags=msg.MSG_ATTN_REUSE_PLAN)

    step()                                           # warm-up (sets kernel attributes)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    out.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert gb.status()[0] == msg.MSG_OK
    assert_attn_close(wl.torch_to_bits(out), oracle_small(spec, host)["out"], "graph mixed")

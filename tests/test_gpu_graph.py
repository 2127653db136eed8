"""CUDA-graph replay of the decode step (plan, store_kv, paged attention).

The whole path runs from device-side metadata with no host synchronisation and
fixed launch shapes, so one captured graph serves every later step of a
fixed-size (padded) decode batch: the caller updates cached_len, the page
table, q and the new k/v in place and replays.  Padding requests point at the
dummy slot, as in a CUDA-graph-padded engine batch ("Engine 与采样器",
初始化的顺序: the extra dummy page and the dummy row).  Replays must match eager
execution of the same step bit for bit."""
import numpy as np
import pytest
import torch

import paged_kv_gqa_store_gb300 as msg
from paged_kv_gqa_store_gb300 import workload as wl

pytestmark = pytest.mark.gpu


def _decode_batch(seed, n_real, n_pad, ctx_lo, ctx_hi, steps_ahead):
    rng = np.random.default_rng(seed)
    ctx = rng.integers(ctx_lo, ctx_hi, size=n_real)
    # room for `steps_ahead` more decode tokens per request
    spec = wl.make_batch("graph", seed, cached_len=ctx - 1 + steps_ahead,
                         extend_len=np.ones(n_real, np.int32), page_size=1,
                         num_pages=int((ctx + steps_ahead).sum()) + 64)
    dummy = spec.num_slots
    width = spec.page_table.shape[1]
    pt = np.zeros((n_real + 1, width), np.int32)
    pt[:n_real] = spec.page_table
    pt[n_real, :] = dummy
    cached = np.r_[ctx - 1, np.zeros(n_pad, np.int64)].astype(np.int32)
    ext = np.ones(n_real + n_pad, np.int32)
    rows = np.r_[np.arange(n_real), np.full(n_pad, n_real)].astype(np.int32)
    return pt, cached, ext, rows, spec.num_slots + 1


def _run_step(pt, cached, ext, rows, qo, loc, ws, q, kn, vn, kp, vp, out):
    msg.msg_plan(pt, cached, ext, q.shape[0], kp.shape[0], ws, req_rows=rows, qo_indptr_out=qo,
                 out_loc_out=loc)
    msg.msg_store_kv(kn, vn, kp, vp, loc)
    msg.msg_paged_attention(q, kp, vp, pt, cached, ext, qo, out, ws, page_size=1, req_rows=rows,
                            max_kv_len=0, flags=msg.MSG_ATTN_REUSE_PLAN | msg.MSG_ATTN_DECODE_ONLY)


def test_graph_replay_matches_eager_over_steps():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    msg.load_library()
    dev = "cuda"
    n_real, n_pad, steps = 6, 2, 3
    pt_np, cached_np, ext_np, rows_np, num_slots = _decode_batch(7, n_real, n_pad, 200, 3000, steps)
    B = n_real + n_pad
    rng = np.random.default_rng(8)
    pool_k = wl.random_bf16(rng, (num_slots, 8, 128))
    pool_v = wl.random_bf16(rng, (num_slots, 8, 128))
    step_in = [{n: wl.random_bf16(rng, shape) for n, shape in
                (("q", (B, 16, 128)), ("k", (B, 8, 128)), ("v", (B, 8, 128)))}
               for _ in range(steps)]

    def tensors():
        return {
            "pt": torch.from_numpy(pt_np).to(dev), "cached": torch.from_numpy(cached_np).to(dev),
            "ext": torch.from_numpy(ext_np).to(dev), "rows": torch.from_numpy(rows_np).to(dev),
            "qo": torch.zeros(B + 1, dtype=torch.int32, device=dev),
            "loc": torch.zeros(B, dtype=torch.int64, device=dev),
            "ws": torch.zeros(msg.msg_workspace_size(B, B), dtype=torch.uint8, device=dev),
            "q": torch.empty(B, 16, 128, dtype=torch.bfloat16, device=dev),
            "kn": torch.empty(B, 8, 128, dtype=torch.bfloat16, device=dev),
            "vn": torch.empty(B, 8, 128, dtype=torch.bfloat16, device=dev),
            "kp": wl.bits_to_torch(pool_k, dev), "vp": wl.bits_to_torch(pool_v, dev),
            "out": torch.empty(B, 16, 128, dtype=torch.bfloat16, device=dev)}

    def load(t, s):
        t["q"].copy_(wl.bits_to_torch(step_in[s]["q"], dev))
        t["kn"].copy_(wl.bits_to_torch(step_in[s]["k"], dev))
        t["vn"].copy_(wl.bits_to_torch(step_in[s]["v"], dev))
        # Req.complete_one on real requests: cached_len advances by one per step
        c = cached_np.copy()
        c[:n_real] += s
        t["cached"].copy_(torch.from_numpy(c).to(dev))

    def args(t):
        return (t["pt"], t["cached"], t["ext"], t["rows"], t["qo"], t["loc"], t["ws"], t["q"],
                t["kn"], t["vn"], t["kp"], t["vp"], t["out"])

    eager, graph_t = tensors(), tensors()
    # warm-up (first calls set kernel attributes), then capture on a side stream
    load(graph_t, 0)
    warm = tensors()
    load(warm, 0)
    _run_step(*args(warm))
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _run_step(*args(graph_t))
    for s in range(steps):
        load(eager, s)
        _run_step(*args(eager))
        load(graph_t, s)
        g.replay()
        torch.cuda.synchronize()
        e = wl.torch_to_bits(eager["out"])[:n_real]
        r = wl.torch_to_bits(graph_t["out"])[:n_real]
        assert np.array_equal(e, r), f"step {s}"
        assert np.isfinite(wl.bf16_bits_to_f64(r)).all()
    real = np.arange(num_slots) != num_slots - 1
    assert np.array_equal(wl.torch_to_bits(eager["kp"])[real], wl.torch_to_bits(graph_t["kp"])[real])
    assert msg.msg_read_device_status(graph_t["ws"])[0] == msg.MSG_OK

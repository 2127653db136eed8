"""msg_paged_attention_noalloc: the attention entry point for callers that cannot
allocate device memory (its scratch is a fixed array inside the library).

Checked through the C ABI against msg_paged_attention with a caller workspace
on two calls in a row on different batches (the shared array keeps the
previous call's contents).  Both run the same kernels on the same plan, so the
outputs must be identical bit for bit, and within the attention tolerance of
the other tests.  This file is collected last on purpose."""
import numpy as np
import pytest
import torch

import paged_kv_gqa_store_gb300 as msg
from paged_kv_gqa_store_gb300 import workload as wl

from _harness import GpuBatch, MAX_ABS, REL_L2

pytestmark = pytest.mark.gpu


def _batch(seed, n_dec, n_ext, page_size):
    rng = np.random.default_rng(seed)
    cached = np.r_[rng.integers(0, 3000, size=n_dec), rng.integers(0, 500, size=n_ext)]
    ext = np.r_[np.ones(n_dec, np.int64), rng.integers(2, 300, size=n_ext)]
    need = int(((cached + ext + page_size - 1) // page_size).sum()) + 5
    return wl.make_batch(f"noalloc{seed}", seed, cached, ext, page_size, num_pages=need,
                         shuffle_rows=True, extra_rows=2)


def _compare(a, b):
    fa = wl.bf16_bits_to_f64(wl.torch_to_bits(a))
    fb = wl.bf16_bits_to_f64(wl.torch_to_bits(b))
    assert np.isfinite(fa).all()
    max_abs = np.abs(fa - fb).max()
    rel = np.linalg.norm(fa - fb) / np.linalg.norm(fb)
    assert max_abs <= MAX_ABS and rel <= REL_L2, (max_abs, rel)


def test_noalloc_matches_workspace_entry_on_two_calls_in_a_row():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    msg.load_library()
    for seed, n_dec, n_ext, P in ((71, 40, 3, 16), (72, 9, 2, 1)):
        spec = _batch(seed, n_dec, n_ext, P)
        host = wl.host_tensors(spec)
        gb = GpuBatch(spec)
        q = wl.bits_to_torch(host["q"], "cuda")
        kp = wl.bits_to_torch(host["k_pool"], "cuda")
        vp = wl.bits_to_torch(host["v_pool"], "cuda")
        loc = gb.plan()
        msg.msg_store_kv(wl.bits_to_torch(host["k_new"], "cuda"),
                         wl.bits_to_torch(host["v_new"], "cuda"), kp, vp, loc)
        ref = gb.attention(q, kp, vp)
        out = torch.full_like(q, float("nan"))
        status = torch.zeros(4, dtype=torch.int32, device="cuda")
        msg.msg_paged_attention_noalloc(q, kp, vp, gb.page_table, gb.cached, gb.extend, gb.qo,
                                        out, page_size=P, req_rows=gb.rows,
                                        max_kv_len=spec.max_kv_len, dev_status=status)
        torch.cuda.synchronize()
        assert msg.msg_read_device_status(status)[0] == msg.MSG_OK
        assert gb.status()[0] == msg.MSG_OK
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
        _compare(out, ref)


def test_noalloc_reuse_plan_needs_a_plan_of_the_same_batch_size():
    """MSG_ATTN_REUSE_PLAN reads the plan a previous call left in the shared
    array, whose place depends on the batch size: a call of another size is
    rejected before anything is enqueued, one of the same size reuses it."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    msg.load_library()
    spec = _batch(73, 11, 2, 1)
    host = wl.host_tensors(spec)
    gb = GpuBatch(spec)
    q = wl.bits_to_torch(host["q"], "cuda")
    kp = wl.bits_to_torch(host["k_pool"], "cuda")
    vp = wl.bits_to_torch(host["v_pool"], "cuda")
    loc = gb.plan()
    msg.msg_store_kv(wl.bits_to_torch(host["k_new"], "cuda"),
                     wl.bits_to_torch(host["v_new"], "cuda"), kp, vp, loc)
    ref = gb.attention(q, kp, vp)
    out = torch.full_like(q, float("nan"))
    args = (q, kp, vp, gb.page_table, gb.cached, gb.extend, gb.qo, out)
    kw = dict(page_size=1, req_rows=gb.rows, max_kv_len=spec.max_kv_len)
    msg.msg_paged_attention_noalloc(*args, **kw)                  # builds the plan
    out2 = torch.full_like(q, float("nan"))
    msg.msg_paged_attention_noalloc(q, kp, vp, gb.page_table, gb.cached, gb.extend, gb.qo, out2,
                                    flags=msg.MSG_ATTN_REUSE_PLAN, **kw)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert torch.equal(out2.view(torch.int16), ref.view(torch.int16))
    # a batch of another size may not reuse that plan
    sub = slice(0, spec.num_reqs - 1)
    with pytest.raises(msg.MsgError) as e:
        msg.msg_paged_attention_noalloc(q, kp, vp, gb.page_table, gb.cached[sub], gb.extend[sub],
                                        gb.qo[:spec.num_reqs], out2,
                                        flags=msg.MSG_ATTN_REUSE_PLAN, **kw)
    assert e.value.status == msg.MSG_ERR_INVALID_ARG


def test_noalloc_rejects_batches_beyond_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = msg.load_library()
    need = msg.msg_workspace_size(100000, 1 << 20)
    assert need > (9 << 20)
    one = torch.zeros(16, dtype=torch.int32, device="cuda")
    x = torch.zeros(8, 16, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(msg.MsgError) as e:
        msg.msg_paged_attention_noalloc(x, x[:, :8], x[:, :8], one.view(1, 16),
                                        torch.zeros(100000, dtype=torch.int32, device="cuda"),
                                        torch.zeros(100000, dtype=torch.int32, device="cuda"),
                                        one, x)
    assert e.value.status == msg.MSG_ERR_WORKSPACE
    assert lib is not None

"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI,
run the oracle on the same inputs, compare."""
from __future__ import annotations

import numpy as np
import torch

import oracle
import paged_kv_gqa_store_gb300 as msg
from paged_kv_gqa_store_gb300 import workload as wl

# Attention tolerance against the fp64 oracle (bf16 inputs, fp32 accumulation).
MAX_ABS = 1e-2
REL_L2 = 2e-3


def i32(a, dev="cuda"):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)


class GpuBatch:
    """Device copies of a batch's metadata plus a workspace sized for it."""

    def __init__(self, spec: wl.BatchSpec, dev="cuda", ws_extra=0):
        self.spec = spec
        self.page_table = i32(spec.page_table, dev)
        self.cached = i32(spec.cached_len, dev)
        self.extend = i32(spec.extend_len, dev)
        self.rows = i32(spec.req_rows, dev)
        T = spec.total_q
        self.qo = torch.zeros(spec.num_reqs + 1, dtype=torch.int32, device=dev)
        self.out_loc = torch.zeros(max(T, 1), dtype=torch.int64, device=dev)[:T]
        self.positions = torch.zeros(max(T, 1), dtype=torch.int32, device=dev)[:T]
        nbytes = msg.msg_workspace_size(max(spec.num_reqs, 1), max(T, 1), spec.num_qo_heads,
                                        spec.head_dim) + ws_extra
        self.ws = torch.zeros(nbytes, dtype=torch.uint8, device=dev)

    def plan(self, out_loc_int64=True):
        if out_loc_int64:
            loc = self.out_loc
        else:
            loc = torch.zeros(max(self.spec.total_q, 1), dtype=torch.int32,
                              device=self.page_table.device)[:self.spec.total_q]
            self.out_loc32 = loc
        msg.msg_plan(self.page_table, self.cached, self.extend, self.spec.total_q,
                     self.spec.num_slots, self.ws, req_rows=self.rows,
                     qo_indptr_out=self.qo, out_loc_out=loc, positions_out=self.positions)
        return loc

    def attention(self, q, k_pool, v_pool, out=None, flags=0, page_size=None, max_kv_len=None):
        if out is None:
            out = torch.empty(q.shape, dtype=torch.bfloat16, device=q.device)
        msg.msg_paged_attention(
            q, k_pool, v_pool, self.page_table, self.cached, self.extend, self.qo, out, self.ws,
            page_size=self.spec.page_size if page_size is None else page_size,
            req_rows=self.rows,
            max_kv_len=self.spec.max_kv_len if max_kv_len is None else max_kv_len, flags=flags)
        return out

    def status(self):
        return msg.msg_read_device_status(self.ws)


def run_small(spec: wl.BatchSpec, host: dict, flags=0, out_loc_int64=True, q_stride_pad=0):
    """Full CUDA path on host-generated inputs: plan, store_kv, attention."""
    dev = "cuda"
    gb = GpuBatch(spec, dev)
    if q_stride_pad:
        T, H, D = host["q"].shape
        qbuf = torch.zeros(T, H + q_stride_pad, D, dtype=torch.bfloat16, device=dev)
        qbuf[:, :H] = wl.bits_to_torch(host["q"], dev)
        q = qbuf[:, :H]
    else:
        q = wl.bits_to_torch(host["q"], dev)
    k_new = wl.bits_to_torch(host["k_new"], dev)
    v_new = wl.bits_to_torch(host["v_new"], dev)
    k_pool = wl.bits_to_torch(host["k_pool"], dev)
    v_pool = wl.bits_to_torch(host["v_pool"], dev)
    loc = gb.plan(out_loc_int64)
    msg.msg_store_kv(k_new, v_new, k_pool, v_pool, loc, dev_status=gb.ws)
    out = gb.attention(q, k_pool, v_pool, flags=flags | msg.MSG_ATTN_REUSE_PLAN)
    torch.cuda.synchronize()
    st, info = gb.status()
    return {"qo": gb.qo.cpu().numpy(), "out_loc": loc.cpu().numpy().astype(np.int64),
            "positions": gb.positions.cpu().numpy(), "out": wl.torch_to_bits(out),
            "k_pool": wl.torch_to_bits(k_pool), "v_pool": wl.torch_to_bits(v_pool),
            "status": st, "status_info": info}


def oracle_small(spec: wl.BatchSpec, host: dict, rows=None):
    meta = oracle.metadata(spec.page_table, spec.cached_len, spec.extend_len, spec.req_rows)
    kp, vp = host["k_pool"].copy(), host["v_pool"].copy()
    oracle.store_kv(host["k_new"], host["v_new"], meta["out_loc"], kp, vp)
    out = oracle.paged_attention(host["q"], kp, vp, spec.page_table, spec.cached_len,
                                 meta["qo_indptr"], spec.num_qo_heads, spec.num_kv_heads,
                                 spec.head_dim, req_rows=spec.req_rows, rows=rows)
    return {**meta, "k_pool": kp, "v_pool": vp, "out": out}


def attn_errors(gpu_bits: np.ndarray, ref: np.ndarray):
    got = wl.bf16_bits_to_f64(gpu_bits).reshape(ref.shape)
    diff = got - ref
    max_abs = float(np.abs(diff).max()) if diff.size else 0.0
    rel = float(np.linalg.norm(diff) / max(np.linalg.norm(ref), 1e-300)) if diff.size else 0.0
    return max_abs, rel


def assert_attn_close(gpu_bits, ref, what=""):
    assert np.isfinite(wl.bf16_bits_to_f64(gpu_bits)).all(), f"{what}: non-finite output"
    max_abs, rel = attn_errors(gpu_bits, ref)
    assert max_abs <= MAX_ABS and rel <= REL_L2, f"{what}: max_abs {max_abs:.3e} rel_l2 {rel:.3e}"
    return max_abs, rel


# ------------------------------------------------------------ full-size sampling
def sampled_oracle(spec: wl.BatchSpec, pools_before: tuple, q, k_new, v_new, reqs,
                   rows_per_req=None, rng=None):
    """Oracle for a subset of requests of a large batch.

    pools_before: (k_pool, v_pool) device tensors holding the state BEFORE store_kv
    (the cached prefixes); call this before the CUDA path runs.  The chosen
    requests' pages are relabelled into a compact host pool; the oracle then
    stores the new K/V and attends.  Returns (gpu_rows, ref) where gpu_rows are
    the global query rows to compare."""
    sub, src_slots = wl.compact_requests(spec, reqs)
    idx = torch.from_numpy(src_slots).to(q.device)
    kp = wl.torch_to_bits(pools_before[0].index_select(0, idx))
    vp = wl.torch_to_bits(pools_before[1].index_select(0, idx))
    # global rows of the chosen requests' new tokens
    qo_full = np.concatenate([[0], np.cumsum(spec.extend_len)]).astype(np.int64)
    tok = np.concatenate([np.arange(qo_full[r], qo_full[r + 1]) for r in reqs])
    tok_t = torch.from_numpy(tok).to(q.device)
    q_sub = wl.torch_to_bits(q.index_select(0, tok_t))
    kn = wl.torch_to_bits(k_new.index_select(0, tok_t))
    vn = wl.torch_to_bits(v_new.index_select(0, tok_t))
    meta = oracle.metadata(sub.page_table, sub.cached_len, sub.extend_len, sub.req_rows)
    oracle.store_kv(kn, vn, meta["out_loc"], kp, vp)
    sub_rows = None
    if rows_per_req is not None:
        rng = rng or np.random.default_rng(0)
        pick = []
        for n in range(sub.num_reqs):
            lo, hi = int(meta["qo_indptr"][n]), int(meta["qo_indptr"][n + 1])
            e = hi - lo
            cand = np.unique(np.concatenate([
                [0, e - 1, min(63, e - 1), min(64, e - 1), min(127, e - 1), min(128, e - 1)],
                rng.integers(0, e, size=min(rows_per_req, e))]))
            pick.append(lo + cand)
        sub_rows = np.concatenate(pick).astype(np.int64)
    ref = oracle.paged_attention(q_sub, kp, vp, sub.page_table, sub.cached_len, meta["qo_indptr"],
                                 sub.num_qo_heads, sub.num_kv_heads, sub.head_dim,
                                 req_rows=sub.req_rows, rows=sub_rows)
    gpu_rows = tok if sub_rows is None else tok[sub_rows]
    return gpu_rows, ref

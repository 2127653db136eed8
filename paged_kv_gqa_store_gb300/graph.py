"""CUDA-graph replay of a whole decode step, over a ladder of padded batch sizes.

A decode step of the attention path is one plan launch followed, per layer, by
one fused store_kv + decode-attention launch (``msg_paged_attention_store``).
Every launch reads its batch from device memory (the plan is built on the
device, launch shapes do not depend on the lengths), so one captured graph
serves every later step of a batch of the same padded size: the caller updates
the metadata and the step's q / k / v rows in place and replays.

This follows the engine's graph runner ("Mini-SGLang 源码解析（四）" 10.2-10.7;
"Mini-SGLang 完整剖析" 4.6.6): graphs are captured for the batch sizes
[1, 2, 4] and every multiple of 8 up to the largest, from the largest to the
smallest into one memory pool, each after a warm-up run; a live batch is padded
to the smallest captured size that holds it, the padding requests being dummy
requests whose page-table row points every token at the dummy slot ("Engine 与
采样器", 初始化的顺序: the extra dummy page).

The runner owns fixed-address device buffers sized for the largest batch:
``q[layer]``, ``k_new[layer]``, ``v_new[layer]`` (the step's inputs, which the
model writes before ``replay``) and ``out[layer]`` (the attention outputs),
plus the metadata.  Row r of each is request r of the live batch; rows past
the live size belong to the padding and their outputs mean nothing.
"""
from __future__ import annotations

import numpy as np

from . import MSG_ATTN_DECODE_ONLY, MSG_ATTN_REUSE_PLAN, msg_paged_attention_store, msg_plan
from . import msg_workspace_size


def graph_batch_sizes(max_bs: int) -> list[int]:
    """The capture ladder: 1, 2, 4, then the multiples of 8 up to max_bs (and
    max_bs itself when it is not one of them)."""
    if max_bs < 1:
        raise ValueError("max_bs must be >= 1")
    sizes = [b for b in (1, 2, 4) if b <= max_bs] + list(range(8, max_bs + 1, 8))
    if sizes[-1] != max_bs:
        sizes.append(max_bs)
    return sizes


def padded_size(sizes: list[int], n: int) -> int:
    """The smallest captured size that holds a live batch of n requests."""
    for b in sorted(sizes):
        if b >= n:
            return b
    raise ValueError(f"batch of {n} exceeds the largest captured size {max(sizes)}")


class DecodeGraphRunner:
    """Captured decode steps for every size of the ladder.

    pools       list of (k_pool, v_pool) per layer, bf16 [slots, Hkv, D].
    page_table  int32 [rows, width] device tensor: the global token table; row
                ``dummy_row`` maps every token to the dummy slot.
    """

    def __init__(self, pools, page_table, dummy_row: int, max_bs: int, page_size: int = 1,
                 num_qo_heads: int = 16, head_dim: int = 128, max_kv_len: int = 0):
        import torch
        self.pools = list(pools)
        self.page_table = page_table
        self.dummy_row = int(dummy_row)
        self.sizes = graph_batch_sizes(max_bs)
        self.max_bs = max(self.sizes)
        self.page_size = int(page_size)
        self.max_kv_len = int(max_kv_len)
        dev = page_table.device
        hkv = int(self.pools[0][0].shape[1])
        B = self.max_bs
        self.num_slots = int(self.pools[0][0].shape[0])
        # per-step metadata: cached_len and page-table rows, one H2D copy a step
        # from pinned staging (the staging is rewritten only after the previous
        # step's copy has run)
        self._host_meta = torch.zeros(2, B, dtype=torch.int32).pin_memory()
        self._meta = torch.zeros(2, B, dtype=torch.int32, device=dev)
        self._copied = torch.cuda.Event()
        self._copied.record()
        self.cached, self.rows = self._meta[0], self._meta[1]
        self.extend = torch.ones(B, dtype=torch.int32, device=dev)
        self.qo = torch.zeros(B + 1, dtype=torch.int32, device=dev)
        self.out_loc = torch.zeros(B, dtype=torch.int64, device=dev)
        self.ws = torch.zeros(msg_workspace_size(B, B, num_qo_heads, head_dim),
                              dtype=torch.uint8, device=dev)
        L = len(self.pools)
        bf = torch.bfloat16
        self.q = [torch.zeros(B, num_qo_heads, head_dim, dtype=bf, device=dev) for _ in range(L)]
        self.k_new = [torch.zeros(B, hkv, head_dim, dtype=bf, device=dev) for _ in range(L)]
        self.v_new = [torch.zeros(B, hkv, head_dim, dtype=bf, device=dev) for _ in range(L)]
        self.out = [torch.zeros(B, num_qo_heads, head_dim, dtype=bf, device=dev)
                    for _ in range(L)]
        self.graphs = {}

    # ---------------------------------------------------------------- one step
    def _step(self, bs: int) -> None:
        """The decode step on the first bs rows of the buffers (eager)."""
        cached, ext, rows = self.cached[:bs], self.extend[:bs], self.rows[:bs]
        qo, loc = self.qo[:bs + 1], self.out_loc[:bs]
        msg_plan(self.page_table, cached, ext, bs, self.num_slots, self.ws, req_rows=rows,
                 qo_indptr_out=qo, out_loc_out=loc)
        flags = MSG_ATTN_REUSE_PLAN | MSG_ATTN_DECODE_ONLY
        for i, (kp, vp) in enumerate(self.pools):
            msg_paged_attention_store(self.q[i][:bs], self.k_new[i][:bs], self.v_new[i][:bs],
                                      kp, vp, self.page_table, cached, ext, qo, self.out[i][:bs],
                                      self.ws, page_size=self.page_size, req_rows=rows,
                                      max_kv_len=self.max_kv_len, flags=flags)

    def capture(self) -> None:
        """Capture one graph per ladder size, largest first, sharing one pool.
        Each capture follows a warm-up run of the same size on the dummy
        batch (every request on the dummy row), as the engine does."""
        import torch
        pool = None
        stream = torch.cuda.Stream(device=self.page_table.device)
        for bs in sorted(self.sizes, reverse=True):
            self._set_meta(0, np.zeros(0, np.int32), np.zeros(0, np.int32), bs)
            stream.wait_stream(torch.cuda.current_stream())
            with torch.cuda.stream(stream):
                self._step(bs)                       # warm-up
            torch.cuda.current_stream().wait_stream(stream)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, pool=pool, stream=stream):
                self._step(bs)
            if pool is None:
                pool = g.pool()
            self.graphs[bs] = g
        torch.cuda.synchronize()

    def _set_meta(self, n: int, cached_len, req_rows, bs: int) -> None:
        h = self._host_meta
        self._copied.synchronize()                   # the last step's copy has read h
        h[0, :n] = torch_from(cached_len[:n])
        h[1, :n] = torch_from(req_rows[:n])
        h[0, n:bs] = 0                               # a dummy request: 1 token on the dummy row
        h[1, n:bs] = self.dummy_row
        self._meta.copy_(h, non_blocking=True)
        self._copied.record()

    def replay(self, cached_len, req_rows) -> int:
        """One decode step of a live batch of len(cached_len) requests: its
        cached lengths (host int arrays; device_len = cached_len + 1) and page
        table rows.  The step's q / k_new / v_new rows must already be in the
        first rows of the buffers.  Pads to the next captured size, replays,
        and returns that size; outputs land in out[layer][:live]."""
        n = len(cached_len)
        bs = padded_size(self.sizes, n)
        if not self.graphs:
            raise RuntimeError("capture() first")
        self._set_meta(n, np.asarray(cached_len, np.int32), np.asarray(req_rows, np.int32), bs)
        self.graphs[bs].replay()
        return bs

    def eager(self, cached_len, req_rows) -> int:
        """The same step without the graph (the reference for replay timing)."""
        n = len(cached_len)
        bs = padded_size(self.sizes, n)
        self._set_meta(n, np.asarray(cached_len, np.int32), np.asarray(req_rows, np.int32), bs)
        self._step(bs)
        return bs


def torch_from(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32))

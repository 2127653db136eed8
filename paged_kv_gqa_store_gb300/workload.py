"""Seeded synthetic inputs for the paged KV store and GQA paged attention.

This module only generates inputs: request lengths, page assignments (the
token-granular page table) and iid N(0,1) bf16 values.  It computes none of the
method's arithmetic (no out_loc, positions, qo_indptr, scores or softmax), so the
CUDA library and the CPU oracle can both consume what it produces without
sharing code.

Shapes follow the Qwen3 attention of "第 0 步：一个能跑的最小推理引擎": 16 query
heads, 8 KV heads, head_dim 128, bf16.  The page table is token-granular, as
"核心数据结构：Req、Batch、Context" (Context) states: entry [row, j] is the pool
slot of token j of that request.  With page_size P > 1, each page is P
consecutive, P-aligned slots, so entry [row, j] = P * page(j // P) + j % P.

Unreferenced pool rows are filled with a NaN canary so that a stray read shows up
in the output and a stray write shows up in the pool.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

HQ = 16
HKV = 8
HEAD_DIM = 128
CANARY_BF16 = 0xFFC1          # a quiet NaN in bf16, never produced by N(0,1)


def align_up(x: int, a: int) -> int:
    return (x + a - 1) // a * a


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (round to nearest, ties to even); return uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_bits_to_f64(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(
        np.float32).astype(np.float64)


def random_bf16(rng: np.random.Generator, shape) -> np.ndarray:
    return f32_to_bf16_bits(rng.standard_normal(size=shape, dtype=np.float32))


@dataclass
class BatchSpec:
    """One batch: per-request lengths and the page table, plus pool geometry."""
    name: str
    cached_len: np.ndarray            # int32 [num_reqs]
    extend_len: np.ndarray            # int32 [num_reqs]
    req_rows: np.ndarray              # int32 [num_reqs], row in page_table
    page_table: np.ndarray            # int32 [rows, width], token-granular slots
    page_size: int
    num_slots: int                    # pool rows (pages * page_size)
    seed: int
    num_layers: int = 1
    num_qo_heads: int = HQ
    num_kv_heads: int = HKV
    head_dim: int = HEAD_DIM
    notes: dict = field(default_factory=dict)

    @property
    def num_reqs(self) -> int:
        return int(self.cached_len.shape[0])

    @property
    def total_q(self) -> int:
        return int(self.extend_len.sum())

    @property
    def device_len(self) -> np.ndarray:
        return self.cached_len.astype(np.int64) + self.extend_len

    @property
    def max_kv_len(self) -> int:
        return int(self.device_len.max()) if self.num_reqs else 0

    @property
    def row_elems(self) -> int:
        return self.num_kv_heads * self.head_dim


def assign_pages(rng: np.random.Generator, device_lens, page_size: int,
                 num_pages: int, num_rows: int | None = None,
                 row_of=None) -> np.ndarray:
    """Token-granular page table: each request gets ceil(len / P) distinct pages
    drawn without replacement from [0, num_pages), in random order."""
    device_lens = np.asarray(device_lens, dtype=np.int64)
    n = device_lens.shape[0]
    pages_needed = (device_lens + page_size - 1) // page_size
    total_pages = int(pages_needed.sum())
    if total_pages > num_pages:
        raise ValueError(f"pool of {num_pages} pages cannot hold {total_pages}")
    chosen = rng.choice(num_pages, size=total_pages, replace=False).astype(np.int64)
    width = align_up(max(int(device_lens.max()) if n else 1, 1), 32)
    rows = num_rows if num_rows is not None else n
    table = np.zeros((rows, width), dtype=np.int32)
    off = 0
    for r in range(n):
        L, npg = int(device_lens[r]), int(pages_needed[r])
        pages = chosen[off:off + npg]
        off += npg
        j = np.arange(L, dtype=np.int64)
        row = r if row_of is None else int(row_of[r])
        table[row, :L] = (pages[j // page_size] * page_size + j % page_size).astype(np.int32)
    return table


def make_batch(name: str, seed: int, cached_len, extend_len, page_size: int,
               num_pages: int, num_layers: int = 1, shuffle_rows: bool = False,
               extra_rows: int = 0, **kw) -> BatchSpec:
    rng = np.random.default_rng(seed)
    cached_len = np.asarray(cached_len, dtype=np.int32)
    extend_len = np.asarray(extend_len, dtype=np.int32)
    n = cached_len.shape[0]
    rows = np.arange(n, dtype=np.int32)
    if shuffle_rows:
        rows = rng.permutation(n + extra_rows)[:n].astype(np.int32)
    table = assign_pages(rng, cached_len.astype(np.int64) + extend_len, page_size,
                         num_pages, num_rows=n + extra_rows, row_of=rows)
    return BatchSpec(name=name, cached_len=cached_len, extend_len=extend_len,
                     req_rows=rows, page_table=table, page_size=page_size,
                     num_slots=num_pages * page_size, seed=seed,
                     num_layers=num_layers, **kw)


# ---------------------------------------------------------------- the 5 configs
# A decode request's "context length" is read as its device_len (the KV length
# after this step, including the new token): cached_len = context - 1, extend 1.

def config_tiny_mixed(seed: int = 1001) -> BatchSpec:
    """1 extend (prompt 6, cached 2 -> extend 4) + decode at context 5, 17, 64;
    page_size 1, pool of 4096 pages, slots a seeded random permutation."""
    return make_batch("tiny_mixed", seed, cached_len=[2, 4, 16, 63],
                      extend_len=[4, 1, 1, 1], page_size=1, num_pages=4096)


def config_decode_28_layers(seed: int = 1002) -> BatchSpec:
    """64 decode requests, context U[512, 4096], page_size 1, 28 layer pools of
    300k pages each, one shared page table."""
    rng = np.random.default_rng(seed)
    ctx = rng.integers(512, 4096 + 1, size=64)
    return make_batch("decode_64x28", seed + 1, cached_len=ctx - 1,
                      extend_len=np.ones(64, np.int32), page_size=1,
                      num_pages=300_000, num_layers=28)


def config_large_decode(num_pages: int, seed: int = 1003) -> BatchSpec:
    """256 decode requests, context U[1024, 8192], page_size 16, pages drawn at
    random from a pool of num_pages pages (sized by the caller to 90% of free
    HBM for one layer)."""
    rng = np.random.default_rng(seed)
    ctx = rng.integers(1024, 8192 + 1, size=256)
    return make_batch("decode_256_p16", seed + 1, cached_len=ctx - 1,
                      extend_len=np.ones(256, np.int32), page_size=16,
                      num_pages=num_pages)


def config_extend(seed: int = 1004, num_pages: int = 65536) -> BatchSpec:
    """8 extend requests, cached U[0, 2048], extend U[512, 4096], page_size 1,
    random slot permutation over a 65536-slot pool."""
    rng = np.random.default_rng(seed)
    cached = rng.integers(0, 2048 + 1, size=8)
    ext = rng.integers(512, 4096 + 1, size=8)
    return make_batch("extend_8", seed + 1, cached_len=cached, extend_len=ext,
                      page_size=1, num_pages=num_pages)


def config_long_mixed(seed: int = 1005, num_pages: int = 32768) -> BatchSpec:
    """32 decode requests at context 32768 + 2 extend requests of 2048 tokens
    over 16384 cached; page_size 64, pages randomly permuted."""
    cached = [32767] * 32 + [16384] * 2
    ext = [1] * 32 + [2048] * 2
    return make_batch("long_mixed_p64", seed, cached_len=cached, extend_len=ext,
                      page_size=64, num_pages=num_pages)


def prefix_slots(spec: BatchSpec) -> np.ndarray:
    """Pool slots holding each request's cached prefix (positions < cached_len)."""
    out = []
    for r in range(spec.num_reqs):
        c = int(spec.cached_len[r])
        out.append(spec.page_table[spec.req_rows[r], :c].astype(np.int64))
    return np.concatenate(out) if out else np.zeros(0, np.int64)


def host_tensors(spec: BatchSpec, layer: int = 0) -> dict:
    """Host-side inputs for one layer (small configs): q, new k/v and both
    pools (canary everywhere except the cached prefixes), all bf16 bits."""
    rng = np.random.default_rng([spec.seed, layer])
    T, H, Hk, D = spec.total_q, spec.num_qo_heads, spec.num_kv_heads, spec.head_dim
    q = random_bf16(rng, (T, H, D))
    k_new = random_bf16(rng, (T, Hk, D))
    v_new = random_bf16(rng, (T, Hk, D))
    k_pool = np.full((spec.num_slots, Hk, D), CANARY_BF16, np.uint16)
    v_pool = np.full((spec.num_slots, Hk, D), CANARY_BF16, np.uint16)
    slots = prefix_slots(spec)
    k_pool[slots] = random_bf16(rng, (slots.shape[0], Hk, D))
    v_pool[slots] = random_bf16(rng, (slots.shape[0], Hk, D))
    return {"q": q, "k_new": k_new, "v_new": v_new, "k_pool": k_pool, "v_pool": v_pool}


# ---------------------------------------------------------------- device side
def bits_to_torch(bits: np.ndarray, device=None):
    """uint16 bf16 bits -> torch.bfloat16 tensor (optionally moved to device)."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.to(device) if device is not None else t


def torch_to_bits(t) -> np.ndarray:
    """torch.bfloat16 tensor -> uint16 numpy bits (copied to host)."""
    import torch
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


def device_tensors(spec: BatchSpec, layer: int = 0, device="cuda", pools=True,
                   chunk_rows: int = 1 << 16, canary: bool = True) -> dict:
    """Inputs for one layer generated directly on the GPU (large configs): q and
    the new k/v as N(0,1) bf16, and (if pools) K/V pools filled with the canary
    except the cached prefixes, which get N(0,1) bf16 rows.  Values come from
    torch's CUDA generator seeded by (seed, layer); nothing of the method runs.
    With canary=False the unused slots are left uninitialised (timing only: no
    slot outside the prefixes and the new tokens is ever read)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(spec.seed) * 1009 + layer)
    T, H, Hk, D = spec.total_q, spec.num_qo_heads, spec.num_kv_heads, spec.head_dim

    def randn(*shape):
        return torch.randn(*shape, generator=g, device=device, dtype=torch.float32).to(
            torch.bfloat16)

    out = {"q": randn(T, H, D), "k_new": randn(T, Hk, D), "v_new": randn(T, Hk, D)}
    if pools:
        if canary:
            fill = torch.tensor([CANARY_BF16], dtype=torch.int32).to(torch.int16).view(
                torch.bfloat16).item()
            kp = torch.full((spec.num_slots, Hk, D), fill, dtype=torch.bfloat16, device=device)
            vp = torch.full((spec.num_slots, Hk, D), fill, dtype=torch.bfloat16, device=device)
        else:
            kp = torch.empty((spec.num_slots, Hk, D), dtype=torch.bfloat16, device=device)
            vp = torch.empty((spec.num_slots, Hk, D), dtype=torch.bfloat16, device=device)
        slots = torch.from_numpy(prefix_slots(spec)).to(device)
        for i in range(0, slots.numel(), chunk_rows):
            idx = slots[i:i + chunk_rows]
            kp.index_copy_(0, idx, randn(idx.numel(), Hk, D))
            vp.index_copy_(0, idx, randn(idx.numel(), Hk, D))
        out["k_pool"], out["v_pool"] = kp, vp
    return out


def compact_requests(spec: BatchSpec, reqs) -> tuple[BatchSpec, np.ndarray]:
    """Relabel the pages of a subset of requests into a small dense pool.

    Returns (sub_spec, src_slots): sub_spec holds the chosen requests (in the
    given order) with a page table that points into a pool of
    len(src_slots) slots, whose slot i holds what src_slots[i] holds in the full
    pool.  Pages keep their size and alignment, so page geometry is preserved;
    only the labels change.
    """
    reqs = np.asarray(reqs, dtype=np.int64)
    P = spec.page_size
    dev = spec.device_len
    width = align_up(max(int(dev[reqs].max()), 1), 32)
    table = np.zeros((len(reqs), width), np.int32)
    page_ids: dict[int, int] = {}
    src_pages = []
    for n, r in enumerate(reqs):
        L = int(dev[r])
        row = spec.page_table[spec.req_rows[r], :L].astype(np.int64)
        first = row[::P] if P > 1 else row
        for pg in (first // P):
            pg = int(pg)
            if pg not in page_ids:
                page_ids[pg] = len(src_pages)
                src_pages.append(pg)
        j = np.arange(L)
        new_pages = np.array([page_ids[int(x)] for x in (row[j - j % P] // P)], np.int64)
        table[n, :L] = (new_pages * P + j % P).astype(np.int32)
    src_pages = np.asarray(src_pages, np.int64)
    src_slots = (src_pages[:, None] * P + np.arange(P)[None, :]).reshape(-1)
    sub = BatchSpec(name=spec.name + "_sub", cached_len=spec.cached_len[reqs].copy(),
                    extend_len=spec.extend_len[reqs].copy(),
                    req_rows=np.arange(len(reqs), dtype=np.int32), page_table=table,
                    page_size=P, num_slots=int(src_slots.shape[0]), seed=spec.seed,
                    num_qo_heads=spec.num_qo_heads, num_kv_heads=spec.num_kv_heads,
                    head_dim=spec.head_dim)
    return sub, src_slots


# ------------------------------------------------------------ sampler inputs
QWEN3_VOCAB = 151936          # Qwen3-0.6B's vocabulary (the model the pages run)


@dataclass
class SamplerSpec:
    """One batch of logits with each request's raw sampling parameters
    (temperature <= 0: greedy; top_k < 1: whole vocabulary; top_p: any float)
    and the uniform each row's draw consumes."""
    name: str
    logits: np.ndarray            # float32 [B, V], or bf16 bits uint16 [B, V]
    is_bf16: bool
    temperature: np.ndarray       # float32 [B]
    top_k: np.ndarray             # int32 [B]
    top_p: np.ndarray             # float32 [B]
    uniforms: np.ndarray          # float32 [B] in [0, 1)

    @property
    def batch(self) -> int:
        return int(self.logits.shape[0])

    @property
    def vocab(self) -> int:
        return int(self.logits.shape[1])

    def logits_f64(self) -> np.ndarray:
        return bf16_bits_to_f64(self.logits) if self.is_bf16 else self.logits.astype(np.float64)


_SAMPLER_MIX = (              # (temperature, top_k, top_p) of a request, drawn per row
    (0.0, -1, 1.0),           # greedy
    (1.0, -1, 1.0),           # plain draw
    (0.7, 50, 1.0),
    (1.0, 20, 0.9),
    (0.8, -1, 0.95),
    (1.3, 1000, 0.5),
    (0.6, 1, 1.0),
    (1.0, -1, 0.9),
)


def sampler_batch(name: str, seed: int, batch: int, vocab: int, bf16: bool = False,
                  mix=_SAMPLER_MIX, greedy_only: bool = False) -> SamplerSpec:
    """Logits shaped like a language model's: N(0, 2^2) per token, plus a few
    boosted tokens per row (none, 1, 3, 10 or 100 tokens raised by U(2, 12)),
    so that the top-p nucleus ranges from one token to most of the vocabulary.
    Rows take their parameters from `mix` in turn (all greedy if
    greedy_only); uniforms are U[0, 1) in float32."""
    rng = np.random.default_rng(seed)
    L = rng.normal(0.0, 2.0, (batch, vocab)).astype(np.float32)
    for r in range(batch):
        n = int(rng.choice([0, 1, 3, 10, 100]))
        n = min(n, vocab)
        if n:
            idx = rng.choice(vocab, n, replace=False)
            L[r, idx] += rng.uniform(2.0, 12.0, n).astype(np.float32)
    params = [(0.0, -1, 1.0)] * batch if greedy_only else [mix[r % len(mix)] for r in range(batch)]
    t = np.array([p[0] for p in params], np.float32)
    k = np.array([p[1] for p in params], np.int32)
    p = np.array([p[2] for p in params], np.float32)
    u = rng.random(batch).astype(np.float32)
    u = np.minimum(u, np.float32(1.0) - np.float32(2.0 ** -24))
    logits = f32_to_bf16_bits(L) if bf16 else L
    return SamplerSpec(name, logits, bf16, t, k, p, u)

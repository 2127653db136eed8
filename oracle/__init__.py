"""fp64 CPU oracle for the paged KV store and GQA paged attention.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import or run
anything in this package.  It shares no code with the CUDA library and never
imports it; the two meet only in the seeded input generators
(``paged_kv_gqa_store_gb300.workload``), which hold none of the method's
arithmetic.

What it computes (each function cites its page and section; see ``oracle.c``):

* ``metadata``          -- qo_indptr, kv_len, positions and out_loc of a batch
                           ("核心数据结构" Batch table; "Engine 与采样器", 手工驱动引擎).
* ``store_kv``          -- the out_loc row scatter into the K and V pools
                           ("Mini-SGLang 完整剖析" 4.4.3).
* ``paged_attention``   -- softmax(q.k / sqrt(D)) v with causal offset and
                           GQA mapping h -> h / (Hq/Hkv), K/V gathered token by
                           token through the page table ("第 0 步" attention
                           operator).
* ``complete_one``      -- the request length transition after a forward
                           ("核心数据结构", Req：请求的三个长度).
* ``build_kv_index``    -- the backends' page-id forms of the global token
                           table: dense per-request page-id table, ragged
                           page-id list with offsets ("Mini-SGLang 完整剖析" 4.6.4).
* ``token_slots``       -- the slot of every token of every request read back
                           through any of the three index forms (same section).
* ``rope_cos_sin_cache``, ``rmsnorm``, ``rope``, ``qk_norm_rope`` -- the step
                           that feeds the path: q_norm / k_norm and the rotary
                           embedding of the new q and k before store_kv
                           ("第 0 步" 四个算子; "Mini-SGLang 完整剖析" 4.5.6, 4.6.7).
* ``sampling_args``, ``sample_filter``, ``inverse_cdf``, ``sample`` -- the
                           batched sampler after the forward: temperature,
                           top-k then top-p, one draw per row from a uniform
                           passed in ("Engine 与采样器" 采样器; "Mini-SGLang
                           源码解析（四）" 14).

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
and its siblings (worked examples printed on the pages, a brute-force
contiguous attention, a pairwise brute-force sampler filter,
torch's scaled_dot_product_attention in float64 for the cached_len = 0 case,
closed forms and invariants).  None is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc (OpenMP if available) into oracle/_build."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:4] + ["-fopenmp"] + base[4:], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True, text=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P, I64, I32, D = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_double
            lib.oracle_metadata.argtypes = [P, I64, P, P, P, I32, P, P, P, P]
            lib.oracle_metadata.restype = None
            lib.oracle_store_kv.argtypes = [P, P, I64, I64, I64, P, P, P, I64]
            lib.oracle_store_kv.restype = None
            lib.oracle_paged_attention_rows.argtypes = [
                P, I64, P, P, I64, P, I64, P, P, P, I32, I32, I32, I32, D, P, I64, P]
            lib.oracle_paged_attention_rows.restype = None
            lib.oracle_num_threads.argtypes = []
            lib.oracle_num_threads.restype = ctypes.c_int
            lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
            lib.oracle_set_num_threads.restype = None
            _lib = lib
    return _lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> None:
    """Threads of later oracle calls (for timing on one core); the results do
    not depend on it."""
    _load().oracle_set_num_threads(int(n))


def metadata(page_table, cached_len, extend_len, req_rows=None):
    """Return dict(qo_indptr, kv_len, positions, out_loc) of a batch.

    page_table: int32 [rows, stride] token-granular slots; cached_len,
    extend_len: int32 [num_reqs]; req_rows: int32 [num_reqs] or None (row r).
    """
    pt = _c(page_table, np.int32)
    c = _c(cached_len, np.int32)
    e = _c(extend_len, np.int32)
    rows = None if req_rows is None else _c(req_rows, np.int32)
    n = int(c.shape[0])
    total = int(e.sum())
    qo = np.zeros(n + 1, np.int32)
    kv = np.zeros(n, np.int32)
    loc = np.zeros(total, np.int64)
    pos = np.zeros(total, np.int32)
    _load().oracle_metadata(_ptr(pt), pt.shape[1], _ptr(rows), _ptr(c), _ptr(e), n,
                            _ptr(qo), _ptr(kv), _ptr(loc), _ptr(pos))
    return {"qo_indptr": qo, "kv_len": kv, "positions": pos, "out_loc": loc}


def store_kv(k, v, out_loc, k_pool, v_pool):
    """Scatter new rows into the pools in place.

    k, v: uint16 (bf16 bits) [T, ...] flattened to [T, row_elems];
    out_loc: [T] integer slots; k_pool, v_pool: uint16 [num_slots, ...] C-contiguous.
    """
    kk = _c(k, np.uint16).reshape(k.shape[0], -1)
    vv = _c(v, np.uint16).reshape(v.shape[0], -1)
    loc = _c(out_loc, np.int64)
    assert k_pool.flags.c_contiguous and v_pool.flags.c_contiguous
    assert k_pool.dtype == np.uint16 and v_pool.dtype == np.uint16
    row = kk.shape[1]
    pool_stride = int(np.prod(k_pool.shape[1:]))
    assert row <= pool_stride and loc.shape[0] == kk.shape[0]
    if loc.size:
        assert loc.min() >= 0 and loc.max() < k_pool.shape[0]
    _load().oracle_store_kv(_ptr(kk), _ptr(vv), row, kk.shape[0], row, _ptr(loc),
                            _ptr(k_pool), _ptr(v_pool), pool_stride)


def paged_attention(q, k_pool, v_pool, page_table, cached_len, qo_indptr,
                    num_qo_heads, num_kv_heads, head_dim, scale=None,
                    req_rows=None, rows=None):
    """fp64 paged GQA attention.

    q: uint16 (bf16 bits) [total_q, Hq, D]; pools: uint16 [num_slots, Hkv, D];
    page_table: int32 [rows, stride]; cached_len: int32 [num_reqs];
    qo_indptr: int32 [num_reqs + 1]; rows: optional int64 list of query rows
    (default all).  Returns float64 [len(rows), Hq, D].
    """
    if scale is None:
        scale = 1.0 / np.sqrt(head_dim)
    qq = _c(q, np.uint16).reshape(q.shape[0], -1)
    assert k_pool.flags.c_contiguous and v_pool.flags.c_contiguous
    pt = _c(page_table, np.int32)
    c = _c(cached_len, np.int32)
    qo = _c(qo_indptr, np.int32)
    rr = None if req_rows is None else _c(req_rows, np.int32)
    if rows is None:
        rows = np.arange(qq.shape[0], dtype=np.int64)
    rows = _c(rows, np.int64)
    assert num_qo_heads % num_kv_heads == 0
    out = np.empty((rows.shape[0], num_qo_heads, head_dim), np.float64)
    pool_stride = int(np.prod(k_pool.shape[1:]))
    _load().oracle_paged_attention_rows(
        _ptr(qq), qq.shape[1], _ptr(k_pool), _ptr(v_pool), pool_stride, _ptr(pt),
        pt.shape[1], _ptr(rr), _ptr(c), _ptr(qo), c.shape[0], num_qo_heads,
        num_kv_heads, head_dim, float(scale), _ptr(rows), rows.shape[0], _ptr(out))
    return out


KV_TOKEN_TABLE, KV_PAGE_TABLE, KV_RAGGED = 0, 1, 2


def build_kv_index(kind, page_size, page_table, cached_len, extend_len, req_rows=None):
    """The backends' form of the global token table for a batch ("Mini-SGLang
    完整剖析" 4.6.4): the global table stores one slot per token; the
    FlashAttention / TRT-LLM backends take every page_size-th column and divide
    it by page_size (a dense [requests, pages] table of page ids), FlashInfer
    concatenates the per-request lists into one 1-D array with offsets.

    Returns a list of per-request page-id lists (plain Python ints), and, for
    the two kinds, the dense table (padded with -1) or (indices, indptr)."""
    P = int(page_size)
    pages = []
    for r in range(len(cached_len)):
        row = r if req_rows is None else int(req_rows[r])
        n = int(cached_len[r]) + int(extend_len[r])
        ids = []
        for i in range((n + P - 1) // P):
            first = int(page_table[row][i * P])
            ids.append(first // P)
        pages.append(ids)
    if kind == KV_PAGE_TABLE:
        width = max([len(x) for x in pages] + [1])
        table = np.full((len(pages), width), -1, np.int32)
        for r, ids in enumerate(pages):
            table[r, :len(ids)] = ids
        return pages, table
    indptr = [0]
    flat = []
    for ids in pages:
        flat.extend(ids)
        indptr.append(len(flat))
    return pages, (np.array(flat, np.int32), np.array(indptr, np.int32))


def token_slots(kind, page_size, table, kv_len, req_rows=None, indptr=None):
    """Slot of token j of request r for j < kv_len[r], read through an index of
    the given kind ("Mini-SGLang 完整剖析" 4.6.4):
      token table : table[row_r][j]                     (every token's own entry)
      page table  : table[row_r][j // P] * P + j % P
      ragged      : table[indptr[r] + j // P] * P + j % P
    Returns an int32 [num_reqs, max(kv_len)] token table (rows = requests,
    unused entries -1) that the other oracle functions read with req_rows=None."""
    P = int(page_size)
    n_req = len(kv_len)
    width = max([int(x) for x in kv_len] + [1])
    out = np.full((n_req, width), -1, np.int64)
    for r in range(n_req):
        for j in range(int(kv_len[r])):
            if kind == KV_TOKEN_TABLE:
                row = r if req_rows is None else int(req_rows[r])
                out[r, j] = int(table[row][j])
            elif kind == KV_PAGE_TABLE:
                row = r if req_rows is None else int(req_rows[r])
                out[r, j] = int(table[row][j // P]) * P + j % P
            else:
                out[r, j] = int(table[int(indptr[r]) + j // P]) * P + j % P
    return out.astype(np.int32)


def rope_cos_sin_cache(theta: float, head_dim: int, max_pos: int) -> np.ndarray:
    """Rotary cache ("Mini-SGLang 完整剖析" 4.5.6: one [max_position, rotary_dim]
    table shared by every layer; "第 0 步" rope: inv_freq_i = theta^(-2i/D),
    angle = pos * inv_freq).  Reading fixed for this library: inv_freq rounded
    once to fp32, the angle one fp32 product, cos / sin of that angle rounded
    once to fp32.  Returns float32 [max_pos, D] = [cos | sin]."""
    half = head_dim // 2
    inv = np.array([float(theta) ** (-2.0 * i / head_dim) for i in range(half)],
                   np.float64).astype(np.float32)
    pos = np.arange(max_pos, dtype=np.float32)
    angle = (pos[:, None] * inv[None, :]).astype(np.float32)       # one fp32 rounding
    a = angle.astype(np.float64)
    return np.concatenate([np.cos(a), np.sin(a)], axis=1).astype(np.float32)


def bf16_bits_to_f64(bits) -> np.ndarray:
    """bf16 bit patterns -> float64 (exact: bf16 is the upper half of a binary32)."""
    u = np.asarray(bits, np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def rmsnorm(x, w, eps):
    """RMSNorm over the last axis ("第 0 步" 四个算子: a scale only, no mean or
    bias): w * x / sqrt(mean(x^2) + eps), in float64."""
    x = np.asarray(x, np.float64)
    return np.asarray(w, np.float64) * (x / np.sqrt((x * x).mean(-1, keepdims=True) + eps))


def rope(x, cos_sin_rows):
    """Rotate the first half of the last axis against the second half ("第 0 步"
    rope, the Hugging Face / Qwen pairing): [x1 c - x2 s, x1 s + x2 c] with c, s
    the cache row of each leading index; float64."""
    x = np.asarray(x, np.float64)
    half = x.shape[-1] // 2
    cs = np.asarray(cos_sin_rows, np.float64)
    c, s = cs[..., :half], cs[..., half:]
    while c.ndim < x.ndim:                        # broadcast over the heads axis
        c, s = c[..., None, :], s[..., None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * c - x2 * s, x1 * s + x2 * c], axis=-1)


def qk_norm_rope(qkv_bits, positions, q_norm_w_bits, k_norm_w_bits, eps, cos_sin,
                 num_qo_heads, num_kv_heads, head_dim):
    """The attention layer's front ("Mini-SGLang 完整剖析" 4.6.7: split qkv, q_norm
    and k_norm per head, rotary at the batch positions; then store_kv): returns
    (q float64 [T, Hq, D], k float64 [T, Hkv, D], v bf16 bits [T, Hkv, D])."""
    T = qkv_bits.shape[0]
    x = bf16_bits_to_f64(np.asarray(qkv_bits).reshape(T, -1))
    Hq, Hk, D = num_qo_heads, num_kv_heads, head_dim
    q = x[:, :Hq * D].reshape(T, Hq, D)
    k = x[:, Hq * D:(Hq + Hk) * D].reshape(T, Hk, D)
    v_bits = np.asarray(qkv_bits).reshape(T, -1)[:, (Hq + Hk) * D:(Hq + 2 * Hk) * D]
    rows = np.asarray(cos_sin)[np.asarray(positions, np.int64)]
    qn = rope(rmsnorm(q, bf16_bits_to_f64(q_norm_w_bits), eps), rows)
    kn = rope(rmsnorm(k, bf16_bits_to_f64(k_norm_w_bits), eps), rows)
    return qn, kn, v_bits.reshape(T, Hk, D).copy()


def complete_one(cached_len: int, device_len: int) -> tuple[int, int]:
    """Request length transition after one forward ("核心数据结构", Req section):
    every token of this step is now cached, and the next step computes one more
    position.  Returns the new (cached_len, device_len)."""
    return device_len, device_len + 1


# ------------------------------------------------------------------ sampler
# "Engine 与采样器" (Sampler, sample_torch) and "Mini-SGLang 源码解析（四）"
# 14.2-14.5, "Mini-SGLang 完整剖析" 4.8.5: the step after the forward in
# forward_batch turns each request's row of logits into its next token.
SAMPLE_MIN_T = 1e-6          # smallest temperature (a greedy request in a mixed batch)
SAMPLE_MIN_P = 1e-6          # smallest top-p


def is_greedy(temperature, top_k, top_p):
    """SamplingParams.is_greedy ("核心数据结构：Req、Batch、Context", section
    SamplingParams; "Mini-SGLang 完整剖析" 4.8.4): a request is greedy when its
    temperature is at most 0 or its top_k is 1, and its top_p is exactly 1 --
    a request with top_p below 1 is not greedy even at temperature 0."""
    return (float(temperature) <= 0.0 or int(top_k) == 1) and float(top_p) == 1.0


def sampling_args(temperature, top_k, top_p, vocab_size):
    """Per-batch sampling arguments (Sampler.prepare, "Engine 与采样器" 采样器;
    "Mini-SGLang 完整剖析" 4.8.5), from per-request (temperature, top_k, top_p).

    Returns (temperatures, top_k, top_p) as float32 / int32 / float32 arrays or
    None: temperatures is None when every request is_greedy (the sampler then
    takes the argmax); otherwise a greedy request gets temperature MIN_T and
    any other max(temperature, MIN_T) (so a temperature <= 0 request with
    top_p < 1 is sampled at MIN_T); top_k < 1 means the whole vocabulary and
    the array is None unless some request restricts it; top_p is clamped to
    [MIN_P, 1] and is None unless some request has top_p < 1."""
    reqs = list(zip([float(x) for x in temperature], [int(k) for k in top_k],
                    [float(p) for p in top_p]))
    greedy = [is_greedy(t, k, p) for t, k, p in reqs]
    if all(greedy):
        return None, None, None
    ts = np.array([max(0.0 if g else t, SAMPLE_MIN_T) for (t, _, _), g in zip(reqs, greedy)],
                  np.float32)
    ks = [k if k >= 1 else int(vocab_size) for _, k, _ in reqs]
    ps = [min(max(p, SAMPLE_MIN_P), 1.0) for _, _, p in reqs]
    k_arr = np.array(ks, np.int32) if any(k != vocab_size for k in ks) else None
    p_arr = np.array(ps, np.float32) if any(p < 1.0 for p in ps) else None
    return ts, k_arr, p_arr


def sample_filter(logits_row, temperature, top_k=None, top_p=None):
    """The distribution one request draws from (sample_torch, "Engine 与采样器";
    "Mini-SGLang 源码解析（四）" 14.4), float64.

    1. p = softmax(logits / T), T = max(temperature, MIN_T).
    2. Order the vocabulary by p, largest first; equal p in increasing token
       index (the pages sort without saying how ties fall: this is the
       library's reading).
    3. top-k (k < 1 or k >= V: no cut): ranks >= k get 0.
    4. top-p (clamped to [MIN_P, 1]): renormalise what is left; a token keeps
       its mass only if the mass ranked before it is below top_p, so the most
       likely token always stays (FlashInfer order: top-k first, then top-p).
    Returns (q, order): q the kept masses renormalised to sum 1, scattered
    back to vocabulary order; order the ranking of step 2."""
    T = float(np.float32(max(float(temperature), SAMPLE_MIN_T)))   # a float32 tensor on the pages
    x = np.asarray(logits_row, np.float64) / T
    e = np.exp(x - x.max())
    p = e / e.sum()
    V = p.shape[0]
    order = np.argsort(-p, kind="stable")
    sp = p[order].copy()
    if top_k is not None:
        k = int(top_k)
        if 1 <= k < V:
            sp[k:] = 0.0
    P = 1.0 if top_p is None else float(np.float32(min(max(float(top_p), SAMPLE_MIN_P), 1.0)))
    if P < 1.0:
        # top_p = 1 cuts nothing: in exact arithmetic the mass before any token
        # that has mass is below 1 (a rounded cumulative sum reaching 1.0 is not
        # a cut)
        sp = sp / sp.sum()
        before = np.concatenate([[0.0], np.cumsum(sp)[:-1]])
        sp[before >= P] = 0.0
    q = np.zeros(V, np.float64)
    q[order] = sp
    return q / q.sum(), order


def inverse_cdf(q, u):
    """The draw (torch.multinomial with one sample in sample_torch): with the
    uniform u in [0, 1) passed in, the token is the smallest index i, in
    vocabulary order, whose cumulative mass q_0 + ... + q_i exceeds u times
    the total."""
    c = np.cumsum(np.asarray(q, np.float64))
    return int(np.searchsorted(c, float(u) * c[-1], side="right"))


def sample(logits, temperatures, top_k, top_p, uniforms):
    """Batched sampler (Sampler.sample): next token of every row of logits
    [B, V] (float32 values, or anything float64 holds exactly).

    temperatures None: every request is greedy and the token is the argmax of
    the row (first index among equal maxima, torch.argmax).  Otherwise each row
    draws from sample_filter(row, T, k, p) with its uniform.  top_k / top_p
    None mean no cut for any row.  Returns int32 [B]."""
    L = np.asarray(logits, np.float64)
    B = L.shape[0]
    out = np.empty(B, np.int32)
    for r in range(B):
        if temperatures is None:
            out[r] = int(np.argmax(L[r]))
            continue
        q, _ = sample_filter(L[r], temperatures[r],
                             None if top_k is None else top_k[r],
                             None if top_p is None else top_p[r])
        out[r] = inverse_cdf(q, uniforms[r])
    return out

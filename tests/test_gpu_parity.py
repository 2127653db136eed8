"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on
seeded inputs, at sizes the oracle finishes in seconds, spanning several tiles,
ragged tails, every supported page size and the degenerate cases.

Bars: metadata and store_kv bit-exact; attention within max-abs 1e-2 and
relative L2 2e-3 of the oracle."""
import numpy as np
import pytest
import torch

import paged_kv_gqa_store_gb300 as msg
from paged_kv_gqa_store_gb300 import workload as wl

from _harness import (GpuBatch, assert_attn_close, oracle_small, run_small)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    msg.load_library()


def _check_full(spec, host, flags=0, out_loc_int64=True, q_stride_pad=0):
    g = run_small(spec, host, flags=flags, out_loc_int64=out_loc_int64, q_stride_pad=q_stride_pad)
    o = oracle_small(spec, host)
    assert g["status"] == msg.MSG_OK, g["status_info"]
    assert np.array_equal(g["qo"], o["qo_indptr"])
    assert np.array_equal(g["out_loc"], o["out_loc"])
    assert np.array_equal(g["positions"], o["positions"])
    assert np.array_equal(g["k_pool"], o["k_pool"]), "store_kv K pool differs"
    assert np.array_equal(g["v_pool"], o["v_pool"]), "store_kv V pool differs"
    assert_attn_close(g["out"], o["out"], spec.name)
    return g, o


# ------------------------------------------------------------ the tiny config
@pytest.mark.parametrize("int64_loc", [True, False])
def test_tiny_mixed_config(int64_loc):
    spec = wl.config_tiny_mixed()
    _check_full(spec, wl.host_tensors(spec), out_loc_int64=int64_loc)


# ------------------------------------------------------------ random ragged batches
def _rand_spec(seed, n_dec, n_ext, page_size, max_ctx=700, max_ext=200, shuffle=True,
               extra_rows=3, **kw):
    rng = np.random.default_rng(seed)
    cached = list(rng.integers(0, max_ctx, size=n_dec)) + list(rng.integers(0, max_ctx, size=n_ext))
    ext = [1] * n_dec + list(rng.integers(2, max_ext + 1, size=n_ext))
    order = rng.permutation(n_dec + n_ext)
    cached = np.asarray(cached)[order]
    ext = np.asarray(ext)[order]
    need = int(((np.asarray(cached) + ext + page_size - 1) // page_size).sum())
    return wl.make_batch(f"rand{seed}_p{page_size}", seed, cached, ext, page_size,
                         num_pages=need + 11, shuffle_rows=shuffle, extra_rows=extra_rows, **kw)


@pytest.mark.parametrize("page_size", [1, 16, 64])
def test_decode_only_ragged(page_size):
    spec = _rand_spec(200 + page_size, n_dec=37, n_ext=0, page_size=page_size)
    _check_full(spec, wl.host_tensors(spec), flags=msg.MSG_ATTN_DECODE_ONLY)


@pytest.mark.parametrize("page_size", [1, 16, 64])
def test_extend_only_ragged(page_size):
    spec = wl.make_batch(f"ext_p{page_size}", 300 + page_size, cached_len=[0, 63, 130, 7],
                         extend_len=[65, 2, 129, 64], page_size=page_size,
                         num_pages=(2048 // page_size) + 8, shuffle_rows=True, extra_rows=2)
    _check_full(spec, wl.host_tensors(spec), flags=msg.MSG_ATTN_EXTEND_ONLY)


@pytest.mark.parametrize("page_size", [1, 16])
def test_mixed_ragged_with_strided_q(page_size):
    spec = _rand_spec(400 + page_size, n_dec=21, n_ext=5, page_size=page_size)
    _check_full(spec, wl.host_tensors(spec), q_stride_pad=16)


def test_long_single_decode_splits_over_all_ctas():
    spec = wl.make_batch("long1", 501, cached_len=[40000], extend_len=[1], page_size=1,
                         num_pages=40100)
    _check_full(spec, wl.host_tensors(spec))


@pytest.mark.parametrize("page_size", [1, 16])
def test_few_long_decodes_both_merge_instances(page_size):
    """A few long decode requests, each cut over 30-70 CTAs: with max_kv_len
    given the library takes the decode instance that merges the splits in two
    levels (groups of 8, then the groups); without it the one-level instance.
    Both match the oracle, and each is bit-identical on repeat."""
    rng = np.random.default_rng(590 + page_size)
    cached = rng.integers(2000, 6000, size=6)
    pages = int(sum((c + page_size) // page_size + 1 for c in cached)) + 32
    spec = wl.make_batch("few_long", 590 + page_size, cached, np.ones(6, np.int32), page_size,
                         num_pages=pages)
    host = wl.host_tensors(spec)
    ref = oracle_small(spec, host)["out"]
    for mkv in (spec.max_kv_len, 0):
        outs = []
        for _ in range(2):
            gb = GpuBatch(spec)
            q = wl.bits_to_torch(host["q"], "cuda")
            kp = wl.bits_to_torch(host["k_pool"], "cuda")
            vp = wl.bits_to_torch(host["v_pool"], "cuda")
            loc = gb.plan()
            msg.msg_store_kv(wl.bits_to_torch(host["k_new"], "cuda"),
                             wl.bits_to_torch(host["v_new"], "cuda"), kp, vp, loc, dev_status=gb.ws)
            out = gb.attention(q, kp, vp, flags=msg.MSG_ATTN_REUSE_PLAN, max_kv_len=mkv)
            torch.cuda.synchronize()
            assert gb.status()[0] == msg.MSG_OK, gb.status()
            outs.append(wl.torch_to_bits(out))
        assert np.array_equal(outs[0], outs[1])
        assert_attn_close(outs[0], ref, f"few_long max_kv_len={mkv}")


@pytest.mark.parametrize("page_size", [1, 16])
def test_fused_store_decode_is_store_then_attend(page_size):
    """msg_paged_attention_store (store_kv done by the decode kernel, the newest
    key gathered from k_new / v_new) gives the output and pool bits of
    msg_store_kv followed by msg_paged_attention, with one request cut across
    most CTAs, and matches the oracle."""
    rng = np.random.default_rng(560 + page_size)
    n = 12
    cached = rng.integers(1, 2000, size=n)
    cached[0] = 12000
    pages = int(sum((c + page_size) // page_size + 1 for c in cached)) + 64
    spec = wl.make_batch("fused", 560 + page_size, cached, np.ones(n, np.int32), page_size,
                         num_pages=pages)
    host = wl.host_tensors(spec)
    ref = run_small(spec, host, flags=msg.MSG_ATTN_DECODE_ONLY)
    assert ref["status"] == msg.MSG_OK, ref["status_info"]
    dev = "cuda"
    gb = GpuBatch(spec, dev)
    q = wl.bits_to_torch(host["q"], dev)
    k_new, v_new = wl.bits_to_torch(host["k_new"], dev), wl.bits_to_torch(host["v_new"], dev)
    k_pool, v_pool = wl.bits_to_torch(host["k_pool"], dev), wl.bits_to_torch(host["v_pool"], dev)
    gb.plan()
    out = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
    msg.msg_paged_attention_store(q, k_new, v_new, k_pool, v_pool, gb.page_table, gb.cached,
                                  gb.extend, gb.qo, out, gb.ws, page_size=spec.page_size,
                                  req_rows=gb.rows, max_kv_len=spec.max_kv_len,
                                  flags=msg.MSG_ATTN_DECODE_ONLY | msg.MSG_ATTN_REUSE_PLAN)
    torch.cuda.synchronize()
    st, info = gb.status()
    assert st == msg.MSG_OK, info
    assert np.array_equal(wl.torch_to_bits(out), ref["out"])
    assert np.array_equal(wl.torch_to_bits(k_pool), ref["k_pool"])
    assert np.array_equal(wl.torch_to_bits(v_pool), ref["v_pool"])
    assert_attn_close(wl.torch_to_bits(out), oracle_small(spec, host)["out"], "fused")


def test_many_tiny_decodes():
    rng = np.random.default_rng(502)
    n = 600
    cached = rng.integers(0, 5, size=n)
    spec = wl.make_batch("tiny_many", 502, cached, np.ones(n, np.int32), 1,
                         num_pages=int(cached.sum()) + n + 10)
    _check_full(spec, wl.host_tensors(spec))


def test_degenerate_lengths():
    # kv_len 1 decode, 2-token prefill from nothing, extend of exactly 64 and 65
    # tokens at a cached length that is a multiple of the key tile.
    spec = wl.make_batch("degenerate", 503, cached_len=[0, 0, 64, 128, 5],
                         extend_len=[1, 2, 64, 65, 1], page_size=1, num_pages=600)
    _check_full(spec, wl.host_tensors(spec))


def test_empty_batches_are_noops():
    spec = wl.make_batch("empty", 504, cached_len=[], extend_len=[], page_size=1, num_pages=16)
    gb = GpuBatch(spec)
    q = torch.zeros(0, 16, 128, dtype=torch.bfloat16, device="cuda")
    pool = torch.zeros(16, 8, 128, dtype=torch.bfloat16, device="cuda")
    gb.attention(q, pool, pool)
    msg.msg_store_kv(q[:, :8], q[:, :8], pool, pool,
                     torch.zeros(0, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()


# ------------------------------------------------------------ invariants on the GPU
def test_page_permutation_gives_identical_bits():
    base = _rand_spec(600, n_dec=9, n_ext=3, page_size=1, shuffle=False, extra_rows=0)
    host = wl.host_tensors(base)
    a = run_small(base, host)
    perm = np.random.default_rng(601).permutation(base.num_slots).astype(np.int32)
    spec2 = wl.BatchSpec(**{**base.__dict__, "page_table": perm[base.page_table]})
    host2 = dict(host)
    inv = np.argsort(perm)
    host2["k_pool"] = host["k_pool"][inv]
    host2["v_pool"] = host["v_pool"][inv]
    b = run_small(spec2, host2)
    assert np.array_equal(a["out"], b["out"])


def test_page_size_gives_identical_bits():
    outs = []
    cached, ext = [70, 0, 130, 300], [1, 65, 1, 40]
    for P in (1, 16, 64):
        spec = wl.make_batch(f"ps{P}", 700 + P, cached, ext, P,
                             num_pages=int(((np.array(cached) + ext + P - 1) // P).sum()) + 3)
        rng = np.random.default_rng(7)      # same values for every geometry
        host = {"q": wl.random_bf16(rng, (spec.total_q, 16, 128)),
                "k_new": wl.random_bf16(rng, (spec.total_q, 8, 128)),
                "v_new": wl.random_bf16(rng, (spec.total_q, 8, 128))}
        kseq = wl.random_bf16(rng, (int(spec.device_len.sum()), 8, 128))
        vseq = wl.random_bf16(rng, (int(spec.device_len.sum()), 8, 128))
        kp = np.full((spec.num_slots, 8, 128), wl.CANARY_BF16, np.uint16)
        vp = kp.copy()
        off = 0
        for r in range(spec.num_reqs):
            c = int(spec.cached_len[r])
            slots = spec.page_table[spec.req_rows[r], :c]
            kp[slots] = kseq[off:off + c]
            vp[slots] = vseq[off:off + c]
            off += int(spec.device_len[r])
        host["k_pool"], host["v_pool"] = kp, vp
        outs.append(run_small(spec, host)["out"])
    assert np.array_equal(outs[0], outs[1]) and np.array_equal(outs[0], outs[2])


def test_constant_v_reproduces_v():
    spec = _rand_spec(800, n_dec=7, n_ext=2, page_size=1)
    host = wl.host_tensors(spec)
    rng = np.random.default_rng(801)
    vconst = wl.random_bf16(rng, (8, 128))
    host["v_pool"] = np.where(host["v_pool"] == wl.CANARY_BF16, wl.CANARY_BF16,
                              np.broadcast_to(vconst, host["v_pool"].shape)).astype(np.uint16)
    host["v_new"] = np.broadcast_to(vconst, host["v_new"].shape).copy()
    g = run_small(spec, host)
    expect = np.repeat(wl.bf16_bits_to_f64(vconst), 2, axis=0)
    got = wl.bf16_bits_to_f64(g["out"])
    assert np.abs(got - expect[None]).max() <= np.abs(expect).max() * 2 ** -8


def test_chunked_prefill_matches_single_extend():
    # The same 150-token extend done at once, in 3 chunks, and as decode steps
    # for the last 5 tokens: per-token outputs agree within the tolerance.
    rng = np.random.default_rng(900)
    L, c0 = 160, 10
    pt = wl.assign_pages(rng, [L], 1, 256)
    q = wl.random_bf16(rng, (L - c0, 16, 128))
    kall = wl.random_bf16(rng, (L, 8, 128))
    vall = wl.random_bf16(rng, (L, 8, 128))
    kp = np.full((256, 8, 128), wl.CANARY_BF16, np.uint16)
    vp = kp.copy()
    kp[pt[0, :c0]] = kall[:c0]
    vp[pt[0, :c0]] = vall[:c0]

    def run(chunks):
        kp_d = wl.bits_to_torch(kp, "cuda")
        vp_d = wl.bits_to_torch(vp, "cuda")
        outs, c = [], c0
        for e in chunks:
            spec = wl.BatchSpec("chunk", np.array([c], np.int32), np.array([e], np.int32),
                                np.array([0], np.int32), pt, 1, 256, 0)
            gb = GpuBatch(spec)
            loc = gb.plan()
            msg.msg_store_kv(wl.bits_to_torch(kall[c:c + e], "cuda"),
                             wl.bits_to_torch(vall[c:c + e], "cuda"), kp_d, vp_d, loc)
            out = gb.attention(wl.bits_to_torch(q[c - c0:c - c0 + e], "cuda"), kp_d, vp_d,
                               flags=msg.MSG_ATTN_REUSE_PLAN)
            outs.append(wl.torch_to_bits(out))
            c += e
        return wl.bf16_bits_to_f64(np.concatenate(outs))

    one = run([L - c0])
    for chunks in ([50, 64, 31, 5], [145, 1, 1, 1, 1, 1]):
        other = run(chunks)
        assert np.abs(one - other).max() <= 1e-2


# ------------------------------------------------------------ padding, reuse, errors
def test_dummy_padding_duplicates_only_touch_the_dummy_slot():
    # Two padding requests point at the dummy slot (the pool's last slot), as a
    # CUDA-graph-padded decode batch does; real requests must be unaffected.
    spec = _rand_spec(1000, n_dec=6, n_ext=1, page_size=1, shuffle=False, extra_rows=0)
    dummy = spec.num_slots
    n = spec.num_reqs
    pt = np.zeros((n + 1, spec.page_table.shape[1]), np.int32)
    pt[:n] = spec.page_table
    pt[n, :] = dummy
    padded = wl.BatchSpec(name="padded", cached_len=np.r_[spec.cached_len, 0, 0].astype(np.int32),
                          extend_len=np.r_[spec.extend_len, 1, 1].astype(np.int32),
                          req_rows=np.r_[np.arange(n), n, n].astype(np.int32), page_table=pt,
                          page_size=1, num_slots=spec.num_slots + 1, seed=spec.seed)
    host = wl.host_tensors(padded)
    g = run_small(padded, host)
    o = oracle_small(padded, host)
    assert g["status"] == msg.MSG_OK
    real = np.arange(padded.num_slots) != dummy
    assert np.array_equal(g["k_pool"][real], o["k_pool"][real])
    assert np.array_equal(g["v_pool"][real], o["v_pool"][real])
    nreal = int(spec.extend_len.sum())
    assert_attn_close(g["out"][:nreal], o["out"][:nreal], "padded batch")


def test_plan_reuse_is_repeatable():
    spec = _rand_spec(1100, n_dec=30, n_ext=2, page_size=16)
    host = wl.host_tensors(spec)
    gb = GpuBatch(spec)
    q = wl.bits_to_torch(host["q"], "cuda")
    kp = wl.bits_to_torch(host["k_pool"], "cuda")
    vp = wl.bits_to_torch(host["v_pool"], "cuda")
    loc = gb.plan()
    msg.msg_store_kv(wl.bits_to_torch(host["k_new"], "cuda"),
                     wl.bits_to_torch(host["v_new"], "cuda"), kp, vp, loc)
    outs = [wl.torch_to_bits(gb.attention(q, kp, vp, flags=msg.MSG_ATTN_REUSE_PLAN))
            for _ in range(3)]
    outs.append(wl.torch_to_bits(gb.attention(q, kp, vp)))       # replans
    assert all(np.array_equal(outs[0], o) for o in outs[1:])
    assert gb.status()[0] == msg.MSG_OK


def test_out_of_range_slot_is_reported_not_faulted():
    spec = _rand_spec(1200, n_dec=4, n_ext=1, page_size=1, shuffle=False, extra_rows=0)
    host = wl.host_tensors(spec)
    bad = spec.page_table.copy()
    bad[0, 0] = spec.num_slots + 5            # outside the pool
    bad_spec = wl.BatchSpec(**{**spec.__dict__, "page_table": bad})
    gb = GpuBatch(bad_spec)
    q = wl.bits_to_torch(host["q"], "cuda")
    kp = wl.bits_to_torch(host["k_pool"], "cuda")
    vp = wl.bits_to_torch(host["v_pool"], "cuda")
    gb.plan()
    gb.attention(q, kp, vp)
    st, info = gb.status()
    assert st == msg.MSG_ERR_DEVICE_CHECK and info[0] == msg.MSG_DEV_SLOT_OUT_OF_RANGE
    msg.msg_clear_device_status(gb.ws)
    assert gb.status()[0] == msg.MSG_OK
    # store_kv with an out-of-range out_loc: the row is skipped and reported
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    loc = torch.tensor([0, spec.num_slots], dtype=torch.int64, device="cuda")
    before = wl.torch_to_bits(kp)
    kn = torch.ones(2, 8, 128, dtype=torch.bfloat16, device="cuda")
    msg.msg_store_kv(kn, kn, kp, vp, loc, dev_status=status)
    st, info = msg.msg_read_device_status(status)
    assert st == msg.MSG_ERR_DEVICE_CHECK and info[0] == msg.MSG_DEV_SLOT_OUT_OF_RANGE
    after = wl.torch_to_bits(kp)
    assert np.array_equal(after[1:], before[1:])


@pytest.mark.parametrize("page_size", [16, 64])
def test_extend_page_outside_the_pool_is_reported_other_requests_still_match(page_size):
    """Pages of 16 or more keys, where the extend kernel loads each 16-key run
    of a page as one tile: an extend request whose first (fully cached) page
    lies past the pool is reported and read as zeros, its output stays finite,
    and every other request's rows still match the oracle."""
    cached = [100, 37, 300, 5, 250, 64]
    ext = [1, 150, 1, 1, 200, 67]
    need = sum((c + e + page_size - 1) // page_size for c, e in zip(cached, ext))
    spec = wl.make_batch(f"badpage_p{page_size}", 1230 + page_size, cached, ext, page_size,
                         num_pages=need + 7)
    host = wl.host_tensors(spec)
    bad_req = 4
    bad = spec.page_table.copy()
    bad[spec.req_rows[bad_req], 0] = spec.num_slots + page_size     # a page past the pool
    g = run_small(wl.BatchSpec(**{**spec.__dict__, "page_table": bad}), host)
    o = oracle_small(spec, host)
    assert g["status"] == msg.MSG_ERR_DEVICE_CHECK
    assert g["status_info"][0] == msg.MSG_DEV_SLOT_OUT_OF_RANGE
    qo = o["qo_indptr"]
    keep = np.ones(spec.total_q, bool)
    keep[qo[bad_req]:qo[bad_req + 1]] = False
    assert np.isfinite(wl.bf16_bits_to_f64(g["out"][~keep])).all()
    assert_attn_close(g["out"][keep], o["out"][keep], spec.name)


def test_phase_flag_contradiction_is_reported():
    spec = _rand_spec(1300, n_dec=3, n_ext=1, page_size=1)
    host = wl.host_tensors(spec)
    gb = GpuBatch(spec)
    q = wl.bits_to_torch(host["q"], "cuda")
    kp = wl.bits_to_torch(host["k_pool"], "cuda")
    vp = wl.bits_to_torch(host["v_pool"], "cuda")
    gb.plan()
    gb.attention(q, kp, vp, flags=msg.MSG_ATTN_DECODE_ONLY)
    st, info = gb.status()
    assert st == msg.MSG_ERR_DEVICE_CHECK and info[0] == msg.MSG_DEV_WRONG_PHASE


# ------------------------------------------------------------ tensor-parallel head slices
@pytest.mark.parametrize("hkv", [4, 2, 1])
@pytest.mark.parametrize("page_size", [1, 16])
def test_tp_head_slice_mixed(hkv, page_size):
    """A tensor-parallel rank holds num_kv_heads / tp KV heads and their 2 query
    heads each ("Mini-SGLang 完整剖析" 4.5: the QKV projection is split by KV
    head); its attention is the same call with fewer heads: 8q/4kv at tp = 2,
    4q/2kv at tp = 4, 2q/1kv at tp = 8."""
    spec = _rand_spec(700 + 10 * hkv + page_size, n_dec=25, n_ext=4, page_size=page_size,
                      num_qo_heads=2 * hkv, num_kv_heads=hkv)
    _check_full(spec, wl.host_tensors(spec))


@pytest.mark.parametrize("hkv", [4, 1])
def test_tp_head_slice_fused_store_long_request(hkv):
    """The fused store + decode call on a head slice, one request cut over
    most CTAs; equals store_kv then attention bit for bit, and the oracle."""
    rng = np.random.default_rng(580 + hkv)
    n = 9
    cached = rng.integers(1, 1500, size=n)
    cached[3] = 20000
    spec = wl.make_batch("fused_tp", 580 + hkv, cached, np.ones(n, np.int32), 1,
                         num_pages=int(cached.sum()) + 64, num_qo_heads=2 * hkv,
                         num_kv_heads=hkv)
    host = wl.host_tensors(spec)
    ref = run_small(spec, host, flags=msg.MSG_ATTN_DECODE_ONLY)
    assert ref["status"] == msg.MSG_OK, ref["status_info"]
    dev = "cuda"
    gb = GpuBatch(spec, dev)
    q = wl.bits_to_torch(host["q"], dev)
    k_new, v_new = wl.bits_to_torch(host["k_new"], dev), wl.bits_to_torch(host["v_new"], dev)
    k_pool, v_pool = wl.bits_to_torch(host["k_pool"], dev), wl.bits_to_torch(host["v_pool"], dev)
    gb.plan()
    out = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
    msg.msg_paged_attention_store(q, k_new, v_new, k_pool, v_pool, gb.page_table, gb.cached,
                                  gb.extend, gb.qo, out, gb.ws, page_size=1, req_rows=gb.rows,
                                  max_kv_len=spec.max_kv_len,
                                  flags=msg.MSG_ATTN_DECODE_ONLY | msg.MSG_ATTN_REUSE_PLAN)
    torch.cuda.synchronize()
    st, info = gb.status()
    assert st == msg.MSG_OK, info
    assert np.array_equal(wl.torch_to_bits(out), ref["out"])
    assert np.array_equal(wl.torch_to_bits(k_pool), ref["k_pool"])
    assert np.array_equal(wl.torch_to_bits(v_pool), ref["v_pool"])
    assert_attn_close(wl.torch_to_bits(out), oracle_small(spec, host)["out"], "fused tp")


def test_tp_rank_reads_its_slice_of_the_full_pools():
    """Rank 1 of tp = 2 on views of a full layer: q heads 8..15 and KV heads
    4..7 of the pools (rows keep the full layer's stride).  Its store writes
    only heads 4..7 and its outputs match the full layer's query heads 8..15
    within tolerance, both checked against the oracle."""
    spec = _rand_spec(731, n_dec=14, n_ext=3, page_size=16)
    host = wl.host_tensors(spec)
    full = oracle_small(spec, host)
    dev = "cuda"
    gb = GpuBatch(spec, dev)
    q = wl.bits_to_torch(host["q"], dev)[:, 8:16]
    k_new = wl.bits_to_torch(host["k_new"], dev)[:, 4:8]
    v_new = wl.bits_to_torch(host["v_new"], dev)[:, 4:8]
    k_pool, v_pool = wl.bits_to_torch(host["k_pool"], dev), wl.bits_to_torch(host["v_pool"], dev)
    loc = gb.plan()
    msg.msg_store_kv(k_new, v_new, k_pool[:, 4:8], v_pool[:, 4:8], loc, dev_status=gb.ws)
    out = torch.empty(q.shape[0], 8, 128, dtype=torch.bfloat16, device=dev)
    msg.msg_paged_attention(q, k_pool[:, 4:8], v_pool[:, 4:8], gb.page_table, gb.cached,
                            gb.extend, gb.qo, out, gb.ws, page_size=16, req_rows=gb.rows,
                            max_kv_len=spec.max_kv_len, flags=msg.MSG_ATTN_REUSE_PLAN)
    torch.cuda.synchronize()
    st, info = gb.status()
    assert st == msg.MSG_OK, info
    kp, vp = wl.torch_to_bits(k_pool), wl.torch_to_bits(v_pool)
    assert np.array_equal(kp[:, 4:8], full["k_pool"][:, 4:8])
    assert np.array_equal(vp[:, 4:8], full["v_pool"][:, 4:8])
    assert np.array_equal(kp[:, :4], host["k_pool"][:, :4])     # the other rank's heads untouched
    assert_attn_close(wl.torch_to_bits(out), full["out"][:, 8:16], "tp rank 1 of 2")

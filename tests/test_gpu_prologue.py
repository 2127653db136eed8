"""GPU parity of the fused attention prologue (q_norm / k_norm, rotary
embedding, store_kv of the rotated K and of V) and of the rotary cache
("Mini-SGLang 完整剖析" 4.5.6, 4.6.7; "第 0 步" 四个算子).

Bars: the cache within one fp32 ulp of the oracle's (both round cos / sin of
the same fp32 angle once); V and the untouched pool slots bit-exact; q and the
stored K within one bf16 ulp of the fp64 oracle (fp32 arithmetic and a single
round-to-nearest), plus an absolute 2^-20 of the head's largest value for
outputs that cancel to near zero; at least 99% of them within half an ulp."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_gqa_store_gb300 as msg
from paged_kv_gqa_store_gb300 import workload as wl

pytestmark = pytest.mark.gpu

HQ, HKV, D = 16, 8, 128
THETA, EPS = 1e6, 1e-6


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    msg.load_library()


def _ulp_bf16(v):
    a = np.abs(v)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, 2.0 ** (e - 7), 2.0 ** -133)


def _check_close(got_bits, ref, what):
    got = wl.bf16_bits_to_f64(got_bits).reshape(ref.shape)
    err = np.abs(got - ref)
    head_max = np.abs(ref).max(axis=-1, keepdims=True)
    assert np.isfinite(got).all(), what
    assert (err <= _ulp_bf16(ref) + 2.0 ** -20 * head_max).all(), \
        f"{what}: worst {float((err / (_ulp_bf16(ref) + 1e-300)).max()):.3f} ulp"
    half = (err <= 0.5 * _ulp_bf16(ref) * (1 + 1e-3) + 2.0 ** -20 * head_max).mean()
    assert half >= 0.99, f"{what}: only {half:.4f} within half an ulp"


def test_rope_cache_matches_oracle():
    max_pos = 40000
    got = msg.msg_rope_cos_sin_cache(THETA, D, max_pos).cpu().numpy()
    want = oracle.rope_cos_sin_cache(THETA, D, max_pos)
    gu, wu = got.view(np.int32).astype(np.int64), want.view(np.int32).astype(np.int64)
    assert np.abs(gu - wu).max() <= 1
    assert (gu != wu).mean() < 1e-4


def _inputs(seed, T, max_pos, num_slots):
    rng = np.random.default_rng(seed)
    qkv = wl.random_bf16(rng, (T, HQ + 2 * HKV, D))
    qw = wl.f32_to_bf16_bits(rng.uniform(0.5, 1.5, D).astype(np.float32))
    kw = wl.f32_to_bf16_bits(rng.uniform(0.5, 1.5, D).astype(np.float32))
    pos = rng.integers(0, max_pos, size=T).astype(np.int32)
    loc = rng.choice(num_slots, size=T, replace=False).astype(np.int64)
    return qkv, qw, kw, pos, loc


@pytest.mark.parametrize("T,in_place,int64_loc", [(1, False, True), (67, True, False),
                                                  (1500, False, True)])
def test_prologue_matches_oracle(T, in_place, int64_loc):
    max_pos, num_slots = 33000, 4096
    qkv, qw, kw, pos, loc = _inputs(900 + T, T, max_pos, num_slots)
    dev = "cuda"
    cs = msg.msg_rope_cos_sin_cache(THETA, D, max_pos)
    qkv_t = wl.bits_to_torch(qkv, dev)
    q_out = qkv_t[:, :HQ] if in_place else torch.empty(T, HQ, D, dtype=torch.bfloat16, device=dev)
    kp = torch.full((num_slots, HKV, D), 0, dtype=torch.int16, device=dev)
    kp.fill_(wl.CANARY_BF16 - 65536 if wl.CANARY_BF16 > 32767 else wl.CANARY_BF16)
    kp = kp.view(torch.bfloat16)
    vp = kp.clone()
    loc_t = torch.from_numpy(loc if int64_loc else loc.astype(np.int32)).to(dev)
    status = torch.zeros(4, dtype=torch.int32, device=dev)
    msg.msg_qk_norm_rope_store(qkv_t, torch.from_numpy(pos).to(dev), wl.bits_to_torch(qw, dev),
                               wl.bits_to_torch(kw, dev), EPS, cs, q_out, kp, vp, loc_t, HQ, HKV,
                               dev_status=status)
    torch.cuda.synchronize()
    assert msg.msg_read_device_status(status)[0] == msg.MSG_OK
    q_ref, k_ref, v_ref = oracle.qk_norm_rope(qkv, pos, qw, kw, EPS,
                                              oracle.rope_cos_sin_cache(THETA, D, max_pos),
                                              HQ, HKV, D)
    _check_close(wl.torch_to_bits(q_out), q_ref, "q")
    kpool, vpool = wl.torch_to_bits(kp), wl.torch_to_bits(vp)
    _check_close(kpool[loc], k_ref, "k")
    assert np.array_equal(vpool[loc], v_ref), "v"
    other = np.setdiff1d(np.arange(num_slots), loc)
    assert (kpool[other] == wl.CANARY_BF16).all() and (vpool[other] == wl.CANARY_BF16).all()
    if in_place:   # the k and v parts of qkv are left as they were
        assert np.array_equal(wl.torch_to_bits(qkv_t)[:, HQ:], qkv[:, HQ:])


def test_prologue_bad_position_and_slot_are_reported_and_skipped():
    T, max_pos, num_slots = 8, 100, 64
    qkv, qw, kw, pos, loc = _inputs(950, T, max_pos, num_slots)
    pos[3] = max_pos                       # outside the cache
    loc[5] = num_slots + 2                 # outside the pool
    dev = "cuda"
    cs = msg.msg_rope_cos_sin_cache(THETA, D, max_pos)
    qkv_t = wl.bits_to_torch(qkv, dev)
    q_out = torch.zeros(T, HQ, D, dtype=torch.bfloat16, device=dev)
    kp = torch.zeros(num_slots, HKV, D, dtype=torch.bfloat16, device=dev)
    vp = torch.zeros_like(kp)
    status = torch.zeros(4, dtype=torch.int32, device=dev)
    msg.msg_qk_norm_rope_store(qkv_t, torch.from_numpy(pos).to(dev), wl.bits_to_torch(qw, dev),
                               wl.bits_to_torch(kw, dev), EPS, cs, q_out, kp, vp,
                               torch.from_numpy(loc).to(dev), HQ, HKV, dev_status=status)
    st, info = msg.msg_read_device_status(status)
    assert st == msg.MSG_ERR_DEVICE_CHECK
    assert info[0] in (msg.MSG_DEV_BAD_POSITION, msg.MSG_DEV_SLOT_OUT_OF_RANGE)
    assert (wl.torch_to_bits(q_out)[3] == 0).all()          # token 3 not written
    assert wl.torch_to_bits(q_out)[5].any()                 # token 5's q still written
    good = np.setdiff1d(np.arange(T), [3, 5])
    assert wl.torch_to_bits(kp)[loc[good]].any(axis=(1, 2)).all()


def test_prologue_full_extend_batch_sampled():
    """The extend batch's token count (8 requests, ~18k new tokens) in the launch
    configuration the benchmark times; a sample of tokens checked."""
    spec = wl.config_extend()
    T = spec.total_q
    max_pos = int(spec.max_kv_len) + 1
    rng = np.random.default_rng(960)
    dev = "cuda"
    qkv_t = torch.randn(T, HQ + 2 * HKV, D, generator=torch.Generator(dev).manual_seed(961),
                        device=dev).to(torch.bfloat16)
    qw = wl.f32_to_bf16_bits(rng.uniform(0.5, 1.5, D).astype(np.float32))
    kw = wl.f32_to_bf16_bits(rng.uniform(0.5, 1.5, D).astype(np.float32))
    meta = oracle.metadata(spec.page_table, spec.cached_len, spec.extend_len, spec.req_rows)
    pos, loc = meta["positions"], meta["out_loc"]
    cs = msg.msg_rope_cos_sin_cache(THETA, D, max_pos)
    q_out = torch.empty(T, HQ, D, dtype=torch.bfloat16, device=dev)
    kp = torch.zeros(spec.num_slots, HKV, D, dtype=torch.bfloat16, device=dev)
    vp = torch.zeros_like(kp)
    msg.msg_qk_norm_rope_store(qkv_t, torch.from_numpy(pos).to(dev), wl.bits_to_torch(qw, dev),
                               wl.bits_to_torch(kw, dev), EPS, cs, q_out, kp, vp,
                               torch.from_numpy(loc).to(dev), HQ, HKV)
    torch.cuda.synchronize()
    pick = np.unique(np.concatenate([[0, T - 1], rng.integers(0, T, size=300)]))
    idx = torch.from_numpy(pick).to(dev)
    qkv_s = wl.torch_to_bits(qkv_t.index_select(0, idx))
    q_ref, k_ref, v_ref = oracle.qk_norm_rope(qkv_s, pos[pick], qw, kw, EPS,
                                              oracle.rope_cos_sin_cache(THETA, D, max_pos),
                                              HQ, HKV, D)
    _check_close(wl.torch_to_bits(q_out.index_select(0, idx)), q_ref, "q")
    sl = torch.from_numpy(loc[pick]).to(dev)
    _check_close(wl.torch_to_bits(kp.index_select(0, sl)), k_ref, "k")
    assert np.array_equal(wl.torch_to_bits(vp.index_select(0, sl)), v_ref)


@pytest.mark.parametrize("hq,hkv,T", [(8, 2, 300), (64, 8, 200), (448, 4, 40)])
def test_prologue_other_head_counts(hq, hkv, T):
    """Head counts other than 16 / 8: a narrow row (12 head rows a token), a wide
    one (80 rows: fewer warps and stages per CTA) and one whose two stages do not
    fit in shared memory (456 rows: the kernel that keeps rows in registers)."""
    max_pos, num_slots = 5000, 1024
    rng = np.random.default_rng(970 + hq)
    qkv = wl.random_bf16(rng, (T, hq + 2 * hkv, D))
    qw = wl.f32_to_bf16_bits(rng.uniform(0.5, 1.5, D).astype(np.float32))
    kw = wl.f32_to_bf16_bits(rng.uniform(0.5, 1.5, D).astype(np.float32))
    pos = rng.integers(0, max_pos, size=T).astype(np.int32)
    loc = rng.choice(num_slots, size=T, replace=False).astype(np.int64)
    dev = "cuda"
    cs = msg.msg_rope_cos_sin_cache(THETA, D, max_pos)
    q_out = torch.empty(T, hq, D, dtype=torch.bfloat16, device=dev)
    kp = torch.zeros(num_slots, hkv, D, dtype=torch.bfloat16, device=dev)
    vp = torch.zeros_like(kp)
    status = torch.zeros(4, dtype=torch.int32, device=dev)
    msg.msg_qk_norm_rope_store(wl.bits_to_torch(qkv, dev), torch.from_numpy(pos).to(dev),
                               wl.bits_to_torch(qw, dev), wl.bits_to_torch(kw, dev), EPS, cs,
                               q_out, kp, vp, torch.from_numpy(loc).to(dev), hq, hkv,
                               dev_status=status)
    torch.cuda.synchronize()
    assert msg.msg_read_device_status(status)[0] == msg.MSG_OK
    q_ref, k_ref, v_ref = oracle.qk_norm_rope(qkv, pos, qw, kw, EPS,
                                              oracle.rope_cos_sin_cache(THETA, D, max_pos),
                                              hq, hkv, D)
    _check_close(wl.torch_to_bits(q_out), q_ref, "q")
    _check_close(wl.torch_to_bits(kp)[loc], k_ref, "k")
    assert np.array_equal(wl.torch_to_bits(vp)[loc], v_ref), "v"
    other = np.setdiff1d(np.arange(num_slots), loc)
    assert not wl.torch_to_bits(kp)[other].any() and not wl.torch_to_bits(vp)[other].any()


def test_prologue_then_fused_decode_reads_the_fresh_step_inputs():
    """The fused decode call (msg_paged_attention_store with a reused plan)
    launched straight after the prologue kernel that writes its q, k_new and
    v_new.  The prologue lets dependent kernels start before it writes them,
    and the decode kernel gathers its first older pool rows before waiting for
    it, so a read of q or of a newest row before that wait would show up as a
    stale value.  Three repeats of the step with new QKV projections: each
    step's output equals the oracle run on that step's q / k_new / v_new, and
    the pools bit for bit."""
    from _harness import GpuBatch, assert_attn_close
    rng = np.random.default_rng(612)
    n = 600
    cached = rng.integers(1, 300, size=n)
    cached[:4] = (9000, 4000, 2500, 1200)
    spec = wl.make_batch("prologue_fused", 612, cached, np.ones(n, np.int32), 1,
                         num_pages=int(cached.sum()) + n + 16)
    host = wl.host_tensors(spec)
    dev = "cuda"
    gb = GpuBatch(spec, dev)
    gb.plan()
    T = spec.total_q
    kp, vp = wl.bits_to_torch(host["k_pool"], dev), wl.bits_to_torch(host["v_pool"], dev)
    kp_h, vp_h = host["k_pool"].copy(), host["v_pool"].copy()
    max_pos = int(cached.max()) + 2
    cs = msg.msg_rope_cos_sin_cache(THETA, D, max_pos)
    qw = wl.f32_to_bf16_bits(rng.uniform(0.5, 1.5, D).astype(np.float32))
    kw = wl.f32_to_bf16_bits(rng.uniform(0.5, 1.5, D).astype(np.float32))
    qw_t, kw_t = wl.bits_to_torch(qw, dev), wl.bits_to_torch(kw, dev)
    pos = torch.from_numpy(cached.astype(np.int32)).to(dev)        # each new token's position
    rows = torch.arange(T, dtype=torch.int64, device=dev)          # k_new / v_new row t <- token t
    q = torch.empty(T, HQ, D, dtype=torch.bfloat16, device=dev)
    k_new = torch.empty(T, HKV, D, dtype=torch.bfloat16, device=dev)
    v_new = torch.empty_like(k_new)
    out = torch.empty_like(q)
    pstat = torch.zeros(4, dtype=torch.int32, device=dev)
    meta = oracle.metadata(spec.page_table, spec.cached_len, spec.extend_len, spec.req_rows)
    for step in range(3):
        qkv = wl.bits_to_torch(wl.random_bf16(rng, (T, HQ + 2 * HKV, D)), dev)
        torch.cuda.synchronize()
        msg.msg_qk_norm_rope_store(qkv, pos, qw_t, kw_t, EPS, cs, q, k_new, v_new, rows, HQ, HKV,
                                   dev_status=pstat)
        msg.msg_paged_attention_store(q, k_new, v_new, kp, vp, gb.page_table, gb.cached,
                                      gb.extend, gb.qo, out, gb.ws, page_size=1,
                                      req_rows=gb.rows, max_kv_len=spec.max_kv_len,
                                      flags=msg.MSG_ATTN_DECODE_ONLY | msg.MSG_ATTN_REUSE_PLAN)
        torch.cuda.synchronize()
        st, info = gb.status()
        assert st == msg.MSG_OK, info
        assert msg.msg_read_device_status(pstat)[0] == msg.MSG_OK
        qh, kh, vh = (wl.torch_to_bits(t) for t in (q, k_new, v_new))
        oracle.store_kv(kh, vh, meta["out_loc"], kp_h, vp_h)
        ref = oracle.paged_attention(qh, kp_h, vp_h, spec.page_table, spec.cached_len,
                                     meta["qo_indptr"], HQ, HKV, D, req_rows=spec.req_rows)
        assert_attn_close(wl.torch_to_bits(out), ref, f"step {step}")
        assert np.array_equal(wl.torch_to_bits(kp), kp_h), f"k pool, step {step}"
        assert np.array_equal(wl.torch_to_bits(vp), vp_h), f"v pool, step {step}"

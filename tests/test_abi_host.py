"""Host-side checks of the C ABI, no GPU needed: the library builds for sm_103a,
loads, exports every entry point include/msg.h declares, and rejects bad
arguments with the documented status before touching the device."""
import ctypes
import subprocess

import pytest

import paged_kv_gqa_store_gb300 as msg
from paged_kv_gqa_store_gb300 import build as msg_build


@pytest.fixture(scope="module")
def lib():
    msg_build.build()
    return msg.load_library()


def test_header_declares_the_boundary():
    names = msg.header_functions()
    for want in ("msg_plan", "msg_store_kv", "msg_paged_attention", "msg_workspace_size",
                 "msg_read_device_status", "msg_clear_device_status", "msg_status_string",
                 "msg_version"):
        assert want in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", msg.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in msg.header_functions():
        assert name in exported, name
        assert getattr(lib, name) is not None


def test_status_strings_and_version(lib):
    assert msg.msg_status_string(0) == "ok"
    for code in (-1, -2, -3, -4, -5, -6):
        assert msg.msg_status_string(code) != "unknown status"
    assert msg.msg_version() >= 100


def test_survey_boundary_names(lib):
    # the boundary's planned names: the workspace size with a split bound, and
    # the device-error read; same sizes and codes as msg_workspace_size and the
    # status block
    for reqs, q in ((1, 1), (64, 64), (256, 18432)):
        for hq in (16, 8, 2):
            assert lib.msg_paged_attention_workspace_size(reqs, q, hq, 128, 64) == \
                lib.msg_workspace_size(reqs, q, hq, 128)
    assert lib.msg_paged_attention_workspace_size(4, 4, 16, 128, 0) == 0
    assert lib.msg_get_device_error(None, None) == msg.MSG_ERR_INVALID_ARG


def test_workspace_size_monotone(lib):
    a = msg.msg_workspace_size(64, 64)
    b = msg.msg_workspace_size(256, 18432)
    assert 0 < a < b
    assert lib.msg_workspace_size(-1, 0, 16, 128) == 0


FAKE = 1 << 20          # a 16-byte-aligned fake device address, never dereferenced


def _attn(lib, **kw):
    a = dict(q=FAKE, q_row_stride=2048, k_pool=FAKE, v_pool=FAKE, pool_row_stride=1024,
             num_slots=100, page_table=FAKE, page_table_stride=32, req_rows=None,
             cached_len=FAKE, extend_len=FAKE, qo_indptr=FAKE, num_reqs=2, total_q=2,
             max_kv_len=0, page_size=1, num_qo_heads=16, num_kv_heads=8, head_dim=128,
             scale=0.088, out=FAKE, workspace=FAKE, workspace_bytes=1 << 30, flags=0,
             stream=None)
    a.update(kw)
    return lib.msg_paged_attention(*a.values())


@pytest.mark.parametrize("kw,status", [
    (dict(head_dim=64), msg.MSG_ERR_UNSUPPORTED),
    (dict(num_qo_heads=24), msg.MSG_ERR_UNSUPPORTED),
    (dict(num_qo_heads=6, num_kv_heads=3), msg.MSG_ERR_UNSUPPORTED),
    (dict(num_qo_heads=16, num_kv_heads=4), msg.MSG_ERR_UNSUPPORTED),    # GQA group 4
    (dict(num_qo_heads=32, num_kv_heads=16), msg.MSG_ERR_UNSUPPORTED),   # more than 8 KV heads
    (dict(num_qo_heads=12, num_kv_heads=6), msg.MSG_ERR_UNSUPPORTED),    # not a slice of 8
    (dict(num_qo_heads=16, num_kv_heads=16), msg.MSG_ERR_UNSUPPORTED),
    (dict(page_size=3), msg.MSG_ERR_UNSUPPORTED),
    (dict(page_size=256), msg.MSG_ERR_UNSUPPORTED),
    (dict(num_reqs=-1), msg.MSG_ERR_INVALID_ARG),
    (dict(scale=0.0), msg.MSG_ERR_INVALID_ARG),
    (dict(flags=msg.MSG_ATTN_DECODE_ONLY | msg.MSG_ATTN_EXTEND_ONLY), msg.MSG_ERR_INVALID_ARG),
    (dict(flags=64), msg.MSG_ERR_INVALID_ARG),
    (dict(q=None), msg.MSG_ERR_INVALID_ARG),
    (dict(q_row_stride=100), msg.MSG_ERR_INVALID_ARG),
    (dict(q=FAKE + 8), msg.MSG_ERR_ALIGNMENT),
    (dict(pool_row_stride=1028), msg.MSG_ERR_ALIGNMENT),
    (dict(workspace=None), msg.MSG_ERR_WORKSPACE),
    (dict(workspace_bytes=1024), msg.MSG_ERR_WORKSPACE),
    (dict(num_reqs=0), msg.MSG_OK),
    (dict(total_q=0), msg.MSG_OK),
])
def test_attention_argument_validation(lib, kw, status):
    assert _attn(lib, **kw) == status


def _attn_store(lib, **kw):
    a = dict(q=FAKE, q_row_stride=2048, k_new=FAKE, v_new=FAKE, kv_row_stride=1024, k_pool=FAKE,
             v_pool=FAKE, pool_row_stride=1024, num_slots=100, page_table=FAKE,
             page_table_stride=32, req_rows=None, cached_len=FAKE, extend_len=FAKE,
             qo_indptr=FAKE, num_reqs=2, total_q=2, max_kv_len=0, page_size=1, num_qo_heads=16,
             num_kv_heads=8, head_dim=128, scale=0.088, out=FAKE, workspace=FAKE,
             workspace_bytes=1 << 30, flags=msg.MSG_ATTN_DECODE_ONLY, stream=None)
    a.update(kw)
    return lib.msg_paged_attention_store(*a.values())


@pytest.mark.parametrize("kw,status", [
    (dict(flags=0), msg.MSG_ERR_INVALID_ARG),                 # decode-only batches alone
    (dict(flags=msg.MSG_ATTN_EXTEND_ONLY), msg.MSG_ERR_INVALID_ARG),
    (dict(k_new=None), msg.MSG_ERR_INVALID_ARG),
    (dict(v_new=None), msg.MSG_ERR_INVALID_ARG),
    (dict(kv_row_stride=512), msg.MSG_ERR_INVALID_ARG),
    (dict(k_new=FAKE + 8), msg.MSG_ERR_ALIGNMENT),
    (dict(kv_row_stride=1028), msg.MSG_ERR_ALIGNMENT),
    (dict(head_dim=64), msg.MSG_ERR_UNSUPPORTED),
    (dict(page_size=3), msg.MSG_ERR_UNSUPPORTED),
    (dict(num_reqs=0), msg.MSG_OK),
])
def test_fused_store_attention_argument_validation(lib, kw, status):
    """msg_paged_attention_store: the store fused into the decode kernel takes
    decode-only batches and the step's new K / V rows (16-byte aligned)."""
    assert _attn_store(lib, **kw) == status


def _store(lib, **kw):
    a = dict(k=FAKE, v=FAKE, kv_row_stride=1024, k_pool=FAKE, v_pool=FAKE,
             pool_row_stride=1024, num_slots=10, out_loc=FAKE, is64=0, num_tokens=3,
             num_kv_heads=8, head_dim=128, dev_status=None, stream=None)
    a.update(kw)
    return lib.msg_store_kv(*a.values())


@pytest.mark.parametrize("kw,status", [
    (dict(num_tokens=0), msg.MSG_OK),
    (dict(num_tokens=-1), msg.MSG_ERR_INVALID_ARG),
    (dict(k=None), msg.MSG_ERR_INVALID_ARG),
    (dict(kv_row_stride=512), msg.MSG_ERR_INVALID_ARG),
    (dict(k=FAKE + 2), msg.MSG_ERR_ALIGNMENT),
    (dict(pool_row_stride=1030), msg.MSG_ERR_ALIGNMENT),
    (dict(num_kv_heads=1, head_dim=4, kv_row_stride=8, pool_row_stride=8), msg.MSG_ERR_UNSUPPORTED),
])
def test_store_argument_validation(lib, kw, status):
    assert _store(lib, **kw) == status


def test_plan_argument_validation(lib):
    P = FAKE
    assert lib.msg_plan(P, 32, None, P, P, -1, 0, 10, None, None, 0, None, P, 1 << 20, None) \
        == msg.MSG_ERR_INVALID_ARG
    assert lib.msg_plan(P, 32, None, P, P, 4, 4, 10, None, None, 0, None, None, 1 << 20, None) \
        == msg.MSG_ERR_WORKSPACE
    assert lib.msg_plan(P, 32, None, P, P, 4, 4, 10, None, None, 0, None, P, 16, None) \
        == msg.MSG_ERR_WORKSPACE


def _kv(**kw):
    a = dict(kind=msg.MSG_KV_RAGGED, page_size=1, table=FAKE, table_stride=0, table_len=-1,
             req_rows=None, indptr=FAKE)
    a.update(kw)
    return msg._KvIndexC(*a.values())


@pytest.mark.parametrize("kw,status", [
    (dict(kind=3), msg.MSG_ERR_UNSUPPORTED),
    (dict(page_size=3), msg.MSG_ERR_UNSUPPORTED),
    (dict(page_size=256), msg.MSG_ERR_UNSUPPORTED),
    (dict(indptr=None), msg.MSG_ERR_INVALID_ARG),
    (dict(kind=msg.MSG_KV_PAGE_TABLE, table_stride=-1), msg.MSG_ERR_INVALID_ARG),
])
def test_kv_index_validation(lib, kw, status):
    c = _kv(**kw)
    assert lib.msg_plan_ex(ctypes.byref(c), FAKE, FAKE, 2, 2, 10, None, None, 0, None, FAKE,
                           1 << 20, None) == status
    a = dict(q=FAKE, q_row_stride=2048, k_pool=FAKE, v_pool=FAKE, pool_row_stride=1024,
             num_slots=100, kv=ctypes.byref(c), cached_len=FAKE, extend_len=FAKE,
             qo_indptr=FAKE, num_reqs=2, total_q=2, max_kv_len=0, num_qo_heads=16,
             num_kv_heads=8, head_dim=128, scale=0.088, out=FAKE, workspace=FAKE,
             workspace_bytes=1 << 30, flags=0, stream=None)
    assert lib.msg_paged_attention_ex(*a.values()) == status


def test_kv_index_null_descriptor(lib):
    assert lib.msg_plan_ex(None, FAKE, FAKE, 2, 2, 10, None, None, 0, None, FAKE, 1 << 20,
                           None) == msg.MSG_ERR_INVALID_ARG


@pytest.mark.parametrize("args,status", [
    (dict(kind=msg.MSG_KV_TOKEN_TABLE), msg.MSG_ERR_UNSUPPORTED),
    (dict(page_size=5), msg.MSG_ERR_UNSUPPORTED),
    (dict(num_reqs=-1), msg.MSG_ERR_INVALID_ARG),
    (dict(out_indptr=None), msg.MSG_ERR_INVALID_ARG),
    (dict(num_reqs=0, out_indptr=None, kind=msg.MSG_KV_PAGE_TABLE), msg.MSG_OK),
])
def test_build_kv_index_validation(lib, args, status):
    a = dict(kind=msg.MSG_KV_RAGGED, page_size=16, page_table=FAKE, page_table_stride=64,
             req_rows=None, cached_len=FAKE, extend_len=FAKE, num_reqs=2, out_table=FAKE,
             out_stride=0, out_capacity=100, out_indptr=FAKE, dev_status=None, stream=None)
    a.update(args)
    assert lib.msg_build_kv_index(*a.values()) == status


def _prologue(lib, **kw):
    a = dict(qkv=FAKE, qkv_row_stride=4096, num_tokens=3, positions=FAKE, q_norm_w=FAKE,
             k_norm_w=FAKE, eps=1e-6, cos_sin=FAKE, max_pos=100, q_out=FAKE,
             q_out_row_stride=2048, k_pool=FAKE, v_pool=FAKE, pool_row_stride=1024,
             num_slots=10, out_loc=FAKE, is64=1, num_qo_heads=16, num_kv_heads=8,
             head_dim=128, dev_status=None, stream=None)
    a.update(kw)
    return lib.msg_qk_norm_rope_store(*a.values())


@pytest.mark.parametrize("kw,status", [
    (dict(num_tokens=0), msg.MSG_OK),
    (dict(num_tokens=-1), msg.MSG_ERR_INVALID_ARG),
    (dict(head_dim=64, qkv_row_stride=2048, q_out_row_stride=1024, pool_row_stride=512),
     msg.MSG_ERR_UNSUPPORTED),
    (dict(qkv_row_stride=4000), msg.MSG_ERR_INVALID_ARG),
    (dict(eps=-1.0), msg.MSG_ERR_INVALID_ARG),
    (dict(max_pos=0), msg.MSG_ERR_INVALID_ARG),
    (dict(positions=None), msg.MSG_ERR_INVALID_ARG),
    (dict(qkv=FAKE + 8), msg.MSG_ERR_ALIGNMENT),
    (dict(qkv_row_stride=4100), msg.MSG_ERR_ALIGNMENT),
])
def test_prologue_argument_validation(lib, kw, status):
    assert _prologue(lib, **kw) == status


@pytest.mark.parametrize("theta,d,n,status", [
    (0.0, 128, 10, msg.MSG_ERR_INVALID_ARG), (1e6, 127, 10, msg.MSG_ERR_INVALID_ARG),
    (1e6, 128, 0, msg.MSG_ERR_INVALID_ARG)])
def test_rope_cache_argument_validation(lib, theta, d, n, status):
    assert lib.msg_rope_cos_sin_cache(theta, d, n, FAKE, None) == status


# ------------------------------------------------------------------ sampler
def _sample(lib, **kw):
    a = dict(logits=FAKE, dtype=msg.MSG_DTYPE_BF16, stride=152000, batch=4, vocab=151936,
             temperatures=FAKE, top_k=None, top_p=None, uniforms=FAKE, tokens=FAKE,
             ws=FAKE, ws_bytes=1 << 24, dev_status=None, stream=None)
    a.update(kw)
    return lib.msg_sample(*a.values())


@pytest.mark.parametrize("kw,status", [
    (dict(batch=0), msg.MSG_OK),
    (dict(batch=-1), msg.MSG_ERR_INVALID_ARG),
    (dict(dtype=7), msg.MSG_ERR_UNSUPPORTED),
    (dict(vocab=0), msg.MSG_ERR_INVALID_ARG),
    (dict(stride=100000), msg.MSG_ERR_INVALID_ARG),
    (dict(vocab=500000, stride=500000), msg.MSG_ERR_UNSUPPORTED),
    (dict(logits=None), msg.MSG_ERR_INVALID_ARG),
    (dict(tokens=None), msg.MSG_ERR_INVALID_ARG),
    (dict(uniforms=None), msg.MSG_ERR_INVALID_ARG),
    (dict(logits=FAKE + 1), msg.MSG_ERR_ALIGNMENT),
    (dict(dtype=msg.MSG_DTYPE_F32, logits=FAKE + 2), msg.MSG_ERR_ALIGNMENT),
    (dict(ws=None), msg.MSG_ERR_WORKSPACE),
    (dict(ws_bytes=1000), msg.MSG_ERR_WORKSPACE),
    (dict(ws=FAKE + 8), msg.MSG_ERR_ALIGNMENT),
])
def test_sample_argument_validation(lib, kw, status):
    assert _sample(lib, **kw) == status


def test_sampling_args_match_the_pages_prepare():
    # the binding's host half of Sampler.prepare against the oracle's statement
    import numpy as np
    import oracle
    cases = [([0.0, 0.0], [-1, 5], [1.0, 0.5]),
             ([0.7, 0.0, 1.2], [-1, 0, -3], [1.0, 1.0, 2.0]),
             ([1.0, 1.0], [50, -1], [0.0, 0.95]),
             ([0.5], [10**6], [1e-9]),
             ([0.0, 0.0], [-1, -1], [1.0, 0.9]),
             ([0.8, 1.5], [1, 1], [1.0, 1.0]),
             ([0.8, 1.5, 0.0], [1, 3, 1], [1.0, 1.0, 0.7])]
    for t, k, p in cases:
        got = msg.sampling_args(t, k, p, 1000, device="cpu")
        want = oracle.sampling_args(t, k, p, 1000)
        for g, w in zip(got, want):
            assert (g is None) == (w is None)
            if g is not None:
                assert np.array_equal(g.numpy(), w)


def test_sample_workspace_size(lib):
    per_row = msg.msg_sample_workspace_size(1, 151936)
    assert 8 * 596 <= per_row <= 16 * 1024
    assert msg.msg_sample_workspace_size(256, 151936) == 256 * per_row
    assert msg.msg_sample_workspace_size(0, 151936) == 0
    assert msg.msg_sample_workspace_size(4, 0) == 0
    assert msg.msg_sample_workspace_size(4, 425985) == 0

// abi.cu -- the extern "C" entry points declared in include/msg.h: argument
// validation, workspace carving and kernel launches.  No entry point allocates
// memory, synchronises the stream (except msg_read_device_status, which exists
// to do so) or lets an exception out.
#include <math.h>
#include <string.h>

#include "internal.cuh"

namespace msg {

int device_sm_count() {
  static int cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      n = 1;
    cache[dev] = n;
  }
  return cache[dev];
}

}  // namespace msg

namespace {

using namespace msg;

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_heads(int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim) {
  if (num_qo_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0) return MSG_ERR_INVALID_ARG;
  if (head_dim != kHeadDim) return MSG_ERR_UNSUPPORTED;
  // the full layer (8 KV heads) or a tensor-parallel slice of it, GQA group 2
  if (num_kv_heads != 8 && num_kv_heads != 4 && num_kv_heads != 2 && num_kv_heads != 1)
    return MSG_ERR_UNSUPPORTED;
  if (num_qo_heads != kGroup * num_kv_heads) return MSG_ERR_UNSUPPORTED;
  return MSG_OK;
}

int from_cuda(cudaError_t e) { return e == cudaSuccess ? MSG_OK : MSG_ERR_CUDA; }

bool pow2_page(int32_t page_size) {
  return page_size >= 1 && page_size <= 128 && (page_size & (page_size - 1)) == 0;
}

int32_t log2_page(int32_t page_size) {
  int32_t shift = 0;
  while ((1 << shift) < page_size) ++shift;
  return shift;
}

KvIndex token_table(const int32_t *page_table, int64_t stride, const int32_t *req_rows,
                    int32_t page_size) {
  KvIndex x{};
  x.table = page_table;
  x.stride = stride;
  x.len = -1;
  x.req_rows = req_rows;
  x.indptr = nullptr;
  x.kind = MSG_KV_TOKEN_TABLE;
  x.page_size = page_size;
  x.page_shift = log2_page(page_size);
  return x;
}

// Validate a caller's msg_kv_index (host struct) into the device-side form.
int make_kv(const msg_kv_index *kv, KvIndex &x) {
  if (kv == nullptr) return MSG_ERR_INVALID_ARG;
  if (kv->kind != MSG_KV_TOKEN_TABLE && kv->kind != MSG_KV_PAGE_TABLE && kv->kind != MSG_KV_RAGGED)
    return MSG_ERR_UNSUPPORTED;
  if (!pow2_page(kv->page_size)) return MSG_ERR_UNSUPPORTED;
  if (kv->kind == MSG_KV_RAGGED ? kv->indptr == nullptr : kv->table_stride < 0)
    return MSG_ERR_INVALID_ARG;
  x = token_table(kv->table, kv->kind == MSG_KV_RAGGED ? 0 : kv->table_stride,
                  kv->kind == MSG_KV_RAGGED ? nullptr : kv->req_rows, kv->page_size);
  x.kind = kv->kind;
  x.len = kv->table_len < 0 ? -1 : kv->table_len;
  x.indptr = kv->kind == MSG_KV_RAGGED ? kv->indptr : nullptr;
  return MSG_OK;
}

int plan_impl(const KvIndex &kv, const int32_t *cached_len, const int32_t *extend_len,
              int32_t num_reqs, int64_t total_q, int64_t num_slots, int32_t *qo_indptr_out,
              void *out_loc_out, int32_t out_loc_is_int64, int32_t *positions_out,
              void *workspace, size_t workspace_bytes, void *stream) {
  if (num_reqs < 0 || total_q < 0 || total_q > INT32_MAX || num_slots < 0)
    return MSG_ERR_INVALID_ARG;
  if (workspace == nullptr) return MSG_ERR_WORKSPACE;
  const WsLayout L = ws_layout(num_reqs, total_q, 0, 0);
  if (workspace_bytes < L.plan_end) return MSG_ERR_WORKSPACE;
  if (num_reqs > 0 && (cached_len == nullptr || extend_len == nullptr)) return MSG_ERR_INVALID_ARG;
  if (total_q > 0 && (out_loc_out || positions_out) && kv.table == nullptr)
    return MSG_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  PlanParams pp{};
  pp.kv = kv;
  pp.cached_len = cached_len;
  pp.extend_len = extend_len;
  pp.qo_in = nullptr;
  pp.num_reqs = num_reqs;
  pp.total_q = total_q;
  pp.status = reinterpret_cast<int32_t *>(ws + L.status);
  pp.hdr = reinterpret_cast<PlanHeader *>(ws + L.header);
  pp.qo_ws = reinterpret_cast<int32_t *>(ws + L.qo_indptr);
  pp.qo_out = qo_indptr_out;
  pp.dec_req = reinterpret_cast<int32_t *>(ws + L.dec_req);
  pp.dec_start = reinterpret_cast<int64_t *>(ws + L.dec_start);
  pp.dec_row = reinterpret_cast<int64_t *>(ws + L.dec_row);
  pp.dec_qrow = reinterpret_cast<int32_t *>(ws + L.dec_qrow);
  pp.counters = reinterpret_cast<int32_t *>(ws + L.counters);
  pp.gcounters = reinterpret_cast<int32_t *>(ws + L.gcounters);
  pp.ext_tiles = reinterpret_cast<int32_t *>(ws + L.ext_tiles);
  pp.max_tiles = L.max_tiles;
  int rc = from_cuda(launch_plan(pp, s));
  if (rc != MSG_OK) return rc;
  if (total_q > 0 && (out_loc_out || positions_out)) {
    TokenMetaParams tp{};
    tp.kv = kv;
    tp.cached_len = cached_len;
    tp.qo_ws = pp.qo_ws;
    tp.num_reqs = num_reqs;
    tp.total_q = total_q;
    tp.num_slots = num_slots;
    tp.out_loc = out_loc_out;
    tp.out_loc_is_int64 = out_loc_is_int64 ? 1 : 0;
    tp.positions = positions_out;
    tp.status = pp.status;
    rc = from_cuda(launch_token_meta(tp, s));
  }
  return rc;
}

int attention_impl(const void *q, int64_t q_row_stride, const void *k_pool, const void *v_pool,
                   int64_t pool_row_stride, int64_t num_slots, const KvIndex &kv,
                   const int32_t *cached_len, const int32_t *extend_len,
                   const int32_t *qo_indptr, int32_t num_reqs, int64_t total_q,
                   int32_t max_kv_len, int32_t num_qo_heads, int32_t num_kv_heads,
                   int32_t head_dim, float scale, void *out, void *workspace,
                   size_t workspace_bytes, uint32_t flags, void *stream,
                   const void *k_new = nullptr, const void *v_new = nullptr,
                   int64_t kv_row_stride = 0);

}  // namespace

extern "C" {

const char *msg_status_string(int status) {
  switch (status) {
    case MSG_OK: return "ok";
    case MSG_ERR_INVALID_ARG: return "invalid argument (null pointer, negative size or bad stride)";
    case MSG_ERR_UNSUPPORTED: return "unsupported shape (needs head_dim 128, 2 query heads per KV "
                                     "head with 8, 4, 2 or 1 KV heads, page_size a power of two "
                                     "<= 128)";
    case MSG_ERR_ALIGNMENT: return "pointer or row stride not 16-byte aligned";
    case MSG_ERR_WORKSPACE: return "workspace missing or smaller than msg_workspace_size()";
    case MSG_ERR_CUDA: return "CUDA runtime error (launch or copy failed)";
    case MSG_ERR_DEVICE_CHECK: return "a kernel recorded a device-side error in the status block";
    default: return "unknown status";
  }
}

int msg_version(void) { return 100; }

size_t msg_workspace_size(int32_t max_reqs, int64_t max_total_q, int32_t num_qo_heads,
                          int32_t head_dim) {
  if (max_reqs < 0 || max_total_q < 0 || num_qo_heads <= 0 || head_dim <= 0) return 0;
  return ws_layout(max_reqs, max_total_q, num_qo_heads, head_dim).total_split;
}

size_t msg_paged_attention_workspace_size(int32_t max_reqs, int64_t max_total_q,
                                          int32_t num_qo_heads, int32_t head_dim,
                                          int32_t max_splits) {
  // the split count is the library's choice and every one it makes fits
  if (max_splits < 1) return 0;
  return msg_workspace_size(max_reqs, max_total_q, num_qo_heads, head_dim);
}

int msg_plan(const int32_t *page_table, int64_t page_table_stride, const int32_t *req_rows,
             const int32_t *cached_len, const int32_t *extend_len, int32_t num_reqs,
             int64_t total_q, int64_t num_slots, int32_t *qo_indptr_out, void *out_loc_out,
             int32_t out_loc_is_int64, int32_t *positions_out, void *workspace,
             size_t workspace_bytes, void *stream) {
  if (page_table_stride < 0) return MSG_ERR_INVALID_ARG;
  return plan_impl(token_table(page_table, page_table_stride, req_rows, 1), cached_len, extend_len,
                   num_reqs, total_q, num_slots, qo_indptr_out, out_loc_out, out_loc_is_int64,
                   positions_out, workspace, workspace_bytes, stream);
}

int msg_plan_ex(const msg_kv_index *kv, const int32_t *cached_len, const int32_t *extend_len,
                int32_t num_reqs, int64_t total_q, int64_t num_slots, int32_t *qo_indptr_out,
                void *out_loc_out, int32_t out_loc_is_int64, int32_t *positions_out,
                void *workspace, size_t workspace_bytes, void *stream) {
  KvIndex x;
  const int rc = make_kv(kv, x);
  if (rc != MSG_OK) return rc;
  return plan_impl(x, cached_len, extend_len, num_reqs, total_q, num_slots, qo_indptr_out,
                   out_loc_out, out_loc_is_int64, positions_out, workspace, workspace_bytes,
                   stream);
}

int msg_store_kv(const void *k, const void *v, int64_t kv_row_stride, void *k_pool, void *v_pool,
                 int64_t pool_row_stride, int64_t num_slots, const void *out_loc,
                 int32_t out_loc_is_int64, int64_t num_tokens, int32_t num_kv_heads,
                 int32_t head_dim, int32_t *dev_status, void *stream) {
  if (num_tokens < 0 || num_slots < 0 || num_kv_heads <= 0 || head_dim <= 0)
    return MSG_ERR_INVALID_ARG;
  if (num_tokens == 0) return MSG_OK;
  if (!k || !v || !k_pool || !v_pool || !out_loc) return MSG_ERR_INVALID_ARG;
  const int64_t row = (int64_t)num_kv_heads * head_dim;
  if (kv_row_stride < row || pool_row_stride < row) return MSG_ERR_INVALID_ARG;
  if ((row * 2) % 16 != 0) return MSG_ERR_UNSUPPORTED;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_pool) || !aligned16(v_pool) ||
      kv_row_stride % 8 != 0 || pool_row_stride % 8 != 0)
    return MSG_ERR_ALIGNMENT;
  StoreParams sp{};
  sp.k = static_cast<const uint8_t *>(k);
  sp.v = static_cast<const uint8_t *>(v);
  sp.in_stride_bytes = kv_row_stride * 2;
  sp.k_pool = static_cast<uint8_t *>(k_pool);
  sp.v_pool = static_cast<uint8_t *>(v_pool);
  sp.pool_stride_bytes = pool_row_stride * 2;
  sp.num_slots = num_slots;
  sp.out_loc = out_loc;
  sp.out_loc_is_int64 = out_loc_is_int64 ? 1 : 0;
  sp.num_tokens = num_tokens;
  sp.row_chunks = (int32_t)(row * 2 / 16);
  sp.status = dev_status;
  return from_cuda(launch_store_kv(sp, static_cast<cudaStream_t>(stream)));
}

int msg_paged_attention(const void *q, int64_t q_row_stride, const void *k_pool,
                        const void *v_pool, int64_t pool_row_stride, int64_t num_slots,
                        const int32_t *page_table, int64_t page_table_stride,
                        const int32_t *req_rows, const int32_t *cached_len,
                        const int32_t *extend_len, const int32_t *qo_indptr, int32_t num_reqs,
                        int64_t total_q, int32_t max_kv_len, int32_t page_size,
                        int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                        float scale, void *out, void *workspace, size_t workspace_bytes,
                        uint32_t flags, void *stream) {
  const int rc = check_heads(num_qo_heads, num_kv_heads, head_dim);
  if (rc != MSG_OK) return rc;
  if (page_table_stride < 0) return MSG_ERR_INVALID_ARG;
  if (!pow2_page(page_size)) return MSG_ERR_UNSUPPORTED;
  return attention_impl(q, q_row_stride, k_pool, v_pool, pool_row_stride, num_slots,
                        token_table(page_table, page_table_stride, req_rows, page_size),
                        cached_len, extend_len, qo_indptr, num_reqs, total_q, max_kv_len,
                        num_qo_heads, num_kv_heads, head_dim, scale, out, workspace,
                        workspace_bytes, flags, stream);
}

int msg_paged_attention_store(const void *q, int64_t q_row_stride, const void *k_new,
                              const void *v_new, int64_t kv_row_stride, void *k_pool,
                              void *v_pool, int64_t pool_row_stride, int64_t num_slots,
                              const int32_t *page_table, int64_t page_table_stride,
                              const int32_t *req_rows, const int32_t *cached_len,
                              const int32_t *extend_len, const int32_t *qo_indptr,
                              int32_t num_reqs, int64_t total_q, int32_t max_kv_len,
                              int32_t page_size, int32_t num_qo_heads, int32_t num_kv_heads,
                              int32_t head_dim, float scale, void *out, void *workspace,
                              size_t workspace_bytes, uint32_t flags, void *stream) {
  const int rc = check_heads(num_qo_heads, num_kv_heads, head_dim);
  if (rc != MSG_OK) return rc;
  if (page_table_stride < 0 || k_new == nullptr || v_new == nullptr) return MSG_ERR_INVALID_ARG;
  if (!pow2_page(page_size)) return MSG_ERR_UNSUPPORTED;
  return attention_impl(q, q_row_stride, k_pool, v_pool, pool_row_stride, num_slots,
                        token_table(page_table, page_table_stride, req_rows, page_size),
                        cached_len, extend_len, qo_indptr, num_reqs, total_q, max_kv_len,
                        num_qo_heads, num_kv_heads, head_dim, scale, out, workspace,
                        workspace_bytes, flags, stream, k_new, v_new, kv_row_stride);
}

int msg_paged_attention_ex(const void *q, int64_t q_row_stride, const void *k_pool,
                           const void *v_pool, int64_t pool_row_stride, int64_t num_slots,
                           const msg_kv_index *kv, const int32_t *cached_len,
                           const int32_t *extend_len, const int32_t *qo_indptr,
                           int32_t num_reqs, int64_t total_q, int32_t max_kv_len,
                           int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                           float scale, void *out, void *workspace, size_t workspace_bytes,
                           uint32_t flags, void *stream) {
  int rc = check_heads(num_qo_heads, num_kv_heads, head_dim);
  if (rc != MSG_OK) return rc;
  KvIndex x;
  rc = make_kv(kv, x);
  if (rc != MSG_OK) return rc;
  return attention_impl(q, q_row_stride, k_pool, v_pool, pool_row_stride, num_slots, x,
                        cached_len, extend_len, qo_indptr, num_reqs, total_q, max_kv_len,
                        num_qo_heads, num_kv_heads, head_dim, scale, out, workspace,
                        workspace_bytes, flags, stream);
}

}  // extern "C"

namespace {

int attention_impl(const void *q, int64_t q_row_stride, const void *k_pool, const void *v_pool,
                   int64_t pool_row_stride, int64_t num_slots, const KvIndex &kv,
                   const int32_t *cached_len, const int32_t *extend_len,
                   const int32_t *qo_indptr, int32_t num_reqs, int64_t total_q,
                   int32_t max_kv_len, int32_t num_qo_heads, int32_t num_kv_heads,
                   int32_t head_dim, float scale, void *out, void *workspace,
                   size_t workspace_bytes, uint32_t flags, void *stream,
                   const void *k_new, const void *v_new, int64_t kv_row_stride) {
  int rc = MSG_OK;
  if (num_reqs < 0 || total_q < 0 || total_q > INT32_MAX || max_kv_len < 0 || num_slots < 0 ||
      !(scale > 0.f) || !isfinite(scale))
    return MSG_ERR_INVALID_ARG;
  if ((flags & ~(MSG_ATTN_REUSE_PLAN | MSG_ATTN_DECODE_ONLY | MSG_ATTN_EXTEND_ONLY)) ||
      ((flags & MSG_ATTN_DECODE_ONLY) && (flags & MSG_ATTN_EXTEND_ONLY)))
    return MSG_ERR_INVALID_ARG;
  if (num_reqs == 0 || total_q == 0) return MSG_OK;
  if (!q || !k_pool || !v_pool || !kv.table || !cached_len || !extend_len || !qo_indptr || !out)
    return MSG_ERR_INVALID_ARG;
  if ((k_new != nullptr) != (v_new != nullptr)) return MSG_ERR_INVALID_ARG;
  if (k_new != nullptr) {                       // the store fused into the decode kernel
    if (!(flags & MSG_ATTN_DECODE_ONLY)) return MSG_ERR_INVALID_ARG;
    if (kv_row_stride < (int64_t)num_kv_heads * head_dim) return MSG_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new) || kv_row_stride % 8 != 0) return MSG_ERR_ALIGNMENT;
  }
  const int64_t row = (int64_t)num_kv_heads * head_dim;
  if (q_row_stride < (int64_t)num_qo_heads * head_dim || pool_row_stride < row)
    return MSG_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(out) ||
      q_row_stride % 8 != 0 || pool_row_stride % 8 != 0)
    return MSG_ERR_ALIGNMENT;
  if (workspace == nullptr) return MSG_ERR_WORKSPACE;
  const WsLayout L = ws_layout(num_reqs, total_q, num_qo_heads, head_dim);
  if (workspace_bytes < L.total) return MSG_ERR_WORKSPACE;
  if (!aligned16(workspace)) return MSG_ERR_ALIGNMENT;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  int32_t *status = reinterpret_cast<int32_t *>(ws + L.status);
  if (!(flags & MSG_ATTN_REUSE_PLAN)) {
    PlanParams pp{};
    pp.kv = kv;
    pp.cached_len = cached_len;
    pp.extend_len = extend_len;
    pp.qo_in = qo_indptr;
    pp.num_reqs = num_reqs;
    pp.total_q = total_q;
    pp.status = status;
    pp.hdr = reinterpret_cast<PlanHeader *>(ws + L.header);
    pp.qo_ws = reinterpret_cast<int32_t *>(ws + L.qo_indptr);
    pp.qo_out = nullptr;
    pp.dec_req = reinterpret_cast<int32_t *>(ws + L.dec_req);
    pp.dec_start = reinterpret_cast<int64_t *>(ws + L.dec_start);
    pp.dec_row = reinterpret_cast<int64_t *>(ws + L.dec_row);
    pp.dec_qrow = reinterpret_cast<int32_t *>(ws + L.dec_qrow);
    pp.counters = reinterpret_cast<int32_t *>(ws + L.counters);
    pp.gcounters = reinterpret_cast<int32_t *>(ws + L.gcounters);
    pp.ext_tiles = reinterpret_cast<int32_t *>(ws + L.ext_tiles);
    pp.max_tiles = L.max_tiles;
    rc = from_cuda(launch_plan(pp, s));
    if (rc != MSG_OK) return rc;
  }

  AttnParams ap{};
  ap.q = static_cast<const uint16_t *>(q);
  ap.q_stride = q_row_stride;
  ap.k_pool = static_cast<const uint8_t *>(k_pool);
  ap.v_pool = static_cast<const uint8_t *>(v_pool);
  ap.pool_stride_bytes = pool_row_stride * 2;
  ap.num_slots = num_slots;
  ap.kv = kv;
  ap.cached_len = cached_len;
  ap.extend_len = extend_len;
  ap.qo_indptr = qo_indptr;
  ap.num_reqs = num_reqs;
  ap.total_q = total_q;
  ap.flags = flags;
  ap.page_size = kv.page_size;
  ap.page_shift = kv.page_shift;
  ap.num_qo_heads = num_qo_heads;
  ap.num_kv_heads = num_kv_heads;
  ap.scale_log2 = scale * 1.4426950408889634f;
  ap.out = static_cast<uint16_t *>(out);
  ap.status = status;
  ap.hdr = reinterpret_cast<const PlanHeader *>(ws + L.header);
  ap.k_new = static_cast<const uint8_t *>(k_new);
  ap.v_new = static_cast<const uint8_t *>(v_new);
  ap.new_stride_bytes = kv_row_stride * 2;
  ap.k_pool_w = static_cast<uint8_t *>(const_cast<void *>(k_pool));
  ap.v_pool_w = static_cast<uint8_t *>(const_cast<void *>(v_pool));
  ap.dec_req = reinterpret_cast<const int32_t *>(ws + L.dec_req);
  ap.dec_start = reinterpret_cast<const int64_t *>(ws + L.dec_start);
  ap.dec_row = reinterpret_cast<const int64_t *>(ws + L.dec_row);
  ap.dec_qrow = reinterpret_cast<const int32_t *>(ws + L.dec_qrow);
  ap.counters = reinterpret_cast<int32_t *>(ws + L.counters);
  ap.gcounters = reinterpret_cast<int32_t *>(ws + L.gcounters);
  ap.ext_tiles = reinterpret_cast<const int32_t *>(ws + L.ext_tiles);
  ap.part_lse = reinterpret_cast<float *>(ws + L.part_lse);
  ap.part_o = reinterpret_cast<float *>(ws + L.part_o);
  if (workspace_bytes >= L.total_split) {     // room for the extend key split
    ap.ext_items = reinterpret_cast<int32_t *>(ws + L.ext_items);
    ap.ext_lse = reinterpret_cast<float *>(ws + L.ext_lse);
    ap.ext_o = reinterpret_cast<float *>(ws + L.ext_o);
  }

  if (!(flags & MSG_ATTN_EXTEND_ONLY)) {
    int64_t grid = (int64_t)device_sm_count() * decode_ctas_per_sm(num_kv_heads);
    if (grid > max_decode_ctas(num_qo_heads)) grid = max_decode_ctas(num_qo_heads);
    if (max_kv_len > 0) {
      const int64_t want = ((int64_t)num_reqs * max_kv_len + 63) / 64;
      if (want < grid) grid = want > 0 ? want : 1;
    }
    // with a reused plan the decode kernel may start its set-up (which reads
    // only the plan and the KV index) while the preceding kernel finishes
    // Few requests with long contexts are each cut over many CTAs: their
    // partials are merged in two levels (shorter dependent-load chains).  Only
    // for such batches: the other instance keeps a leaner merge.
    const bool two_level = num_reqs <= 16 && max_kv_len > 768;
    rc = from_cuda(
        launch_decode(ap, (int)grid, (flags & MSG_ATTN_REUSE_PLAN) != 0, two_level, s));
    if (rc != MSG_OK) return rc;
  }
  if (!(flags & MSG_ATTN_DECODE_ONLY)) {
    // the persistent extend kernel takes work items from a counter in the plan header
    PlanHeader *hdr = reinterpret_cast<PlanHeader *>(ws + L.header);
    rc = from_cuda(cudaMemsetAsync(&hdr->ext_next, 0, 2 * sizeof(int32_t), s));
    if (rc != MSG_OK) return rc;
    rc = from_cuda(launch_extend(ap, L.max_tiles, max_kv_len, s));
    if (rc != MSG_OK) return rc;
  }
  return MSG_OK;
}

}  // namespace

extern "C" {

int msg_read_device_status(const void *dev_status, int32_t *host_out, void *stream) {
  if (dev_status == nullptr || host_out == nullptr) return MSG_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(host_out, dev_status, MSG_STATUS_BYTES, cudaMemcpyDeviceToHost, s) !=
      cudaSuccess)
    return MSG_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MSG_ERR_CUDA;
  return host_out[0] == MSG_DEV_OK ? MSG_OK : MSG_ERR_DEVICE_CHECK;
}

int msg_get_device_error(const void *workspace, void *stream) {
  int32_t host[4] = {0, 0, 0, 0};
  const int rc = msg_read_device_status(workspace, host, stream);
  if (rc != MSG_OK && rc != MSG_ERR_DEVICE_CHECK) return rc;
  return host[0];
}

int msg_clear_device_status(void *dev_status, void *stream) {
  if (dev_status == nullptr) return MSG_ERR_INVALID_ARG;
  return from_cuda(
      cudaMemsetAsync(dev_status, 0, MSG_STATUS_BYTES, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

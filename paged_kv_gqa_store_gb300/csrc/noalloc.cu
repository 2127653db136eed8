// noalloc.cu -- msg_paged_attention_noalloc: paged attention whose scratch
// workspace (plan, split-KV partials, merge counters, status block) lives in a
// fixed array inside the library instead of a caller-allocated buffer.
//
// For callers that cannot allocate device memory themselves: code that runs
// under a framework whose allocator owns every byte of device memory and
// forbids raw cudaMalloc, C or plugin callers that have no device allocator at
// hand, and latency-critical loops that cannot afford cudaMalloc / cudaFree
// (both may synchronise the device).  They still pass their inputs and outputs.
//
// The array is a file-scope __device__ object: every GPU that loads the
// library holds MSG_NOALLOC_SCRATCH_BYTES of it until the process exits.  Host
// code cannot use the symbol as a device address, so the first call on each
// device looks the address up with cudaGetSymbolAddress (with that device
// current) and caches it; that first call should therefore come before any
// stream capture.  All calls share the one array: calls that overlap on the GPU
// (on different streams, or from different threads without ordering) race on
// it and must not be issued.
#include "internal.cuh"

namespace {

static __device__ __align__(256) uint8_t g_noalloc_scratch[MSG_NOALLOC_SCRATCH_BYTES];

// Batch size (num_reqs, total_q) of the plan the last successful call without
// MSG_ATTN_REUSE_PLAN left in the array, per device; {-1, -1}: none yet.  The
// plan's offsets in the array depend on that size, so a call that reuses the
// plan must have the same one.
struct PlanSize {
  int32_t num_reqs = -1;
  int64_t total_q = -1;
};
PlanSize g_plan_size[64];

void *scratch_address(int *rc) {
  static void *addr[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    *rc = MSG_ERR_CUDA;
    return nullptr;
  }
  if (addr[dev] == nullptr) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      *rc = MSG_ERR_CUDA;
      return nullptr;
    }
    addr[dev] = p;
  }
  *rc = MSG_OK;
  return addr[dev];
}

}  // namespace

extern "C" int msg_paged_attention_noalloc(
    const void *q, int64_t q_row_stride, const void *k_pool, const void *v_pool,
    int64_t pool_row_stride, int64_t num_slots, const int32_t *page_table,
    int64_t page_table_stride, const int32_t *req_rows, const int32_t *cached_len,
    const int32_t *extend_len, const int32_t *qo_indptr, int32_t num_reqs, int64_t total_q,
    int32_t max_kv_len, int32_t page_size, int32_t num_qo_heads, int32_t num_kv_heads,
    int32_t head_dim, float scale, void *out, uint32_t flags, int32_t *dev_status,
    void *stream) {
  if (num_reqs < 0 || total_q < 0 || num_qo_heads <= 0 || head_dim <= 0)
    return MSG_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (num_reqs == 0 || total_q == 0) {
    // nothing to do; the caller's status block reports this call: clean
    if (dev_status != nullptr &&
        cudaMemsetAsync(dev_status, 0, MSG_STATUS_BYTES, s) != cudaSuccess)
      return MSG_ERR_CUDA;
    return MSG_OK;
  }
  // the part a call needs (the scratch leaves out the extend key split's
  // partial slots: batches with few extend items take them whole here)
  const size_t need = msg::ws_layout(num_reqs, total_q, num_qo_heads, head_dim).total;
  if (need == 0) return MSG_ERR_INVALID_ARG;
  if (need > (size_t)MSG_NOALLOC_SCRATCH_BYTES) return MSG_ERR_WORKSPACE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MSG_ERR_CUDA;
  PlanSize &plan = g_plan_size[dev];
  const bool reuse = (flags & MSG_ATTN_REUSE_PLAN) != 0;
  if (reuse && (plan.num_reqs != num_reqs || plan.total_q != total_q))
    return MSG_ERR_INVALID_ARG;        // no plan of this batch size in the array
  int rc = MSG_OK;
  uint8_t *ws = static_cast<uint8_t *>(scratch_address(&rc));
  if (rc != MSG_OK) return rc;
  // The status block must start at zero so that it reports this call only.
  if (cudaMemsetAsync(ws, 0, MSG_STATUS_BYTES, s) != cudaSuccess) return MSG_ERR_CUDA;
  if (!reuse) plan = PlanSize{};       // the plan is rewritten below
  rc = msg_paged_attention(q, q_row_stride, k_pool, v_pool, pool_row_stride, num_slots,
                           page_table, page_table_stride, req_rows, cached_len, extend_len,
                           qo_indptr, num_reqs, total_q, max_kv_len, page_size, num_qo_heads,
                           num_kv_heads, head_dim, scale, out, ws, MSG_NOALLOC_SCRATCH_BYTES,
                           flags, stream);
  if (rc != MSG_OK) return rc;
  if (!reuse) {
    plan.num_reqs = num_reqs;
    plan.total_q = total_q;
  }
  if (dev_status != nullptr &&
      cudaMemcpyAsync(dev_status, ws, MSG_STATUS_BYTES, cudaMemcpyDeviceToDevice, s) !=
          cudaSuccess)
    return MSG_ERR_CUDA;
  return MSG_OK;
}

// kv_index.cu -- a1, the backends' forms of the global page table
// ("Mini-SGLang 完整剖析" 4.6.4): the engine keeps one token-granular table
// (entry = pool slot of a token); the FlashAttention / TRT-LLM backends read a
// dense per-request table of page ids (every page_size-th column divided by
// page_size), FlashInfer a 1-D ragged list of the same ids with int32 offsets.
#include "internal.cuh"

namespace msg {

namespace {

constexpr int kScanThreads = 1024;

struct IndexParams {
  int32_t kind;
  int32_t page_size, page_shift;
  const int32_t *page_table;
  int64_t pt_stride;
  const int32_t *req_rows;
  const int32_t *cached_len;
  const int32_t *extend_len;
  int32_t num_reqs;
  int32_t *out;
  int64_t out_stride;           // page-id table
  int64_t out_capacity;         // ragged list
  int32_t *indptr;              // ragged offsets (written by the scan)
  int32_t *status;
};

// Pages of request r, or -1 if its lengths are invalid (reported).
__device__ __forceinline__ int64_t pages_of(const IndexParams &p, int32_t r) {
  const int64_t c = p.cached_len[r], e = p.extend_len[r];
  const int64_t n = c + e;
  if (c < 0 || e < 0 || n > p.pt_stride) {
    report(p.status, MSG_DEV_BAD_LENGTHS, r, n);
    return -1;
  }
  return (n + p.page_size - 1) >> p.page_shift;
}

// Ragged offsets: exclusive prefix sum of the page counts, one CTA.
__global__ void __launch_bounds__(kScanThreads) indptr_kernel(IndexParams p) {
  __shared__ int64_t part[kScanThreads];
  const int tid = threadIdx.x;
  const int32_t per = (p.num_reqs + kScanThreads - 1) / kScanThreads;
  const int32_t r0 = tid * per;
  int64_t sum = 0;
  for (int32_t r = r0; r < r0 + per && r < p.num_reqs; ++r) {
    const int64_t n = pages_of(p, r);
    sum += n > 0 ? n : 0;
  }
  part[tid] = sum;
  __syncthreads();
  // inclusive Hillis-Steele scan over the per-thread sums
  for (int o = 1; o < kScanThreads; o <<= 1) {
    const int64_t add = tid >= o ? part[tid - o] : 0;
    __syncthreads();
    part[tid] += add;
    __syncthreads();
  }
  int64_t off = tid ? part[tid - 1] : 0;
  for (int32_t r = r0; r < r0 + per && r < p.num_reqs; ++r) {
    p.indptr[r] = (int32_t)off;
    const int64_t n = pages_of(p, r);
    off += n > 0 ? n : 0;
  }
  if (tid == kScanThreads - 1) {
    const int64_t total = part[kScanThreads - 1];
    p.indptr[p.num_reqs] = (int32_t)total;
    if (total > p.out_capacity) report(p.status, MSG_DEV_BAD_LENGTHS, p.num_reqs, total);
  }
}

// One CTA per request (grid-stride): entry i = page_table[row, i * P] / P.
__global__ void fill_kernel(IndexParams p) {
  for (int32_t r = blockIdx.x; r < p.num_reqs; r += gridDim.x) {
    const int64_t n = pages_of(p, r);
    if (n <= 0) continue;
    int64_t base, limit;
    if (p.kind == MSG_KV_RAGGED) {
      base = p.indptr[r];
      limit = p.out_capacity;
    } else {
      if (n > p.out_stride) {
        if (threadIdx.x == 0) report(p.status, MSG_DEV_BAD_LENGTHS, r, n);
        continue;
      }
      base = (int64_t)r * p.out_stride;
      limit = base + p.out_stride;
    }
    const int64_t row = p.req_rows ? p.req_rows[r] : r;
    const int32_t *src = p.page_table + row * p.pt_stride;
    for (int64_t i = threadIdx.x; i < n && base + i < limit; i += blockDim.x) {
      const int32_t first = src[i << p.page_shift];
      int32_t id = -1;
      if (first < 0) report(p.status, MSG_DEV_SLOT_OUT_OF_RANGE, r, first);
      else if (first & (p.page_size - 1)) report(p.status, MSG_DEV_PAGE_MISALIGNED, r, first);
      else id = first >> p.page_shift;
      p.out[base + i] = id;
    }
  }
}

}  // namespace

}  // namespace msg

extern "C" int msg_build_kv_index(int32_t kind, int32_t page_size, const int32_t *page_table,
                                  int64_t page_table_stride, const int32_t *req_rows,
                                  const int32_t *cached_len, const int32_t *extend_len,
                                  int32_t num_reqs, int32_t *out_table, int64_t out_stride,
                                  int64_t out_capacity, int32_t *out_indptr, int32_t *dev_status,
                                  void *stream) {
  using namespace msg;
  if (kind != MSG_KV_PAGE_TABLE && kind != MSG_KV_RAGGED) return MSG_ERR_UNSUPPORTED;
  if (page_size < 1 || page_size > 128 || (page_size & (page_size - 1))) return MSG_ERR_UNSUPPORTED;
  if (num_reqs < 0 || page_table_stride < 0) return MSG_ERR_INVALID_ARG;
  if (kind == MSG_KV_RAGGED && (out_indptr == nullptr || out_capacity < 0))
    return MSG_ERR_INVALID_ARG;
  if (kind == MSG_KV_PAGE_TABLE && out_stride < 0) return MSG_ERR_INVALID_ARG;
  if (num_reqs == 0) {
    if (kind == MSG_KV_RAGGED)
      return cudaMemsetAsync(out_indptr, 0, sizeof(int32_t), static_cast<cudaStream_t>(stream)) ==
                     cudaSuccess
                 ? MSG_OK
                 : MSG_ERR_CUDA;
    return MSG_OK;
  }
  if (!page_table || !cached_len || !extend_len || !out_table) return MSG_ERR_INVALID_ARG;
  IndexParams p{};
  p.kind = kind;
  p.page_size = page_size;
  while ((1 << p.page_shift) < page_size) ++p.page_shift;
  p.page_table = page_table;
  p.pt_stride = page_table_stride;
  p.req_rows = req_rows;
  p.cached_len = cached_len;
  p.extend_len = extend_len;
  p.num_reqs = num_reqs;
  p.out = out_table;
  p.out_stride = out_stride;
  p.out_capacity = out_capacity;
  p.indptr = out_indptr;
  p.status = dev_status;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (kind == MSG_KV_RAGGED) {
    indptr_kernel<<<1, kScanThreads, 0, s>>>(p);
    if (cudaGetLastError() != cudaSuccess) return MSG_ERR_CUDA;
  }
  int64_t grid = num_reqs;
  const int64_t cap = (int64_t)device_sm_count() * 4;
  if (grid > cap) grid = cap;
  fill_kernel<<<(unsigned)grid, 256, 0, s>>>(p);
  return cudaGetLastError() == cudaSuccess ? MSG_OK : MSG_ERR_CUDA;
}

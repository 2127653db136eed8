// store_kv.cu -- a2, the KV-pool write path.
//
// "Mini-SGLang 完整剖析" 4.4.3 / 4.6.7: the pool of one layer is a
// [slots, kv_heads, head_dim] array per K and V; at the start of the attention
// backend's forward, row i of the step's new K (and V) is copied to pool row
// out_loc[i].  4.9.4 states the shape contract (rows of kv_heads * head_dim
// elements, int32 or int64 indices, one dtype); 4.9.5 describes the upstream
// warp-per-row copy in 16-byte packets.
//
// GB300 design: a grid-stride loop over 16-byte units (token, K|V, chunk) so
// that consecutive threads move consecutive 16 B of one 2 KiB row (coalesced
// on both sides); each thread issues 4 independent loads before its stores to
// keep many requests in flight.  Slots outside [0, num_slots) are reported in
// the status block and not written.
#include "internal.cuh"

namespace msg {

namespace {

constexpr int kStoreThreads = 256;
constexpr int kStoreUnroll = 4;

__device__ __forceinline__ uint4 ld_stream(const uint8_t *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__global__ void __launch_bounds__(kStoreThreads) store_kv_kernel(StoreParams p) {
  grid_dep_wait();      // k / v come from, and the pools are read by, the kernels around it
  grid_dep_launch();
  const int64_t per_tok = 2 * (int64_t)p.row_chunks;
  const int64_t total = p.num_tokens * per_tok;
  const int64_t step = (int64_t)gridDim.x * kStoreThreads * kStoreUnroll;
  for (int64_t base = (int64_t)blockIdx.x * kStoreThreads * kStoreUnroll + threadIdx.x;
       base < total; base += step) {
    uint4 val[kStoreUnroll];
    uint8_t *dst[kStoreUnroll];
#pragma unroll
    for (int u = 0; u < kStoreUnroll; ++u) {
      const int64_t unit = base + (int64_t)u * kStoreThreads;
      dst[u] = nullptr;
      if (unit < total) {
        const int64_t tok = unit / per_tok;
        const int64_t rem = unit - tok * per_tok;
        const int which = rem >= p.row_chunks;           // 0 = K, 1 = V
        const int64_t chunk = rem - (which ? p.row_chunks : 0);
        const int64_t slot = p.out_loc_is_int64
                                 ? static_cast<const int64_t *>(p.out_loc)[tok]
                                 : (int64_t) static_cast<const int32_t *>(p.out_loc)[tok];
        if (slot < 0 || slot >= p.num_slots) {
          if (chunk == 0 && !which) report(p.status, MSG_DEV_SLOT_OUT_OF_RANGE, (int32_t)tok, slot);
          continue;
        }
        const uint8_t *src = (which ? p.v : p.k) + tok * p.in_stride_bytes + chunk * 16;
        val[u] = ld_stream(src);
        dst[u] = (which ? p.v_pool : p.k_pool) + slot * p.pool_stride_bytes + chunk * 16;
      }
    }
#pragma unroll
    for (int u = 0; u < kStoreUnroll; ++u)
      if (dst[u]) *reinterpret_cast<uint4 *>(dst[u]) = val[u];
  }
}

}  // namespace

cudaError_t launch_store_kv(const StoreParams &p, cudaStream_t s) {
  const int64_t total = p.num_tokens * 2 * (int64_t)p.row_chunks;
  if (total <= 0) return cudaSuccess;
  int64_t blocks = (total + kStoreThreads * kStoreUnroll - 1) / (kStoreThreads * kStoreUnroll);
  const int64_t cap = (int64_t)device_sm_count() * 8;
  if (blocks > cap) blocks = cap;
  return launch_k(store_kv_kernel, dim3((unsigned)blocks), dim3(kStoreThreads), 0, s, true, p);
}

}  // namespace msg

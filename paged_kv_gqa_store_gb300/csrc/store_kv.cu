// store_kv.cu -- a2, the KV-pool write path.
//
// "Mini-SGLang 完整剖析" 4.4.3 / 4.6.7: the pool of one layer is a
// [slots, kv_heads, head_dim] array per K and V; at the start of the attention
// backend's forward, row i of the step's new K (and V) is copied to pool row
// out_loc[i].  4.9.4 states the shape contract (rows of kv_heads * head_dim
// elements, int32 or int64 indices, one dtype); 4.9.5 describes the upstream
// warp-per-row copy in 16-byte packets.
//
// GB300 design: one warp per token, over a grid sized to the SMs.  The warp
// moves the token's K and V rows in 16-byte chunks (lane l takes chunks l,
// l + 32, ...: coalesced on both sides), issuing all of a row pair's loads (8
// per lane for 2 KiB rows) together with the token's slot before any store,
// so no load waits on the slot.  Slots outside [0, num_slots) are reported in
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
  const int lane = threadIdx.x & 31;
  const int64_t first = ((int64_t)blockIdx.x * kStoreThreads + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * kStoreThreads) >> 5;
  const int rc = p.row_chunks;
  for (int64_t tok = first; tok < p.num_tokens; tok += nwarps) {
    const int64_t slot = p.out_loc_is_int64 ? static_cast<const int64_t *>(p.out_loc)[tok]
                                            : (int64_t) static_cast<const int32_t *>(p.out_loc)[tok];
    const uint8_t *ks = p.k + tok * p.in_stride_bytes, *vs = p.v + tok * p.in_stride_bytes;
    const bool ok = slot >= 0 && slot < p.num_slots;
    if (!ok && lane == 0) report(p.status, MSG_DEV_SLOT_OUT_OF_RANGE, (int32_t)tok, slot);
    uint8_t *kd = p.k_pool + (ok ? slot : 0) * p.pool_stride_bytes;
    uint8_t *vd = p.v_pool + (ok ? slot : 0) * p.pool_stride_bytes;
    for (int c0 = 0; c0 < rc; c0 += 32 * kStoreUnroll) {
      uint4 kv[kStoreUnroll], vv[kStoreUnroll];
#pragma unroll
      for (int u = 0; u < kStoreUnroll; ++u) {
        const int c = c0 + u * 32 + lane;
        if (c < rc) {
          kv[u] = ld_stream(ks + (int64_t)c * 16);
          vv[u] = ld_stream(vs + (int64_t)c * 16);
        }
      }
      if (!ok) continue;
#pragma unroll
      for (int u = 0; u < kStoreUnroll; ++u) {
        const int c = c0 + u * 32 + lane;
        if (c < rc) {
          *reinterpret_cast<uint4 *>(kd + (int64_t)c * 16) = kv[u];
          *reinterpret_cast<uint4 *>(vd + (int64_t)c * 16) = vv[u];
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_store_kv(const StoreParams &p, cudaStream_t s) {
  if (p.num_tokens <= 0 || p.row_chunks <= 0) return cudaSuccess;
  constexpr int kWarps = kStoreThreads / 32;               // one warp per token
  int64_t blocks = (p.num_tokens + kWarps - 1) / kWarps;
  const int64_t cap = (int64_t)device_sm_count() * 8;
  if (blocks > cap) blocks = cap;
  return launch_k(store_kv_kernel, dim3((unsigned)blocks), dim3(kStoreThreads), 0, s, true, p);
}

}  // namespace msg

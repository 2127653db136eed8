// internal.cuh -- shared definitions of the sm_103a kernels behind msg.h:
// workspace layout, kernel parameter blocks and small device helpers
// (bf16 unpacking, mbarrier / bulk-copy PTX, the device status block).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/msg.h"

namespace msg {

constexpr int kHeadDim = 128;
constexpr int kGroup = 2;                 // query heads per KV head
constexpr int kMaxKvHeads = 8;            // KV heads of a full layer (16 query heads); a
                                          // tensor-parallel slice passes 4, 2 or 1
constexpr int kMaxDecodeCtas = 512;       // decode CTAs at 8 KV heads (2 partial slots each)
// Group counters of the two-level split merge, one per (partial slot, KV
// head): slots x KV heads is at most 2 kMaxDecodeCtas x 8 at every head count
// (fewer heads, proportionally more CTAs).
constexpr int kGroupCounters = 2 * kMaxDecodeCtas * kMaxKvHeads;
// The decode plan lays the requests' keys end to end with this many empty
// key positions after each request: the decode CTAs split that space evenly,
// so a CTA whose range holds a request boundary (a second segment: its q, its
// own normalisation and partial) gets correspondingly fewer keys.  Below the
// decode kernel's 32 keys per CTA, so no CTA range lies inside a gap.
constexpr int kDecSegPad = 24;

// Decode CTAs the split-KV partials have room for with hq query heads: the
// partial arrays are sized for 16 heads x kMaxDecodeCtas, so fewer heads per
// CTA leave room for proportionally more CTAs.
inline int64_t max_decode_ctas(int64_t hq) {
  return hq > 0 && hq < kGroup * kMaxKvHeads ? kMaxDecodeCtas * (kGroup * kMaxKvHeads / hq)
                                             : kMaxDecodeCtas;
}
constexpr int kExtendTileTokens = 128;    // query tokens per extend tile
// Extend batches with few work items split them along the keys over the CTAs
// (see extend.cu): partial slots for up to kExtMaxCtas CTAs, a tile prefix of
// up to kExtMaxTiles tiles, a list of the split items (one entry per slot).
constexpr int kExtMaxCtas = 160;
constexpr int kExtMaxItems = 4 * kExtMaxCtas;
constexpr int kExtMaxTiles = 256;
constexpr int kExtSlots = 2 * kExtMaxCtas;
constexpr int kPlanThreads = 1024;

// Bound of every mbarrier wait (2 s, far beyond any legitimate wait); on expiry
// the kernel records MSG_DEV_TIMEOUT and unwinds instead of hanging the GPU.
constexpr uint64_t kWaitNs = 2000000000ull;

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Workspace layout.  Per-request arrays come first and depend only on the
// batch size (num_reqs, total_q), so msg_plan and msg_paged_attention agree on
// them; the split-KV partials (which depend on the head count) follow.
struct WsLayout {
  size_t status = 0;       // int32[4]
  size_t header = 0;       // PlanHeader
  size_t qo_indptr = 0;    // int32[num_reqs + 1]   (plan's own, checked copy)
  size_t dec_req = 0;      // int32[num_reqs]       decode request list
  size_t dec_start = 0;    // int64[num_reqs + 1]   prefix of decode kv lengths + gaps
  size_t dec_row = 0;      // int64[num_reqs]       index row offset of each decode request
  size_t dec_qrow = 0;     // int32[num_reqs]       its query row (qo_indptr)
  size_t counters = 0;     // int32[num_reqs * 8]   split merge counters (request, KV head)
  size_t gcounters = 0;    // int32[kGroupCounters] group merge counters (slot, KV head)
  size_t ext_tiles = 0;    // int32x2[max_tiles]    (request, query tile)
  size_t part_lse = 0;     // float[2 * max_decode_ctas(Hq) * Hq]
  size_t part_o = 0;       // float[2 * max_decode_ctas(Hq) * Hq * D]
  size_t plan_end = 0;     // bytes used by the plan part
  size_t total = 0;        // bytes a call needs
  // optional: the extend key split (used when the workspace holds it)
  size_t ext_items = 0;    // int32x4[kExtSlots]  split items (item, first CTA, last CTA, shift),
                           //                     ext_split_count of them, in arrival order
  size_t ext_lse = 0;      // float[2 * kExtMaxCtas][2][128]
  size_t ext_o = 0;        // float[2 * kExtMaxCtas][2][128][128]
  size_t total_split = 0;  // bytes with the extend key split (msg_workspace_size)
  int64_t max_tiles = 0;
};

struct PlanHeader {
  int32_t num_reqs;        // requests planned
  int32_t dec_count;       // decode requests
  int32_t ext_tile_count;  // extend tiles
  int32_t ext_count;       // extend requests
  int64_t dec_keys;        // sum of decode kv lengths + a gap (kDecSegPad) per request
  int64_t total_q;         // sum of extend lengths
  int32_t ext_next;        // extend work-item counter  } both zeroed before each
  int32_t ext_split_count; // split extend items listed } extend launch
  int32_t ext_split_ready; // the plan filled ext_units
  int32_t pad2;
  int64_t ext_units;       // key tiles over the extend tiles (128 keys each, per KV head)
};

inline WsLayout ws_layout(int64_t num_reqs, int64_t total_q, int64_t hq, int64_t d) {
  WsLayout L;
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t o = off; off = align_up(off + bytes, 256); return o; };
  L.status = take(MSG_STATUS_BYTES);
  L.header = take(sizeof(PlanHeader));
  L.qo_indptr = take(sizeof(int32_t) * (num_reqs + 1));
  L.dec_req = take(sizeof(int32_t) * (num_reqs + 1));
  L.dec_start = take(sizeof(int64_t) * (num_reqs + 1));
  L.dec_row = take(sizeof(int64_t) * (num_reqs + 1));
  L.dec_qrow = take(sizeof(int32_t) * (num_reqs + 1));
  L.counters = take(sizeof(int32_t) * (num_reqs + 1) * kMaxKvHeads);
  L.gcounters = take(sizeof(int32_t) * kGroupCounters);
  L.max_tiles = (total_q + kExtendTileTokens - 1) / kExtendTileTokens + num_reqs + 1;
  L.ext_tiles = take(sizeof(int32_t) * 2 * L.max_tiles);
  L.ext_items = take(sizeof(int32_t) * 4 * kExtSlots);
  L.plan_end = off;
  L.part_lse = take(sizeof(float) * 2 * max_decode_ctas(hq) * hq);
  L.part_o = take(sizeof(float) * 2 * (size_t)max_decode_ctas(hq) * hq * d);
  L.total = off;
  L.ext_lse = take(sizeof(float) * 2 * kExtMaxCtas * 2 * 128);
  L.ext_o = take(sizeof(float) * (size_t)2 * kExtMaxCtas * 2 * 128 * kHeadDim);
  L.total_split = off;
  return L;
}

// ------------------------------------------------------------------ params
// Where the pool slot of token j of a request is found (msg_kv_index).
struct KvIndex {
  const int32_t *table;
  int64_t stride;               // entries between rows (token / page-id tables)
  int64_t len;                  // entries in table, -1 unknown
  const int32_t *req_rows;      // row per request (token / page-id tables), null = r
  const int32_t *indptr;        // ragged: request r's entries at [indptr[r], indptr[r+1])
  int32_t kind;                 // MSG_KV_*
  int32_t page_size;
  int32_t page_shift;           // log2(page_size)
};

struct PlanParams {
  KvIndex kv;                   // row capacities are checked against device_len
  const int32_t *cached_len;
  const int32_t *extend_len;
  const int32_t *qo_in;         // caller's qo_indptr to check, or null
  int32_t num_reqs;
  int64_t total_q;
  int32_t *status;
  PlanHeader *hdr;
  int32_t *qo_ws;               // plan's qo_indptr
  int32_t *qo_out;              // optional user copy
  int32_t *dec_req;
  int64_t *dec_start;
  int64_t *dec_row;             // offset of the request's row (or ragged range) in the index
  int32_t *dec_qrow;
  int32_t *counters;
  int32_t *gcounters;           // kGroupCounters, zeroed with the counters
  int32_t *ext_tiles;           // pairs
  int64_t max_tiles;
};

struct TokenMetaParams {
  KvIndex kv;
  const int32_t *cached_len;
  const int32_t *qo_ws;
  int32_t num_reqs;
  int64_t total_q;
  int64_t num_slots;
  void *out_loc;
  int32_t out_loc_is_int64;
  int32_t *positions;
  int32_t *status;
};

struct StoreParams {
  const uint8_t *k;
  const uint8_t *v;
  int64_t in_stride_bytes;
  uint8_t *k_pool;
  uint8_t *v_pool;
  int64_t pool_stride_bytes;
  int64_t num_slots;
  const void *out_loc;
  int32_t out_loc_is_int64;
  int64_t num_tokens;
  int32_t row_chunks;           // 16-byte chunks per row
  int32_t *status;
};

struct AttnParams {
  const uint16_t *q;
  int64_t q_stride;             // elements between tokens
  const uint8_t *k_pool;
  const uint8_t *v_pool;
  int64_t pool_stride_bytes;
  int64_t num_slots;
  const int32_t *cached_len;
  const int32_t *extend_len;
  const int32_t *qo_indptr;
  int32_t num_reqs;
  int64_t total_q;
  uint32_t flags;
  int32_t page_size;
  int32_t page_shift;           // log2(page_size)
  int32_t num_qo_heads;
  int32_t num_kv_heads;
  float scale_log2;             // scale * log2(e)
  uint16_t *out;
  int32_t *status;
  const PlanHeader *hdr;
  // decode only: the step's new K / V rows (row = the request's q row), read
  // for each request's newest key in place of the pool and stored to the pool
  // by the decode kernel itself; NULL when they are already in the pool
  const uint8_t *k_new, *v_new;
  int64_t new_stride_bytes;
  uint8_t *k_pool_w, *v_pool_w;
  const int32_t *dec_req;
  const int64_t *dec_start;
  const int64_t *dec_row;
  const int32_t *dec_qrow;
  int32_t *counters;
  int32_t *gcounters;           // group counters of the two-level split merge
  const int32_t *ext_tiles;
  float *part_lse;
  float *part_o;
  // extend key split: the split items and their partial slots (null: not available)
  int32_t *ext_items;
  float *ext_lse;
  float *ext_o;
  KvIndex kv;                   // where the keys' slots are found
};

// ------------------------------------------------------------------ launchers
// Launch with an optional programmatic-stream-serialization attribute (see
// grid_dep_wait).
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                     cudaStream_t s, bool pdl, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

cudaError_t launch_plan(const PlanParams &p, cudaStream_t s);
cudaError_t launch_token_meta(const TokenMetaParams &p, cudaStream_t s);
cudaError_t launch_store_kv(const StoreParams &p, cudaStream_t s);
// two_level: the decode instance that merges requests cut into many splits in
// two levels (taken by the host for batches of few long requests).
cudaError_t launch_decode(const AttnParams &p, int grid, bool pdl, bool two_level,
                          cudaStream_t s);
cudaError_t launch_extend(const AttnParams &p, int64_t max_tiles, int64_t max_kv_len,
                          cudaStream_t s);
int device_sm_count();
int decode_ctas_per_sm(int num_kv_heads);

}  // namespace msg

// ------------------------------------------------------------------ device helpers
#ifdef __CUDACC__
namespace msg {

// Record the first device error: code, request index, value (lo/hi words).
__device__ __forceinline__ void report(int32_t *status, int32_t code, int32_t idx,
                                       int64_t val) {
  if (status == nullptr) return;
  if (atomicCAS(status, 0, code) == 0) {
    status[1] = idx;
    status[2] = (int32_t)(uint32_t)((uint64_t)val & 0xffffffffu);
    status[3] = (int32_t)(uint32_t)((uint64_t)val >> 32);
  }
}

// Two bf16 in a 32-bit word -> two floats (exact: bf16 is the high half of fp32).
__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Two floats -> packed bf16x2 (round to nearest even), lo in the low half.
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- mbarrier (shared::cta)
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}
// Bounded wait for the phase with the given parity to complete: gives up after
// kWaitNs of wall-clock time (far beyond any legitimate wait) and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 0 && global_ns() - t0 > kWaitNs) return false;
  }
}

// ---- bulk global -> shared copy completing on an mbarrier (TMA, non-tensor)
__device__ __forceinline__ void bulk_g2s(void *dst_smem, const void *src, uint32_t bytes,
                                         uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst_smem)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// ---- Ampere-style 16-byte async copy (used by the extend kernel)
__device__ __forceinline__ void cp_async16(void *dst_smem, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst_smem)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ int64_t imin64(int64_t a, int64_t b) { return a < b ? a : b; }

// Named barrier over a subset of warps (id 0 is __syncthreads).
__device__ __forceinline__ void named_barrier(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---- programmatic dependent launch
// A kernel launched with launch_k(..., pdl = true) may start while the kernel
// before it on the stream is still running.  Every such kernel calls
// grid_dep_wait() before it touches anything the earlier kernels write (and
// before it writes anything they read), and grid_dep_launch() only after that
// wait.  So when a kernel starts early, everything launched at least two
// kernels before it has completed: only data that old (the plan, the KV index)
// may be read before the wait.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---- KV index layouts ("Mini-SGLang 完整剖析" 4.6.4)
// Entries of request r: its table row, or its ragged range.
__device__ __forceinline__ const int32_t *kv_row(const KvIndex &x, int32_t r) {
  if (x.kind == MSG_KV_RAGGED) return x.table + x.indptr[r];
  return x.table + (int64_t)(x.req_rows ? x.req_rows[r] : r) * x.stride;
}
// Index in the row of the entry that locates token j: the token table holds
// one entry per token but only page starts are read; the page-id forms hold
// one entry per page.
__device__ __forceinline__ int64_t kv_entry(const KvIndex &x, int64_t j) {
  if (x.page_size == 1) return j;                 // every form: one entry per token
  return x.kind == MSG_KV_TOKEN_TABLE ? (j & ~(int64_t)(x.page_size - 1)) : (j >> x.page_shift);
}
// Entries a row needs for n tokens.
__device__ __forceinline__ int64_t kv_entries(const KvIndex &x, int64_t n) {
  return x.kind == MSG_KV_TOKEN_TABLE ? n : (n + x.page_size - 1) >> x.page_shift;
}
// Pool slot of token j from the entry e that locates it, or -1 if e names no
// valid page (recorded in status when `status` is non-null).
__device__ __forceinline__ int64_t kv_slot(const KvIndex &x, int64_t e, int64_t j, int64_t num_slots,
                                           int32_t *status, int32_t req) {
  if (x.page_size == 1) {                          // every form: the entry is the slot
    if (e < 0 || e >= num_slots) {
      if (status) report(status, MSG_DEV_SLOT_OUT_OF_RANGE, req, e);
      return -1;
    }
    return e;
  }
  const int64_t first = x.kind == MSG_KV_TOKEN_TABLE ? e : e << x.page_shift;
  if (e < 0 || first + x.page_size > num_slots) {
    if (status) report(status, MSG_DEV_SLOT_OUT_OF_RANGE, req, e);
    return -1;
  }
  if (first & (x.page_size - 1)) {
    if (status) report(status, MSG_DEV_PAGE_MISALIGNED, req, e);
    return -1;
  }
  return first + (j & (x.page_size - 1));
}

}  // namespace msg
#endif

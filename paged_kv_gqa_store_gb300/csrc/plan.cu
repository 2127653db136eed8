// plan.cu -- a1, per-batch metadata prep on the device (no host sync, one
// launch, graph-capturable).
//
// From per-request (cached_len, extend_len) it builds, as "核心数据结构：Req、
// Batch、Context" (Batch table) and "Engine 与采样器" (手工驱动引擎) define them:
//   qo_indptr  = exclusive prefix sum of extend_len (ragged concatenation),
//   positions  = cached_len .. device_len-1 per request,
//   out_loc    = the slots of tokens cached_len .. device_len-1 of each request,
//                through the batch's KV index (token table, page ids, ragged),
// and the attention plan used by the decode and extend kernels:
//   - the decode list (requests with extend_len == 1) with the prefix sum of
//     their KV lengths, over which the decode kernel splits work evenly;
//   - the extend tile list (request, 64-token query tile), the heaviest tile of
//     each request first (causal: later query tiles see more keys);
//   - zeroed split-merge counters.
#include "internal.cuh"

namespace msg {

namespace {

// Block-wide exclusive scan of 4 int64 lanes over kPlanThreads threads.
struct Scan4 {
  int64_t v[4];
};

__device__ __forceinline__ Scan4 block_exclusive_scan(Scan4 x, Scan4 *total, int64_t (*warp_sums)[4]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  Scan4 inc = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      int64_t y = __shfl_up_sync(0xffffffffu, inc.v[k], o);
      if (lane >= o) inc.v[k] += y;
    }
  }
  if (lane == 31)
    for (int k = 0; k < 4; ++k) warp_sums[warp][k] = inc.v[k];
  __syncthreads();
  if (warp == 0) {
    Scan4 w;
    for (int k = 0; k < 4; ++k) w.v[k] = (lane < (int)(blockDim.x >> 5)) ? warp_sums[lane][k] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        int64_t y = __shfl_up_sync(0xffffffffu, w.v[k], o);
        if (lane >= o) w.v[k] += y;
      }
    }
    for (int k = 0; k < 4; ++k) warp_sums[lane][k] = w.v[k];   // inclusive over warps
  }
  __syncthreads();
  Scan4 ex;
  for (int k = 0; k < 4; ++k) {
    int64_t before_warp = warp ? warp_sums[warp - 1][k] : 0;
    ex.v[k] = before_warp + inc.v[k] - x.v[k];
    total->v[k] = warp_sums[(blockDim.x >> 5) - 1][k];
  }
  __syncthreads();
  return ex;
}

// Does request r's row (or ragged range) hold the entries of n tokens, inside
// the index array when its length is known?
__device__ __forceinline__ bool row_fits(const KvIndex &x, int32_t r, int64_t n) {
  const int64_t need = kv_entries(x, n);
  if (x.kind == MSG_KV_RAGGED) {
    const int64_t b = x.indptr[r], e = x.indptr[r + 1];
    return b >= 0 && e - b >= need && (x.len < 0 || e <= x.len);
  }
  const int64_t row = x.req_rows ? x.req_rows[r] : r;
  return row >= 0 && need <= x.stride && (x.len < 0 || (row + 1) * x.stride <= x.len);
}

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(PlanParams p) {
  grid_dep_wait();      // the previous step's kernels still read the plan
  grid_dep_launch();
  __shared__ int64_t warp_sums[32][4];
  __shared__ int64_t carry[4];     // qo, decode count, decode keys, extend tiles
  __shared__ int32_t ext_reqs;
  __shared__ unsigned long long ext_units;
  const int tid = threadIdx.x;
  if (tid < 4) carry[tid] = 0;
  if (tid == 0) {
    ext_reqs = 0;
    ext_units = 0;
  }
  for (int i = tid; i < kGroupCounters; i += kPlanThreads) p.gcounters[i] = 0;
  __syncthreads();

  for (int32_t base = 0; base < p.num_reqs; base += kPlanThreads) {
    const int32_t r = base + tid;
    int64_t c = 0, e = 0;
    if (r < p.num_reqs) {
      c = p.cached_len[r];
      e = p.extend_len[r];
      if (c < 0 || e < 0 || !row_fits(p.kv, r, c + e)) {
        report(p.status, MSG_DEV_BAD_LENGTHS, r, c + e);
        e = 0;
      }
    }
    const bool is_dec = (e == 1);
    const bool is_ext = (e >= 2);
    const int64_t ntiles = is_ext ? (e + kExtendTileTokens - 1) / kExtendTileTokens : 0;
    Scan4 x{{e, is_dec ? 1 : 0, is_dec ? c + e + kDecSegPad : 0, ntiles}};
    Scan4 tot;
    Scan4 ex = block_exclusive_scan(x, &tot, warp_sums);
    if (r < p.num_reqs) {
      const int64_t qo = carry[0] + ex.v[0];
      p.qo_ws[r] = (int32_t)qo;
      if (p.qo_out) p.qo_out[r] = (int32_t)qo;
      if (p.qo_in && p.qo_in[r] != qo) report(p.status, MSG_DEV_BAD_LENGTHS, r, p.qo_in[r]);
      for (int h = 0; h < kMaxKvHeads; ++h) p.counters[(int64_t)r * kMaxKvHeads + h] = 0;
      if (is_dec) {
        const int64_t i = carry[1] + ex.v[1];
        p.dec_req[i] = r;
        p.dec_start[i] = carry[2] + ex.v[2];
        // what the decode kernel needs to start a segment, in one place
        p.dec_row[i] = kv_row(p.kv, r) - p.kv.table;
        p.dec_qrow[i] = (int32_t)qo;
      }
      if (is_ext) {
        atomicAdd(&ext_reqs, 1);
        const int64_t t0 = carry[3] + ex.v[3];
        unsigned long long units = 0;       // key tiles of the request's query tiles
        for (int64_t t = 0; t < ntiles; ++t) {
          if (t0 + t < p.max_tiles) {
            const int32_t qt = (int32_t)(ntiles - 1 - t);
            p.ext_tiles[2 * (t0 + t)] = r;
            p.ext_tiles[2 * (t0 + t) + 1] = qt;
            const int64_t q0 = (int64_t)qt * kExtendTileTokens;
            const int64_t kv_end = c + q0 + (e - q0 < kExtendTileTokens ? e - q0 : kExtendTileTokens);
            units += (unsigned long long)((kv_end + kExtendTileTokens - 1) / kExtendTileTokens);
          }
        }
        atomicAdd(&ext_units, units);
      }
    }
    __syncthreads();
    if (tid < 4) carry[tid] += tot.v[tid];
    __syncthreads();
  }
  if (tid == 0) {
    const int64_t total = carry[0];
    p.qo_ws[p.num_reqs] = (int32_t)total;
    if (p.qo_out) p.qo_out[p.num_reqs] = (int32_t)total;
    if (total != p.total_q) report(p.status, MSG_DEV_BAD_LENGTHS, p.num_reqs, total);
    if (p.qo_in && p.qo_in[p.num_reqs] != total)
      report(p.status, MSG_DEV_BAD_LENGTHS, p.num_reqs, p.qo_in[p.num_reqs]);
    p.dec_start[carry[1]] = carry[2];
    p.hdr->num_reqs = p.num_reqs;
    p.hdr->dec_count = (int32_t)carry[1];
    p.hdr->dec_keys = carry[2];
    p.hdr->ext_tile_count = (int32_t)(carry[3] < p.max_tiles ? carry[3] : p.max_tiles);
    p.hdr->ext_count = ext_reqs;
    p.hdr->total_q = total;
    p.hdr->ext_units = (int64_t)ext_units;
    p.hdr->ext_split_ready = 1;
  }
}

// out_loc and positions, one thread per new token.
__global__ void token_meta_kernel(TokenMetaParams p) {
  grid_dep_wait();
  grid_dep_launch();
  for (int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; t < p.total_q;
       t += (int64_t)gridDim.x * blockDim.x) {
    // request owning token t: last r with qo[r] <= t (empty requests skipped)
    int32_t lo = 0, hi = p.num_reqs;   // invariant qo[lo] <= t < qo[hi]
    if (t >= p.qo_ws[p.num_reqs]) continue;   // inconsistent total_q, already reported
    while (hi - lo > 1) {
      int32_t mid = (lo + hi) >> 1;
      if (p.qo_ws[mid] <= t) lo = mid; else hi = mid;
    }
    const int32_t r = lo;
    const int64_t pos = (int64_t)p.cached_len[r] + (t - p.qo_ws[r]);
    const int64_t slot = kv_slot(p.kv, kv_row(p.kv, r)[kv_entry(p.kv, pos)], pos, p.num_slots,
                                 p.status, r);
    if (p.positions) p.positions[t] = (int32_t)pos;
    if (p.out_loc) {
      if (p.out_loc_is_int64) static_cast<int64_t *>(p.out_loc)[t] = slot;
      else static_cast<int32_t *>(p.out_loc)[t] = (int32_t)slot;
    }
  }
}

}  // namespace

cudaError_t launch_plan(const PlanParams &p, cudaStream_t s) {
  return launch_k(plan_kernel, dim3(1), dim3(kPlanThreads), 0, s, true, p);
}

cudaError_t launch_token_meta(const TokenMetaParams &p, cudaStream_t s) {
  if (p.total_q <= 0) return cudaSuccess;
  const int threads = 256;
  int64_t blocks = (p.total_q + threads - 1) / threads;
  const int64_t cap = (int64_t)device_sm_count() * 8;
  if (blocks > cap) blocks = cap;
  return launch_k(token_meta_kernel, dim3((unsigned)blocks), dim3(threads), 0, s, true, p);
}

}  // namespace msg

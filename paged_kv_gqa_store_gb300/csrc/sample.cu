// sample.cu -- the batched sampler that follows the forward in forward_batch
// ("Engine 与采样器", 采样器: Sampler.prepare / Sampler.sample / sample_torch;
// "Mini-SGLang 源码解析（四）" 14.2-14.5; "Mini-SGLang 完整剖析" 4.8.5-4.8.6).
//
// Per row: p = softmax(logits / T); keep the k most likely tokens (ties in
// token order); renormalise and keep a token only while the mass ranked ahead
// of it is below top_p; draw the token whose cumulative kept mass, in
// vocabulary order, first exceeds u times the kept total.  Without
// temperatures every row is greedy and the token is the first maximum.
//
// GB300 layout: one thread-block cluster per row.  The row is split into
// C contiguous slices (C = 1..8), each CTA reads its slice from HBM exactly
// once into shared memory (up to ~76 KB for a 151,936-token vocabulary with
// C = 8, two CTAs per SM), and every later step runs out of shared memory.
// There is no sort: the k-th token and the top-p boundary are found by radix
// selection over a 30-bit order key, one 8-bit digit per pass, with the
// per-bucket counts or masses of all C CTAs summed through distributed shared
// memory after a cluster barrier.  Masses are fixed point (e * 2^40, floor),
// so every sum is exact integer arithmetic, identical in every CTA of the
// cluster and from run to run.
#include <math.h>

#include "internal.cuh"

namespace msg {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kBuckets = 256;
constexpr int kMaxCluster = 8;
constexpr int kSliceAlign = 8;                 // elements: every CTA starts 16-byte aligned
constexpr int kSliceTwoPerSm = 24576;          // <= 96 KB of fp32: two CTAs per SM
constexpr int kSliceMax = 53248;               // <= 208 KB of fp32: one CTA per SM
constexpr uint32_t kOneBits = 0x3F800000u;     // bits of 1.0f
constexpr uint32_t kPadBits = 0x80000000u;     // -0.0f: key above every real key
constexpr float kMinT = 1e-6f;                 // Sampler.prepare's MIN_T
constexpr float kMinP = 1e-6f;                 // Sampler.prepare's MIN_P
constexpr float kMassScale = 1099511627776.0f; // 2^40

struct SampleParams {
  const uint8_t *logits;
  int64_t row_bytes;                           // bytes between rows
  int32_t batch, vocab, slice;                 // slice: elements per CTA (multiple of 8)
  const float *temperature;                    // null: every row greedy
  const int32_t *top_k;                        // null: no top-k
  const float *top_p;                          // null: no top-p
  const float *uniform;
  int32_t *tokens;
  int32_t *status;
};

// Shared state beside the staged slice.  Buffers read by other CTAs of the
// cluster alternate between two slots, so a slot is rewritten only after the
// barrier that follows every CTA's last read of it.
struct Shared {
  unsigned long long hist[2][kBuckets];        // published per-CTA histogram
  unsigned long long scal[2][2];               // published per-CTA scalars
  unsigned long long scan[kWarps];
  unsigned long long wmass[kWarps];            // draw: mass below the threshold key, per warp
  uint32_t wties[kWarps];                      //       keys equal to it, per warp
  uint32_t pick[4];                            // selected bucket / flags
  unsigned long long pick64[2];
};
static_assert(sizeof(Shared) % 16 == 0, "the staged slice after Shared must be 16-byte aligned");

// ---- cluster primitives
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Every thread of every CTA of the cluster arrives (release) and waits
// (acquire): shared-memory writes before it are visible to every CTA after it.
__device__ __forceinline__ void cluster_barrier() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
               "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ unsigned long long ld_cluster_u64(const void *local, uint32_t rank) {
  uint32_t remote;
  unsigned long long v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
  asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(remote) : "memory");
  return v;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Order key: ascending key = descending probability (e in [0, 1]).
__device__ __forceinline__ uint32_t key_of(uint32_t bits) { return kOneBits - bits; }
// Fixed-point mass of a probability weight: floor(e * 2^40).
__device__ __forceinline__ unsigned long long mass_of(uint32_t bits) {
  return __float2ull_rz(__uint_as_float(bits) * kMassScale);
}
// Float -> unsigned key with the same order (finite values).
__device__ __forceinline__ uint32_t orderable(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ unsigned long long warp_sum(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Exclusive scan over the block of one value per thread (thread order);
// `total` receives the block sum.  Contains two __syncthreads.
__device__ __forceinline__ unsigned long long block_excl_scan(unsigned long long v, Shared &sh,
                                                              unsigned long long &total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sh.scan[warp] = x;
  __syncthreads();
  unsigned long long before = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const unsigned long long t = sh.scan[w];
    if (w < warp) before += t;
    tot += t;
  }
  __syncthreads();
  total = tot;
  return before + x - v;
}

// Digit d of the 30-bit key: bits [shift, shift + width).
__device__ __forceinline__ int digit_shift(int d) { return d < 3 ? 22 - 8 * d : 0; }
__device__ __forceinline__ int digit_width(int d) { return d < 3 ? 8 : 6; }

// Cluster sum of this thread's bucket (thread b, bucket b), then the bucket
// with excl(b) < target <= excl(b) + h(b), published in shared memory:
// pick[0] = bucket, pick64[0] = excl, pick64[1] = h.  `adjust` is taken off
// bucket adj_bucket first.  False if no bucket qualifies (target above the
// total).
__device__ __forceinline__ bool select_bucket(Shared &sh, int slot, int C,
                                              unsigned long long target, int adj_bucket,
                                              unsigned long long adjust,
                                              unsigned long long *total_out) {
  const int b = threadIdx.x;
  unsigned long long h = 0;
  for (int c = 0; c < C; ++c) h += ld_cluster_u64(&sh.hist[slot][b], (uint32_t)c);
  if (b == adj_bucket) h -= adjust;
  unsigned long long total;
  const unsigned long long excl = block_excl_scan(h, sh, total);
  if (threadIdx.x == 0) sh.pick[1] = 0;
  __syncthreads();
  if (excl < target && target <= excl + h) {
    sh.pick[0] = (uint32_t)b;
    sh.pick[1] = 1;
    sh.pick64[0] = excl;
    sh.pick64[1] = h;
  }
  if (total_out) *total_out = total;
  __syncthreads();
  return sh.pick[1] != 0;
}

template <bool kBf16>
__device__ __forceinline__ void load8(const uint8_t *p, float v[8]) {
  if (kBf16) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    v[0] = bf16lo(r.x); v[1] = bf16hi(r.x); v[2] = bf16lo(r.y); v[3] = bf16hi(r.y);
    v[4] = bf16lo(r.z); v[5] = bf16hi(r.z); v[6] = bf16lo(r.w); v[7] = bf16hi(r.w);
  } else {
    float4 a, b;
    asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(a.x), "=f"(a.y), "=f"(a.z), "=f"(a.w) : "l"(p));
    asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(b.x), "=f"(b.y), "=f"(b.z), "=f"(b.w) : "l"(p + 16));
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
}

template <bool kBf16>
__device__ __forceinline__ float load1(const uint8_t *row, int64_t j) {
  if (kBf16) return __uint_as_float((uint32_t)reinterpret_cast<const uint16_t *>(row)[j] << 16);
  return reinterpret_cast<const float *>(row)[j];
}

template <bool kBf16, bool kGreedy>
__global__ void __launch_bounds__(kThreads, kGreedy ? 4 : 2) sample_kernel(SampleParams p) {
  extern __shared__ __align__(16) uint8_t smem[];
  Shared &sh = *reinterpret_cast<Shared *>(smem);
  uint32_t *val = reinterpret_cast<uint32_t *>(smem + sizeof(Shared));
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int C = (int)(gridDim.x / (uint32_t)p.batch);     // cluster size
  const uint32_t rank = cluster_rank();
  const int row = (int)(blockIdx.x / (uint32_t)C);
  const int64_t lo = (int64_t)rank * p.slice;
  const int64_t left = (int64_t)p.vocab - lo;
  const int n = left <= 0 ? 0 : (int)(left < p.slice ? left : p.slice);
  const uint8_t *rowp = p.logits + (int64_t)row * p.row_bytes;
  constexpr int kEsz = kBf16 ? 2 : 4;

  // ---- pass 0: the slice from HBM (once), its maximum, finiteness.  Rows need
  //      not be 16-byte aligned: the first h < 16 / esz elements (up to the
  //      next 16-byte boundary) and the ragged end are read one by one, the
  //      rest as 16-byte vectors.  Element j of the slice sits at val[off + j]
  //      with off chosen so that the vector part lands 16-byte aligned in
  //      shared memory; val[0, off) and the end of the last group hold pads.
  float vmax = -INFINITY;
  bool finite = true;
  unsigned long long best = 0;                 // greedy: (orderable value, ~index), max wins
  const uint8_t *sp = rowp + lo * kEsz;        // first element of the slice
  const int h = min(n, (int)(((16u - (uint32_t)(reinterpret_cast<uintptr_t>(sp) & 15u)) & 15u) / kEsz));
  const int off = (4 - (h & 3)) & 3;
  const int nchunk = (n - h) >> 3;
  const int n4 = (off + n + 3) >> 2;
  auto take = [&](float x, int j) {            // element j of the slice, read one by one
    finite &= isfinite(x);
    if (kGreedy) {
      const unsigned long long key = ((unsigned long long)orderable(x + 0.f) << 32) |
                                     (0xffffffffu - (uint32_t)(lo + j));
      best = key > best ? key : best;
    } else {
      vmax = fmaxf(vmax, x);
      val[off + j] = __float_as_uint(x);
    }
  };
  for (int c0 = tid; c0 < nchunk; c0 += 4 * kThreads) {
    float v[4][8];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (c0 + u * kThreads < nchunk) load8<kBf16>(sp + (h + 8 * (c0 + u * kThreads)) * kEsz, v[u]);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int c = c0 + u * kThreads;
      if (c >= nchunk) break;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        finite &= isfinite(v[u][e]);
        if (kGreedy) {
          const unsigned long long key = ((unsigned long long)orderable(v[u][e] + 0.f) << 32) |
                                         (0xffffffffu - (uint32_t)(lo + h + 8 * c + e));
          best = key > best ? key : best;
        } else {
          vmax = fmaxf(vmax, v[u][e]);
        }
      }
      if (!kGreedy) {
        uint4 *dst = reinterpret_cast<uint4 *>(val + off + h + 8 * c);
        dst[0] = make_uint4(__float_as_uint(v[u][0]), __float_as_uint(v[u][1]),
                            __float_as_uint(v[u][2]), __float_as_uint(v[u][3]));
        dst[1] = make_uint4(__float_as_uint(v[u][4]), __float_as_uint(v[u][5]),
                            __float_as_uint(v[u][6]), __float_as_uint(v[u][7]));
      }
    }
  }
  if (tid < h) take(load1<kBf16>(sp, tid), tid);                      // head
  {
    const int j = h + 8 * nchunk + (tid - 32);                      // ragged end (warp 1)
    if (tid >= 32 && j < n && tid < 40) take(load1<kBf16>(sp, j), j);
  }
  if (!kGreedy) {                                                   // pads
    if (tid >= 64 && tid < 64 + off) val[tid - 64] = kPadBits;
    const int i = off + n + (tid - 96);
    if (tid >= 96 && tid < 100 && i < 4 * n4) val[i] = kPadBits;
  }
  // block reduce, publish, cluster reduce
  const int any_bad = __syncthreads_or(!finite);
  if (kGreedy) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long y = __shfl_xor_sync(0xffffffffu, best, o);
      best = y > best ? y : best;
    }
    if (lane == 0) sh.scan[warp] = best;
  } else {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, o));
    if (lane == 0) sh.scan[warp] = __float_as_uint(vmax);
  }
  __syncthreads();
  if (tid == 0) {
    unsigned long long r = 0;
    float m = -INFINITY;
    for (int w = 0; w < kWarps; ++w) {
      if (kGreedy) r = sh.scan[w] > r ? sh.scan[w] : r;
      else m = fmaxf(m, __uint_as_float((uint32_t)sh.scan[w]));
    }
    sh.scal[0][0] = kGreedy ? r : (unsigned long long)__float_as_uint(m);
    sh.scal[0][1] = any_bad ? 1ull : 0ull;
  }
  cluster_barrier();
  unsigned long long red = 0;
  float M = -INFINITY;
  bool bad = false;
  for (int c = 0; c < C; ++c) {
    const unsigned long long a = ld_cluster_u64(&sh.scal[0][0], (uint32_t)c);
    bad |= ld_cluster_u64(&sh.scal[0][1], (uint32_t)c) != 0;
    if (kGreedy) red = a > red ? a : red;
    else M = fmaxf(M, __uint_as_float((uint32_t)a));
  }
  if (kGreedy) {
    if (tid == 0 && rank == 0) {
      if (bad) {
        report(p.status, MSG_DEV_BAD_LOGIT, row, 0);
        p.tokens[row] = -1;
      } else {
        p.tokens[row] = (int32_t)(0xffffffffu - (uint32_t)(red & 0xffffffffu));
      }
    }
    cluster_barrier();                         // no CTA leaves while its scalars are read
    return;
  }

  // ---- row parameters (Sampler.prepare's clamps), identical in every CTA
  const float T = p.temperature[row];
  const float u = p.uniform[row];
  int64_t k = p.vocab;
  if (p.top_k != nullptr && p.top_k[row] >= 1 && p.top_k[row] < p.vocab) k = p.top_k[row];
  float P = 1.f;
  if (p.top_p != nullptr) P = fminf(fmaxf(p.top_p[row], kMinP), 1.f);
  const bool params_ok = isfinite(T) && u >= 0.f && u < 1.f &&
                         (p.top_p == nullptr || !isnan(p.top_p[row]));
  if (bad || !params_ok) {
    if (tid == 0 && rank == 0) {
      report(p.status, bad ? MSG_DEV_BAD_LOGIT : MSG_DEV_BAD_SAMPLING, row, 0);
      p.tokens[row] = -1;
    }
    cluster_barrier();
    return;
  }
  const bool topk_on = k < p.vocab;
  const bool topp_on = P < 1.f;
  // (l - max) * log2(e) / T, then 2^x: the pages' softmax(logits / T) numerator
  const float kx = 1.4426950408889634f / fmaxf(T, kMinT);

  // ---- pass 1: e = exp((l - max) / T) in place (pads stay above every key),
  //      and the first digit's histogram when a cut is on
  int slot = 1;
  const bool hist1 = topk_on || topp_on;
  if (hist1) {
    sh.hist[slot][tid] = 0;
    __syncthreads();
  }
  for (int g = tid; g < n4; g += kThreads) {
    uint4 w = reinterpret_cast<uint4 *>(val)[g];
    uint32_t b[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int j = 4 * g + q - off;            // element of the slice, or a pad
      if (j >= 0 && j < n) b[q] = __float_as_uint(ex2((__uint_as_float(b[q]) - M) * kx));
      else b[q] = kPadBits;
      if (hist1) {
        const uint32_t key = key_of(b[q]);
        if ((key >> 30) == 0)
          atomicAdd(&sh.hist[slot][key >> 22], topk_on ? 1ull : mass_of(b[q]));
      }
    }
    reinterpret_cast<uint4 *>(val)[g] = make_uint4(b[0], b[1], b[2], b[3]);
  }
  __syncthreads();                              // the draw reads other threads' groups

  // ---- top-k: the key d_k of rank k-1 (ascending key, ties in token order)
  uint32_t dk = 0x7fffffffu;                    // every real key is below this when top-k is off
  unsigned long long rk = 0, ties_k = 0;        // ties of d_k kept, ties of d_k in all
  bool ok = true;
  if (topk_on) {
    uint32_t prefix = 0;
    unsigned long long need = (unsigned long long)k;
    for (int d = 0; d < 4; ++d) {
      const int sh_ = digit_shift(d), wd = digit_width(d), hi = sh_ + wd;
      if (d > 0) {
        slot ^= 1;
        sh.hist[slot][tid] = 0;
        __syncthreads();
        for (int g = tid; g < n4; g += kThreads) {
          const uint4 w = reinterpret_cast<const uint4 *>(val)[g];
          const uint32_t b[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint32_t key = key_of(b[q]);
            if ((key >> hi) == (prefix >> hi))
              atomicAdd(&sh.hist[slot][(key >> sh_) & ((1u << wd) - 1)], 1ull);
          }
        }
      }
      cluster_barrier();
      ok &= select_bucket(sh, slot, C, need, -1, 0, nullptr);
      if (!ok) break;
      need -= sh.pick64[0];
      prefix |= sh.pick[0] << sh_;
      if (d == 3) ties_k = sh.pick64[1];
    }
    dk = prefix;
    rk = need;
  }

  // ---- top-p over the top-k set: the key d_p where the mass ranked ahead
  //      first reaches tau = ceil(P * S_k), and how many of its ties stay
  uint32_t dsel = topk_on ? dk : kOneBits + 1; // final threshold key
  unsigned long long tsel = topk_on ? rk : 0;  //   and ties of it kept
  if (ok && topp_on) {
    const unsigned long long wk = topk_on ? mass_of(kOneBits - dk) : 0;
    const unsigned long long drop = topk_on ? (ties_k - rk) * wk : 0;
    uint32_t prefix = 0;
    unsigned long long tau = 0, A = 0, wsel = 0;
    for (int d = 0; d < 4; ++d) {
      const int sh_ = digit_shift(d), wd = digit_width(d), hi = sh_ + wd;
      if (d > 0 || topk_on) {
        slot ^= 1;
        sh.hist[slot][tid] = 0;
        __syncthreads();
        for (int g = tid; g < n4; g += kThreads) {
          const uint4 w = reinterpret_cast<const uint4 *>(val)[g];
          const uint32_t b[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint32_t key = key_of(b[q]);
            if ((key >> hi) == (prefix >> hi) && key <= dk)
              atomicAdd(&sh.hist[slot][(key >> sh_) & ((1u << wd) - 1)], mass_of(b[q]));
          }
        }
      }
      cluster_barrier();
      // the ties of d_k beyond the first rk are not in the top-k set
      const int adj = (topk_on && (dk >> hi) == (prefix >> hi)) ? (int)((dk >> sh_) & ((1u << wd) - 1)) : -1;
      if (d == 0) {
        unsigned long long S = 0;
        // first the total (S_k), then the selection against tau
        const int b = tid;
        unsigned long long h = 0;
        for (int c = 0; c < C; ++c) h += ld_cluster_u64(&sh.hist[slot][b], (uint32_t)c);
        if (b == adj) h -= drop;
        S = warp_sum(h);
        if (lane == 0) sh.scan[warp] = S;
        __syncthreads();
        S = 0;
        for (int w = 0; w < kWarps; ++w) S += sh.scan[w];
        __syncthreads();
        tau = (unsigned long long)ceil((double)P * (double)S);
      }
      ok &= select_bucket(sh, slot, C, tau - A, adj, drop, nullptr);
      if (!ok) break;
      A += sh.pick64[0];
      prefix |= sh.pick[0] << sh_;
      if (d == 3) wsel = sh.pick64[1];
    }
    if (ok) {
      // every tie of d_p has the same mass w; keep ties while the mass ahead
      // of them is below tau
      const unsigned long long w = mass_of(kOneBits - prefix);
      const unsigned long long avail = w ? wsel / w : 0;
      unsigned long long nt = w ? (tau - A + w - 1) / w : 0;
      if (nt < 1) nt = 1;
      if (nt > avail) nt = avail;
      ok = w != 0 && avail != 0;
      dsel = prefix;
      tsel = nt;
    }
  }

  // ---- the draw, part 1: per warp (contiguous ranges) and per CTA, the
  //      mass of keys below dsel and the count of keys equal to it
  const int G = (n4 + kWarps - 1) / kWarps;    // groups of 4 per warp
  const int g0 = warp * G, g1 = min(n4, g0 + G);
  unsigned long long mlt = 0, teq = 0;
  for (int g = g0 + lane; g < g1; g += 32) {
    const uint4 w = reinterpret_cast<const uint4 *>(val)[g];
    const uint32_t b[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t key = key_of(b[q]);
      if (key < dsel) mlt += mass_of(b[q]);
      teq += key == dsel;
    }
  }
  mlt = warp_sum(mlt);
  teq = warp_sum(teq);
  if (lane == 0) {
    sh.wmass[warp] = mlt;
    sh.wties[warp] = (uint32_t)teq;
  }
  __syncthreads();
  if (tid == 0) {                               // scal[0] held pass 0's values: use scal[1]
    unsigned long long a = 0, t = 0;
    for (int w = 0; w < kWarps; ++w) {
      a += sh.wmass[w];
      t += sh.wties[w];
    }
    sh.scal[1][0] = a;
    sh.scal[1][1] = t;
  }
  cluster_barrier();
  const unsigned long long wd = dsel <= kOneBits ? mass_of(kOneBits - dsel) : 0;
  unsigned long long S = 0, base = 0, tie_base = 0, ties_before = 0;
  int cstar = -1;
  {
    unsigned long long Kc[kMaxCluster], tc[kMaxCluster];
#pragma unroll
    for (int c = 0; c < kMaxCluster; ++c) {
      Kc[c] = tc[c] = 0;
      if (c >= C) continue;
      const unsigned long long m = ld_cluster_u64(&sh.scal[1][0], (uint32_t)c);
      tc[c] = ld_cluster_u64(&sh.scal[1][1], (uint32_t)c);
      const unsigned long long keep =
          tsel > ties_before ? (tsel - ties_before < tc[c] ? tsel - ties_before : tc[c]) : 0;
      Kc[c] = m + keep * wd;
      ties_before += tc[c];
      S += Kc[c];
    }
    const unsigned long long U = (unsigned long long)floor((double)u * (double)S);
    unsigned long long run = 0, tb = 0;
#pragma unroll
    for (int c = 0; c < kMaxCluster; ++c) {
      if (c >= C) break;
      if (cstar < 0 && run + Kc[c] > U) {
        cstar = c;
        base = U - run;                         // target inside CTA c: first cum > base
        tie_base = tb;
      }
      run += Kc[c];
      tb += tc[c];
    }
  }
  cluster_barrier();                            // every remote read is done
  if (!ok || S == 0 || cstar < 0) {
    if (tid == 0 && rank == 0) {
      report(p.status, MSG_DEV_INTERNAL, row, 0);
      p.tokens[row] = -1;
    }
    return;
  }
  if ((int)rank != cstar) return;

  // ---- the draw, part 2 (one CTA): the warp, then the token
  int wstar = -1;
  unsigned long long wbase = 0, wtie = 0;
  {
    unsigned long long run = 0, tb = tie_base;
    for (int w = 0; w < kWarps; ++w) {
      const unsigned long long keep =
          tsel > tb ? (tsel - tb < sh.wties[w] ? tsel - tb : sh.wties[w]) : 0;
      const unsigned long long Kw = sh.wmass[w] + keep * wd;
      if (wstar < 0 && run + Kw > base) {
        wstar = w;
        wbase = base - run;
        wtie = tb;
      }
      run += Kw;
      tb += sh.wties[w];
    }
  }
  if (warp != wstar) return;
  unsigned long long run = 0, ties = wtie;
  for (int gb = g0; gb < g1; gb += 32) {
    const int g = gb + lane;
    uint32_t b[4] = {kPadBits, kPadBits, kPadBits, kPadBits};
    if (g < g1) {
      const uint4 w = reinterpret_cast<const uint4 *>(val)[g];
      b[0] = w.x; b[1] = w.y; b[2] = w.z; b[3] = w.w;
    }
    uint32_t my_ties = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q) my_ties += key_of(b[q]) == dsel;
    uint32_t tie_excl = my_ties;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xffffffffu, tie_excl, o);
      if (lane >= o) tie_excl += y;
    }
    const uint32_t tie_total = __shfl_sync(0xffffffffu, tie_excl, 31);
    tie_excl -= my_ties;
    unsigned long long m[4], mine = 0;
#pragma unroll
    for (int q = 0, t = 0; q < 4; ++q) {
      const uint32_t key = key_of(b[q]);
      m[q] = 0;
      if (key < dsel) m[q] = mass_of(b[q]);
      else if (key == dsel) {
        if (ties + tie_excl + t < tsel) m[q] = wd;
        ++t;
      }
      mine += m[q];
    }
    unsigned long long incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const unsigned long long y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const unsigned int hit = __ballot_sync(0xffffffffu, run + incl > wbase);
    if (hit) {
      if (lane == __ffs(hit) - 1) {
        unsigned long long acc = run + incl - mine;
        int q = 0;
        for (; q < 3; ++q) {
          acc += m[q];
          if (acc > wbase) break;
        }
        p.tokens[row] = (int32_t)(lo + 4 * (int64_t)g + q - off);
      }
      return;
    }
    run += __shfl_sync(0xffffffffu, incl, 31);
    ties += tie_total;
  }
  if (lane == 0) {
    report(p.status, MSG_DEV_INTERNAL, row, 1);
    p.tokens[row] = -1;
  }
}

template <bool kBf16, bool kGreedy>
cudaError_t launch_sample(const SampleParams &p, int C, cudaStream_t s) {
  auto kernel = sample_kernel<kBf16, kGreedy>;
  const size_t smem = sizeof(Shared) + (kGreedy ? 0 : ((size_t)p.slice + 8) * 4);
  static size_t configured = 0;
  if (smem > 48 * 1024 && smem > configured) {
    const cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    configured = smem;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.batch * C));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

}  // namespace

}  // namespace msg

extern "C" int msg_sample_slices(int32_t vocab, int32_t *cluster_out, int32_t *slice_out) {
  using namespace msg;
  if (vocab < 1) return MSG_ERR_INVALID_ARG;
  int C = 1;
  while (C < kMaxCluster && (vocab + C - 1) / C > kSliceTwoPerSm) C *= 2;
  int64_t slice = ((int64_t)vocab + C - 1) / C;
  slice = (slice + kSliceAlign - 1) / kSliceAlign * kSliceAlign;
  if (slice > kSliceMax) return MSG_ERR_UNSUPPORTED;
  if (cluster_out) *cluster_out = C;
  if (slice_out) *slice_out = (int32_t)slice;
  return MSG_OK;
}

extern "C" int msg_sample(const void *logits, int32_t logits_dtype, int64_t logits_row_stride,
                          int32_t batch, int32_t vocab, const float *temperatures,
                          const int32_t *top_k, const float *top_p, const float *uniforms,
                          int32_t *tokens_out, int32_t *dev_status, void *stream) {
  using namespace msg;
  if (logits_dtype != MSG_DTYPE_F32 && logits_dtype != MSG_DTYPE_BF16) return MSG_ERR_UNSUPPORTED;
  if (batch < 0 || vocab < 1 || logits_row_stride < vocab) return MSG_ERR_INVALID_ARG;
  int32_t C = 0, slice = 0;
  const int rc = msg_sample_slices(vocab, &C, &slice);
  if (rc != MSG_OK) return rc;
  if (batch == 0) return MSG_OK;
  if (logits == nullptr || tokens_out == nullptr) return MSG_ERR_INVALID_ARG;
  if (temperatures != nullptr && uniforms == nullptr) return MSG_ERR_INVALID_ARG;
  if ((int64_t)batch * C > 0x7fffffffLL) return MSG_ERR_INVALID_ARG;
  const int esz = logits_dtype == MSG_DTYPE_BF16 ? 2 : 4;
  if (reinterpret_cast<uintptr_t>(logits) % esz) return MSG_ERR_ALIGNMENT;
  SampleParams p{};
  p.logits = static_cast<const uint8_t *>(logits);
  p.row_bytes = logits_row_stride * esz;
  p.batch = batch;
  p.vocab = vocab;
  p.slice = slice;
  p.temperature = temperatures;
  p.top_k = top_k;
  p.top_p = top_p;
  p.uniform = uniforms;
  p.tokens = tokens_out;
  p.status = dev_status;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  const bool bf = logits_dtype == MSG_DTYPE_BF16;
  if (temperatures == nullptr)
    e = bf ? launch_sample<true, true>(p, C, s) : launch_sample<false, true>(p, C, s);
  else
    e = bf ? launch_sample<true, false>(p, C, s) : launch_sample<false, false>(p, C, s);
  return e == cudaSuccess ? MSG_OK : MSG_ERR_CUDA;
}

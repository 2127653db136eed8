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
// GB300 layout: a scan kernel over all SMs reads every row from HBM once and
// keeps, per chunk of 256 logits, its maximum and its mass relative to that
// maximum, plus a sparse sample of the row; a batch of bf16 logits (78 MB for
// 256 x 151,936) then stays in L2 for the few later reads by the row kernel,
// one CTA per row.  A row without a cut draws straight from the chunk masses
// (one more read of a single chunk).  With a cut, the k-th token or the top-p
// boundary is located inside a small window of logit values: the window is
// estimated from the chunk maxima or from the sample (for top-p, a second
// estimate corrected by the exact mass the first gather measured at its edge
// when the first window misses), tightened when needed by probe passes that
// count logits and sum masses above four pivots, then gathered (at most kCap
// logits), sorted by (logit desc, index asc) and resolved exactly.  The kept set is "every token ranked at or before the threshold
// token", so the draw needs no rank bookkeeping: either the whole kept set is
// in the window (a sort by index and one scan), or the gather also summed,
// per chunk, the mass above the window and the draw walks the chunks.
//
// Masses are fp32 2^((l - max) * log2(e) / T) summed in a fixed order (no
// atomics), so a row's token is deterministic.
//
// The row kernel's CTAs take the rows in order of a cost class read from the
// parameters (top-p cuts over whole distributions first), so each long row
// gets an SM of its own.  A batch without temperatures (every row greedy)
// runs one kernel instead: a CTA per row reads it once and keeps its first
// maximum.
#include <math.h>
#include <stddef.h>

#include "internal.cuh"

namespace msg {

namespace {

constexpr int kT = 512;                        // threads: one CTA per row
constexpr int kW = kT / 32;
constexpr int kLE = 8;                         // logits a lane holds of a chunk
constexpr int kChunk = 32 * kLE;               // logits per chunk
constexpr int kMaxVocab = 425984;
constexpr int kMaxChunks = (kMaxVocab / kLE + 31) / 32 + 2;   // + the head and tail chunks
constexpr int kSortChunks = 2048;              // power of two >= kMaxChunks
constexpr int kCap = 4096;                     // window capacity (logits)
constexpr int kMaxSamples = 4096;
constexpr int kMaxProbes = 48;
constexpr float kMinT = 1e-6f;                 // Sampler.prepare's MIN_T
constexpr float kMinP = 1e-6f;                 // Sampler.prepare's MIN_P
constexpr unsigned long long kKeyEnd = 1ull << 32;   // one past every order key
static_assert(kMaxChunks <= kSortChunks, "chunk maxima are sorted in one power-of-two array");

struct SampleParams {
  const uint8_t *logits;
  int64_t row_bytes;                           // bytes between rows
  int32_t batch, vocab;
  const float *temperature;                    // null: every row greedy
  const int32_t *top_k;                        // null: no top-k
  const float *top_p;                          // null: no top-p
  const float *uniform;
  int32_t *tokens;
  int32_t *status;
};

struct Smem {
  float cmax[kMaxChunks];                      // per chunk: largest logit
  float cmass[kMaxChunks];                     //   mass (rel. to cmax, then to the row max)
  float cabove[kMaxChunks];                    //   mass above the window / kept mass
  unsigned long long csort[kSortChunks];       // (~key << 32) | chunk of the chunk maxima, ascending
  float csamp[kMaxChunks];                     // per chunk: mass of its sample points
  uint32_t samp[kMaxSamples];                  // ~key of the sample, sorted ascending
  unsigned long long list[kCap];               // window: (~key << 32) | index, sorted ascending
  float lcum[kCap];                            // window: cumulative masses in list order
  float fred[kW];
  unsigned long long ured[kW];
  int ival[8];
  float fval[4];
};
// the draw reuses the sample's array for per-chunk 64-bit sums
static_assert(offsetof(Smem, samp) % 8 == 0 && kMaxSamples / 2 >= kMaxChunks,
              "samp holds kMaxChunks 64-bit sums");

// ---- keys and masses
// Order key of a logit: increasing with the value (-0 is read as +0).
__device__ __forceinline__ uint32_t key_of(float f) {
  const uint32_t u = __float_as_uint(f + 0.f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float value_of(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}
// Key of the chunk maximum at position i of csort.
__device__ __forceinline__ uint32_t ckey(const Smem &sm, int i) {
  return ~(uint32_t)(sm.csort[i] >> 32);
}
// last_at_least over csort positions [p0, p1).
__device__ __forceinline__ int last_at_least_c(const Smem &sm, int p0, int p1, uint32_t K) {
  int lo = p0, hi = p1;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (ckey(sm, mid) >= K) lo = mid + 1;
    else hi = mid;
  }
  return lo - 1;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Pairwise fp32 arithmetic (one instruction for two IEEE round-to-nearest
// operations) and a maximum that returns NaN when either input is NaN.
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float fmax_nan(float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}

// ---- block primitives (every thread calls; every thread gets the result)
__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ float warp_max_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float block_sum_f(float v, Smem &sm) {
  v = warp_sum_f(v);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) sm.fred[threadIdx.x >> 5] = v;
  __syncthreads();
  float s = 0.f;
#pragma unroll
  for (int w = 0; w < kW; ++w) s += sm.fred[w];
  return s;
}
__device__ __forceinline__ float block_max_f(float v, Smem &sm) {
  v = warp_max_f(v);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) sm.fred[threadIdx.x >> 5] = v;
  __syncthreads();
  float s = -INFINITY;
#pragma unroll
  for (int w = 0; w < kW; ++w) s = fmaxf(s, sm.fred[w]);
  return s;
}
__device__ __forceinline__ unsigned long long block_sum_u(unsigned long long v, Smem &sm) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) sm.ured[threadIdx.x >> 5] = v;
  __syncthreads();
  unsigned long long s = 0;
#pragma unroll
  for (int w = 0; w < kW; ++w) s += sm.ured[w];
  return s;
}
__device__ __forceinline__ unsigned long long block_max_u(unsigned long long v, Smem &sm) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long y = __shfl_xor_sync(0xffffffffu, v, o);
    v = y > v ? y : v;
  }
  __syncthreads();
  if ((threadIdx.x & 31) == 0) sm.ured[threadIdx.x >> 5] = v;
  __syncthreads();
  unsigned long long s = 0;
#pragma unroll
  for (int w = 0; w < kW; ++w) s = sm.ured[w] > s ? sm.ured[w] : s;
  return s;
}
__device__ __forceinline__ int block_min_i(int v, Smem &sm) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
  __syncthreads();
  if ((threadIdx.x & 31) == 0) sm.ured[threadIdx.x >> 5] = (unsigned long long)(uint32_t)v;
  __syncthreads();
  int s = v;
#pragma unroll
  for (int w = 0; w < kW; ++w) s = min(s, (int)(uint32_t)sm.ured[w]);
  return s;
}
// Exclusive scan of one float per thread, in thread order; the total in *tot.
__device__ __forceinline__ float block_excl_scan_f(float v, Smem &sm, float *tot) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  __syncthreads();
  if (lane == 31) sm.fred[warp] = x;
  __syncthreads();
  float before = 0.f, all = 0.f;
#pragma unroll
  for (int w = 0; w < kW; ++w) {
    const float t = sm.fred[w];
    if (w < warp) before += t;
    all += t;
  }
  *tot = all;
  return before + x - v;
}

// Ascending bitonic sort of n (a power of two, >= 2) entries in shared
// memory.  Stages whose pairs lie inside one warp's contiguous segment of
// n / kW entries synchronise only that warp; the others the whole block.
template <typename T>
__device__ void bitonic_sort_smem(T *a, int n) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int seg = n >= 2 * kW ? n / kW : n;     // entries per warp segment
  const bool warp_local = n >= 2 * kW;
  for (int k = 2; k <= n; k <<= 1) {
    int j = k >> 1;
    for (; j > 0 && (!warp_local || j >= seg); j >>= 1) {   // block-wide stages
      for (int i = threadIdx.x; i < (n >> 1); i += kT) {
        const int lo = 2 * i - (i & (j - 1)), hi = lo + j;
        const T x = a[lo], y = a[hi];
        if ((x > y) == ((lo & k) == 0)) {
          a[lo] = y;
          a[hi] = x;
        }
      }
      __syncthreads();
    }
    if (j == 0) continue;
    T *b = a + warp * seg;                      // warp-local stages
    const int base = warp * seg;
    for (; j > 0; j >>= 1) {
      for (int i = lane; i < (seg >> 1); i += 32) {
        const int lo = 2 * i - (i & (j - 1)), hi = lo + j;
        const T x = b[lo], y = b[hi];
        if ((x > y) == (((base + lo) & k) == 0)) {
          b[lo] = y;
          b[hi] = x;
        }
      }
      __syncwarp();
    }
    __syncthreads();
  }
}
// The same sort for n = kT * E: thread t holds entries t*E .. t*E+E-1 in
// registers.  A stage with pair distance j < E exchanges registers of one
// thread, E <= j < 32 E exchanges with lane ^ (j / E) by shuffle, and only
// the stages with j >= 32 E go through shared memory (the whole block).
template <typename T, int E>
__device__ void bitonic_sort_reg(T *a) {
  constexpr int n = kT * E;
  const int t = threadIdx.x;
  T r[E];
#pragma unroll
  for (int e = 0; e < E; ++e) r[e] = a[t * E + e];
  for (int k = 2; k <= n; k <<= 1) {
    int j = k >> 1;
    if (j >= 32 * E) {                          // pairs across warps: shared memory
#pragma unroll
      for (int e = 0; e < E; ++e) a[t * E + e] = r[e];
      __syncthreads();
      for (; j >= 32 * E; j >>= 1) {
        for (int i = t; i < (n >> 1); i += kT) {
          const int lo = 2 * i - (i & (j - 1)), hi = lo + j;
          const T x = a[lo], y = a[hi];
          if ((x > y) == ((lo & k) == 0)) {
            a[lo] = y;
            a[hi] = x;
          }
        }
        __syncthreads();
      }
#pragma unroll
      for (int e = 0; e < E; ++e) r[e] = a[t * E + e];
    }
    // pairs across lanes: every register of the thread is on the same side
    const bool up = ((t * E) & k) == 0;         // k > j >= E: the same for all e
    for (; j >= E; j >>= 1) {
      const bool keep_min = (((t * E) & j) == 0) == up;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const T o = __shfl_xor_sync(0xffffffffu, r[e], j / E);
        r[e] = keep_min ? (o < r[e] ? o : r[e]) : (o > r[e] ? o : r[e]);
      }
    }
    // pairs inside the thread
#pragma unroll
    for (int jj = E >> 1; jj > 0; jj >>= 1) {
      if (jj < k) {
#pragma unroll
        for (int e = 0; e < E; ++e) {
          if (e & jj) continue;
          const T x = r[e], y = r[e + jj];
          if ((x > y) == (((t * E + e) & k) == 0)) {
            r[e] = y;
            r[e + jj] = x;
          }
        }
      }
    }
  }
  __syncthreads();                              // every read of a[] above is done
#pragma unroll
  for (int e = 0; e < E; ++e) a[t * E + e] = r[e];
  __syncthreads();
}

// Ascending sort of n (a power of two, >= 2) entries in shared memory.
template <typename T>
__device__ void bitonic_sort(T *a, int n) {
  if (n == 8 * kT) {
    bitonic_sort_reg<T, 8>(a);
  } else if (n == 4 * kT) {
    bitonic_sort_reg<T, 4>(a);
  } else if (n == 2 * kT) {
    bitonic_sort_reg<T, 2>(a);
  } else if (n == kT) {
    bitonic_sort_reg<T, 1>(a);
  } else {
    bitonic_sort_smem(a, n);
  }
}

__device__ __forceinline__ int pow2_at_least(int n) {
  int p = 2;
  while (p < n) p <<= 1;
  return p;
}

// ---- the row: a head of h logits up to the first 16-byte boundary, nvec
// vectors of 8 logits (16 bytes of bf16, 32 of fp32), a tail of < 8 logits.
// Logical chunk 0 is the head (lane 0), chunks 1..nch hold 32 vectors each,
// chunk nch + 1 is the tail (lane 0); chunk order is index order.
struct RowRef {
  const uint8_t *p;
  int V, h, nvec, nch, tail;
};

template <bool kBf16>
__device__ __forceinline__ RowRef row_ref(const uint8_t *p, int V) {
  constexpr int esz = kBf16 ? 2 : 4;
  int h = (int)(((16u - (uint32_t)(reinterpret_cast<uintptr_t>(p) & 15u)) & 15u) / esz);
  if (h > V) h = V;
  const int nvec = (V - h) / kLE;
  return {p, V, h, nvec, (nvec + 31) / 32, V - h - kLE * nvec};
}

template <bool kBf16>
__device__ __forceinline__ float load1(const uint8_t *row, int j) {
  if (kBf16) return __uint_as_float((uint32_t)reinterpret_cast<const uint16_t *>(row)[j] << 16);
  return reinterpret_cast<const float *>(row)[j];
}

template <bool kBf16>
__device__ __forceinline__ void load8(const uint8_t *p, float v[kLE]) {
  if (kBf16) {
    uint4 r;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    v[0] = bf16lo(r.x); v[1] = bf16hi(r.x); v[2] = bf16lo(r.y); v[3] = bf16hi(r.y);
    v[4] = bf16lo(r.z); v[5] = bf16hi(r.z); v[6] = bf16lo(r.w); v[7] = bf16hi(r.w);
  } else {
    float4 a, b;
    asm volatile("ld.global.nc.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(a.x), "=f"(a.y), "=f"(a.z), "=f"(a.w) : "l"(p));
    asm volatile("ld.global.nc.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(b.x), "=f"(b.y), "=f"(b.z), "=f"(b.w) : "l"(p + 16));
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
}

// The lane's logits of logical chunk c: how many (0..8), and the first one's index.
template <bool kBf16>
__device__ __forceinline__ int chunk_lane(const RowRef &r, int c, int lane, float v[kLE], int &idx0) {
  constexpr int esz = kBf16 ? 2 : 4;
  int n = 0;
  if (c == 0 || c == r.nch + 1) {
    idx0 = c == 0 ? 0 : r.h + kLE * r.nvec;
    n = lane == 0 ? (c == 0 ? r.h : r.tail) : 0;
#pragma unroll
    for (int j = 0; j < kLE; ++j) v[j] = j < n ? load1<kBf16>(r.p, idx0 + j) : 0.f;
  } else {
    const int vi = 32 * (c - 1) + lane;
    idx0 = r.h + kLE * vi;
    if (vi < r.nvec) {
      n = kLE;
      load8<kBf16>(r.p + (int64_t)idx0 * esz, v);
    } else {
#pragma unroll
      for (int j = 0; j < kLE; ++j) v[j] = 0.f;
    }
  }
  return n;
}

// Chunk holding token index i.
__device__ __forceinline__ int chunk_of(const RowRef &r, int i) {
  if (i < r.h) return 0;
  if (i >= r.h + kLE * r.nvec) return r.nch + 1;
  return 1 + (i - r.h) / kChunk;
}

constexpr int kPassUnrollBf16 = 4;             // chunks a warp has in flight in a row pass
constexpr int kPassUnrollF32 = 2;

// A pass over the row's chunks: warp w takes logical chunks 1 + w, 1 + w + kW,
// ... with 4 (bf16) or 2 (fp32) chunks' loads in flight, then the head and tail chunks
// (warps 0 and 1).  A chunk with keep(c) false is not read; skip(c) runs
// instead (lane-uniform).  body(v, n, i0, c) sees the lane's logits.
template <bool kBf16, typename Keep, typename Skip, typename Body>
__device__ __forceinline__ void for_chunks(const RowRef &r, Keep keep, Skip skip, Body body) {
  constexpr int esz = kBf16 ? 2 : 4;
  constexpr int kWords = kBf16 ? 1 : 2;
  constexpr int kPassUnroll = kBf16 ? kPassUnrollBf16 : kPassUnrollF32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int c0 = 1 + warp; c0 <= r.nch; c0 += kW * kPassUnroll) {
    uint4 raw[kPassUnroll][kWords];
    bool on[kPassUnroll];
#pragma unroll
    for (int q = 0; q < kPassUnroll; ++q) {
      const int c = c0 + q * kW;
      on[q] = c <= r.nch && keep(c);
      const int vi = 32 * (c - 1) + lane;
      if (on[q] && vi < r.nvec) {
        const uint8_t *src = r.p + (int64_t)(r.h + kLE * vi) * esz;
#pragma unroll
        for (int w = 0; w < kWords; ++w)
          asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                       : "=r"(raw[q][w].x), "=r"(raw[q][w].y), "=r"(raw[q][w].z), "=r"(raw[q][w].w)
                       : "l"(src + 16 * w));
      }
    }
#pragma unroll
    for (int q = 0; q < kPassUnroll; ++q) {
      const int c = c0 + q * kW;
      if (c > r.nch) break;                     // warp-uniform
      if (!on[q]) {
        skip(c);
        continue;
      }
      const int vi = 32 * (c - 1) + lane;
      const int n = vi < r.nvec ? kLE : 0;
      float v[kLE];
      if (kBf16) {
        const uint4 w = raw[q][0];
        v[0] = bf16lo(w.x); v[1] = bf16hi(w.x); v[2] = bf16lo(w.y); v[3] = bf16hi(w.y);
        v[4] = bf16lo(w.z); v[5] = bf16hi(w.z); v[6] = bf16lo(w.w); v[7] = bf16hi(w.w);
      } else {
        const uint4 a = raw[q][0], b = raw[q][kWords - 1];
        v[0] = __uint_as_float(a.x); v[1] = __uint_as_float(a.y);
        v[2] = __uint_as_float(a.z); v[3] = __uint_as_float(a.w);
        v[4] = __uint_as_float(b.x); v[5] = __uint_as_float(b.y);
        v[6] = __uint_as_float(b.z); v[7] = __uint_as_float(b.w);
      }
      body(v, n, r.h + kLE * vi, c);
    }
  }
  if (warp < 2) {                               // head (warp 0) and tail (warp 1)
    const int c = warp == 0 ? 0 : r.nch + 1;
    if (!keep(c)) {
      skip(c);
    } else {
      float v[kLE];
      int i0;
      const int n = chunk_lane<kBf16>(r, c, lane, v, i0);
      body(v, n, i0, c);
    }
  }
}

// ---- row state (every thread holds the same copy)
struct Ctx {
  RowRef r;
  int nl;                                      // logical chunks
  float M, kx;                                 // row maximum, log2(e) / T
  float S;                                     // row mass (relative to M)
  int ns;                                      // valid samples (sorted, first)
  int spc;                                     // samples per vector chunk
};

__device__ __forceinline__ float mass_of(const Ctx &x, float l) { return ex2((l - x.M) * x.kx); }

// Load the lane's 8 logits of vector chunk c (1-based logical index) into raw.
template <bool kBf16>
__device__ __forceinline__ bool load_chunk_raw(const RowRef &r, int c, int lane, uint4 raw[2]) {
  const int vi = 32 * (c - 1) + lane;
  if (vi >= r.nvec) return false;
  const uint8_t *src = r.p + (int64_t)(r.h + kLE * vi) * (kBf16 ? 2 : 4);
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(raw[0].x), "=r"(raw[0].y), "=r"(raw[0].z), "=r"(raw[0].w) : "l"(src));
  if (!kBf16)
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(raw[1].x), "=r"(raw[1].y), "=r"(raw[1].z), "=r"(raw[1].w) : "l"(src + 16));
  return true;
}
template <bool kBf16>
__device__ __forceinline__ void unpack_raw(const uint4 raw[2], float v[kLE]) {
  if (kBf16) {
    const uint4 w = raw[0];
    v[0] = bf16lo(w.x); v[1] = bf16hi(w.x); v[2] = bf16lo(w.y); v[3] = bf16hi(w.y);
    v[4] = bf16lo(w.z); v[5] = bf16hi(w.z); v[6] = bf16lo(w.w); v[7] = bf16hi(w.w);
  } else {
    v[0] = __uint_as_float(raw[0].x); v[1] = __uint_as_float(raw[0].y);
    v[2] = __uint_as_float(raw[0].z); v[3] = __uint_as_float(raw[0].w);
    v[4] = __uint_as_float(raw[1].x); v[5] = __uint_as_float(raw[1].y);
    v[6] = __uint_as_float(raw[1].z); v[7] = __uint_as_float(raw[1].w);
  }
}

// Smallest logit value whose order key is >= K (K up to 2^32): -inf when
// every value qualifies, NaN (every comparison false) when none does.  So
// key_of(f) >= K exactly when f >= min_value_at_least(K), for every non-NaN f.
__device__ __forceinline__ float min_value_at_least(unsigned long long K) {
  if (K <= key_of(-INFINITY)) return -INFINITY;
  if (K > key_of(INFINITY)) return __uint_as_float(0x7fffffffu);
  if (K == 0x7fffffffull) return 0.f;          // the key of -0, which no logit has
  return value_of((uint32_t)K);
}

// One chunk of the gather (all lanes): window logits appended; returns the
// lane's mass of the logits above the window (the caller sums the warp).
// f_lo / f_above: min_value_at_least of the window's bounds lo and hi.
__device__ __forceinline__ float gather_chunk(const Ctx &x, Smem &sm, const float v[kLE], int n,
                                              int i0, float f_lo, float f_above, uint32_t &ca) {
  float ma = 0.f;
  uint32_t wmask = 0;
#pragma unroll
  for (int j = 0; j < kLE; ++j) {
    if (j < n && v[j] >= f_lo) {
      if (v[j] >= f_above) {
        ++ca;
        ma += mass_of(x, v[j]);
      } else {
        wmask |= 1u << j;
      }
    }
  }
  if (wmask) {                                  // window logits are few: a slot reservation per lane
    int base = atomicAdd(&sm.ival[0], __popc(wmask));
#pragma unroll
    for (int j = 0; j < kLE; ++j)
      if ((wmask >> j) & 1u) {
        if (base < kCap) sm.list[base] = ((unsigned long long)(~key_of(v[j])) << 32) | (uint32_t)(i0 + j);
        ++base;
      }
  }
  return ma;
}

// Window [lo, hi) of order keys: gather its logits into the list (at most kCap
// stored; the full count is returned), and per chunk the mass of the logits
// at or above hi (cabove); *cnt_above / *mass_above get their totals.
template <bool kBf16>
__device__ int gather(const Ctx &x, Smem &sm, uint32_t lo, unsigned long long hi,
                      unsigned long long *cnt_above, float *mass_above) {
  constexpr int U = kBf16 ? kPassUnrollBf16 : kPassUnrollF32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();
  if (threadIdx.x == 0) sm.ival[0] = 0;
  __syncthreads();
  uint32_t ca = 0;
  // keys in [lo, hi) are in the window, keys at or above hi above it
  const float f_lo = min_value_at_least(lo);
  const float f_above = min_value_at_least(hi);
  for (int c0 = 1 + warp; c0 <= x.r.nch; c0 += kW * U) {
    uint4 raw[U][2];
    bool on[U], got[U];
#pragma unroll
    for (int q = 0; q < U; ++q) {
      const int c = c0 + q * kW;
      on[q] = c <= x.r.nch && sm.cmax[c] != -INFINITY && key_of(sm.cmax[c]) >= lo;
      got[q] = on[q] && load_chunk_raw<kBf16>(x.r, c, lane, raw[q]);
    }
    float ma[U];
#pragma unroll
    for (int q = 0; q < U; ++q) {
      const int c = c0 + q * kW;
      ma[q] = 0.f;
      if (c > x.r.nch || !on[q]) continue;      // warp-uniform
      float v[kLE];
      unpack_raw<kBf16>(raw[q], v);
      ma[q] = gather_chunk(x, sm, v, got[q] ? kLE : 0, x.r.h + kLE * (32 * (c - 1) + lane), f_lo,
                           f_above, ca);
    }
    // the chunks' above-window masses, reduced together
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
#pragma unroll
      for (int q = 0; q < U; ++q) ma[q] += __shfl_xor_sync(0xffffffffu, ma[q], o);
    if (lane == 0) {
#pragma unroll
      for (int q = 0; q < U; ++q)
        if (c0 + q * kW <= x.r.nch) sm.cabove[c0 + q * kW] = ma[q];
    }
  }
  if (warp < 2) {                               // head (warp 0) and tail (warp 1)
    const int c = warp == 0 ? 0 : x.r.nch + 1;
    if (sm.cmax[c] != -INFINITY && key_of(sm.cmax[c]) >= lo) {
      float v[kLE];
      int i0;
      const int n = chunk_lane<kBf16>(x.r, c, lane, v, i0);
      const float ma = warp_sum_f(gather_chunk(x, sm, v, n, i0, f_lo, f_above, ca));
      if (lane == 0) sm.cabove[c] = ma;
    } else if (lane == 0) {
      sm.cabove[c] = 0.f;
    }
  }
  *cnt_above = block_sum_u(ca, sm);
  float part = 0.f;                            // fixed order: thread t sums chunks t, t + kT, ...
  for (int c = threadIdx.x; c < x.nl; c += kT) part += sm.cabove[c];
  *mass_above = block_sum_f(part, sm);
  return sm.ival[0];
}

// Sort the gathered window (n <= kCap entries) and write cumulative masses.
__device__ void sort_window(const Ctx &x, Smem &sm, int n) {
  const int np = pow2_at_least(n);
  for (int i = n + threadIdx.x; i < np; i += kT) sm.list[i] = ~0ull;
  __syncthreads();
  bitonic_sort(sm.list, np);
  const int per = (n + kT - 1) / kT;           // thread t owns entries [t * per, (t + 1) * per)
  const int a = min(n, (int)threadIdx.x * per), b = min(n, a + per);
  float s = 0.f;
  for (int i = a; i < b; ++i) s += mass_of(x, value_of(~(uint32_t)(sm.list[i] >> 32)));
  float tot;
  float run = block_excl_scan_f(s, sm, &tot);
  for (int i = a; i < b; ++i) {
    run += mass_of(x, value_of(~(uint32_t)(sm.list[i] >> 32)));
    sm.lcum[i] = run;
  }
  __syncthreads();
}

// First list position (< n) whose cumulative mass plus `base` reaches tau; n if none.
__device__ int window_crossing(Smem &sm, int n, float base, float tau) {
  int best = n;
  for (int i = threadIdx.x; i < n; i += kT)
    if (base + sm.lcum[i] >= tau) {
      best = i;
      break;
    }
  return block_min_i(best, sm);
}

// Probe pass: count and mass of the logits at or above each of four pivots
// (descending keys); chunks whose maximum is below the smallest are skipped.
// f0..f3: min_value_at_least of the pivots (a value >= f_t has key >= piv[t]).
__device__ __forceinline__ void probe_chunk(const Ctx &x, const float v[kLE], int n, float f0,
                                            float f1, float f2, float f3, bool want_mass,
                                            uint32_t c4[4], float m4[4]) {
#pragma unroll
  for (int j = 0; j < kLE; ++j) {
    if (j >= n || !(v[j] >= f3)) continue;
    const float e = want_mass ? mass_of(x, v[j]) : 0.f;
    ++c4[3];
    m4[3] += e;
    const bool g2 = v[j] >= f2, g1 = v[j] >= f1, g0 = v[j] >= f0;
    c4[2] += g2;
    c4[1] += g1;
    c4[0] += g0;
    m4[2] += g2 ? e : 0.f;
    m4[1] += g1 ? e : 0.f;
    m4[0] += g0 ? e : 0.f;
  }
}

template <bool kBf16>
__device__ void probe(const Ctx &x, Smem &sm, const uint32_t piv[4], bool want_mass,
                      unsigned long long cnt[4], float mass[4]) {
  constexpr int U = kBf16 ? kPassUnrollBf16 : kPassUnrollF32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t c4[4] = {0, 0, 0, 0};
  float m4[4] = {0.f, 0.f, 0.f, 0.f};
  const uint32_t p3 = piv[3];
  const float f0 = min_value_at_least(piv[0]), f1 = min_value_at_least(piv[1]),
              f2 = min_value_at_least(piv[2]), f3 = min_value_at_least(p3);
  for (int c0 = 1 + warp; c0 <= x.r.nch; c0 += kW * U) {
    uint4 raw[U][2];
    bool got[U];
#pragma unroll
    for (int q = 0; q < U; ++q) {
      const int c = c0 + q * kW;
      got[q] = c <= x.r.nch && sm.cmax[c] != -INFINITY && key_of(sm.cmax[c]) >= p3 &&
               load_chunk_raw<kBf16>(x.r, c, lane, raw[q]);
    }
#pragma unroll
    for (int q = 0; q < U; ++q) {
      if (!got[q]) continue;
      float v[kLE];
      unpack_raw<kBf16>(raw[q], v);
      probe_chunk(x, v, kLE, f0, f1, f2, f3, want_mass, c4, m4);
    }
  }
  if (warp < 2) {
    const int c = warp == 0 ? 0 : x.r.nch + 1;
    if (sm.cmax[c] != -INFINITY && key_of(sm.cmax[c]) >= p3) {
      float v[kLE];
      int i0;
      const int n = chunk_lane<kBf16>(x.r, c, lane, v, i0);
      probe_chunk(x, v, n, f0, f1, f2, f3, want_mass, c4, m4);
    }
  }
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    cnt[q] = block_sum_u(c4[q], sm);
    mass[q] = want_mass ? block_sum_f(m4[q], sm) : 0.f;
  }
}

// Lower bound for the top-p boundary from the chunk maxima (csort, descending
// keys): the maxima at or above `lo` are distinct logits, so if the first r of
// them hold tau the boundary is at or above the r-th.  0 if they never do.
__device__ uint32_t chunk_max_bound(const Ctx &x, Smem &sm, uint32_t lo, float tau) {
  const int per = (x.nl + kT - 1) / kT;
  const int a = min(x.nl, (int)threadIdx.x * per), b = min(x.nl, a + per);
  float part = 0.f;
  for (int i = a; i < b; ++i) {
    const uint32_t kk = ckey(sm, i);
    if (sm.csort[i] != ~0ull && kk >= lo) part += mass_of(x, value_of(kk));
  }
  float tot;
  float run = block_excl_scan_f(part, sm, &tot);
  int first = x.nl;
  for (int i = a; i < b; ++i) {
    const uint32_t kk = ckey(sm, i);
    if (sm.csort[i] != ~0ull && kk >= lo) {
      run += mass_of(x, value_of(kk));
      if (run >= tau) {
        first = i;
        break;
      }
    }
  }
  first = block_min_i(first, sm);
  return first < x.nl ? ckey(sm, first) : 0u;
}

// Last position in [p0, p1) of a descending-key array stored as ~key
// (ascending) whose key is >= K; p0 - 1 if none.
__device__ __forceinline__ int last_at_least(const uint32_t *arr, int p0, int p1, uint32_t K) {
  int lo = p0, hi = p1;                         // first position with key < K
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (~arr[mid] >= K) lo = mid + 1;
    else hi = mid;
  }
  return lo - 1;
}

// Pivots for a top-p target inside (lo, hi): the mass at or above a key X is
// estimated as the exact mass at hi, plus the chunk maxima in [X, hi) (real
// logits, so the heavy tail of a peaked row is counted exactly), plus the
// sample points in [X, hi) weighted by the logits they stand for (the sample
// leaves out points that are their chunk's maximum, so nothing is counted
// twice; it carries the bulk of a flat row).  The
// pivots are the highest keys where the estimate reaches tau + g * f,
// f = -1/4, -1/12, 1/12, 1/4, with the spread g given by the caller.  Uses
// lcum and cabove as scratch.
__device__ void estimate_pivots(const Ctx &x, Smem &sm, uint32_t lo, unsigned long long hi, int a,
                                int b, int s, float g, float mass_hi, float tau, uint32_t piv[4]) {
  // chunk maxima strictly inside (lo, hi): positions [ca, cb) of csort
  unsigned long long ge_hi = 0, gt_lo = 0;
  for (int i = threadIdx.x; i < x.nl; i += kT) {
    if (sm.csort[i] == ~0ull) continue;
    const uint32_t kk = ckey(sm, i);
    ge_hi += (unsigned long long)kk >= hi;
    gt_lo += kk > lo;
  }
  const int ca = (int)block_sum_u(ge_hi, sm), cb = (int)block_sum_u(gt_lo, sm);
  // prefix masses: samples into lcum[a, b), chunk maxima into cabove[ca, cb)
  {
    const int per = (b - a + kT - 1) / kT;
    const int ta = min(b, a + (int)threadIdx.x * per), tb = min(b, ta + per);
    float part = 0.f;
    for (int i = ta; i < tb; ++i) part += (float)s * mass_of(x, value_of(~sm.samp[i]));
    float tot;
    float run = block_excl_scan_f(part, sm, &tot);
    for (int i = ta; i < tb; ++i) {
      run += (float)s * mass_of(x, value_of(~sm.samp[i]));
      sm.lcum[i] = run;
    }
  }
  {
    const int per = (cb - ca + kT - 1) / kT;
    const int ta = min(cb, ca + (int)threadIdx.x * per), tb = min(cb, ta + per);
    float part = 0.f;
    for (int i = ta; i < tb; ++i) part += mass_of(x, value_of(ckey(sm, i)));
    float tot;
    float run = block_excl_scan_f(part, sm, &tot);
    for (int i = ta; i < tb; ++i) {
      run += mass_of(x, value_of(ckey(sm, i)));
      sm.cabove[i] = run;
    }
  }
  __syncthreads();
  const float frac[4] = {-0.25f, -1.f / 12.f, 1.f / 12.f, 0.25f};
  const int ps = (b - a + kT - 1) / kT, pc = (cb - ca + kT - 1) / kT;
  const int sa = min(b, a + (int)threadIdx.x * ps), sb = min(b, sa + ps);
  const int qa = min(cb, ca + (int)threadIdx.x * pc), qb = min(cb, qa + pc);
  for (int t = 0; t < 4; ++t) {
    const float want = tau + frac[t] * g;
    int fs = b, fc = cb;
    for (int i = sa; i < sb; ++i) {
      const int r = last_at_least_c(sm, ca, cb, ~sm.samp[i]);
      const float e = mass_hi + sm.lcum[i] + (r >= ca ? sm.cabove[r] : 0.f);
      if (e >= want) {
        fs = i;
        break;
      }
    }
    for (int i = qa; i < qb; ++i) {
      const int r = last_at_least(sm.samp, a, b, ckey(sm, i));
      const float e = mass_hi + sm.cabove[i] + (r >= a ? sm.lcum[r] : 0.f);
      if (e >= want) {
        fc = i;
        break;
      }
    }
    fs = block_min_i(fs, sm);
    fc = block_min_i(fc, sm);
    uint32_t kp = lo + 1;                       // nothing reaches it: the bottom
    if (fs < b) kp = ~sm.samp[fs];
    if (fc < cb && ckey(sm, fc) > kp) kp = ckey(sm, fc);
    piv[t] = kp;
  }
}

// A window [lo, hi) of keys around the top-p boundary of the whole row.  The
// mass at or above X is the row's mass minus the mass below X, and the mass
// below is the light part of each chunk: the chunks whose maximum is below X
// count with their exact mass, and in the others the sample points below X
// count with the logits they stand for.  The window spans `d` sample points on
// either side of the first point where that estimate reaches tau.  The window
// stays inside [rlo, rhi), where the boundary is known to lie: mass(>= rlo)
// >= tau (or rlo = 0) and mass(>= rhi) < tau.  With a reference key kref whose
// exact mass mref a gather has measured, the estimate is shifted by its error
// there.  Needs the sample sorted and csort; uses lcum and the list as scratch.
__device__ void estimate_window(const Ctx &x, Smem &sm, float tau, int d, uint32_t rlo,
                                unsigned long long rhi, bool has_ref, uint32_t kref, float mref,
                                uint32_t &lo, unsigned long long &hi) {
  const float w = (float)(kChunk / x.spc);
  float *cs = reinterpret_cast<float *>(sm.list);          // chunk-mass prefix, csort order
  float *css = cs + kSortChunks;                            // sample-mass prefix, csort order
  const int nc = x.nl;
  // prefixes over csort (descending maxima) and over the sorted sample
  {
    const int per = (nc + kT - 1) / kT;
    const int a = min(nc, (int)threadIdx.x * per), b = min(nc, a + per);
    float p1 = 0.f, p2 = 0.f;
    for (int i = a; i < b; ++i)
      if (sm.csort[i] != ~0ull) {
        const int c = (int)(uint32_t)sm.csort[i];
        p1 += sm.cmass[c];
        p2 += sm.csamp[c];
      }
    float t1, t2;
    float r1 = block_excl_scan_f(p1, sm, &t1);
    float r2 = block_excl_scan_f(p2, sm, &t2);
    for (int i = a; i < b; ++i) {
      if (sm.csort[i] != ~0ull) {
        const int c = (int)(uint32_t)sm.csort[i];
        r1 += sm.cmass[c];
        r2 += sm.csamp[c];
      }
      cs[i] = r1;
      css[i] = r2;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      sm.fval[1] = t1;
      sm.fval[2] = t2;
    }
  }
  {
    const int per = (x.ns + kT - 1) / kT;
    const int a = min(x.ns, (int)threadIdx.x * per), b = min(x.ns, a + per);
    float part = 0.f;
    for (int i = a; i < b; ++i) part += mass_of(x, value_of(~sm.samp[i]));
    float tot;
    float run = block_excl_scan_f(part, sm, &tot);
    for (int i = a; i < b; ++i) {
      run += mass_of(x, value_of(~sm.samp[i]));
      sm.lcum[i] = run;
    }
    if (threadIdx.x == 0) sm.fval[3] = tot;
  }
  __syncthreads();
  const float cs_tot = sm.fval[1], css_tot = sm.fval[2], samp_tot = sm.fval[3];
  // estimated mass at or above K, given the mass of the sample points at or above K
  auto estimate = [&](uint32_t K, float samp_ge) {
    const int r = last_at_least_c(sm, 0, nc, K);            // chunks with maximum >= K
    const float cs_lt = cs_tot - (r >= 0 ? cs[r] : 0.f);
    const float css_lt = css_tot - (r >= 0 ? css[r] : 0.f);
    return x.S - cs_lt - w * fmaxf(0.f, samp_tot - samp_ge - css_lt);
  };
  float bias = 0.f;
  if (has_ref) {
    int q0 = 0, q1 = x.ns;                                  // sample points with key >= kref
    while (q0 < q1) {
      const int mid = (q0 + q1) >> 1;
      if (~sm.samp[mid] >= kref) q0 = mid + 1;
      else q1 = mid;
    }
    bias = mref - estimate(kref, q0 > 0 ? sm.lcum[q0 - 1] : 0.f);
  }
  // first sample point (descending) whose estimate reaches tau; points at or
  // below rlo reach it, points at or above rhi do not
  int first = x.ns;
  const int per = (x.ns + kT - 1) / kT;
  const int a = min(x.ns, (int)threadIdx.x * per), b = min(x.ns, a + per);
  for (int i = a; i < b; ++i) {
    const uint32_t K = ~sm.samp[i];
    if ((unsigned long long)K >= rhi) continue;
    if ((rlo > 0 && K <= rlo) || estimate(K, sm.lcum[i]) + bias >= tau) {
      first = i;
      break;
    }
  }
  first = block_min_i(first, sm);
  lo = first + d < x.ns ? ~sm.samp[first + d] : 0u;
  hi = first - d >= 0 ? (unsigned long long)(~sm.samp[first - d]) : kKeyEnd;
  if (lo < rlo) lo = rlo;
  if (hi > rhi) hi = rhi;
  if (hi <= lo) {
    hi = rhi;
    if (hi <= lo) lo = rlo;
  }
}

// Sort the sample once (descending keys, invalid points last); x.ns = valid points.
__device__ void sort_sample(Ctx &x, Smem &sm) {
  if (x.ns >= 0) return;
  const int nsamp = x.r.nch * x.spc;
  const int np = pow2_at_least(nsamp);
  for (int i = nsamp + threadIdx.x; i < np; i += kT) sm.samp[i] = ~0u;
  __syncthreads();
  bitonic_sort(sm.samp, np);
  unsigned long long valid = 0;
  for (int i = threadIdx.x; i < nsamp; i += kT) valid += sm.samp[i] != ~0u;
  x.ns = (int)block_sum_u(valid, sm);
}

// Sample points strictly inside (lo, hi): positions [a, b) of the sorted sample.
__device__ void sample_span(const Ctx &x, Smem &sm, uint32_t lo, unsigned long long hi, int &a,
                            int &b) {
  unsigned long long ge_hi = 0, gt_lo = 0;
  for (int i = threadIdx.x; i < x.ns; i += kT) {
    const uint32_t kk = ~sm.samp[i];
    ge_hi += (unsigned long long)kk >= hi;
    gt_lo += kk > lo;
  }
  a = (int)block_sum_u(ge_hi, sm);
  b = (int)block_sum_u(gt_lo, sm);
}

// Pivots strictly inside (lo, hi), non-increasing.
__device__ __forceinline__ void clamp_pivots(uint32_t piv[4], uint32_t lo, unsigned long long hi) {
  for (int t = 0; t < 4; ++t) {
    if ((unsigned long long)piv[t] >= hi) piv[t] = (uint32_t)(hi - 1);
    if (piv[t] <= lo) piv[t] = lo + 1;
    if (t && piv[t] > piv[t - 1]) piv[t] = piv[t - 1];
  }
}

// Tighten [lo, hi) (with the counts and masses at lo and at hi) until it holds
// at most kCap logits or a single key.  Target: the k-th logit (count(>= X)
// >= k) or the top-p boundary (mass(>= X) >= tau).  Pivots are sample points
// around the sample's estimate of the target while the sample has enough
// points inside, else the key range split in five.  False if the probes ran out.
template <bool kBf16>
__device__ bool narrow(Ctx &x, Smem &sm, bool want_mass, unsigned long long k, float tau,
                       uint32_t &lo, unsigned long long &hi, unsigned long long &cnt_lo,
                       float &mass_lo, unsigned long long &cnt_hi, float &mass_hi) {
  const int s = kChunk / x.spc;                // logits per sample point
  sort_sample(x, sm);
  float spread = 0.16f * x.S;                   // top-p pivot spread; widens after a miss
  for (int it = 0; it < kMaxProbes; ++it) {
    if (cnt_lo - cnt_hi <= (unsigned long long)kCap || hi - lo <= 1) return true;
    int a, b;
    sample_span(x, sm, lo, hi, a, b);
    uint32_t piv[4];
    if (want_mass && it < kMaxProbes / 2) {
      estimate_pivots(x, sm, lo, hi, a, b, s, fminf(spread, mass_lo - mass_hi), mass_hi, tau, piv);
    } else if (b - a >= 8 && it < kMaxProbes / 2) {
      // the k-th logit: the sample point at the estimated rank, and around it
      long long need = ((long long)k - (long long)cnt_hi) / s;
      if (need < 0) need = 0;
      if (need > b - a - 1) need = b - a - 1;
      const int centre = a + (int)need;
      const int span = max(2, (int)(3.f * sqrtf((float)(centre - a + 1))) + 2);
      const int q[4] = {centre - span, centre - span / 3, centre + span / 3, centre + span};
      for (int t = 0; t < 4; ++t) piv[t] = ~sm.samp[min(b - 1, max(a, q[t]))];
    } else {
      const unsigned long long w = hi - lo;
      for (int t = 0; t < 4; ++t) piv[t] = (uint32_t)(lo + (w * (unsigned long long)(4 - t)) / 5);
    }
    clamp_pivots(piv, lo, hi);
    unsigned long long pc[4];
    float pm[4];
    probe<kBf16>(x, sm, piv, want_mass, pc, pm);
    // the largest pivot that still holds the target becomes lo, the one above it hi
    int sel = -1;
    for (int t = 0; t < 4 && sel < 0; ++t)
      if (want_mass ? pm[t] >= tau : pc[t] >= k) sel = t;
    spread = (sel == 0 || sel < 0) ? spread * 4.f : spread * 0.5f;   // a miss widens
    if (sel >= 0) {
      if (sel > 0) {
        hi = piv[sel - 1];
        cnt_hi = pc[sel - 1];
        mass_hi = pm[sel - 1];
      }
      lo = piv[sel];
      cnt_lo = pc[sel];
      mass_lo = pm[sel];
    } else {
      hi = piv[3];
      cnt_hi = pc[3];
      mass_hi = pm[3];
    }
  }
  return cnt_lo - cnt_hi <= (unsigned long long)kCap || hi - lo <= 1;
}

// Ties: the window is the single key v, holding more logits than kCap.  Writes
// per chunk the mass above v (cabove) and the count of v (cmass, as a float),
// and returns the index of the t-th (0-based) logit equal to v in index order.
template <bool kBf16>
__device__ int tie_index(const Ctx &x, Smem &sm, uint32_t v, unsigned long long t) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for_chunks<kBf16>(
      x.r, [&](int) { return true; }, [&](int) {},
      [&](const float vv[kLE], int n, int, int c) {
        float ma = 0.f;
        int ties = 0;
#pragma unroll
        for (int j = 0; j < kLE; ++j) {
          const uint32_t k = key_of(vv[j]);
          if (j < n && k > v) ma += mass_of(x, vv[j]);
          ties += j < n && k == v;
        }
        ma = warp_sum_f(ma);
        ties = __reduce_add_sync(0xffffffffu, ties);
        if (lane == 0) {
          sm.cabove[c] = ma;
          sm.cmass[c] = (float)ties;
        }
      });
  __syncthreads();
  const int per = (x.nl + kT - 1) / kT;
  const int a = min(x.nl, (int)threadIdx.x * per), b = min(x.nl, a + per);
  float s = 0.f;
  for (int c = a; c < b; ++c) s += sm.cmass[c];
  float tot;
  float run = block_excl_scan_f(s, sm, &tot);
  if (threadIdx.x == 0) {
    sm.ival[1] = -1;
    sm.ival[3] = -1;
  }
  __syncthreads();
  for (int c = a; c < b; ++c) {
    if (run <= (float)t && (float)t < run + sm.cmass[c]) {
      sm.ival[1] = c;
      sm.ival[2] = (int)((float)t - run);
    }
    run += sm.cmass[c];
  }
  __syncthreads();
  const int c = sm.ival[1], want = sm.ival[2];
  if (c >= 0 && warp == 0) {
    float vv[kLE];
    int i0;
    const int n = chunk_lane<kBf16>(x.r, c, lane, vv, i0);
    int mine = 0;
#pragma unroll
    for (int j = 0; j < kLE; ++j) mine += j < n && key_of(vv[j]) == v;
    int incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const int excl = incl - mine;
    if (excl <= want && want < incl) {
      int r = excl;
      for (int j = 0; j < n; ++j)
        if (key_of(vv[j]) == v) {
          if (r == want) sm.ival[3] = i0 + j;
          ++r;
        }
    }
  }
  __syncthreads();
  return sm.ival[3];
}

// The draw over the per-chunk kept masses in cabove: the chunk whose
// cumulative mass first exceeds u times the total, then the token inside it.
// Kept: key > vk, or key == vk and index <= ik.
template <bool kBf16>
__device__ int draw_chunks(const Ctx &x, Smem &sm, float u, uint32_t vk, int ik) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int per = (x.nl + kT - 1) / kT;
  const int a = min(x.nl, (int)threadIdx.x * per), b = min(x.nl, a + per);
  float s = 0.f;
  for (int c = a; c < b; ++c) s += sm.cabove[c];
  float tot;
  float run = block_excl_scan_f(s, sm, &tot);
  const float U = u * tot;
  if (threadIdx.x == 0) {
    sm.ival[4] = -1;
    sm.ival[5] = -1;
  }
  __syncthreads();
  for (int c = a; c < b; ++c) {
    const float K = sm.cabove[c];
    if (K > 0.f) {
      if (run <= U && U < run + K) {
        sm.ival[4] = c;
        sm.fval[0] = U - run;
      }
      atomicMax(&sm.ival[5], c);               // the last chunk with mass (rounding fallback)
    }
    run += K;
  }
  __syncthreads();
  int c = sm.ival[4];
  float target = sm.fval[0];
  if (c < 0) {                                  // u * total rounded past the last mass
    c = sm.ival[5];
    target = INFINITY;
  }
  if (warp == 0 && c >= 0) {
    float v[kLE];
    int i0;
    const int n = chunk_lane<kBf16>(x.r, c, lane, v, i0);
    float m[kLE], mine = 0.f;
    int last = -1;
#pragma unroll
    for (int j = 0; j < kLE; ++j) {
      const uint32_t k = key_of(v[j]);
      const bool kept = j < n && (k > vk || (k == vk && i0 + j <= ik));
      m[j] = kept ? mass_of(x, v[j]) : 0.f;
      if (m[j] > 0.f) last = i0 + j;
      mine += m[j];
    }
    float incl = mine;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    const unsigned hit = __ballot_sync(0xffffffffu, incl > target && mine > 0.f);
    int tok = -1;
    if (hit) {
      const int hl = __ffs(hit) - 1;
      if (lane == hl) {
        float acc = incl - mine;
        for (int j = 0; j < kLE; ++j)
          if (m[j] > 0.f) {
            acc += m[j];
            if (acc > target) {
              tok = i0 + j;
              break;
            }
          }
        if (tok < 0) tok = last;
      }
      tok = __shfl_sync(0xffffffffu, tok, hl);
    } else {
      // rounding left the target past the chunk: its last kept token
      const unsigned has = __ballot_sync(0xffffffffu, last >= 0);
      if (has) tok = __shfl_sync(0xffffffffu, last, 31 - __clz(has));
    }
    if (lane == 0) sm.ival[6] = tok;
  }
  __syncthreads();
  return c >= 0 ? sm.ival[6] : -1;
}

// Rewrite the first n window entries as (index << 32) | mass bits, sorted by index.
__device__ void window_by_index(const Ctx &x, Smem &sm, int n) {
  for (int i = threadIdx.x; i < n; i += kT) {
    const unsigned long long e = sm.list[i];
    const float l = value_of(~(uint32_t)(e >> 32));
    sm.list[i] = ((unsigned long long)(uint32_t)e << 32) | __float_as_uint(mass_of(x, l));
  }
  const int np = pow2_at_least(n);
  for (int i = n + threadIdx.x; i < np; i += kT) sm.list[i] = ~0ull;
  __syncthreads();
  bitonic_sort(sm.list, np);
}

// The draw when the whole kept set is the first n window entries.
__device__ int draw_list(const Ctx &x, Smem &sm, int n, float u) {
  window_by_index(x, sm, n);
  const int per = (n + kT - 1) / kT;
  const int a = min(n, (int)threadIdx.x * per), b = min(n, a + per);
  float s = 0.f;
  for (int i = a; i < b; ++i) s += __uint_as_float((uint32_t)sm.list[i]);
  float tot;
  float run = block_excl_scan_f(s, sm, &tot);
  const float U = u * tot;
  if (threadIdx.x == 0) sm.ival[7] = -1;
  __syncthreads();
  int last = -1;
  for (int i = a; i < b; ++i) {
    const float m = __uint_as_float((uint32_t)sm.list[i]);
    if (m > 0.f) {
      if (run <= U && U < run + m) sm.ival[7] = (int)(sm.list[i] >> 32);
      last = (int)(sm.list[i] >> 32);
    }
    run += m;
  }
  __syncthreads();
  const int tok = sm.ival[7];
  if (tok >= 0) return tok;
  return (int)block_max_u((unsigned long long)(last + 1), sm) - 1;   // rounding: the last one
}

// Per-chunk summaries written by the scan kernel for the row kernel.
struct WsRef {
  float *cmax, *cmass;                         // [row][nl_cap]
  uint32_t *samp;                              // [row][ns_cap]
  uint32_t *bad;                               // [row][nparts]: a non-finite logit seen
  int nl_cap, ns_cap, nparts;
};

constexpr int kScanThreads = 256;
constexpr int kScanWarps = kScanThreads / 32;
constexpr int kChunksPerCta = 64;              // vector chunks of a scan CTA (16384 logits)
constexpr int kScanPerWarp = kChunksPerCta / kScanWarps;

// ---- the scan (HBM, once): per chunk its maximum and its mass relative to
// it, the sample, and the part's finiteness.  Grid (parts, rows).
template <bool kBf16>
__global__ void __launch_bounds__(kScanThreads) sample_scan_kernel(SampleParams p, WsRef ws) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int part = blockIdx.x, row = blockIdx.y;
  const RowRef r = row_ref<kBf16>(p.logits + (int64_t)row * p.row_bytes, p.vocab);
  const int spc = r.nch <= kMaxSamples / 4 ? 4 : 2;
  const float kx = 1.4426950408889634f / fmaxf(p.temperature[row], kMinT);
  float *cmax = ws.cmax + (int64_t)row * ws.nl_cap, *cmass = ws.cmass + (int64_t)row * ws.nl_cap;
  uint32_t *samp = ws.samp + (int64_t)row * ws.ns_cap;
  bool finite = true;
  auto chunk = [&](const float v[kLE], int n, int c_logical, int i0, int sample_slot) {
    float m = -INFINITY;
#pragma unroll
    for (int j = 0; j < kLE; ++j)
      if (j < n) m = fmaxf(m, v[j]);
    m = warp_max_f(m);
    // sum of 2^((v - m) kx), even and odd positions apart, in pairs
    float2 s2 = make_float2(0.f, 0.f);
    const float2 nm2 = make_float2(-m, -m), kx2 = make_float2(kx, kx);
#pragma unroll
    for (int j = 0; j < kLE; j += 2) {
      const float2 y = fmul2(fadd2(make_float2(v[j], v[j + 1]), nm2), kx2);
      s2 = fadd2(s2, make_float2(j < n ? ex2(y.x) : 0.f, j + 1 < n ? ex2(y.y) : 0.f));
    }
    float s = warp_sum_f(s2.x + s2.y);
    // a NaN turns the mass into NaN, +inf the maximum; -inf is a zero-mass logit
    if (m == -INFINITY) s = 0.f;
    finite &= m != INFINITY && s == s;
    if (lane == 0) {
      cmax[c_logical] = m;
      cmass[c_logical] = s;
    }
    if (sample_slot >= 0) samp[sample_slot] = (n && v[0] != m) ? ~key_of(v[0]) : ~0u;
  };
  const int cbeg = part * kChunksPerCta + warp;
  uint4 raw[kScanPerWarp][kBf16 ? 1 : 2];
  int n[kScanPerWarp];
#pragma unroll
  for (int q = 0; q < kScanPerWarp; ++q) {     // every load of the warp in flight at once
    const int c = cbeg + q * kScanWarps, vi = 32 * c + lane;
    n[q] = (c < r.nch && vi < r.nvec) ? kLE : 0;
    if (n[q]) {
      const uint8_t *src = r.p + (int64_t)(r.h + kLE * vi) * (kBf16 ? 2 : 4);
      asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                   : "=r"(raw[q][0].x), "=r"(raw[q][0].y), "=r"(raw[q][0].z), "=r"(raw[q][0].w)
                   : "l"(src));
      if (!kBf16)
        asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(raw[q][kBf16 ? 0 : 1].x), "=r"(raw[q][kBf16 ? 0 : 1].y),
                       "=r"(raw[q][kBf16 ? 0 : 1].z), "=r"(raw[q][kBf16 ? 0 : 1].w)
                     : "l"(src + 16));
    }
  }
  auto unpack = [&](int q, float v[kLE]) {
    if (kBf16) {
      const uint4 w = raw[q][0];
      v[0] = bf16lo(w.x); v[1] = bf16hi(w.x); v[2] = bf16lo(w.y); v[3] = bf16hi(w.y);
      v[4] = bf16lo(w.z); v[5] = bf16hi(w.z); v[6] = bf16lo(w.w); v[7] = bf16hi(w.w);
    } else {
      const uint4 a = raw[q][0], b = raw[q][kBf16 ? 0 : 1];
      v[0] = __uint_as_float(a.x); v[1] = __uint_as_float(a.y);
      v[2] = __uint_as_float(a.z); v[3] = __uint_as_float(a.w);
      v[4] = __uint_as_float(b.x); v[5] = __uint_as_float(b.y);
      v[6] = __uint_as_float(b.z); v[7] = __uint_as_float(b.w);
    }
  };
  const int every = 32 / spc;
  // the warp's chunks side by side: maxima, then masses relative to them,
  // each reduced over the warp for all chunks at once
  float m[kScanPerWarp], sm2[kScanPerWarp];
#pragma unroll
  for (int q = 0; q < kScanPerWarp; ++q) {
    float v[kLE];
    unpack(q, v);
    m[q] = -INFINITY;
#pragma unroll
    for (int j = 0; j < kLE; ++j)
      if (j < n[q]) m[q] = fmaxf(m[q], v[j]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
#pragma unroll
    for (int q = 0; q < kScanPerWarp; ++q) m[q] = fmaxf(m[q], __shfl_xor_sync(0xffffffffu, m[q], o));
#pragma unroll
  for (int q = 0; q < kScanPerWarp; ++q) {
    float v[kLE];
    unpack(q, v);
    float2 s2 = make_float2(0.f, 0.f);
    const float2 nm2 = make_float2(-m[q], -m[q]), kx2 = make_float2(kx, kx);
#pragma unroll
    for (int j = 0; j < kLE; j += 2) {
      const float2 y = fmul2(fadd2(make_float2(v[j], v[j + 1]), nm2), kx2);
      s2 = fadd2(s2, make_float2(j < n[q] ? ex2(y.x) : 0.f, j + 1 < n[q] ? ex2(y.y) : 0.f));
    }
    sm2[q] = s2.x + s2.y;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
#pragma unroll
    for (int q = 0; q < kScanPerWarp; ++q) sm2[q] += __shfl_xor_sync(0xffffffffu, sm2[q], o);
#pragma unroll
  for (int q = 0; q < kScanPerWarp; ++q) {
    const int c = cbeg + q * kScanWarps;
    if (c >= r.nch) break;                    // warp-uniform
    // a NaN turns the mass into NaN, +inf the maximum; -inf is a zero-mass logit
    const float s = m[q] == -INFINITY ? 0.f : sm2[q];
    finite &= m[q] != INFINITY && s == s;
    if (lane == 0) {
      cmax[c + 1] = m[q];
      cmass[c + 1] = s;
    }
    if ((lane & (every - 1)) == 0) {
      float v0[kLE];
      unpack(q, v0);
      samp[c * spc + lane / every] = (n[q] && v0[0] != m[q]) ? ~key_of(v0[0]) : ~0u;
    }
  }
  if (part == 0 && warp == 0) {                 // head and tail chunks
    for (int c = 0; c < r.nch + 2; c += r.nch + 1) {
      float v[kLE];
      int i0;
      const int nn = chunk_lane<kBf16>(r, c, lane, v, i0);
      chunk(v, nn, c, i0, -1);
    }
  }
  const bool bad = __syncthreads_or(!finite);
  if (threadIdx.x == 0) ws.bad[(int64_t)row * ws.nparts + part] = bad ? 1u : 0u;
  grid_dep_launch();
}

// ---- which row a CTA takes
// Cost class of row i from its parameters alone: 0 = a top-p cut with no
// top-k below the window capacity (its boundary is searched over a whole
// distribution: the long rows), 1 = another cut, 2 = none.
__device__ __forceinline__ int row_class(const SampleParams &p, int i) {
  unsigned long long k = (unsigned long long)p.vocab;
  if (p.top_k != nullptr && p.top_k[i] >= 1 && p.top_k[i] < p.vocab) k = (unsigned long long)p.top_k[i];
  const bool topp = p.top_p != nullptr && p.top_p[i] < 1.f;   // NaN: no cut (reported later)
  if (topp && k > (unsigned long long)kCap) return 0;
  return (topp || k < (unsigned long long)p.vocab) ? 1 : 2;
}

// The row of this CTA: rows in order of cost class (the long rows first,
// index order within a class).  The first wave of CTAs is spread one per SM,
// so each long row gets an SM of its own instead of sharing its issue slots
// with another long row for its whole run.  Batches above 2 kT rows keep
// CTA b on row b.  Reads only the parameters (every thread calls).
__device__ int row_of_block(const SampleParams &p, Smem &sm) {
  const int b = (int)blockIdx.x, B = p.batch, t = threadIdx.x;
  const int lane = t & 31, warp = t >> 5;
  if (B > 2 * kT) return b;
  const int c0 = t < B ? row_class(p, t) : 3, c1 = t + kT < B ? row_class(p, t + kT) : 3;
  if (t < 4) sm.ival[t] = 0;
  __syncthreads();
  if (c0 < 3) atomicAdd(&sm.ival[c0], 1);
  if (c1 < 3) atomicAdd(&sm.ival[c1], 1);
  __syncthreads();
  int cls = 0, off = 0;
  while (cls < 2 && b >= off + sm.ival[cls]) off += sm.ival[cls++];
  const int rank = b - off;                     // this CTA takes the rank-th row of class cls
  const unsigned m0 = __ballot_sync(0xffffffffu, c0 == cls);
  const unsigned m1 = __ballot_sync(0xffffffffu, c1 == cls);
  if (lane == 0) sm.ured[warp] = (unsigned long long)__popc(m0) | ((unsigned long long)__popc(m1) << 32);
  __syncthreads();
  int pre0 = 0, pre1 = 0, tot0 = 0;
  for (int w = 0; w < kW; ++w) {
    const int n0 = (int)(sm.ured[w] & 0xffffffffu), n1 = (int)(sm.ured[w] >> 32);
    tot0 += n0;
    if (w < warp) {
      pre0 += n0;
      pre1 += n1;
    }
  }
  const unsigned lt = (1u << lane) - 1u;
  pre0 += __popc(m0 & lt);
  pre1 += tot0 + __popc(m1 & lt);
  if (c0 == cls && pre0 == rank) sm.ival[4] = t;
  if (c1 == cls && pre1 == rank) sm.ival[4] = t + kT;
  __syncthreads();
  const int row = sm.ival[4];
  __syncthreads();                              // ival and ured are reused by the row's work
  return row;
}

// ---- the row (one CTA each): everything after the scan
template <bool kBf16>
__global__ void __launch_bounds__(kT, 2) sample_row_kernel(SampleParams p, WsRef ws) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  Smem &sm = *reinterpret_cast<Smem *>(smem_raw);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int row = row_of_block(p, sm);
  Ctx x;
  x.r = row_ref<kBf16>(p.logits + (int64_t)row * p.row_bytes, p.vocab);
  x.nl = x.r.nch + 2;
  x.spc = x.r.nch <= kMaxSamples / 4 ? 4 : 2;
  x.ns = -1;                                    // the sample is sorted on first use
  x.M = 0.f;

  // ---- row parameters (Sampler.prepare's clamps)
  const float T = p.temperature[row], u = p.uniform[row];
  float P = 1.f;
  unsigned long long k = (unsigned long long)p.vocab;
  bool params_ok = true;
  if (p.top_k != nullptr && p.top_k[row] >= 1 && p.top_k[row] < p.vocab) k = p.top_k[row];
  if (p.top_p != nullptr) {
    P = fminf(fmaxf(p.top_p[row], kMinP), 1.f);
    params_ok = !isnan(p.top_p[row]);
  }
  params_ok = params_ok && isfinite(T) && u >= 0.f && u < 1.f;
  x.kx = 1.4426950408889634f / fmaxf(T, kMinT);
  grid_dep_wait();                              // the scan's summaries
  bool bad = false;
  for (int i = threadIdx.x; i < ws.nparts; i += kT) bad |= ws.bad[(int64_t)row * ws.nparts + i] != 0;
  bad = __syncthreads_or(bad);
  if (bad || !params_ok) {
    if (threadIdx.x == 0) {
      report(p.status, bad ? MSG_DEV_BAD_LOGIT : MSG_DEV_BAD_SAMPLING, row, 0);
      p.tokens[row] = -1;
    }
    return;
  }
  {
    const float *cmax = ws.cmax + (int64_t)row * ws.nl_cap, *cmass = ws.cmass + (int64_t)row * ws.nl_cap;
    float m = -INFINITY;
    for (int c = threadIdx.x; c < x.nl; c += kT) {
      sm.cmax[c] = cmax[c];
      sm.cmass[c] = cmass[c];
      m = fmaxf(m, sm.cmax[c]);
    }
    x.M = block_max_f(m, sm);
  }
  if (x.M == -INFINITY) {                       // every logit -inf: no distribution
    if (threadIdx.x == 0) {
      report(p.status, MSG_DEV_BAD_LOGIT, row, 1);
      p.tokens[row] = -1;
    }
    return;
  }
  float S;                                      // chunk masses relative to the row maximum
  {
    float part = 0.f;
    for (int c = threadIdx.x; c < x.nl; c += kT) {
      const float cm = sm.cmass[c] > 0.f ? sm.cmass[c] * ex2((sm.cmax[c] - x.M) * x.kx) : 0.f;
      sm.cmass[c] = cm;
      part += cm;
    }
    S = block_sum_f(part, sm);
    x.S = S;
  }
  const bool topk_on = k < (unsigned long long)p.vocab;
  const bool topp_on = P < 1.f;
  int tok = -1;
  if (!topk_on && !topp_on) {
    // ---- no cut: the chunk masses are the kept masses
    for (int c = threadIdx.x; c < x.nl; c += kT) sm.cabove[c] = sm.cmass[c];
    __syncthreads();
    tok = draw_chunks<kBf16>(x, sm, u, 0u, p.vocab);
  } else {
    {                                           // the sample (sorted on first use), and
      const uint32_t *samp = ws.samp + (int64_t)row * ws.ns_cap;   // its mass per chunk
      const int ns4 = (x.r.nch * x.spc) >> 2;                       // spc is 4 or 2: whole uint4s
      for (int i = threadIdx.x; i < ns4; i += kT)
        reinterpret_cast<uint4 *>(sm.samp)[i] = reinterpret_cast<const uint4 *>(samp)[i];
      for (int i = 4 * ns4 + threadIdx.x; i < x.r.nch * x.spc; i += kT) sm.samp[i] = samp[i];
      __syncthreads();
      for (int c = threadIdx.x; c < x.nl; c += kT) {
        float m = 0.f;
        if (c >= 1 && c <= x.r.nch)
          for (int i = 0; i < x.spc; ++i) {
            const uint32_t e = sm.samp[(c - 1) * x.spc + i];
            if (e != ~0u) m += mass_of(x, value_of(~e));
          }
        sm.csamp[c] = m;
      }
    }
    // chunk maxima sorted by descending key (invalid chunks last)
    const int npc = pow2_at_least(x.nl);
    for (int i = threadIdx.x; i < npc; i += kT)
      sm.csort[i] = (i < x.nl && sm.cmax[i] != -INFINITY)
                        ? ((unsigned long long)(~key_of(sm.cmax[i])) << 32) | (uint32_t)i
                        : ~0ull;
    __syncthreads();
    bitonic_sort(sm.csort, npc);
    bool ok = true, tie_mode = false;
    uint32_t vk = 0;                            // the threshold token: its key and index
    int ik = -1;
    int n_win = 0;                              // kept entries at the head of the list
    unsigned long long cnt_above = 0;           // logits above the window
    float mass_above = 0.f;
    uint32_t region_lo = 0;                     // where stage 2 may search
    float S_k = S;
    // ---- stage 1: the k-th token
    if (topk_on) {
      bool gathered = false;
      if (k <= (unsigned long long)x.nl) {
        // the k-th largest chunk maximum bounds the k-th logit from below
        if (sm.csort[k - 1] != ~0ull) {
          n_win = gather<kBf16>(x, sm, ckey(sm, (int)k - 1), kKeyEnd, &cnt_above, &mass_above);
          gathered = n_win <= kCap;
        }
      }
      if (!gathered) {
        uint32_t lo = 0;
        unsigned long long hi = kKeyEnd, cnt_lo = (unsigned long long)p.vocab, cnt_hi = 0;
        float mass_lo = S, mass_hi = 0.f;
        ok = narrow<kBf16>(x, sm, false, k, 0.f, lo, hi, cnt_lo, mass_lo, cnt_hi, mass_hi);
        if (ok && cnt_lo - cnt_hi <= (unsigned long long)kCap) {
          n_win = gather<kBf16>(x, sm, lo, hi, &cnt_above, &mass_above);
          ok = n_win <= kCap && cnt_above < k && k <= cnt_above + (unsigned long long)n_win;
          region_lo = hi >= kKeyEnd ? 0xffffffffu : (uint32_t)hi;
        } else if (ok) {
          tie_mode = true;                      // one key with more logits than kCap
          vk = lo;
          cnt_above = cnt_hi;
          region_lo = vk + 1;
        }
      }
      if (ok && !tie_mode) {
        sort_window(x, sm, n_win);
        const int pk = (int)(k - cnt_above - 1);
        vk = ~(uint32_t)(sm.list[pk] >> 32);
        ik = (int)(uint32_t)sm.list[pk];
        S_k = mass_above + sm.lcum[pk];
        n_win = pk + 1;
      } else if (ok) {
        const unsigned long long t = k - cnt_above - 1;
        ik = tie_index<kBf16>(x, sm, vk, t);
        float part = 0.f;
        for (int c = threadIdx.x; c < x.nl; c += kT) part += sm.cabove[c];
        mass_above = block_sum_f(part, sm);
        S_k = mass_above + (float)(t + 1) * mass_of(x, value_of(vk));
        ok = ik >= 0;
      }
    }
    // ---- stage 2: the top-p boundary inside the top-k set
    if (ok && topp_on) {
      const float tau = P * S_k;
      if (topk_on && mass_above < tau) {
        if (!tie_mode) {                        // inside the sorted window
          const int pp = window_crossing(sm, n_win, mass_above, tau);
          const int pos = min(pp, n_win - 1);
          vk = ~(uint32_t)(sm.list[pos] >> 32);
          ik = (int)(uint32_t)sm.list[pos];
          n_win = pos + 1;
        } else {                                // inside the tie group
          const float w = mass_of(x, value_of(vk));
          unsigned long long t = w > 0.f ? (unsigned long long)ceilf((tau - mass_above) / w) : 1;
          t = max(1ull, min(t, k - cnt_above));
          ik = tie_index<kBf16>(x, sm, vk, t - 1);
          ok = ik >= 0;
        }
      } else {
        // the boundary lies above the top-k window (or there is no top-k)
        uint32_t lo = topk_on ? region_lo : 0;
        unsigned long long hi = kKeyEnd;
        unsigned long long cnt_lo = topk_on ? cnt_above : (unsigned long long)p.vocab, cnt_hi = 0;
        float mass_lo = topk_on ? mass_above : S, mass_hi = 0.f;
        tie_mode = false;
        // the largest chunk maxima are logits of their own: the first r of them
        // whose masses reach tau put the boundary at or above the r-th
        const uint32_t cm = chunk_max_bound(x, sm, lo, tau);
        bool gathered = false, sorted = false;
        if (cm != 0u) {
          n_win = gather<kBf16>(x, sm, cm, kKeyEnd, &cnt_above, &mass_above);
          gathered = n_win <= kCap;
        }
        if (!gathered) {
          // a gather around the estimate; a miss still tells which side, and
          // the exact mass it measured at that edge corrects the estimate for
          // a second gather on that side
          sort_sample(x, sm);
          bool side_above = false;
          int dwin = 16;
          for (int attempt = 0; attempt < 2 && !gathered; ++attempt) {
            uint32_t piv[4];
            if (attempt == 1 || (lo == 0 && hi == kKeyEnd)) {
              uint32_t wl;
              unsigned long long wh;
              estimate_window(x, sm, tau, dwin, lo, hi, attempt == 1,
                              side_above ? lo : (uint32_t)hi, side_above ? mass_lo : mass_hi,
                              wl, wh);
              piv[0] = wh >= kKeyEnd ? 0xffffffffu : (uint32_t)wh;
              piv[3] = wl;
              piv[1] = piv[2] = piv[3];
              if (attempt == 0) clamp_pivots(piv, lo, hi);
            } else {
              int a, b;
              sample_span(x, sm, lo, hi, a, b);
              estimate_pivots(x, sm, lo, hi, a, b, kChunk / x.spc,
                              fminf(0.1f * x.S, mass_lo - mass_hi), mass_hi, tau, piv);
              clamp_pivots(piv, lo, hi);
            }
            n_win = gather<kBf16>(x, sm, piv[3], piv[0], &cnt_above, &mass_above);
            if (n_win <= kCap && mass_above >= tau) {
              // the boundary lies above the window: known without sorting it
              lo = piv[0];
              cnt_lo = cnt_above;
              mass_lo = mass_above;
              side_above = true;
            } else if (n_win <= kCap) {
              sort_window(x, sm, n_win);
              const float wm = n_win > 0 ? sm.lcum[n_win - 1] : 0.f;
              if (tau <= mass_above + wm) {
                gathered = sorted = true;
              } else {
                hi = piv[3];
                cnt_hi = cnt_above + (unsigned long long)n_win;
                mass_hi = mass_above + wm;
                side_above = false;
              }
            } else if (mass_above >= tau) {
              lo = piv[0];
              cnt_lo = cnt_above;
              mass_lo = mass_above;
              side_above = true;
            } else {                            // too many in the window: the boundary is below its top
              hi = piv[0];
              cnt_hi = cnt_above;
              mass_hi = mass_above;
              side_above = false;
              dwin = 8;
            }
          }
        }
        if (!gathered)
          ok = narrow<kBf16>(x, sm, true, 0, tau, lo, hi, cnt_lo, mass_lo, cnt_hi, mass_hi);
        if (gathered || (ok && cnt_lo - cnt_hi <= (unsigned long long)kCap)) {
          if (!gathered) n_win = gather<kBf16>(x, sm, lo, hi, &cnt_above, &mass_above);
          ok = n_win <= kCap && n_win > 0;
          if (ok) {
            if (!sorted) sort_window(x, sm, n_win);
            const int pp = window_crossing(sm, n_win, mass_above, tau);
            const int pos = min(pp, n_win - 1);
            vk = ~(uint32_t)(sm.list[pos] >> 32);
            ik = (int)(uint32_t)sm.list[pos];
            n_win = pos + 1;
          }
        } else if (ok) {
          tie_mode = true;
          vk = lo;
          cnt_above = cnt_hi;
          const float w = mass_of(x, value_of(vk));
          unsigned long long t =
              w > 0.f ? (unsigned long long)ceilf((tau - mass_hi) / w) : 1;
          t = max(1ull, min(t, cnt_lo - cnt_hi));
          ik = tie_index<kBf16>(x, sm, vk, t - 1);
          ok = ik >= 0;
        }
      }
    }
    // ---- the draw
    if (ok) {
      if (!tie_mode && cnt_above == 0) {
        tok = draw_list(x, sm, n_win, u);
      } else {
        if (!tie_mode) {
          // add the kept window entries to their chunks: per chunk a 64-bit
          // fixed-point sum (2^-40 of the row maximum's mass), exact and so
          // independent of the order of the atomics; the sample's array is
          // free by now
          unsigned long long *acc = reinterpret_cast<unsigned long long *>(sm.samp);
          for (int c = threadIdx.x; c < x.nl; c += kT) acc[c] = 0ull;
          __syncthreads();
          for (int i = threadIdx.x; i < n_win; i += kT) {
            const unsigned long long e = sm.list[i];
            const float m = mass_of(x, value_of(~(uint32_t)(e >> 32)));
            atomicAdd(&acc[chunk_of(x.r, (int)(uint32_t)e)], __float2ull_rn(m * 1099511627776.f));
          }
          __syncthreads();
          for (int c = threadIdx.x; c < x.nl; c += kT)
            if (acc[c]) sm.cabove[c] += __ull2float_rn(acc[c]) * 9.094947017729282e-13f;
        } else {
          // cabove holds the mass above vk, cmass the count of vk, per chunk:
          // ties with index <= ik are kept
          const float w = mass_of(x, value_of(vk));
          const int cik = chunk_of(x.r, ik);
          for (int c = threadIdx.x; c < cik; c += kT) sm.cabove[c] += sm.cmass[c] * w;
          __syncthreads();
          if (warp == 0) {
            float v[kLE];
            int i0;
            const int n = chunk_lane<kBf16>(x.r, cik, lane, v, i0);
            int tc = 0;
            for (int j = 0; j < n; ++j) tc += key_of(v[j]) == vk && i0 + j <= ik;
            tc = __reduce_add_sync(0xffffffffu, tc);
            if (lane == 0) sm.cabove[cik] += (float)tc * w;
          }
        }
        __syncthreads();
        tok = draw_chunks<kBf16>(x, sm, u, vk, ik);
      }
    }
  }
  if (threadIdx.x == 0) {
    if (tok < 0) report(p.status, MSG_DEV_INTERNAL, row, 0);
    p.tokens[row] = tok;
  }
}

// ---- every row greedy (no temperatures): the token is the row's first
// maximum.  One CTA per row (two per SM, so a batch of up to twice the SMs is
// resident at once) reads the row once from HBM, each thread with 128 bytes
// of logits in flight (8 vectors of 8 bf16, 4 of 8 fp32), keeping the
// largest (key, ~index) it sees; a NaN anywhere marks the row bad.  One
// launch, no workspace traffic.
constexpr int kGreedyThreads = 512;

template <bool kBf16>
__global__ void __launch_bounds__(kGreedyThreads, 2) sample_greedy_kernel(SampleParams p) {
  constexpr int esz = kBf16 ? 2 : 4;
  constexpr int kGreedyUnroll = kBf16 ? 8 : 4;
  const int row = blockIdx.x, t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const RowRef r = row_ref<kBf16>(p.logits + (int64_t)row * p.row_bytes, p.vocab);
  bool bad = false;
  unsigned long long best = 0;                  // (key << 32) | ~index, max wins
  auto take = [&](const float v[kLE], int n, int i0) {
    float mv = -INFINITY;
#pragma unroll
    for (int j = 0; j < kLE; ++j)
      if (j < n) mv = fmax_nan(mv, v[j]);
    bad |= mv != mv;
    const unsigned long long kmv = (unsigned long long)key_of(mv) << 32;
    if (n > 0 && (kmv | 0xffffffffu) > best) {  // this vector may hold a better (key, index)
      int jj = 0;
#pragma unroll
      for (int j = kLE - 1; j >= 0; --j)
        if (j < n && v[j] == mv) jj = j;
      const unsigned long long kk = kmv | (0xffffffffu - (uint32_t)(i0 + jj));
      best = kk > best ? kk : best;
    }
  };
  for (int base = t; base < r.nvec; base += kGreedyUnroll * kGreedyThreads) {
    uint4 raw[kGreedyUnroll][kBf16 ? 1 : 2];
#pragma unroll
    for (int u = 0; u < kGreedyUnroll; ++u) {   // every load of the round in flight at once
      const int vi = base + u * kGreedyThreads;
      if (vi < r.nvec) {
        const uint8_t *src = r.p + (int64_t)(r.h + kLE * vi) * esz;
        asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(raw[u][0].x), "=r"(raw[u][0].y), "=r"(raw[u][0].z), "=r"(raw[u][0].w)
                     : "l"(src));
        if (!kBf16)
          asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                       : "=r"(raw[u][kBf16 ? 0 : 1].x), "=r"(raw[u][kBf16 ? 0 : 1].y),
                         "=r"(raw[u][kBf16 ? 0 : 1].z), "=r"(raw[u][kBf16 ? 0 : 1].w)
                       : "l"(src + 16));
      }
    }
#pragma unroll
    for (int u = 0; u < kGreedyUnroll; ++u) {
      const int vi = base + u * kGreedyThreads;
      if (vi < r.nvec) {
        float v[kLE];
        if (kBf16) {
          const uint4 w = raw[u][0];
          v[0] = bf16lo(w.x); v[1] = bf16hi(w.x); v[2] = bf16lo(w.y); v[3] = bf16hi(w.y);
          v[4] = bf16lo(w.z); v[5] = bf16hi(w.z); v[6] = bf16lo(w.w); v[7] = bf16hi(w.w);
        } else {
          const uint4 a = raw[u][0], b = raw[u][kBf16 ? 0 : 1];
          v[0] = __uint_as_float(a.x); v[1] = __uint_as_float(a.y);
          v[2] = __uint_as_float(a.z); v[3] = __uint_as_float(a.w);
          v[4] = __uint_as_float(b.x); v[5] = __uint_as_float(b.y);
          v[6] = __uint_as_float(b.z); v[7] = __uint_as_float(b.w);
        }
        take(v, kLE, r.h + kLE * vi);
      }
    }
  }
  if (t == 0) {                                 // the head and the tail (< 8 logits each)
    for (int c = 0; c < r.nch + 2; c += r.nch + 1) {
      float v[kLE];
      int i0;
      const int n = chunk_lane<kBf16>(r, c, 0, v, i0);
      take(v, n, i0);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long y = __shfl_xor_sync(0xffffffffu, best, o);
    best = y > best ? y : best;
  }
  __shared__ unsigned long long wbest[kGreedyThreads / 32];
  if (lane == 0) wbest[warp] = best;
  bad = __syncthreads_or(bad);
  if (t == 0) {
    for (int w = 1; w < kGreedyThreads / 32; ++w) best = wbest[w] > best ? wbest[w] : best;
    if (bad) report(p.status, MSG_DEV_BAD_LOGIT, row, 0);
    p.tokens[row] = bad ? -1 : (int32_t)(0xffffffffu - (uint32_t)(best & 0xffffffffu));
  }
  grid_dep_launch();
}

template <bool kBf16, bool kGreedy>
cudaError_t launch_sample(const SampleParams &p, const WsRef &ws, cudaStream_t s) {
  if (kGreedy) {
    sample_greedy_kernel<kBf16><<<dim3((unsigned)p.batch), kGreedyThreads, 0, s>>>(p);
    return cudaGetLastError();
  }
  auto scan = sample_scan_kernel<kBf16>;
  auto rowk = sample_row_kernel<kBf16>;
  static bool configured = false;
  if (!configured) {
    const cudaError_t e =
        cudaFuncSetAttribute(rowk, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(Smem));
    if (e != cudaSuccess) return e;
    configured = true;
  }
  scan<<<dim3((unsigned)ws.nparts, (unsigned)p.batch), kScanThreads, 0, s>>>(p, ws);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_k(rowk, dim3((unsigned)p.batch), dim3(kT), sizeof(Smem), s, true, p, ws);
}

// Workspace of a batch: per row the chunk maxima and masses, the sample, and
// per scan part its greedy key and finiteness flag.
struct WsSizes {
  int nl_cap, ns_cap, nparts;
  size_t bytes;
};
inline WsSizes ws_sizes(int64_t batch, int32_t vocab) {
  WsSizes z;
  const int nch_cap = (vocab + kChunk - 1) / kChunk;
  z.nl_cap = nch_cap + 2;
  z.ns_cap = 4 * nch_cap;
  z.nparts = (nch_cap + kChunksPerCta - 1) / kChunksPerCta;
  if (z.nparts < 1) z.nparts = 1;
  const size_t per_row = align_up((size_t)z.nl_cap * 4, 16) * 2 + align_up((size_t)z.ns_cap * 4, 16) +
                         align_up((size_t)z.nparts * 4, 16);
  z.bytes = per_row * (size_t)batch;
  return z;
}

}  // namespace

}  // namespace msg

extern "C" size_t msg_sample_workspace_size(int32_t batch, int32_t vocab) {
  if (batch < 0 || vocab < 1 || vocab > msg::kMaxVocab) return 0;
  return msg::ws_sizes(batch, vocab).bytes;
}

extern "C" int msg_sample(const void *logits, int32_t logits_dtype, int64_t logits_row_stride,
                          int32_t batch, int32_t vocab, const float *temperatures,
                          const int32_t *top_k, const float *top_p, const float *uniforms,
                          int32_t *tokens_out, void *workspace, size_t workspace_bytes,
                          int32_t *dev_status, void *stream) {
  using namespace msg;
  if (logits_dtype != MSG_DTYPE_F32 && logits_dtype != MSG_DTYPE_BF16) return MSG_ERR_UNSUPPORTED;
  if (batch < 0 || vocab < 1 || logits_row_stride < vocab) return MSG_ERR_INVALID_ARG;
  if (vocab > kMaxVocab) return MSG_ERR_UNSUPPORTED;
  if (batch == 0) return MSG_OK;
  if (logits == nullptr || tokens_out == nullptr) return MSG_ERR_INVALID_ARG;
  if (temperatures != nullptr && uniforms == nullptr) return MSG_ERR_INVALID_ARG;
  const int esz = logits_dtype == MSG_DTYPE_BF16 ? 2 : 4;
  if (reinterpret_cast<uintptr_t>(logits) % esz) return MSG_ERR_ALIGNMENT;
  const WsSizes z = ws_sizes(batch, vocab);
  if (workspace == nullptr || workspace_bytes < z.bytes) return MSG_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 15u) return MSG_ERR_ALIGNMENT;
  SampleParams p{};
  p.logits = static_cast<const uint8_t *>(logits);
  p.row_bytes = logits_row_stride * esz;
  p.batch = batch;
  p.vocab = vocab;
  p.temperature = temperatures;
  p.top_k = top_k;
  p.top_p = top_p;
  p.uniform = uniforms;
  p.tokens = tokens_out;
  p.status = dev_status;
  uint8_t *w = static_cast<uint8_t *>(workspace);
  WsRef ws{};
  ws.nl_cap = z.nl_cap;
  ws.ns_cap = z.ns_cap;
  ws.nparts = z.nparts;
  ws.cmax = reinterpret_cast<float *>(w);
  w += align_up((size_t)z.nl_cap * 4, 16) * batch;
  ws.cmass = reinterpret_cast<float *>(w);
  w += align_up((size_t)z.nl_cap * 4, 16) * batch;
  ws.samp = reinterpret_cast<uint32_t *>(w);
  w += align_up((size_t)z.ns_cap * 4, 16) * batch;
  ws.bad = reinterpret_cast<uint32_t *>(w);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  const bool bf = logits_dtype == MSG_DTYPE_BF16;
  if (temperatures == nullptr)
    e = bf ? launch_sample<true, true>(p, ws, s) : launch_sample<false, true>(p, ws, s);
  else
    e = bf ? launch_sample<true, false>(p, ws, s) : launch_sample<false, false>(p, ws, s);
  return e == cudaSuccess ? MSG_OK : MSG_ERR_CUDA;
}

// decode.cu -- a3 + a4: split-KV GQA decode attention through the page table,
// with the log-sum-exp merge of the splits.
//
// Math ("第 0 步：一个能跑的最小推理引擎", attention operator): a decode query
// (extend_len 1) of request r sits at position device_len - 1 and sees every
// key of the request, so
//   o[h] = sum_j exp(s_j - m) V_j[h/2] / sum_j exp(s_j - m),  s_j = scale * q[h].K_j[h/2].
// K_j / V_j are gathered through the page table ("Mini-SGLang 完整剖析" 4.6.4).
//
// GB300 design (bandwidth bound, ~1 flop per byte; 16 query / 8 KV heads):
// - Work split.  The decode requests' keys are laid end to end (prefix sum from
//   the plan) and cut into equal ranges, one per CTA, two CTAs per SM.  A CTA
//   walks the requests its range touches.  A request cut by a range boundary
//   leaves per-CTA partials (normalised o and its log-sum-exp) for each KV
//   head; the warp that finishes last for (request, KV head) -- an atomic
//   counter with acquire-release semantics -- merges them.  No CTA or warp
//   ever waits on another.
// - Data movement.  One producer warp owns all global reads: it prefetches the
//   page-table entries one tile ahead, gathers whole token rows (8 KV heads x
//   256 B = 2 KiB) of K and V with cp.async.bulk (TMA, non-tensor) into a
//   3-stage shared-memory ring, copies the request's q row with the first tile
//   of a segment, and writes a small tile header (request, output row, split
//   slot).  mbarriers guard the ring (full: transaction bytes; empty: one
//   arrival per consumer warp).
// - Compute.  8 consumer warps, one per KV head; each computes BOTH query heads
//   of its GQA group from every K/V row it reads.  A lane holds 4 of the 128
//   dims; the 16 partial dot products of a tile (8 keys x 2 heads) are
//   reduce-scattered across the warp in 16 shuffles with no selects (each lane
//   walks the keys and heads in an XOR-permuted order so that the butterfly
//   never has to pick halves), then an fp32 online softmax in base 2 (scale *
//   log2 e folded into q) and the P.V accumulation, with packed f32x2 FMAs.
// - Fused store (the kFused instantiations, msg_paged_attention_store): with
//   the step's new K / V rows given, the one CTA whose range holds a request's
//   newest key gathers it from those rows instead of the pool and its producer
//   warp writes them to the key's pool slot -- store_kv done by this kernel,
//   bit-identical to running it first.
// - Waits are bounded by wall-clock time: an expired wait records
//   MSG_DEV_TIMEOUT, raises an abort flag that ends every loop, and the
//   producer drains its copies before the CTA exits.  There are no CTA-wide
//   barriers after set-up.
#include <math.h>

#include "internal.cuh"

namespace msg {

namespace {

constexpr int kTileKeys = 8;
constexpr int kStages = 3;
constexpr int64_t kMinKeysPerCta = 32;
static_assert(kDecSegPad < kMinKeysPerCta, "a CTA range must reach past any gap");

// Launch shape for HKV KV heads (query heads 2 HKV): one consumer warp per KV
// head plus the producer warp; a stage holds kTileKeys whole token rows of K
// and of V (all HKV heads), one q row and a tile header.
// Atomic add with acquire-release semantics at GPU scope: the arrival
// publishes the warp's partial (its lanes' stores ordered before it by
// __syncwarp), and the last arrival sees every earlier one's.
__device__ __forceinline__ int32_t atom_add_acq_rel(int32_t *p, int32_t v) {
  int32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v)
               : "memory");
  return old;
}

template <int HKV>
struct Dec {
  static constexpr int kHkv = HKV;
  static constexpr int kHq = kGroup * HKV;
  static constexpr int kWarps = HKV;                              // consumer warps
  static constexpr int kThreads = (kWarps + 1) * 32;              // + producer warp
  static constexpr int kRowBytes = HKV * kHeadDim * 2;            // one token's K row
  static constexpr int kKBytes = kTileKeys * kRowBytes;
  static constexpr int kQBytes = kHq * kHeadDim * 2;              // one q row
  static constexpr int kOffV = kKBytes;
  static constexpr int kOffQ = 2 * kKBytes;
  static constexpr int kOffHdr = 2 * kKBytes + kQBytes;
  static constexpr int kStageBytes = kOffHdr + 64;
  static constexpr int kPbufBytes = kWarps * kTileKeys * 4 * 4;   // per key: {p0,p0,p1,p1}
  static constexpr size_t kSmem =
      (size_t)kStages * kStageBytes + kPbufBytes + 2 * kStages * 8 + 16;
  // 16 / HKV CTAs per SM would keep the bytes in flight per SM equal for every
  // head count; the register file (96 per thread, no spills) caps it below 8
  // KV heads: 2, 4, 6, 10 CTAs for 8, 4, 2, 1 heads.
  static constexpr int kCtasPerSm = HKV == 8 ? 2 : HKV == 4 ? 4 : HKV == 2 ? 6 : 10;
};

enum : int32_t { kFirst = 1, kLast = 2, kFinal = 4, kNoRow = 8 };

struct TileHdr {
  int32_t nkeys, flags, r, qrow;
  int32_t part_slot, bf, bl, head_shift;
};

__device__ __forceinline__ int64_t cta_begin(int64_t b, int64_t K, int64_t g) { return b * K / g; }
// Largest CTA index b < g whose range starts at or before key s.
__device__ __forceinline__ int64_t cta_of_key(int64_t s, int64_t K, int64_t g) {
  int64_t b = ((s + 1) * g - 1) / K;
  return b < g - 1 ? b : g - 1;
}

// ---- packed fp32x2 arithmetic (sm_100+)
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
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
__device__ __forceinline__ float2 bf2(uint32_t w) { return make_float2(bf16lo(w), bf16hi(w)); }

// One segment: the part of decode request i that lies in this CTA's range.
struct Seg {
  int64_t S, E, lo, hi;        // request keys [S, E) and this CTA's part [lo, hi)
  const int32_t *row;          // page-table row
  int32_t r, qrow, part_slot, bf, bl, head_shift;
};

__device__ __forceinline__ Seg load_seg(const AttnParams &p, int32_t i, int64_t begin, int64_t end,
                                        int64_t b, int64_t K, int64_t g) {
  Seg s;
  s.S = p.dec_start[i];
  s.E = p.dec_start[i + 1] - kDecSegPad;      // the request's keys; a gap follows them
  s.lo = s.S > begin ? s.S : begin;
  s.hi = s.E < end ? s.E : end;
  s.r = p.dec_req[i];
  s.row = p.kv.table + p.dec_row[i];
  const int64_t q = p.dec_qrow[i];
  s.qrow = (q >= 0 && q < p.total_q) ? (int32_t)q : -1;
  const bool whole = s.S >= begin && s.E <= end;
  s.part_slot = whole ? -1 : (int32_t)(2 * b + (s.lo == begin ? 0 : 1));
  s.bf = (int32_t)cta_of_key(s.S, K, g);
  s.bl = (int32_t)cta_of_key(s.E - 1, K, g);
  s.head_shift = s.S > cta_begin(s.bf, K, g) ? 1 : 0;
  return s;
}

// Raw index entry that locates local key j (token table: the page's first
// slot; page-id forms: the page).  Loaded ahead of use; validated by raw_to_slot.
// kPage1: page_size 1, where every index form holds the slot itself.
constexpr int kMergeBatch = 4;                // split partials loaded before any is applied
constexpr int kMergeGroup = 8;                // two-level merge: splits per group
constexpr int kMergeOneLevel = 16;            // ... taken for requests cut more ways than this

template <bool kPage1>
__device__ __forceinline__ int32_t load_raw(const AttnParams &p, const int32_t *row, int64_t j) {
  return __ldg(row + (kPage1 ? j : kv_entry(p.kv, j)));
}
// Whether the index entry of key j names a slot in the pool (no report).
template <bool kPage1>
__device__ __forceinline__ bool raw_ok(const AttnParams &p, int32_t raw, int64_t j) {
  if (kPage1) return raw >= 0 && raw < p.num_slots;
  return kv_slot(p.kv, raw, j, p.num_slots, nullptr, 0) >= 0;
}
// Slot of key j; an invalid entry is reported and redirected to slot 0.
template <bool kPage1>
__device__ __forceinline__ int64_t raw_to_slot(const AttnParams &p, int32_t raw, int64_t j,
                                               int32_t r) {
  if (kPage1) {
    if (raw < 0 || raw >= p.num_slots) {
      report(p.status, MSG_DEV_SLOT_OUT_OF_RANGE, r, raw);
      return 0;
    }
    return raw;
  }
  const int64_t slot = kv_slot(p.kv, raw, j, p.num_slots, p.status, r);
  return slot < 0 ? 0 : slot;
}

// kFused: the step's new K / V rows are given (p.k_new): each request's newest
// key is read from them and stored to the pool here (compiled apart, so the
// plain kernel carries none of it).
// kTwoLevel: the instance for batches of few long requests, whose requests
// are cut into many splits; it merges those in two levels (see the merge).
template <int HKV, bool kPage1, bool kFused, bool kTwoLevel>
__global__ void __launch_bounds__(Dec<HKV>::kThreads, Dec<HKV>::kCtasPerSm)
    decode_kernel(AttnParams p) {
  using S = Dec<HKV>;
  constexpr int kHkv = S::kHkv, kHq = S::kHq, kWarps = S::kWarps, kRowBytes = S::kRowBytes;
  constexpr int kQBytes = S::kQBytes, kOffV = S::kOffV, kOffQ = S::kOffQ, kOffHdr = S::kOffHdr;
  constexpr int kStageBytes = S::kStageBytes, kPbufBytes = S::kPbufBytes;
  extern __shared__ __align__(128) uint8_t smem[];
  float *pbuf = reinterpret_cast<float *>(smem + (size_t)kStages * kStageBytes);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)kStages * kStageBytes + kPbufBytes);
  uint64_t *empty = full + kStages;
  volatile int32_t *abort_flag = reinterpret_cast<volatile int32_t *>(empty + kStages);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const PlanHeader hdr = *p.hdr;
  // A decode-only call whose plan lists extend tiles is reported by thread 0,
  // after grid_dep_wait(): the status block may still be written by the
  // kernel before this one.
  const bool wrong_phase = blockIdx.x == 0 && tid == 0 && (p.flags & MSG_ATTN_DECODE_ONLY) &&
                           hdr.ext_tile_count > 0;
  const int64_t K = hdr.dec_keys;
  const int32_t nd = hdr.dec_count;
  if (K <= 0 || nd <= 0) {
    if (wrong_phase) {
      grid_dep_wait();
      report(p.status, MSG_DEV_WRONG_PHASE, hdr.ext_count, hdr.ext_tile_count);
    }
    return;
  }
  int64_t g = gridDim.x;
  const int64_t gmax = K / kMinKeysPerCta > 0 ? K / kMinKeysPerCta : 1;
  if (g > gmax) g = gmax;
  const int64_t b = blockIdx.x;
  if (b >= g) return;
  const int64_t begin = cta_begin(b, K, g), end = cta_begin(b + 1, K, g);

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kWarps);
    }
    *abort_flag = 0;
    mbar_fence_init();
  }
  __syncthreads();

  if (warp == kWarps) {
    // ------------------------------------------------------------ producer
    // first request of this CTA's range: the last i with dec_start[i] <= begin,
    // found by the whole warp 32 entries at a time (2 dependent loads for up
    // to 1024 decode requests, instead of log2(n))
    int32_t i = 0;
    {
      int32_t lo = 0, hi = nd;   // dec_start[lo] <= begin < dec_start[hi]
      while (hi - lo > 1) {
        const int32_t step = (hi - lo + 31) / 32;
        const int32_t idx = lo + lane * step;
        const bool le = idx < hi && p.dec_start[idx] <= begin;
        const uint32_t m = __ballot_sync(0xffffffffu, le);   // lane 0 always set
        const int32_t last = 31 - __clz(m);
        lo = lo + last * step;
        const int32_t nhi = lo + step;
        hi = nhi < hi ? nhi : hi;
      }
      i = lo;
    }
    Seg sg = load_seg(p, i, begin, end, b, K, g);
    // begin in a gap: the range starts with the next request (there is one:
    // a range is longer than a gap, and the last request's gap ends the space)
    if (sg.lo >= sg.hi && i + 1 < nd) sg = load_seg(p, ++i, begin, end, b, K, g);
    int64_t kt = sg.lo;                        // flattened key index of the tile
    int32_t raw = 0;
    {
      const int64_t n0 = imin64(kTileKeys, sg.hi - kt);
      if (lane < n0) raw = load_raw<kPage1>(p, sg.row, kt - sg.S + lane);
    }
    // Everything above reads only the plan and the KV index.  q and the step's
    // new rows are read after the preceding kernel.  With the new rows given
    // (kFused) the first ring stages of older pool rows are gathered before
    // that wait, while the preceding kernel's last CTAs finish.
    bool waited = !kFused;
    if (waited) {
      grid_dep_wait();
      grid_dep_launch();
    }
    // the wait, then the q rows of segments whose first tile went before it
    // (tiles issued before the wait are tiles 0 .. n-1 in stages 0 .. n-1)
    auto wait_preceding = [&](uint32_t n) {
      grid_dep_wait();
      grid_dep_launch();
      waited = true;
      if (lane == 0) {
        for (uint32_t j = 0; j < n; ++j) {
          uint8_t *stg = smem + (size_t)j * kStageBytes;
          const TileHdr *th = reinterpret_cast<const TileHdr *>(stg + kOffHdr);
          if (th->flags & kFirst) {
            const int64_t qr = th->qrow < 0 ? 0 : th->qrow;
            bulk_g2s(stg + kOffQ, p.q + qr * p.q_stride, kQBytes, &full[j]);
          }
        }
      }
      __syncwarp();
    };
    uint32_t it = 0, issued = 0;
    bool ok = true;
    while (true) {
      const int nkeys = (int)imin64(kTileKeys, sg.hi - kt);
      const bool first = (kt == sg.lo);
      const bool last = (kt + nkeys == sg.hi);
      // the range ends with this segment, or in the gap after it
      const bool fin = last && (sg.hi == end || i + 1 >= nd || sg.E + kDecSegPad >= end);
      // look one tile ahead: next segment metadata and page-table entries
      Seg nsg = sg;
      int64_t nkt = kt + nkeys;
      int32_t nraw = 0;
      if (!fin) {
        if (last) {
          nsg = load_seg(p, i + 1, begin, end, b, K, g);
          nkt = nsg.lo;
        }
        const int64_t nn = imin64(kTileKeys, nsg.hi - nkt);
        if (lane < nn) nraw = load_raw<kPage1>(p, nsg.row, nkt - nsg.S + lane);
      }
      const int st = it % kStages;
      if (!waited) {
        // wait first for a tile with a new row (the segment's last, when it
        // ends the request), one that would report, or the first to reuse a
        // stage (the consumers that free it wait too)
        const bool bad = lane < nkeys && !raw_ok<kPage1>(p, raw, kt - sg.S + lane);
        if (__any_sync(0xffffffffu, bad) || it >= (uint32_t)kStages || (last && sg.hi == sg.E) ||
            sg.qrow < 0)
          wait_preceding(issued);
      }
      if (ok && it >= (uint32_t)kStages && !mbar_wait(&empty[st], ((it / kStages) & 1) ^ 1)) {
        ok = false;
        if (lane == 0) {
          *abort_flag = 1;
          report(p.status, MSG_DEV_TIMEOUT, sg.r, kt);
        }
      }
      if (*abort_flag) ok = false;
      if (ok) {
        uint8_t *stage = smem + (size_t)st * kStageBytes;
        int64_t slot = 0;
        if (lane < nkeys) slot = raw_to_slot<kPage1>(p, raw, kt - sg.S + lane, sg.r);
        if (lane == 0) {
          TileHdr *h = reinterpret_cast<TileHdr *>(stage + kOffHdr);
          h->nkeys = nkeys;
          h->flags = (first ? kFirst : 0) | (last ? kLast : 0) | (fin ? kFinal : 0) |
                     (sg.qrow < 0 ? kNoRow : 0);
          h->r = sg.r;
          h->qrow = sg.qrow;
          h->part_slot = sg.part_slot;
          h->bf = sg.bf;
          h->bl = sg.bl;
          h->head_shift = sg.head_shift;
          if (first && sg.qrow < 0) report(p.status, MSG_DEV_BAD_LENGTHS, sg.r, p.qo_indptr[sg.r]);
          mbar_arrive_expect_tx(&full[st], (uint32_t)nkeys * 2 * kRowBytes + (first ? kQBytes : 0));
        }
        __syncwarp();
        // with the step's new rows given, a request's newest key comes from
        // them (and is stored to its pool slot below)
        const int newest = (kFused && last && sg.hi == sg.E && sg.qrow >= 0) ? nkeys - 1 : -1;
        if (lane < nkeys) {
          const int64_t off = slot * p.pool_stride_bytes;
          const uint8_t *ks = p.k_pool + off, *vs = p.v_pool + off;
          if (kFused && lane == newest) {
            ks = p.k_new + (int64_t)sg.qrow * p.new_stride_bytes;
            vs = p.v_new + (int64_t)sg.qrow * p.new_stride_bytes;
          }
          bulk_g2s(stage + lane * kRowBytes, ks, kRowBytes, &full[st]);
          bulk_g2s(stage + kOffV + lane * kRowBytes, vs, kRowBytes, &full[st]);
        }
        if (kFused && newest >= 0) {
          // store_kv of that token: its slot, the same bits the gathers read
          const int64_t nslot = __shfl_sync(0xffffffffu, slot, newest);
          const uint4 *ks = reinterpret_cast<const uint4 *>(p.k_new + (int64_t)sg.qrow * p.new_stride_bytes);
          const uint4 *vs = reinterpret_cast<const uint4 *>(p.v_new + (int64_t)sg.qrow * p.new_stride_bytes);
          const bool slot_ok = raw_ok<kPage1>(p, __shfl_sync(0xffffffffu, raw, newest),
                                              kt + newest - sg.S);
          if (slot_ok) {
            uint4 *kd = reinterpret_cast<uint4 *>(p.k_pool_w + nslot * p.pool_stride_bytes);
            uint4 *vd = reinterpret_cast<uint4 *>(p.v_pool_w + nslot * p.pool_stride_bytes);
            // two rounds of at most 2 K + 2 V chunks per lane in flight (the
            // producer's registers are the kernel's tightest)
            constexpr int kChunks = kRowBytes / 16, kPer = (kChunks + 31) / 32;
            constexpr int kRound = kPer < 2 ? kPer : 2;
#pragma unroll
            for (int u0 = 0; u0 < kPer; u0 += kRound) {
              uint4 a[kRound], c[kRound];
#pragma unroll
              for (int u = 0; u < kRound; ++u) {
                if ((u0 + u) * 32 + lane < kChunks) {
                  a[u] = ks[(u0 + u) * 32 + lane];
                  c[u] = vs[(u0 + u) * 32 + lane];
                }
              }
#pragma unroll
              for (int u = 0; u < kRound; ++u) {
                if ((u0 + u) * 32 + lane < kChunks) {
                  kd[(u0 + u) * 32 + lane] = a[u];
                  vd[(u0 + u) * 32 + lane] = c[u];
                }
              }
            }
          }
        }
        if (first && lane == 0 && waited) {
          const int64_t qr = sg.qrow < 0 ? 0 : sg.qrow;
          bulk_g2s(stage + kOffQ, p.q + qr * p.q_stride, kQBytes, &full[st]);
        }
        issued = it + 1;
      }
      ++it;
      if (fin || !ok) break;
      if (last) {
        sg = nsg;
        ++i;
      }
      kt = nkt;
      raw = nraw;
    }
    if (!waited) wait_preceding(issued);
    // Drain: the last issued use of every stage must have landed before exit.
    for (uint32_t j = issued > (uint32_t)kStages ? issued - kStages : 0; j < issued; ++j)
      mbar_wait(&full[j % kStages], (j / kStages) & 1);
    return;
  }

  // -------------------------------------------------------------- consumers
  grid_dep_wait();      // out, the split partials and the merge counters
  if (wrong_phase) report(p.status, MSG_DEV_WRONG_PHASE, hdr.ext_count, hdr.ext_tile_count);
  const int gh = warp;                          // KV head
  const int kx = (lane >> 2) & 7, hx = (lane >> 1) & 1;
  const int kl = kx, hl = hx;                   // after the butterfly: this lane's key / head
  uint32_t koff[kTileKeys];
#pragma unroll
  for (int t = 0; t < kTileKeys; ++t)
    koff[t] = (uint32_t)((t ^ kx) * kRowBytes + gh * (kHeadDim * 2) + lane * 8);
  const uint32_t voff = (uint32_t)(kOffV + gh * (kHeadDim * 2) + lane * 8);
  float *my_p = pbuf + warp * kTileKeys * 4;
  const float sl2 = p.scale_log2;

  float2 qa01 = make_float2(0.f, 0.f), qa23 = qa01, qb01 = qa01, qb23 = qa01;
  float m0 = -INFINITY, m1 = -INFINITY, lsum = 0.f;
  float2 o0a = make_float2(0.f, 0.f), o0b = o0a, o1a = o0a, o1b = o0a;

  for (uint32_t it = 0;; ++it) {
    const int st = it % kStages;
    const uint8_t *stage = smem + (size_t)st * kStageBytes;
    if (*abort_flag) break;
    if (!mbar_wait(&full[st], (it / kStages) & 1)) {
      if (lane == 0) {
        *abort_flag = 1;
        report(p.status, MSG_DEV_TIMEOUT, -1, (int64_t)it);
      }
      break;
    }
    const TileHdr h = *reinterpret_cast<const TileHdr *>(stage + kOffHdr);
    if (h.flags & kFirst) {
      const uint2 wa = *reinterpret_cast<const uint2 *>(stage + kOffQ + (2 * gh + hx) * 256 + lane * 8);
      const uint2 wb =
          *reinterpret_cast<const uint2 *>(stage + kOffQ + (2 * gh + (hx ^ 1)) * 256 + lane * 8);
      const float2 sc2 = make_float2(sl2, sl2);
      qa01 = fmul2(bf2(wa.x), sc2);
      qa23 = fmul2(bf2(wa.y), sc2);
      qb01 = fmul2(bf2(wb.x), sc2);
      qb23 = fmul2(bf2(wb.y), sc2);
      m0 = m1 = -INFINITY;
      lsum = 0.f;
      o0a = o0b = o1a = o1b = make_float2(0.f, 0.f);
    }
    const int nk = h.nkeys;

    // ---- scores: slot (t, hh) of this lane holds key t ^ kx, head hh ^ hx
    float s[16];
#pragma unroll
    for (int t = 0; t < kTileKeys; ++t) {
      const uint2 w = *reinterpret_cast<const uint2 *>(stage + koff[t]);
      const float2 k01 = bf2(w.x), k23 = bf2(w.y);
      float2 a = fmul2(k01, qa01);
      a = ffma2(k23, qa23, a);
      float2 c = fmul2(k01, qb01);
      c = ffma2(k23, qb23, c);
      s[2 * t] = a.x + a.y;
      s[2 * t + 1] = c.x + c.y;
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) s[j] += __shfl_xor_sync(0xffffffffu, s[j + 8], 16);
#pragma unroll
    for (int j = 0; j < 4; ++j) s[j] += __shfl_xor_sync(0xffffffffu, s[j + 4], 8);
#pragma unroll
    for (int j = 0; j < 2; ++j) s[j] += __shfl_xor_sync(0xffffffffu, s[j + 2], 4);
    s[0] += __shfl_xor_sync(0xffffffffu, s[1], 2);
    s[0] += __shfl_xor_sync(0xffffffffu, s[0], 1);

    // ---- online softmax (lane holds key kl, head hl)
    const float sc = kl < nk ? s[0] : -INFINITY;
    float mx = sc;
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
    const float mo = __shfl_xor_sync(0xffffffffu, mx, 2);
    const float mn0 = fmaxf(m0, hl ? mo : mx), mn1 = fmaxf(m1, hl ? mx : mo);
    const float a0 = exp2f(m0 - mn0), a1 = exp2f(m1 - mn1);
    m0 = mn0;
    m1 = mn1;
    const float pr = exp2f(sc - (hl ? mn1 : mn0));
    lsum = lsum * (hl ? a1 : a0) + pr;
    o0a = fmul2(o0a, make_float2(a0, a0));
    o0b = fmul2(o0b, make_float2(a0, a0));
    o1a = fmul2(o1a, make_float2(a1, a1));
    o1b = fmul2(o1b, make_float2(a1, a1));
    if (!(lane & 1)) *reinterpret_cast<float2 *>(my_p + kl * 4 + hl * 2) = make_float2(pr, pr);
    __syncwarp();
#pragma unroll
    for (int t = 0; t < kTileKeys; ++t) {
      if (t < nk) {
        const float4 pp = *reinterpret_cast<const float4 *>(my_p + t * 4);
        const uint2 w = *reinterpret_cast<const uint2 *>(stage + voff + t * kRowBytes);
        const float2 v01 = bf2(w.x), v23 = bf2(w.y);
        o0a = ffma2(v01, make_float2(pp.x, pp.y), o0a);
        o0b = ffma2(v23, make_float2(pp.x, pp.y), o0b);
        o1a = ffma2(v01, make_float2(pp.z, pp.w), o1a);
        o1b = ffma2(v23, make_float2(pp.z, pp.w), o1b);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);

    if (h.flags & kLast) {
      // ---- end of this request's part: normalise and write out or a partial
      float lv = (lane & 1) ? 0.f : lsum;
      lv += __shfl_xor_sync(0xffffffffu, lv, 4);
      lv += __shfl_xor_sync(0xffffffffu, lv, 8);
      lv += __shfl_xor_sync(0xffffffffu, lv, 16);
      const float l0 = __shfl_sync(0xffffffffu, lv, 0), l1 = __shfl_sync(0xffffffffu, lv, 2);
      const float i0f = 1.f / l0, i1f = 1.f / l1;
      const bool row_ok = !(h.flags & kNoRow);
      uint16_t *op = p.out + (int64_t)h.qrow * kHq * kHeadDim + (2 * gh) * kHeadDim + lane * 4;
      if (h.part_slot < 0) {
        if (row_ok) {
          *reinterpret_cast<uint2 *>(op) = make_uint2(pack_bf16(o0a.x * i0f, o0a.y * i0f),
                                                      pack_bf16(o0b.x * i0f, o0b.y * i0f));
          *reinterpret_cast<uint2 *>(op + kHeadDim) = make_uint2(
              pack_bf16(o1a.x * i1f, o1a.y * i1f), pack_bf16(o1b.x * i1f, o1b.y * i1f));
        }
      } else {
        const int64_t slot = h.part_slot;
        float *po = p.part_o + (slot * kHq + 2 * gh) * kHeadDim + lane * 4;
        *reinterpret_cast<float4 *>(po) =
            make_float4(o0a.x * i0f, o0a.y * i0f, o0b.x * i0f, o0b.y * i0f);
        *reinterpret_cast<float4 *>(po + kHeadDim) =
            make_float4(o1a.x * i1f, o1a.y * i1f, o1b.x * i1f, o1b.y * i1f);
        if (lane == 0) {
          p.part_lse[slot * kHq + 2 * gh] = m0 + log2f(l0);
          p.part_lse[slot * kHq + 2 * gh + 1] = m1 + log2f(l1);
        }
        __syncwarp();                               // released by the counter's atomic
        if constexpr (kTwoLevel) {
          // Two-level merge.  A request cut into at most kMergeOneLevel splits
          // is merged as in the one-level instance.  One cut into more is
          // merged in two levels, so that the last warp's chain of
          // dependent loads stays short: each group of kMergeGroup consecutive
          // splits by the last of its warps to finish (into the group's first
          // slot, as one more normalised partial with its lse), then the groups
          // by the last group.  The partials to merge are the slots
          // slot_of(mb + ms i), i < mn; sums run in index order at each level.
          const int ns = h.bl - h.bf + 1;
          auto slot_of = [&](int k) {
            return 2 * (int64_t)(h.bf + k) + (k == 0 ? h.head_shift : 0);
          };
          int mb = 0, ms = 1, mn = ns;
          bool to_out = ns <= kMergeOneLevel;
          {
            int32_t *ctr = &p.counters[(int64_t)h.r * kHkv + gh];
            if (!to_out) {
              mb = ((int)blockIdx.x - h.bf) / kMergeGroup * kMergeGroup;
              mn = ns - mb < kMergeGroup ? ns - mb : kMergeGroup;
              ctr = &p.gcounters[slot_of(mb) * kHkv + gh];
            }
            int old = 0;
            if (lane == 0) old = atom_add_acq_rel(ctr, 1);
            old = __shfl_sync(0xffffffffu, old, 0);
            if (old != mn - 1) mn = 0;                 // not the last: nothing to merge
          }
          while (mn > 0) {
            // the last of these partials' warps: merge them.  Their lse values
            // are loaded by the lanes side by side (partial k by lane k % 32),
            // the o rows partial after partial with several loads in flight.
            __syncwarp();                             // after lane 0's acquire
            auto mslot = [&](int k) { return slot_of(mb + ms * k); };
            // partial `lane`'s lse values and the first batch of o rows, all in
            // flight at once; the lse values stay in their lanes for the weights
            float4 xs[kMergeBatch], ys[kMergeBatch];
  #pragma unroll
            for (int u = 0; u < kMergeBatch; ++u) {
              if (u < mn) {
                const float *pr0 = p.part_o + (mslot(u) * kHq + 2 * gh) * kHeadDim + lane * 4;
                xs[u] = __ldcg(reinterpret_cast<const float4 *>(pr0));
                ys[u] = __ldcg(reinterpret_cast<const float4 *>(pr0 + kHeadDim));
              }
            }
            float l0 = -INFINITY, l1 = -INFINITY;
            if (lane < mn) {
              const int64_t sl = mslot(lane);
              l0 = __ldcg(p.part_lse + sl * kHq + 2 * gh);
              l1 = __ldcg(p.part_lse + sl * kHq + 2 * gh + 1);
            }
            float L0 = l0, L1 = l1;
            for (int k = lane + 32; k < mn; k += 32) {
              const int64_t sl = mslot(k);
              L0 = fmaxf(L0, __ldcg(p.part_lse + sl * kHq + 2 * gh));
              L1 = fmaxf(L1, __ldcg(p.part_lse + sl * kHq + 2 * gh + 1));
            }
  #pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
              L0 = fmaxf(L0, __shfl_xor_sync(0xffffffffu, L0, o));
              L1 = fmaxf(L1, __shfl_xor_sync(0xffffffffu, L1, o));
            }
            float4 n0 = make_float4(0.f, 0.f, 0.f, 0.f), n1 = n0;
            float d0 = 0.f, d1 = 0.f;
            for (int k0 = 0; k0 < mn; k0 += 32) {
              float w0 = 0.f, w1 = 0.f;
              if (k0 == 0) {
                if (lane < mn) {
                  w0 = exp2f(l0 - L0);
                  w1 = exp2f(l1 - L1);
                }
              } else if (k0 + lane < mn) {
                const int64_t sl = mslot(k0 + lane);
                w0 = exp2f(__ldcg(p.part_lse + sl * kHq + 2 * gh) - L0);
                w1 = exp2f(__ldcg(p.part_lse + sl * kHq + 2 * gh + 1) - L1);
              }
              const int nk = mn - k0 < 32 ? mn - k0 : 32;
              for (int j0 = 0; j0 < nk; j0 += kMergeBatch) {
                if (k0 > 0 || j0 > 0) {
  #pragma unroll
                  for (int u = 0; u < kMergeBatch; ++u) {   // the batch's loads, all in flight
                    if (j0 + u < nk) {
                      const float *pr0 =
                          p.part_o + (mslot(k0 + j0 + u) * kHq + 2 * gh) * kHeadDim + lane * 4;
                      xs[u] = __ldcg(reinterpret_cast<const float4 *>(pr0));
                      ys[u] = __ldcg(reinterpret_cast<const float4 *>(pr0 + kHeadDim));
                    }
                  }
                }
  #pragma unroll
                for (int u = 0; u < kMergeBatch; ++u) {
                  if (j0 + u >= nk) break;
                  const float a0 = __shfl_sync(0xffffffffu, w0, j0 + u);
                  const float a1 = __shfl_sync(0xffffffffu, w1, j0 + u);
                  const float4 x = xs[u], y = ys[u];
                  n0.x = fmaf(a0, x.x, n0.x); n0.y = fmaf(a0, x.y, n0.y);
                  n0.z = fmaf(a0, x.z, n0.z); n0.w = fmaf(a0, x.w, n0.w);
                  n1.x = fmaf(a1, y.x, n1.x); n1.y = fmaf(a1, y.y, n1.y);
                  n1.z = fmaf(a1, y.z, n1.z); n1.w = fmaf(a1, y.w, n1.w);
                  d0 += a0;
                  d1 += a1;
                }
              }
            }
            const float e0 = 1.f / d0, e1 = 1.f / d1;
            if (to_out) {
              if (row_ok) {
                *reinterpret_cast<uint2 *>(op) =
                    make_uint2(pack_bf16(n0.x * e0, n0.y * e0), pack_bf16(n0.z * e0, n0.w * e0));
                *reinterpret_cast<uint2 *>(op + kHeadDim) =
                    make_uint2(pack_bf16(n1.x * e1, n1.y * e1), pack_bf16(n1.z * e1, n1.w * e1));
              }
              if (lane == 0) p.counters[(int64_t)h.r * kHkv + gh] = 0;
              break;
            }
            // a group: its merged partial replaces the group's first one
            const int64_t gs = mslot(0);
            float *po = p.part_o + (gs * kHq + 2 * gh) * kHeadDim + lane * 4;
            *reinterpret_cast<float4 *>(po) = make_float4(n0.x * e0, n0.y * e0, n0.z * e0, n0.w * e0);
            *reinterpret_cast<float4 *>(po + kHeadDim) =
                make_float4(n1.x * e1, n1.y * e1, n1.z * e1, n1.w * e1);
            if (lane == 0) {
              p.part_lse[gs * kHq + 2 * gh] = L0 + log2f(d0);
              p.part_lse[gs * kHq + 2 * gh + 1] = L1 + log2f(d1);
              p.gcounters[gs * kHkv + gh] = 0;
            }
            __syncwarp();
            const int ng = (ns + kMergeGroup - 1) / kMergeGroup;
            int old = 0;
            if (lane == 0) old = atom_add_acq_rel(&p.counters[(int64_t)h.r * kHkv + gh], 1);
            old = __shfl_sync(0xffffffffu, old, 0);
            if (old != ng - 1) break;                  // not the last group
            mb = 0;
            ms = kMergeGroup;
            mn = ng;
            to_out = true;
          }
        } else {
          int old = 0;
          if (lane == 0) old = atom_add_acq_rel(&p.counters[(int64_t)h.r * kHkv + gh], 1);
          old = __shfl_sync(0xffffffffu, old, 0);
          if (old == h.bl - h.bf) {
            // last of the (request, KV head) splits: merge them (one level).  The splits'
            // lse values are loaded by the lanes side by side (split bf + k by
            // lane k % 32), the o rows split after split with several loads in
            // flight; the sums run in split order.
            __syncwarp();                             // after lane 0's acquire
            const int ns = h.bl - h.bf + 1;
            auto slot_of = [&](int k) {
              return 2 * (int64_t)(h.bf + k) + (k == 0 ? h.head_shift : 0);
            };
            // split `lane`'s lse values and the first batch of o rows, all in
            // flight at once; the lse values stay in their lanes for the weights
            float4 xs[kMergeBatch], ys[kMergeBatch];
  #pragma unroll
            for (int u = 0; u < kMergeBatch; ++u) {
              if (u < ns) {
                const float *pr0 = p.part_o + (slot_of(u) * kHq + 2 * gh) * kHeadDim + lane * 4;
                xs[u] = __ldcg(reinterpret_cast<const float4 *>(pr0));
                ys[u] = __ldcg(reinterpret_cast<const float4 *>(pr0 + kHeadDim));
              }
            }
            float l0 = -INFINITY, l1 = -INFINITY;
            if (lane < ns) {
              const int64_t sl = slot_of(lane);
              l0 = __ldcg(p.part_lse + sl * kHq + 2 * gh);
              l1 = __ldcg(p.part_lse + sl * kHq + 2 * gh + 1);
            }
            float L0 = l0, L1 = l1;
            for (int k = lane + 32; k < ns; k += 32) {
              const int64_t sl = slot_of(k);
              L0 = fmaxf(L0, __ldcg(p.part_lse + sl * kHq + 2 * gh));
              L1 = fmaxf(L1, __ldcg(p.part_lse + sl * kHq + 2 * gh + 1));
            }
  #pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
              L0 = fmaxf(L0, __shfl_xor_sync(0xffffffffu, L0, o));
              L1 = fmaxf(L1, __shfl_xor_sync(0xffffffffu, L1, o));
            }
            float4 n0 = make_float4(0.f, 0.f, 0.f, 0.f), n1 = n0;
            float d0 = 0.f, d1 = 0.f;
            for (int k0 = 0; k0 < ns; k0 += 32) {
              float w0 = 0.f, w1 = 0.f;
              if (k0 == 0) {
                if (lane < ns) {
                  w0 = exp2f(l0 - L0);
                  w1 = exp2f(l1 - L1);
                }
              } else if (k0 + lane < ns) {
                const int64_t sl = slot_of(k0 + lane);
                w0 = exp2f(__ldcg(p.part_lse + sl * kHq + 2 * gh) - L0);
                w1 = exp2f(__ldcg(p.part_lse + sl * kHq + 2 * gh + 1) - L1);
              }
              const int nk = ns - k0 < 32 ? ns - k0 : 32;
              for (int j0 = 0; j0 < nk; j0 += kMergeBatch) {
                if (k0 > 0 || j0 > 0) {
  #pragma unroll
                  for (int u = 0; u < kMergeBatch; ++u) {   // the batch's loads, all in flight
                    if (j0 + u < nk) {
                      const float *pr0 =
                          p.part_o + (slot_of(k0 + j0 + u) * kHq + 2 * gh) * kHeadDim + lane * 4;
                      xs[u] = __ldcg(reinterpret_cast<const float4 *>(pr0));
                      ys[u] = __ldcg(reinterpret_cast<const float4 *>(pr0 + kHeadDim));
                    }
                  }
                }
  #pragma unroll
                for (int u = 0; u < kMergeBatch; ++u) {
                  if (j0 + u >= nk) break;
                  const float a0 = __shfl_sync(0xffffffffu, w0, j0 + u);
                  const float a1 = __shfl_sync(0xffffffffu, w1, j0 + u);
                  const float4 x = xs[u], y = ys[u];
                  n0.x = fmaf(a0, x.x, n0.x); n0.y = fmaf(a0, x.y, n0.y);
                  n0.z = fmaf(a0, x.z, n0.z); n0.w = fmaf(a0, x.w, n0.w);
                  n1.x = fmaf(a1, y.x, n1.x); n1.y = fmaf(a1, y.y, n1.y);
                  n1.z = fmaf(a1, y.z, n1.z); n1.w = fmaf(a1, y.w, n1.w);
                  d0 += a0;
                  d1 += a1;
                }
              }
            }
            if (row_ok) {
              const float e0 = 1.f / d0, e1 = 1.f / d1;
              *reinterpret_cast<uint2 *>(op) =
                  make_uint2(pack_bf16(n0.x * e0, n0.y * e0), pack_bf16(n0.z * e0, n0.w * e0));
              *reinterpret_cast<uint2 *>(op + kHeadDim) =
                  make_uint2(pack_bf16(n1.x * e1, n1.y * e1), pack_bf16(n1.z * e1, n1.w * e1));
            }
            if (lane == 0) p.counters[(int64_t)h.r * kHkv + gh] = 0;
          }
        }
      }
    }
    if (h.flags & kFinal) break;
  }
}

template <int HKV>
cudaError_t launch_decode_h(const AttnParams &p, int grid, bool pdl, bool two_level,
                            cudaStream_t s) {
  using S = Dec<HKV>;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    for (auto k : {decode_kernel<HKV, true, false, false>, decode_kernel<HKV, false, false, false>,
                   decode_kernel<HKV, true, true, false>, decode_kernel<HKV, false, true, false>,
                   decode_kernel<HKV, true, false, true>, decode_kernel<HKV, false, false, true>,
                   decode_kernel<HKV, true, true, true>, decode_kernel<HKV, false, true, true>}) {
      e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)S::kSmem);
      if (e != cudaSuccess) return e;
    }
    attr_set[dev] = true;
  }
  const bool fused = p.k_new != nullptr;
  auto k = two_level
               ? (p.page_size == 1 ? (fused ? decode_kernel<HKV, true, true, true>
                                            : decode_kernel<HKV, true, false, true>)
                                   : (fused ? decode_kernel<HKV, false, true, true>
                                            : decode_kernel<HKV, false, false, true>))
               : (p.page_size == 1 ? (fused ? decode_kernel<HKV, true, true, false>
                                            : decode_kernel<HKV, true, false, false>)
                                   : (fused ? decode_kernel<HKV, false, true, false>
                                            : decode_kernel<HKV, false, false, false>));
  return launch_k(k, dim3(grid), dim3(S::kThreads), S::kSmem, s, pdl, p);
}

template <int HKV>
int ctas_per_sm_h() {
  static int cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  if (cache[dev] == 0) {
    int n = 0;
    // the shared memory of the launch decides how many CTAs share an SM
    if (cudaFuncSetAttribute(decode_kernel<HKV, true, false, false>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)Dec<HKV>::kSmem) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_kernel<HKV, true, false, false>,
                                                      Dec<HKV>::kThreads,
                                                      Dec<HKV>::kSmem) != cudaSuccess ||
        n <= 0)
      n = 1;
    cache[dev] = n < Dec<HKV>::kCtasPerSm ? n : Dec<HKV>::kCtasPerSm;
  }
  return cache[dev];
}

}  // namespace

cudaError_t launch_decode(const AttnParams &p, int grid, bool pdl, bool two_level,
                          cudaStream_t s) {
  if (p.num_qo_heads != kGroup * p.num_kv_heads) return cudaErrorInvalidValue;
  switch (p.num_kv_heads) {
    case 8: return launch_decode_h<8>(p, grid, pdl, two_level, s);
    case 4: return launch_decode_h<4>(p, grid, pdl, two_level, s);
    case 2: return launch_decode_h<2>(p, grid, pdl, two_level, s);
    case 1: return launch_decode_h<1>(p, grid, pdl, two_level, s);
    default: return cudaErrorInvalidValue;
  }
}

int decode_ctas_per_sm(int num_kv_heads) {
  switch (num_kv_heads) {
    case 8: return ctas_per_sm_h<8>();
    case 4: return ctas_per_sm_h<4>();
    case 2: return ctas_per_sm_h<2>();
    case 1: return ctas_per_sm_h<1>();
    default: return 1;
  }
}

}  // namespace msg

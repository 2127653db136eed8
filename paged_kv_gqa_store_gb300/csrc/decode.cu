// decode.cu -- a3 + a4: split-KV GQA decode attention through the page table,
// with the log-sum-exp merge of the splits.
//
// Math ("第 0 步：一个能跑的最小推理引擎", attention operator): a decode query
// (extend_len 1) of request r sits at position device_len - 1 and sees every
// key of the request, so
//   o[h] = sum_j exp(s_j - m) V_j[h/2] / sum_j exp(s_j - m),  s_j = scale * q[h].K_j[h/2].
// K_j / V_j are gathered through the page table ("Mini-SGLang 完整剖析" 4.6.4).
//
// GB300 design (bandwidth bound, ~1 flop per byte):
// - Work split.  The decode requests' keys are laid end to end (prefix sum from
//   the plan) and cut into gridDim.x equal ranges, one per persistent CTA (one
//   CTA per SM).  A CTA walks the requests its range touches; a request cut by
//   a range boundary yields per-CTA partials (normalised o and lse) that the
//   last CTA to finish that request merges (atomic counter + fence, no CTA
//   ever waits on another).  This balances any length mix to within one tile.
// - Data movement.  One producer warp gathers whole token rows (all KV heads,
//   kv_heads * 256 B) with cp.async.bulk (TMA, non-tensor) into a 3-stage
//   shared-memory ring guarded by mbarriers (full: transaction bytes; empty:
//   16 consumer-warp arrivals).  Each 2 KiB row is one contiguous HBM read.
// - Compute.  16 consumer warps; warp w owns KV head w % Hkv and 8 keys of each
//   tile, and computes BOTH query heads of the GQA group from each K/V load.
//   A lane holds 4 of the 128 dims; the 16 partial dot products (8 keys x 2
//   heads) are reduce-scattered across the warp in 16 shuffles (one score per
//   lane pair), followed by an fp32 online softmax in base 2 (scale * log2 e
//   folded into q) and the P.V accumulation.
// - Waits are bounded: an expired wait records MSG_DEV_TIMEOUT, sets an abort
//   flag that short-circuits every later wait, and the producer drains its
//   copies before the CTA exits.
#include <math.h>

#include "internal.cuh"

namespace msg {

namespace {

constexpr int64_t kMinKeysPerCta = 64;

template <int HKV>
struct Dec {
  static constexpr int kNsub = 16 / HKV;                   // warps per KV head
  static constexpr int kConsumerWarps = 16;
  static constexpr int kConsumerThreads = kConsumerWarps * 32;
  static constexpr int kThreads = kConsumerThreads + 32;   // + producer warp
  static constexpr int kTileKeys = 8 * kNsub;              // keys per stage
  static constexpr int kRowBytes = HKV * kHeadDim * 2;     // one token's K row
  static constexpr int kStages = 3;
  static constexpr int kHalfStage = kTileKeys * kRowBytes; // 32 KiB (K or V)
  static constexpr int kStageBytes = 2 * kHalfStage;
  static constexpr int kStateFloats = 4 + 2 * kHeadDim;    // m0 m1 l0 l1 o0[128] o1[128]
  static constexpr int kMergeBytes = kConsumerWarps * kStateFloats * 4;
  static constexpr int kPbufBytes = kConsumerWarps * 16 * 4;
  static constexpr size_t kSmem =
      (size_t)kStages * kStageBytes + kMergeBytes + kPbufBytes + 2 * kStages * 8 + 16;
};

__device__ __forceinline__ int64_t cta_begin(int64_t b, int64_t K, int64_t g) { return b * K / g; }
// Largest CTA index b < g whose range starts at or before key s.
__device__ __forceinline__ int64_t cta_of_key(int64_t s, int64_t K, int64_t g) {
  int64_t b = ((s + 1) * g - 1) / K;
  return b < g - 1 ? b : g - 1;
}

template <int HKV>
__global__ void __launch_bounds__(Dec<HKV>::kThreads, 1) decode_kernel(AttnParams p) {
  using C = Dec<HKV>;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t *stages = smem;
  float *merge = reinterpret_cast<float *>(smem + (size_t)C::kStages * C::kStageBytes);
  float *pbuf = merge + C::kMergeBytes / 4;
  uint64_t *full = reinterpret_cast<uint64_t *>(pbuf + C::kPbufBytes / 4);
  uint64_t *empty = full + C::kStages;
  volatile int32_t *flag = reinterpret_cast<volatile int32_t *>(empty + C::kStages);  // [0] abort [1] merge

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const PlanHeader hdr = *p.hdr;
  if (blockIdx.x == 0 && tid == 0 && (p.flags & MSG_ATTN_DECODE_ONLY) && hdr.ext_tile_count > 0)
    report(p.status, MSG_DEV_WRONG_PHASE, hdr.ext_count, hdr.ext_tile_count);
  const int64_t K = hdr.dec_keys;
  const int32_t nd = hdr.dec_count;
  if (K <= 0 || nd <= 0) return;
  int64_t g = gridDim.x;
  const int64_t gmax = K / kMinKeysPerCta > 0 ? K / kMinKeysPerCta : 1;
  if (g > gmax) g = gmax;
  const int64_t b = blockIdx.x;
  if (b >= g) return;
  const int64_t begin = cta_begin(b, K, g), end = cta_begin(b + 1, K, g);

  if (tid == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], C::kConsumerWarps);
    }
    flag[0] = 0;
    flag[1] = 0;
    mbar_fence_init();
  }
  __syncthreads();

  // First decode request whose keys reach this CTA's range.
  int32_t i0 = 0;
  {
    int32_t lo = 0, hi = nd;   // dec_start[lo] <= begin < dec_start[hi]
    while (hi - lo > 1) {
      const int32_t mid = (lo + hi) >> 1;
      if (p.dec_start[mid] <= begin) lo = mid; else hi = mid;
    }
    i0 = lo;
  }

  if (warp == C::kConsumerWarps) {
    // ------------------------------------------------------------ producer
    uint32_t it = 0, issued = 0;
    bool ok = true;
    int64_t pos = begin;
    for (int32_t i = i0; pos < end; ++i) {
      const int64_t S = p.dec_start[i], E = p.dec_start[i + 1];
      const int64_t seg_end = E < end ? E : end;
      const int32_t r = p.dec_req[i];
      const int64_t row = p.req_rows ? p.req_rows[r] : r;
      const int32_t *row_ptr = p.page_table + row * p.pt_stride;
      for (int64_t kt = pos - S; kt < seg_end - S; kt += C::kTileKeys) {
        const int nkeys = (int)imin64(C::kTileKeys, seg_end - S - kt);
        const int st = it % C::kStages;
        if (ok && it >= (uint32_t)C::kStages &&
            !mbar_wait(&empty[st], ((it / C::kStages) & 1) ^ 1)) {
          ok = false;
          if (lane == 0) {
            flag[0] = 1;
            report(p.status, MSG_DEV_TIMEOUT, r, kt);
          }
        }
        if (flag[0]) ok = false;
        if (ok) {
          if (lane == 0) mbar_arrive_expect_tx(&full[st], (uint32_t)nkeys * C::kRowBytes * 2);
          __syncwarp();
          uint8_t *kdst = stages + (size_t)st * C::kStageBytes;
          uint8_t *vdst = kdst + C::kHalfStage;
          for (int l = lane; l < nkeys; l += 32) {
            const int64_t slot =
                page_slot(row_ptr, kt + l, p.page_size, p.page_shift, p.num_slots, p.status, r);
            const int64_t off = slot * p.pool_stride_bytes;
            bulk_g2s(kdst + l * C::kRowBytes, p.k_pool + off, C::kRowBytes, &full[st]);
            bulk_g2s(vdst + l * C::kRowBytes, p.v_pool + off, C::kRowBytes, &full[st]);
          }
          issued = it + 1;
        }
        ++it;
      }
      pos = seg_end;
    }
    // Drain: the last issued use of every stage must have landed before exit.
    for (uint32_t j = issued > (uint32_t)C::kStages ? issued - C::kStages : 0; j < issued; ++j)
      mbar_wait(&full[j % C::kStages], (j / C::kStages) & 1);
    return;
  }

  // -------------------------------------------------------------- consumers
  const int gh = warp % HKV;            // KV head of this warp
  const int sub = warp / HKV;           // which 8 keys of each tile
  const int hq = p.num_qo_heads;
  float *my_p = pbuf + warp * 16;
  uint32_t it = 0;
  int64_t pos = begin;
  for (int32_t i = i0; pos < end; ++i) {
    const int64_t S = p.dec_start[i], E = p.dec_start[i + 1];
    const int64_t seg_end = E < end ? E : end;
    const int32_t r = p.dec_req[i];
    const bool whole = (pos == S) && (seg_end == E);
    const int64_t qrow = p.qo_indptr[r];
    const bool row_ok = qrow >= 0 && qrow < p.total_q;
    if (!row_ok && tid == 0) report(p.status, MSG_DEV_BAD_LENGTHS, r, qrow);

    float q0[4] = {0.f, 0.f, 0.f, 0.f}, q1[4] = {0.f, 0.f, 0.f, 0.f};
    if (row_ok) {
      const uint16_t *qp = p.q + qrow * p.q_stride + (2 * gh) * kHeadDim + lane * 4;
      const uint2 a = *reinterpret_cast<const uint2 *>(qp);
      const uint2 c = *reinterpret_cast<const uint2 *>(qp + kHeadDim);
      q0[0] = bf16lo(a.x) * p.scale_log2; q0[1] = bf16hi(a.x) * p.scale_log2;
      q0[2] = bf16lo(a.y) * p.scale_log2; q0[3] = bf16hi(a.y) * p.scale_log2;
      q1[0] = bf16lo(c.x) * p.scale_log2; q1[1] = bf16hi(c.x) * p.scale_log2;
      q1[2] = bf16lo(c.y) * p.scale_log2; q1[3] = bf16hi(c.y) * p.scale_log2;
    }
    float m0 = -INFINITY, m1 = -INFINITY, lsum = 0.f;
    float o0[4] = {0.f, 0.f, 0.f, 0.f}, o1[4] = {0.f, 0.f, 0.f, 0.f};

    for (int64_t kt = pos - S; kt < seg_end - S; kt += C::kTileKeys) {
      const int nkeys = (int)imin64(C::kTileKeys, seg_end - S - kt);
      const int st = it % C::kStages;
      bool ok = !flag[0];
      if (ok && !mbar_wait(&full[st], (it / C::kStages) & 1)) {
        ok = false;
        if (lane == 0) {
          flag[0] = 1;
          report(p.status, MSG_DEV_TIMEOUT, r, kt);
        }
      }
      int nk = nkeys - sub * 8;
      nk = nk < 0 ? 0 : (nk > 8 ? 8 : nk);
      if (ok && nk > 0) {
        const uint8_t *kb = stages + (size_t)st * C::kStageBytes + (sub * 8) * C::kRowBytes +
                            gh * (kHeadDim * 2) + lane * 8;
        const uint8_t *vb = kb + C::kHalfStage;
        float s[16];
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          const uint2 w = *reinterpret_cast<const uint2 *>(kb + t * C::kRowBytes);
          const float k0 = bf16lo(w.x), k1 = bf16hi(w.x), k2 = bf16lo(w.y), k3 = bf16hi(w.y);
          s[2 * t] = fmaf(q0[0], k0, fmaf(q0[1], k1, fmaf(q0[2], k2, q0[3] * k3)));
          s[2 * t + 1] = fmaf(q1[0], k0, fmaf(q1[1], k1, fmaf(q1[2], k2, q1[3] * k3)));
        }
        // Reduce-scatter the 16 partial dots: afterwards lane l holds the full
        // score of key (l >> 2) for head ((l >> 1) & 1).
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const bool up = lane & 16;
          const float send = up ? s[j] : s[j + 8];
          const float keep = up ? s[j + 8] : s[j];
          s[j] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const bool up = lane & 8;
          const float send = up ? s[j] : s[j + 4];
          const float keep = up ? s[j + 4] : s[j];
          s[j] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const bool up = lane & 4;
          const float send = up ? s[j] : s[j + 2];
          const float keep = up ? s[j + 2] : s[j];
          s[j] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
        }
        {
          const bool up = lane & 2;
          const float send = up ? s[0] : s[1];
          const float keep = up ? s[1] : s[0];
          s[0] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
        }
        s[0] += __shfl_xor_sync(0xffffffffu, s[0], 1);

        const int kl = lane >> 2, hm = (lane >> 1) & 1;
        const float sc = kl < nk ? s[0] : -INFINITY;
        float mx = sc;
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        const float mo = __shfl_xor_sync(0xffffffffu, mx, 2);
        const float mn0 = fmaxf(m0, hm ? mo : mx), mn1 = fmaxf(m1, hm ? mx : mo);
        const float a0 = exp2f(m0 - mn0), a1 = exp2f(m1 - mn1);
        m0 = mn0;
        m1 = mn1;
        const float pr = exp2f(sc - (hm ? mn1 : mn0));
        lsum = lsum * (hm ? a1 : a0) + pr;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          o0[c] *= a0;
          o1[c] *= a1;
        }
        if (!(lane & 1)) my_p[lane >> 1] = pr;
        __syncwarp();
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          if (t < nk) {
            const float2 pp = *reinterpret_cast<const float2 *>(my_p + 2 * t);
            const uint2 w = *reinterpret_cast<const uint2 *>(vb + t * C::kRowBytes);
            const float v[4] = {bf16lo(w.x), bf16hi(w.x), bf16lo(w.y), bf16hi(w.y)};
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              o0[c] = fmaf(pp.x, v[c], o0[c]);
              o1[c] = fmaf(pp.y, v[c], o1[c]);
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
      ++it;
    }

    // ---- end of segment: combine the kNsub warps of each KV head
    float lv = (lane & 1) ? 0.f : lsum;
    lv += __shfl_xor_sync(0xffffffffu, lv, 4);
    lv += __shfl_xor_sync(0xffffffffu, lv, 8);
    lv += __shfl_xor_sync(0xffffffffu, lv, 16);
    const float l0 = __shfl_sync(0xffffffffu, lv, 0), l1 = __shfl_sync(0xffffffffu, lv, 2);
    {
      float *ms = merge + warp * C::kStateFloats;
      if (lane == 0) {
        ms[0] = m0; ms[1] = m1; ms[2] = l0; ms[3] = l1;
      }
      *reinterpret_cast<float4 *>(ms + 4 + lane * 4) = make_float4(o0[0], o0[1], o0[2], o0[3]);
      *reinterpret_cast<float4 *>(ms + 4 + kHeadDim + lane * 4) =
          make_float4(o1[0], o1[1], o1[2], o1[3]);
    }
    named_barrier(1, C::kConsumerThreads);
    if (sub == 0) {
      float M0 = -INFINITY, M1 = -INFINITY;
#pragma unroll
      for (int s = 0; s < C::kNsub; ++s) {
        const float *ms = merge + (s * HKV + gh) * C::kStateFloats;
        M0 = fmaxf(M0, ms[0]);
        M1 = fmaxf(M1, ms[1]);
      }
      float L0 = 0.f, L1 = 0.f, O0[4] = {0.f, 0.f, 0.f, 0.f}, O1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int s = 0; s < C::kNsub; ++s) {
        const float *ms = merge + (s * HKV + gh) * C::kStateFloats;
        const float w0 = exp2f(ms[0] - M0), w1 = exp2f(ms[1] - M1);
        L0 = fmaf(ms[2], w0, L0);
        L1 = fmaf(ms[3], w1, L1);
        const float4 x = *reinterpret_cast<const float4 *>(ms + 4 + lane * 4);
        const float4 y = *reinterpret_cast<const float4 *>(ms + 4 + kHeadDim + lane * 4);
        O0[0] = fmaf(x.x, w0, O0[0]); O0[1] = fmaf(x.y, w0, O0[1]);
        O0[2] = fmaf(x.z, w0, O0[2]); O0[3] = fmaf(x.w, w0, O0[3]);
        O1[0] = fmaf(y.x, w1, O1[0]); O1[1] = fmaf(y.y, w1, O1[1]);
        O1[2] = fmaf(y.z, w1, O1[2]); O1[3] = fmaf(y.w, w1, O1[3]);
      }
      const float i0f = 1.f / L0, i1f = 1.f / L1;
      if (whole) {
        if (row_ok) {
          uint16_t *op = p.out + qrow * (int64_t)hq * kHeadDim + (2 * gh) * kHeadDim + lane * 4;
          *reinterpret_cast<uint2 *>(op) =
              make_uint2(pack_bf16(O0[0] * i0f, O0[1] * i0f), pack_bf16(O0[2] * i0f, O0[3] * i0f));
          *reinterpret_cast<uint2 *>(op + kHeadDim) =
              make_uint2(pack_bf16(O1[0] * i1f, O1[1] * i1f), pack_bf16(O1[2] * i1f, O1[3] * i1f));
        }
      } else {
        const int64_t slot = 2 * b + (pos == begin ? 0 : 1);
        float *po = p.part_o + (slot * hq + 2 * gh) * kHeadDim + lane * 4;
        *reinterpret_cast<float4 *>(po) = make_float4(O0[0] * i0f, O0[1] * i0f, O0[2] * i0f, O0[3] * i0f);
        *reinterpret_cast<float4 *>(po + kHeadDim) =
            make_float4(O1[0] * i1f, O1[1] * i1f, O1[2] * i1f, O1[3] * i1f);
        if (lane == 0) {
          p.part_lse[slot * hq + 2 * gh] = M0 + log2f(L0);
          p.part_lse[slot * hq + 2 * gh + 1] = M1 + log2f(L1);
        }
      }
    }
    if (!whole) {
      __threadfence();
      named_barrier(1, C::kConsumerThreads);
      if (tid == 0) {
        const int64_t nsplit = cta_of_key(E - 1, K, g) - cta_of_key(S, K, g) + 1;
        const int old = atomicAdd(&p.counters[r], 1);
        flag[1] = (old == nsplit - 1) ? 1 : 0;
      }
      named_barrier(1, C::kConsumerThreads);
      if (flag[1]) {
        __threadfence();
        const int64_t bf = cta_of_key(S, K, g), bl = cta_of_key(E - 1, K, g);
        const int64_t head_shift = (S > cta_begin(bf, K, g)) ? 1 : 0;
        for (int idx = tid; idx < hq * kHeadDim; idx += C::kConsumerThreads) {
          const int h = idx / kHeadDim, d = idx % kHeadDim;
          float L = -INFINITY;
          for (int64_t bb = bf; bb <= bl; ++bb) {
            const int64_t slot = 2 * bb + (bb == bf ? head_shift : 0);
            L = fmaxf(L, __ldcg(p.part_lse + slot * hq + h));
          }
          float num = 0.f, den = 0.f;
          for (int64_t bb = bf; bb <= bl; ++bb) {
            const int64_t slot = 2 * bb + (bb == bf ? head_shift : 0);
            const float w = exp2f(__ldcg(p.part_lse + slot * hq + h) - L);
            num = fmaf(w, __ldcg(p.part_o + (slot * hq + h) * kHeadDim + d), num);
            den += w;
          }
          if (row_ok) {
            __nv_bfloat16 ob = __float2bfloat16_rn(num / den);
            p.out[qrow * (int64_t)hq * kHeadDim + idx] = *reinterpret_cast<uint16_t *>(&ob);
          }
        }
        if (tid == 0) p.counters[r] = 0;
      }
    }
    named_barrier(1, C::kConsumerThreads);
    pos = seg_end;
  }
}

template <int HKV>
cudaError_t launch_decode_t(const AttnParams &p, int grid, cudaStream_t s) {
  using C = Dec<HKV>;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(decode_kernel<HKV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)C::kSmem);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  decode_kernel<HKV><<<grid, C::kThreads, C::kSmem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const AttnParams &p, int grid, cudaStream_t s) {
  switch (p.num_kv_heads) {
    case 1: return launch_decode_t<1>(p, grid, s);
    case 2: return launch_decode_t<2>(p, grid, s);
    case 4: return launch_decode_t<4>(p, grid, s);
    case 8: return launch_decode_t<8>(p, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace msg

// prologue.cu -- the step that feeds the path: q_norm / k_norm (RMSNorm per
// head), rotary embedding, and store_kv of the rotated K and of V, fused into
// one pass over the QKV projection's output ("Mini-SGLang 完整剖析" 4.6.7,
// AttentionLayer.forward; "第 0 步：一个能跑的最小推理引擎", 四个算子: rmsnorm is a
// scale with no mean or bias, rope rotates the first half of a head against
// the second half, Qwen3 norms q and k before rotating them).
//
// One warp per token, two head rows at a time: lane l works on row 2m + l/16
// of the pair and holds elements 4j .. 4j+3 and 64+4j .. 64+4j+3 (j = l % 16),
// so each element and its rotation partner sit in the same thread and the
// mean of squares is a 4-step butterfly within the half-warp.  Every row is
// two coalesced 128-byte reads and two 128-byte writes; the warp loads 8 row
// pairs (4 KB) before it processes any, and reads the token's cos/sin row
// once for all its heads.  Registers are capped for 3 CTAs (24 warps) per SM:
// the kernel is bound by how many loads are in flight and by issue, not by
// its arithmetic.  The rotary cache itself ("Mini-SGLang 完整剖析" 4.5.6) is
// built once per model by cos_sin_kernel.
#include <math.h>

#include "internal.cuh"

namespace msg {

namespace {

constexpr int kD = 128;            // head_dim
constexpr int kHalfD = kD / 2;

struct PrologueParams {
  const uint16_t *qkv;
  int64_t qkv_stride;              // elements between token rows
  int64_t num_tokens;
  const int32_t *positions;
  const uint16_t *q_w, *k_w;
  float eps;
  const float *cos_sin;
  int64_t max_pos;
  uint16_t *q_out;
  int64_t q_out_stride;
  uint8_t *k_pool, *v_pool;
  int64_t pool_stride_bytes;
  int64_t num_slots;
  const void *out_loc;
  int32_t out_loc_is_int64;
  int32_t hq, hkv;
  int32_t *status;
};

__device__ __forceinline__ float bf16_lo_f(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi_f(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

constexpr int kPairs = 8;          // row pairs of a token loaded before any is processed

__device__ __forceinline__ void unpack4(uint2 w, float (&x)[4]) {
  x[0] = bf16_lo_f(w.x);
  x[1] = bf16_hi_f(w.x);
  x[2] = bf16_lo_f(w.y);
  x[3] = bf16_hi_f(w.y);
}

__global__ void __launch_bounds__(256, 3) prologue_kernel(PrologueParams p) {
  grid_dep_wait();
  grid_dep_launch();
  const int lane = threadIdx.x & 31;
  const int h = lane >> 4;                        // which row of a pair this half-warp takes
  const int j4 = 4 * (lane & 15);                 // elements j4 .. j4+3 and 64+j4 .. 64+j4+3
  const int64_t first = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t stride = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int nk = p.hq + p.hkv;                    // q and k rows: normed and rotated
  const int units = nk + p.hkv;                   // then the v rows: copied
  const int npn = (nk + 1) / 2, nps = npn + (p.hkv + 1) / 2;   // row pairs
  float qw1[4], qw2[4], kw1[4], kw2[4];
  unpack4(*reinterpret_cast<const uint2 *>(p.q_w + j4), qw1);
  unpack4(*reinterpret_cast<const uint2 *>(p.q_w + kHalfD + j4), qw2);
  unpack4(*reinterpret_cast<const uint2 *>(p.k_w + j4), kw1);
  unpack4(*reinterpret_cast<const uint2 *>(p.k_w + kHalfD + j4), kw2);
  // one warp per token, a row pair per step: kPairs pairs in flight at a time
  for (int64_t t = first; t < p.num_tokens; t += stride) {
    const int64_t pos = p.positions[t];
    if (pos < 0 || pos >= p.max_pos) {
      if (lane == 0) report(p.status, MSG_DEV_BAD_POSITION, (int32_t)t, pos);
      continue;
    }
    const int64_t slot = p.out_loc_is_int64 ? static_cast<const int64_t *>(p.out_loc)[t]
                                            : (int64_t) static_cast<const int32_t *>(p.out_loc)[t];
    const bool slot_ok = slot >= 0 && slot < p.num_slots;
    if (!slot_ok && lane == 0) report(p.status, MSG_DEV_SLOT_OUT_OF_RANGE, (int32_t)t, slot);
    const uint16_t *row = p.qkv + t * p.qkv_stride + j4;
    const float4 c4 = *reinterpret_cast<const float4 *>(p.cos_sin + pos * kD + j4);
    const float4 s4 = *reinterpret_cast<const float4 *>(p.cos_sin + pos * kD + kHalfD + j4);
    const float cc[4] = {c4.x, c4.y, c4.z, c4.w}, sn[4] = {s4.x, s4.y, s4.z, s4.w};
    for (int s0 = 0; s0 < nps; s0 += kPairs) {
      uint2 lo[kPairs], hi[kPairs];
#pragma unroll
      for (int k = 0; k < kPairs; ++k) {
        const int s = s0 + k;
        const int u = s < npn ? 2 * s + h : nk + 2 * (s - npn) + h;
        const bool ok = s < nps && (s < npn ? u < nk : u < units);
        lo[k] = ok ? *reinterpret_cast<const uint2 *>(row + (int64_t)u * kD) : make_uint2(0, 0);
        hi[k] = ok ? *reinterpret_cast<const uint2 *>(row + (int64_t)u * kD + kHalfD)
                   : make_uint2(0, 0);
      }
#pragma unroll
      for (int k = 0; k < kPairs; ++k) {
        const int s = s0 + k;
        if (s >= nps) break;
        if (s >= npn) {                           // V: a bit copy
          const int g = 2 * (s - npn) + h;
          if (g < p.hkv && slot_ok) {
            uint8_t *dst = p.v_pool + slot * p.pool_stride_bytes + (int64_t)g * kD * 2 + 2 * j4;
            *reinterpret_cast<uint2 *>(dst) = lo[k];
            *reinterpret_cast<uint2 *>(dst + kD) = hi[k];
          }
          continue;
        }
        const int u = 2 * s + h;
        const bool is_q = u < p.hq;
        float x1[4], x2[4];
        unpack4(lo[k], x1);
        unpack4(hi[k], x2);
        // RMSNorm: x * w / sqrt(mean(x^2) + eps), the sum over the half-warp
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e) ss += x1[e] * x1[e] + x2[e] * x2[e];
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
        const float r = rsqrtf(ss * (1.f / kD) + p.eps);
        float o1[4], o2[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float y1 = (is_q ? qw1[e] : kw1[e]) * (x1[e] * r);
          const float y2 = (is_q ? qw2[e] : kw2[e]) * (x2[e] * r);
          o1[e] = y1 * cc[e] - y2 * sn[e];        // x1 c - x2 s
          o2[e] = y1 * sn[e] + y2 * cc[e];        // x1 s + x2 c
        }
        uint2 a, b;
        a.x = pack_bf16(o1[0], o1[1]);
        a.y = pack_bf16(o1[2], o1[3]);
        b.x = pack_bf16(o2[0], o2[1]);
        b.y = pack_bf16(o2[2], o2[3]);
        if (u >= nk) continue;
        if (is_q) {
          uint16_t *dst = p.q_out + t * p.q_out_stride + (int64_t)u * kD + j4;
          *reinterpret_cast<uint2 *>(dst) = a;
          *reinterpret_cast<uint2 *>(dst + kHalfD) = b;
        } else if (slot_ok) {
          uint8_t *dst = p.k_pool + slot * p.pool_stride_bytes + (int64_t)(u - p.hq) * kD * 2 + 2 * j4;
          *reinterpret_cast<uint2 *>(dst) = a;
          *reinterpret_cast<uint2 *>(dst + kD) = b;
        }
      }
    }
  }
}

// Rotary cache row p: cos of the fp32 angles, then their sin.
__global__ void cos_sin_kernel(double theta, int32_t d, int64_t max_pos, float *out) {
  const int32_t half = d / 2;
  const int64_t n = max_pos * half;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < n;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int64_t pos = e / half;
    const int32_t i = (int32_t)(e - pos * half);
    const float inv_freq = (float)pow(theta, -2.0 * (double)i / (double)d);
    const float angle = __fmul_rn((float)pos, inv_freq);
    out[pos * d + i] = (float)cos((double)angle);
    out[pos * d + half + i] = (float)sin((double)angle);
  }
}

}  // namespace

}  // namespace msg

extern "C" int msg_rope_cos_sin_cache(double theta, int32_t head_dim, int64_t max_pos, float *out,
                                      void *stream) {
  using namespace msg;
  if (!(theta > 0.0) || head_dim <= 0 || (head_dim & 1) || max_pos < 1 || out == nullptr)
    return MSG_ERR_INVALID_ARG;
  const int64_t n = max_pos * (head_dim / 2);
  int64_t blocks = (n + 255) / 256;
  const int64_t cap = (int64_t)device_sm_count() * 16;
  if (blocks > cap) blocks = cap;
  cos_sin_kernel<<<(unsigned)blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(theta, head_dim,
                                                                                 max_pos, out);
  return cudaGetLastError() == cudaSuccess ? MSG_OK : MSG_ERR_CUDA;
}

extern "C" int msg_qk_norm_rope_store(const void *qkv, int64_t qkv_row_stride, int64_t num_tokens,
                                      const int32_t *positions, const void *q_norm_w,
                                      const void *k_norm_w, float eps, const float *cos_sin,
                                      int64_t max_pos, void *q_out, int64_t q_out_row_stride,
                                      void *k_pool, void *v_pool, int64_t pool_row_stride,
                                      int64_t num_slots, const void *out_loc,
                                      int32_t out_loc_is_int64, int32_t num_qo_heads,
                                      int32_t num_kv_heads, int32_t head_dim, int32_t *dev_status,
                                      void *stream) {
  using namespace msg;
  if (num_tokens < 0 || num_qo_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || max_pos < 1 ||
      num_slots < 0 || !(eps >= 0.f) || !isfinite(eps))
    return MSG_ERR_INVALID_ARG;
  if (head_dim != kD) return MSG_ERR_UNSUPPORTED;
  if (num_tokens == 0) return MSG_OK;
  if (!qkv || !positions || !q_norm_w || !k_norm_w || !cos_sin || !q_out || !k_pool || !v_pool ||
      !out_loc)
    return MSG_ERR_INVALID_ARG;
  const int64_t row = (int64_t)(num_qo_heads + 2 * num_kv_heads) * head_dim;
  if (qkv_row_stride < row || q_out_row_stride < (int64_t)num_qo_heads * head_dim ||
      pool_row_stride < (int64_t)num_kv_heads * head_dim)
    return MSG_ERR_INVALID_ARG;
  auto a16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
  if (!a16(qkv) || !a16(q_out) || !a16(k_pool) || !a16(v_pool) || !a16(cos_sin) ||
      !a16(q_norm_w) || !a16(k_norm_w) || qkv_row_stride % 8 || q_out_row_stride % 8 ||
      pool_row_stride % 8)
    return MSG_ERR_ALIGNMENT;
  PrologueParams p{};
  p.qkv = static_cast<const uint16_t *>(qkv);
  p.qkv_stride = qkv_row_stride;
  p.num_tokens = num_tokens;
  p.positions = positions;
  p.q_w = static_cast<const uint16_t *>(q_norm_w);
  p.k_w = static_cast<const uint16_t *>(k_norm_w);
  p.eps = eps;
  p.cos_sin = cos_sin;
  p.max_pos = max_pos;
  p.q_out = static_cast<uint16_t *>(q_out);
  p.q_out_stride = q_out_row_stride;
  p.k_pool = static_cast<uint8_t *>(k_pool);
  p.v_pool = static_cast<uint8_t *>(v_pool);
  p.pool_stride_bytes = pool_row_stride * 2;
  p.num_slots = num_slots;
  p.out_loc = out_loc;
  p.out_loc_is_int64 = out_loc_is_int64 ? 1 : 0;
  p.hq = num_qo_heads;
  p.hkv = num_kv_heads;
  p.status = dev_status;
  int64_t blocks = (num_tokens + 7) / 8;           // one warp per token
  const int64_t cap = (int64_t)device_sm_count() * 3;   // persistent: the 3 CTAs an SM holds
  if (blocks > cap) blocks = cap;
  return launch_k(prologue_kernel, dim3((unsigned)blocks), dim3(256), 0,
                  static_cast<cudaStream_t>(stream), true, p) == cudaSuccess
             ? MSG_OK
             : MSG_ERR_CUDA;
}

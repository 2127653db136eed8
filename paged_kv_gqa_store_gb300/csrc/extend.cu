// extend.cu -- a5: causal GQA extend (prefill / chunked prefill / prefix hit)
// attention through the page table, on tensor cores.
//
// Math ("第 0 步：一个能跑的最小推理引擎", attention operator): new token i of
// request r sits at absolute position p = cached_len + i and sees keys j <= p;
// query head h reads KV head h / 2; scores are scale * q.k, softmax, weighted V.
//
// Tiling: one CTA per (request, 64-token query tile, KV head).  The two query
// heads of the GQA group are stacked, so the tile is M = 128 rows (row = head *
// 64 + token) against key tiles of 64 gathered through the page table.  Q.K^T
// and P.V run as bf16 MMAs with fp32 accumulation; the online softmax is fp32 in
// base 2.  P is rounded to bf16 for the P.V product and the row sums add up the
// same rounded values, so a constant V is reproduced exactly.  Key tiles that
// lie wholly below the causal diagonal skip the mask; tiles past the last query
// position are never visited.
#include <math.h>

#include "internal.cuh"

namespace msg {

namespace {

constexpr int kBM = kExtendTileTokens;        // 64 query tokens
constexpr int kRows = kBM * kGroup;           // 128 rows
constexpr int kBN = 64;                       // keys per tile
constexpr int kThreads = 256;                 // 8 warps x 16 rows
constexpr int kRowBytes = kHeadDim * 2;       // 256 B per (token, head)
constexpr int kQBytes = kRows * kRowBytes;    // 32 KiB
constexpr int kKVBytes = kBN * kRowBytes;     // 16 KiB
constexpr size_t kSmem = kQBytes + 4 * (size_t)kKVBytes;   // Q + 2 x (K, V)

// 16-byte chunk c of row r in a 256-byte-row tile, XOR-swizzled so that the 8
// rows an ldmatrix phase touches fall in 8 different bank groups.
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return (uint32_t)(r * kRowBytes + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                          uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float *c, const uint32_t *a, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__global__ void __launch_bounds__(kThreads, 1) extend_kernel(AttnParams p) {
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t *qs = smem;
  uint8_t *ks[2] = {smem + kQBytes, smem + kQBytes + 2 * kKVBytes};
  uint8_t *vs[2] = {smem + kQBytes + kKVBytes, smem + kQBytes + 3 * kKVBytes};

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const PlanHeader hdr = *p.hdr;
  if (blockIdx.x == 0 && blockIdx.y == 0 && tid == 0 && (p.flags & MSG_ATTN_EXTEND_ONLY) &&
      hdr.dec_count > 0)
    report(p.status, MSG_DEV_WRONG_PHASE, hdr.dec_count, hdr.dec_keys);
  if ((int)blockIdx.x >= hdr.ext_tile_count) return;
  const int32_t r = p.ext_tiles[2 * blockIdx.x];
  const int32_t qt = p.ext_tiles[2 * blockIdx.x + 1];
  const int gh = blockIdx.y;
  const int64_t cached = p.cached_len[r];
  const int64_t ext = p.extend_len[r];
  const int64_t q0 = (int64_t)qt * kBM;
  const int nq = (int)imin64(kBM, ext - q0);
  const int64_t qrow0 = (int64_t)p.qo_indptr[r] + q0;
  if (qrow0 < 0 || qrow0 + nq > p.total_q) {
    if (tid == 0 && gh == 0) report(p.status, MSG_DEV_BAD_LENGTHS, r, qrow0);
    return;
  }
  const int64_t row = p.req_rows ? p.req_rows[r] : r;
  const int32_t *row_ptr = p.page_table + row * p.pt_stride;
  const int64_t kv_end = cached + q0 + nq;              // keys [0, kv_end)
  const int n_tiles = (int)((kv_end + kBN - 1) / kBN);
  const int hq = p.num_qo_heads;

  // ---- Q tile: rows m = h * 64 + t (t < nq), zero rows past the extend
  for (int idx = tid; idx < kRows * 16; idx += kThreads) {
    const int m = idx >> 4, c = idx & 15;
    const int h = m / kBM, t = m % kBM;
    uint8_t *dst = qs + swz(m, c);
    if (t < nq) {
      const uint16_t *src = p.q + (qrow0 + t) * p.q_stride + (2 * gh + h) * kHeadDim + c * 8;
      cp_async16(dst, src);
    } else {
      *reinterpret_cast<uint4 *>(dst) = make_uint4(0, 0, 0, 0);
    }
  }
  auto load_kv = [&](int kt, int stage) {
    for (int idx = tid; idx < kBN * 16; idx += kThreads) {
      const int n = idx >> 4, c = idx & 15;
      const int64_t j = (int64_t)kt * kBN + n;
      uint8_t *kd = ks[stage] + swz(n, c);
      uint8_t *vd = vs[stage] + swz(n, c);
      if (j < kv_end) {
        const int64_t slot =
            page_slot(row_ptr, j, p.page_size, p.page_shift, p.num_slots, p.status, r);
        const int64_t off = slot * p.pool_stride_bytes + gh * kRowBytes + c * 16;
        cp_async16(kd, p.k_pool + off);
        cp_async16(vd, p.v_pool + off);
      } else {
        *reinterpret_cast<uint4 *>(kd) = make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4 *>(vd) = make_uint4(0, 0, 0, 0);
      }
    }
  };
  load_kv(0, 0);
  cp_async_commit();

  const uint32_t qs_a = smem_u32(qs);
  uint32_t qf[8][4];
  float oacc[16][4];
#pragma unroll
  for (int j = 0; j < 16; ++j) oacc[j][0] = oacc[j][1] = oacc[j][2] = oacc[j][3] = 0.f;
  float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};
  const int lr = lane >> 2;                       // local row (and +8)
  const int m_base = warp * 16;
  const int h_warp = m_base / kBM;                // head of this warp's rows
  const int64_t pos0 = cached + q0 + (m_base % kBM) + lr;   // position of row lr
  const int64_t min_pos = cached + q0;                       // smallest position in the tile
  const float sl2 = p.scale_log2;

  for (int kt = 0; kt < n_tiles; ++kt) {
    const int st = kt & 1;
    if (kt + 1 < n_tiles) {
      load_kv(kt + 1, st ^ 1);
      cp_async_commit();
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    if (kt == 0) {
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const int m = m_base + (lane & 15), c = kk * 2 + (lane >> 4);
        ldsm_x4(qs_a + swz(m, c), qf[kk][0], qf[kk][1], qf[kk][2], qf[kk][3]);
      }
    }
    // ---- S = Q K^T (16 rows x 64 keys per warp)
    float sacc[8][4];
#pragma unroll
    for (int j = 0; j < 8; ++j) sacc[j][0] = sacc[j][1] = sacc[j][2] = sacc[j][3] = 0.f;
    const uint32_t ks_a = smem_u32(ks[st]);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        const int n = np * 16 + (lane & 7) + ((lane >> 4) << 3);
        const int c = kk * 2 + ((lane >> 3) & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(ks_a + swz(n, c), b0, b1, b2, b3);
        mma_bf16(sacc[2 * np], qf[kk], b0, b1);
        mma_bf16(sacc[2 * np + 1], qf[kk], b2, b3);
      }
    }
    // ---- scale, causal mask, online softmax (rows lr and lr + 8)
    const int64_t kbase = (int64_t)kt * kBN;
    const bool need_mask = kbase + kBN - 1 > min_pos;
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float v = sacc[j][e] * sl2;
        if (need_mask) {
          const int64_t key = kbase + j * 8 + 2 * (lane & 3) + (e & 1);
          const int64_t pos = pos0 + ((e >> 1) << 3);
          if (key > pos) v = -INFINITY;
        }
        sacc[j][e] = v;
        mx[e >> 1] = fmaxf(mx[e >> 1], v);
      }
    }
    float alpha[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 1));
      mx[i] = fmaxf(mx[i], __shfl_xor_sync(0xffffffffu, mx[i], 2));
      const float mn = fmaxf(mrow[i], mx[i]);
      alpha[i] = exp2f(mrow[i] - mn);
      mrow[i] = mn;
      lrow[i] *= alpha[i];
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      oacc[j][0] *= alpha[0];
      oacc[j][1] *= alpha[0];
      oacc[j][2] *= alpha[1];
      oacc[j][3] *= alpha[1];
    }
    // ---- O += P V with P carried as a bf16 pair (hi + lo): a single bf16 P
    // costs ~2.2e-3 relative L2 on top of the output rounding; the pair keeps
    // ~16 bits of P.  Row sums add the same hi + lo values.
    const uint32_t vs_a = smem_u32(vs[st]);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t ph[4], pl[4];
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int j = 2 * kk + half;
        const float p0 = exp2f(sacc[j][0] - mrow[0]), p1 = exp2f(sacc[j][1] - mrow[0]);
        const float p2 = exp2f(sacc[j][2] - mrow[1]), p3 = exp2f(sacc[j][3] - mrow[1]);
        const uint32_t h01 = pack_bf16(p0, p1), h23 = pack_bf16(p2, p3);
        const float r0 = p0 - bf16lo(h01), r1 = p1 - bf16hi(h01);
        const float r2 = p2 - bf16lo(h23), r3 = p3 - bf16hi(h23);
        const uint32_t l01 = pack_bf16(r0, r1), l23 = pack_bf16(r2, r3);
        lrow[0] += (bf16lo(h01) + bf16lo(l01)) + (bf16hi(h01) + bf16hi(l01));
        lrow[1] += (bf16lo(h23) + bf16lo(l23)) + (bf16hi(h23) + bf16hi(l23));
        ph[half * 2 + 0] = h01;
        ph[half * 2 + 1] = h23;
        pl[half * 2 + 0] = l01;
        pl[half * 2 + 1] = l23;
      }
#pragma unroll
      for (int dp = 0; dp < 8; ++dp) {
        const int n = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
        const int c = dp * 2 + (lane >> 4);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vs_a + swz(n, c), b0, b1, b2, b3);
        mma_bf16(oacc[2 * dp], ph, b0, b1);
        mma_bf16(oacc[2 * dp + 1], ph, b2, b3);
        mma_bf16(oacc[2 * dp], pl, b0, b1);
        mma_bf16(oacc[2 * dp + 1], pl, b2, b3);
      }
    }
    __syncthreads();
  }

  // ---- normalise and store rows with t < nq
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    lrow[i] += __shfl_xor_sync(0xffffffffu, lrow[i], 1);
    lrow[i] += __shfl_xor_sync(0xffffffffu, lrow[i], 2);
  }
  const float inv[2] = {1.f / lrow[0], 1.f / lrow[1]};
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int t = (m_base % kBM) + lr + i * 8;
    if (t < nq) {
      uint16_t *op = p.out + (qrow0 + t) * (int64_t)hq * kHeadDim + (2 * gh + h_warp) * kHeadDim +
                     2 * (lane & 3);
#pragma unroll
      for (int j = 0; j < 16; ++j)
        *reinterpret_cast<uint32_t *>(op + j * 8) =
            pack_bf16(oacc[j][2 * i] * inv[i], oacc[j][2 * i + 1] * inv[i]);
    }
  }
}

}  // namespace

cudaError_t launch_extend(const AttnParams &p, int64_t max_tiles, cudaStream_t s) {
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    e = cudaFuncSetAttribute(extend_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  if (max_tiles <= 0) return cudaSuccess;
  dim3 grid((unsigned)max_tiles, (unsigned)p.num_kv_heads);
  extend_kernel<<<grid, kThreads, kSmem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace msg

// extend.cu -- a5: causal GQA extend (prefill / chunked prefill / prefix hit)
// attention through the page table, on the sm_100-family tensor cores
// (tcgen05 MMA with TMEM accumulators, TMA loads).
//
// Math ("第 0 步：一个能跑的最小推理引擎", attention operator): new token i of
// request r sits at absolute position p = cached_len + i and sees keys j <= p;
// query head h reads KV head h / 2; scores are scale * q.k, softmax, weighted V.
//
// Work item = (request, 128-token query tile, KV head), as two sub-tiles a / b
// of 64 tokens; one persistent CTA per SM takes items until none is left.  In a
// sub-tile the two query heads of the GQA group are
// stacked, so each sub-tile is M = 128 rows (row = head * 64 + token) and both
// sub-tiles share every K/V tile of N = 128 keys (twice the MMA work per byte
// loaded).
//
//  warps 1-3    producers: K and V rows gathered through the page table with
//               TMA tile::gather4 (4 rows of 128 B per instruction, the 64
//               instructions of a tile spread over the three warps) into
//               128B-swizzled shared memory, in a ring of five 32 KiB slots
//               (K_j, V_j, K_j+1, ...).  With pages of 16 or more keys a
//               16-key run of one page is contiguous in the pool and comes
//               in as one 16-row tile load (16 instructions per K or V tile).
//  warp 0       allocates TMEM (S_a | S_b | O_a | O_b, 128 fp32 columns each),
//               loads Q by TMA (3-D tensor map over q), and one lane issues the
//               MMAs, alternating the sub-tiles:
//               O_a += P_a V_{j-1}, S_a = Q_a K_j^T, O_b += P_b V_{j-1},
//               S_b = Q_b K_j^T.  Q.K^T has both operands K-major in shared
//               memory; P.V reads P from TMEM and V (MN-major) from shared
//               memory.  So each sub-tile's softmax overlaps the other's MMAs.
//  warps 4-7,   softmax of sub-tile a, b: one thread per row (= TMEM lane
//  8-11         32 (warp % 4) + lane).  Reads its whole S row with tcgen05.ld, scale * log2 e and the causal mask
//               (only on tiles that reach the diagonal), running max (O is
//               rescaled in TMEM only when the max grows by more than 2^8 --
//               rare, and the normalisation stays exact), then writes P back
//               over S as a bf16 pair hi + lo (a single bf16 P costs ~2.2e-3
//               relative L2 on top of the output rounding; the pair keeps ~16
//               bits).  The row's denominator sums the fp32 P (within 2^-16 of
//               the pair).  P is published to the issuer once per key tile
//               (each wait the issuer makes between MMA groups lets the tensor
//               pipe drain, and the softmax runs well ahead of its P.V).  The
//               epilogue normalises O and stores bf16 rows.
//
// A batch with fewer than 4 items per SM (a chunked-prefill tile over a long
// prefix, a few long extends) leaves SMs idle when items are taken whole; for
// one that has at least 8 key tiles per SM the kernel instead splits the
// items' key tiles evenly over every CTA (the Split geometry below): a range
// boundary inside an item leaves each side's rows normalised by their own sum,
// in fp32, with their lse, and a second kernel (ext_merge_kernel) combines the
// pieces.  The host launches that split-capable instance (kSplit) only for a
// batch that can have few items; other batches run the plain work queue.
//
// All cross-role hand-offs are mbarriers; every wait is bounded in time and an
// expired one records MSG_DEV_TIMEOUT and unwinds.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <math.h>

#include <type_traits>

#include "internal.cuh"

namespace msg {

namespace {

constexpr int kSubTok = 64;                   // tokens per sub-tile
constexpr int kBN = 128;                      // keys per tile
constexpr int kThreads = 384;                 // 12 warps
constexpr int kHalf = 128 * 128;              // one 64-element-wide region of 128 rows (16 KiB)
constexpr int kQSub = 2 * kHalf;              // 32 KiB of Q per sub-tile
constexpr int kSlot = 2 * kHalf;              // 32 KiB ring slot: a K or V tile (two halves)
constexpr int kSlots = 5;
constexpr int kOffQ = 0;
constexpr int kOffRing = 2 * kQSub;
constexpr int kOffBar = kOffRing + kSlots * kSlot;
constexpr int kBarBytes = 512;               // mbarriers, TMEM address, abort flag
constexpr int kItemQueue = 8;                 // work pieces published ahead of the slowest role
constexpr int kQEntry = 12;                   // int32 per queue entry: the piece, then its item
// key split (few work items): the tiles' key-tile prefix, then the piece queue
constexpr int kOffPre = kOffBar + kBarBytes;
constexpr int kOffQueue = kOffPre + (kExtMaxTiles + 4) * 4;
constexpr int kOffGrab = kOffQueue + kItemQueue * kQEntry * 4;   // the grabber's state (GrabState)
constexpr size_t kSmem = (size_t)kOffGrab + 64 + 1024;   // + 1 KiB alignment slack
static_assert(kSmem <= 232448, "227 KiB of shared memory per CTA");
static_assert(kBN == kExtendTileTokens, "the plan counts key tiles of kExtendTileTokens keys");
constexpr uint32_t kTmemCols = 512;           // S_a | S_b | O_a | O_b
constexpr uint32_t kColS = 0, kColO = 256;
constexpr float kRescaleThreshold = 8.0f;     // log2 units: rescale O when max grows > 2^8

// mbarrier slots inside the barrier block
enum {
  kBarQFull = 0, kBarQFree = 1, kBarFull = 2, kBarEmpty = 7, kBarSFull = 12, kBarPReady = 14,
  kBarODone = 18, kBarOFree = 20, kBarEpi = 22, kBarFinal = 23, kBarItem = 24, kNumBars = 40
};  // kBarPReady + 2 x: P of sub-tile x written (kBarPReady + 2 x + 1 unused)
static_assert(kBarItem + kItemQueue <= kNumBars, "one mbarrier per queue entry");

// ---------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, int c0, int c1,
                                            int c2, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tma_gather4(void *dst, const CUtensorMap *map, int col, int r0,
                                            int r1, int r2, int r3, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(col), "r"(r0), "r"(r1), "r"(r2), "r"(r3),
      "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem desc] * B[smem desc]
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem desc]
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
        "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
        "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
      "%14,%15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
      "%13,%14,%15,%16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
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
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

// Shared-memory matrix descriptor, 128-byte swizzle (sm_100 format: start,
// leading and stride byte offsets in 16-byte units, version 1, layout 2).
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}
// Instruction descriptor, kind::f16: D fp32, A and B bf16, M = 128, N = 128.
constexpr uint32_t kIdescQK = (1u << 4) | (1u << 7) | (1u << 10) | ((128u >> 3) << 17) |
                              ((128u >> 4) << 24);
constexpr uint32_t kIdescPV = kIdescQK | (1u << 16);   // B (V) is MN-major

struct ExtParams {
  AttnParams a;
  int32_t kv_rows_per_slot;     // 64-element rows per pool slot (pool_row_stride / 64)
  int32_t kv_rows_total;        // rows of the K/V gather maps (row >= this: zero fill)
};

__device__ __forceinline__ bool aborted(volatile int32_t *f) { return *f != 0; }

// One work item: (extend tile of 128 query tokens, KV head).
struct Item {
  int64_t cached, q0, qrow0, kv_end;
  int32_t r, gh, nq, n_tiles;
  int32_t n_a;        // key tiles sub-tile a needs (its last query sits 64 tokens earlier)
  bool ok;
};

// An item as the grabber publishes it in the piece queue (every length and
// row index fits int32), and as the other roles read it back: the plan's
// global loads are made once, ahead of the roles that wait on the item.
__device__ __forceinline__ void put_item(volatile int32_t *q, const Item &it) {
  q[4] = (int32_t)it.cached;
  q[5] = (int32_t)it.q0;
  q[6] = (int32_t)it.qrow0;
  q[7] = it.r;
  q[8] = it.gh;
  q[9] = it.nq;
  q[10] = it.ok ? 1 : 0;
}
__device__ __forceinline__ Item get_item(const volatile int32_t *q) {
  Item it;
  it.cached = q[4];
  it.q0 = q[5];
  it.qrow0 = q[6];
  it.r = q[7];
  it.gh = q[8];
  it.nq = q[9];
  it.ok = q[10] != 0;
  it.kv_end = it.cached + it.q0 + it.nq;
  it.n_tiles = it.ok ? (int)((it.kv_end + kBN - 1) / kBN) : 0;
  const int64_t kv_a = it.cached + it.q0 + (it.nq < kSubTok ? it.nq : kSubTok);
  it.n_a = it.ok ? (int)((kv_a + kBN - 1) / kBN) : 0;
  return it;
}

__device__ __forceinline__ Item load_item(const AttnParams &p, int w) {
  Item it;
  const int tile = w / p.num_kv_heads;
  it.gh = w % p.num_kv_heads;
  it.r = p.ext_tiles[2 * tile];
  const int32_t qt = p.ext_tiles[2 * tile + 1];
  it.cached = p.cached_len[it.r];
  const int64_t ext = p.extend_len[it.r];
  it.q0 = (int64_t)qt * kExtendTileTokens;
  it.nq = (int)imin64(kExtendTileTokens, ext - it.q0);
  it.qrow0 = (int64_t)p.qo_indptr[it.r] + it.q0;
  it.ok = it.nq > 0 && it.qrow0 >= 0 && it.qrow0 + it.nq <= p.total_q;
  it.kv_end = it.cached + it.q0 + it.nq;              // keys [0, kv_end)
  it.n_tiles = it.ok ? (int)((it.kv_end + kBN - 1) / kBN) : 0;
  const int64_t kv_a = it.cached + it.q0 + (it.nq < kSubTok ? it.nq : kSubTok);
  it.n_a = it.ok ? (int)((kv_a + kBN - 1) / kBN) : 0;
  return it;
}

// A piece of work: key tiles [j0, j1) of item w (j1 < 0: to the item's end).
// meta, for a piece that is not the whole item: the first and the last CTA
// holding a piece of the item (bits 0-14, 15-29), whether the first CTA's
// piece is its second piece (bit 30), and bit 31 set.
struct Piece {
  int32_t w, j0, j1;
  uint32_t meta;
};

// Key split of a batch with few items (< 4 per CTA, at least 8 key tiles per
// CTA): the items, ordered KV head by KV head and within a head in the plan's
// tile order (so that neighbouring CTAs read the same K/V), laid end to end
// as units of one key tile; CTA c takes units [B(c), B(c+1)).  A boundary
// inside an item moves down (by at most one unit) so that both sub-tiles keep
// a key tile on each side.  pre[t] = first unit of tile t within a head, bit
// 31 set when sub-tile a needs one key tile fewer than sub-tile b.
struct Split {
  const int32_t *pre;
  int32_t tiles, heads, G;
  int64_t wt, w;                 // units per head, in all
  __device__ int32_t start(int t) const { return pre[t] & 0x7fffffff; }
  // largest tile t whose first unit is <= u (u within a head's units)
  __device__ int tile_of(int64_t u) const {
    int lo = 0, hi = tiles;        // start(lo) <= u < start(hi)
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (start(mid) <= u) lo = mid; else hi = mid;
    }
    return lo;
  }
  __device__ int64_t snap(int64_t u) const {
    if (u <= 0 || u >= w) return u <= 0 ? 0 : w;
    const int64_t gh = u / wt, lu = u - gh * wt;
    const int t = tile_of(lu);
    const int64_t j = lu - start(t);
    if (j == 0) return u;
    const int64_t n = start(t + 1) - start(t), na = n - (pre[t] < 0 ? 1 : 0);
    int64_t jj = j < na - 1 ? j : na - 1;
    if (jj < 0) jj = 0;
    return u - j + jj;
  }
  __device__ int64_t bound(int64_t b) const { return snap(b * w / G); }
  // the CTA whose range holds unit v
  __device__ int cta_of(int64_t v) const {
    int64_t b = ((v + 1) * G - 1) / w;
    if (b > G - 1) b = G - 1;
    if (b + 1 < G && bound(b + 1) <= v) ++b;
    return (int)b;
  }
};
// The grabber's state, in shared memory (kept out of the roles' registers).
struct GrabState {
  Split sp;
  int64_t su, su_end;               // its position in this CTA's range
  int32_t split;                    // key split (else the global counter)
};
static_assert(sizeof(GrabState) <= 64, "grabber state block");

// Next piece of CTA c's split range; a split item is also appended to the list
// (by its first piece) for the merge kernel.
__device__ Piece next_split_piece(GrabState *gs, int c, int32_t *ext_items, int32_t *count) {
  const Split &sp = gs->sp;
  if (gs->su >= gs->su_end) return Piece{-1, 0, 0, 0u};
  const int64_t su = gs->su;
  const int64_t gh = su / sp.wt, lu = su - gh * sp.wt;
  const int t = sp.tile_of(lu);
  const int64_t first = gh * sp.wt + sp.start(t);
  const int64_t n = sp.start(t + 1) - sp.start(t);
  const int32_t j0 = (int32_t)(su - first);
  const int32_t j1 = (int32_t)(n < j0 + (gs->su_end - su) ? n : j0 + (gs->su_end - su));
  const int32_t w = (int32_t)(t * sp.heads + gh);
  uint32_t meta = 0;
  if (j0 != 0 || j1 != n) {
    const int cf = sp.cta_of(first), cl = sp.cta_of(first + n - 1);
    const int hs = first > sp.bound(cf) ? 1 : 0;
    meta = (uint32_t)cf | ((uint32_t)cl << 15) | ((uint32_t)hs << 30) | (1u << 31);
    const int idx = c == cf ? atomicAdd(count, 1) : kExtSlots;
    if (idx < kExtSlots) {
      int32_t *e = ext_items + 4 * idx;
      e[1] = cf;
      e[2] = cl;
      e[3] = hs;
      e[0] = w;
    }
  }
  gs->su = su + (j1 - j0);
  return Piece{w, j0, j1, meta};
}

// Persistent: each CTA takes work items of the plan's extend tile list x KV
// heads (heaviest tiles first) from a global counter until none is left, or,
// for a batch with few items, its own range of the key split above.  TMEM,
// the mbarriers and the K/V ring live across items; every role counts tiles,
// ring items and items globally, so the phases line up without any CTA-wide
// sync.
// kSplit: the instance that may take the key split (the host launches it only
// for a batch that may have few items); the other is the plain work queue.
template <bool kSplit>
__global__ void __launch_bounds__(kThreads, 1)
    extend_kernel(const __grid_constant__ ExtParams ep, const __grid_constant__ CUtensorMap tmap_q,
                  const __grid_constant__ CUtensorMap tmap_k,
                  const __grid_constant__ CUtensorMap tmap_v,
                  const __grid_constant__ CUtensorMap tmap_kp,
                  const __grid_constant__ CUtensorMap tmap_vp) {
  extern __shared__ uint8_t smem_raw[];
  const AttnParams &p = ep.a;
  // 1 KiB-aligned base: the 128B swizzle pattern repeats every 1 KiB.
  const uint32_t raw_u32 = smem_u32(smem_raw);
  uint8_t *smem = smem_raw + (((raw_u32 + 1023u) & ~1023u) - raw_u32);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffBar);
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + kOffBar + kNumBars * 8);
  volatile int32_t *abort_flag =
      reinterpret_cast<volatile int32_t *>(smem + kOffBar + kNumBars * 8 + 8);
  volatile int32_t *piece_q = reinterpret_cast<volatile int32_t *>(smem + kOffQueue);
  int32_t *tile_pre = reinterpret_cast<int32_t *>(smem + kOffPre);
  GrabState *gs = reinterpret_cast<GrabState *>(smem + kOffGrab);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  grid_dep_wait();      // (launched without early start; kept for any launch path)
  grid_dep_launch();
  const PlanHeader hdr = *p.hdr;
  int32_t *next_ctr = const_cast<int32_t *>(&p.hdr->ext_next);
  const int items = hdr.ext_tile_count * p.num_kv_heads;
  const int G = (int)gridDim.x;
  const int64_t units = hdr.ext_units * p.num_kv_heads;
  // the key split, for a batch with few items and enough key tiles
  const bool split = kSplit && p.ext_o != nullptr && hdr.ext_split_ready != 0 && G <= kExtMaxCtas &&
                     hdr.ext_tile_count <= kExtMaxTiles && items <= kExtMaxItems &&
                     items < 4 * G && units >= 8 * (int64_t)G && units < (1ll << 30);
  // k-th piece of this CTA: taken by the producer warp 1 (lane 0) just before
  // it starts loading it (from the global counter, or the next piece of this
  // CTA's split range), published with the item's fields through the
  // kItemQueue-entry queue; every role reads the same sequence.  w = -1: no
  // more work.
  auto fetch_piece = [&](uint32_t k, bool grab, bool whole_warp, Item &it) -> Piece {
    const int e = (int)(k % kItemQueue);
    volatile int32_t *qe = piece_q + kQEntry * e;
    if (grab) {
      Piece pc{-1, 0, -1, 0u};
      if (kSplit && gs->split) {
        pc = next_split_piece(gs, (int)blockIdx.x, p.ext_items,
                              const_cast<int32_t *>(&p.hdr->ext_split_count));
      } else {
        pc.w = atomicAdd(next_ctr, 1);
        if (pc.w >= hdr.ext_tile_count * p.num_kv_heads) pc.w = -1;
      }
      qe[0] = pc.w;
      if (kSplit) {
        qe[1] = pc.j0;
        qe[2] = pc.j1;
        qe[3] = (int32_t)pc.meta;
      }
      if (pc.w >= 0) put_item(qe, load_item(p, pc.w));
      mbar_arrive(&bars[kBarItem + e]);
    }
    if (whole_warp) __syncwarp();
    if (!mbar_wait(&bars[kBarItem + e], (k / kItemQueue) & 1)) {
      *abort_flag = 1;
      report(p.status, MSG_DEV_TIMEOUT, -1, -3);
      return Piece{-1, 0, 0, 0u};
    }
    const Piece pc = kSplit ? Piece{qe[0], qe[1], qe[2], (uint32_t)qe[3]}
                            : Piece{qe[0], 0, -1, 0u};   // whole items
    if (pc.w >= 0) it = get_item(qe);
    return pc;
  };
  if (blockIdx.x == 0 && tid == 0 && (p.flags & MSG_ATTN_EXTEND_ONLY) && hdr.dec_count > 0)
    report(p.status, MSG_DEV_WRONG_PHASE, hdr.dec_count, hdr.dec_keys);
  if (!split && (int)blockIdx.x >= items) return;

  if (tid == 0) {
    mbar_init(&bars[kBarQFull], 1);
    mbar_init(&bars[kBarQFree], 1);
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(&bars[kBarFull + s], 3);          // one expect-tx arrival per producer warp
      mbar_init(&bars[kBarEmpty + s], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&bars[kBarSFull + x], 1);
      mbar_init(&bars[kBarPReady + 2 * x], 4);
      mbar_init(&bars[kBarODone + x], 1);
      mbar_init(&bars[kBarOFree + x], 4);
    }
    mbar_init(&bars[kBarEpi], 8);
    mbar_init(&bars[kBarFinal], 1);
    for (int e = 0; e < kItemQueue; ++e) mbar_init(&bars[kBarItem + e], 1);
    gs->split = split ? 1 : 0;
    gs->su = gs->su_end = 0;
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 0) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp >= 1 && warp <= 3) {
    // ------------------------------------------------------------ producers
    // Each ring item is 64 gather4 units u = half * 32 + g (keys 4g .. 4g+3,
    // 64-dim half `half` of the head slice); unit u is issued by warp
    // 1 + u % 3, lane u / 3.
    const int u = (warp - 1) + 3 * lane;
    const bool active = u < 64;
    const int half = u >> 5, kg4 = u & 31;
    const int n_units = (64 - (warp - 1) + 2) / 3;     // units of this warp: 22, 21, 21
    const int n_units16 = (16 - (warp - 1) + 2) / 3;   // with 16-key page units: 6, 5, 5
    const int oob = ep.kv_rows_total;                   // a row past the map: zero fill
    if (kSplit && split && warp == 1) {
      // the tiles' key-tile prefix (and sub-tile a's one tile fewer), then this
      // CTA's range; only the grabber (lane 0) uses them
      int64_t carry = 0;
      for (int base = 0; base < hdr.ext_tile_count; base += 32) {
        const int t = base + lane;
        int32_t n = 0, short_a = 0;
        if (t < hdr.ext_tile_count) {
          const Item ti = load_item(p, t * p.num_kv_heads);
          n = ti.n_tiles;
          short_a = ti.n_a < ti.n_tiles ? 1 : 0;
        }
        int32_t incl = n;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int32_t y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        if (t < hdr.ext_tile_count)
          tile_pre[t] = (int32_t)(carry + incl - n) | (short_a ? (int32_t)0x80000000u : 0);
        carry += __shfl_sync(0xffffffffu, incl, 31);
      }
      __syncwarp();                                  // every lane's entries, for lane 0
      if (lane == 0) {
        tile_pre[hdr.ext_tile_count] = (int32_t)carry;
        Split &sp = gs->sp;
        sp.pre = tile_pre;
        sp.tiles = hdr.ext_tile_count;
        sp.heads = p.num_kv_heads;
        sp.G = G;
        sp.wt = carry;
        sp.w = carry * p.num_kv_heads;
        if (sp.w > 0) {
          gs->su = sp.bound(blockIdx.x);
          gs->su_end = sp.bound((int64_t)blockIdx.x + 1);
        }
      }
      __syncwarp();
    }
    uint32_t N = 0;                                     // ring items issued
    bool ok = true;
    for (uint32_t k = 0; ok; ++k) {
      Item it;
      const Piece pc = fetch_piece(k, warp == 1 && lane == 0, true, it);
      if (pc.w < 0) break;
      const int j0 = pc.j0, j1 = pc.j1 < 0 ? it.n_tiles : pc.j1;
      const int na = (j1 < it.n_a ? j1 : it.n_a) - j0;
      if (j1 <= j0 || na <= 0) continue;
      const int32_t *row_ptr = kv_row(p.kv, it.r);
      // The tile loop, compiled once for page_size 1 (the entry is the slot in
      // every index form) and once for larger pages, so that the common case
      // carries none of the page arithmetic.
      auto stream_item = [&](auto page1) {
        constexpr bool kPage1 = decltype(page1)::value;
        // Index entries of this lane's 4 keys are read two tiles ahead of their
        // use, so their latency hides behind the previous tiles' waits.
        auto read_pt = [&](int j, int32_t (&raw)[4]) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int64_t key = (int64_t)j * kBN + kg4 * 4 + e;
            if (active && j < it.n_tiles && key < it.kv_end)
              raw[e] = __ldg(row_ptr + (kPage1 ? key : kv_entry(p.kv, key)));
            else
              raw[e] = 0;
          }
        };
        int32_t cur[4], nxt[4], nxt2[4];
        read_pt(j0, cur);
        read_pt(j0 + 1, nxt);
        for (int j = j0; ok && j < j1; ++j) {
          read_pt(j + 2, nxt2);
          // gather rows of this lane's 4 keys; an invalid entry (reported once,
          // by the half-0 lane) reads zeros
          int rk[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int64_t key = (int64_t)j * kBN + kg4 * 4 + e;
            rk[e] = oob;
            if (active && key < it.kv_end) {
              int64_t slot = -1;
              if constexpr (kPage1) {
                const int64_t first = cur[e];
                if (first >= 0 && first < p.num_slots) slot = first;
                else if (half == 0) report(p.status, MSG_DEV_SLOT_OUT_OF_RANGE, it.r, first);
              } else {
                slot = kv_slot(p.kv, cur[e], key, p.num_slots, half == 0 ? p.status : nullptr, it.r);
              }
              if (slot >= 0) rk[e] = (int)(slot * ep.kv_rows_per_slot + 2 * it.gh + half);
            }
            cur[e] = nxt[e];
            nxt[e] = nxt2[e];
          }
#pragma unroll
          for (int kv = 0; kv < 2; ++kv) {          // 0: K_j, 1: V_j
            const uint32_t n = N + 2 * (j - j0) + kv;
            const int s = n % kSlots;
            if (n >= (uint32_t)kSlots && !mbar_wait(&bars[kBarEmpty + s], ((n / kSlots) & 1) ^ 1)) {
              if (lane == 0) {
                *abort_flag = 1;
                report(p.status, MSG_DEV_TIMEOUT, it.r, j);
              }
              ok = false;
              break;
            }
            if (aborted(abort_flag)) {
              ok = false;
              break;
            }
            if (lane == 0) mbar_arrive_expect_tx(&bars[kBarFull + s], (uint32_t)n_units * 512u);
            __syncwarp();
            if (active)
              tma_gather4(smem + kOffRing + s * kSlot + half * kHalf + kg4 * 4 * 128,
                          kv ? &tmap_v : &tmap_k, 0, rk[0], rk[1], rk[2], rk[3], &bars[kBarFull + s]);
          }
        }
      };
      // Pages of 16 or more keys: each unit is 16 consecutive keys of one
      // page and one 64-dim half (so 16 units per K or V tile instead of 64),
      // loaded as one 16-row tile (3-D map over (half row, head half, slot))
      // when all 16 keys belong to the item, else by gather4 with zero rows
      // past the item's keys.  One index entry per unit, read two tiles ahead.
      auto stream_pages = [&]() {
        const bool act = u < 16;
        const int hf = u >> 3, g = u & 7;
        auto read_e = [&](int j) -> int32_t {
          const int64_t key = (int64_t)j * kBN + g * 16;
          return (act && j < it.n_tiles && key < it.kv_end) ? __ldg(row_ptr + kv_entry(p.kv, key))
                                                            : 0;
        };
        int32_t cur = read_e(j0), nxt = read_e(j0 + 1);
        for (int j = j0; ok && j < j1; ++j) {
          const int32_t nxt2 = read_e(j + 2);
          const int64_t key0 = (int64_t)j * kBN + g * 16;
          int64_t slot0 = -1;
          if (act && key0 < it.kv_end)
            slot0 = kv_slot(p.kv, cur, key0, p.num_slots, hf == 0 ? p.status : nullptr, it.r);
          const int64_t nvalid = imin64(16, it.kv_end - key0);   // keys of the unit in the item
          cur = nxt;
          nxt = nxt2;
#pragma unroll
          for (int kv = 0; kv < 2; ++kv) {          // 0: K_j, 1: V_j
            const uint32_t n = N + 2 * (j - j0) + kv;
            const int s = n % kSlots;
            if (n >= (uint32_t)kSlots && !mbar_wait(&bars[kBarEmpty + s], ((n / kSlots) & 1) ^ 1)) {
              if (lane == 0) {
                *abort_flag = 1;
                report(p.status, MSG_DEV_TIMEOUT, it.r, j);
              }
              ok = false;
              break;
            }
            if (aborted(abort_flag)) {
              ok = false;
              break;
            }
            if (lane == 0) mbar_arrive_expect_tx(&bars[kBarFull + s], (uint32_t)n_units16 * 2048u);
            __syncwarp();
            if (act) {
              uint8_t *dst = smem + kOffRing + s * kSlot + hf * kHalf + g * 16 * 128;
              if (slot0 >= 0 && nvalid >= 16) {
                tma_load_3d(dst, kv ? &tmap_vp : &tmap_kp, 0, 2 * it.gh + hf, (int)slot0,
                            &bars[kBarFull + s]);
              } else {
                for (int q4 = 0; q4 < 4; ++q4) {
                  int rr[4];
#pragma unroll
                  for (int e = 0; e < 4; ++e) {
                    const int k = 4 * q4 + e;
                    rr[e] = (slot0 >= 0 && k < nvalid)
                                ? (int)((slot0 + k) * ep.kv_rows_per_slot + 2 * it.gh + hf)
                                : oob;
                  }
                  tma_gather4(dst + q4 * 4 * 128, kv ? &tmap_v : &tmap_k, 0, rr[0], rr[1], rr[2],
                              rr[3], &bars[kBarFull + s]);
                }
              }
            }
          }
        }
      };
      if (p.page_size == 1) stream_item(std::true_type{});
      else if (p.page_size >= 16) stream_pages();
      else stream_item(std::false_type{});
      N += 2u * (uint32_t)(j1 - j0);
    }
    // drain: every issued ring item must have landed before the CTA can exit
    for (uint32_t n = N > (uint32_t)kSlots ? N - kSlots : 0; n < N; ++n)
      mbar_wait(&bars[kBarFull + n % kSlots], (n / kSlots) & 1);
    return;
  }

  if (warp == 0) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t q_base = smem_u32(smem + kOffQ);
      const uint32_t ring = smem_u32(smem + kOffRing);
      // descriptors differ only in the start address (low 14 bits, 16-byte units)
      const uint64_t dq0 = sdesc(q_base, 16, 1024);
      const uint64_t dring = sdesc(ring, 16, 1024);
      const uint64_t dv0 = sdesc(ring, kHalf, 1024);
      uint32_t Ts[2] = {0, 0}, N = 0, V = 0;       // tiles per sub-tile, ring items, items done
      bool ok = true;
      for (uint32_t k = 0; ok; ++k) {
        Item it;
        const Piece pc = fetch_piece(k, false, false, it);   // lane 0 alone
        if (pc.w < 0) break;
        const int j1 = pc.j1 < 0 ? it.n_tiles : pc.j1;
        const int n = j1 - pc.j0;                        // key tiles of sub-tile b
        const int na = (j1 < it.n_a ? j1 : it.n_a) - pc.j0;   // of sub-tile a
        if (n <= 0 || na <= 0) continue;
        // Q of this item, once the previous item's Q.K^T products are done
        if (V > 0 && !mbar_wait(&bars[kBarQFree], (V - 1) & 1)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&bars[kBarQFull], 2 * kQSub);
        for (int x = 0; x < 2; ++x)
          for (int h = 0; h < 2; ++h)
            for (int half = 0; half < 2; ++half)
              tma_load_3d(smem + kOffQ + x * kQSub + half * kHalf + h * (kHalf / 2), &tmap_q, 0,
                          (2 * it.gh + h) * 2 + half, (int)(it.qrow0 + x * kSubTok),
                          &bars[kBarQFull]);
        if (!mbar_wait(&bars[kBarQFull], V & 1)) {
          ok = false;
          break;
        }
        for (int j = 0; ok && j <= n; ++j) {
          const uint32_t nk = N + 2 * j, nv = N + 2 * j - 1;   // ring items K_j and V_{j-1}
          bool k_ready = false, v_ready = false;
          for (int x = 0; x < 2 && ok; ++x) {
            const int nx = x ? n : na;                 // tiles this sub-tile uses
            if (j >= 1 && j - 1 < nx) {
              // O_x += P_x(j-1) . V_{j-1}, P as the pair hi + lo
              if ((x == 0 && aborted(abort_flag)) ||
                  !mbar_wait(&bars[kBarPReady + 2 * x], (Ts[x] + j - 1) & 1) ||
                  (!v_ready && !mbar_wait(&bars[kBarFull + nv % kSlots], (nv / kSlots) & 1)) ||
                  (j == 1 && V > 0 && !mbar_wait(&bars[kBarOFree + x], (V - 1) & 1))) {
                ok = false;
                break;
              }
              v_ready = true;
              tc_fence_after();
              const uint64_t vd = dv0 + (uint64_t)(((nv % kSlots) * kSlot) >> 4);
              const uint32_t p_col = tmem + kColS + 128u * x;
              const uint32_t o_col = tmem + kColO + 128u * x;
#pragma unroll
              for (int kk = 0; kk < 8; ++kk) {
                // keys 16kk .. 16kk+15: P hi at columns 32(kk/2) + 8(kk%2), lo 16 further
                const uint32_t pc = p_col + 32u * (kk >> 1) + 8u * (kk & 1);
                const uint64_t bd = vd + (uint64_t)((kk * 2048) >> 4);
                mma_ts(o_col, pc, bd, kIdescPV, (j > 1 || kk > 0) ? 1u : 0u);
                mma_ts(o_col, pc + 16u, bd, kIdescPV, 1u);
              }
              if (!ok) break;
              mma_commit(&bars[kBarODone + x]);
            }
            if (x == 1 && j >= 1) mma_commit(&bars[kBarEmpty + nv % kSlots]);
            if (j < nx) {
              // S_x = Q_x . K_j^T
              if (!k_ready && !mbar_wait(&bars[kBarFull + nk % kSlots], (nk / kSlots) & 1)) {
                ok = false;
                break;
              }
              k_ready = true;
              tc_fence_after();
              const uint64_t kd = dring + (uint64_t)(((nk % kSlots) * kSlot) >> 4);
              const uint64_t qd = dq0 + (uint64_t)((x * kQSub) >> 4);
#pragma unroll
              for (int k = 0; k < 8; ++k) {
                const uint64_t off = (uint64_t)(((k >> 2) * kHalf + (k & 3) * 32) >> 4);
                mma_ss(tmem + kColS + 128u * x, qd + off, kd + off, kIdescQK, k > 0 ? 1u : 0u);
              }
              mma_commit(&bars[kBarSFull + x]);
            }
            if (x == 1 && j < n) {
              mma_commit(&bars[kBarEmpty + nk % kSlots]);
              if (j == n - 1) mma_commit(&bars[kBarQFree]);   // Q no longer read
            }
          }
        }
        Ts[0] += (uint32_t)na;
        Ts[1] += (uint32_t)n;
        N += 2u * (uint32_t)n;
        V += 1;
      }
      if (!ok) {
        *abort_flag = 1;
        report(p.status, MSG_DEV_TIMEOUT, -1, -1);
      }
      // every MMA of this thread must complete before TMEM is released
      mma_commit(&bars[kBarFinal]);
      mbar_wait(&bars[kBarFinal], 0);
      mbar_wait(&bars[kBarEpi], 0);
    }
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
    return;
  }

  // ---------------------------------------------------------------- softmax
  const int x = (warp - 4) >> 2;                    // sub-tile
  const int row = (warp & 3) * 32 + lane;           // = TMEM lane (warp % 4 picks the quarter)
  const int tsub = x * kSubTok + (row % kSubTok);   // token inside the item's 128-token tile
  const int hh = row / kSubTok;                     // head inside the GQA group
  const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
  const uint32_t s_col = lane_base + kColS + 128u * x;
  const uint32_t o_col = lane_base + kColO + 128u * x;
  const float sl2 = p.scale_log2;
  uint32_t T = 0;
  bool ok = true;
  for (uint32_t k = 0; ok; ++k) {
    Item it;
    const Piece pc = fetch_piece(k, false, true, it);
    if (pc.w < 0) break;
    if (it.n_tiles == 0) {
      if (x == 0 && row == 0 && !it.ok) report(p.status, MSG_DEV_BAD_LENGTHS, it.r, it.qrow0);
      continue;
    }
    const int j0 = pc.j0, j1 = pc.j1 < 0 ? it.n_tiles : pc.j1;
    const int na = (j1 < it.n_a ? j1 : it.n_a) - j0;
    if (j1 <= j0 || na <= 0) continue;
    const int64_t pos = it.cached + it.q0 + tsub;   // this row's absolute position
    const int64_t min_pos = it.cached + it.q0 + x * kSubTok;
    const int nx = x ? j1 - j0 : na;                 // key tiles this sub-tile uses
    float m = -INFINITY;                             // (stays so while every key seen is masked,
                                                     // possible in a piece that starts late)
    float2 la = make_float2(0.f, 0.f), lb = la;      // independent partial sums
    for (int j = 0; j < nx; ++j) {
      if (aborted(abort_flag) || !mbar_wait(&bars[kBarSFull + x], (T + j) & 1)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int64_t kbase = (int64_t)(j0 + j) * kBN;
      const bool need_mask = kbase + kBN - 1 > min_pos;
      // keys i of the tile with i > lim are masked (only on diagonal tiles)
      const int lim = need_mask ? (int)imin64(pos - kbase, kBN) : kBN;
      uint32_t v[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(s_col + 32u * c, v[c]);
      tmem_wait_ld();
      if (need_mask) {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (32 * c + i > lim) v[c][i] = __float_as_uint(-INFINITY);
      }
      // row max of the tile (raw scores; the scale is positive), 4 independent chains
      float mm[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) mm[q] = __uint_as_float(v[0][q]);
#pragma unroll
      for (int i = 4; i < 128; ++i)
        mm[i & 3] = fmaxf(mm[i & 3], __uint_as_float(v[i >> 5][i & 31]));
      const float mx = fmaxf(fmaxf(mm[0], mm[1]), fmaxf(mm[2], mm[3])) * sl2;
      if (j == 0) {
        m = fmaxf(mx, -1e30f);   // finite even when every key of the tile is masked
      } else if (mx > m + kRescaleThreshold) {
        // O_x holds tiles < j (their P.V completed before this S): rescale in place
        if (!mbar_wait(&bars[kBarODone + x], (T + j - 1) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const float alpha = ex2(m - mx);
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
          uint32_t o[16];
          tmem_ld16(o_col + 16u * c, o);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st16(o_col + 16u * c, o);
        }
        tmem_wait_st();
        const float2 a2 = make_float2(alpha, alpha);
        la = fmul2(la, a2);
        lb = fmul2(lb, a2);
        m = mx;
      }
      // P = exp2(s * scale - m) as a bf16 pair (hi, lo), written over S chunk by chunk:
      // chunk c (keys 32c..32c+31) -> hi in columns 32c..+15, lo in 32c+16..+31
      const float2 sc2 = make_float2(sl2, sl2), nm2 = make_float2(-m, -m);
      const float2 neg1 = make_float2(-1.f, -1.f);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t wh[16], wl[16];
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const float2 xx = ffma2(
              make_float2(__uint_as_float(v[c][i]), __uint_as_float(v[c][i + 1])), sc2, nm2);
          const float2 pp = make_float2(ex2(xx.x), ex2(xx.y));
          const uint32_t hi = pack_bf16(pp.x, pp.y);
          const float2 rr = ffma2(make_float2(bf16lo(hi), bf16hi(hi)), neg1, pp);
          wh[i >> 1] = hi;
          wl[i >> 1] = pack_bf16(rr.x, rr.y);
          if ((i >> 1) & 1) lb = fadd2(lb, pp);
          else la = fadd2(la, pp);
        }
        tmem_st16(s_col + 32u * c, wh);
        tmem_st16(s_col + 32u * c + 16u, wl);
        if (c == 3) {
          // the whole of P is in TMEM: let the MMA issuer use it
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars[kBarPReady + 2 * x]);
        }
      }
    }
    if (!ok) break;
    // ---- epilogue: O / l -> bf16, then hand O_x back to the MMA issuer
    if (!mbar_wait(&bars[kBarODone + x], (T + nx - 1) & 1)) {
      ok = false;
      break;
    }
    tc_fence_after();
    const float2 lsum2 = fadd2(la, lb);
    const float lsum = lsum2.x + lsum2.y;
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
    uint16_t *op = p.out + (it.qrow0 + tsub) * (int64_t)p.num_qo_heads * kHeadDim +
                   (2 * it.gh + hh) * kHeadDim;
    const bool part = kSplit && (pc.meta >> 31) != 0;   // one piece of a split item
    const int cf = (int)(pc.meta & 0x7fffu), hs = (int)((pc.meta >> 30) & 1u);
    // a piece's slot: 2 c for a CTA's first piece, 2 c + 1 for its last
    const int slot = 2 * (int)blockIdx.x + ((int)blockIdx.x == cf ? hs : 0);
    const int64_t prow = ((int64_t)slot * 2 + x) * 128 + row;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t o[32];
      tmem_ld32(o_col + 32u * c, o);
      tmem_wait_ld();
      if (tsub < it.nq && !part) {
#pragma unroll
        for (int i = 0; i < 32; i += 8) {
          uint4 q4;
          q4.x = pack_bf16(__uint_as_float(o[i]) * inv, __uint_as_float(o[i + 1]) * inv);
          q4.y = pack_bf16(__uint_as_float(o[i + 2]) * inv, __uint_as_float(o[i + 3]) * inv);
          q4.z = pack_bf16(__uint_as_float(o[i + 4]) * inv, __uint_as_float(o[i + 5]) * inv);
          q4.w = pack_bf16(__uint_as_float(o[i + 6]) * inv, __uint_as_float(o[i + 7]) * inv);
          *reinterpret_cast<uint4 *>(op + 32 * c + i) = q4;
        }
      } else if (tsub < it.nq) {
        // the piece's normalised rows in fp32, for the merge kernel
        float4 *po = reinterpret_cast<float4 *>(p.ext_o + prow * kHeadDim + 32 * c);
#pragma unroll
        for (int i = 0; i < 32; i += 4)
          po[i / 4] = make_float4(__uint_as_float(o[i]) * inv, __uint_as_float(o[i + 1]) * inv,
                                  __uint_as_float(o[i + 2]) * inv, __uint_as_float(o[i + 3]) * inv);
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars[kBarOFree + x]);
    T += (uint32_t)nx;
    // lse of a piece's rows (log2 units; -inf for a row none of whose keys
    // the piece holds), for the merge kernel
    if (part && tsub < it.nq) p.ext_lse[prow] = lsum > 0.f ? m + log2f(lsum) : -INFINITY;
  }
  if (!ok && lane == 0) {
    *abort_flag = 1;
    report(p.status, MSG_DEV_TIMEOUT, -1, -2);
  }
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(&bars[kBarEpi]);
}

// ---------------------------------------------------------------- split merge
// The extend kernel's grabbers append each split item once to the list (the
// item, the first and the last CTA holding a piece of it, and whether the
// first CTA's piece is its second one; ext_split_count entries, zeroed before
// each extend launch).  One wave of CTAs strides over (entry, block rb of 32
// rows of sub-tile rb / 4: consecutive tokens of one query head), 4 rows per
// warp:
// o = sum_k 2^(lse_k - L) o_k / sum_k 2^(lse_k - L) over the pieces in order,
// written as bf16 rows.  Lane k holds piece k's lse (L and the sum are warp
// reductions); lane l holds dims 4 l .. 4 l + 3 of the rows, so every load and
// store covers whole rows, and 4 rows of 4 pieces are in flight at once.
constexpr int kMergeThreads = 256;
constexpr int kMergeBlocks = 8;               // 2 sub-tiles x 4 blocks of 32 rows
constexpr int kMergeRows = 4;                 // rows per warp
constexpr int kMergePieces = 4;               // pieces in flight per row
constexpr int kMergeCtasPerSm = 2;
// One unit of merge work: 32 rows (4 per warp) of listed split item idx.
__device__ void merge_unit(const AttnParams &p, int idx, int rb, int G);
__global__ void __launch_bounds__(kMergeThreads, kMergeCtasPerSm) ext_merge_kernel(AttnParams p) {
  grid_dep_wait();                      // the extend kernel's partials and list
  grid_dep_launch();
  int n = __ldcg(&p.hdr->ext_split_count);
  if (n > kExtSlots) n = kExtSlots;
  const int G = (int)gridDim.x / kMergeCtasPerSm;   // the extend grid
  for (int u = blockIdx.x; u < n * kMergeBlocks; u += gridDim.x)
    merge_unit(p, u / kMergeBlocks, u % kMergeBlocks, G);
}

__device__ void merge_unit(const AttnParams &p, int idx, int rb, int G) {
  const int32_t *e = p.ext_items + 4 * idx;
  const int w = __ldcg(e);
  const int cf = __ldcg(e + 1), cl = __ldcg(e + 2), hs = __ldcg(e + 3);
  // an entry the extend kernel of this grid cannot have made is reported, not used
  if (w < 0 || w >= p.hdr->ext_tile_count * p.num_kv_heads || cf < 0 || cl < cf || cl >= G ||
      (hs != 0 && hs != 1)) {
    if (threadIdx.x == 0 && rb == 0)
      report(p.status, MSG_DEV_BAD_LENGTHS, w, (int64_t)cf * 65536 + cl);
    return;
  }
  const Item it = load_item(p, w);
  if (!it.ok) return;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int x = rb / 4, r0 = (rb % 4) * 32 + warp * kMergeRows;   // this warp's first row
  const int tsub0 = x * kSubTok + r0 % kSubTok;
  int rows = it.nq - tsub0;
  if (rows <= 0) return;
  if (rows > kMergeRows) rows = kMergeRows;
  const int np = cl - cf + 1;
  auto prow = [&](int k, int r) {       // partial row of piece k, row r0 + r of sub-tile x
    return ((int64_t)(2 * (cf + k) + (k == 0 ? hs : 0)) * 2 + x) * 128 + r0 + r;
  };
  // lane j holds piece k0 + j's lse of each row (32 pieces per group): L is a
  // warp max over all groups, then each group's weights 2^(lse - L) stay in
  // their lanes (summed into den by a warp reduction and shuffled to every
  // lane for its dims), and the group's rows are loaded 8 pieces at a time
  float L[kMergeRows], den[kMergeRows];
  float4 acc[kMergeRows];
#pragma unroll
  for (int r = 0; r < kMergeRows; ++r) {
    L[r] = -INFINITY;
    den[r] = 0.f;
    acc[r] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  for (int g0 = 0; g0 < np; g0 += 32) {
#pragma unroll
    for (int r = 0; r < kMergeRows; ++r)
      if (g0 + lane < np && r < rows) L[r] = fmaxf(L[r], __ldcg(p.ext_lse + prow(g0 + lane, r)));
  }
#pragma unroll
  for (int r = 0; r < kMergeRows; ++r)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L[r] = fmaxf(L[r], __shfl_xor_sync(0xffffffffu, L[r], o));
  for (int g0 = 0; g0 < np; g0 += 32) {
    float wl[kMergeRows];               // this lane's piece's weight of each row
#pragma unroll
    for (int r = 0; r < kMergeRows; ++r) {
      wl[r] = (g0 + lane < np && r < rows) ? exp2f(__ldcg(p.ext_lse + prow(g0 + lane, r)) - L[r])
                                           : 0.f;
      float d = wl[r];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
      den[r] += d;
    }
    const int gn = np - g0 < 32 ? np - g0 : 32;
    for (int j0 = 0; j0 < gn; j0 += kMergePieces) {
      float4 v[kMergePieces][kMergeRows];
#pragma unroll
      for (int j = 0; j < kMergePieces; ++j)
#pragma unroll
        for (int r = 0; r < kMergeRows; ++r)
          v[j][r] = (j0 + j < gn && r < rows)
                        ? __ldcg(reinterpret_cast<const float4 *>(
                                     p.ext_o + prow(g0 + j0 + j, r) * kHeadDim) + lane)
                        : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int j = 0; j < kMergePieces; ++j) {
#pragma unroll
        for (int r = 0; r < kMergeRows; ++r) {
          const float wk = __shfl_sync(0xffffffffu, wl[r], (j0 + j) & 31);
          acc[r].x = fmaf(wk, v[j][r].x, acc[r].x);
          acc[r].y = fmaf(wk, v[j][r].y, acc[r].y);
          acc[r].z = fmaf(wk, v[j][r].z, acc[r].z);
          acc[r].w = fmaf(wk, v[j][r].w, acc[r].w);
        }
      }
    }
  }
  const int64_t ors = (int64_t)p.num_qo_heads * kHeadDim;
  uint16_t *out = p.out + (it.qrow0 + tsub0) * ors + (2 * it.gh + r0 / kSubTok) * kHeadDim;
#pragma unroll
  for (int r = 0; r < kMergeRows; ++r) {
    if (r < rows) {
      const float rd = 1.f / den[r];
      *reinterpret_cast<uint2 *>(out + (int64_t)r * ors + 4 * lane) = make_uint2(
          pack_bf16(acc[r].x * rd, acc[r].y * rd), pack_bf16(acc[r].z * rd, acc[r].w * rd));
    }
  }
}

// ---------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (fn == nullptr) {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// 2-D map over a pool viewed as rows of 64 bf16 (128 B): box 64 x 1, 128B swizzle.
bool encode_rows(CUtensorMap *m, const void *base, uint64_t rows) {
  const cuuint64_t dims[2] = {64, rows};
  const cuuint64_t strides[1] = {128};
  const cuuint32_t box[2] = {64, 1};
  const cuuint32_t es[2] = {1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims,
                     strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

// 3-D map over a pool as (64-element half rows, half rows per slot, slots):
// box 64 x 1 x 16, one 64-dim half of 16 consecutive slots, 128B swizzle.
bool encode_pages(CUtensorMap *m, const void *base, uint64_t rows_per_slot, uint64_t slots,
                  uint64_t slot_bytes) {
  const cuuint64_t dims[3] = {64, rows_per_slot, slots};
  const cuuint64_t strides[2] = {128, slot_bytes};
  const cuuint32_t box[3] = {64, 1, 16};
  const cuuint32_t es[3] = {1, 1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims,
                     strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

// 3-D map over q: (64-element half rows, 2 per head, tokens); box 64 x 1 x 64.
bool encode_q(CUtensorMap *m, const void *q, int32_t hq, int64_t total_q, int64_t row_stride) {
  const cuuint64_t dims[3] = {64, (cuuint64_t)hq * 2, (cuuint64_t)total_q};
  const cuuint64_t strides[2] = {128, (cuuint64_t)row_stride * 2};
  const cuuint32_t box[3] = {64, 1, (cuuint32_t)kSubTok};
  const cuuint32_t es[3] = {1, 1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(q), dims, strides,
                     box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_extend(const AttnParams &p, int64_t max_tiles, int64_t max_kv_len,
                          cudaStream_t s) {
  if (max_tiles <= 0) return cudaSuccess;
  if (encode_fn() == nullptr) return cudaErrorNotSupported;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    for (auto k : {extend_kernel<false>, extend_kernel<true>}) {
      e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
      if (e != cudaSuccess) return e;
    }
    attr_set[dev] = true;
  }
  ExtParams ep{};
  ep.a = p;
  const int64_t pool_stride_elems = p.pool_stride_bytes / 2;
  if (pool_stride_elems % 64 != 0) return cudaErrorInvalidValue;
  ep.kv_rows_per_slot = (int32_t)(pool_stride_elems / 64);
  const uint64_t rows = (uint64_t)p.num_slots * (uint64_t)ep.kv_rows_per_slot;
  if (rows == 0 || rows >= (1ull << 31)) return cudaErrorInvalidValue;
  ep.kv_rows_total = (int32_t)rows;
  CUtensorMap mq, mk, mv, mkp, mvp;
  if (!encode_q(&mq, p.q, p.num_qo_heads, p.total_q, p.q_stride) ||
      !encode_rows(&mk, p.k_pool, rows) || !encode_rows(&mv, p.v_pool, rows))
    return cudaErrorInvalidValue;
  if (p.page_size >= 16) {
    if (!encode_pages(&mkp, p.k_pool, (uint64_t)ep.kv_rows_per_slot, (uint64_t)p.num_slots,
                      (uint64_t)p.pool_stride_bytes) ||
        !encode_pages(&mvp, p.v_pool, (uint64_t)ep.kv_rows_per_slot, (uint64_t)p.num_slots,
                      (uint64_t)p.pool_stride_bytes))
      return cudaErrorInvalidValue;
  } else {
    mkp = mk;   // not read: smaller pages take the gather4 path
    mvp = mv;
  }
  // persistent: one CTA per SM (the kernel's shared memory allows no more).
  // The instance that may take the key split, with a CTA on every SM, only
  // where the batch may have few items: its partial slots are there, fewer
  // than 4 items per CTA are possible (every extend token but one per
  // request sits in a 128-token tile, so at least H (total_q - num_reqs) /
  // 128 items), and, with max_kv_len given, 8 key tiles per CTA are.
  int64_t grid = (int64_t)device_sm_count();
  const int64_t items = max_tiles * p.num_kv_heads;
  const int64_t items_lo = (int64_t)p.num_kv_heads * ((p.total_q - p.num_reqs) / kBN);
  bool may_split = p.ext_o != nullptr && grid <= kExtMaxCtas && items_lo < 4 * grid;
  if (may_split && max_kv_len > 0 && items * ((max_kv_len + kBN - 1) / kBN) < 8 * grid)
    may_split = false;
  if (!may_split && grid > items) grid = items;
  if (may_split)
    extend_kernel<true><<<(unsigned)grid, kThreads, kSmem, s>>>(ep, mq, mk, mv, mkp, mvp);
  else
    extend_kernel<false><<<(unsigned)grid, kThreads, kSmem, s>>>(ep, mq, mk, mv, mkp, mvp);
  e = cudaGetLastError();
  if (e != cudaSuccess || !may_split) return e;
  // the split items' merge: one wave of CTAs over (listed item, 32-row block)
  return launch_k(ext_merge_kernel, dim3(kMergeCtasPerSm * (unsigned)grid), dim3(kMergeThreads), 0,
                  s, true, p);
}

}  // namespace msg

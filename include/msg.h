/*
 * msg.h -- C ABI of the GB300 (sm_103a) paged KV store and GQA paged attention.
 *
 * The library implements the attention step inside a mini-sglang style
 * Engine.forward_batch: the step's new K/V rows are scattered into a paged KV
 * pool (store_kv through out_loc), then GQA attention runs for a mixed batch of
 * decode and causal extend requests, reading K/V straight through the page
 * table.  Sources (page title, section):
 *   [CORE]   "核心数据结构：Req、Batch、Context" (mini-sglang handbook, core):
 *            sections "Req：请求的三个长度", "Batch：谁来填哪个字段", "Context".
 *   [ENGINE] "Engine 与采样器" (mini-sglang handbook, engine): sections
 *            "初始化的顺序" and "手工驱动引擎".
 *   [TINY]   "第 0 步：一个能跑的最小推理引擎": section "这份代码在做什么"
 *            (the attention operator: GQA by repeat_interleave, scale
 *            1/sqrt(D), causal mask at absolute positions).
 *   [TINY0]  the same page and section, its item "四个算子" (rmsnorm: a
 *            scale without mean or bias; rope: rotation of the first half
 *            against the second half of the head; q and k normed before the
 *            rotation, Qwen3).
 *   [WALK]   "Mini-SGLang 完整剖析": 4.4.3 (KV pool layout, store_kv),
 *            4.5.6 (one cos/sin cache of max_position x rotary_dim shared by
 *            every layer), 4.6.7 (AttentionLayer.forward: q_norm and k_norm
 *            in place, rotary in place, then store_kv and attention),
 *            4.6.4 (page table reading per backend: the dense per-request
 *            page-id table of the FlashAttention / TRT-LLM backends and the
 *            1-D ragged index list of FlashInfer), 4.6.5 (cu_seqlens),
 *            4.6.7 (store before attend), 4.9.4-4.9.5 (store kernel contract),
 *            4.8.5-4.8.6 (Sampler.prepare's sparse arguments, the sampler's
 *            four-way dispatch).
 *   [SAMPLE] "Engine 与采样器", section "采样器" (Sampler.prepare,
 *            Sampler.sample, sample_torch: softmax of logits / T, top-k, then
 *            top-p on the renormalised rest, one draw per row) and section
 *            "测试"; "Mini-SGLang 源码解析（四）" 14.2-14.5 (greedy batches
 *            take the argmax; MIN_T and MIN_P clamps).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Pointers are DEVICE pointers unless stated otherwise.  The caller allocates
 *   and owns every buffer (inputs, outputs, workspace).  The library allocates
 *   no device memory, never synchronises the stream, and enqueues all work on
 *   `stream` (a cudaStream_t passed as void*; NULL = legacy default stream).
 * - bf16 tensors are raw bf16 bit patterns.  Attention shapes are the Qwen3
 *   ones: head_dim 128, 16 query heads over 8 KV heads (GQA group of 2), or a
 *   tensor-parallel rank's slice of them split by KV head ([WALK] 4.5: 8, 4,
 *   2 or 1 KV heads with 2 query heads each, e.g. 8 q / 4 kv at tp = 2); other
 *   shapes return MSG_ERR_UNSUPPORTED.  store_kv accepts any row of
 *   num_kv_heads * head_dim bf16 values that is a multiple of 16 bytes.
 * - Pool layout ([WALK] 4.4.3): one K pool and one V pool per layer, each a
 *   [num_slots, num_kv_heads, head_dim] bf16 array whose consecutive slots are
 *   pool_row_stride elements apart.  slot = page * page_size + offset.
 * - page_table ([CORE] Context; [ENGINE] 初始化的顺序): int32 [rows,
 *   page_table_stride], token granular: entry [row, j] is the pool slot of
 *   token j of the request in that row.  With page_size P > 1 the caller
 *   guarantees that every page is P consecutive, P-aligned slots; the attention
 *   kernels then read one entry per page (the first token's) and add the offset
 *   ([WALK] 4.6.4, FlashAttention/TRT-LLM reading).
 * - Requests ([CORE] Req): cached_len[r] tokens already in the pool, extend_len[r]
 *   new tokens this step, device_len = cached_len + extend_len.  A request with
 *   extend_len == 1 is a decode request; extend_len >= 2 is an extend (prefill,
 *   chunked prefill or prefix-cache hit) request.  extend_len == 0 contributes
 *   nothing.  New tokens are concatenated in request order without padding;
 *   qo_indptr[r] is the first token of request r ([CORE] Batch).
 * - Alignment: every bf16 base pointer 16-byte aligned, every row stride a
 *   multiple of 8 elements; otherwise MSG_ERR_ALIGNMENT.
 * - Early start: the library's kernels are launched with programmatic
 *   stream serialization, so each may begin while the kernel before it on the
 *   stream is finishing; it waits for that kernel before touching anything it
 *   writes or reads.  The one exception is the decode kernel of a call with
 *   MSG_ATTN_REUSE_PLAN, which reads the plan (workspace) and the KV index
 *   before that wait, and in msg_paged_attention_store also the first K/V
 *   pool rows of its key range (up to three 32-key tiles per CTA, never a
 *   request's newest key, which comes from k_new / v_new): those must not be
 *   written by the kernel launched immediately before the call unless that
 *   kernel completes before it lets dependents start (every kernel that does
 *   not opt into programmatic launch, and every kernel of this library,
 *   qualifies: each lets dependents start only after its own wait).
 * - Errors: entry points return MSG_OK (0) or a negative status before
 *   enqueuing anything; no exception crosses the ABI, nothing aborts and no
 *   kernel traps.  Data-dependent problems found on the device (a slot outside
 *   [0, num_slots), a misaligned page, inconsistent lengths, a bounded wait that
 *   expired) are recorded in a device status block and the offending access is
 *   redirected to slot 0 or skipped; read the block with msg_read_device_status.
 */
#ifndef MSG_H
#define MSG_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Host-side status codes returned by every entry point. */
#define MSG_OK 0
#define MSG_ERR_INVALID_ARG -1    /* null pointer, negative size, bad stride    */
#define MSG_ERR_UNSUPPORTED -2    /* head_dim, head counts or page_size         */
#define MSG_ERR_ALIGNMENT -3      /* 16-byte alignment of a pointer or stride   */
#define MSG_ERR_WORKSPACE -4      /* workspace missing or too small             */
#define MSG_ERR_CUDA -5           /* a CUDA runtime call or launch failed       */
#define MSG_ERR_DEVICE_CHECK -6   /* msg_read_device_status found a device error */

/* Device-side error codes (first field of the device status block). */
#define MSG_DEV_OK 0
#define MSG_DEV_SLOT_OUT_OF_RANGE 1  /* out_loc or page-table slot not in [0, num_slots) */
#define MSG_DEV_PAGE_MISALIGNED 2    /* page_size > 1 and a page's first slot % page_size != 0 */
#define MSG_DEV_BAD_LENGTHS 3        /* negative length, a row shorter than device_len,
                                        or qo_indptr inconsistent with extend_len */
#define MSG_DEV_TIMEOUT 4            /* a bounded wait inside a kernel expired */
#define MSG_DEV_WRONG_PHASE 5        /* decode-only / extend-only flag contradicted */
#define MSG_DEV_BAD_POSITION 6       /* a position outside the rotary cache */
#define MSG_DEV_BAD_LOGIT 7          /* msg_sample: a NaN logit (+inf when sampling),
                                        or a row of -inf only */
#define MSG_DEV_BAD_SAMPLING 8       /* msg_sample: non-finite temperature, NaN top_p,
                                        or a uniform outside [0, 1) */
#define MSG_DEV_INTERNAL 9           /* msg_sample: an internal consistency check failed */

/* Element types of msg_sample's logits. */
#define MSG_DTYPE_F32 0
#define MSG_DTYPE_BF16 1

/* Flags of msg_paged_attention. */
#define MSG_ATTN_REUSE_PLAN 1u   /* workspace already holds the plan of this batch
                                    (made by msg_plan / msg_plan_ex, or by a
                                    previous attention call, with the same
                                    lengths and the same KV index); skip the
                                    plan kernel */
#define MSG_ATTN_DECODE_ONLY 2u  /* every request has extend_len <= 1: skip the
                                    extend kernel launch */
#define MSG_ATTN_EXTEND_ONLY 4u  /* no request has extend_len == 1: skip the
                                    decode kernel launch */

/*
 * KV index layouts ([WALK] 4.6.4).  The engine keeps one global, token
 * granular page table; the attention backends read it in one of three forms:
 *
 *   MSG_KV_TOKEN_TABLE  table[row, j] is the pool slot of token j (the global
 *                       table itself).  With page_size P > 1 only the entry of
 *                       each page's first token is read (j rounded down to a
 *                       multiple of P) and must be P-aligned; slot = entry +
 *                       j % P.  This is what msg_plan / msg_paged_attention use.
 *   MSG_KV_PAGE_TABLE   table[row, j / P] is a page id (FlashAttention and
 *                       TRT-LLM: every P-th column of the global table divided
 *                       by P, a dense [requests, ceil(max_len / P)] table);
 *                       slot = id * P + j % P.
 *   MSG_KV_RAGGED       table[indptr[r] + j / P] is a page id (FlashInfer: the
 *                       per-request lists concatenated in one 1-D array with
 *                       int32 offsets indptr [num_reqs + 1]; with P = 1 the
 *                       entries are slots); slot = id * P + j % P.
 *
 * Rows of the two table forms are req_rows[r] (NULL = r) and table_stride
 * entries apart; the ragged form ignores req_rows and table_stride.
 * table_len (entries of `table`, or -1 if unknown) lets the plan reject rows
 * or offsets that would leave the array (MSG_DEV_BAD_LENGTHS).  A request of
 * device_len n needs n entries in its row (token table) or ceil(n / P)
 * (page-id forms); fewer is MSG_DEV_BAD_LENGTHS, and an entry that names a
 * slot outside the pool MSG_DEV_SLOT_OUT_OF_RANGE.
 */
#define MSG_KV_TOKEN_TABLE 0
#define MSG_KV_PAGE_TABLE 1
#define MSG_KV_RAGGED 2

typedef struct msg_kv_index {
  int32_t kind;              /* MSG_KV_* */
  int32_t page_size;         /* power of two in [1, 128] */
  const int32_t *table;      /* device int32 entries */
  int64_t table_stride;      /* entries between rows (table forms) */
  int64_t table_len;         /* entries in `table`, or -1 */
  const int32_t *req_rows;   /* device int32 [num_reqs] or NULL (table forms) */
  const int32_t *indptr;     /* device int32 [num_reqs + 1] (ragged form) */
} msg_kv_index;

/* Size in bytes of the device status block (4 x int32: code, request index,
 * low and high 32 bits of the offending value).  It sits at the start of the
 * workspace; a standalone block may be passed to msg_store_kv. */
#define MSG_STATUS_BYTES 16

/* Human-readable text for a host status code (static storage). */
const char *msg_status_string(int status);

/* ABI version (major * 10000 + minor * 100 + patch). */
int msg_version(void);

/*
 * Workspace bytes needed by msg_plan and msg_paged_attention for batches of at
 * most max_reqs requests and max_total_q new tokens, with num_qo_heads query
 * heads of head_dim.  The workspace holds the status block, the plan (per
 * request lengths, decode partition, extend tile list and list of split
 * extend items, merge counters) and the split-KV partial results, then
 * ~42 MB of partial slots for the extend key split: an extend batch of fewer
 * than 4 work items (query tile x KV head) per SM, whose items hold at least
 * 8 key tiles of 128 keys per SM (e.g. a chunked-prefill tile over a long
 * cached prefix), has its key tiles split evenly over every SM and the split
 * items' partial results merged by a second kernel.  A workspace that holds
 * everything but those slots is accepted too (the no-alloc entry point's
 * scratch is one): such batches then take their items whole.  Returns 0 on
 * invalid arguments.  Any workspace of at least this size serves every
 * smaller batch.
 */
size_t msg_workspace_size(int32_t max_reqs, int64_t max_total_q,
                          int32_t num_qo_heads, int32_t head_dim);

/*
 * The workspace size under the boundary's planned name: msg_workspace_size for
 * batches of at most max_reqs requests and max_total_q new tokens.  The
 * split-KV split count is the library's own choice (at most two partial
 * results per decode CTA, whose number it caps to what this size holds), so
 * every max_splits >= 1 gives the same size; max_splits < 1 or any invalid
 * argument returns 0.
 */
size_t msg_paged_attention_workspace_size(int32_t max_reqs, int64_t max_total_q,
                                          int32_t num_qo_heads, int32_t head_dim,
                                          int32_t max_splits);

/*
 * a1. Per-batch metadata prep ([CORE] Batch table; [ENGINE] 手工驱动引擎;
 * [WALK] 4.6.5).  From per-request (req_rows, cached_len, extend_len):
 *   qo_indptr[r+1] = qo_indptr[r] + extend_len[r]          (qo_indptr[0] = 0)
 *   positions[qo_indptr[r] + i] = cached_len[r] + i          (i < extend_len[r])
 *   out_loc[qo_indptr[r] + i]   = page_table[row_r, cached_len[r] + i]
 * and writes the attention plan (decode partition, extend tile list, zeroed
 * merge counters) into `workspace`, so msg_paged_attention may pass
 * MSG_ATTN_REUSE_PLAN for this batch.
 *
 * page_table      int32 [*, page_table_stride]; rows read: req_rows[r].
 * req_rows        int32 [num_reqs] page-table row per request, or NULL = r.
 * cached_len      int32 [num_reqs];  extend_len  int32 [num_reqs].
 * total_q         host value: sum of extend_len (sizes the output arrays and
 *                 the launch; a mismatch is reported as MSG_DEV_BAD_LENGTHS).
 * num_slots       pool rows, for the range check of out_loc.
 * qo_indptr_out   int32 [num_reqs + 1] or NULL.
 * out_loc_out     [total_q] int32 (out_loc_is_int64 = 0) or int64 (= 1), or NULL.
 * positions_out   int32 [total_q] or NULL.
 * workspace       device buffer of workspace_bytes >= msg_workspace_size(...).
 * Errors: MSG_ERR_INVALID_ARG, MSG_ERR_WORKSPACE, MSG_ERR_CUDA.
 */
int msg_plan(const int32_t *page_table, int64_t page_table_stride,
             const int32_t *req_rows, const int32_t *cached_len,
             const int32_t *extend_len, int32_t num_reqs, int64_t total_q,
             int64_t num_slots, int32_t *qo_indptr_out, void *out_loc_out,
             int32_t out_loc_is_int64, int32_t *positions_out, void *workspace,
             size_t workspace_bytes, void *stream);

/*
 * a1 with any index layout: as msg_plan, but the slots of out_loc are read
 * through `kv` (a host pointer to the descriptor; its arrays are device
 * arrays), including its page size.  msg_plan(page_table, stride, req_rows,
 * ...) equals msg_plan_ex with {MSG_KV_TOKEN_TABLE, page_size 1, page_table,
 * stride, -1, req_rows, NULL}.
 * Errors: as msg_plan, plus MSG_ERR_UNSUPPORTED for an unknown kind or a page
 * size that is not a power of two in [1, 128].
 */
int msg_plan_ex(const msg_kv_index *kv, const int32_t *cached_len,
                const int32_t *extend_len, int32_t num_reqs, int64_t total_q,
                int64_t num_slots, int32_t *qo_indptr_out, void *out_loc_out,
                int32_t out_loc_is_int64, int32_t *positions_out, void *workspace,
                size_t workspace_bytes, void *stream);

/*
 * a1, backend metadata ([WALK] 4.6.4): the per-request page-id forms of the
 * global token table for the requests of a batch.
 *   kind MSG_KV_PAGE_TABLE: out_table[r, i] = page_table[row_r, i * P] / P for
 *       i < ceil(device_len_r / P); out_stride entries per row (>= the
 *       longest row); out_indptr unused (NULL).
 *   kind MSG_KV_RAGGED: out_indptr[0] = 0, out_indptr[r + 1] = out_indptr[r] +
 *       ceil(device_len_r / P); out_table[out_indptr[r] + i] = page_table[row_r,
 *       i * P] / P (the slots themselves when P = 1).  out_capacity bounds the
 *       entries written; the total needed is reported by MSG_DEV_BAD_LENGTHS
 *       when it does not fit (nothing is written past out_capacity).
 * page_table is the global token-granular table (MSG_KV_TOKEN_TABLE form);
 * device_len_r = cached_len[r] + extend_len[r].  The result serves
 * msg_plan_ex / msg_paged_attention_ex with the same page size.  A page-start
 * slot that is negative or not a multiple of P is recorded as
 * MSG_DEV_SLOT_OUT_OF_RANGE / MSG_DEV_PAGE_MISALIGNED in dev_status (may be
 * NULL) and written as -1.
 * Errors: MSG_ERR_INVALID_ARG, MSG_ERR_UNSUPPORTED, MSG_ERR_CUDA.
 */
int msg_build_kv_index(int32_t kind, int32_t page_size, const int32_t *page_table,
                       int64_t page_table_stride, const int32_t *req_rows,
                       const int32_t *cached_len, const int32_t *extend_len,
                       int32_t num_reqs, int32_t *out_table, int64_t out_stride,
                       int64_t out_capacity, int32_t *out_indptr, int32_t *dev_status,
                       void *stream);

/*
 * a2. store_kv ([WALK] 4.4.3, 4.6.7 step 1; shape contract of 4.9.4):
 *   k_pool[out_loc[i], :, :] = k[i, :, :];  v_pool[out_loc[i], :, :] = v[i, :, :]
 * for i < num_tokens, bit-exact copies of num_kv_heads * head_dim bf16 values.
 *
 * k, v            bf16 [num_tokens, num_kv_heads, head_dim], rows kv_row_stride
 *                 elements apart (heads contiguous inside a row).
 * k_pool, v_pool  bf16 pools, rows pool_row_stride elements apart, num_slots rows.
 * out_loc         [num_tokens] int32 (out_loc_is_int64 = 0) or int64 (= 1).
 *                 Only padding may repeat a slot (the dummy slot); which
 *                 duplicate lands is unspecified.
 * dev_status      MSG_STATUS_BYTES device block or NULL.  A slot outside
 *                 [0, num_slots) is recorded there and its row is not written.
 * Must be enqueued before msg_paged_attention on the same stream: attention
 * reads the step's own K/V from the pool.  num_tokens == 0 is a no-op.
 * Errors: MSG_ERR_INVALID_ARG, MSG_ERR_UNSUPPORTED, MSG_ERR_ALIGNMENT, MSG_ERR_CUDA.
 */
int msg_store_kv(const void *k, const void *v, int64_t kv_row_stride,
                 void *k_pool, void *v_pool, int64_t pool_row_stride,
                 int64_t num_slots, const void *out_loc, int32_t out_loc_is_int64,
                 int64_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                 int32_t *dev_status, void *stream);

/*
 * a3-a6. GQA paged attention for a mixed batch ([TINY] attention operator;
 * [WALK] 4.6.4, 4.6.7 step 2).  For new token i of request r (absolute position
 * p = cached_len[r] + i) and query head h with kv head g = h / 2:
 *   out[qo_indptr[r] + i, h, :] = sum_{j <= p} softmax_j(scale * q.K_j[g]) V_j[g]
 * where K_j, V_j are read from the pools at the slot the page table gives for
 * token j of row req_rows[r].  Decode requests (extend_len == 1) run a split-KV,
 * bandwidth-bound kernel whose partial results are merged by log-sum-exp in the
 * workspace; extend requests run a tensor-core kernel tiled over query chunks
 * with the causal mask offset by cached_len.
 *
 * q               bf16 [total_q, num_qo_heads, head_dim], rows q_row_stride apart.
 * k_pool, v_pool  as in msg_store_kv; the step's K/V must already be stored.
 * qo_indptr       int32 [num_reqs + 1] (e.g. from msg_plan), consistent with
 *                 extend_len.
 * max_kv_len      host hint: an upper bound of device_len, or 0 if unknown; it
 *                 only sizes the decode launch for tiny batches.
 * page_size       power of two in [1, 128]; see the page_table convention.
 * scale           softmax scale (1/sqrt(head_dim) for the configs here).
 * out             bf16 [total_q, num_qo_heads, head_dim], contiguous.
 * workspace       >= msg_workspace_size(num_reqs, total_q, num_qo_heads, head_dim).
 * flags           MSG_ATTN_* bits.
 * Consecutive calls that share one workspace must be ordered on one stream.
 * Errors: MSG_ERR_INVALID_ARG, MSG_ERR_UNSUPPORTED, MSG_ERR_ALIGNMENT,
 *         MSG_ERR_WORKSPACE, MSG_ERR_CUDA.
 */
int msg_paged_attention(const void *q, int64_t q_row_stride, const void *k_pool,
                        const void *v_pool, int64_t pool_row_stride,
                        int64_t num_slots, const int32_t *page_table,
                        int64_t page_table_stride, const int32_t *req_rows,
                        const int32_t *cached_len, const int32_t *extend_len,
                        const int32_t *qo_indptr, int32_t num_reqs,
                        int64_t total_q, int32_t max_kv_len, int32_t page_size,
                        int32_t num_qo_heads, int32_t num_kv_heads,
                        int32_t head_dim, float scale, void *out,
                        void *workspace, size_t workspace_bytes, uint32_t flags,
                        void *stream);

/*
 * a2 + a3/a4 fused for a decode step ([WALK] 4.6.7 steps 1 and 2: store_kv, then
 * attention): a decode-only batch (flags must include MSG_ATTN_DECODE_ONLY)
 * whose new K / V rows have not been stored yet.  Equivalent to
 *   msg_store_kv(k_new, v_new, kv_row_stride, k_pool, v_pool, ..., out_loc, ...)
 *   msg_paged_attention(q, ..., k_pool, v_pool, ...)
 * with out_loc[qo_indptr[r]] = the slot of token cached_len[r] of request r's
 * row (the slot msg_plan writes to out_loc): the decode kernel gathers each
 * request's newest key from k_new / v_new row qo_indptr[r] instead of the
 * pool, and the CTA that owns that key writes the two rows to its pool slot.
 * Outputs and pools are bit-identical to the two calls; one kernel launch
 * instead of two.
 *
 * k_new, v_new    bf16 [total_q, num_kv_heads, head_dim], rows kv_row_stride
 *                 elements apart (16-byte aligned rows), in q's row order.
 * k_pool, v_pool  written at the new tokens' slots (the only writes).
 * Other arguments as msg_paged_attention.  A slot outside the pool is
 * recorded in the workspace's status block and not written.
 * Errors: as msg_paged_attention; MSG_ERR_INVALID_ARG also without
 *         MSG_ATTN_DECODE_ONLY or with a NULL k_new / v_new.
 */
int msg_paged_attention_store(const void *q, int64_t q_row_stride, const void *k_new,
                              const void *v_new, int64_t kv_row_stride, void *k_pool,
                              void *v_pool, int64_t pool_row_stride, int64_t num_slots,
                              const int32_t *page_table, int64_t page_table_stride,
                              const int32_t *req_rows, const int32_t *cached_len,
                              const int32_t *extend_len, const int32_t *qo_indptr,
                              int32_t num_reqs, int64_t total_q, int32_t max_kv_len,
                              int32_t page_size, int32_t num_qo_heads, int32_t num_kv_heads,
                              int32_t head_dim, float scale, void *out, void *workspace,
                              size_t workspace_bytes, uint32_t flags, void *stream);

/*
 * a3-a6 with any index layout: as msg_paged_attention, with the slots of each
 * request's keys read through `kv` (host pointer to the descriptor, device
 * arrays; its page_size replaces the page_size argument).
 * msg_paged_attention(..., page_table, stride, req_rows, ..., page_size, ...)
 * equals msg_paged_attention_ex with {MSG_KV_TOKEN_TABLE, page_size,
 * page_table, stride, -1, req_rows, NULL}.
 * Errors: as msg_paged_attention.
 */
int msg_paged_attention_ex(const void *q, int64_t q_row_stride, const void *k_pool,
                           const void *v_pool, int64_t pool_row_stride, int64_t num_slots,
                           const msg_kv_index *kv, const int32_t *cached_len,
                           const int32_t *extend_len, const int32_t *qo_indptr,
                           int32_t num_reqs, int64_t total_q, int32_t max_kv_len,
                           int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                           float scale, void *out, void *workspace, size_t workspace_bytes,
                           uint32_t flags, void *stream);

/*
 * Rotary cos/sin cache ([WALK] 4.5.6; [TINY0] rope): fp32 [max_pos, head_dim],
 * row p = cos(a_p,0 .. a_p,D/2-1) followed by sin(a_p,0 .. a_p,D/2-1) with
 *   inv_freq_i = theta^(-2i / D) rounded once to fp32,
 *   a_p,i      = fp32(p) * inv_freq_i in fp32 (one rounding),
 *   cos, sin   of that fp32 angle, rounded once to fp32.
 * Built once per model on the device (double-precision pow / cos / sin), read
 * by msg_qk_norm_rope_store.  head_dim even, theta > 0, max_pos >= 1.
 * Errors: MSG_ERR_INVALID_ARG, MSG_ERR_CUDA.
 */
int msg_rope_cos_sin_cache(double theta, int32_t head_dim, int64_t max_pos, float *out,
                           void *stream);

/*
 * Fused attention prologue ([WALK] 4.6.7; [TINY0] rmsnorm, rope): for token t
 * of num_tokens, with qkv row t = [q (Hq x D) | k (Hkv x D) | v (Hkv x D)] bf16
 * as the QKV projection writes it, and p = positions[t]:
 *   q_out[t, h, :]             = rope(rmsnorm(q[t, h, :], q_norm_w), p)
 *   k_pool[out_loc[t], g, :]   = rope(rmsnorm(k[t, g, :], k_norm_w), p)
 *   v_pool[out_loc[t], g, :]   = v[t, g, :]                      (bit copy)
 * rmsnorm(x, w)_d = w_d * x_d / sqrt(mean_d(x_d^2) + eps);
 * rope(x, p): x1 = x[0 : D/2], x2 = x[D/2 : D], c = cos_sin[p, 0 : D/2],
 *   s = cos_sin[p, D/2 : D]; result = [x1 c - x2 s, x1 s + x2 c].
 * Arithmetic in fp32 from the bf16 inputs, one round-to-nearest-even to bf16
 * per output.  This is store_kv with the norm and the rotation of K fused in:
 * the step's K is written to the pool already rotated, and Q lands in q_out
 * ready for msg_paged_attention (q_out may be qkv itself, same row stride: the
 * q part is then rotated in place).
 *
 * qkv         bf16 rows of (Hq + 2 Hkv) x D values, qkv_row_stride elements apart.
 * positions   int32 [num_tokens] (from msg_plan), each in [0, max_pos).
 * q_norm_w, k_norm_w  bf16 [D].
 * cos_sin     fp32 [max_pos, D] from msg_rope_cos_sin_cache.
 * q_out       bf16 [num_tokens, Hq, D], rows q_out_row_stride elements apart.
 * k_pool, v_pool, pool_row_stride, num_slots, out_loc, out_loc_is_int64: as
 *             msg_store_kv (the slot of token t is out_loc[t]).
 * dev_status  MSG_STATUS_BYTES block or NULL: a slot outside the pool or a
 *             position outside the cache is recorded, and that token's K/V
 *             (resp. its q and K/V) are not written.
 * Supported: head_dim 128 (other shapes MSG_ERR_UNSUPPORTED); any head counts.
 * Errors: MSG_ERR_INVALID_ARG, MSG_ERR_UNSUPPORTED, MSG_ERR_ALIGNMENT, MSG_ERR_CUDA.
 */
int msg_qk_norm_rope_store(const void *qkv, int64_t qkv_row_stride, int64_t num_tokens,
                           const int32_t *positions, const void *q_norm_w,
                           const void *k_norm_w, float eps, const float *cos_sin,
                           int64_t max_pos, void *q_out, int64_t q_out_row_stride,
                           void *k_pool, void *v_pool, int64_t pool_row_stride,
                           int64_t num_slots, const void *out_loc, int32_t out_loc_is_int64,
                           int32_t num_qo_heads, int32_t num_kv_heads, int32_t head_dim,
                           int32_t *dev_status, void *stream);

/*
 * Copy the device status block (a workspace, or a standalone
 * MSG_STATUS_BYTES block) to the host array host_out[4], synchronising
 * `stream`.  Returns MSG_OK if no device error was recorded,
 * MSG_ERR_DEVICE_CHECK if one was (host_out[0] holds its MSG_DEV_* code),
 * MSG_ERR_CUDA if the copy failed.
 */
int msg_read_device_status(const void *dev_status, int32_t *host_out, void *stream);

/*
 * The device error of a workspace (or standalone status block) under the
 * boundary's planned name: synchronises `stream` like msg_read_device_status
 * and returns the recorded MSG_DEV_* code (MSG_DEV_OK = 0 when none), or a
 * negative host status (MSG_ERR_INVALID_ARG for NULL, MSG_ERR_CUDA if the
 * copy failed).
 */
int msg_get_device_error(const void *workspace, void *stream);

/* Zero a device status block (asynchronously, on `stream`). */
int msg_clear_device_status(void *dev_status, void *stream);

/*
 * Paged attention without a caller-allocated workspace.  (No counterpart on
 * the pages: this is a convenience of this library.)
 *
 * Identical to msg_paged_attention, except that its scratch (plan, split-KV
 * partial results, merge counters, status block) lives in one fixed array of
 * MSG_NOALLOC_SCRATCH_BYTES inside the library rather than in a workspace the
 * caller allocates.  It exists for callers that cannot allocate device memory:
 * code running under a framework whose allocator owns all device memory and
 * forbids raw cudaMalloc, C or plugin callers with no device allocator at hand,
 * and latency-critical loops that cannot pay for cudaMalloc / cudaFree (which
 * may synchronise the device).  The caller still passes its inputs and outputs.
 *
 * - The array is a file-scope device object: every GPU that loads the library
 *   holds MSG_NOALLOC_SCRATCH_BYTES until the process exits.  That fits every
 *   batch of up to 1024 requests and 65536 new tokens at 16 query heads of
 *   head_dim 128; a batch whose msg_workspace_size(...) exceeds it is rejected
 *   with MSG_ERR_WORKSPACE before anything is enqueued.
 * - The first call on a device looks up the array's device address (with that
 *   device current) and caches it; make that first call before any stream
 *   capture.
 * - Every call shares the one array and it keeps the last call's contents: the
 *   status block is cleared at the start of each call, and MSG_ATTN_REUSE_PLAN
 *   reuses the plan left by the last successful call of this entry point on
 *   this device that built one (called without MSG_ATTN_REUSE_PLAN).  The
 *   library remembers that call's (num_reqs, total_q) on the host and rejects
 *   MSG_ATTN_REUSE_PLAN with MSG_ERR_INVALID_ARG when no plan was built yet
 *   or the batch size differs (the plan's place in the array depends on it);
 *   that the lengths and index are the same is, as for msg_paged_attention,
 *   the caller's promise.  Calls that overlap on the GPU (different streams,
 *   or unordered threads) race on the array and must not be issued.
 * - dev_status: optional MSG_STATUS_BYTES device block, or NULL.  When the
 *   call returns MSG_OK it receives this call's device status (copied at the
 *   end of the call; zeroed for an empty batch).  When the call returns an
 *   error it is not written.
 * - Nothing is allocated: no cudaMalloc, cudaFree or allocating library call.
 * Errors: as msg_paged_attention; MSG_ERR_INVALID_ARG also for
 *         MSG_ATTN_REUSE_PLAN without a plan of this batch size.
 */
#define MSG_NOALLOC_SCRATCH_BYTES (9u << 20)

int msg_paged_attention_noalloc(const void *q, int64_t q_row_stride, const void *k_pool,
                                const void *v_pool, int64_t pool_row_stride,
                                int64_t num_slots, const int32_t *page_table,
                                int64_t page_table_stride, const int32_t *req_rows,
                                const int32_t *cached_len, const int32_t *extend_len,
                                const int32_t *qo_indptr, int32_t num_reqs,
                                int64_t total_q, int32_t max_kv_len, int32_t page_size,
                                int32_t num_qo_heads, int32_t num_kv_heads,
                                int32_t head_dim, float scale, void *out, uint32_t flags,
                                int32_t *dev_status, void *stream);

/*
 * Batched sampler: the next token of every row of logits [SAMPLE].
 *
 * Per row r (B rows of V logits):
 *   temperatures == NULL: every request is greedy (Sampler.prepare returned
 *     no temperatures); token = the first index of the row's maximum
 *     (torch.argmax).  top_k, top_p and uniforms are ignored and may be NULL.
 *   otherwise, sample_torch's steps in order:
 *     T = max(temperatures[r], 1e-6)   (a greedy request of a mixed batch
 *                                       passes T <= 0 and gets MIN_T);
 *     p = softmax(logits[r] / T);
 *     top-k (top_k != NULL and 1 <= top_k[r] < V): keep the top_k[r] most
 *       likely tokens, equal probabilities in increasing token index;
 *     top-p (top_p != NULL and clamp(top_p[r], 1e-6, 1) < 1): renormalise
 *       what is left and keep a token only while the mass ranked ahead of it
 *       is below top_p (the most likely token always stays);
 *     draw: token = the smallest index i, in vocabulary order, whose
 *       cumulative kept mass exceeds uniforms[r] times the kept total (the
 *       inverse CDF; uniforms[r] in [0, 1) comes from the caller's generator).
 *   The kernel computes p in fp32 as 2^((l - max) * log2(e) / T) and sums in
 *   a fixed order, so a row's token is deterministic.  It differs from an
 *   exact (fp64) evaluation only when the uniform or a cut falls within about
 *   1e-5 (relative to the kept mass) of a boundary between two tokens.
 *
 * Arguments:
 *   logits             device, B rows of V elements of logits_dtype
 *                      (MSG_DTYPE_F32 or MSG_DTYPE_BF16; bf16 values are used
 *                      exactly, as logits.float() would); rows
 *                      logits_row_stride elements apart (>= V, any value); the
 *                      pointer aligned to the element size (MSG_ERR_ALIGNMENT).
 *                      Read only.
 *   batch, vocab       B >= 0, 1 <= V <= 425984 (larger V: MSG_ERR_UNSUPPORTED).
 *   temperatures       device float32 [B] or NULL (see above).
 *   top_k              device int32 [B] or NULL (values < 1 or >= V: no cut).
 *   top_p              device float32 [B] or NULL (clamped to [1e-6, 1]).
 *   uniforms           device float32 [B], required with temperatures.
 *   tokens_out         device int32 [B]: the tokens; -1 for a row that failed
 *                      a device check.
 *   workspace          device scratch of msg_sample_workspace_size(B, V) bytes
 *                      or more, 16-byte aligned (MSG_ERR_WORKSPACE if missing
 *                      or smaller; MSG_ERR_ALIGNMENT if misaligned); owned by
 *                      the caller, its contents are not kept between calls.
 *   dev_status         MSG_STATUS_BYTES device block or NULL: a NaN logit, a
 *                      +inf logit when sampling (softmax is undefined), or a
 *                      row whose every logit is -inf (MSG_DEV_BAD_LOGIT); a
 *                      non-finite temperature, NaN top_p or a uniform outside
 *                      [0, 1) (MSG_DEV_BAD_SAMPLING).  -inf logits are tokens
 *                      of probability zero; a greedy row takes a +inf logit as
 *                      its maximum.
 *   stream             cudaStream_t (NULL: the legacy default stream).
 * With temperatures: two kernel launches on `stream`, a scan that reads every
 * logit from HBM once (many CTAs per row) and a row kernel (one CTA per row,
 * started early by programmatic dependent launch) that re-reads at most a few
 * chunks of a row, or, for a top-p boundary deep inside a flat distribution,
 * the row a few times (from L2 when the batch fits there).  Without them (every
 * row greedy): one launch, a CTA per row reading it once; the workspace is
 * still checked but not used.
 * Errors: MSG_ERR_INVALID_ARG, MSG_ERR_UNSUPPORTED, MSG_ERR_ALIGNMENT,
 *         MSG_ERR_WORKSPACE, MSG_ERR_CUDA.
 */
int msg_sample(const void *logits, int32_t logits_dtype, int64_t logits_row_stride,
               int32_t batch, int32_t vocab, const float *temperatures,
               const int32_t *top_k, const float *top_p, const float *uniforms,
               int32_t *tokens_out, void *workspace, size_t workspace_bytes,
               int32_t *dev_status, void *stream);

/*
 * Bytes of msg_sample's workspace for `batch` rows of `vocab` logits (per
 * row: each 256-logit chunk's maximum and mass, a sparse sample, and the scan
 * parts' finiteness flags; about 14.0 KB per row at V = 151,936).  0 for an
 * invalid or unsupported size.  Host only.
 */
size_t msg_sample_workspace_size(int32_t batch, int32_t vocab);


#ifdef __cplusplus
}
#endif
#endif /* MSG_H */

/*
 * mla.h - C ABI of the GB300 (sm_103a) MLA prefill attention library.
 *
 * What it computes. Causal prefill attention for DeepSeek-style multi-head
 * latent attention (MLA) in weight-absorbed form, as served for GLM-5.3 on the
 * pages "More throughput from fewer GPUs: profiling and fixing GLM-5.3
 * prefill on NVIDIA B300" (section System architecture: one latent vector per
 * token shared by all heads; FP8 KV cache) and "GLM-5.3-Optimierungen, Teil 2:
 * PCP, DCP und Hybrid HiSparse auf 16 H200s" (section "Warum nicht TP oder
 * DP?": 64 heads share the latent row, an indexer scores every earlier token
 * and keeps 2,048; section Ausprobieren: sparse MLA runs as MQA; footnote 1:
 * QK over 576 dims, PV over 512; footnote 3: indexer keys are 128 FP8 values
 * and a 4-byte scale).
 *
 * Data layout (all row-major, all device memory unless named *_host):
 *   query rows     q       bf16  [Tq, H, 576]   dims 0..511 latent, 512..575 RoPE
 *                                                (RoPE already applied)
 *   latent cache   kv      e4m3  [num_blocks, 256, 576]   one row per token
 *   cache scales   kv_scale f32  [num_blocks, 256]        K_s = kv_scale_s * dec(kv_s)
 *   output         out     bf16  [Tq, H, 512]
 *   log-sum-exp    lse     f32   [Tq, H]   natural log, optional (NULL = skip)
 *   indexer q      qi      e4m3  [Tq, 64, 128]
 *   indexer w      w       f32   row t at w + t*w_token_stride (64 values)
 *   indexer keys   ki      e4m3  [num_blocks, 256, 128]
 *   indexer scale  ki_scale f32  [num_blocks, 256]
 *   top-k indices  idx     int32 [Tq, topk]  positions within the sequence,
 *                                            distinct, -1 padding at the end
 * Position s of sequence b lives at page block_table[b*max_blocks_per_seq +
 * s/256], slot s%256. New token i of sequence b is at position prefix_lens[b]
 * + i and attends to positions 0..prefix_lens[b]+i (itself included); its
 * cache row must already be written.
 *
 * Ownership. The caller owns every buffer, workspace included. The library
 * allocates no device or host memory, never synchronises, and enqueues all
 * work asynchronously on the given stream. Host mirrors (cu_seqlens_q_host,
 * prefix_lens_host) are read during the call only.
 *
 * Errors. Arguments are validated on the host before any launch; a failing
 * check returns a status and launches nothing. mla_last_error() then returns
 * a message (thread-local, valid until the thread's next call). Data that only
 * the device sees (a page id outside [0, num_blocks), a sparse index outside
 * [-1, position]) never traps: the kernel skips the offending key and ORs a
 * MLA_DEVERR_* bit into *dev_err (if dev_err is not NULL); the caller reads it
 * after synchronising. A kernel launch failure returns MLA_ERR_CUDA.
 */
#ifndef MLA_H_
#define MLA_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MLA_OK = 0,
    MLA_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, bad size or shape */
    MLA_ERR_UNSUPPORTED = 2,   /* valid but not implemented (e.g. H not in {16,32,64,128}) */
    MLA_ERR_CUDA = 3,          /* a CUDA call or kernel launch failed */
    MLA_ERR_WORKSPACE = 4      /* workspace NULL or smaller than mla_workspace_size() */
} mla_status_t;

/* Bits ORed into *dev_err by the kernels. */
#define MLA_DEVERR_BAD_PAGE 1   /* block table entry outside [0, num_blocks) */
#define MLA_DEVERR_BAD_INDEX 2  /* sparse index outside [-1, position of the query] */
#define MLA_DEVERR_TIMEOUT 4    /* a bounded wait inside a kernel gave up; that CTA's rows are not written */
#define MLA_DEVERR_INTERNAL 8   /* a kernel invariant failed (a library bug); the row is -1 filled */
#define MLA_DEVERR_SEQ_MISMATCH 16  /* the device cu_seqlens_q disagrees with its host mirror: no row at or
                                       past the host's count is read or written; a unit of work (a pair of
                                       row tiles, a group of indexer tokens) that either side does not
                                       count in full is skipped whole, leaving its rows unwritten */

typedef enum {
    MLA_OP_DENSE = 0,
    MLA_OP_INDEXER = 1,
    MLA_OP_SPARSE = 2,
    MLA_OP_DENSE_HOST = 3,  /* mla_prefill_dense_host, any chunk count */
    MLA_OP_MHA = 4,         /* mla_prefill_mha */
    MLA_OP_DENSE_DS = 5     /* mla_prefill_dense_ds */
} mla_op_t;

/* Ragged batch of sequences over one paged cache (256-token pages). */
typedef struct {
    int32_t batch;                      /* B >= 1 */
    const int32_t *cu_seqlens_q;        /* device [B+1], cu[0] = 0, non-decreasing */
    const int32_t *cu_seqlens_q_host;   /* host mirror of cu_seqlens_q */
    const int32_t *prefix_lens;         /* device [B], cached tokens before the new ones */
    const int32_t *prefix_lens_host;    /* host mirror of prefix_lens */
    const int32_t *block_table;         /* device [B, max_blocks_per_seq] page ids */
    int32_t max_blocks_per_seq;         /* >= ceil((prefix+new)/256) for every sequence */
    int32_t num_blocks;                 /* pages in the cache */
} mla_seqs_t;

/* Bytes of workspace the op needs for this batch (0 means none is needed and
 * workspace may be NULL). Returns 0 on invalid arguments as well; the op call
 * itself reports those. */
size_t mla_workspace_size(mla_op_t op, const mla_seqs_t *seqs, int32_t num_heads, int32_t topk);

/* Dense causal MLA prefill, weight-absorbed (MQA over the shared latent row).
 * For each new token t (position p) and head h:
 *   logit_s = sm_scale * sum_{d<576} q[t,h,d] * kv_scale_s * dec(kv_s[d]),  s = 0..p
 *   out[t,h,:] = sum_s softmax(logit)_s * kv_scale_s * dec(kv_s[0:512])
 *   lse[t,h]   = ln sum_s exp(logit_s)
 * (More throughput from fewer GPUs, section System architecture; GLM-5.3
 * Teil 2, footnote 1.) Work is scheduled by pairing query tile i with tile
 * n-1-i of the same sequence, the load-balanced chunk pairing of GLM-5.3 Teil
 * 2, section "PCP: teile die Token, nicht die Köpfe", applied across CTAs.
 * num_heads in {16, 32, 64, 128}. Pointers: q, out 16-byte aligned; kv
 * 16-byte aligned. workspace: mla_workspace_size(MLA_OP_DENSE, ...) bytes,
 * 16-byte aligned. */
mla_status_t mla_prefill_dense(const mla_seqs_t *seqs, const void *q_bf16, int32_t num_heads,
                               const uint8_t *kv_e4m3, const float *kv_scale, float sm_scale,
                               void *out_bf16, float *lse, void *workspace, size_t workspace_bytes,
                               int32_t *dev_err, cudaStream_t stream);

/* Indexer score and top-k selection (GLM-5.3 Teil 2, section "Warum nicht TP
 * oder DP?": score every earlier token, keep 2,048; footnote 3: 128 FP8 values
 * and a 4-byte scale per key). For new token t at position p:
 *   score(t,s) = ki_scale_s * sum_{h<64} w[t,h] * max(0, sum_{d<128} dec(qi[t,h,d]) * dec(ki_s[d]))
 * for s = 0..p; idx[t,:] = the min(topk, p+1) positions with the largest
 * scores, ties going to the lower position. A row with p+1 <= topk holds
 * 0..p and then -1; a longer row holds its topk distinct positions in an
 * order that is fixed for given inputs (not necessarily ascending). Scores
 * are accumulated in fp32 (exact when q and k hold small integers).
 * w_token_stride 0 shares one 64-value row among all
 * tokens; otherwise it is a multiple of 4. topk in [1, 2048]. qi, ki, w and
 * ki_scale 16-byte aligned. The scores never leave the GPU's on-chip memory:
 * one CTA streams every key a group of three tokens can see and keeps each
 * token's candidates in shared memory (a threshold set from a sample of the
 * keys decides which enter; a group the fast path cannot finish exactly is
 * redone by an exact streaming pass). workspace: mla_workspace_size(
 * MLA_OP_INDEXER, ...) bytes: a 16-byte work item and a 4-byte flag per group
 * of three tokens, whatever the context length. */
mla_status_t mla_indexer_topk(const mla_seqs_t *seqs, const uint8_t *qi_e4m3, const float *w,
                              int64_t w_token_stride, const uint8_t *ki_e4m3, const float *ki_scale,
                              int32_t topk, int32_t *idx_out, void *workspace, size_t workspace_bytes,
                              int32_t *dev_err, cudaStream_t stream);

/* Sparse MLA over selected rows, run as MQA: every gathered latent row serves
 * all heads (GLM-5.3 Teil 2, section Ausprobieren; footnote 1). As
 * mla_prefill_dense, but token t attends only to the positions idx[t, 0..topk)
 * (entries -1 are skipped; an index above the token's position or below -1
 * sets MLA_DEVERR_BAD_INDEX and is skipped). A row whose list holds no valid
 * index gets out = 0 and lse = -inf. topk in [1, 2048]. */
mla_status_t mla_prefill_sparse(const mla_seqs_t *seqs, const void *q_bf16, int32_t num_heads,
                                const uint8_t *kv_e4m3, const float *kv_scale, float sm_scale,
                                const int32_t *idx, int32_t topk, void *out_bf16, float *lse,
                                void *workspace, size_t workspace_bytes, int32_t *dev_err,
                                cudaStream_t stream);

/* Bytes of one row of the alternative cache layout: the 656-byte row of
 * GLM-5.3 Teil 2, footnote 1 (656 FP8 KV bytes per token, FlashMLA's
 * fp8_ds_mla format), read as 512 e4m3 latent codes (bytes 0..511), one fp32
 * scale per 128 latent dims (bytes 512..527, little-endian; dim d of the latent
 * is scales[d/128] * dec(code[d])) and the 64 RoPE dims as bf16 (bytes
 * 528..655). Pages hold 256 rows, as for the 580-byte layout. */
#define MLA_DS_ROW_BYTES 656

/* Dense causal MLA prefill on a cache of 656-byte rows kv_ds [num_blocks, 256,
 * 656]: what mla_prefill_dense computes, with K_s[d] = scales_s[d/128] *
 * dec(code_s[d]) for d < 512 and K_s[512+i] = the bf16 RoPE value i, V_s =
 * K_s[0:512]. Every key row the new tokens see is first dequantised once into
 * an f16 row in the workspace (relative to the row's largest group scale, so
 * the scale ratios and the RoPE values are rounded once to 11 significant
 * bits), and the attention kernel multiplies those rows on the tensor cores in
 * f16 with fp32 accumulation. workspace: mla_workspace_size(MLA_OP_DENSE_DS,
 * ...) bytes, 256-byte aligned: the work list plus about 1,164 bytes per key
 * row of every sequence's context (its f16 row and metadata). Arguments and
 * errors otherwise as mla_prefill_dense; kv_ds 16-byte aligned. */
mla_status_t mla_prefill_dense_ds(const mla_seqs_t *seqs, const void *q_bf16, int32_t num_heads,
                                  const uint8_t *kv_ds, float sm_scale, void *out_bf16, float *lse,
                                  void *workspace, size_t workspace_bytes, int32_t *dev_err, cudaStream_t stream);

/* Sparse MLA over selected rows of a cache of 656-byte rows: what
 * mla_prefill_sparse computes, with the rows read as in mla_prefill_dense_ds.
 * No workspace. */
mla_status_t mla_prefill_sparse_ds(const mla_seqs_t *seqs, const void *q_bf16, int32_t num_heads,
                                   const uint8_t *kv_ds, float sm_scale, const int32_t *idx, int32_t topk,
                                   void *out_bf16, float *lse, int32_t *dev_err, cudaStream_t stream);

/* Non-absorbed (MHA) dense causal prefill, the path GLM-5.3 Teil 2 (section
 * Ausprobieren) describes for prefill batches whose prompts fit within the
 * top-k of 2,048 tokens when sparse_mla_force_mqa is off. Per head h, with c_s
 * = kv_scale_s * dec(kv_s[0:512]) and r_s = kv_scale_s * dec(kv_s[512:576]):
 *   k[s,h] = [ W_UK_h c_s ; r_s ]  (192 dims),   v[s,h] = W_UV_h c_s  (128 dims)
 *   out[t,h,:] = sum_s softmax_s(sm_scale * q[t,h,:] . k[s,h]) v[s,h],  s = 0..p
 *   lse[t,h]   = ln sum_s exp(sm_scale * q[t,h,:] . k[s,h])
 * q_bf16: [Tq, H, 192] (128 no-RoPE dims, then 64 RoPE dims with RoPE applied);
 * w_ukv_bf16: [H, 256, 512], rows 0..127 of head h are W_UK_h and rows
 * 128..255 W_UV_h (k[s,h][i] = sum_d W_UK_h[i][d] c_s[d]); out_bf16: [Tq, H,
 * 128]; lse: [Tq, H] or NULL. The keys and values of every sequence's whole
 * context are first up-projected into the workspace as f16 (k and v rows of
 * 256 bytes per head, 128 bytes of RoPE dims per row; each context padded to
 * 128 rows), then attended with the queries converted to f16 and P in f16 (so
 * every value must lie inside the f16 range). Any prompt length works; the workspace grows with
 * the context times the heads, which is why the path suits short prompts.
 * num_heads in {16, 32, 64, 128}; q, w_ukv, out and kv 16-byte aligned.
 * workspace: mla_workspace_size(MLA_OP_MHA, ...) bytes, 256-byte aligned.
 * Errors as mla_prefill_dense. */
mla_status_t mla_prefill_mha(const mla_seqs_t *seqs, const void *q_bf16, int32_t num_heads, const void *w_ukv_bf16,
                             const uint8_t *kv_e4m3, const float *kv_scale, float sm_scale, void *out_bf16,
                             float *lse, void *workspace, size_t workspace_bytes, int32_t *dev_err,
                             cudaStream_t stream);

/* Largest work list mla_prefill_dense_static can hold: 65,536 items of 16
 * bytes (1 MiB of device memory, reserved on every GPU that loads the library
 * for the life of the process). One item covers two 64-row query tiles, so
 * with 64 heads a call can carry about 131,000 new tokens. */
#define MLA_DENSE_STATIC_MAX_WORK_ITEMS 65536

/* Dense prefill for callers that cannot allocate device memory. This entry
 * point has no counterpart on the source pages: it exists for code that is
 * given only its inputs and outputs (a plugin inside a framework that owns
 * the whole device pool, or a caller that must avoid the implicit device
 * synchronisation of cudaMalloc). It computes exactly what mla_prefill_dense
 * computes and takes the same arguments minus the workspace; it calls no
 * allocator (CUDA's or any library's) and copies nothing from the host.
 * Its scratch space (the tile work list) is a fixed device array inside the
 * library. The first call on each device looks that array's address up
 * (cudaGetSymbolAddress, with the device current); make that first call
 * before capturing the stream into a graph. All calls share the array: two
 * calls whose work overlaps on the GPU (different streams, no ordering
 * between them) race and may return wrong results; calls on one stream are
 * ordered and safe. Nothing in the array needs to start at zero: each call
 * writes every entry it reads. The array's address is looked up once per
 * device and kept for the life of the process: after cudaDeviceReset() on a
 * device, do not call this entry point on that device again. A batch needing
 * more than MLA_DENSE_STATIC_MAX_WORK_ITEMS items returns
 * MLA_ERR_UNSUPPORTED. The work list is built on the GPU from the device
 * cu_seqlens_q; if it disagrees with the host mirror, MLA_DEVERR_SEQ_MISMATCH
 * is set and only rows both count are computed. */
mla_status_t mla_prefill_dense_static(const mla_seqs_t *seqs, const void *q_bf16, int32_t num_heads,
                                      const uint8_t *kv_e4m3, const float *kv_scale, float sm_scale,
                                      void *out_bf16, float *lse, int32_t *dev_err, cudaStream_t stream);

/* Most pieces mla_prefill_dense_host cuts the new tokens into. */
#define MLA_DENSE_HOST_MAX_CHUNKS 64

/* Dense prefill from host memory to host memory, with the copies overlapped
 * with the attention. This entry point has no counterpart on the source pages:
 * it serves callers whose queries and cache sit in host memory. It computes
 * exactly what mla_prefill_dense computes (the same tiles with the same
 * arithmetic, so the results are identical) and leaves the results in host
 * memory:
 *   1. the cache (kv_host, kv_scale_host: num_blocks * 256 rows) is copied to
 *      kv_e4m3 / kv_scale;
 *   2. the new tokens are cut into n_chunks near-equal pieces of consecutive
 *      tokens (moved to tile boundaries: 64 rows of token x head), and each
 *      piece's query rows are copied from q_host to q_bf16 (same [Tq, H, 576]
 *      layout), its attention runs as soon as its rows have arrived, and its
 *      out and lse rows are copied back to out_host / lse_host ([Tq, H, 512]
 *      bf16, [Tq, H] f32) as soon as it has finished.
 * Copies to the device, attention and copies back run on three sets of
 * streams of the call's own, so piece c+1's queries travel while piece c is
 * computed and piece c-1's output travels back. The call is ordered on
 * `stream`: it starts after the work queued there and that stream waits for
 * its last copy back; the host buffers may be read after synchronising with
 * `stream`. Host buffers should be page-locked (cudaHostAlloc or registered),
 * or the copies do not overlap. q_bf16, kv_e4m3, kv_scale, out_bf16 and lse
 * are device buffers the caller owns, with mla_prefill_dense's layout and
 * alignment; lse may be NULL only with lse_host NULL. n_chunks in [1,
 * MLA_DENSE_HOST_MAX_CHUNKS]. workspace: mla_workspace_size(MLA_OP_DENSE_HOST,
 * ...) bytes, 16-byte aligned. Errors: the checks of mla_prefill_dense, plus
 * MLA_ERR_INVALID_ARG for a NULL host pointer or n_chunks out of range. */
mla_status_t mla_prefill_dense_host(const mla_seqs_t *seqs, const void *q_host, int32_t num_heads,
                                    const uint8_t *kv_host, const float *kv_scale_host, float sm_scale,
                                    void *out_host, float *lse_host, void *q_bf16, uint8_t *kv_e4m3,
                                    float *kv_scale, void *out_bf16, float *lse, int32_t n_chunks,
                                    void *workspace, size_t workspace_bytes, int32_t *dev_err,
                                    cudaStream_t stream);

/* The tensors of one sparse step, once in host memory and once on the device
 * (mla_prefill_sparse_host). Layouts as in mla_indexer_topk and
 * mla_prefill_sparse; w holds one 64-value row (w_token_stride 0) or a row per
 * token at w + t * w_token_stride. */
typedef struct {
    void *q_bf16;       /* [Tq, H, 576] bf16 */
    uint8_t *qi_e4m3;   /* [Tq, 64, 128] */
    float *w;           /* indexer head weights */
    uint8_t *kv_e4m3;   /* [num_blocks, 256, 576] */
    float *kv_scale;    /* [num_blocks, 256] */
    uint8_t *ki_e4m3;   /* [num_blocks, 256, 128] */
    float *ki_scale;    /* [num_blocks, 256] */
} mla_sparse_inputs_t;

typedef struct {
    void *out_bf16;     /* [Tq, H, 512] bf16 */
    float *lse;         /* [Tq, H], or NULL */
    int32_t *idx;       /* [Tq, topk] selected positions */
} mla_sparse_outputs_t;

/* The sparse step (mla_indexer_topk, then mla_prefill_sparse over the
 * selected rows) from host memory to host memory, with the copies overlapped
 * with the kernels. This entry point has no counterpart on the source pages:
 * it serves callers whose inputs sit in host memory. It computes exactly what
 * the two device calls compute (identical indices and outputs):
 *   1. w, the latent cache and the indexer keys are copied to the device
 *      buffers of `dev_in`;
 *   2. the new tokens are cut into n_chunks near-equal pieces of consecutive
 *      tokens (moved to the indexer's 3-token group boundaries); each piece's
 *      qi and q rows are copied in, its indexer scores, top-k and sparse
 *      attention run as soon as they have arrived, and its out, lse and idx
 *      rows are copied back to `host_out` as soon as it has finished.
 * Streams, ordering and page-locking as in mla_prefill_dense_host. Every
 * pointer of host_in, dev_in, host_out and dev_out must be set, except the
 * lse pair: NULL in both or set in both. topk in [1, 2048]; n_chunks in [1,
 * MLA_DENSE_HOST_MAX_CHUNKS]. workspace: mla_workspace_size(MLA_OP_INDEXER,
 * ...) bytes, 256-byte aligned. Errors: the checks of the two device calls,
 * plus MLA_ERR_INVALID_ARG for a NULL pointer or n_chunks out of range. */
mla_status_t mla_prefill_sparse_host(const mla_seqs_t *seqs, int32_t num_heads, float sm_scale,
                                     int64_t w_token_stride, int32_t topk, const mla_sparse_inputs_t *host_in,
                                     const mla_sparse_inputs_t *dev_in, const mla_sparse_outputs_t *host_out,
                                     const mla_sparse_outputs_t *dev_out, int32_t n_chunks, void *workspace,
                                     size_t workspace_bytes, int32_t *dev_err, cudaStream_t stream);

/* Cache write of the new tokens: the step before attention, which reads the
 * rows this call stores ("More throughput from fewer GPUs", section System
 * architecture: FP8 KV cache, one latent row per token; section KV hand-off
 * and caching: 256-token chunks; GLM-5.3 Teil 2, footnote 3: indexer keys of
 * 128 FP8 values plus a 4-byte scale). For new token t of sequence b, at
 * position p = prefix_lens[b] + t - cu_seqlens_q[b] (page block_table[b][p/256],
 * slot p%256):
 *   kv_scale[p] = max(amax / 448, 2^-126), amax = max_d |latent[t,d]| (d < 576);
 *                 1 if amax = 0
 *   kv[p][d]    = the e4m3 code nearest to latent[t,d] * (1 / kv_scale[p]),
 *                 ties to the even code, magnitudes above 448 stored as 448
 * where the division, the reciprocal and the product are IEEE binary32
 * operations (the floor keeps the reciprocal finite). With kidx_bf16 set, the
 * 128-dim indexer key kidx[t] goes the same way into ki[p] / ki_scale[p];
 * with it NULL, ki and ki_scale are not used. Layouts: latent bf16 [Tq, 576],
 * kidx bf16 [Tq, 128], caches as in the data layout above. Nothing but the
 * new tokens' rows is written; two new tokens must not map to one cache row.
 * Inputs must be finite (a NaN or infinity makes that row unspecified). A page
 * id outside [0, num_blocks) sets MLA_DEVERR_BAD_PAGE and that token writes
 * nothing. latent, kidx, kv and ki 16-byte aligned; kv_scale, ki_scale 4-byte
 * aligned. No workspace. */
mla_status_t mla_kv_append(const mla_seqs_t *seqs, const void *latent_bf16, const void *kidx_bf16,
                           uint8_t *kv_e4m3, float *kv_scale, uint8_t *ki_e4m3, float *ki_scale,
                           int32_t *dev_err, cudaStream_t stream);

/* Most partial results one mla_merge_attn call combines. */
#define MLA_MERGE_MAX_PARTS 8

/* Merge of partial attention results over disjoint key sets: the
 * log-sum-exp combination by which attention split over shards of the cache
 * is put back together (GLM-5.3 Teil 2, section "DCP: Sharding auch des
 * KV-Caches": each GPU attends over its own shard and the partial results are
 * combined through their log-sum-exp). Part i holds, per row (one (token,
 * head) pair), the output o_i of attention over its keys and lse_i, as written
 * by mla_prefill_dense / mla_prefill_sparse. For each row:
 *   lse = ln sum_i exp(lse_i),   out = sum_i exp(lse_i - lse) * o_i
 * which is attention over the union of the parts' keys. A part with lse_i =
 * -inf (no keys) adds nothing; a row whose parts are all -inf gets out = 0,
 * lse = -inf. Arithmetic in fp32, out rounded once to bf16.
 * outs_bf16, lses: HOST arrays of n_parts DEVICE pointers; part i is bf16
 * [rows, 512] (16-byte aligned) and f32 [rows] (4-byte aligned). out_bf16:
 * bf16 [rows, 512], 16-byte aligned; it may be one of the parts (in place).
 * lse_out: f32 [rows] or NULL. n_parts in [1, MLA_MERGE_MAX_PARTS]; a NaN or
 * +inf lse gives an unspecified row. No workspace. */
mla_status_t mla_merge_attn(int32_t n_parts, const void *const *outs_bf16, const float *const *lses, int64_t rows,
                            void *out_bf16, float *lse_out, cudaStream_t stream);

/* Message for the last non-OK status returned on this thread ("" if none). */
const char *mla_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* MLA_H_ */

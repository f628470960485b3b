// Launch interfaces between the C ABI layer and the kernels (internal).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace mla {

struct AttnArgs {
    const __nv_bfloat16 *q;      // [Tq, H, 576]
    const uint8_t *kv;           // [num_blocks, 256, 576] e4m3
    const float *kv_scale;       // [num_blocks, 256]
    const int32_t *block_table;  // [batch, max_blocks]
    int32_t max_blocks, num_blocks;
    const int32_t *cu_seqlens;   // [batch+1]
    const int32_t *prefix_lens;  // [batch]
    int32_t batch;
    __nv_bfloat16 *out;          // [Tq, H, 512]
    float *lse;                  // [Tq, H] or null
    int32_t H;
    float sm_scale_log2;         // sm_scale * log2(e)
    const int32_t *idx;          // sparse: [Tq, topk]
    int32_t topk;
    int32_t *dev_err;
    int64_t tok_begin, tok_end;  // sparse: the new tokens this launch attends for (global indices)
    int64_t total_q;             // new tokens by the host mirror of cu_seqlens: no row at or past total_q * H
                                 // is read or written whatever the device copy says
    // dense calls on 656-byte rows: the converted keys (f16 [rows][576], each
    // sequence's rows from conv_base[b], padded to 80-key tiles) and their tile metadata
    __half *kconv;
    uint8_t *kmeta;
    const int32_t *conv_base;    // [batch], converted row of each sequence's key 0
    const int32_t *conv_ctx;     // [batch], keys each sequence has (prefix + new)
};

// Dense attention on e4m3 operands (kind::f8f6f4). Work item: x = sequence,
// y = 64-row tile, z = paired row tile or -1. tmap_kv: the latent cache as
// [num_blocks * 256 rows][576 B], 128 x 128 boxes, 128-byte swizzle (encode_kv_tmap).
cudaError_t launch_dense_f8(const AttnArgs &a, const int4 *work, int n_work, const CUtensorMap &tmap_kv, cudaStream_t st);
bool encode_kv_tmap(CUtensorMap *map, const uint8_t *kv, int32_t num_blocks);
// Sparse attention on e4m3 operands: rows gathered by index (cp.async), two
// tokens x 64 heads per CTA, for the tokens [a.tok_begin, a.tok_end).
cudaError_t launch_sparse_f8(const AttnArgs &a, cudaStream_t st);

// The same two on a cache of 656-byte rows (512 e4m3 latent codes, four fp32
// group scales, 64 bf16 RoPE values; a.kv_scale unused): tcgen05 kind::f16, 64
// query rows x 80 keys per tile. Dense: the rows are first converted to f16
// (a.kconv, a.kmeta; n_conv_rows rows) and loaded by TMA through tmap_conv
// ([rows][576] f16, 64 x 80 boxes, 128-byte swizzle); sparse: gathered and
// converted in shared memory.
constexpr int kDsTileKeys = 80;
constexpr int kDsMetaBytes = 960;     // one key tile's metadata
cudaError_t launch_dense_ds(const AttnArgs &a, const int4 *work, int n_work, int64_t n_conv_rows,
                            const CUtensorMap &tmap_conv, cudaStream_t st);
cudaError_t launch_sparse_ds(const AttnArgs &a, cudaStream_t st);

// Non-absorbed (MHA) path: per-head keys [W_UK c ; r] (192 dims) and values
// W_UV c (128 dims), up-projected from the 580-byte cache rows into a workspace,
// then causal attention per head.
constexpr int kDr = 64;        // RoPE dims
constexpr int kDvh = 128;      // no-RoPE key dims and value dims per head
struct MhaArgs {
    const __nv_bfloat16 *q;      // [Tq, H, 192]
    const uint8_t *kv;           // [num_blocks, 256, 576] e4m3
    const float *kv_scale;       // [num_blocks, 256]
    const int32_t *block_table;  // [batch, max_blocks]
    int32_t max_blocks, num_blocks;
    __half *kn;                  // [H, R, 128] up-projected no-RoPE keys (f16)
    __half *v;                   // [H, R, 128] up-projected values (f16)
    __half *kr;                  // [R, 64] RoPE dims of the keys (f16)
    int64_t R;                   // key rows: each sequence's context padded to 128
    __nv_bfloat16 *out;          // [Tq, H, 128]
    float *lse;                  // [Tq, H] or null
    int32_t H;
    int32_t up_heads;            // heads per up-projection CTA (divides H)
    float sm_scale_log2;
    int32_t *dev_err;
    int64_t total_q;             // new tokens (rows of q) by the host mirror of cu_seqlens
    int32_t ahead;               // attention: CTA blockIdx.x + ahead is the one expected to follow
                                 // on the same SM (the SM count; set by the launcher)
};
// Up-projection: work item = {sequence, first position (a multiple of 128),
// key-row base of those rows, context length}; tmap_w: w_ukv as [H*256 rows][512]
// bf16, 64 x 128 boxes (a half head's rows), 128-byte swizzle.
cudaError_t launch_mha_up(const MhaArgs &a, const int4 *work, int n_work, const CUtensorMap &tmap_w, cudaStream_t st);
// Attention: work item = two int4, {sequence, first new token in it, that
// token's global index, valid rows <= 128} and {prefix, key-row base, key tiles
// of 64, 0}; one CTA per item and head (q is read row by row into TMEM).
// tmap_kn / tmap_v: f16 [H*R rows][128], 64 x 64 boxes; tmap_kr: f16 [R][64],
// 64 x 64 boxes; all with the 128-byte swizzle.
cudaError_t launch_mha_attn(const MhaArgs &a, const int4 *work, int n_work, const CUtensorMap &tmap_kn,
                            const CUtensorMap &tmap_kr, const CUtensorMap &tmap_v, cudaStream_t st);

struct IndexerArgs {
    const uint8_t *qi;           // [Tq, 64, 128] e4m3
    const float *w;              // row t at w + t * w_stride
    int64_t w_stride;
    const uint8_t *ki;           // [num_blocks, 256, 128] e4m3
    const float *ki_scale;       // [num_blocks, 256]
    const int32_t *block_table;
    int32_t max_blocks, num_blocks;
    const int32_t *cu_seqlens;
    const int32_t *prefix_lens;
    int32_t batch;
    int32_t topk;
    int32_t *idx_out;            // [Tq, topk]
    int32_t *dev_err;
    int64_t total_q;             // new tokens by the host mirror of cu_seqlens
    int32_t *fail;               // one flag per work item: the fast path left the group to the exact path
};

// Indexer scores and streaming exact top-k in one kernel. Work item: x =
// sequence, y = first new token (in-sequence), z = token count (<=
// kIdxTokensPerCta); the CTA streams every key those tokens see. tmap_k: the
// key cache as [num_blocks * 256 rows][128 B]; tmap_q: the queries as [Tq * 64
// rows][128 B]; both with 128-byte-wide boxes and the 128-byte swizzle (boxes of
// 128 key rows and of kIdxTokensPerCta * 64 query rows). Each token keeps up to
// kIdxCandidates candidates in shared memory. Two launches: the fast path
// (sampled threshold) for every item, then the exact streaming path for the
// items it flagged in a.fail (one int32 per item, written by the first launch).
constexpr int kIdxTokensPerCta = 3;
constexpr int kIdxCandidates = 5120;
cudaError_t launch_indexer_topk(const IndexerArgs &a, const int4 *work, int n_work, const CUtensorMap &tmap_k,
                                const CUtensorMap &tmap_q, cudaStream_t st);

struct AppendArgs {
    const __nv_bfloat16 *latent; // [Tq, 576]
    const __nv_bfloat16 *kidx;   // [Tq, 128] or null
    uint8_t *kv;                 // [num_blocks, 256, 576] e4m3
    float *kv_scale;             // [num_blocks, 256]
    uint8_t *ki;                 // [num_blocks, 256, 128] e4m3 (unused without kidx)
    float *ki_scale;             // [num_blocks, 256]
    const int32_t *block_table;
    int32_t max_blocks, num_blocks;
    const int32_t *cu_seqlens;
    const int32_t *prefix_lens;
    int32_t batch;
    int64_t n_tokens;
    int32_t *dev_err;
};

// Cache write of the new tokens (per-token absmax/448 e4m3 rows), one warp per token.
cudaError_t launch_kv_append(const AppendArgs &a, cudaStream_t st);

constexpr int kMergeMaxParts = 8;
struct MergeArgs {
    const uint4 *outs[kMergeMaxParts];   // part i: bf16 [rows, 512]
    const float *lses[kMergeMaxParts];   // part i: f32 [rows]
    int32_t n_parts;
    int64_t rows;
    uint4 *out;                          // bf16 [rows, 512] (may be one of the parts)
    float *lse;                          // f32 [rows] or null
};
// Log-sum-exp merge of partial attention results, one warp per row.
cudaError_t launch_merge(const MergeArgs &a, cudaStream_t st);

}  // namespace mla

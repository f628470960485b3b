// C ABI of the MLA prefill attention library: argument checks, scheduling,
// workspace layout and kernel launches. Every entry point is declared and
// documented in include/mla.h.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "../../include/mla.h"
#include "kernels.h"

static_assert(MLA_MERGE_MAX_PARTS == mla::kMergeMaxParts, "merge part limit");

namespace {

thread_local std::string g_err;

mla_status_t fail(mla_status_t s, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = buf;
    return s;
}

mla_status_t cuda_fail(cudaError_t e, const char *where) {
    return fail(MLA_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

constexpr int kBM = 64;               // query rows per dense tile
constexpr size_t kWsAlign = 256;

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

mla_status_t check_seqs(const mla_seqs_t *s) {
    if (!s) return fail(MLA_ERR_INVALID_ARG, "seqs is NULL");
    if (s->batch < 1) return fail(MLA_ERR_INVALID_ARG, "batch must be >= 1 (got %d)", s->batch);
    if (!s->cu_seqlens_q || !s->cu_seqlens_q_host || !s->prefix_lens || !s->prefix_lens_host || !s->block_table)
        return fail(MLA_ERR_INVALID_ARG, "cu_seqlens_q, prefix_lens (device and host) and block_table must be set");
    if (s->max_blocks_per_seq < 1 || s->num_blocks < 1)
        return fail(MLA_ERR_INVALID_ARG, "max_blocks_per_seq and num_blocks must be >= 1");
    if (static_cast<int64_t>(s->num_blocks) * 256 > INT32_MAX)
        return fail(MLA_ERR_UNSUPPORTED, "num_blocks * 256 must fit in int32");
    if (s->cu_seqlens_q_host[0] != 0) return fail(MLA_ERR_INVALID_ARG, "cu_seqlens_q[0] must be 0");
    for (int b = 0; b < s->batch; ++b) {
        const int64_t t = static_cast<int64_t>(s->cu_seqlens_q_host[b + 1]) - s->cu_seqlens_q_host[b];
        const int64_t p = s->prefix_lens_host[b];
        if (t < 0) return fail(MLA_ERR_INVALID_ARG, "cu_seqlens_q must be non-decreasing (sequence %d)", b);
        if (p < 0) return fail(MLA_ERR_INVALID_ARG, "prefix_lens[%d] < 0", b);
        if (p + t > INT32_MAX - 256) return fail(MLA_ERR_UNSUPPORTED, "sequence %d too long", b);
        if ((p + t + 255) / 256 > s->max_blocks_per_seq)
            return fail(MLA_ERR_INVALID_ARG, "sequence %d needs %lld pages > max_blocks_per_seq %d", b,
                        static_cast<long long>((p + t + 255) / 256), s->max_blocks_per_seq);
    }
    return MLA_OK;
}

bool heads_ok(int32_t h) { return h == 16 || h == 32 || h == 64 || h == 128; }

// Paired row tiles: tile i with tile n-1-i of the same sequence (the V-shaped
// chunk pairing of the PCP scheme, applied at tile granularity), items sorted
// by decreasing work so the costliest go first. Only the tiles of the new
// tokens [t0, t1) (global indices, on tile boundaries of their sequences) are
// scheduled; within each sequence's share of that range the first tile pairs
// with the last.
std::vector<int4> dense_schedule_range(const mla_seqs_t *s, int32_t H, int64_t t0, int64_t t1) {
    struct Item {
        int4 v;
        int64_t cost;
    };
    std::vector<Item> items;
    for (int b = 0; b < s->batch; ++b) {
        const int64_t c0 = s->cu_seqlens_q_host[b], c1 = s->cu_seqlens_q_host[b + 1];
        const int64_t l0 = std::max(t0, c0) - c0, l1 = std::min(t1, c1) - c0;
        if (l1 <= l0) continue;
        const int64_t P = s->prefix_lens_host[b];
        const int64_t rows = (c1 - c0) * H;
        const int64_t i_lo = l0 * H / kBM, i_hi = (l1 * H + kBM - 1) / kBM;
        auto tile_keys = [&](int64_t i) {
            const int64_t last_row = std::min(rows, (i + 1) * kBM) - 1;
            return P + last_row / H + 1;
        };
        for (int64_t m = 0; m < (i_hi - i_lo + 1) / 2; ++m) {
            const int64_t i = i_lo + m, j = i_hi - 1 - m;
            Item it;
            it.v = make_int4(b, static_cast<int>(i), j != i ? static_cast<int>(j) : -1, 0);
            it.cost = tile_keys(i) + (j != i ? tile_keys(j) : 0);
            items.push_back(it);
        }
    }
    std::stable_sort(items.begin(), items.end(), [](const Item &x, const Item &y) { return x.cost > y.cost; });
    std::vector<int4> out(items.size());
    for (size_t i = 0; i < items.size(); ++i) out[i] = items[i].v;
    return out;
}

std::vector<int4> dense_schedule(const mla_seqs_t *s, int32_t H) {
    return dense_schedule_range(s, H, 0, s->cu_seqlens_q_host[s->batch]);
}

// Token boundaries of n_chunks near-equal pieces of the new tokens, each moved
// down to a tile boundary of the sequence it falls in (a tile is 64 rows of
// token x head, i.e. 64/H tokens for H <= 64); pieces may come out empty.
std::vector<int64_t> dense_chunk_bounds(const mla_seqs_t *s, int32_t H, int32_t n_chunks) {
    const int64_t tq = s->cu_seqlens_q_host[s->batch];
    const int64_t g = H < kBM ? kBM / H : 1;     // tokens per tile
    std::vector<int64_t> bnd(static_cast<size_t>(n_chunks) + 1);
    bnd[0] = 0;
    bnd[n_chunks] = tq;
    int b = 0;
    for (int c = 1; c < n_chunks; ++c) {
        const int64_t t = tq * c / n_chunks;
        while (b + 1 < s->batch && s->cu_seqlens_q_host[b + 1] <= t) ++b;
        const int64_t c0 = s->cu_seqlens_q_host[b];
        bnd[c] = std::max(bnd[c - 1], c0 + (t - c0) / g * g);
    }
    return bnd;
}

// Upper bound of the items of all pieces: a piece's share of a sequence adds at
// most half a pair to the plain schedule, and the shares number at most
// batch + n_chunks.
size_t dense_host_items_bound(const mla_seqs_t *s, int32_t H) {
    size_t tiles = 0;
    for (int b = 0; b < s->batch; ++b) {
        const int64_t rows = static_cast<int64_t>(s->cu_seqlens_q_host[b + 1] - s->cu_seqlens_q_host[b]) * H;
        tiles += static_cast<size_t>((rows + kBM - 1) / kBM);
    }
    return tiles / 2 + static_cast<size_t>(s->batch) + MLA_DENSE_HOST_MAX_CHUNKS + 1;
}

// Work items of the indexer: (sequence, first token, token count, 0) for every
// group of kIdxTokensPerCta tokens whose first token lies in [t0, t1) (global
// indices; groups start every kIdxTokensPerCta tokens from the start of their
// sequence). A CTA streams every key its group can see, so the items are sorted
// by that count, longest first (LPT), to keep the last wave short.
std::vector<int4> indexer_schedule(const mla_seqs_t *s, int64_t t0, int64_t t1) {
    struct Item {
        int4 v;
        int64_t keys;
    };
    std::vector<Item> items;
    for (int b = 0; b < s->batch; ++b) {
        const int64_t c0 = s->cu_seqlens_q_host[b];
        const int t = s->cu_seqlens_q_host[b + 1] - s->cu_seqlens_q_host[b];
        const int P = s->prefix_lens_host[b];
        for (int i0 = 0; i0 < t; i0 += mla::kIdxTokensPerCta) {
            if (c0 + i0 < t0 || c0 + i0 >= t1) continue;
            const int nt = std::min(mla::kIdxTokensPerCta, t - i0);
            items.push_back({make_int4(b, i0, nt, 0), static_cast<int64_t>(P) + i0 + nt});
        }
    }
    std::stable_sort(items.begin(), items.end(), [](const Item &x, const Item &y) { return x.keys > y.keys; });
    std::vector<int4> out(items.size());
    for (size_t i = 0; i < items.size(); ++i) out[i] = items[i].v;
    return out;
}

// Indexer workspace: the work list (16 bytes per item), then one int32 flag per
// item (the fast path marks the items it leaves to the exact path).
size_t indexer_ws_bytes(size_t n_items) {
    return round_up(n_items * sizeof(int4), kWsAlign) + round_up(n_items * sizeof(int32_t), kWsAlign);
}

size_t indexer_groups(const mla_seqs_t *s) {
    size_t n = 0;
    for (int b = 0; b < s->batch; ++b) {
        const int t = s->cu_seqlens_q_host[b + 1] - s->cu_seqlens_q_host[b];
        n += static_cast<size_t>((t + mla::kIdxTokensPerCta - 1) / mla::kIdxTokensPerCta);
    }
    return n;
}

// 2-D tensor map over a row-major u8 matrix [rows][width] for TMA copies of
// box_rows x 128-byte boxes with the 128-byte swizzle (bytes past the row end
// read as zero). The encoder is fetched from the driver once; no link against
// the driver library is needed.
using EncodeTiled = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                 const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiled tiled_encoder() {
    static EncodeTiled encode = nullptr;
    if (!encode) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn)
            return nullptr;
        encode = reinterpret_cast<EncodeTiled>(fn);
    }
    return encode;
}

// Tensor map over a 16-bit (bf16 or f16) tensor of rank 2 or 3 (dims innermost
// first, byte strides of the outer dims), 128-byte swizzle, zero fill past the edges.
bool encode_16bit(CUtensorMap *map, CUtensorMapDataType type, const void *base, cuuint32_t rank,
                  const cuuint64_t *dims, const cuuint64_t *strides, const cuuint32_t *box) {
    const EncodeTiled encode = tiled_encoder();
    if (!encode) return false;
    const cuuint32_t estr[3] = {1, 1, 1};
    return encode(map, type, rank, const_cast<void *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_u8_rows(CUtensorMap *map, const void *base, uint64_t width, uint64_t rows, uint32_t box_rows) {
    const EncodeTiled encode = tiled_encoder();
    if (!encode) return false;
    const cuuint64_t dims[2] = {width, rows};
    const cuuint64_t strides[1] = {width};
    const cuuint32_t box[2] = {128, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
bool encode_rows128(CUtensorMap *map, const void *base, uint64_t rows, uint32_t box_rows) {
    return encode_u8_rows(map, base, 128, rows, box_rows);
}

// The non-absorbed path's plan: key rows (each sequence with new tokens gets
// its context padded to 128 rows), the up-projection items (one per 128 rows)
// and the attention items (one per 128 new tokens, two int4 each, longest
// first), and the workspace layout.
struct MhaPlan {
    std::vector<int4> up, at;
    int64_t R = 0;
    size_t off_at = 0, off_up = 0, off_kn = 0, off_v = 0, off_kr = 0, bytes = 0;
};
MhaPlan mha_plan(const mla_seqs_t *s, int32_t H) {
    MhaPlan p;
    struct At {
        int4 a, b;
    };
    std::vector<At> at;
    for (int b = 0; b < s->batch; ++b) {
        const int64_t c0 = s->cu_seqlens_q_host[b], q = s->cu_seqlens_q_host[b + 1] - c0;
        if (q <= 0) continue;
        const int64_t P = s->prefix_lens_host[b], ctx = P + q;
        const int64_t kb = p.R;
        for (int64_t y = 0; y < ctx; y += 128)
            p.up.push_back(make_int4(b, static_cast<int>(y), static_cast<int>(kb + y), static_cast<int>(ctx)));
        for (int64_t i0 = 0; i0 < q; i0 += 128) {
            const int64_t nv = std::min<int64_t>(128, q - i0);
            const int64_t n_tiles = (P + i0 + nv + 63) / 64;
            at.push_back({make_int4(b, static_cast<int>(i0), static_cast<int>(c0 + i0), static_cast<int>(nv)),
                          make_int4(static_cast<int>(P), static_cast<int>(kb), static_cast<int>(n_tiles), 0)});
        }
        p.R += (ctx + 127) / 128 * 128;
    }
    std::stable_sort(at.begin(), at.end(), [](const At &x, const At &y) { return x.b.z > y.b.z; });
    for (const At &x : at) {
        p.at.push_back(x.a);
        p.at.push_back(x.b);
    }
    p.off_at = 0;
    p.off_up = round_up(p.at.size() * sizeof(int4), kWsAlign);
    p.off_kn = p.off_up + round_up(p.up.size() * sizeof(int4), kWsAlign);
    const size_t kv_bytes = round_up(static_cast<size_t>(H) * static_cast<size_t>(p.R) * 256, kWsAlign);
    p.off_v = p.off_kn + kv_bytes;
    p.off_kr = p.off_v + kv_bytes;
    p.bytes = p.off_kr + round_up(static_cast<size_t>(p.R) * 128, kWsAlign);
    return p;
}

// Dense calls on 656-byte rows: each sequence with new tokens gets its keys
// converted to f16 rows from conv_base[b] (its context padded to whole 80-key
// tiles). Workspace: work list | conv_base, conv_ctx | f16 rows | tile metadata.
struct DsPlan {
    std::vector<int4> work;
    std::vector<int32_t> base, ctx;
    int64_t rows = 0;
    size_t off_ints = 0, off_rows = 0, off_meta = 0, bytes = 0;
};
DsPlan ds_plan(const mla_seqs_t *s, int32_t H) {
    DsPlan p;
    p.work = dense_schedule(s, H);
    p.base.assign(static_cast<size_t>(s->batch), 0);
    p.ctx.assign(static_cast<size_t>(s->batch), 0);
    for (int b = 0; b < s->batch; ++b) {
        const int64_t q = s->cu_seqlens_q_host[b + 1] - s->cu_seqlens_q_host[b];
        p.base[b] = static_cast<int32_t>(p.rows);
        if (q <= 0) continue;
        const int64_t ctx = s->prefix_lens_host[b] + q;
        p.ctx[b] = static_cast<int32_t>(ctx);
        p.rows += (ctx + mla::kDsTileKeys - 1) / mla::kDsTileKeys * mla::kDsTileKeys;
    }
    p.off_ints = round_up(p.work.size() * sizeof(int4), kWsAlign);
    p.off_rows = p.off_ints + round_up(2 * static_cast<size_t>(s->batch) * sizeof(int32_t), kWsAlign);
    p.off_meta = p.off_rows + round_up(static_cast<size_t>(p.rows) * 576 * 2, kWsAlign);
    p.bytes = p.off_meta + round_up(static_cast<size_t>(p.rows / mla::kDsTileKeys) * mla::kDsMetaBytes, kWsAlign);
    return p;
}

mla::AttnArgs attn_args(const mla_seqs_t *s, const void *q, int32_t H, const uint8_t *kv, const float *kv_scale,
                        float sm_scale, void *out, float *lse, int32_t *dev_err) {
    mla::AttnArgs a{};
    a.q = static_cast<const __nv_bfloat16 *>(q);
    a.kv = kv;
    a.kv_scale = kv_scale;
    a.block_table = s->block_table;
    a.max_blocks = s->max_blocks_per_seq;
    a.num_blocks = s->num_blocks;
    a.cu_seqlens = s->cu_seqlens_q;
    a.prefix_lens = s->prefix_lens;
    a.batch = s->batch;
    a.out = static_cast<__nv_bfloat16 *>(out);
    a.lse = lse;
    a.H = H;
    a.sm_scale_log2 = sm_scale * 1.4426950408889634f;
    a.dev_err = dev_err;
    a.total_q = s->cu_seqlens_q_host[s->batch];
    return a;
}

mla_status_t check_attn_ptrs(const void *q, const uint8_t *kv, const float *kv_scale, const void *out,
                             const float *lse, float sm_scale) {
    if (!q || !kv || !kv_scale || !out) return fail(MLA_ERR_INVALID_ARG, "q, kv, kv_scale and out must be set");
    if (!aligned(q, 16) || !aligned(kv, 16) || !aligned(out, 16))
        return fail(MLA_ERR_INVALID_ARG, "q, kv and out must be 16-byte aligned");
    if (!aligned(kv_scale, 4) || (lse && !aligned(lse, 4)))
        return fail(MLA_ERR_INVALID_ARG, "kv_scale and lse must be 4-byte aligned");
    if (!std::isfinite(sm_scale)) return fail(MLA_ERR_INVALID_ARG, "sm_scale must be finite");
    return MLA_OK;
}

}  // namespace

extern "C" {

const char *mla_last_error(void) { return g_err.c_str(); }

size_t mla_workspace_size(mla_op_t op, const mla_seqs_t *seqs, int32_t num_heads, int32_t topk) {
    (void)topk;
    if (check_seqs(seqs) != MLA_OK) return 0;
    switch (op) {
        case MLA_OP_DENSE:
            if (!heads_ok(num_heads)) return 0;
            return round_up(dense_schedule(seqs, num_heads).size() * sizeof(int4), kWsAlign);
        case MLA_OP_INDEXER:
            // the work list and a flag per item: the scores stay on chip
            return indexer_ws_bytes(indexer_groups(seqs));
        case MLA_OP_SPARSE:
            return 0;
        case MLA_OP_DENSE_HOST:
            if (!heads_ok(num_heads)) return 0;
            return round_up(dense_host_items_bound(seqs, num_heads) * sizeof(int4), kWsAlign);
        case MLA_OP_MHA:
            if (!heads_ok(num_heads)) return 0;
            return mha_plan(seqs, num_heads).bytes;
        case MLA_OP_DENSE_DS:
            if (!heads_ok(num_heads)) return 0;
            return ds_plan(seqs, num_heads).bytes;
    }
    return 0;
}

mla_status_t mla_prefill_dense(const mla_seqs_t *seqs, const void *q_bf16, int32_t num_heads,
                               const uint8_t *kv_e4m3, const float *kv_scale, float sm_scale, void *out_bf16,
                               float *lse, void *workspace, size_t workspace_bytes, int32_t *dev_err,
                               cudaStream_t stream) {
    g_err.clear();
    mla_status_t st = check_seqs(seqs);
    if (st != MLA_OK) return st;
    if (!heads_ok(num_heads)) return fail(MLA_ERR_UNSUPPORTED, "num_heads must be 16, 32, 64 or 128 (got %d)", num_heads);
    if ((st = check_attn_ptrs(q_bf16, kv_e4m3, kv_scale, out_bf16, lse, sm_scale)) != MLA_OK) return st;
    const std::vector<int4> work = dense_schedule(seqs, num_heads);
    const size_t need = round_up(work.size() * sizeof(int4), kWsAlign);
    if (work.empty()) return MLA_OK;
    if (!workspace || workspace_bytes < need || !aligned(workspace, 16))
        return fail(MLA_ERR_WORKSPACE, "dense needs %zu workspace bytes (16-byte aligned), got %zu", need,
                    workspace ? workspace_bytes : 0);
    if (static_cast<int64_t>(work.size()) > INT32_MAX)
        return fail(MLA_ERR_UNSUPPORTED, "too many tiles");
    cudaError_t e = cudaMemcpyAsync(workspace, work.data(), work.size() * sizeof(int4), cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return cuda_fail(e, "schedule upload");
    const mla::AttnArgs a = attn_args(seqs, q_bf16, num_heads, kv_e4m3, kv_scale, sm_scale, out_bf16, lse, dev_err);
    CUtensorMap tmap_kv;
    if (!mla::encode_kv_tmap(&tmap_kv, kv_e4m3, seqs->num_blocks))
        return fail(MLA_ERR_CUDA, "tensor map encoding for the latent cache failed");
    e = mla::launch_dense_f8(a, static_cast<const int4 *>(workspace), static_cast<int>(work.size()), tmap_kv, stream);
    if (e != cudaSuccess) return cuda_fail(e, "dense launch");
    return MLA_OK;
}

namespace {
// Streams and events of one host-to-host call; destroyed when the call returns
// (CUDA releases them once the work queued on them has finished).
struct HostPipe {
    cudaStream_t s_in = nullptr, s_out = nullptr, s_c[2] = {nullptr, nullptr};
    std::vector<cudaEvent_t> ev;
    ~HostPipe() {
        for (cudaEvent_t e : ev) cudaEventDestroy(e);
        for (cudaStream_t x : {s_in, s_out, s_c[0], s_c[1]})
            if (x) cudaStreamDestroy(x);
    }
    cudaError_t event(cudaEvent_t *e) {
        cudaError_t r = cudaEventCreateWithFlags(e, cudaEventDisableTiming);
        if (r == cudaSuccess) ev.push_back(*e);
        return r;
    }
};
}  // namespace

mla_status_t mla_prefill_dense_host(const mla_seqs_t *seqs, const void *q_host, int32_t num_heads,
                                    const uint8_t *kv_host, const float *kv_scale_host, float sm_scale,
                                    void *out_host, float *lse_host, void *q_bf16, uint8_t *kv_e4m3, float *kv_scale,
                                    void *out_bf16, float *lse, int32_t n_chunks, void *workspace,
                                    size_t workspace_bytes, int32_t *dev_err, cudaStream_t stream) {
    g_err.clear();
    mla_status_t st = check_seqs(seqs);
    if (st != MLA_OK) return st;
    if (!heads_ok(num_heads)) return fail(MLA_ERR_UNSUPPORTED, "num_heads must be 16, 32, 64 or 128 (got %d)", num_heads);
    if ((st = check_attn_ptrs(q_bf16, kv_e4m3, kv_scale, out_bf16, lse, sm_scale)) != MLA_OK) return st;
    if (!q_host || !kv_host || !kv_scale_host || !out_host)
        return fail(MLA_ERR_INVALID_ARG, "q_host, kv_host, kv_scale_host and out_host must be set");
    if (lse_host && !lse) return fail(MLA_ERR_INVALID_ARG, "lse_host needs the device lse buffer");
    if (n_chunks < 1 || n_chunks > MLA_DENSE_HOST_MAX_CHUNKS)
        return fail(MLA_ERR_INVALID_ARG, "n_chunks must be in [1, %d] (got %d)", MLA_DENSE_HOST_MAX_CHUNKS, n_chunks);
    const int64_t tq = seqs->cu_seqlens_q_host[seqs->batch];
    if (tq == 0) return MLA_OK;
    const std::vector<int64_t> bnd = dense_chunk_bounds(seqs, num_heads, n_chunks);
    std::vector<int4> work;
    std::vector<size_t> off(static_cast<size_t>(n_chunks) + 1, 0);
    for (int c = 0; c < n_chunks; ++c) {
        const std::vector<int4> w = dense_schedule_range(seqs, num_heads, bnd[c], bnd[c + 1]);
        work.insert(work.end(), w.begin(), w.end());
        off[c + 1] = work.size();
    }
    const size_t need = round_up(work.size() * sizeof(int4), kWsAlign);
    if (work.size() > dense_host_items_bound(seqs, num_heads))   // the bound the workspace size promises
        return fail(MLA_ERR_INVALID_ARG, "internal: %zu work items above the workspace bound", work.size());
    if (!workspace || workspace_bytes < need || !aligned(workspace, 16))
        return fail(MLA_ERR_WORKSPACE, "dense from host needs %zu workspace bytes (16-byte aligned), got %zu", need,
                    workspace ? workspace_bytes : 0);
    const mla::AttnArgs a = attn_args(seqs, q_bf16, num_heads, kv_e4m3, kv_scale, sm_scale, out_bf16, lse, dev_err);
    CUtensorMap tmap_kv;
    if (!mla::encode_kv_tmap(&tmap_kv, kv_e4m3, seqs->num_blocks))
        return fail(MLA_ERR_CUDA, "tensor map encoding for the latent cache failed");

    HostPipe p;
    cudaError_t e;
    cudaEvent_t ev_entry, ev_end;
#define MLA_TRY(x, what)                       \
    if ((e = (x)) != cudaSuccess) return cuda_fail(e, what)
    MLA_TRY(cudaStreamCreateWithFlags(&p.s_in, cudaStreamNonBlocking), "stream");
    MLA_TRY(cudaStreamCreateWithFlags(&p.s_out, cudaStreamNonBlocking), "stream");
    MLA_TRY(cudaStreamCreateWithFlags(&p.s_c[0], cudaStreamNonBlocking), "stream");
    MLA_TRY(cudaStreamCreateWithFlags(&p.s_c[1], cudaStreamNonBlocking), "stream");
    MLA_TRY(p.event(&ev_entry), "event");
    MLA_TRY(p.event(&ev_end), "event");
    // everything queued on `stream` before this call comes first
    MLA_TRY(cudaEventRecord(ev_entry, stream), "event record");
    for (cudaStream_t x : {p.s_in, p.s_out, p.s_c[0], p.s_c[1]}) MLA_TRY(cudaStreamWaitEvent(x, ev_entry, 0), "wait");
    // the cache and the work lists first, then the queries piece by piece
    const size_t rows_kv = static_cast<size_t>(seqs->num_blocks) * 256;
    MLA_TRY(cudaMemcpyAsync(kv_e4m3, kv_host, rows_kv * 576, cudaMemcpyHostToDevice, p.s_in), "cache copy");
    MLA_TRY(cudaMemcpyAsync(kv_scale, kv_scale_host, rows_kv * sizeof(float), cudaMemcpyHostToDevice, p.s_in),
            "cache scale copy");
    MLA_TRY(cudaMemcpyAsync(workspace, work.data(), work.size() * sizeof(int4), cudaMemcpyHostToDevice, p.s_in),
            "schedule upload");
    const size_t q_row = static_cast<size_t>(num_heads) * 576 * 2, o_row = static_cast<size_t>(num_heads) * 512 * 2,
                 l_row = static_cast<size_t>(num_heads) * sizeof(float);
    const int4 *dwork = static_cast<const int4 *>(workspace);
    for (int c = 0; c < n_chunks; ++c) {
        if (bnd[c + 1] == bnd[c]) continue;
        const size_t t0 = static_cast<size_t>(bnd[c]), nt = static_cast<size_t>(bnd[c + 1] - bnd[c]);
        cudaEvent_t ev_in, ev_done;
        MLA_TRY(p.event(&ev_in), "event");
        MLA_TRY(p.event(&ev_done), "event");
        MLA_TRY(cudaMemcpyAsync(static_cast<char *>(q_bf16) + t0 * q_row, static_cast<const char *>(q_host) + t0 * q_row,
                                nt * q_row, cudaMemcpyHostToDevice, p.s_in),
                "query copy");
        MLA_TRY(cudaEventRecord(ev_in, p.s_in), "event record");
        // pieces share no data, so consecutive ones go to two streams and the
        // start of one overlaps the last CTAs of the other
        cudaStream_t cs = p.s_c[c & 1];
        MLA_TRY(cudaStreamWaitEvent(cs, ev_in, 0), "wait");
        const int n_items = static_cast<int>(off[c + 1] - off[c]);
        if (n_items > 0) MLA_TRY(mla::launch_dense_f8(a, dwork + off[c], n_items, tmap_kv, cs), "dense launch");
        MLA_TRY(cudaEventRecord(ev_done, cs), "event record");
        MLA_TRY(cudaStreamWaitEvent(p.s_out, ev_done, 0), "wait");
        MLA_TRY(cudaMemcpyAsync(static_cast<char *>(out_host) + t0 * o_row, static_cast<const char *>(out_bf16) + t0 * o_row,
                                nt * o_row, cudaMemcpyDeviceToHost, p.s_out),
                "output copy");
        if (lse_host)
            MLA_TRY(cudaMemcpyAsync(reinterpret_cast<char *>(lse_host) + t0 * l_row,
                                    reinterpret_cast<const char *>(lse) + t0 * l_row, nt * l_row,
                                    cudaMemcpyDeviceToHost, p.s_out),
                    "lse copy");
    }
    // the caller's stream resumes after the last copy back
    MLA_TRY(cudaEventRecord(ev_end, p.s_out), "event record");
    MLA_TRY(cudaStreamWaitEvent(stream, ev_end, 0), "wait");
#undef MLA_TRY
    return MLA_OK;
}

namespace {
mla_status_t check_indexer_args(const mla_seqs_t *seqs, const uint8_t *qi_e4m3, const float *w, int64_t w_token_stride,
                                const uint8_t *ki_e4m3, const float *ki_scale, int32_t topk, const int32_t *idx_out) {
    if (!qi_e4m3 || !w || !ki_e4m3 || !ki_scale || !idx_out)
        return fail(MLA_ERR_INVALID_ARG, "qi, w, ki, ki_scale and idx_out must be set");
    if (!aligned(qi_e4m3, 16) || !aligned(ki_e4m3, 16))
        return fail(MLA_ERR_INVALID_ARG, "qi and ki must be 16-byte aligned");
    if (!aligned(w, 16) || !aligned(ki_scale, 16))
        return fail(MLA_ERR_INVALID_ARG, "w and ki_scale must be 16-byte aligned");
    if (!aligned(idx_out, 4)) return fail(MLA_ERR_INVALID_ARG, "idx_out must be 4-byte aligned");
    if (w_token_stride < 0 || w_token_stride % 4 != 0)
        return fail(MLA_ERR_INVALID_ARG, "w_token_stride must be a non-negative multiple of 4");
    if (topk < 1 || topk > 2048) return fail(MLA_ERR_UNSUPPORTED, "topk must be in [1, 2048] (got %d)", topk);
    if (static_cast<int64_t>(seqs->cu_seqlens_q_host[seqs->batch]) * 64 > INT32_MAX)
        return fail(MLA_ERR_UNSUPPORTED, "too many query tokens for the indexer (Tq * 64 > 2^31 - 1)");
    return MLA_OK;
}

mla::IndexerArgs indexer_args(const mla_seqs_t *seqs, const uint8_t *qi_e4m3, const float *w, int64_t w_token_stride,
                              const uint8_t *ki_e4m3, const float *ki_scale, int32_t topk, int32_t *idx_out,
                              int32_t *dev_err) {
    mla::IndexerArgs a{};
    a.qi = qi_e4m3;
    a.w = w;
    a.w_stride = w_token_stride;
    a.ki = ki_e4m3;
    a.ki_scale = ki_scale;
    a.block_table = seqs->block_table;
    a.max_blocks = seqs->max_blocks_per_seq;
    a.num_blocks = seqs->num_blocks;
    a.cu_seqlens = seqs->cu_seqlens_q;
    a.prefix_lens = seqs->prefix_lens;
    a.batch = seqs->batch;
    a.topk = topk;
    a.idx_out = idx_out;
    a.dev_err = dev_err;
    a.total_q = seqs->cu_seqlens_q_host[seqs->batch];
    return a;
}
}  // namespace

mla_status_t mla_indexer_topk(const mla_seqs_t *seqs, const uint8_t *qi_e4m3, const float *w, int64_t w_token_stride,
                              const uint8_t *ki_e4m3, const float *ki_scale, int32_t topk, int32_t *idx_out,
                              void *workspace, size_t workspace_bytes, int32_t *dev_err, cudaStream_t stream) {
    g_err.clear();
    mla_status_t st = check_seqs(seqs);
    if (st != MLA_OK) return st;
    if ((st = check_indexer_args(seqs, qi_e4m3, w, w_token_stride, ki_e4m3, ki_scale, topk, idx_out)) != MLA_OK)
        return st;
    const int64_t tq = seqs->cu_seqlens_q_host[seqs->batch];
    if (tq == 0) return MLA_OK;
    const std::vector<int4> work = indexer_schedule(seqs, 0, tq);
    const size_t need = indexer_ws_bytes(work.size());
    if (!workspace || workspace_bytes < need || !aligned(workspace, 16))
        return fail(MLA_ERR_WORKSPACE, "indexer needs %zu workspace bytes (16-byte aligned), got %zu", need,
                    workspace ? workspace_bytes : 0);
    if (work.size() > static_cast<size_t>(INT32_MAX)) return fail(MLA_ERR_UNSUPPORTED, "too many query tokens");
    int4 *dwork = static_cast<int4 *>(workspace);
    cudaError_t e = cudaMemcpyAsync(dwork, work.data(), work.size() * sizeof(int4), cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return cuda_fail(e, "schedule upload");
    mla::IndexerArgs a = indexer_args(seqs, qi_e4m3, w, w_token_stride, ki_e4m3, ki_scale, topk, idx_out, dev_err);
    a.fail = reinterpret_cast<int32_t *>(static_cast<char *>(workspace) + round_up(work.size() * sizeof(int4), kWsAlign));
    CUtensorMap tmap_k, tmap_q;
    if (!encode_rows128(&tmap_k, ki_e4m3, static_cast<uint64_t>(seqs->num_blocks) * 256, 128) ||
        !encode_rows128(&tmap_q, qi_e4m3, static_cast<uint64_t>(tq) * 64, mla::kIdxTokensPerCta * 64))
        return fail(MLA_ERR_CUDA, "tensor map encoding for the indexer failed");
    if ((e = mla::launch_indexer_topk(a, dwork, static_cast<int>(work.size()), tmap_k, tmap_q, stream)) != cudaSuccess)
        return cuda_fail(e, "indexer launch");
    return MLA_OK;
}

mla_status_t mla_prefill_sparse(const mla_seqs_t *seqs, const void *q_bf16, int32_t num_heads,
                                const uint8_t *kv_e4m3, const float *kv_scale, float sm_scale, const int32_t *idx,
                                int32_t topk, void *out_bf16, float *lse, void *workspace, size_t workspace_bytes,
                                int32_t *dev_err, cudaStream_t stream) {
    (void)workspace;
    (void)workspace_bytes;
    g_err.clear();
    mla_status_t st = check_seqs(seqs);
    if (st != MLA_OK) return st;
    if (!heads_ok(num_heads)) return fail(MLA_ERR_UNSUPPORTED, "num_heads must be 16, 32, 64 or 128 (got %d)", num_heads);
    if ((st = check_attn_ptrs(q_bf16, kv_e4m3, kv_scale, out_bf16, lse, sm_scale)) != MLA_OK) return st;
    if (!idx || !aligned(idx, 4)) return fail(MLA_ERR_INVALID_ARG, "idx must be set and 4-byte aligned");
    if (topk < 1 || topk > 2048) return fail(MLA_ERR_UNSUPPORTED, "topk must be in [1, 2048] (got %d)", topk);
    const int64_t tq = seqs->cu_seqlens_q_host[seqs->batch];
    if (tq == 0) return MLA_OK;
    if (tq > INT32_MAX) return fail(MLA_ERR_UNSUPPORTED, "too many query tokens");
    mla::AttnArgs a = attn_args(seqs, q_bf16, num_heads, kv_e4m3, kv_scale, sm_scale, out_bf16, lse, dev_err);
    a.idx = idx;
    a.topk = topk;
    a.tok_begin = 0;
    a.tok_end = tq;
    cudaError_t e = mla::launch_sparse_f8(a, stream);
    if (e != cudaSuccess) return cuda_fail(e, "sparse launch");
    return MLA_OK;
}

mla_status_t mla_prefill_sparse_host(const mla_seqs_t *seqs, int32_t num_heads, float sm_scale,
                                     int64_t w_token_stride, int32_t topk, const mla_sparse_inputs_t *host_in,
                                     const mla_sparse_inputs_t *dev_in, const mla_sparse_outputs_t *host_out,
                                     const mla_sparse_outputs_t *dev_out, int32_t n_chunks, void *workspace,
                                     size_t workspace_bytes, int32_t *dev_err, cudaStream_t stream) {
    g_err.clear();
    mla_status_t st = check_seqs(seqs);
    if (st != MLA_OK) return st;
    if (!host_in || !dev_in || !host_out || !dev_out)
        return fail(MLA_ERR_INVALID_ARG, "host_in, dev_in, host_out and dev_out must be set");
    const mla_sparse_inputs_t &hi = *host_in, &di = *dev_in;
    const mla_sparse_outputs_t &ho = *host_out, &dO = *dev_out;
    if (!hi.q_bf16 || !hi.qi_e4m3 || !hi.w || !hi.kv_e4m3 || !hi.kv_scale || !hi.ki_e4m3 || !hi.ki_scale ||
        !ho.out_bf16 || !ho.idx)
        return fail(MLA_ERR_INVALID_ARG, "every host pointer but lse must be set");
    if (!ho.lse != !dO.lse) return fail(MLA_ERR_INVALID_ARG, "lse must be set on both sides or on neither");
    if (!heads_ok(num_heads)) return fail(MLA_ERR_UNSUPPORTED, "num_heads must be 16, 32, 64 or 128 (got %d)", num_heads);
    if ((st = check_indexer_args(seqs, di.qi_e4m3, di.w, w_token_stride, di.ki_e4m3, di.ki_scale, topk, dO.idx)) !=
        MLA_OK)
        return st;
    if ((st = check_attn_ptrs(di.q_bf16, di.kv_e4m3, di.kv_scale, dO.out_bf16, dO.lse, sm_scale)) != MLA_OK) return st;
    if (n_chunks < 1 || n_chunks > MLA_DENSE_HOST_MAX_CHUNKS)
        return fail(MLA_ERR_INVALID_ARG, "n_chunks must be in [1, %d] (got %d)", MLA_DENSE_HOST_MAX_CHUNKS, n_chunks);
    const int64_t tq = seqs->cu_seqlens_q_host[seqs->batch];
    if (tq == 0) return MLA_OK;
    // pieces on indexer group boundaries, each with its key chunk and work list
    std::vector<int64_t> bnd(static_cast<size_t>(n_chunks) + 1);
    bnd[0] = 0;
    bnd[n_chunks] = tq;
    for (int c = 1, b = 0; c < n_chunks; ++c) {
        const int64_t t = tq * c / n_chunks;
        while (b + 1 < seqs->batch && seqs->cu_seqlens_q_host[b + 1] <= t) ++b;
        const int64_t c0 = seqs->cu_seqlens_q_host[b];
        bnd[c] = std::max(bnd[c - 1], c0 + (t - c0) / mla::kIdxTokensPerCta * mla::kIdxTokensPerCta);
    }
    std::vector<int4> work;
    std::vector<size_t> off(static_cast<size_t>(n_chunks) + 1, 0);
    for (int c = 0; c < n_chunks; ++c) {
        if (bnd[c + 1] > bnd[c]) {
            const std::vector<int4> w = indexer_schedule(seqs, bnd[c], bnd[c + 1]);
            work.insert(work.end(), w.begin(), w.end());
        }
        off[c + 1] = work.size();
    }
    const size_t need = indexer_ws_bytes(work.size());
    if (!workspace || workspace_bytes < need || !aligned(workspace, 16))
        return fail(MLA_ERR_WORKSPACE, "sparse from host needs %zu workspace bytes (16-byte aligned), got %zu", need,
                    workspace ? workspace_bytes : 0);
    int4 *dwork = static_cast<int4 *>(workspace);
    int32_t *dfail = reinterpret_cast<int32_t *>(static_cast<char *>(workspace) +
                                                 round_up(work.size() * sizeof(int4), kWsAlign));
    mla::IndexerArgs ia = indexer_args(seqs, di.qi_e4m3, di.w, w_token_stride, di.ki_e4m3, di.ki_scale, topk, dO.idx,
                                       dev_err);
    mla::AttnArgs aa = attn_args(seqs, di.q_bf16, num_heads, di.kv_e4m3, di.kv_scale, sm_scale, dO.out_bf16, dO.lse,
                                 dev_err);
    aa.idx = dO.idx;
    aa.topk = topk;
    CUtensorMap tmap_k, tmap_q;
    if (!encode_rows128(&tmap_k, di.ki_e4m3, static_cast<uint64_t>(seqs->num_blocks) * 256, 128) ||
        !encode_rows128(&tmap_q, di.qi_e4m3, static_cast<uint64_t>(tq) * 64, mla::kIdxTokensPerCta * 64))
        return fail(MLA_ERR_CUDA, "tensor map encoding for the indexer failed");

    HostPipe p;
    cudaError_t e;
    cudaEvent_t ev_entry, ev_end;
#define MLA_TRY(x, what)                       \
    if ((e = (x)) != cudaSuccess) return cuda_fail(e, what)
    MLA_TRY(cudaStreamCreateWithFlags(&p.s_in, cudaStreamNonBlocking), "stream");
    MLA_TRY(cudaStreamCreateWithFlags(&p.s_out, cudaStreamNonBlocking), "stream");
    MLA_TRY(cudaStreamCreateWithFlags(&p.s_c[0], cudaStreamNonBlocking), "stream");
    MLA_TRY(cudaStreamCreateWithFlags(&p.s_c[1], cudaStreamNonBlocking), "stream");
    MLA_TRY(p.event(&ev_entry), "event");
    MLA_TRY(p.event(&ev_end), "event");
    MLA_TRY(cudaEventRecord(ev_entry, stream), "event record");
    for (cudaStream_t x : {p.s_in, p.s_out, p.s_c[0], p.s_c[1]}) MLA_TRY(cudaStreamWaitEvent(x, ev_entry, 0), "wait");
    // weights, caches and work lists first, then qi and q piece by piece
    const size_t rows_kv = static_cast<size_t>(seqs->num_blocks) * 256;
    const size_t w_floats = w_token_stride ? static_cast<size_t>(tq - 1) * static_cast<size_t>(w_token_stride) + 64 : 64;
    MLA_TRY(cudaMemcpyAsync(di.w, hi.w, w_floats * sizeof(float), cudaMemcpyHostToDevice, p.s_in), "weight copy");
    MLA_TRY(cudaMemcpyAsync(di.ki_e4m3, hi.ki_e4m3, rows_kv * 128, cudaMemcpyHostToDevice, p.s_in), "key copy");
    MLA_TRY(cudaMemcpyAsync(di.ki_scale, hi.ki_scale, rows_kv * sizeof(float), cudaMemcpyHostToDevice, p.s_in),
            "key scale copy");
    MLA_TRY(cudaMemcpyAsync(di.kv_e4m3, hi.kv_e4m3, rows_kv * 576, cudaMemcpyHostToDevice, p.s_in), "cache copy");
    MLA_TRY(cudaMemcpyAsync(di.kv_scale, hi.kv_scale, rows_kv * sizeof(float), cudaMemcpyHostToDevice, p.s_in),
            "cache scale copy");
    if (!work.empty())
        MLA_TRY(cudaMemcpyAsync(dwork, work.data(), work.size() * sizeof(int4), cudaMemcpyHostToDevice, p.s_in),
                "schedule upload");
    const size_t q_row = static_cast<size_t>(num_heads) * 576 * 2, qi_row = 64 * 128,
                 o_row = static_cast<size_t>(num_heads) * 512 * 2, l_row = static_cast<size_t>(num_heads) * sizeof(float),
                 i_row = static_cast<size_t>(topk) * sizeof(int32_t);
    auto at = [](const void *base, size_t bytes) { return static_cast<char *>(const_cast<void *>(base)) + bytes; };
    for (int c = 0; c < n_chunks; ++c) {
        if (bnd[c + 1] == bnd[c]) continue;
        const size_t t0 = static_cast<size_t>(bnd[c]), nt = static_cast<size_t>(bnd[c + 1] - bnd[c]);
        cudaEvent_t ev_in, ev_done;
        MLA_TRY(p.event(&ev_in), "event");
        MLA_TRY(p.event(&ev_done), "event");
        MLA_TRY(cudaMemcpyAsync(at(di.qi_e4m3, t0 * qi_row), at(hi.qi_e4m3, t0 * qi_row), nt * qi_row,
                                cudaMemcpyHostToDevice, p.s_in),
                "indexer query copy");
        MLA_TRY(cudaMemcpyAsync(at(di.q_bf16, t0 * q_row), at(hi.q_bf16, t0 * q_row), nt * q_row,
                                cudaMemcpyHostToDevice, p.s_in),
                "query copy");
        MLA_TRY(cudaEventRecord(ev_in, p.s_in), "event record");
        // pieces share no data (each writes its own index and output rows), so
        // consecutive ones go to two streams
        cudaStream_t cs = p.s_c[c & 1];
        MLA_TRY(cudaStreamWaitEvent(cs, ev_in, 0), "wait");
        const int n_items = static_cast<int>(off[c + 1] - off[c]);
        mla::IndexerArgs pa = ia;
        pa.fail = dfail + off[c];
        if (n_items > 0)
            MLA_TRY(mla::launch_indexer_topk(pa, dwork + off[c], n_items, tmap_k, tmap_q, cs), "indexer launch");
        mla::AttnArgs sa = aa;
        sa.tok_begin = bnd[c];
        sa.tok_end = bnd[c + 1];
        MLA_TRY(mla::launch_sparse_f8(sa, cs), "sparse launch");
        MLA_TRY(cudaEventRecord(ev_done, cs), "event record");
        MLA_TRY(cudaStreamWaitEvent(p.s_out, ev_done, 0), "wait");
        MLA_TRY(cudaMemcpyAsync(at(ho.out_bf16, t0 * o_row), at(dO.out_bf16, t0 * o_row), nt * o_row,
                                cudaMemcpyDeviceToHost, p.s_out),
                "output copy");
        if (ho.lse)
            MLA_TRY(cudaMemcpyAsync(at(ho.lse, t0 * l_row), at(dO.lse, t0 * l_row), nt * l_row, cudaMemcpyDeviceToHost,
                                    p.s_out),
                    "lse copy");
        MLA_TRY(cudaMemcpyAsync(at(ho.idx, t0 * i_row), at(dO.idx, t0 * i_row), nt * i_row, cudaMemcpyDeviceToHost,
                                p.s_out),
                "index copy");
    }
    MLA_TRY(cudaEventRecord(ev_end, p.s_out), "event record");
    MLA_TRY(cudaStreamWaitEvent(stream, ev_end, 0), "wait");
#undef MLA_TRY
    return MLA_OK;
}

mla_status_t mla_prefill_dense_ds(const mla_seqs_t *seqs, const void *q_bf16, int32_t num_heads, const uint8_t *kv_ds,
                                  float sm_scale, void *out_bf16, float *lse, void *workspace, size_t workspace_bytes,
                                  int32_t *dev_err, cudaStream_t stream) {
    g_err.clear();
    mla_status_t st = check_seqs(seqs);
    if (st != MLA_OK) return st;
    if (!heads_ok(num_heads)) return fail(MLA_ERR_UNSUPPORTED, "num_heads must be 16, 32, 64 or 128 (got %d)", num_heads);
    // the row format carries its own scales: any 4-byte-aligned stand-in passes the scale check
    if ((st = check_attn_ptrs(q_bf16, kv_ds, reinterpret_cast<const float *>(kv_ds), out_bf16, lse, sm_scale)) != MLA_OK)
        return st;
    const DsPlan p = ds_plan(seqs, num_heads);
    if (p.work.empty()) return MLA_OK;
    if (!workspace || workspace_bytes < p.bytes || !aligned(workspace, kWsAlign))
        return fail(MLA_ERR_WORKSPACE, "dense (656-byte rows) needs %zu workspace bytes (256-byte aligned), got %zu",
                    p.bytes, workspace ? workspace_bytes : 0);
    if (static_cast<int64_t>(p.work.size()) > INT32_MAX || p.rows > INT32_MAX / 36)
        return fail(MLA_ERR_UNSUPPORTED, "too many tiles");
    char *ws = static_cast<char *>(workspace);
    std::vector<char> head(p.off_rows, 0);
    std::memcpy(head.data(), p.work.data(), p.work.size() * sizeof(int4));
    std::memcpy(head.data() + p.off_ints, p.base.data(), p.base.size() * sizeof(int32_t));
    std::memcpy(head.data() + p.off_ints + p.base.size() * sizeof(int32_t), p.ctx.data(), p.ctx.size() * sizeof(int32_t));
    cudaError_t e = cudaMemcpyAsync(ws, head.data(), head.size(), cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return cuda_fail(e, "schedule upload");
    mla::AttnArgs a = attn_args(seqs, q_bf16, num_heads, kv_ds, nullptr, sm_scale, out_bf16, lse, dev_err);
    a.conv_base = reinterpret_cast<const int32_t *>(ws + p.off_ints);
    a.conv_ctx = a.conv_base + seqs->batch;
    a.kconv = reinterpret_cast<__half *>(ws + p.off_rows);
    a.kmeta = reinterpret_cast<uint8_t *>(ws + p.off_meta);
    CUtensorMap tmap;
    const cuuint64_t dims[2] = {576, static_cast<cuuint64_t>(p.rows)}, strides[1] = {1152};
    const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(mla::kDsTileKeys)};
    if (!encode_16bit(&tmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, a.kconv, 2, dims, strides, box))
        return fail(MLA_ERR_CUDA, "tensor map encoding failed");
    e = mla::launch_dense_ds(a, reinterpret_cast<const int4 *>(ws), static_cast<int>(p.work.size()), p.rows, tmap,
                             stream);
    if (e != cudaSuccess) return cuda_fail(e, "dense launch");
    return MLA_OK;
}

mla_status_t mla_prefill_mha(const mla_seqs_t *seqs, const void *q_bf16, int32_t num_heads, const void *w_ukv_bf16,
                             const uint8_t *kv_e4m3, const float *kv_scale, float sm_scale, void *out_bf16,
                             float *lse, void *workspace, size_t workspace_bytes, int32_t *dev_err,
                             cudaStream_t stream) {
    g_err.clear();
    mla_status_t st = check_seqs(seqs);
    if (st != MLA_OK) return st;
    if (!heads_ok(num_heads)) return fail(MLA_ERR_UNSUPPORTED, "num_heads must be 16, 32, 64 or 128 (got %d)", num_heads);
    if ((st = check_attn_ptrs(q_bf16, kv_e4m3, kv_scale, out_bf16, lse, sm_scale)) != MLA_OK) return st;
    if (!w_ukv_bf16 || !aligned(w_ukv_bf16, 16)) return fail(MLA_ERR_INVALID_ARG, "w_ukv must be set and 16-byte aligned");
    const MhaPlan p = mha_plan(seqs, num_heads);
    if (p.at.empty()) return MLA_OK;
    if (!workspace || workspace_bytes < p.bytes || !aligned(workspace, kWsAlign))
        return fail(MLA_ERR_WORKSPACE, "mha needs %zu workspace bytes (256-byte aligned), got %zu", p.bytes,
                    workspace ? workspace_bytes : 0);
    const int64_t tq = seqs->cu_seqlens_q_host[seqs->batch];
    if (static_cast<int64_t>(num_heads) * p.R > INT32_MAX || tq > INT32_MAX ||
        static_cast<int64_t>(p.at.size() / 2) * num_heads > INT32_MAX)
        return fail(MLA_ERR_UNSUPPORTED, "batch too large for the non-absorbed path");
    char *ws = static_cast<char *>(workspace);
    std::vector<int4> lists(p.off_kn / sizeof(int4), make_int4(0, 0, 0, 0));
    std::copy(p.at.begin(), p.at.end(), lists.begin() + p.off_at / sizeof(int4));
    std::copy(p.up.begin(), p.up.end(), lists.begin() + p.off_up / sizeof(int4));
    cudaError_t e = cudaMemcpyAsync(ws, lists.data(), p.off_kn, cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) return cuda_fail(e, "schedule upload");

    mla::MhaArgs a{};
    a.q = static_cast<const __nv_bfloat16 *>(q_bf16);
    a.kv = kv_e4m3;
    a.kv_scale = kv_scale;
    a.block_table = seqs->block_table;
    a.max_blocks = seqs->max_blocks_per_seq;
    a.num_blocks = seqs->num_blocks;
    a.kn = reinterpret_cast<__half *>(ws + p.off_kn);
    a.v = reinterpret_cast<__half *>(ws + p.off_v);
    a.kr = reinterpret_cast<__half *>(ws + p.off_kr);
    a.R = p.R;
    a.out = static_cast<__nv_bfloat16 *>(out_bf16);
    a.lse = lse;
    a.H = num_heads;
    // heads per up-projection CTA: the fewest waves of CTAs times the work of one,
    // counting the decode of a CTA's 128 rows as two heads' worth
    {
        int sms = 148;
        int dev = 0;
        if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        const int64_t n_up = static_cast<int64_t>(p.up.size());
        int64_t best = -1;
        for (int g = 8; g <= num_heads; g *= 2) {
            const int64_t ctas = n_up * (num_heads / g), waves = (ctas + sms - 1) / sms;
            const int64_t cost = waves * (g + 2);
            if (best < 0 || cost < best) {
                best = cost;
                a.up_heads = g;
            }
        }
    }
    a.sm_scale_log2 = sm_scale * 1.4426950408889634f;
    a.dev_err = dev_err;
    a.total_q = tq;

    const cuuint64_t H = static_cast<cuuint64_t>(num_heads), R = static_cast<cuuint64_t>(p.R);
    CUtensorMap tw, tkn, tkr, tv;
    const cuuint64_t w_dims[2] = {512, H * 256}, w_str[1] = {1024};
    const cuuint32_t w_box[2] = {64, 128};
    const cuuint64_t kv_dims[2] = {128, H * R}, kv_str[1] = {256};
    const cuuint64_t kr_dims[2] = {64, R}, kr_str[1] = {128};
    const cuuint32_t k_box[2] = {64, 64};
    const CUtensorMapDataType BF = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, F16 = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    if (!encode_16bit(&tw, BF, w_ukv_bf16, 2, w_dims, w_str, w_box) ||
        !encode_16bit(&tkn, F16, a.kn, 2, kv_dims, kv_str, k_box) ||
        !encode_16bit(&tv, F16, a.v, 2, kv_dims, kv_str, k_box) ||
        !encode_16bit(&tkr, F16, a.kr, 2, kr_dims, kr_str, k_box))
        return fail(MLA_ERR_CUDA, "tensor map encoding failed");
    e = mla::launch_mha_up(a, reinterpret_cast<const int4 *>(ws + p.off_up), static_cast<int>(p.up.size()), tw, stream);
    if (e != cudaSuccess) return cuda_fail(e, "mha up-projection launch");
    e = mla::launch_mha_attn(a, reinterpret_cast<const int4 *>(ws + p.off_at), static_cast<int>(p.at.size() / 2), tkn,
                             tkr, tv, stream);
    if (e != cudaSuccess) return cuda_fail(e, "mha attention launch");
    return MLA_OK;
}

mla_status_t mla_prefill_sparse_ds(const mla_seqs_t *seqs, const void *q_bf16, int32_t num_heads, const uint8_t *kv_ds,
                                   float sm_scale, const int32_t *idx, int32_t topk, void *out_bf16, float *lse,
                                   int32_t *dev_err, cudaStream_t stream) {
    g_err.clear();
    mla_status_t st = check_seqs(seqs);
    if (st != MLA_OK) return st;
    if (!heads_ok(num_heads)) return fail(MLA_ERR_UNSUPPORTED, "num_heads must be 16, 32, 64 or 128 (got %d)", num_heads);
    if ((st = check_attn_ptrs(q_bf16, kv_ds, reinterpret_cast<const float *>(kv_ds), out_bf16, lse, sm_scale)) != MLA_OK)
        return st;
    if (!idx || !aligned(idx, 4)) return fail(MLA_ERR_INVALID_ARG, "idx must be set and 4-byte aligned");
    if (topk < 1 || topk > 2048) return fail(MLA_ERR_UNSUPPORTED, "topk must be in [1, 2048] (got %d)", topk);
    const int64_t tq = seqs->cu_seqlens_q_host[seqs->batch];
    if (tq == 0) return MLA_OK;
    if (tq > INT32_MAX) return fail(MLA_ERR_UNSUPPORTED, "too many query tokens");
    mla::AttnArgs a = attn_args(seqs, q_bf16, num_heads, kv_ds, nullptr, sm_scale, out_bf16, lse, dev_err);
    a.idx = idx;
    a.topk = topk;
    a.tok_begin = 0;
    a.tok_end = tq;
    const cudaError_t e = mla::launch_sparse_ds(a, stream);
    if (e != cudaSuccess) return cuda_fail(e, "sparse launch");
    return MLA_OK;
}

mla_status_t mla_kv_append(const mla_seqs_t *seqs, const void *latent_bf16, const void *kidx_bf16,
                           uint8_t *kv_e4m3, float *kv_scale, uint8_t *ki_e4m3, float *ki_scale,
                           int32_t *dev_err, cudaStream_t stream) {
    g_err.clear();
    mla_status_t st = check_seqs(seqs);
    if (st != MLA_OK) return st;
    if (!latent_bf16 || !kv_e4m3 || !kv_scale) return fail(MLA_ERR_INVALID_ARG, "latent, kv and kv_scale must be set");
    if (!aligned(latent_bf16, 16) || !aligned(kv_e4m3, 16))
        return fail(MLA_ERR_INVALID_ARG, "latent and kv must be 16-byte aligned");
    if (!aligned(kv_scale, 4)) return fail(MLA_ERR_INVALID_ARG, "kv_scale must be 4-byte aligned");
    if (kidx_bf16) {
        if (!ki_e4m3 || !ki_scale) return fail(MLA_ERR_INVALID_ARG, "ki and ki_scale must be set with kidx");
        if (!aligned(kidx_bf16, 16) || !aligned(ki_e4m3, 16))
            return fail(MLA_ERR_INVALID_ARG, "kidx and ki must be 16-byte aligned");
        if (!aligned(ki_scale, 4)) return fail(MLA_ERR_INVALID_ARG, "ki_scale must be 4-byte aligned");
    }
    const int64_t tq = seqs->cu_seqlens_q_host[seqs->batch];
    if (tq == 0) return MLA_OK;
    if (tq > INT32_MAX) return fail(MLA_ERR_UNSUPPORTED, "too many new tokens");
    mla::AppendArgs a{};
    a.latent = static_cast<const __nv_bfloat16 *>(latent_bf16);
    a.kidx = static_cast<const __nv_bfloat16 *>(kidx_bf16);
    a.kv = kv_e4m3;
    a.kv_scale = kv_scale;
    a.ki = kidx_bf16 ? ki_e4m3 : nullptr;
    a.ki_scale = kidx_bf16 ? ki_scale : nullptr;
    a.block_table = seqs->block_table;
    a.max_blocks = seqs->max_blocks_per_seq;
    a.num_blocks = seqs->num_blocks;
    a.cu_seqlens = seqs->cu_seqlens_q;
    a.prefix_lens = seqs->prefix_lens;
    a.batch = seqs->batch;
    a.n_tokens = tq;
    a.dev_err = dev_err;
    const cudaError_t e = mla::launch_kv_append(a, stream);
    if (e != cudaSuccess) return cuda_fail(e, "kv append launch");
    return MLA_OK;
}

mla_status_t mla_merge_attn(int32_t n_parts, const void *const *outs_bf16, const float *const *lses, int64_t rows,
                            void *out_bf16, float *lse_out, cudaStream_t stream) {
    g_err.clear();
    if (n_parts < 1 || n_parts > MLA_MERGE_MAX_PARTS)
        return fail(MLA_ERR_UNSUPPORTED, "n_parts must be in [1, %d] (got %d)", MLA_MERGE_MAX_PARTS, n_parts);
    if (!outs_bf16 || !lses || !out_bf16) return fail(MLA_ERR_INVALID_ARG, "outs, lses and out must be set");
    if (rows < 0) return fail(MLA_ERR_INVALID_ARG, "rows must be >= 0");
    if (!aligned(out_bf16, 16)) return fail(MLA_ERR_INVALID_ARG, "out must be 16-byte aligned");
    if (lse_out && !aligned(lse_out, 4)) return fail(MLA_ERR_INVALID_ARG, "lse must be 4-byte aligned");
    mla::MergeArgs a{};
    for (int i = 0; i < n_parts; ++i) {
        if (!outs_bf16[i] || !lses[i]) return fail(MLA_ERR_INVALID_ARG, "part %d: out and lse must be set", i);
        if (!aligned(outs_bf16[i], 16) || !aligned(lses[i], 4))
            return fail(MLA_ERR_INVALID_ARG, "part %d: out must be 16-byte and lse 4-byte aligned", i);
        a.outs[i] = static_cast<const uint4 *>(outs_bf16[i]);
        a.lses[i] = lses[i];
    }
    if (rows == 0) return MLA_OK;
    if ((rows + 7) / 8 > INT32_MAX) return fail(MLA_ERR_UNSUPPORTED, "too many rows");
    a.n_parts = n_parts;
    a.rows = rows;
    a.out = static_cast<uint4 *>(out_bf16);
    a.lse = lse_out;
    const cudaError_t e = mla::launch_merge(a, stream);
    if (e != cudaSuccess) return cuda_fail(e, "merge launch");
    return MLA_OK;
}

}  // extern "C"

// Helpers shared with the allocation-free dense entry point (dense_noalloc.cu).
namespace mla {
bool encode_kv_tmap(CUtensorMap *map, const uint8_t *kv, int32_t num_blocks) {
    // rows of 576 e4m3 codes (512 latent + 64 RoPE); 128-row boxes (a dense key tile)
    // start at multiples of 128 and never straddle a 256-row page
    return num_blocks > 0 && encode_u8_rows(map, kv, 576, static_cast<uint64_t>(num_blocks) * 256, 128);
}
mla_status_t check_dense_args(const mla_seqs_t *seqs, const void *q, int32_t H, const uint8_t *kv,
                              const float *kv_scale, const void *out, const float *lse, float sm_scale) {
    g_err.clear();
    mla_status_t st = check_seqs(seqs);
    if (st != MLA_OK) return st;
    if (!heads_ok(H)) return fail(MLA_ERR_UNSUPPORTED, "num_heads must be 16, 32, 64 or 128 (got %d)", H);
    return check_attn_ptrs(q, kv, kv_scale, out, lse, sm_scale);
}
mla_status_t report(mla_status_t s, const char *msg) { return fail(s, "%s", msg); }
AttnArgs make_attn_args(const mla_seqs_t *s, const void *q, int32_t H, const uint8_t *kv, const float *kv_scale,
                        float sm_scale, void *out, float *lse, int32_t *dev_err) {
    return attn_args(s, q, H, kv, kv_scale, sm_scale, out, lse, dev_err);
}
}  // namespace mla

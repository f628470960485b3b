// Indexer score and exact top-k selection (sm_103a).
//
// score(t,s) = sigmaI_s * sum_h w[t,h] * max(0, q_{t,h} . k_s), s <= position(t)
// (GLM-5.3 Teil 2, section "Warum nicht TP oder DP?": the indexer scores every
// earlier token to pick 2,048; footnote 3: keys are 128 FP8 values + a 4-byte
// scale). Scores go to an fp32 workspace row per token; the top-k kernel then
// finds, per token, the exact k-th largest of the 64-bit keys
//   (order-preserving bits of the score) << 32 | (0xFFFFFFFF - s)
// which are all distinct, so "score descending, lower position first" is a
// total order, and writes the positions whose key is >= that threshold in
// ascending position order.
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"

namespace mla {
namespace idx {

constexpr int NT = 256;             // 8 warps = 8 query tokens per CTA
constexpr int KT = 128;             // keys per smem tile
constexpr int kRow = kDidx;         // 128 B per e4m3 key row

__device__ __forceinline__ uint32_t sw128(uint32_t base, int row, int chunk) {
    return base + row * 128 + ((chunk ^ (row & 7)) << 4);
}

__device__ __forceinline__ int find_seq(const int32_t *cu, int batch, int64_t t) {
    int lo = 0, hi = batch - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(cu + mid) <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
}

__global__ void __launch_bounds__(NT, 1) score_kernel(const IndexerArgs a, const int4 *__restrict__ work) {
    __shared__ __align__(128) uint8_t sk[2][KT * kRow];
    __shared__ int64_t srow[2][KT];
    __shared__ float ssig[2][KT];

    const int4 it = work[blockIdx.x];
    const int b = it.x, i0 = it.y, ntok = it.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t4 = lane & 3;
    const int q0 = __ldg(a.cu_seqlens + b), P = __ldg(a.prefix_lens + b);
    const int32_t *bt = a.block_table + static_cast<int64_t>(b) * a.max_blocks;
    const int k_lo = it.w * kIdxKeyChunk;
    const int k_hi = min(k_lo + kIdxKeyChunk, P + i0 + ntok);       // exclusive
    const bool tok_ok = warp < ntok;
    const int64_t tg = static_cast<int64_t>(q0) + i0 + warp;        // global token of this warp
    const int limit = P + i0 + warp;                                // last visible position

    // this token's 64 heads x 128 dims as m16n8k32 B fragments (n = head, k = dim)
    uint32_t bq[8][4][2];
    float wv[8][2];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
        const int head = 8 * nt + g;
        const uint8_t *qrow = a.qi + (tg * kHidx + head) * kDidx + 4 * t4;
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
            bq[nt][ks][0] = tok_ok ? __ldg(reinterpret_cast<const uint32_t *>(qrow + 32 * ks)) : 0u;
            bq[nt][ks][1] = tok_ok ? __ldg(reinterpret_cast<const uint32_t *>(qrow + 32 * ks + 16)) : 0u;
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) wv[nt][j] = tok_ok ? __ldg(a.w + tg * a.w_stride + 8 * nt + 2 * t4 + j) : 0.f;
    }

    const int n_tiles = (k_hi - k_lo + KT - 1) / KT;
    auto meta = [&](int buf, int tile) {
        const int k = threadIdx.x;
        if (k < KT) {
            const int pos = k_lo + tile * KT + k;
            const int64_t row = pos < k_hi ? cache_row(bt, a.max_blocks, a.num_blocks, pos, a.dev_err) : -1;
            srow[buf][k] = row;
            ssig[buf][k] = row >= 0 ? __ldg(a.ki_scale + row) : 0.f;
        }
    };
    auto issue = [&](int buf) {
        const uint32_t base = smem_u32(sk[buf]);
#pragma unroll
        for (int i = 0; i < (KT * kRow / 16) / NT; ++i) {
            const int c = threadIdx.x + NT * i;
            const int key = c >> 3, part = c & 7;
            const int64_t row = srow[buf][key];
            cp_async16(sw128(base, key, part), a.ki + (row >= 0 ? row : 0) * kRow + part * 16, row >= 0 ? 16 : 0);
        }
        cp_async_commit();
    };

    if (n_tiles > 0) {
        meta(0, 0);
        __syncthreads();
        issue(0);
    }
    for (int j = 0; j < n_tiles; ++j) {
        const int buf = j & 1;
        cp_async_wait<0>();
        __syncthreads();
        if (j + 1 < n_tiles) meta(buf ^ 1, j + 1);
        __syncthreads();
        if (j + 1 < n_tiles) issue(buf ^ 1);

        const uint32_t base = smem_u32(sk[buf]);
        const int tile0 = k_lo + j * KT;
#pragma unroll 1
        for (int st = 0; st < KT / 16; ++st) {
            if (!tok_ok || tile0 + 16 * st > limit) break;
            uint32_t af[4][4];
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                ldsm_x4(sw128(base, 16 * st + (lane & 7) + (((lane >> 3) & 1) << 3), 2 * ks + (lane >> 4)),
                        af[ks][0], af[ks][1], af[ks][2], af[ks][3]);
            float e0 = 0.f, e1 = 0.f;
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                float c[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_e4m3_16832(c, af[ks][0], af[ks][1], af[ks][2], af[ks][3], bq[nt][ks][0], bq[nt][ks][1]);
                e0 = fmaf(wv[nt][0], fmaxf(c[0], 0.f), e0);
                e0 = fmaf(wv[nt][1], fmaxf(c[1], 0.f), e0);
                e1 = fmaf(wv[nt][0], fmaxf(c[2], 0.f), e1);
                e1 = fmaf(wv[nt][1], fmaxf(c[3], 0.f), e1);
            }
            e0 += __shfl_xor_sync(0xffffffffu, e0, 1);
            e1 += __shfl_xor_sync(0xffffffffu, e1, 1);
            e0 += __shfl_xor_sync(0xffffffffu, e0, 2);
            e1 += __shfl_xor_sync(0xffffffffu, e1, 2);
            if (t4 < 2) {
                const int kk = 16 * st + g + 8 * t4;
                const int pos = tile0 + kk;
                if (pos <= limit && pos < k_hi) {
                    const float v = t4 == 0 ? e0 : e1;
                    a.scores[tg * a.score_stride + pos] = srow[buf][kk] >= 0 ? ssig[buf][kk] * v : -INFINITY;
                }
            }
        }
    }
}

// ---------------------------------------------------------------------------
// exact top-k over one score row per token
// ---------------------------------------------------------------------------
constexpr int TK_NT = 1024;
constexpr int TK_CAP = 6144;
constexpr int TK_SMEM = TK_CAP * 8 + 4096 * 4;

__device__ __forceinline__ uint32_t ord_f32(float x) {
    if (x != x) return 0u;          // NaN ranks below everything
    if (x == 0.f) x = 0.f;          // -0 and +0 tie
    const uint32_t u = __float_as_uint(x);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ uint64_t key64(float sc, int s) {
    return (static_cast<uint64_t>(ord_f32(sc)) << 32) | static_cast<uint32_t>(0xFFFFFFFFu - static_cast<uint32_t>(s));
}
__device__ __forceinline__ bool prefix_match(uint64_t k, uint64_t prefix, int bits) {
    return bits == 0 || (k >> (64 - bits)) == (prefix >> (64 - bits));
}

struct TkState {
    uint64_t prefix;
    int bits;
    uint32_t krem, cnt, ncand;
    uint32_t wtot[32];
    uint32_t base;
};

// Pick the digit holding the krem-th largest key; warp 0 only.
__device__ void pick_digit(const uint32_t *hist, int width, int shift, TkState &st) {
    const int lane = threadIdx.x & 31;
    const int nb = 1 << width, per = nb / 32;
    uint32_t sum = 0;
    for (int d = lane * per; d < lane * per + per; ++d) sum += hist[d];
    // above = sum over lanes with higher bins
    uint32_t incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_down_sync(0xffffffffu, incl, o);
        if (lane + o < 32) incl += v;
    }
    const uint32_t above = incl - sum;
    const uint32_t krem = st.krem;
    if (above < krem && krem <= above + sum) {
        uint32_t acc = above;
        for (int d = lane * per + per - 1; d >= lane * per; --d) {
            if (acc + hist[d] >= krem) {
                st.prefix |= static_cast<uint64_t>(d) << shift;
                st.bits += width;
                st.krem = krem - acc;
                st.cnt = hist[d];
                break;
            }
            acc += hist[d];
        }
    }
}

__global__ void __launch_bounds__(TK_NT, 1) topk_kernel(const IndexerArgs a) {
    extern __shared__ __align__(16) uint8_t tk_raw[];
    uint64_t *cand = reinterpret_cast<uint64_t *>(tk_raw);
    uint32_t *hist = reinterpret_cast<uint32_t *>(tk_raw + TK_CAP * 8);
    __shared__ TkState st;

    const int64_t t = blockIdx.x;
    const int b = find_seq(a.cu_seqlens, a.batch, t);
    const int64_t n = static_cast<int64_t>(__ldg(a.prefix_lens + b)) + (t - __ldg(a.cu_seqlens + b)) + 1;
    int32_t *out = a.idx_out + t * a.topk;
    const int tid = threadIdx.x;
    if (n <= a.topk) {
        for (int j = tid; j < a.topk; j += TK_NT) out[j] = j < n ? j : -1;
        return;
    }
    const float *row = a.scores + t * a.score_stride;
    const int widths[6] = {12, 12, 8, 12, 12, 8};
    if (tid == 0) {
        st.prefix = 0;
        st.bits = 0;
        st.krem = static_cast<uint32_t>(a.topk);
        st.cnt = static_cast<uint32_t>(n);
    }
    __syncthreads();
    int di = 0;
    // phase A: digit passes over the global row until the candidates fit in smem
    while (di < 6 && st.bits < 64 && st.cnt > TK_CAP) {
        const int width = widths[di++], shift = 64 - st.bits - width;
        const uint64_t prefix = st.prefix;
        const int bits = st.bits;
        for (int d = tid; d < (1 << width); d += TK_NT) hist[d] = 0;
        __syncthreads();
        for (int64_t s = tid; s < n; s += TK_NT) {
            const uint64_t k = key64(row[s], static_cast<int>(s));
            if (prefix_match(k, prefix, bits)) atomicAdd(&hist[(k >> shift) & ((1u << width) - 1)], 1u);
        }
        __syncthreads();
        if (tid < 32) pick_digit(hist, width, shift, st);
        __syncthreads();
    }
    // phase B: compact the keys matching the prefix into smem
    if (st.bits < 64) {
        if (tid == 0) st.ncand = 0;
        __syncthreads();
        const uint64_t prefix = st.prefix;
        const int bits = st.bits;
        for (int64_t s = tid; s < n; s += TK_NT) {
            const uint64_t k = key64(row[s], static_cast<int>(s));
            if (prefix_match(k, prefix, bits)) cand[atomicAdd(&st.ncand, 1u)] = k;
        }
        __syncthreads();
        // phase C: remaining digits in smem
        const uint32_t nc = st.ncand;
        while (di < 6 && st.bits < 64) {
            const int width = widths[di++], shift = 64 - st.bits - width;
            const uint64_t pf = st.prefix;
            const int bb = st.bits;
            for (int d = tid; d < (1 << width); d += TK_NT) hist[d] = 0;
            __syncthreads();
            for (uint32_t i = tid; i < nc; i += TK_NT) {
                const uint64_t k = cand[i];
                if (prefix_match(k, pf, bb)) atomicAdd(&hist[(k >> shift) & ((1u << width) - 1)], 1u);
            }
            __syncthreads();
            if (tid < 32) pick_digit(hist, width, shift, st);
            __syncthreads();
        }
    }
    // every digit must have been picked (the counts guarantee it); if not,
    // report instead of writing an arbitrary selection
    if (st.bits != 64) {
        if (tid == 0) set_dev_err(a.dev_err, MLA_DEVERR_INTERNAL);
        for (int j = tid; j < a.topk; j += TK_NT) out[j] = -1;
        return;
    }
    // phase D: positions with key >= threshold, in ascending position order
    const uint64_t kth = st.prefix;
    const int warp = tid >> 5, lane = tid & 31;
    if (tid == 0) st.base = 0;
    __syncthreads();
    for (int64_t c0 = 0; c0 < n; c0 += TK_NT) {
        const int64_t s = c0 + tid;
        const bool f = s < n && key64(row[s], static_cast<int>(s)) >= kth;
        const uint32_t m = __ballot_sync(0xffffffffu, f);
        if (lane == 0) st.wtot[warp] = __popc(m);
        __syncthreads();
        uint32_t off = st.base;
        for (int w = 0; w < warp; ++w) off += st.wtot[w];
        if (f) {
            const uint32_t o = off + __popc(m & ((1u << lane) - 1u));
            if (o < static_cast<uint32_t>(a.topk)) out[o] = static_cast<int32_t>(s);
        }
        __syncthreads();
        if (tid == 0) {
            uint32_t tot = 0;
            for (int w = 0; w < 32; ++w) tot += st.wtot[w];
            st.base += tot;
        }
        __syncthreads();
    }
}

}  // namespace idx

cudaError_t launch_indexer_scores(const IndexerArgs &a, const int4 *work, int n_work, cudaStream_t st) {
    if (n_work > 0) idx::score_kernel<<<n_work, idx::NT, 0, st>>>(a, work);
    return cudaGetLastError();
}

cudaError_t launch_topk(const IndexerArgs &a, int64_t n_tokens, cudaStream_t st) {
    cudaError_t e = cudaFuncSetAttribute(idx::topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, idx::TK_SMEM);
    if (e != cudaSuccess) return e;
    if (n_tokens > 0) idx::topk_kernel<<<static_cast<unsigned>(n_tokens), idx::TK_NT, idx::TK_SMEM, st>>>(a);
    return cudaGetLastError();
}

}  // namespace mla

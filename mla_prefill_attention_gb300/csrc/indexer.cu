// Exact top-k selection over the indexer's scores (sm_103a); the scores come
// from indexer_tc.cu.
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

__device__ __forceinline__ int find_seq(const int32_t *cu, int batch, int64_t t) {
    int lo = 0, hi = batch - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(cu + mid) <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
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

cudaError_t launch_topk(const IndexerArgs &a, int64_t n_tokens, cudaStream_t st) {
    cudaError_t e = cudaFuncSetAttribute(idx::topk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, idx::TK_SMEM);
    if (e != cudaSuccess) return e;
    if (n_tokens > 0) idx::topk_kernel<<<static_cast<unsigned>(n_tokens), idx::TK_NT, idx::TK_SMEM, st>>>(a);
    return cudaGetLastError();
}

}  // namespace mla

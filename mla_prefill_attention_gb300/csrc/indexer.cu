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
constexpr int TK_SEL = 2048;            // selected positions (max topk), sorted before the write
constexpr int TK_SMEM = TK_CAP * 8 + 4096 * 4 + TK_SEL * 4;

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

// Exclusive block-wide prefix sum of v (every thread of the block calls it);
// also returns the block total. wsum: 32 words of shared scratch.
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t *wsum, uint32_t &total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const uint32_t w = wsum[lane];
        uint32_t wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t u = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += u;
        }
        wsum[lane] = wi - w;                 // exclusive prefix of the warp totals
        if (lane == 31) wsum[32] = wi;       // block total
    }
    __syncthreads();
    const uint32_t r = wsum[warp] + incl - v;
    total = wsum[32];
    __syncthreads();                         // wsum is reused by the next call
    return r;
}

// Histogram of one digit over the keys that match the current prefix; lanes
// that hit the same bin add once (scores of the integer-valued indexer are
// concentrated in few bins, so plain per-key atomics serialise).
__device__ __forceinline__ void hist_add(uint32_t *hist, bool act, uint32_t bin) {
    const uint32_t m = __activemask();
    const uint32_t peers = __match_any_sync(m, act ? bin : 0xFFFFFFFFu);
    if (act && (threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&hist[bin], static_cast<uint32_t>(__popc(peers)));
}

// Per token: the exact top-k under the total order of key64 (score desc, then
// lower position first). Phase A: digit histograms over the global row until
// the keys sharing the k-th key's prefix fit in shared memory. Phase B, one
// more pass: keys above that prefix are winners and go straight to the output;
// keys with the prefix are gathered into shared memory. Phase C resolves the
// remaining digits there and phase D adds the candidates at or above the k-th
// key. Both runs are gathered in position order in shared memory and merged,
// so the row is written in ascending position order.
__global__ void __launch_bounds__(TK_NT, 1) topk_kernel(const IndexerArgs a) {
    extern __shared__ __align__(16) uint8_t tk_raw[];
    uint64_t *cand = reinterpret_cast<uint64_t *>(tk_raw);
    uint32_t *hist = reinterpret_cast<uint32_t *>(tk_raw + TK_CAP * 8);
    int32_t *sel = reinterpret_cast<int32_t *>(tk_raw + TK_CAP * 8 + 4096 * 4);
    __shared__ TkState st;
    __shared__ uint32_t wsum[33];

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
    const float4 *row4 = reinterpret_cast<const float4 *>(row);
    const int widths[6] = {12, 12, 8, 12, 12, 8};
    if (tid == 0) {
        st.prefix = 0;
        st.bits = 0;
        st.krem = static_cast<uint32_t>(a.topk);
        st.cnt = static_cast<uint32_t>(n);
    }
    __syncthreads();
    int di = 0;
    // ---- phase A: digit passes over the global row while the prefix holds too many keys ----
    while (di < 6 && st.bits < 64 && st.cnt > TK_CAP) {
        const int width = widths[di++], shift = 64 - st.bits - width;
        const uint64_t prefix = st.prefix;
        const int bits = st.bits;
        for (int d = tid; d < (1 << width); d += TK_NT) hist[d] = 0;
        __syncthreads();
        for (int64_t s4 = tid; 4 * s4 < n; s4 += TK_NT) {
            const float4 v = row4[s4];
            const float f[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int64_t s = 4 * s4 + e;
                const uint64_t k = key64(f[e], static_cast<int>(s));
                hist_add(hist, s < n && prefix_match(k, prefix, bits),
                         static_cast<uint32_t>((k >> shift) & ((1u << width) - 1)));
            }
        }
        __syncthreads();
        if (tid < 32) pick_digit(hist, width, shift, st);
        __syncthreads();
    }
    const uint64_t prefix = st.prefix;
    const int bits = st.bits;
    const uint32_t need = st.krem;                       // still to pick among the prefix's keys
    const uint32_t n_win = static_cast<uint32_t>(a.topk) - need;
    // ---- phase B: winners above the prefix to the output, the prefix's keys to smem ----
    {
        uint32_t wbase = 0, cbase = 0;
        for (int64_t c0 = 0; c0 < n; c0 += 4 * TK_NT) {
            const int64_t s0 = c0 + 4 * tid;
            uint64_t k[4];
            uint32_t win = 0, cnd = 0;
            if (s0 < n) {
                const float4 v = row4[s0 >> 2];
                const float f[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    k[e] = key64(f[e], static_cast<int>(s0 + e));
                    if (s0 + e < n) {
                        if (bits > 0 && (k[e] >> (64 - bits)) > (prefix >> (64 - bits))) win |= 1u << e;
                        else if (prefix_match(k[e], prefix, bits)) cnd |= 1u << e;
                    }
                }
            }
            uint32_t tot;
            const uint32_t off = block_excl_scan((static_cast<uint32_t>(__popc(cnd)) << 16) | __popc(win), wsum, tot);
            uint32_t wo = wbase + (off & 0xFFFFu), co = cbase + (off >> 16);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if (win >> e & 1u) {
                    if (wo < n_win) sel[wo] = static_cast<int32_t>(s0 + e);
                    ++wo;
                } else if (cnd >> e & 1u) {
                    if (co < TK_CAP) cand[co] = k[e];
                    ++co;
                }
            }
            wbase += tot & 0xFFFFu;
            cbase += tot >> 16;
        }
        if (tid == 0) st.ncand = cbase;
        __syncthreads();
        if (wbase != n_win || cbase > TK_CAP) {   // the histograms guarantee both; report instead of guessing
            if (tid == 0) set_dev_err(a.dev_err, MLA_DEVERR_INTERNAL);
            for (int j = tid; j < a.topk; j += TK_NT) out[j] = -1;
            return;
        }
    }
    // ---- phase C: remaining digits among the candidates, in shared memory ----
    const uint32_t nc = st.ncand;
    if (tid == 0) st.krem = need;
    __syncthreads();
    while (di < 6 && st.bits < 64) {
        const int width = widths[di++], shift = 64 - st.bits - width;
        const uint64_t pf = st.prefix;
        const int bb = st.bits;
        for (int d = tid; d < (1 << width); d += TK_NT) hist[d] = 0;
        __syncthreads();
        for (uint32_t i = tid; i < nc; i += TK_NT) {
            const uint64_t k = cand[i];
            hist_add(hist, prefix_match(k, pf, bb), static_cast<uint32_t>((k >> shift) & ((1u << width) - 1)));
        }
        __syncthreads();
        if (tid < 32) pick_digit(hist, width, shift, st);
        __syncthreads();
    }
    if (st.bits != 64) {
        if (tid == 0) set_dev_err(a.dev_err, MLA_DEVERR_INTERNAL);
        for (int j = tid; j < a.topk; j += TK_NT) out[j] = -1;
        return;
    }
    // ---- phase D: candidates at or above the k-th key, after the winners ----
    const uint64_t kth = st.prefix;
    uint32_t base = n_win;
    for (uint32_t c0 = 0; c0 < nc; c0 += TK_NT) {
        const uint32_t i = c0 + tid;
        const bool f = i < nc && cand[i] >= kth;
        uint32_t tot;
        const uint32_t off = block_excl_scan(f ? 1u : 0u, wsum, tot);
        if (f && base + off < static_cast<uint32_t>(a.topk))
            sel[base + off] = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(cand[i] & 0xFFFFFFFFu));
        base += tot;
    }
    if (base != static_cast<uint32_t>(a.topk)) {  // exactly `need` distinct keys sit at or above the k-th
        if (tid == 0) set_dev_err(a.dev_err, MLA_DEVERR_INTERNAL);
        for (int j = tid; j < a.topk; j += TK_NT) out[j] = -1;
        return;
    }
    // ---- ascending positions: merge the two ascending runs (winners, then candidates);
    // an element's output slot is its rank in its own run plus the number of smaller
    // elements in the other run (positions are distinct) ----
    __syncthreads();
    const int na = static_cast<int>(n_win), nb = a.topk - na;
    for (int i = tid; i < a.topk; i += TK_NT) {
        const bool in_a = i < na;
        const int x = sel[i];
        const int *other = in_a ? sel + na : sel;
        int lo = 0, hi = in_a ? nb : na;       // count of elements < x in the other run
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (other[mid] < x) lo = mid + 1; else hi = mid;
        }
        out[(in_a ? i : i - na) + lo] = x;
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

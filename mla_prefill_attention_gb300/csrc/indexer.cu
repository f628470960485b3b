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
#include "tc.cuh"

namespace mla {
namespace idx {

// ---------------------------------------------------------------------------
// exact top-k over one score row per token
// ---------------------------------------------------------------------------
constexpr int TK_NT = 512;              // two CTAs per SM hide each other's barriers
constexpr int TK_NW = TK_NT / 32;
constexpr int TK_U = 4;                 // float4 loads in flight per thread and pass step
constexpr int TK_STEP = 4 * TK_U * TK_NT;   // scores per step of a global pass
constexpr int TK_CAP = 8192;            // keys sharing the k-th key's prefix kept in shared memory
constexpr int TK_SEL = 2048;            // selected positions (max topk)
constexpr int TK_SMEM = TK_CAP * 8 + 4096 * 4 + TK_SEL * 4;
static_assert(TK_STEP < 65536 && TK_CAP < 65536, "per-step counts are packed in 16 bits");

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
    uint64_t prefix;    // digits fixed so far (high bits of the k-th key)
    int bits;           // how many
    uint32_t krem;      // rank of the k-th key among the keys with that prefix (1-based)
    uint32_t cnt;       // how many keys share the prefix
};

// Exclusive block-wide prefix sum of v in thread order; also the block total.
// wsum: TK_NW + 1 words of shared scratch. Every thread of the block calls it.
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
        const uint32_t w = lane < TK_NW ? wsum[lane] : 0u;
        uint32_t wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t u = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += u;
        }
        if (lane < TK_NW) wsum[lane] = wi - w;
        if (lane == 31) wsum[TK_NW] = wi;
    }
    __syncthreads();
    const uint32_t r = wsum[warp] + incl - v;
    total = wsum[TK_NW];
    __syncthreads();                         // wsum is reused by the next call
    return r;
}

// The same over TK_U values per thread, ordered (u, thread): r[u] counts the
// values of every earlier u and of the lower threads at the same u.
// wsum: TK_U * TK_NW + 1 words.
__device__ __forceinline__ void block_excl_scan_u(const uint32_t (&v)[TK_U], uint32_t (&r)[TK_U], uint32_t *wsum,
                                                  uint32_t &total) {
    static_assert(TK_U * TK_NW == 64, "warp 0 scans two words per lane");
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t incl[TK_U];
#pragma unroll
    for (int u = 0; u < TK_U; ++u) {
        incl[u] = v[u];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t x = __shfl_up_sync(0xffffffffu, incl[u], o);
            if (lane >= o) incl[u] += x;
        }
    }
    if (lane == 31) {
#pragma unroll
        for (int u = 0; u < TK_U; ++u) wsum[u * TK_NW + warp] = incl[u];
    }
    __syncthreads();
    if (warp == 0) {
        const uint32_t w0 = wsum[lane], w1 = wsum[lane + 32];
        uint32_t a = w0, b = w1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t xa = __shfl_up_sync(0xffffffffu, a, o);
            const uint32_t xb = __shfl_up_sync(0xffffffffu, b, o);
            if (lane >= o) { a += xa; b += xb; }
        }
        const uint32_t ta = __shfl_sync(0xffffffffu, a, 31);
        wsum[lane] = a - w0;
        wsum[lane + 32] = ta + b - w1;
        if (lane == 31) wsum[64] = ta + b;
    }
    __syncthreads();
#pragma unroll
    for (int u = 0; u < TK_U; ++u) r[u] = wsum[u * TK_NW + warp] + incl[u] - v[u];
    total = wsum[64];
    __syncthreads();
}

// Histogram of one digit over the keys that match the current prefix; lanes
// that hit the same bin add once (scores of the integer-valued indexer are
// concentrated in few bins, so plain per-key atomics serialise).
__device__ __forceinline__ void hist_add(uint32_t *hist, bool act, uint32_t bin) {
    const uint32_t m = __activemask();
    const uint32_t peers = __match_any_sync(m, act ? bin : 0xFFFFFFFFu);
    if (act && (threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&hist[bin], static_cast<uint32_t>(__popc(peers)));
}

// Pick the digit (one of 2^width bins, PER bins per thread) that holds the
// krem-th largest key and narrow the state to it. Every thread calls it; bins
// are taken in descending order so a block scan gives the keys above each.
template <int PER>    // 4096 bins: PER = 8, all threads in range; 256 bins: PER = 1
__device__ __forceinline__ void pick_digit(const uint32_t *hist, int width, int shift, TkState &st, uint32_t *wsum) {
    const int nb = 1 << width;
    const int tid = threadIdx.x;
    const int lo = nb - PER * (tid + 1);            // this thread's lowest bin
    uint32_t h[PER];
    uint32_t sum = 0;
    if constexpr (PER % 4 == 0) {
#pragma unroll
        for (int i = 0; i < PER; i += 4) {
            const uint4 w = *reinterpret_cast<const uint4 *>(hist + lo + i);
            h[i] = w.x; h[i + 1] = w.y; h[i + 2] = w.z; h[i + 3] = w.w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < PER; ++i) h[i] = lo >= 0 ? hist[lo + i] : 0u;
    }
#pragma unroll
    for (int i = 0; i < PER; ++i) sum += h[i];
    uint32_t tot;
    const uint32_t above = block_excl_scan(sum, wsum, tot);
    const uint32_t krem = st.krem;
    if (above < krem && krem <= above + sum) {      // exactly one thread
        uint32_t acc = above;
#pragma unroll
        for (int i = PER - 1; i >= 0; --i) {
            if (acc < krem && krem <= acc + h[i]) {
                st.prefix |= static_cast<uint64_t>(lo + i) << shift;
                st.bits += width;
                st.krem = krem - acc;
                st.cnt = h[i];
            }
            acc += h[i];
        }
    }
    __syncthreads();
}

__device__ __noinline__ void pick(const uint32_t *hist, int width, int shift, TkState &st, uint32_t *wsum) {
    static_assert(TK_NT == 512, "bins per thread assume 512 threads");
    if (width == 12) pick_digit<8>(hist, width, shift, st, wsum);
    else if (width == 11) pick_digit<4>(hist, width, shift, st, wsum);
    else if (width == 10) pick_digit<2>(hist, width, shift, st, wsum);
    else pick_digit<1>(hist, width, shift, st, wsum);   // up to 512 bins, one per thread
}

__device__ __forceinline__ void topk_fail(const IndexerArgs &a, int32_t *out) {
    if (threadIdx.x == 0) set_dev_err(a.dev_err, MLA_DEVERR_INTERNAL);
    for (int j = threadIdx.x; j < a.topk; j += TK_NT) out[j] = -1;
}

// Exact radix path (any input; the fallback of the sampled path). Phase A:
// digit histograms over the global row until the keys sharing the k-th key's
// prefix fit in shared memory. Phase B, one more pass: keys above that prefix
// are winners and their positions are kept in order; keys with the prefix are
// gathered, in order, into shared memory. Phase C resolves the remaining digits
// there and phase D appends the candidates at or above the k-th key. The two
// ascending runs are merged, so the row is written in ascending position order.
__device__ __noinline__ void topk_radix(const IndexerArgs &a, const float4 *row4, int n, int32_t *out, uint64_t *cand,
                                        uint32_t *hist, int32_t *sel, TkState &st, uint32_t *wsum) {
    const int tid = threadIdx.x;
    const int n4 = (n + 3) >> 2;           // the row stride is a multiple of 4 floats
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
    while (di < 6 && st.cnt > TK_CAP) {
        const int width = widths[di++], shift = 64 - st.bits - width;
        const uint64_t prefix = st.prefix;
        const int bits = st.bits;
        for (int d = tid; d < (1 << width); d += TK_NT) hist[d] = 0;
        __syncthreads();
        for (int q0 = 0; q0 < n4; q0 += TK_U * TK_NT) {
            float4 v[TK_U];
#pragma unroll
            for (int u = 0; u < TK_U; ++u) {
                const int q = q0 + u * TK_NT + tid;
                v[u] = q < n4 ? row4[q] : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < TK_U; ++u) {
                const int s0 = 4 * (q0 + u * TK_NT + tid);
                const float f[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const uint64_t k = key64(f[e], s0 + e);
                    hist_add(hist, s0 + e < n && prefix_match(k, prefix, bits),
                             static_cast<uint32_t>((k >> shift) & ((1u << width) - 1)));
                }
            }
        }
        __syncthreads();
        pick(hist, width, shift, st, wsum);
    }
    const uint64_t prefix = st.prefix;
    const int bits = st.bits;
    const uint32_t need = st.krem;                       // still to pick among the prefix's keys
    const uint32_t n_win = static_cast<uint32_t>(a.topk) - need;
    // ---- phase B: positions above the prefix in order, the prefix's keys to smem ----
    uint32_t nc;
    {
        uint32_t wbase = 0, cbase = 0;
        for (int q0 = 0; q0 < n4; q0 += TK_U * TK_NT) {
            float4 v[TK_U];
#pragma unroll
            for (int u = 0; u < TK_U; ++u) {
                const int q = q0 + u * TK_NT + tid;
                v[u] = q < n4 ? row4[q] : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            uint32_t win[TK_U], cnd[TK_U], cnt[TK_U], off[TK_U];
#pragma unroll
            for (int u = 0; u < TK_U; ++u) {
                const int s0 = 4 * (q0 + u * TK_NT + tid);
                const float f[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
                win[u] = 0;
                cnd[u] = 0;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const uint64_t k = key64(f[e], s0 + e);
                    if (s0 + e < n) {
                        if (bits > 0 && (k >> (64 - bits)) > (prefix >> (64 - bits))) win[u] |= 1u << e;
                        else if (prefix_match(k, prefix, bits)) cnd[u] |= 1u << e;
                    }
                }
                cnt[u] = (static_cast<uint32_t>(__popc(cnd[u])) << 16) | static_cast<uint32_t>(__popc(win[u]));
            }
            uint32_t tot;
            block_excl_scan_u(cnt, off, wsum, tot);
#pragma unroll
            for (int u = 0; u < TK_U; ++u) {
                const int s0 = 4 * (q0 + u * TK_NT + tid);
                const float f[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
                uint32_t wo = wbase + (off[u] & 0xFFFFu), co = cbase + (off[u] >> 16);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if (win[u] >> e & 1u) {
                        if (wo < n_win) sel[wo] = s0 + e;
                        ++wo;
                    } else if (cnd[u] >> e & 1u) {
                        if (co < TK_CAP) cand[co] = key64(f[e], s0 + e);
                        ++co;
                    }
                }
            }
            wbase += tot & 0xFFFFu;
            cbase += tot >> 16;
        }
        if (wbase != n_win || cbase > TK_CAP) {   // the histograms guarantee both; report instead of guessing
            topk_fail(a, out);
            return;
        }
        nc = cbase;
    }
    // ---- phase C: remaining digits among the candidates, in shared memory ----
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
        pick(hist, width, shift, st, wsum);
    }
    if (st.bits != 64) {
        topk_fail(a, out);
        return;
    }
    // ---- phase D: candidates at or above the k-th key, in order, after the winners ----
    const uint64_t kth = st.prefix;
    uint32_t base = n_win;
    for (uint32_t c0 = 0; c0 < nc; c0 += 4 * TK_NT) {
        const uint32_t i0 = c0 + 4 * tid;
        uint32_t f = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (i0 + j < nc && cand[i0 + j] >= kth) f |= 1u << j;
        uint32_t tot;
        uint32_t o = base + block_excl_scan(static_cast<uint32_t>(__popc(f)), wsum, tot);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (f >> j & 1u) {
                if (o < static_cast<uint32_t>(a.topk))
                    sel[o] = static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(cand[i0 + j] & 0xFFFFFFFFu));
                ++o;
            }
        }
        base += tot;
    }
    if (base != static_cast<uint32_t>(a.topk)) {  // exactly `need` distinct keys sit at or above the k-th
        topk_fail(a, out);
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

// Block-wide bitonic sort of v[0..P) in shared memory (P a power of two).
template <typename T, bool kDescending>
__device__ __forceinline__ void bitonic_sort(T *v, int P) {
    // Pair (lo, hi) of index i at stride s <= 32 lies inside elements 64w .. 64w+63
    // of the warp w that owns i (i mod 512 in 32w .. 32w+31), so those stages only
    // need the warp's own lanes in step; a block barrier follows each wider stage
    // and the last stage of every size (the next size starts wide).
    for (int size = 2; size <= P; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int i = threadIdx.x; i < P / 2; i += TK_NT) {
                const int lo = 2 * i - (i & (stride - 1)), hi = lo + stride;
                const bool asc = ((lo & size) == 0) != kDescending;
                const T x = v[lo], y = v[hi];
                if (asc ? x > y : x < y) {
                    v[lo] = y;
                    v[hi] = x;
                }
            }
            if (stride > 32 || stride == 1) __syncthreads();
            else __syncwarp();
        }
    }
}

constexpr int TK_SAMPLE = 1024;
constexpr int TK_CH = 16;   // consecutive scores per lane and step of a sampled pass (four float4)
static_assert(TK_CH == 16 && TK_CH * 32 < 65536, "a warp step's counts are packed in 16 bits");

__device__ __forceinline__ int bit_width(uint32_t x) { return x ? 32 - __clz(x) : 0; }

// The float whose order key is t, for t != 0 (0 is the key of every NaN). The
// key 0xFFFFFFFF maps to a NaN, which no score exceeds.
__device__ __forceinline__ float ord_inv(uint32_t t) {
    return __uint_as_float((t & 0x80000000u) ? (t & 0x7FFFFFFFu) : ~t);
}

// A lane's TK_CH consecutive scores from position TK_CH * c as four float4 loads
// inside the row's float4 span (the row stride is a multiple of 4 floats); bit j
// of vm marks position TK_CH * c + j < n.
__device__ __forceinline__ void load_chunk(const float4 *row4, int c, bool live, int n4, int n, float4 (&v)[4],
                                           uint32_t &vm) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int q = 4 * c + u;
        v[u] = live && q < n4 ? row4[q] : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    const int lim = live ? n - TK_CH * c : 0;
    vm = lim >= TK_CH ? 0xFFFFu : (lim > 0 ? (1u << lim) - 1u : 0u);
}

// Bit j of wm: score j of the chunk lies above the bracket; of gm: at or above
// its low end. Float compares with the ends' floats decide what the order keys
// would: the keys keep the order of non-NaN floats and tie -0 with +0; a NaN
// (key 0) is above no end and at or above the low end only when that end is
// key 0 (lo_all).
__device__ __forceinline__ void classify(const float4 (&v)[4], float f_hi, float f_lo, bool lo_all, uint32_t &wm,
                                         uint32_t &gm) {
    wm = 0;
    gm = 0;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const float f[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            if (f[e] > f_hi) wm |= 1u << (4 * u + e);
            if (lo_all || f[e] >= f_lo) gm |= 1u << (4 * u + e);
        }
    }
}

// One step of a warp's pass over the row: lane chunk c classified into winner
// and candidate masks, and the warp scan of their counts (winners in the low 16
// bits, candidates in the high 16): ex counts the lower lanes, tot the warp.
__device__ __forceinline__ void pass_step(const float4 *row4, int c, bool live, int n4, int n, float f_hi, float f_lo,
                                          bool lo_all, uint32_t &wm, uint32_t &cm, uint32_t &ex, uint32_t &tot) {
    float4 v[4];
    uint32_t vm, gm;
    load_chunk(row4, c, live, n4, n, v, vm);
    classify(v, f_hi, f_lo, lo_all, wm, gm);
    wm &= vm;
    cm = gm & ~wm & vm;
    const uint32_t x = (static_cast<uint32_t>(__popc(cm)) << 16) | static_cast<uint32_t>(__popc(wm));
    const int lane = threadIdx.x & 31;
    uint32_t incl = x;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += y;
    }
    tot = __shfl_sync(0xffffffffu, incl, 31);
    ex = incl - x;
}

// A lane's winners (positions) from slot pw and candidates ((order key,
// position); the score is read again, an L1 hit, rather than picked from
// registers) from slot pc, in position order; slots at or past wcap / ccap are
// not written.
__device__ __forceinline__ void put_hits(const float *row, int s0, uint32_t wm, uint32_t cm, uint32_t pw, uint32_t pc,
                                         uint32_t wcap, uint32_t ccap, int32_t *wdst, uint64_t *cdst) {
    while (wm) {
        if (pw < wcap) wdst[pw] = s0 + __ffs(wm) - 1;
        ++pw;
        wm &= wm - 1;
    }
    while (cm) {
        if (pc < ccap) {
            const int s = s0 + __ffs(cm) - 1;
            cdst[pc] = (static_cast<uint64_t>(ord_f32(row[s])) << 32) | static_cast<uint32_t>(s);
        }
        ++pc;
        cm &= cm - 1;
    }
}

// The warp whose run of final slots holds slot d: the last w with first slot
// <= d (a warp with an empty run shares its first slot with the next warp).
__device__ __forceinline__ int run_owner(const uint32_t (*first)[2], int which, uint32_t d) {
    int w = 0;
#pragma unroll
    for (int step = TK_NW / 2; step > 0; step >>= 1)
        if (w + step < TK_NW && first[w + step][which] <= d) w += step;
    return w;
}

// A candidate (order key << 32 | position) as a digit key: its offset from the
// bracket's low key in the top kb bits (kb <= 32), so the digits cover only the
// bits in which the candidates can differ.
__device__ __forceinline__ uint32_t cand_key(uint64_t c, uint32_t t_lo, int kb) {
    return kb ? (static_cast<uint32_t>(c >> 32) - t_lo) << (32 - kb) : 0u;
}

// Sampled path: the k-th largest score is bracketed from an evenly spaced sample
// of 1,024 scores (ranks expected +- 4 standard deviations + 2); one pass over
// the row follows, each warp over its own contiguous segment and each lane over
// 16 consecutive scores per step, with no atomics and no block barrier: the
// winners (above the bracket) and candidates (inside it) go, as positions and
// as (order key, position), in position order into slots of the warp's own and
// are then compacted; a second, ordered pass runs only when a warp has more
// than its slots hold. Radix digits over the bracket's significant key bits find
// the k-th candidate score; the candidates above it and the first ones equal to
// it (lowest positions first, as the key order wants) follow the winners, and
// the two ascending runs are merged. Returns false, having written nothing, when
// the bracket misses (too few or too many scores inside it); the caller then
// takes the radix path.
__device__ __noinline__ bool topk_sampled(const IndexerArgs &a, const float *row, const float4 *row4, int n,
                                          int32_t *out, uint64_t *cand, uint32_t *hist, int32_t *sel,
                                          uint32_t (*wcnt)[2], uint32_t *info, TkState &st, uint32_t *wsum) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int k = a.topk;
    uint32_t *samp = hist;
    for (int i = tid; i < TK_SAMPLE; i += TK_NT)
        samp[i] = ord_f32(row[static_cast<int>((static_cast<int64_t>(i) * n) / TK_SAMPLE)]);
    __syncthreads();
    bitonic_sort<uint32_t, true>(samp, TK_SAMPLE);
    const float e = static_cast<float>(k) * TK_SAMPLE / static_cast<float>(n);
    const float mg = 4.f * sqrtf(e) + 2.f;
    const int rh = static_cast<int>(floorf(e - mg)), rl = static_cast<int>(ceilf(e + mg));
    const uint32_t t_hi = rh >= 0 ? samp[rh] : 0xFFFFFFFFu;   // winners: key > t_hi
    const uint32_t t_lo = rl < TK_SAMPLE ? samp[rl] : 0u;      // candidates: t_lo <= key <= t_hi
    __syncthreads();                                          // samp is reused as the histogram
    if (t_hi == 0u) return false;                             // NaNs above the bracket: radix path
    const float f_hi = ord_inv(t_hi), f_lo = t_lo ? ord_inv(t_lo) : 0.f;
    const bool lo_all = t_lo == 0u;
    const int n4 = (n + 3) >> 2;
    const int nch = (n + TK_CH - 1) / TK_CH;
    const int segc = (nch + TK_NW - 1) / TK_NW;
    const int c_lo = warp * segc, c_hi = min(nch, c_lo + segc);
    // ---- one pass: each warp puts its winners' positions and its candidates'
    // (key, position) in position order into slots of its own; the counts run on
    // past the slots, so an overflow is seen ----
    constexpr uint32_t kWinSlots = TK_SEL / TK_NW, kCandSlots = TK_CAP / TK_NW;
    uint32_t wn = 0, cn = 0;
    for (int c0 = c_lo; c0 < c_hi; c0 += 32) {
        const int c = c0 + lane;
        uint32_t wm, cm, ex, tot;
        pass_step(row4, c, c < c_hi, n4, n, f_hi, f_lo, lo_all, wm, cm, ex, tot);
        put_hits(row, TK_CH * c, wm, cm, wn + (ex & 0xFFFFu), cn + (ex >> 16), kWinSlots, kCandSlots,
                 sel + warp * kWinSlots, cand + warp * kCandSlots);
        wn += tot & 0xFFFFu;
        cn += tot >> 16;
    }
    if (lane == 0) {
        wcnt[warp][0] = wn;
        wcnt[warp][1] = cn;
    }
    __syncthreads();
    if (tid == 0) {
        uint32_t tw = 0, tc = 0, fits = 1;
        for (int w = 0; w < TK_NW; ++w) {
            const uint32_t x = wcnt[w][0], y = wcnt[w][1];
            if (x > kWinSlots || y > kCandSlots) fits = 0;
            wcnt[w][0] = tw;                                  // from here on: the warp's first final slot
            wcnt[w][1] = tc;
            tw += x;
            tc += y;
        }
        info[0] = tw;
        info[1] = tc;
        info[2] = (tw <= static_cast<uint32_t>(k) && static_cast<uint32_t>(k) <= tw + tc && tc <= TK_CAP) ? 1u : 0u;
        info[3] = fits;
    }
    __syncthreads();
    if (!info[2]) return false;
    const uint32_t n_win = info[0], nc = info[1];
    if (info[3]) {
        // ---- compaction: final slot d takes entry d - first(w) of the warp w whose
        // run holds d. Every entry moves down (a warp's first final slot is at most
        // its own first slot), so in rounds of TK_NT final slots a round's stores
        // land below every later round's sources; one barrier inside a round
        // separates its loads from its stores ----
        const uint32_t rounds = (max(n_win, nc) + TK_NT - 1) / TK_NT;
        for (uint32_t r = 0; r < rounds; ++r) {
            const uint32_t d = r * TK_NT + tid;
            int32_t wv = 0;
            uint64_t cv = 0;
            if (d < n_win) {
                const int w = run_owner(wcnt, 0, d);
                wv = sel[w * kWinSlots + (d - wcnt[w][0])];
            }
            if (d < nc) {
                const int w = run_owner(wcnt, 1, d);
                cv = cand[w * kCandSlots + (d - wcnt[w][1])];
            }
            __syncthreads();
            if (d < n_win) sel[d] = wv;
            if (d < nc) cand[d] = cv;
        }
    } else {
        // ---- a warp's slots overflowed: a second pass writes every entry straight
        // to its final slot ----
        uint32_t wo = wcnt[warp][0], co = wcnt[warp][1];
        for (int c0 = c_lo; c0 < c_hi; c0 += 32) {
            const int c = c0 + lane;
            uint32_t wm, cm, ex, tot;
            pass_step(row4, c, c < c_hi, n4, n, f_hi, f_lo, lo_all, wm, cm, ex, tot);
            put_hits(row, TK_CH * c, wm, cm, wo + (ex & 0xFFFFu), co + (ex >> 16), TK_SEL, TK_CAP, sel, cand);
            wo += tot & 0xFFFFu;
            co += tot >> 16;
        }
    }
    // ---- the k-th candidate score: digits over the kb bits in which candidates differ ----
    const uint32_t need = static_cast<uint32_t>(k) - n_win;
    const int kb = bit_width(t_hi - t_lo);
    if (tid == 0) {
        st.prefix = 0;
        st.bits = 0;
        st.krem = need;
    }
    __syncthreads();
    if (need > 0) {
        // kb bits in at most three digits of at most 12 bits (4,096 bins):
        // one for kb <= 12, two near-equal ones for kb <= 24, else 12 + 12 + rest
        int widths[3] = {kb, 0, 0};
        if (kb > 24) {
            widths[0] = 12;
            widths[1] = 12;
            widths[2] = kb - 24;
        } else if (kb > 12) {
            widths[0] = kb - kb / 2;
            widths[1] = kb / 2;
        }
        int di = 0;
        while (di < 3 && st.bits < kb) {     // 32-bit keys: the state's prefix holds them in its top half
            const int width = widths[di++], bb = st.bits, shift = 32 - bb - width;
            const uint32_t pf = static_cast<uint32_t>(st.prefix >> 32);
            for (int d = tid; d < (1 << width); d += TK_NT) hist[d] = 0;
            __syncthreads();
            for (uint32_t i = tid; i < nc; i += TK_NT) {
                const uint32_t key = cand_key(cand[i], t_lo, kb);
                hist_add(hist, bb == 0 || (key >> (32 - bb)) == (pf >> (32 - bb)), (key >> shift) & ((1u << width) - 1));
            }
            __syncthreads();
            pick(hist, width, shift + 32, st, wsum);
        }
        if (st.bits < kb) {   // every digit finds its bin; unreachable
            topk_fail(a, out);
            return true;
        }
        // ---- candidates above the k-th score, and the first `take` equal to it, after the winners ----
        const uint32_t kth = static_cast<uint32_t>(st.prefix >> 32);
        const uint32_t take = st.krem;
        uint32_t base_a = 0, base_e = 0;
        for (uint32_t c0 = 0; c0 < nc; c0 += 4 * TK_NT) {
            const uint32_t i0 = c0 + 4 * tid;
            uint32_t fa = 0, fe = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (i0 + j < nc) {
                    const uint32_t key = cand_key(cand[i0 + j], t_lo, kb);
                    if (key > kth) fa |= 1u << j;
                    else if (key == kth) fe |= 1u << j;
                }
            }
            uint32_t tot;
            const uint32_t ex = block_excl_scan((static_cast<uint32_t>(__popc(fe)) << 16) |
                                                    static_cast<uint32_t>(__popc(fa)), wsum, tot);
            uint32_t ra = base_a + (ex & 0xFFFFu), re = base_e + (ex >> 16);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (fa >> j & 1u) {
                    const uint32_t o = n_win + ra + min(re, take);
                    if (o < static_cast<uint32_t>(k)) sel[o] = static_cast<int32_t>(cand[i0 + j] & 0xFFFFFFFFu);
                    ++ra;
                } else if (fe >> j & 1u) {
                    const uint32_t o = n_win + ra + re;
                    if (re < take && o < static_cast<uint32_t>(k))
                        sel[o] = static_cast<int32_t>(cand[i0 + j] & 0xFFFFFFFFu);
                    ++re;
                }
            }
            base_a += tot & 0xFFFFu;
            base_e += tot >> 16;
        }
        if (base_a + take != need || base_e < take) {   // the digits guarantee both; report instead of guessing
            topk_fail(a, out);
            return true;
        }
    }
    // ---- merge the two ascending runs (winners, chosen candidates) ----
    __syncthreads();
    const int na = static_cast<int>(n_win), nb = k - na;
    for (int i = tid; i < k; i += TK_NT) {
        const bool in_a = i < na;
        const int x = sel[i];
        const int *other = in_a ? sel + na : sel;
        int lo = 0, hi = in_a ? nb : na;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (other[mid] < x) lo = mid + 1; else hi = mid;
        }
        out[(in_a ? i : i - na) + lo] = x;
    }
    return true;
}

__global__ void __launch_bounds__(TK_NT, 2) topk_kernel(const IndexerArgs a) {
    extern __shared__ __align__(16) uint8_t tk_raw[];
    uint64_t *cand = reinterpret_cast<uint64_t *>(tk_raw);
    uint32_t *hist = reinterpret_cast<uint32_t *>(tk_raw + TK_CAP * 8);   // also the sample
    int32_t *sel = reinterpret_cast<int32_t *>(tk_raw + TK_CAP * 8 + 4096 * 4);
    __shared__ TkState st;
    __shared__ uint32_t wsum[TK_U * TK_NW + 1];
    __shared__ uint32_t wcnt[TK_NW][2];
    __shared__ uint32_t info[4];

    const int64_t t = a.tok0 + blockIdx.x;
    const int b = find_seq(a.cu_seqlens, a.batch, t);
    const int n = __ldg(a.prefix_lens + b) + static_cast<int>(t - __ldg(a.cu_seqlens + b)) + 1;
    int32_t *out = a.idx_out + t * a.topk;
    if (n <= a.topk) {
        for (int j = threadIdx.x; j < a.topk; j += TK_NT) out[j] = j < n ? j : -1;
        return;
    }
    const float *row = a.scores + t * a.score_stride;
    const float4 *row4 = reinterpret_cast<const float4 *>(row);
    if (threadIdx.x == 0) {
        // the whole row into L2 while the sample is read and sorted, so the pass
        // over it reads L2 (rows start 16-byte aligned; whole float4s)
        const uint32_t bytes = static_cast<uint32_t>((n + 3) >> 2) * 16u;
        for (uint32_t off = 0; off < bytes; off += 65536u)
            tc::bulk_prefetch_l2(reinterpret_cast<const char *>(row) + off, min(65536u, bytes - off));
    }
    if (!topk_sampled(a, row, row4, n, out, cand, hist, sel, wcnt, info, st, wsum)) {
        __syncthreads();
        topk_radix(a, row4, n, out, cand, hist, sel, st, wsum);
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

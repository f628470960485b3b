// Indexer scores and exact streaming top-k selection in one kernel
// (tcgen05 kind::f8f6f4 for the scores; the scores never leave the SM).
//
// score(t,s) = sigmaI_s * sum_h w[t,h] * max(0, q_{t,h} . k_s),   s <= position(t)
// (GLM-5.3 Teil 2, section "Warum nicht TP oder DP?": the indexer scores every
// earlier token and keeps 2,048; footnote 3: an indexer key is 128 FP8 values
// plus a 4-byte scale.) The kept set is the first min(topk, p+1) positions in
// the order (score descending, position ascending).
//
// One CTA takes 3 query tokens (x 64 heads) of one sequence and streams every
// key they can see, 128 at a time (a first launch on the fast path, a second,
// for the groups the first flagged, on the exact streaming path):
//
//   D[key][64 j + h] = k_key . q_{t_j,h}    tcgen05.mma e4m3 x e4m3 -> f32,
//                                           M = 128 keys, N = 192 = 3 tokens x 64
//                                           heads, K = 128 (4 steps of 32)
//
// so TMEM lane = key, and each epilogue thread owns one key of one token: the
// head sum sum_h w[t,h] max(0, D) is a per-thread loop over its own columns.
// The products of the codes are exact in f32 and the sums are exact while they
// stay below 2^24 units of the smallest product, which integer-valued queries
// and keys guarantee.
//
// Selection, fast path (per token, by its four epilogue warps). Scores are
// ranked by 64-bit keys (32-bit order key of the score: the float order, -0
// ties +0, NaN lowest; then the complement of the position), which are all
// distinct and order "score descending, position ascending". The CTA visits a
// spread sample of S key tiles first (S grows with the context, 8 to 32; none
// when every key fits the candidate buffer) and every key of those tiles enters
// the buffer. From the sample the token sets a threshold: the sample's r-th
// largest score, r a few standard deviations past the rank the k-th largest
// score is expected at. Then the other tiles stream in position order and a key
// enters only if its score is at or above the threshold. Each warp appends to
// its own quarter of the buffer (no barrier per tile). At the end the k-th
// largest key over the whole buffer is found by radix digits (8 bits at a time
// from the highest bit in which the keys differ) and the k positions at or
// above it are written, quarter by quarter in each quarter's stored order (so
// the row's order is deterministic, though not ascending). This is exact
// whenever at least k keys reached the buffer: every key at or above the
// threshold did. When fewer did
// (the sample put the threshold too high) or a warp's quarter overflowed, the
// group is flagged and a second launch of the exact streaming path redoes it.
//
// Selection, exact streaming path (the fallback). A token keeps up to kCap
// (order key, position) entries in ascending position order and a threshold: a
// key enters if its order key is above it (every key enters until the first
// compaction). Keys arrive in ascending position order, so a later key whose
// score equals the k-th kept score ranks below it and need not enter. When the
// buffer could overflow on the next tile it is compacted: radix digits locate
// the k-th largest order key among the entries; after two digits the bin holding
// it bounds it from below and, if that keeps few enough entries, every entry at
// or above the bin's lower edge stays and the threshold becomes that edge;
// otherwise the digits run to the exact k-th key and ties at it keep the lowest
// positions. Every key of the final top-k is at or above the k-th key of any
// subset seen earlier, so no compaction drops one. An exact compaction at the
// end leaves the k entries, in ascending position order. The four warps of a
// token exchange per-tile counts behind a named barrier so every slot follows
// position order.
//
// Tokens whose position p has p + 1 <= topk keep 0..p (-1 padded) and select
// nothing; a group of such tokens only writes its rows.
//
// Warps: 0-11 epilogue (warp w: token w/4, TMEM lane quadrant w%4 = keys
// 32(w%4)..+31 of a tile), 12 TMA producer, 13 MMA issue + TMEM owner. Key
// tiles go through a 4-stage ring, the accumulator is double-buffered in TMEM
// (2 x 192 of 512 columns). Every wait is bounded and reports
// MLA_DEVERR_TIMEOUT; a warp whose wait gave up stops waiting but still runs
// every named barrier of its token, so none is left waiting; before the CTA
// exits the producer waits for its copies.
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace mla {
namespace idxf {

using namespace tc;

constexpr int TOK = kIdxTokensPerCta;   // 3 query tokens per CTA
constexpr int KT = 128;                 // keys per tile
constexpr int STAGES = 4;
constexpr int kEpiWarps = 4 * TOK;      // tokens x 4 TMEM lane quadrants
constexpr int kDCols = 256;             // TMEM columns per accumulator buffer (TOK x 64 used)
constexpr int NT = 32 * (kEpiWarps + 2);
constexpr int kProducerWarp = kEpiWarps, kIssuerWarp = kEpiWarps + 1;
constexpr int kQBytes = TOK * kHidx * kDidx;       // 24 KB
constexpr int kTileBytes = KT * kDidx;             // 16 KB
constexpr int kCap = kIdxCandidates;               // candidate entries per token
constexpr int kCapW = kCap / 4;                    // fast path: each warp's quarter of a token's buffer
constexpr int kKeepMax = kCap / 2;                 // most entries an inexact compaction keeps
constexpr int kSampleMin = 8, kSampleMax = 32;     // fast path: sample tiles
constexpr int kBins = 256;                         // 8-bit digits
constexpr int kOffK = kQBytes;
constexpr int kOffOrd = kOffK + STAGES * kTileBytes;
constexpr int kOffPos = kOffOrd + TOK * kCap * 4;
constexpr int kOffHist = kOffPos + TOK * kCap * 4;
constexpr int kRing = 8;                           // tiles of key scales staged ahead of the epilogue
constexpr int kOffScale = kOffHist + TOK * kBins * 4;
constexpr int kDynSmem = 1024 + kOffScale + kRing * KT * 4;
constexpr long long kWaitCycles = 200000000LL;
static_assert(kPage % KT == 0, "a key tile must not straddle a page");
static_assert(kCap - KT >= 2048 + kBins && kKeepMax + KT <= kCap, "candidate buffer too small for topk 2048");
static_assert(kDynSmem <= 232448, "shared memory");
static_assert(kSampleMax * 32 < kCapW, "every sampled key of a warp fits its quarter");

enum Bar {
    B_Q_FULL = 0,
    B_K_FULL = 1,                       // [STAGES]  TMA -> issuer
    B_K_EMPTY = B_K_FULL + STAGES,      // [STAGES]  issuer (commit) -> producer
    B_D_FULL = B_K_EMPTY + STAGES,      // [2]       issuer (commit) -> epilogue
    B_D_EMPTY = B_D_FULL + 2,           // [2]       epilogue (12 warps) -> issuer
    B_FINAL = B_D_EMPTY + 2,
    B_S_FULL = B_FINAL + 1,             // [kRing]   producer (+ scale copy) -> epilogue
    NBAR = B_S_FULL + kRing
};

// Radix state of one token's selection (written by one thread, read by the
// token's 128 threads after a barrier).
struct Sel {
    uint32_t prefix;    // digits fixed so far
    uint32_t above;     // entries above the prefix's bin, over all digits so far
    uint32_t krem;      // rank of the k-th key among the entries sharing the prefix (1-based)
    uint32_t bincnt;    // entries sharing the prefix
};

// Radix state of a fast-path selection over 64-bit keys.
struct Sel64 {
    uint64_t prefix;    // digits fixed so far (the key's top nbits)
    uint32_t krem;      // rank of the k-th key among the entries sharing the prefix (1-based)
    uint32_t bincnt;    // entries sharing the prefix
};

struct Shared {
    uint64_t bar[NBAR];
    uint32_t tmem_base;
    int32_t ring_tile[kRing];                 // the key tile of step i sits in slot i % kRing,
    int32_t ring_bad[kRing];                  // with its page flagged bad, and its 128 key scales
    uint32_t cta_fail;                        // fast path: some token of the group needs the exact path
    uint32_t fail_tok[TOK];                   // fast path: a warp of the token gave up or overflowed
    uint32_t wcnt[TOK][4];                    // fast path: entries in each warp's quarter
    uint64_t red[TOK][4][2];                  // fast path: per-warp largest and smallest key
    Sel64 sel64[TOK];
    __align__(16) uint32_t cntx[TOK][2][4];   // per tile parity: candidates of each quadrant's warp
    __align__(16) uint32_t wx[TOK][2][4][2];  // compaction rounds: (above, equal) counts per warp
    uint32_t wtot[TOK][4];                    // digit pick: bin sums per warp
    Sel sel[TOK];
};

__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ float sum2(uint64_t v) {
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
    return lo + hi;
}
// acc += a * b, elementwise on two packed floats
__device__ __forceinline__ void ffma2(uint64_t &acc, uint64_t a, uint64_t b) {
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(a), "l"(b));
}
// Twice max(x, 0), as x + |x| (exact: 0 or 2x): an add with an absolute-value
// operand on the FMA pipe instead of a max on the integer/logic pipe. The
// weights are halved (exact), so each product equals w * max(x, 0).
__device__ __forceinline__ float relu2_bits(uint32_t x) {
    const float f = __uint_as_float(x);
    return f + fabsf(f);
}

// Order key of a score: larger score, larger key; -0 and +0 tie; NaN is 0.
__device__ __forceinline__ uint32_t ord_f32(float x) {
    if (x != x) return 0u;
    if (x == 0.f) x = 0.f;
    const uint32_t u = __float_as_uint(x);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// The named barrier of token j's four epilogue warps.
__device__ __forceinline__ void token_bar(int j) {
    asm volatile("bar.sync %0, %1;\n" ::"r"(1 + j), "r"(128) : "memory");
}
__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

__device__ __forceinline__ bool wait_bar(Shared &sh, int32_t *dev_err, int b, uint32_t parity) {
    if (mbar_wait_cycles(smem_u32(&sh.bar[b]), parity, kWaitCycles)) return true;
    set_dev_err(dev_err, MLA_DEVERR_TIMEOUT);
    return false;
}

// Compaction of token j's candidate buffer (n entries in position order) by its
// 128 threads (t = 0..127): keep the entries that can still be among the top k.
// exact: keep exactly the top k (n >= k), else possibly more (see the file
// comment). Returns the new entry count and sets the insertion threshold (a
// later key enters iff warm is false or its order key is above thr).
__device__ __noinline__ int compact(Shared &sh, int j, int t, uint32_t *ord, int32_t *pos, uint32_t *hist, int n,
                                    int k, bool exact, uint32_t &thr, bool &warm) {
    const int lane = t & 31, wq = t >> 5;
    token_bar(j);                                     // every insert of the token is visible
    if (n <= k) return n;                             // nothing to drop
    Sel &st = sh.sel[j];
    if (t == 0) {
        st.prefix = 0;
        st.above = 0;
        st.krem = static_cast<uint32_t>(k);
        st.bincnt = static_cast<uint32_t>(n);
    }
    int bits = 0;
    uint32_t prefix = 0;
    bool whole_bin = false;
    for (;;) {
        const int shift = 24 - bits;
        hist[2 * t] = 0;
        hist[2 * t + 1] = 0;
        token_bar(j);
        // the state is written only between the two barriers of the pick below: read it here
        prefix = st.prefix;
        const uint32_t krem = st.krem;
        for (int e0 = 0; e0 < n; e0 += 128) {
            const int e = e0 + t;
            const uint32_t o = e < n ? ord[e] : 0u;
            const bool in = e < n && (bits == 0 || (o >> (32 - bits)) == prefix);
            const uint32_t bin = (o >> shift) & (kBins - 1);
            const uint32_t peers = __match_any_sync(0xffffffffu, in ? bin : 0xFFFFFFFFu);
            if (in && lane == __ffs(peers) - 1) atomicAdd(&hist[bin], static_cast<uint32_t>(__popc(peers)));
        }
        token_bar(j);
        // bins in descending order: thread t holds bins 255 - 2t and 254 - 2t
        const uint32_t hh = hist[kBins - 1 - 2 * t], hl = hist[kBins - 2 - 2 * t];
        const uint32_t s = hh + hl;
        uint32_t inc = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t v = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += v;
        }
        if (lane == 31) sh.wtot[j][wq] = inc;
        token_bar(j);
        uint32_t ab = inc - s;
        for (int w = 0; w < wq; ++w) ab += sh.wtot[j][w];
        if (ab < krem && krem <= ab + s) {            // exactly one thread
            const bool hi = krem <= ab + hh;
            const uint32_t bin = hi ? kBins - 1 - 2 * t : kBins - 2 - 2 * t;
            const uint32_t before = hi ? ab : ab + hh;
            st.prefix = (prefix << 8) | bin;
            st.above += before;
            st.krem = krem - before;
            st.bincnt = hi ? hh : hl;
        }
        token_bar(j);
        bits += 8;
        prefix = st.prefix;
        if (st.bincnt == st.krem) {                   // the whole bin is in the top k
            whole_bin = true;
            break;
        }
        if (bits == 32) break;                        // the exact k-th key
        if (!exact && bits >= 16 && st.above + st.bincnt <= static_cast<uint32_t>(kKeepMax)) break;
    }
    const uint32_t lo = bits == 32 ? prefix : prefix << (32 - bits);   // lower edge of the bin
    const bool ties = bits == 32 && !whole_bin;                         // keep the first krem equal keys
    const uint32_t krem = ties ? st.krem : 0u;
    // stable compaction in rounds of 128 entries; an entry moves down only, and a
    // round's loads all precede its stores (the barrier of the count exchange)
    uint32_t kept = 0, eq_seen = 0;
    for (int e0 = 0, r = 0; e0 < n; e0 += 128, ++r) {
        const int e = e0 + t;
        const uint32_t o = e < n ? ord[e] : 0u;
        const int32_t p = e < n ? pos[e] : 0;
        const bool a = e < n && (ties ? o > lo : o >= lo);
        const bool q = ties && e < n && o == lo;
        const uint32_t ma = __ballot_sync(0xffffffffu, a), me = __ballot_sync(0xffffffffu, q);
        if (lane == 0) {
            sh.wx[j][r & 1][wq][0] = __popc(ma);
            sh.wx[j][r & 1][wq][1] = __popc(me);
        }
        token_bar(j);
        uint32_t kb = kept, kept_all = 0, eq_all = 0, eq_mine = 0;
        for (int w = 0; w < 4; ++w) {
            const uint32_t na = sh.wx[j][r & 1][w][0], ne = sh.wx[j][r & 1][w][1];
            const uint32_t before = eq_seen + eq_all;
            const uint32_t take = before >= krem ? 0u : min(ne, krem - before);
            if (w < wq) kb += na + take;
            if (w == wq) eq_mine = before;
            kept_all += na + take;
            eq_all += ne;
        }
        const bool keep = a || (q && eq_mine + static_cast<uint32_t>(__popc(me & lanemask_lt())) < krem);
        const uint32_t mk = __ballot_sync(0xffffffffu, keep);
        if (keep) {
            const uint32_t d = kb + __popc(mk & lanemask_lt());
            ord[d] = o;
            pos[d] = p;
        }
        kept += kept_all;
        eq_seen += eq_all;
    }
    token_bar(j);                                     // the compacted buffer is visible
    // a later key must rank above what every kept-set bound so far allows: above the
    // exact k-th key (later equal keys rank below it), or at or above the bin's edge
    if (bits == 32 || lo > 0) {
        const uint32_t t_new = bits == 32 ? lo : lo - 1;
        thr = warm ? max(thr, t_new) : t_new;
        warm = true;
    }
    return static_cast<int>(kept);
}

// ---------------------------------------------------------------------------
// fast path
// ---------------------------------------------------------------------------
// Sample tiles of a token group's stream: none when every key fits a token's
// buffer, else one per g = n_tiles / S tiles (8 to 32 of them).
__device__ __forceinline__ int sample_tiles(int n_tiles) {
    if (n_tiles * KT <= kCap) return 0;
    return min(kSampleMax, max(kSampleMin, n_tiles / 32));
}
// The key tiles of a group's stream in visiting order, one per call of next():
// the S sample tiles (i*g + g/2) first, then every other tile in ascending
// order (blocks of g tiles less their sample tile, then the tail past S*g).
// Incremental, so no division runs per tile; past the last tile it returns
// values >= n_tiles.
struct TileSeq {
    int S, g, o, per, i, jb, q, tail;
    __device__ __forceinline__ TileSeq(int n_tiles, int S_) : S(S_), i(0), jb(0), q(0), tail(0) {
        g = S ? n_tiles / S : 1;
        o = g / 2;
        per = g - 1;
    }
    __device__ __forceinline__ int next() {
        int t;
        if (i < S) {
            t = i * g + o;
        } else if (jb < S) {
            t = jb * g + q + (q >= o ? 1 : 0);
            if (++q == per) {
                q = 0;
                ++jb;
            }
        } else {
            t = S * g + tail++;
        }
        ++i;
        return t;
    }
};

// The float whose order key is t, for t at or above the key of -inf (0x007FFFFF).
__device__ __forceinline__ float ord_inv(uint32_t t) {
    return __uint_as_float((t & 0x80000000u) ? (t & 0x7FFFFFFFu) : ~t);
}

__device__ __forceinline__ uint64_t key64(uint32_t ord, int32_t pos) {
    return (static_cast<uint64_t>(ord) << 32) | static_cast<uint32_t>(0xFFFFFFFFu - static_cast<uint32_t>(pos));
}

// The k-th largest 64-bit key over the union of the four quarters of token j's
// buffer (quarter q: entries q*kCapW .. + cnt[q]), by the token's 128 threads
// (t = 0..127); 1 <= k <= total. Returns lo with exactly k keys >= lo (the keys
// are distinct). Radix digits of 8 bits start at the highest bit in which the
// keys differ and stop when the k-th key's bin holds exactly the keys still
// needed.
__device__ __noinline__ uint64_t select_top(Shared &sh, int j, int t, const uint32_t *ord, const int32_t *pos,
                                            const uint32_t (&cnt)[4], uint32_t k, uint32_t *hist) {
    const int lane = t & 31, wq = t >> 5;
    uint64_t mx = 0, mn = ~0ull;
    for (int r = 0; r < 4; ++r)
        for (uint32_t e = t; e < cnt[r]; e += 128) {
            const uint64_t key = key64(ord[r * kCapW + e], pos[r * kCapW + e]);
            mx = max(mx, key);
            mn = min(mn, key);
        }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
    }
    if (lane == 0) {
        sh.red[j][wq][0] = mx;
        sh.red[j][wq][1] = mn;
    }
    token_bar(j);
    for (int w = 0; w < 4; ++w) {
        mx = max(mx, sh.red[j][w][0]);
        mn = min(mn, sh.red[j][w][1]);
    }
    token_bar(j);                                     // red is read before it is written again
    if (mx == mn) return mx;                          // one key in all
    int nbits = __clzll(mx ^ mn);                     // bits every key shares
    uint64_t prefix = nbits ? mx >> (64 - nbits) : 0;
    uint32_t krem = k;
    for (;;) {
        const int width = min(8, 64 - nbits), shift = 64 - nbits - width;
        hist[2 * t] = 0;
        hist[2 * t + 1] = 0;
        token_bar(j);
        for (int r = 0; r < 4; ++r)
            for (uint32_t e = t; e < cnt[r]; e += 128) {
                const uint64_t key = key64(ord[r * kCapW + e], pos[r * kCapW + e]);
                if (nbits == 0 || (key >> (64 - nbits)) == prefix)
                    atomicAdd(&hist[static_cast<uint32_t>(key >> shift) & ((1u << width) - 1)], 1u);
            }
        token_bar(j);
        // bins in descending order: thread t holds bins 255 - 2t and 254 - 2t
        const uint32_t hh = hist[kBins - 1 - 2 * t], hl = hist[kBins - 2 - 2 * t];
        const uint32_t sum = hh + hl;
        uint32_t inc = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t v = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += v;
        }
        if (lane == 31) sh.wtot[j][wq] = inc;
        token_bar(j);
        uint32_t ab = inc - sum;
        for (int w = 0; w < wq; ++w) ab += sh.wtot[j][w];
        if (ab < krem && krem <= ab + sum) {          // exactly one thread
            const bool hi = krem <= ab + hh;
            const uint32_t bin = hi ? kBins - 1 - 2 * t : kBins - 2 - 2 * t;
            sh.sel64[j].prefix = (prefix << width) | bin;
            sh.sel64[j].krem = krem - (hi ? ab : ab + hh);
            sh.sel64[j].bincnt = hi ? hh : hl;
        }
        token_bar(j);
        prefix = sh.sel64[j].prefix;
        krem = sh.sel64[j].krem;
        const uint32_t bincnt = sh.sel64[j].bincnt;
        nbits += width;
        if (bincnt == krem || nbits == 64) return nbits == 64 ? prefix : prefix << (64 - nbits);
    }
}

// kFallback = false: the fast path (sampled threshold), flagging in a.fail the
// groups it could not finish; true: the exact streaming path, run only for the
// flagged groups.
template <bool kFallback>
__global__ void __launch_bounds__(NT, 1)
    indexer_topk_kernel(const IndexerArgs a, const int4 *__restrict__ work, const __grid_constant__ CUtensorMap tmap_k,
                        const __grid_constant__ CUtensorMap tmap_q) {
    extern __shared__ __align__(1024) uint8_t dsm[];
    __shared__ Shared sh;
    const uint32_t raw = smem_u32(dsm);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    uint8_t *sbase = dsm + pad;
    const uint32_t sq = raw + pad, sk = sq + kOffK, sscale = sq + kOffScale;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (kFallback && __ldg(a.fail + blockIdx.x) == 0) return;   // the fast path finished this group
    const int4 it = work[blockIdx.x];
    const int b = it.x, i0 = it.y, ntok = it.z;
    const int q0 = __ldg(a.cu_seqlens + b), P = __ldg(a.prefix_lens + b);
    const int32_t *bt = a.block_table + static_cast<int64_t>(b) * a.max_blocks;
    const int k_hi = P + i0 + ntok;                                   // keys 0 .. k_hi-1
    const int n_tiles = (k_hi + KT - 1) / KT;
    const int S = kFallback ? 0 : sample_tiles(n_tiles);
    if (static_cast<int64_t>(q0) + i0 + ntok > a.total_q) {   // the device cu_seqlens points past the host's count
        if (tid == 0) {
            set_dev_err(a.dev_err, MLA_DEVERR_SEQ_MISMATCH);
            if (!kFallback) a.fail[blockIdx.x] = 0;
        }
        return;
    }
    // tokens with p + 1 <= topk keep every position: a group of only those writes its rows
    if (P + i0 + ntok <= a.topk) {
        for (int j = 0; j < ntok; ++j) {
            const int p = P + i0 + j;
            int32_t *row = a.idx_out + static_cast<int64_t>(q0 + i0 + j) * a.topk;
            for (int e = tid; e < a.topk; e += NT) row[e] = e <= p ? e : -1;
        }
        if (!kFallback && tid == 0) a.fail[blockIdx.x] = 0;
        return;
    }

    if (tid == 0) {
        for (int i = 0; i < NBAR; ++i) mbar_init(smem_u32(&sh.bar[i]), (i == B_D_EMPTY || i == B_D_EMPTY + 1) ? kEpiWarps : 1);
        mbar_fence_init();
        sh.cta_fail = 0;
        for (int j = 0; j < TOK; ++j) sh.fail_tok[j] = 0;
    }
    if (warp == kIssuerWarp) {
        tmem_alloc(smem_u32(&sh.tmem_base), 512);
        tmem_relinquish();
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = sh.tmem_base;

    if (warp == kProducerWarp) {
        // =================== TMA producer ===================
        if (lane == 0) {
            tma_prefetch_desc(&tmap_k);
            tma_prefetch_desc(&tmap_q);
            mbar_expect_tx(smem_u32(&sh.bar[B_Q_FULL]), kQBytes);
            tma_load_2d(sq, &tmap_q, 0, (q0 + i0) * kHidx, smem_u32(&sh.bar[B_Q_FULL]));
            int armed[STAGES], armed_r[kRing];
#pragma unroll
            for (int s = 0; s < STAGES; ++s) armed[s] = -1;
#pragma unroll
            for (int s = 0; s < kRing; ++s) armed_r[s] = -1;
            TileSeq seq(n_tiles, S);
            for (int i = 0; i < n_tiles; ++i) {
                const int s = i % STAGES, r = i % kRing;
                if (i >= STAGES && !wait_bar(sh, a.dev_err, B_K_EMPTY + s, ((i / STAGES) - 1) & 1)) break;
                const int tile = seq.next();
                const int pos0 = tile * KT;
                const int page = pos0 / kPage;
                int blk = page < a.max_blocks ? __ldg(bt + page) : -1;
                const bool bad = blk < 0 || blk >= a.num_blocks;
                if (bad) {   // reported; the epilogue masks these keys
                    set_dev_err(a.dev_err, MLA_DEVERR_BAD_PAGE);
                    blk = 0;
                }
                // ring slot r was last read for step i - kRing: every epilogue warp has
                // started step i - 6 (the producer runs at most STAGES steps ahead of the
                // MMA and the MMA two ahead of the slowest warp), so it is free
                sh.ring_tile[r] = tile;
                sh.ring_bad[r] = bad ? 1 : 0;
                mbar_expect_tx(smem_u32(&sh.bar[B_S_FULL + r]), bad ? 0u : KT * 4u);
                if (!bad)
                    bulk_load(sscale + r * KT * 4, a.ki_scale + static_cast<int64_t>(blk) * kPage + pos0 % kPage, KT * 4,
                              smem_u32(&sh.bar[B_S_FULL + r]));
                armed_r[r] = (i / kRing) & 1;
                mbar_expect_tx(smem_u32(&sh.bar[B_K_FULL + s]), kTileBytes);
                tma_load_2d(sk + s * kTileBytes, &tmap_k, 0, blk * kPage + pos0 % kPage, smem_u32(&sh.bar[B_K_FULL + s]));
                armed[s] = (i / STAGES) & 1;
            }
            // drain: the query copy and the last copy into every stage and ring slot have landed
            bool drained = mbar_wait_cycles(smem_u32(&sh.bar[B_Q_FULL]), 0, kWaitCycles);
            for (int s = 0; s < STAGES; ++s)
                if (armed[s] >= 0)
                    drained = mbar_wait_cycles(smem_u32(&sh.bar[B_K_FULL + s]), armed[s], kWaitCycles) && drained;
            for (int s = 0; s < kRing; ++s)
                if (armed_r[s] >= 0)
                    drained = mbar_wait_cycles(smem_u32(&sh.bar[B_S_FULL + s]), armed_r[s], kWaitCycles) && drained;
            if (!drained) set_dev_err(a.dev_err, MLA_DEVERR_TIMEOUT);
        }
        __syncwarp();
    } else if (warp == kIssuerWarp) {
        // =================== MMA issuer ===================
        if (lane == 0) {
            const uint32_t id = idesc_e4m3(KT, TOK * kHidx, false, false);
            const uint64_t dq = sdesc(sq, 16, 1024, kSw128);
            const uint64_t dk0 = sdesc(sk, 16, 1024, kSw128);
            bool ok = wait_bar(sh, a.dev_err, B_Q_FULL, 0);
            for (int i = 0; i < n_tiles && ok; ++i) {
                const int s = i % STAGES, db = i & 1;
                if (!(ok = wait_bar(sh, a.dev_err, B_K_FULL + s, (i / STAGES) & 1))) break;
                if (i >= 2 && !(ok = wait_bar(sh, a.dev_err, B_D_EMPTY + db, ((i >> 1) - 1) & 1))) break;
                fence_after_sync();
                const uint64_t dk = dk0 + static_cast<uint64_t>((s * kTileBytes) >> 4);
#pragma unroll
                for (int ks = 0; ks < kDidx / 32; ++ks)
                    mma_e4m3_ss(tmem + kDCols * db, dk + 2 * ks, dq + 2 * ks, id, ks > 0 ? 1u : 0u);
                mma_commit(smem_u32(&sh.bar[B_K_EMPTY + s]));
                mma_commit(smem_u32(&sh.bar[B_D_FULL + db]));
            }
            mma_commit(smem_u32(&sh.bar[B_FINAL]));
        }
        __syncwarp();
    } else {
        // =================== epilogue + selection (warps 0-11) ===================
        const int quad = warp & 3, j = warp >> 2;                     // keys 32 quad.., token j
        const int t128 = tid - 128 * j;                               // thread within the token's four warps
        const uint32_t lane_addr = static_cast<uint32_t>(32 * quad) << 16;
        const int kk = 32 * quad + lane;                              // key within the tile
        const int p_tok = P + i0 + j;                                 // this token's position
        const bool live = j < ntok;
        const bool select = live && p_tok + 1 > a.topk;              // the same in the token's four warps
        uint32_t *ordb = reinterpret_cast<uint32_t *>(sbase + kOffOrd) + j * kCap;
        int32_t *posb = reinterpret_cast<int32_t *>(sbase + kOffPos) + j * kCap;
        uint32_t *hist = reinterpret_cast<uint32_t *>(sbase + kOffHist) + j * kBins;
        // the token's head weights, halved (see relu2_bits), as pairs, for every tile
        const float4 *wg = reinterpret_cast<const float4 *>(a.w + static_cast<int64_t>(q0 + i0 + min(j, ntok - 1)) *
                                                            a.w_stride);
        uint64_t wp[kHidx / 2];
#pragma unroll
        for (int h4 = 0; h4 < kHidx / 4; ++h4) {
            const float4 w4 = __ldg(wg + h4);
            wp[2 * h4] = pack2(0.5f * w4.x, 0.5f * w4.y);
            wp[2 * h4 + 1] = pack2(0.5f * w4.z, 0.5f * w4.w);
        }
        const float *ring_scale = reinterpret_cast<const float *>(sbase + kOffScale);
        // exact path: the token's whole buffer in position order; fast path: this warp's quarter
        int n_c = 0;
        uint32_t thr = 0;
        bool warm = false;                 // exact path: a threshold is set; fast path: the sample's threshold is
        bool ok = true;                    // every wait so far succeeded
        bool fits = true;                  // fast path: this warp's quarter has not overflowed
        uint32_t *my_ord = ordb + (kFallback ? 0 : quad * kCapW);
        int32_t *my_pos = posb + (kFallback ? 0 : quad * kCapW);
        float thr_f = 0.f;                 // fast path: the float whose order key is thr
        for (int i = 0; i < n_tiles; ++i) {
            const int db = i & 1, r = i % kRing;
            // A wait that gives up must not leave the token's other warps at a named
            // barrier: the warp stops waiting (fast path) or carries the failure through
            // the count exchange so all four leave at the same tile (exact path).
            bool got = false;
            if (kFallback || ok) {
                got = wait_bar(sh, a.dev_err, B_S_FULL + r, (i / kRing) & 1) &&
                      wait_bar(sh, a.dev_err, B_D_FULL + db, (i >> 1) & 1);
                if (!got && (!kFallback || !select)) ok = false;
            }
            // the step's tile, page flag and this thread's key scale, staged by the producer
            const int pos = sh.ring_tile[r] * KT + kk;
            const bool ok_key = sh.ring_bad[r] == 0;
            const float sig = ring_scale[r * KT + kk];
            if (kFallback && !got && !select) break;
            uint64_t acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};   // eight independent chains
            if (got) {
                fence_after_sync();
                // heads in four chunks of 16 columns, the load of chunk c+1 in flight
                // while chunk c is reduced
                const uint32_t col0 = tmem + lane_addr + kDCols * db + 64u * j;
                uint32_t d[2][16];
                tmem_ld16(col0, d[0]);
                tmem_ld_wait();
#pragma unroll
                for (int c = 0; c < 4; ++c) {              // heads 16c .. 16c+15
                    if (c < 3) tmem_ld16(col0 + 16u * (c + 1), d[(c + 1) & 1]);
#pragma unroll
                    for (int pi = 0; pi < 8; ++pi) {
                        const uint32_t *x = d[c & 1] + 2 * pi;
                        ffma2(acc[pi], wp[8 * c + pi], pack2(relu2_bits(x[0]), relu2_bits(x[1])));
                    }
                    if (c < 3) tmem_ld_wait();
                    if (c == 2) {      // every column read: the buffer goes back to the MMA
                        fence_before_sync();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(smem_u32(&sh.bar[B_D_EMPTY + db]));
                    }
                }
            }
            if (!select) continue;
            const float sc = ((sum2(acc[0]) + sum2(acc[1])) + (sum2(acc[2]) + sum2(acc[3]))) +
                             ((sum2(acc[4]) + sum2(acc[5])) + (sum2(acc[6]) + sum2(acc[7])));
            const float sv = ok_key ? sig * sc : -INFINITY;
            if constexpr (!kFallback) {
                // ---- fast path: append to this warp's quarter, no barrier ----
                // Past the sample a key enters iff its order key is >= thr, decided on the
                // floats (the order keys keep the order of non-NaN floats and tie -0 with
                // +0; thr is at or above the key of -inf, so its float is no NaN, and a NaN
                // score compares false, as its key 0 would). An overflowing warp keeps consuming tiles (the MMA waits
                // for every warp) but inserts nothing more: the exact path redoes the group.
                const bool hit = ok && fits && pos <= p_tok && (!warm || sv >= thr_f);
                const uint32_t m = __ballot_sync(0xffffffffu, hit);
                if (m != 0u) {
                    const int c = __popc(m);
                    if (n_c + c > kCapW) {
                        fits = false;
                    } else {
                        if (hit) {
                            const int e = n_c + __popc(m & lanemask_lt());
                            my_ord[e] = ord_f32(sv);
                            my_pos[e] = pos;
                        }
                        n_c += c;
                    }
                }
                if (i == S - 1) {
                    // ---- end of the sample: the threshold (the same in the token's warps) ----
                    if (lane == 0) {
                        sh.wcnt[j][quad] = static_cast<uint32_t>(n_c);
                        if (!ok || !fits) sh.fail_tok[j] = 1;
                    }
                    token_bar(j);
                    const uint32_t cnt[4] = {sh.wcnt[j][0], sh.wcnt[j][1], sh.wcnt[j][2], sh.wcnt[j][3]};
                    const uint32_t m_s = cnt[0] + cnt[1] + cnt[2] + cnt[3];
                    const bool bad = sh.fail_tok[j] != 0;
                    token_bar(j);                          // wcnt is read before it is written again
                    // the k-th largest score is expected at sample rank e; the threshold sits
                    // four standard deviations (and 4) past it
                    const float ex = static_cast<float>(a.topk) * static_cast<float>(m_s) / static_cast<float>(p_tok + 1);
                    const uint32_t r = static_cast<uint32_t>(ceilf(ex + 4.f * sqrtf(ex) + 4.f));
                    if (!bad && r < m_s) {
                        thr = static_cast<uint32_t>(select_top(sh, j, t128, ordb, posb, cnt, r, hist) >> 32);
                        // below the key of -inf (only NaN scores rank there) every key enters
                        warm = thr >= 0x007FFFFFu;
                        thr_f = warm ? ord_inv(thr) : 0.f;
                        // keep this quarter's sample entries at or above the threshold (in order)
                        int kept = 0;
                        for (int e0 = 0; e0 < n_c; e0 += 32) {
                            const int e = e0 + lane;
                            const uint32_t oe = e < n_c ? my_ord[e] : 0u;
                            const int32_t pe = e < n_c ? my_pos[e] : 0;
                            const bool keep = e < n_c && oe >= thr;
                            const uint32_t mk = __ballot_sync(0xffffffffu, keep);
                            if (keep) {
                                const int d2 = kept + __popc(mk & lanemask_lt());
                                my_ord[d2] = oe;
                                my_pos[d2] = pe;
                            }
                            kept += __popc(mk);
                        }
                        n_c = kept;
                    }
                }
            } else {
                // ---- exact path: per-tile count exchange, slots in position order ----
                const uint32_t o = ord_f32(sv);
                const bool hit = got && pos <= p_tok && (!warm || o > thr);
                const uint32_t m = __ballot_sync(0xffffffffu, hit);
                if (lane == 0) sh.cntx[j][i & 1][quad] = static_cast<uint32_t>(__popc(m)) | (got ? 0u : 0x80000000u);
                token_bar(j);
                uint4 c4 = *reinterpret_cast<const uint4 *>(sh.cntx[j][i & 1]);
                if ((c4.x | c4.y | c4.z | c4.w) & 0x80000000u) {   // a warp of the token gave up
                    ok = false;
                    break;
                }
                const uint32_t before = (quad > 0 ? c4.x : 0u) + (quad > 1 ? c4.y : 0u) + (quad > 2 ? c4.z : 0u);
                if (hit) {
                    const int e = n_c + static_cast<int>(before + __popc(m & lanemask_lt()));
                    ordb[e] = o;
                    posb[e] = pos;
                }
                n_c += static_cast<int>(c4.x + c4.y + c4.z + c4.w);
                if (n_c > kCap - KT) n_c = compact(sh, j, t128, ordb, posb, hist, n_c, a.topk, false, thr, warm);
            }
        }
        if (live) {
            int32_t *row = a.idx_out + static_cast<int64_t>(q0 + i0 + j) * a.topk;
            if (!select) {
                for (int e = t128; e < a.topk; e += 128) row[e] = e <= p_tok ? e : -1;
            } else if constexpr (!kFallback) {
                // ---- fast path: exact top k of the union of the four quarters ----
                if (lane == 0) {
                    sh.wcnt[j][quad] = static_cast<uint32_t>(n_c);
                    if (!ok || !fits) sh.fail_tok[j] = 1;
                }
                token_bar(j);
                const uint32_t cnt[4] = {sh.wcnt[j][0], sh.wcnt[j][1], sh.wcnt[j][2], sh.wcnt[j][3]};
                const uint32_t total = cnt[0] + cnt[1] + cnt[2] + cnt[3];
                const uint32_t k = static_cast<uint32_t>(a.topk);
                if (sh.fail_tok[j] != 0 || total < k) {
                    if (t128 == 0) sh.cta_fail = 1;        // the threshold was too high, or a quarter overflowed
                } else {
                    const uint64_t lo = select_top(sh, j, t128, ordb, posb, cnt, k, hist);
                    // the k positions at or above lo, quarter by quarter, each quarter in its
                    // stored order: a deterministic order, as every quarter's contents are
                    uint32_t base = 0;
                    for (int r = 0; r < 4; ++r)
                        for (uint32_t e0 = 0; e0 < cnt[r]; e0 += 128) {
                            const uint32_t e = e0 + t128;
                            const bool keep = e < cnt[r] && key64(ordb[r * kCapW + e], posb[r * kCapW + e]) >= lo;
                            const uint32_t mk = __ballot_sync(0xffffffffu, keep);
                            if (lane == 0) sh.wcnt[j][quad] = static_cast<uint32_t>(__popc(mk));
                            token_bar(j);
                            uint32_t before = base;
                            for (int w = 0; w < quad; ++w) before += sh.wcnt[j][w];
                            const uint32_t all = sh.wcnt[j][0] + sh.wcnt[j][1] + sh.wcnt[j][2] + sh.wcnt[j][3];
                            if (keep) {
                                const uint32_t d2 = before + __popc(mk & lanemask_lt());
                                if (d2 < k) row[d2] = posb[r * kCapW + e];
                            }
                            base += all;
                            token_bar(j);            // wcnt is read before it is written again
                        }
                    if (base != k) {       // exactly k keys are at or above lo; report instead of guessing
                        if (t128 == 0) set_dev_err(a.dev_err, MLA_DEVERR_INTERNAL);
                        for (int e = t128; e < a.topk; e += 128) row[e] = -1;
                    }
                }
            } else if (ok) {
                n_c = compact(sh, j, t128, ordb, posb, hist, n_c, a.topk, true, thr, warm);
                if (n_c == a.topk) {
                    for (int e = t128; e < a.topk; e += 128) row[e] = posb[e];
                } else {       // the compaction leaves exactly topk entries; report instead of guessing
                    if (t128 == 0) set_dev_err(a.dev_err, MLA_DEVERR_INTERNAL);
                    for (int e = t128; e < a.topk; e += 128) row[e] = -1;
                }
            }
        }
    }

    // ----- teardown -----
    __syncthreads();
    if (!kFallback && tid == 0) a.fail[blockIdx.x] = sh.cta_fail;
    if (warp == kIssuerWarp) {
        if (!mbar_wait_cycles(smem_u32(&sh.bar[B_FINAL]), 0, kWaitCycles)) set_dev_err(a.dev_err, MLA_DEVERR_TIMEOUT);
        fence_after_sync();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace idxf

cudaError_t launch_indexer_topk(const IndexerArgs &a, const int4 *work, int n_work, const CUtensorMap &tmap_k,
                                const CUtensorMap &tmap_q, cudaStream_t st) {
    for (auto fn : {idxf::indexer_topk_kernel<false>, idxf::indexer_topk_kernel<true>}) {
        const cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, idxf::kDynSmem);
        if (e != cudaSuccess) return e;
    }
    if (n_work > 0) {
        idxf::indexer_topk_kernel<false><<<n_work, idxf::NT, idxf::kDynSmem, st>>>(a, work, tmap_k, tmap_q);
        idxf::indexer_topk_kernel<true><<<n_work, idxf::NT, idxf::kDynSmem, st>>>(a, work, tmap_k, tmap_q);
    }
    return cudaGetLastError();
}

}  // namespace mla

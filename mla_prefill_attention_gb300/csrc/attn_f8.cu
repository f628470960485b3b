// MLA prefill attention, dense and sparse, with e4m3 tensor-core operands
// (tcgen05 kind::f8f6f4).
//
// The cache holds e4m3 codes, so the key/value operand needs no conversion: key
// tiles go straight from the pages into 128-byte-swizzled shared memory (dense:
// TMA boxes; sparse: rows gathered by index) and both MMAs read the codes as
// they are. The other operand of each product is split into two e4m3 terms whose
// sum carries bf16 precision:
//
//   Q/s_Q = Qh + Ql   (s_Q a power of two per row; for bf16 input the split is
//                      exact while |Q/s_Q| >= 2^-2, and the largest element sits
//                      in [128, 256))
//   P     = Ph + Pl   (P rounded to f16 first; 8 significant bits in total)
//
//   S   = Qh K^T + Ql K^T          M=64, N=BN keys, K=576 (A = Qh, Ql in TMEM)
//   u   = S s_Q sigma sm_scale log2(e) + log2(sigma)
//   P   = 2^(u - m + 6),  l += P / sigma     (m: reference max, log2 domain)
//   O  += Ph V + Pl V              M=64, N=256 x 2 chunks of the 512 value dims
//
// and out = O / l, lse = ln2 (m - 6 + log2 l). The offset 6 keeps the largest
// weights of a row in the normal e4m3 range (a P of 1 would leave most of the
// row's mass in subnormals); the reference max moves when a tile raises a row's
// max by more than 2 (log2 units), so P never exceeds 2^8 < 448.
//
// Each M=64 e4m3 MMA runs at 4096 MAC/clk per SM, twice the f16 rate, so the two
// terms cost what one f16 product would; what goes away is the conversion pass
// (no warp writes key data to shared memory) and half of the operand bytes.
//
// TMEM (M=64 layout: row r in lane 32*(r/16) + r%16 + 16*h, h = lane half)
//   h=0 cols   0..143 : Qh (576 codes, four per column)
//   h=0 cols 144..287 : Ql
//   h=0 cols 288..    : S (dense: one buffer of 128 columns; sparse: two of 96)
//   h=1 cols   0..511 : O
//
// Shared memory
//   dense: 2 stages x 5 slices x [128 keys][128 B]; sparse: 3 stages x 5 slices x
//     [96 keys][128 B]; 128-byte swizzle. Slices 0-3 are the value dims (K-major
//     for QK, MN-major for PV); slice 4 holds the 64 RoPE dims (upper 64 bytes
//     unused). A dense stage is released in three parts as the tensor core is done
//     with them (the RoPE slice after QK, value dims 0-255 and 256-511 after the
//     two PV chunks); a sparse stage is released whole after PV.
//   P: 2 buffers x {Ph, Pl} x [64 rows][BN keys], K-major without swizzle
//     (16-byte x 8-row core matrices; 128 B apart along the keys, BN/16 * 128 B
//     apart along the rows)
//
// Warps
//   dense (10): 0-7 softmax (two per TMEM lane quadrant, 64 keys of a tile each;
//     they also split Q into TMEM and run the epilogue), 8 TMA producer and key
//     metadata, 9 MMA issue.
//   sparse (9): 0-3 softmax (96 keys each), two pairs of gather warps (4 and 6,
//     7 and 8: cp.async rows by index, completing on the stage barrier), 5 MMA
//     issue.
// Keys past a row's causal limit, padding indices and invalid pages are zeroed in
// shared memory (an unwritten cache row could hold a NaN code, which a zero
// weight would not cancel). Every wait is bounded; one that runs out sets
// MLA_DEVERR_TIMEOUT.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <type_traits>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace mla {
namespace f8attn {

using namespace tc;

constexpr int BM = 64;                          // query rows per tile
// Key tiles: dense 128 keys (a QK MMA of N=128 runs at its nominal rate under a full
// SM; N=96 loses ~40%), sparse 96. Dense keeps two stages, each released in three
// parts (RoPE after QK, value dims 0-255 and 256-511 after the two PV chunks), and one
// S buffer; sparse keeps three whole stages and two S buffers.
template <bool S> constexpr int kBN = S ? 96 : 128;
template <bool S> constexpr int kStages = S ? 3 : 2;
template <bool S> constexpr int kParts = S ? 1 : 3;
template <bool S> constexpr int kSBufs = S ? 2 : 1;
constexpr int kBNMax = 128;
// Warps. dense: 10 = 8 softmax (two per TMEM lane quadrant, 64 of a tile's 128 keys
// each: the softmax of tile t then ends before QK(t+1) does), TMA producer (8),
// issuer (9). sparse: 9 = 4 softmax (96 keys each; with eight, the register cap of
// 13 warps costs more than the shorter softmax gains), issuer (5) and two pairs of
// gather warps (4, 6 and 7, 8: a warp keeps only so many row copies in flight).
template <bool kSparse> constexpr int kSmWarps = kSparse ? 4 : 8;
template <bool kSparse> constexpr int kSmKeys = kBN<kSparse> * 4 / kSmWarps<kSparse>;   // keys per softmax warp
template <bool kSparse> constexpr int kThreads = kSparse ? 288 : 320;
template <bool kSparse> constexpr int kIssuerWarp = kSparse ? 5 : 9;
constexpr int kProducerWarp = 8;   // dense
// Gather pair 0 (warps 4, 6) takes even tiles, pair 1 (7, 8) odd ones; each warp of
// a pair copies half of the tile's rows. A pair waits for a stage at most one
// phase ahead of its completed one (its previous tile waited for the phase before),
// which keeps the parity waits exact.
__device__ __forceinline__ int gather_pair(int warp) { return warp == 4 || warp == 6 ? 0 : 1; }
__device__ __forceinline__ int gather_half(int warp) { return warp == 4 || warp == 7 ? 0 : 1; }
constexpr int kSlices = 5;
template <bool S> constexpr int kSliceBytes = kBN<S> * 128;
template <bool S> constexpr int kStageBytes = kSlices * kSliceBytes<S>;
template <bool S> constexpr int kPBytes = BM * kBN<S>;          // one e4m3 term of P
template <bool S> constexpr int kPSbo = kBN<S> / 16 * 128;      // P: 8-row band stride
template <bool S> constexpr int kOffP = kStages<S> * kStageBytes<S>;
template <bool S> constexpr int kDynSmem = 1024 + kOffP<S> + 4 * kPBytes<S>;
constexpr int kGroupRows = 32;                  // sparse metadata: keys per lane round
constexpr long long kWaitCycles = 200000000LL;
constexpr float kRescaleThreshold = 2.0f;
constexpr float kPOffset = 6.0f;
static_assert(kPage % kBN<false> == 0, "a dense key tile must not straddle a page");

constexpr uint32_t kColQh = 0, kColQl = 144, kColS = 288;
constexpr uint32_t kHalf1 = 16u << 16;

enum Bar {
    B_FULL = 0,          // [part * stages + stage] producer (+TMA bytes) -> issuer: loaded
    B_EMPTY = 9,         // [part * stages + stage] issuer (commit) -> producer: done with it
    B_META = 18,         // [4] producer -> softmax: key metadata of tile t, ring t&3
    B_S_FULL = 22,       // [2] issuer (commit) -> softmax
    B_S_FREE = 24,       // [2] softmax -> issuer
    B_P_FULL = 26,       // [2] softmax -> issuer (P written, O rescaled)
    B_PV_DONE = 28,      // [2] issuer (commit) -> softmax
    B_Q_FULL = 30,       //     softmax -> issuer
    B_O_FREE = 31,       //     softmax -> issuer: epilogue done with O
    B_FINAL = 32,        //     issuer -> teardown
    B_FIX = 33,          //     producer's own: a tile whose tail it zeroes
    B_XCH = 34,          // [4] the two softmax warps of a quadrant: tile maxima, then row sums
    NBAR = 38
};

struct __align__(16) KeyMeta {
    float4 sl[kBNMax / 2];    // sigma of keys 2p, 2p+1; log2 sigma of both (-inf: masked)
    float2 isig[kBNMax / 2];  // 1/sigma of both
};

struct Shared {
    KeyMeta meta[4];
    float xmax[2][4][2][16];   // [tile parity][quadrant][key half][row]: tile maxima
    float xsum[4][2][16];      // [quadrant][key half][row]: row sums at the epilogue
    uint64_t bar[NBAR];
    uint32_t tmem_base;
};

struct Wait {
    Shared *sh;
    int32_t *dev_err;
    __device__ bool operator()(int b, uint32_t parity) const {
        if (mbar_wait_cycles(smem_u32(&sh->bar[b]), parity, kWaitCycles)) return true;
        set_dev_err(dev_err, MLA_DEVERR_TIMEOUT);
        return false;
    }
};

struct RowTile {
    int64_t grow0;      // first global query row (token*H + head)
    int nvalid;         // valid rows
    int n_ktiles;       // key tiles to visit
    int key_last;       // dense: last key position visible to any row; sparse: the token's position
    int b;              // sequence
    int64_t tok;        // sparse: the token
};

// Dense: row tile `tile` of sequence b. Sparse: heads h0.. of token tok, whose
// top-k indices give its keys.
template <bool kSparse>
__device__ __forceinline__ RowTile make_tile(const AttnArgs &a, int b, int tile, int64_t tok, int h0) {
    RowTile rt;
    if (kSparse) {
        rt.b = find_seq(a.cu_seqlens, a.batch, tok);
        rt.tok = tok;
        rt.grow0 = tok * a.H + h0;
        rt.nvalid = min(BM, a.H - h0);
        rt.key_last = __ldg(a.prefix_lens + rt.b) + static_cast<int>(tok - __ldg(a.cu_seqlens + rt.b));
        rt.n_ktiles = (a.topk + kBN<true> - 1) / kBN<true>;
    } else {
        const int q0 = __ldg(a.cu_seqlens + b), qn = __ldg(a.cu_seqlens + b + 1) - q0;
        const int P = __ldg(a.prefix_lens + b);
        const int rows = qn * a.H, r_lo = tile * BM;
        rt.b = b;
        rt.tok = -1;
        rt.grow0 = static_cast<int64_t>(q0) * a.H + r_lo;
        rt.nvalid = min(BM, rows - r_lo);
        rt.key_last = P + (r_lo + rt.nvalid - 1) / a.H;
        rt.n_ktiles = rt.key_last / kBN<false> + 1;
    }
    return rt;
}

// A dense work item is backed when each of its row tiles lies wholly inside both
// the device's and the host's count of rows. An item that is not (an empty filler
// item, or a device cu_seqlens that disagrees with its host mirror) is skipped
// whole, before any barrier or TMEM is set up, so no row at or past the host's
// count is ever touched. Out of line: the check runs once per CTA and must not
// share registers with the kernel's loops.
__device__ __noinline__ bool dense_item_backed(const AttnArgs &a, int b, int tile0, int tile1) {
    auto ok = [&](int tile) {
        if (tile < 0) return false;
        const int64_t q0 = __ldg(a.cu_seqlens + b), qn = __ldg(a.cu_seqlens + b + 1) - q0;
        const int64_t rows = qn * a.H, r_lo = static_cast<int64_t>(tile) * BM;
        const int64_t nvalid = min(static_cast<int64_t>(BM), rows - r_lo);
        return nvalid > 0 && q0 * a.H + r_lo + nvalid <= a.total_q * a.H;
    };
    return ok(tile0) && (tile1 < 0 || ok(tile1));
}

// Last key position row `row` may see (dense), the token's position (sparse); -1: no row.
template <bool kSparse>
__device__ __forceinline__ int row_limit(const AttnArgs &a, const RowTile &rt, int row) {
    if (row >= rt.nvalid) return -1;
    if (kSparse) return rt.key_last;
    const int r_lo = static_cast<int>(rt.grow0 - static_cast<int64_t>(__ldg(a.cu_seqlens + rt.b)) * a.H);
    return __ldg(a.prefix_lens + rt.b) + (r_lo + row) / a.H;
}

__device__ __forceinline__ uint32_t swz(int row, int chunk) {  // byte offset in a [rows][128 B] SW128 slice
    return static_cast<uint32_t>((row >> 3) * 1024 + (row & 7) * 128 + ((chunk ^ (row & 7)) << 4));
}
__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst), "l"(src) : "memory");
}
// The mbarrier receives one arrival once all of this thread's earlier cp.async copies
// have landed (its expected count includes these arrivals); the thread does not wait.
__device__ __forceinline__ void cp_async_arrive(uint32_t mbar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(mbar) : "memory");
}
__device__ __align__(16) uint8_t g_zero_row[128];   // the source of padding rows

struct Walk {
    int n0, total;
    __device__ int r(int t) const { return t < n0 ? 0 : 1; }
    __device__ int j(int t) const { return t < n0 ? t : t - n0; }
};

// ---------------------------------------------------------------------------
// e4m3 conversions
// ---------------------------------------------------------------------------
// Two floats -> e4m3 codes (lo in byte 0), round to nearest even, saturating.
__device__ __forceinline__ uint32_t e4m3x2_of(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}
__device__ __forceinline__ uint32_t e4m3x2_of_f16x2(uint32_t h) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(r) : "r"(h));
    return r;
}
__device__ __forceinline__ uint32_t f16x2_of_e4m3x2(uint32_t c) {
    uint32_t r;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(static_cast<uint16_t>(c)));
    return r;
}
__device__ __forceinline__ uint32_t hsub2_bits(uint32_t x, uint32_t y) {
    uint32_t r;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(x), "r"(y));
    return r;
}
__device__ __forceinline__ float2 float2_of_f16x2(uint32_t h) {
    __half2 v;
    *reinterpret_cast<uint32_t *>(&v) = h;
    return __half22float2(v);
}
// (p0, p1) -> (head codes) | (tail codes) << 16: head = e4m3 of the f16 values
// (rounded to nearest, so the remainder is at most half a head ulp), tail =
// e4m3 of what the head leaves (exact in f16).
__device__ __forceinline__ uint32_t split_p2(float p0, float p1) {
    const uint32_t h = pack_half2(p0, p1);
    const uint32_t hd = e4m3x2_of_f16x2(h);
    const uint32_t tl = e4m3x2_of_f16x2(hsub2_bits(h, f16x2_of_e4m3x2(hd)));
    return hd | (tl << 16);
}
// paired f32 arithmetic (two IEEE operations per instruction)
__device__ __forceinline__ uint64_t pk2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ float2 upk2(uint64_t v) {
    float2 f;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(f.x), "=f"(f.y) : "l"(v));
    return f;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// Q rows ra, rb of the tile -> Qh, Ql in TMEM (lane half 0; 16x256b layout:
// column group g holds dims 32g + 8tc .. +7 of this thread's rows). Returns the
// logit scale s_Q * sm_scale * log2(e) per row.
__device__ __noinline__ void load_q_split(const AttnArgs &a, const RowTile &rt, uint32_t tq_addr, int ra, int rb,
                                             int tc, int g_first, int g_count, float &rs_a, float &rs_b) {
    const bool oka = ra < rt.nvalid, okb = rb < rt.nvalid;
    const uint4 *qa = reinterpret_cast<const uint4 *>(a.q + (rt.grow0 + (oka ? ra : 0)) * kDqk + 8 * tc);
    const uint4 *qb = reinterpret_cast<const uint4 *>(a.q + (rt.grow0 + (okb ? rb : 0)) * kDqk + 8 * tc);
    float mxa = 0.f, mxb = 0.f;
#pragma unroll 9
    for (int g = 0; g < 18; ++g) {
        const uint4 va = oka ? __ldg(qa + 4 * g) : make_uint4(0, 0, 0, 0);
        const uint4 vb = okb ? __ldg(qb + 4 * g) : make_uint4(0, 0, 0, 0);
        const __nv_bfloat162 *ha = reinterpret_cast<const __nv_bfloat162 *>(&va);
        const __nv_bfloat162 *hb = reinterpret_cast<const __nv_bfloat162 *>(&vb);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 fa = __bfloat1622float2(ha[e]), fb = __bfloat1622float2(hb[e]);
            mxa = fmaxf(mxa, fmaxf(fabsf(fa.x), fabsf(fa.y)));
            mxb = fmaxf(mxb, fmaxf(fabsf(fb.x), fabsf(fb.y)));
        }
    }
    mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, 1));
    mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, 1));
    mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, 2));
    mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, 2));
    // s_Q = 2^(e - 8) for max = f 2^e, f in [0.5, 1): the largest |Q/s_Q| is in [128, 256)
    int ea = 0, eb = 0;
    if (mxa > 0.f) frexpf(mxa, &ea);
    if (mxb > 0.f) frexpf(mxb, &eb);
    const float ia = mxa > 0.f ? ldexpf(1.f, 8 - ea) : 1.f, ib = mxb > 0.f ? ldexpf(1.f, 8 - eb) : 1.f;
    rs_a = a.sm_scale_log2 / ia;
    rs_b = a.sm_scale_log2 / ib;
    // a row's 8 dims of one group -> (head word pair, tail word pair)
    auto split8 = [](const uint4 &v, float inv, uint32_t (&hd)[2], uint32_t (&tl)[2]) {
        const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&v);
#pragma unroll
        for (int w = 0; w < 2; ++w) {
            const float2 f0 = __bfloat1622float2(h[2 * w]), f1 = __bfloat1622float2(h[2 * w + 1]);
            const float x0 = f0.x * inv, x1 = f0.y * inv, x2 = f1.x * inv, x3 = f1.y * inv;
            const uint32_t h01 = e4m3x2_of(x0, x1), h23 = e4m3x2_of(x2, x3);
            const float2 g01 = float2_of_f16x2(f16x2_of_e4m3x2(h01)), g23 = float2_of_f16x2(f16x2_of_e4m3x2(h23));
            hd[w] = h01 | (h23 << 16);
            tl[w] = e4m3x2_of(x0 - g01.x, x1 - g01.y) | (e4m3x2_of(x2 - g23.x, x3 - g23.y) << 16);
        }
    };
    // this warp's column groups g_first .. g_first + g_count - 1 (all 18, or one half), four
    // at a time, the next four groups' loads in flight while the current ones are split
    constexpr int kC = 4;
    uint4 buf[2][2 * kC];
    auto fetch = [&](int g0, uint4 (&b)[2 * kC]) {
#pragma unroll
        for (int i = 0; i < kC; ++i) {
            const int g = g0 + i;
            const bool in = g < g_first + g_count;
            b[2 * i] = in && oka ? __ldg(qa + 4 * g) : make_uint4(0, 0, 0, 0);
            b[2 * i + 1] = in && okb ? __ldg(qb + 4 * g) : make_uint4(0, 0, 0, 0);
        }
    };
    fetch(g_first, buf[0]);
#pragma unroll
    for (int c = 0; c < (18 + kC - 1) / kC; ++c) {
        const int g0 = g_first + kC * c;
        if (g0 >= g_first + g_count) break;
        if (g0 + kC < g_first + g_count) fetch(g0 + kC, buf[(c + 1) & 1]);
        uint32_t wh[4 * kC], wl[4 * kC];
#pragma unroll
        for (int i = 0; i < kC; ++i) {
            uint32_t ha[2], la[2], hb[2], lb[2];
            split8(buf[c & 1][2 * i], ia, ha, la);
            split8(buf[c & 1][2 * i + 1], ib, hb, lb);
            wh[4 * i + 0] = ha[0];
            wh[4 * i + 1] = ha[1];
            wh[4 * i + 2] = hb[0];
            wh[4 * i + 3] = hb[1];
            wl[4 * i + 0] = la[0];
            wl[4 * i + 1] = la[1];
            wl[4 * i + 2] = lb[0];
            wl[4 * i + 3] = lb[1];
        }
        const int left = g_first + g_count - g0;        // 4 or more, 2 (all 18) or 1 (a half)
        if (left >= kC) {
            tmem_st_16x256b_x4(tq_addr + kColQh + 8 * g0, wh);
            tmem_st_16x256b_x4(tq_addr + kColQl + 8 * g0, wl);
        } else if (left == 2) {
            tmem_st_16x256b_x2(tq_addr + kColQh + 8 * g0, wh);
            tmem_st_16x256b_x2(tq_addr + kColQl + 8 * g0, wl);
        } else {
            tmem_st_16x256b_x1(tq_addr + kColQh + 8 * g0, wh);
            tmem_st_16x256b_x1(tq_addr + kColQl + 8 * g0, wl);
        }
    }
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
template <bool kSparse>
__global__ void __launch_bounds__(kThreads<kSparse>, 1)
    attn_f8_kernel(const AttnArgs a, const int4 *__restrict__ work, const __grid_constant__ CUtensorMap tmap_kv) {
    extern __shared__ __align__(1024) uint8_t dsm[];
    __shared__ Shared sh;
    const uint32_t raw = smem_u32(dsm);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    uint8_t *sbase = dsm + pad;
    const uint32_t sbase_a = raw + pad;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // the CTA's two row tiles: dense, a work item (sequence, tile, tile or -1);
    // sparse, tokens 2x and 2x+1 (if any) for heads 64y..
    int b = 0, tiles[2] = {-1, -1}, h0 = 0;
    int64_t toks[2] = {-1, -1};
    int n_rt;
    if (kSparse) {
        toks[0] = a.tok_begin + 2 * static_cast<int64_t>(blockIdx.x);
        toks[1] = toks[0] + 1 < a.tok_end ? toks[0] + 1 : -1;
        h0 = blockIdx.y * BM;
        n_rt = toks[1] >= 0 ? 2 : 1;
    } else {
        const int4 it = work[blockIdx.x];
        b = it.x;
        tiles[0] = it.y;
        tiles[1] = it.z;
        n_rt = tiles[1] >= 0 ? 2 : 1;
    }
    auto tile_of = [&](int r) { return make_tile<kSparse>(a, b, tiles[r], toks[r], h0); };
    if (!kSparse && !dense_item_backed(a, b, tiles[0], tiles[1])) {
        // (filler items are reported by the kernel that wrote them)
        if (tid == 0 && tiles[0] >= 0) set_dev_err(a.dev_err, MLA_DEVERR_SEQ_MISMATCH);
        return;
    }
    Walk walk;
    walk.n0 = tile_of(0).n_ktiles;
    walk.total = walk.n0 + (n_rt > 1 ? tile_of(1).n_ktiles : 0);

    if (tid == 0) {
        for (int i = 0; i < NBAR; ++i) {
            uint32_t cnt = 1;
            if ((i >= B_S_FREE && i < B_S_FREE + 2) || (i >= B_P_FULL && i < B_P_FULL + 2) || i == B_Q_FULL ||
                i == B_O_FREE)
                cnt = kSmWarps<kSparse>;
            if (kSparse && i >= B_FULL && i < B_FULL + kStages<true>) cnt = 64;  // every lane of a gather pair
            if (i >= B_XCH && i < B_XCH + 4) cnt = 2;                          // the quadrant's two softmax warps
            mbar_init(smem_u32(&sh.bar[i]), cnt);
        }
        mbar_fence_init();
    }
    if (warp == kIssuerWarp<kSparse>) {
        tmem_alloc(smem_u32(&sh.tmem_base), 512);
        tmem_relinquish();
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = sh.tmem_base;
    const Wait wait{&sh, a.dev_err};

    if (!kSparse && warp == kProducerWarp) {
        // =================== TMA producer + key metadata ===================
        // Tile t: one 128-row box per slice (a tile lies in one page). Its parts go
        // as they are released: the RoPE slice once QK(t-2) is done with it, value
        // slices 0-1 and 2-3 once the two PV chunks of tile t-2 are. The block-table
        // and scale loads are issued before the first wait. A tile that reaches past
        // the causal limit is loaded whole, then its tail rows are zeroed (an
        // unwritten cache row could hold a NaN code, which a zero weight would not
        // cancel), and all three parts are released together.
        constexpr int BN = kBN<false>, ST = kStages<false>;
        if (lane == 0) tma_prefetch_desc(&tmap_kv);
        RowTile rt = tile_of(0);
        const int32_t *bt = a.block_table + static_cast<int64_t>(b) * a.max_blocks;
        uint32_t fix_phase = 0;
        bool ok = true;
        // parity of the last phase armed on each full barrier (and the fix barrier),
        // -1 if none: before the CTA exits, each of those phases is waited for, so no
        // TMA write lands in shared memory after a CTA that gave up has left
        int armed[3][ST] = {{-1, -1}, {-1, -1}, {-1, -1}};
        int fix_armed = -1;
        auto wait_empty = [&](int part, int t) -> bool {
            return t < ST || wait(B_EMPTY + part * ST + t % ST, ((t / ST) - 1) & 1);
        };
        for (int t = 0; t < walk.total && ok; ++t) {
            const int st = t % ST;
            if (t > 0 && walk.r(t) != walk.r(t - 1)) rt = tile_of(1);
            const int key0 = walk.j(t) * BN;
            int64_t krow[BN / 32];
            float ksig[BN / 32];
#pragma unroll
            for (int i = 0; i < BN / 32; ++i) {
                const int pos = key0 + lane + 32 * i;
                krow[i] = pos <= rt.key_last ? cache_row(bt, a.max_blocks, a.num_blocks, pos, a.dev_err) : -1;
            }
#pragma unroll
            for (int i = 0; i < BN / 32; ++i) ksig[i] = krow[i] >= 0 ? __ldg(a.kv_scale + krow[i]) : 1.f;
            const int64_t brow = __shfl_sync(0xffffffffu, krow[0], 0);       // the tile's first key
            const int nval = brow < 0 ? 0 : max(0, min(BN, rt.key_last - key0 + 1));
            const uint32_t sdst = sbase_a + st * kStageBytes<false>;
            auto load = [&](int s, int part) {
                tma_load_2d(sdst + s * kSliceBytes<false>, &tmap_kv, 128 * s, static_cast<int>(brow),
                            smem_u32(&sh.bar[B_FULL + part * ST + st]));
            };
            auto meta = [&]() {
                // its ring slot was last read by the softmax of tile t-4, long before
                KeyMeta &mt = sh.meta[t & 3];
#pragma unroll
                for (int i = 0; i < BN / 32; ++i) {
                    const int k = lane + 32 * i;
                    float *sl = reinterpret_cast<float *>(&mt.sl[k >> 1]);
                    sl[k & 1] = ksig[i];
                    sl[2 + (k & 1)] = krow[i] >= 0 ? __log2f(ksig[i]) : -INFINITY;
                    reinterpret_cast<float *>(&mt.isig[k >> 1])[k & 1] = 1.f / ksig[i];
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&sh.bar[B_META + (t & 3)]));
            };
            const int ph = (t / ST) & 1;
            if (nval == BN) {
                if (!(ok = wait_empty(0, t))) break;
                if (lane == 0) {
                    mbar_expect_tx(smem_u32(&sh.bar[B_FULL + 0 * ST + st]), kSliceBytes<false>);
                    load(4, 0);
                }
                armed[0][st] = ph;
                meta();
                if (!(ok = wait_empty(1, t))) break;
                if (lane == 0) {
                    mbar_expect_tx(smem_u32(&sh.bar[B_FULL + 1 * ST + st]), 2 * kSliceBytes<false>);
                    load(0, 1);
                    load(1, 1);
                }
                armed[1][st] = ph;
                if (!(ok = wait_empty(2, t))) break;
                if (lane == 0) {
                    mbar_expect_tx(smem_u32(&sh.bar[B_FULL + 2 * ST + st]), 2 * kSliceBytes<false>);
                    load(2, 2);
                    load(3, 2);
                }
                armed[2][st] = ph;
            } else {
                if (!(ok = wait_empty(0, t) && wait_empty(1, t) && wait_empty(2, t))) break;
                meta();
                if (nval > 0) {
                    if (lane == 0) {
                        mbar_expect_tx(smem_u32(&sh.bar[B_FIX]), kSlices * kSliceBytes<false>);
                        for (int s = 0; s < kSlices; ++s)
                            tma_load_2d(sdst + s * kSliceBytes<false>, &tmap_kv, 128 * s, static_cast<int>(brow),
                                        smem_u32(&sh.bar[B_FIX]));
                    }
                    fix_armed = static_cast<int>(fix_phase);
                    if (!(ok = wait(B_FIX, fix_phase))) break;
                    fix_phase ^= 1;
                    fix_armed = -1;
                }
                // rows nval..BN-1 of every slice (a row is 128 contiguous bytes)
                for (int s = 0; s < kSlices; ++s) {
                    uint8_t *sl = sbase + st * kStageBytes<false> + s * kSliceBytes<false>;
                    for (int o = nval * 128 + 16 * lane; o < kSliceBytes<false>; o += 512)
                        *reinterpret_cast<uint4 *>(sl + o) = make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async();
                __syncwarp();
                if (lane == 0)
                    for (int part = 0; part < 3; ++part) mbar_arrive(smem_u32(&sh.bar[B_FULL + part * ST + st]));
                for (int part = 0; part < 3; ++part) armed[part][st] = ph;
            }
        }
        // drain: every phase armed above has completed once its copies have landed
        if (lane == 0) {
            bool drained = fix_armed < 0 || mbar_wait_cycles(smem_u32(&sh.bar[B_FIX]), fix_armed, kWaitCycles);
            for (int part = 0; part < 3; ++part)
                for (int s2 = 0; s2 < ST; ++s2)
                    if (armed[part][s2] >= 0)
                        drained = mbar_wait_cycles(smem_u32(&sh.bar[B_FULL + part * ST + s2]), armed[part][s2],
                                                   kWaitCycles) && drained;
            if (!drained) set_dev_err(a.dev_err, MLA_DEVERR_TIMEOUT);
        }
        __syncwarp();
    } else if (kSparse && warp >= kSmWarps<kSparse> && warp != kIssuerWarp<kSparse>) {
        // =================== row gathers (sparse): pair p takes tiles p, p+2, ... ===================
        // Key k's 576 bytes go by 16-byte cp.async into the swizzled slices, eight
        // lanes per row (one 128-byte slice row per instruction and row), four rows
        // per warp instruction; a key that is padding (-1) or invalid copies zeros.
        // Copies complete asynchronously on the stage's barrier, so a pair's next
        // tile is on its way before the previous one has landed.
        constexpr int BN = kBN<true>, ST = kStages<true>, kBoxes = BN / kGroupRows;
        constexpr int kSliceB = kSliceBytes<true>, kStageB = kStageBytes<true>;
        const int gk = lane >> 3, gc = lane & 7;
        const int half = gather_half(warp);
        bool ok = true;
        for (int t = gather_pair(warp); t < walk.total && ok; t += 2) {
            const int st = t % ST;
            const RowTile rt = tile_of(walk.r(t));
            const int32_t *bt = a.block_table + static_cast<int64_t>(rt.b) * a.max_blocks;
            const int key0 = walk.j(t) * BN;
            int64_t krow[kBoxes];
            float ksig[kBoxes];
#pragma unroll
            for (int i = 0; i < kBoxes; ++i) {
                const int kk = key0 + lane + 32 * i;
                int pos = kk < a.topk ? __ldg(a.idx + rt.tok * a.topk + kk) : -1;
                if (pos < -1 || pos > rt.key_last) {
                    set_dev_err(a.dev_err, MLA_DEVERR_BAD_INDEX);
                    pos = -1;
                }
                krow[i] = pos >= 0 ? cache_row(bt, a.max_blocks, a.num_blocks, pos, a.dev_err) : -1;
            }
#pragma unroll
            for (int i = 0; i < kBoxes; ++i) ksig[i] = krow[i] >= 0 ? __ldg(a.kv_scale + krow[i]) : 1.f;
            if (t >= ST && !(ok = wait(B_EMPTY + st, ((t / ST) - 1) & 1))) break;
            if (half == 0) {
                KeyMeta &mt = sh.meta[t & 3];
#pragma unroll
                for (int i = 0; i < kBoxes; ++i) {
                    const int k = lane + 32 * i;
                    float *sl = reinterpret_cast<float *>(&mt.sl[k >> 1]);
                    sl[k & 1] = ksig[i];
                    sl[2 + (k & 1)] = krow[i] >= 0 ? __log2f(ksig[i]) : -INFINITY;
                    reinterpret_cast<float *>(&mt.isig[k >> 1])[k & 1] = 1.f / ksig[i];
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&sh.bar[B_META + (t & 3)]));
            }
            const uint32_t sst = sbase_a + st * kStageB;
#pragma unroll 4
            for (int g = half * (BN / 8); g < (half + 1) * (BN / 8); ++g) {
                const int k = 4 * g + gk, kb = (4 * g) >> 5;     // kb: the same for the four rows
                const int64_t r0 = kb == 0 ? krow[0] : (kb == 1 ? krow[1] : krow[2]);
                const int64_t row = __shfl_sync(0xffffffffu, r0, k & 31);
                const uint8_t *src = row >= 0 ? a.kv + row * kDqk + 16 * gc : g_zero_row + 16 * gc;
                const int sstep = row >= 0 ? 128 : 0;
#pragma unroll
                for (int s = 0; s < kSlices; ++s) {
                    if (s == kSlices - 1 && gc >= 4) break;      // the RoPE slice holds 64 bytes
                    cp_async16(sst + s * kSliceB + swz(k, gc), src + sstep * s);
                }
            }
            // no wait: each lane's arrival lands on the stage's barrier when its copies
            // have (the issuer fences them into the async proxy before its MMAs)
            cp_async_arrive(smem_u32(&sh.bar[B_FULL + st]));
        }
        // before the CTA can exit (also after a wait that gave up): this lane's copies have landed
        asm volatile("cp.async.wait_all;\n" ::: "memory");
    } else if (warp == kIssuerWarp<kSparse>) {
        // =================== MMA issuer (lane 0; the other lanes wait at the end) ===================
        // One thread issues: the same instruction stream issued warp-wide with a
        // leader predicate runs ~1.5x slower (measured), as the issue itself
        // becomes the bottleneck of M=64 MMAs.
        if (lane == 0) {
            const uint32_t lead = 1u;
            constexpr int BN = kBN<kSparse>, ST = kStages<kSparse>, SB = kSBufs<kSparse>;
            const uint32_t id_qk = idesc_e4m3(BM, BN, false, false);
            const uint32_t id_pv = idesc_e4m3(BM, 256, false, true);
            const uint64_t dk0 = sdesc(sbase_a, 16, 1024, kSw128);              // K-major key slices
            const uint64_t dv0 = sdesc(sbase_a, kSliceBytes<kSparse>, 1024, kSw128);   // MN-major value chunks
            const uint64_t dp0 = sdesc(sbase_a + kOffP<kSparse>, 128, kPSbo<kSparse>, kSwNone);   // P terms
            bool ok = true;
            // QK(t): the RoPE slice first (dense: released right after), then value slices
            // 0-3; dense waits for each part as it lands
            auto qk = [&](int t) -> bool {
                const int sb = t % SB, st = t % ST, ph = (t / ST) & 1;
                if (t >= SB && !wait(B_S_FREE + sb, ((t / SB) - 1) & 1)) return false;
                const uint32_t d = tmem + kColS + BN * sb;
                auto slice = [&](int s, uint32_t acc0) {
                    const uint64_t db = dk0 + static_cast<uint64_t>((st * kStageBytes<kSparse> + s * kSliceBytes<kSparse>) >> 4);
                    const int nks = s < 4 ? 4 : 2;   // the RoPE slice holds 64 dims
#pragma unroll 4
                    for (int ks = 0; ks < nks; ++ks) {
                        mma_e4m3_ts_w(d, tmem + kColQh + 32 * s + 8 * ks, db + 2 * ks, id_qk, (acc0 || ks > 0) ? 1u : 0u, lead);
                        mma_e4m3_ts_w(d, tmem + kColQl + 32 * s + 8 * ks, db + 2 * ks, id_qk, 1u, lead);
                    }
                };
                if (!wait(B_FULL + 0 * ST + st, ph)) return false;
                fence_after_sync();
                if (kSparse) fence_proxy_async();   // the gathers' cp.async writes, for the MMAs
                slice(4, 0u);
                if (kParts<kSparse> == 3) {
                    mma_commit_w(smem_u32(&sh.bar[B_EMPTY + 0 * ST + st]), lead);   // RoPE slice free
                    if (!wait(B_FULL + 1 * ST + st, ph)) return false;
                    fence_after_sync();
                }
                slice(0, 1u);
                slice(1, 1u);
                if (kParts<kSparse> == 3) {
                    if (!wait(B_FULL + 2 * ST + st, ph)) return false;
                    fence_after_sync();
                }
                slice(2, 1u);
                slice(3, 1u);
                mma_commit_w(smem_u32(&sh.bar[B_S_FULL + sb]), lead);
                return true;
            };
            auto pv = [&](int t) -> bool {
                const int pb = t & 1, st = t % ST, j = walk.j(t), r = walk.r(t);
                if (j == 0 && r > 0 && !wait(B_O_FREE, (r - 1) & 1)) return false;
                if (!wait(B_P_FULL + pb, (t >> 1) & 1)) return false;
                fence_after_sync();
                const uint64_t dph = dp0 + static_cast<uint64_t>(((2 * pb) * kPBytes<kSparse>) >> 4);
                const uint64_t dpl = dp0 + static_cast<uint64_t>(((2 * pb + 1) * kPBytes<kSparse>) >> 4);
#pragma unroll 1
                for (int c = 0; c < 2; ++c) {
                    const uint64_t dv = dv0 + static_cast<uint64_t>((st * kStageBytes<kSparse> + 2 * c * kSliceBytes<kSparse>) >> 4);
                    const uint32_t d = tmem + kHalf1 + 256u * c;
#pragma unroll
                    for (int ks = 0; ks < BN / 32; ++ks) {
                        mma_e4m3_ss_w(d, dph + 16 * ks, dv + 256 * ks, id_pv, (j > 0 || ks > 0) ? 1u : 0u, lead);
                        mma_e4m3_ss_w(d, dpl + 16 * ks, dv + 256 * ks, id_pv, 1u, lead);
                    }
                    if (kParts<kSparse> == 3)   // value slices 2c, 2c+1 free
                        mma_commit_w(smem_u32(&sh.bar[B_EMPTY + (1 + c) * ST + st]), lead);
                }
                if (kParts<kSparse> == 1) mma_commit_w(smem_u32(&sh.bar[B_EMPTY + st]), lead);
                mma_commit_w(smem_u32(&sh.bar[B_PV_DONE + pb]), lead);
                return true;
            };
            if (walk.total > 0) ok = wait(B_Q_FULL, 0) && qk(0);
            for (int t = 0; t < walk.total && ok; ++t) {
                const bool more = t + 1 < walk.total;
                const bool new_rt = more && walk.r(t + 1) != walk.r(t);
                if (more && !new_rt && !(ok = qk(t + 1))) break;
                if (!(ok = pv(t))) break;
                if (new_rt) {
                    if (!(ok = wait(B_Q_FULL, walk.r(t + 1) & 1))) break;
                    if (!(ok = qk(t + 1))) break;
                }
            }
            mma_commit_w(smem_u32(&sh.bar[B_FINAL]), lead);
        } else if (kSparse && lane == 1 && n_rt > 1) {
            // the second token's queries are split long after they are first needed
            // in L2: fetch them now, so that split reads L2 instead of HBM
            const RowTile rt1 = tile_of(1);
            bulk_prefetch_l2(a.q + rt1.grow0 * kDqk, static_cast<uint32_t>(rt1.nvalid) * kDqk * 2);
        }
        __syncwarp();
    } else {
        // =================== softmax / correction ===================
        // warp w: TMEM quadrant w % 4, keys kSmKeys * (w / 4) .. of each tile; with two
        // warps per quadrant they trade tile maxima (and, at the end, row sums) in smem
        constexpr int kKeys = kSmKeys<kSparse>;
        constexpr bool kPair = kSmWarps<kSparse> == 8;
        constexpr int BN = kBN<kSparse>, SB = kSBufs<kSparse>;
        constexpr int kGroups = 18 * kKeys / BN;         // Q column groups per warp
        constexpr int kOCols = 512 * kKeys / BN;         // O columns per warp
        const int q = warp & 3, kh = warp >> 2;
        uint32_t xph = 0;
        auto xch = [&]() -> bool {      // both warps of the quadrant arrive, then wait
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&sh.bar[B_XCH + q]));
            const bool w = wait(B_XCH + q, xph);
            xph ^= 1;
            return w;
        };
        const int tq = lane >> 2, tc = lane & 3;
        const int ra = 16 * q + tq, rb = ra + 8;
        const uint32_t lane_lo = static_cast<uint32_t>(32 * q) << 16;
        const uint32_t lane_hi = lane_lo + kHalf1;
        // P word (own row, keys 8i + 4(tc/2) .. +3) at (row/8)*SBO + (i/2)*128 + (row%8)*16 + 8(i&1) + 4(tc/2)
        const bool even = (tc & 1) == 0;
        const int prow = even ? ra : rb;
        const uint32_t poff = static_cast<uint32_t>((prow >> 3) * kPSbo<kSparse> + (prow & 7) * 16 + 4 * (tc >> 1));
        uint8_t *pbase = sbase + kOffP<kSparse>;
        bool ok = true;
        RowTile rt = tile_of(0);
        float rs_a, rs_b;
        load_q_split(a, rt, tmem + lane_lo, ra, rb, tc, kGroups * kh, kGroups, rs_a, rs_b);
        tmem_st_wait();
        fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sh.bar[B_Q_FULL]));
        int t = 0;
        for (int r = 0; r < n_rt && ok; ++r) {
            float m_a = -INFINITY, m_b = -INFINITY;
            float l_a = 0.f, l_b = 0.f;
            const int lim_a = row_limit<kSparse>(a, rt, ra), lim_b = row_limit<kSparse>(a, rt, rb);
            const int lim_min = min(lim_a, lim_b);
            for (int j = 0; j < rt.n_ktiles && ok; ++j, ++t) {
                const int sb = t % SB, pbf = t & 1;     // S buffer, P buffer
                if (!(ok = wait(B_META + (t & 3), (t >> 2) & 1))) break;
                if (!(ok = wait(B_S_FULL + sb, (t / SB) & 1))) break;
                fence_after_sync();
                uint32_t sv[kKeys / 2];
                if constexpr (kKeys == 64) {
                    tmem_ld_16x256b_x8(tmem + lane_lo + kColS + BN * sb + kKeys * kh, sv);
                } else {
                    tmem_ld_16x256b_x8(tmem + lane_lo + kColS + BN * sb, sv);
                    tmem_ld_16x256b_x4(tmem + lane_lo + kColS + BN * sb + 64, sv + 32);
                }
                tmem_ld_wait();
                fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&sh.bar[B_S_FREE + sb]));
                const KeyMeta &meta = sh.meta[t & 3];
                const int key0 = j * BN + kKeys * kh;     // this warp's first key
                const bool full = kSparse ? lim_min >= 0 : key0 + kKeys - 1 <= lim_min;
                const float mu_a0 = m_a == -INFINITY ? 0.f : m_a - kPOffset;
                const float mu_b0 = m_b == -INFINITY ? 0.f : m_b - kPOffset;
                float mx_a = -INFINITY, mx_b = -INFINITY;
                uint64_t lt2a = 0, lt2b = 0;    // per-thread partial sums of P / sigma, two keys per word
                const uint64_t rs2a = pk2(rs_a, rs_a), rs2b = pk2(rs_b, rs_b);
                const uint64_t mu2a0 = pk2(mu_a0, mu_a0), mu2b0 = pk2(mu_b0, mu_b0);
                uint32_t pa[kKeys / 8], pb[kKeys / 8];   // per 8-key group: this thread's pair of row a / row b, head | tail << 16
                {   // logits, tile maxima and (against the reference max in force) P; for
                    // j == 0 that P is recomputed below once the max is known
#pragma unroll
                    for (int i = 0; i < kKeys / 8; ++i) {
                        const int k0 = 8 * i + 2 * tc;
                        const float4 m = meta.sl[kKeys / 2 * kh + 4 * i + tc];
                        const uint64_t sg = pk2(m.x, m.y), l2 = pk2(m.z, m.w);
                        const float2 ua = upk2(fma2(mul2(pk2(__uint_as_float(sv[4 * i + 0]), __uint_as_float(sv[4 * i + 1])), sg), rs2a, l2));
                        const float2 ub = upk2(fma2(mul2(pk2(__uint_as_float(sv[4 * i + 2]), __uint_as_float(sv[4 * i + 3])), sg), rs2b, l2));
                        float u0 = ua.x, u1 = ua.y, u2 = ub.x, u3 = ub.y;
                        if (!full) {
                            const bool va0 = kSparse ? lim_a >= 0 : key0 + k0 <= lim_a;
                            const bool va1 = kSparse ? lim_a >= 0 : key0 + k0 + 1 <= lim_a;
                            const bool vb0 = kSparse ? lim_b >= 0 : key0 + k0 <= lim_b;
                            const bool vb1 = kSparse ? lim_b >= 0 : key0 + k0 + 1 <= lim_b;
                            u0 = va0 ? u0 : -INFINITY;
                            u1 = va1 ? u1 : -INFINITY;
                            u2 = vb0 ? u2 : -INFINITY;
                            u3 = vb1 ? u3 : -INFINITY;
                        }
                        sv[4 * i + 0] = __float_as_uint(u0);
                        sv[4 * i + 1] = __float_as_uint(u1);
                        sv[4 * i + 2] = __float_as_uint(u2);
                        sv[4 * i + 3] = __float_as_uint(u3);
                        mx_a = max3(mx_a, u0, u1);
                        mx_b = max3(mx_b, u2, u3);
                        {
                            const float2 is = meta.isig[kKeys / 2 * kh + 4 * i + tc];
                            const uint64_t isg = pk2(is.x, is.y);
                            const float2 da = upk2(sub2(pk2(u0, u1), mu2a0)), db = upk2(sub2(pk2(u2, u3), mu2b0));
                            const float p0 = fast_exp2(da.x), p1 = fast_exp2(da.y);
                            const float p2 = fast_exp2(db.x), p3 = fast_exp2(db.y);
                            lt2a = fma2(pk2(p0, p1), isg, lt2a);
                            lt2b = fma2(pk2(p2, p3), isg, lt2b);
                            pa[i] = split_p2(p0, p1);
                            pb[i] = split_p2(p2, p3);
                        }
                    }
                }
                mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 1));
                mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 1));
                mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 2));
                mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 2));
                if constexpr (kPair) {   // the other key half's maxima of the same rows
                    float (*xm)[16] = sh.xmax[t & 1][q];
                    if (tc == 0) {
                        xm[kh][tq] = mx_a;
                        xm[kh][8 + tq] = mx_b;
                    }
                    if (!(ok = xch())) break;
                    mx_a = fmaxf(mx_a, xm[kh ^ 1][tq]);
                    mx_b = fmaxf(mx_b, xm[kh ^ 1][8 + tq]);
                }
                float al_a = 1.f, al_b = 1.f;
                bool resc = false;
                if (j == 0) {
                    m_a = mx_a;
                    m_b = mx_b;
                } else {
                    if (mx_a > m_a + kRescaleThreshold) {
                        al_a = fast_exp2(m_a - mx_a);
                        m_a = mx_a;
                        resc = true;
                    }
                    if (mx_b > m_b + kRescaleThreshold) {
                        al_b = fast_exp2(m_b - mx_b);
                        m_b = mx_b;
                        resc = true;
                    }
                }
                const bool any_resc = __any_sync(0xffffffffu, resc);
                if (j == 0 || any_resc) {
                    const float mu_a = m_a == -INFINITY ? 0.f : m_a - kPOffset;
                    const float mu_b = m_b == -INFINITY ? 0.f : m_b - kPOffset;
                    lt2a = 0;
                    lt2b = 0;
                    const uint64_t mu2a = pk2(mu_a, mu_a), mu2b = pk2(mu_b, mu_b);
#pragma unroll
                    for (int i = 0; i < kKeys / 8; ++i) {
                        const float2 is = meta.isig[kKeys / 2 * kh + 4 * i + tc];
                        const uint64_t isg = pk2(is.x, is.y);
                        const float2 da = upk2(sub2(pk2(__uint_as_float(sv[4 * i + 0]), __uint_as_float(sv[4 * i + 1])), mu2a));
                        const float2 db = upk2(sub2(pk2(__uint_as_float(sv[4 * i + 2]), __uint_as_float(sv[4 * i + 3])), mu2b));
                        const float p0 = fast_exp2(da.x), p1 = fast_exp2(da.y);
                        const float p2 = fast_exp2(db.x), p3 = fast_exp2(db.y);
                        lt2a = fma2(pk2(p0, p1), isg, lt2a);
                        lt2b = fma2(pk2(p2, p3), isg, lt2b);
                        pa[i] = split_p2(p0, p1);
                        pb[i] = split_p2(p2, p3);
                    }
                }
                {
                    const float2 sa = upk2(lt2a), sb = upk2(lt2b);
                    l_a = fmaf(l_a, al_a, sa.x + sa.y);
                    l_b = fmaf(l_b, al_b, sb.x + sb.y);
                }
                if (any_resc) {
                    if (!(ok = wait(B_PV_DONE + ((t - 1) & 1), ((t - 1) >> 1) & 1))) break;
                    fence_after_sync();
#pragma unroll 1
                    for (int c0 = kOCols * kh; c0 < kOCols * kh + kOCols; c0 += 64) {   // this warp's O columns
                        uint32_t o[32];
                        tmem_ld_16x256b_x8(tmem + lane_hi + c0, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            o[4 * i + 0] = __float_as_uint(__uint_as_float(o[4 * i + 0]) * al_a);
                            o[4 * i + 1] = __float_as_uint(__uint_as_float(o[4 * i + 1]) * al_a);
                            o[4 * i + 2] = __float_as_uint(__uint_as_float(o[4 * i + 2]) * al_b);
                            o[4 * i + 3] = __float_as_uint(__uint_as_float(o[4 * i + 3]) * al_b);
                        }
                        tmem_st_16x256b_x8(tmem + lane_hi + c0, o);
                    }
                    tmem_st_wait();
                }
                // ---- P terms into buffer t&1 (last read by PV(t-2)) ----
                if (t >= 2 && !(ok = wait(B_PV_DONE + pbf, ((t >> 1) - 1) & 1))) break;
                uint8_t *ph = pbase + (2 * pbf) * kPBytes<kSparse>, *pl = ph + kPBytes<kSparse>;
#pragma unroll
                for (int i = 0; i < kKeys / 8; ++i) {
                    // the even lane of a pair writes row a's word, the odd lane row b's
                    const uint32_t own = even ? pa[i] : pb[i];
                    const uint32_t oth = __shfl_xor_sync(0xffffffffu, even ? pb[i] : pa[i], 1);
                    const uint32_t lo2 = even ? own : oth, hi2 = even ? oth : own;   // lower keys first
                    const uint32_t hw = (lo2 & 0xFFFFu) | (hi2 << 16);
                    const uint32_t lw = (lo2 >> 16) | (hi2 & 0xFFFF0000u);
                    const int ig = kKeys / 8 * kh + i;           // 8-key group within the tile
                    const uint32_t off = poff + (ig >> 1) * 128 + 8 * (ig & 1);
                    *reinterpret_cast<uint32_t *>(ph + off) = hw;
                    *reinterpret_cast<uint32_t *>(pl + off) = lw;
                }
                fence_proxy_async();
                fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&sh.bar[B_P_FULL + pbf]));
            }
            if (!ok) break;
            const RowTile rt_done = rt;
            float rs_na = 0.f, rs_nb = 0.f;
            if (r + 1 < n_rt) {
                rt = tile_of(r + 1);
                load_q_split(a, rt, tmem + lane_lo, ra, rb, tc, kGroups * kh, kGroups, rs_na, rs_nb);
                tmem_st_wait();
                fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&sh.bar[B_Q_FULL]));
            }
            // ---- epilogue: O / l to bf16, lse ----
            if (!(ok = wait(B_PV_DONE + ((t - 1) & 1), ((t - 1) >> 1) & 1))) break;
            fence_after_sync();
            l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
            l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
            l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
            l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);
            if constexpr (kPair) {   // plus the other key half's sums
                if (tc == 0) {
                    sh.xsum[q][kh][tq] = l_a;
                    sh.xsum[q][kh][8 + tq] = l_b;
                }
                if (!(ok = xch())) break;
                l_a += sh.xsum[q][kh ^ 1][tq];
                l_b += sh.xsum[q][kh ^ 1][8 + tq];
                if (!(ok = xch())) break;      // both read before the next row tile writes again
            }
            const bool va = lim_a >= 0, vb = lim_b >= 0;
            if (tc == 0 && kh == 0 && a.lse) {
                if (va) a.lse[rt_done.grow0 + ra] = l_a > 0.f ? (m_a - kPOffset + __log2f(l_a)) * kLn2 : -INFINITY;
                if (vb) a.lse[rt_done.grow0 + rb] = l_b > 0.f ? (m_b - kPOffset + __log2f(l_b)) * kLn2 : -INFINITY;
            }
            const float ia = l_a > 0.f ? 1.f / l_a : 0.f, ib = l_b > 0.f ? 1.f / l_b : 0.f;
            __nv_bfloat16 *da = a.out + (rt_done.grow0 + ra) * kDv + 2 * tc;
            __nv_bfloat16 *db = a.out + (rt_done.grow0 + rb) * kDv + 2 * tc;
#pragma unroll 1
            for (int c0 = kOCols * kh; c0 < kOCols * kh + kOCols; c0 += 64) {     // this warp's O columns
                uint32_t o[32];
                tmem_ld_16x256b_x8(tmem + lane_hi + c0, o);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if (va)
                        *reinterpret_cast<uint32_t *>(da + c0 + 8 * i) =
                            pack_bf162(__uint_as_float(o[4 * i + 0]) * ia, __uint_as_float(o[4 * i + 1]) * ia);
                    if (vb)
                        *reinterpret_cast<uint32_t *>(db + c0 + 8 * i) =
                            pack_bf162(__uint_as_float(o[4 * i + 2]) * ib, __uint_as_float(o[4 * i + 3]) * ib);
                }
            }
            fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&sh.bar[B_O_FREE]));
            rs_a = rs_na;
            rs_b = rs_nb;
        }
    }

    // ----- teardown: every MMA complete before TMEM is released -----
    __syncthreads();
    if (warp == kIssuerWarp<kSparse>) {
        if (!mbar_wait_cycles(smem_u32(&sh.bar[B_FINAL]), 0, kWaitCycles)) set_dev_err(a.dev_err, MLA_DEVERR_TIMEOUT);
        fence_after_sync();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace f8attn

cudaError_t launch_dense_f8(const AttnArgs &a, const int4 *work, int n_work, const CUtensorMap &tmap_kv,
                            cudaStream_t st) {
    cudaError_t e = cudaFuncSetAttribute(f8attn::attn_f8_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         f8attn::kDynSmem<false>);
    if (e != cudaSuccess) return e;
    if (n_work > 0)
        f8attn::attn_f8_kernel<false><<<n_work, f8attn::kThreads<false>, f8attn::kDynSmem<false>, st>>>(a, work, tmap_kv);
    return cudaGetLastError();
}

cudaError_t launch_sparse_f8(const AttnArgs &a, cudaStream_t st) {
    const int64_t n_tokens = a.tok_end - a.tok_begin;
    cudaError_t e = cudaFuncSetAttribute(f8attn::attn_f8_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         f8attn::kDynSmem<true>);
    if (e != cudaSuccess) return e;
    const CUtensorMap unused{};   // the gather path reads rows with cp.async
    const dim3 grid(static_cast<unsigned>((n_tokens + 1) / 2), (a.H + f8attn::BM - 1) / f8attn::BM);
    if (n_tokens > 0)
        f8attn::attn_f8_kernel<true><<<grid, f8attn::kThreads<true>, f8attn::kDynSmem<true>, st>>>(a, nullptr, unused);
    return cudaGetLastError();
}

}  // namespace mla

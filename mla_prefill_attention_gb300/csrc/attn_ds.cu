// MLA prefill attention over a cache of 656-byte rows (tcgen05 kind::f16).
//
// The row (GLM-5.3-Optimierungen Teil 2, footnote 1: 656 FP8 KV bytes per
// token in the fp8_ds_mla format; read as 512 e4m3 latent codes, one fp32 scale
// per 128 latent dims, then 64 bf16 RoPE values) carries a scale per group of
// dims, so unlike the 580-byte row its scales cannot all be folded into the
// logits and P: they sit inside both products. The loader warps therefore
// dequantise each key row into f16 in shared memory, relative to the row's
// largest group scale sigma (its reference):
//
//   K'[d] = dec(c[d]) * 2^-8 * (sigma_g / sigma)   d < 512, g = d / 128
//   K'[d] = r[d - 512] * 2^-8 / sigma             d >= 512 (the bf16 RoPE values)
//
// so K = 2^8 sigma K', and every other step is the per-token-scale kernel's:
//
//   S   = Q K'^T         tcgen05.mma kind::f16, M=64 N=80, K=576; A = Q in TMEM
//   u   = S*sigma'*rowscale + log2(sigma)        (log2 domain, sigma' = 2^8 sigma)
//   P   = 2^(u - m),  l += P / sigma             (m: running reference max)
//   O  += P V'           M=64 N=128 x 4 chunks of the 512 value dims, A = P in smem
//
// and at the end out = 2^8 O / l, lse = ln2 (m + log2 l). dec(c) * 2^-8 is
// exact in f16 (the code's bits moved into place, see f16x2_of_e4m3x2); the
// group ratio and the RoPE value are rounded once to f16 (11 significant bits).
//
// Shapes and the memory budget. An fp32 O for 64 rows x 512 dims fills one
// TMEM lane half (lanes 16..31 of each 32-lane quadrant, 512 columns); Q
// (64 rows x 576 f16 = 288 columns) and the two score tiles share the other
// half, so shared memory holds only key slices and P. M=64 MMAs run at half
// the M=128 rate (2048 MAC/clk per SM) and take at least ~45 clocks each, so
// N=80 keys is the smallest tile whose QK runs near that rate while leaving
// room for the ring of key slices below.
//
// TMEM (M=64 layout: row r lives in lane 32*(r/16) + r%16 + 16*h; h = lane half)
//   h=0 cols   0..287 : Q (576 dims as f16 pairs)
//   h=0 cols 288..367 : S buffer 0,  cols 368..447 : S buffer 1
//   h=1 cols   0..511 : O
//
// Shared memory
//   18 nope slots x [80 keys][64 dims] f16, 128B-swizzled K-major (10 KB each):
//      a FIFO ring; key tile t's slice s (dims 64s..64s+63) sits in slot
//      (8t + s) mod 18, so slices 2c, 2c+1 always share a slot pair and serve as
//      the N=128 MN-major B operand of PV chunk c
//   2 RoPE slots (the RoPE slice of tiles t, t+1)
//   2 P buffers [64 rows][80 keys] f16, K-major without swizzle (8x16-B core
//      matrices; 128 B apart along the keys, 1280 B apart along the rows)
//
// Warps: 0-3 softmax/correction (warp w owns TMEM quadrant w and reads S with
// the 16-lane shapes, so each thread holds rows 16w + l/4 and 16w + l/4 + 8 x
// 20 keys; the same warps prescale Q into TMEM and run the epilogue), 4-6
// and 8-9 loaders (16 keys each, four lanes per 64-dim slice row; the raw
// bytes and group scales of the next tile are fetched into registers while the
// current one is converted), 7 MMA issue, 10-11 idle.
//
// Dense calls convert first: a conversion kernel writes every key row, once,
// as the f16 K' row above into a workspace in sequence order (each sequence's
// rows padded to whole 80-key tiles) together with each tile's key metadata;
// the attention kernel then loads its slices by TMA (one producer thread, 10 KB
// boxes straight into the ring) instead of converting each row in every CTA that
// reads it (loads in registers were the bound: tensor pipe 45% busy, stalled on
// their latency). Sparse calls gather rows by index and convert them in the
// loader warps as described above.
//
// Tensor-core order: QK(t+1) is issued before PV(t), so the softmax of tile t
// overlaps QK(t+1), and the ring lets the loaders fill tile t+2 while tiles t
// and t+1 are in use. Every wait is bounded; a wait that runs out sets
// MLA_DEVERR_TIMEOUT and the CTA abandons its tile.
#include <cuda_runtime.h>

#include <type_traits>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace mla {
namespace dsattn {

using namespace tc;

constexpr int BM = 64;              // query rows per CTA tile
constexpr int BN = 80;              // keys per tile
constexpr int NT = 384;             // 12 warps
constexpr int kLoaders = 5;         // loader warps: 4, 5, 6, 8, 9
constexpr int kIssuerWarp = 7;      // the only busy warp on its scheduler besides softmax warp 3

// Warp w runs on scheduler w % 4; the issuer's scheduler gets no loader warp.
__device__ __forceinline__ bool is_loader(int warp) { return warp == 4 || warp == 5 || warp == 6 || warp == 8 || warp == 9; }
__device__ __forceinline__ int loader_index(int warp) { return warp < 7 ? warp - 4 : warp - 5; }
constexpr int kSlot = BN * 128;     // one 64-dim slice of a key tile: 10240 B
constexpr int kNopeSlots = 18;      // ring of nope slices (2.25 tiles)
constexpr int kPairs = kNopeSlots / 2;
constexpr int kPBuf = BM * BN * 2;  // 10240 B
constexpr int kOffRope = kNopeSlots * kSlot;
constexpr int kOffP = kOffRope + 2 * kSlot;
constexpr int kDynSmem = 1024 + kOffP + 2 * kPBuf;
constexpr long long kWaitCycles = 200000000LL;   // ~0.1 s: every wait here covers at most one tile of work
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only when the max grows by > 2^8
constexpr float kCodeScale = 256.0f;       // K', V' hold code * 2^-8
constexpr int kRow = 656;                  // bytes per cache row
constexpr int kOffScales = 512, kOffRopeBytes = 528;   // within a row

// TMEM columns
constexpr uint32_t kColQ = 0, kColS = 288, kColO = 0;
constexpr uint32_t kHalf1 = 16u << 16;     // lane offset of the upper half

enum Bar {
    B_FULL_ROPE = 0,                    // [2]  loaders -> issuer: RoPE slot b converted
    B_FULL_PAIR = 2,                    // [9]  loaders -> issuer: nope slot pair converted
    B_FREE_PAIR = 11,                   // [9]  issuer (commit) -> loaders: PV chunk done with the pair
    B_S_FULL = 20,                      // [2]  issuer (commit) -> softmax, loaders: QK of the tile complete
    B_S_FREE = 22,                      // [2]  softmax -> issuer: S buffer read out
    B_P_FULL = 24,                      // [2]  softmax -> issuer: P buffer written (and O rescaled)
    B_PV_DONE = 26,                     // [2]  issuer (commit) -> softmax: PV of the tile complete
    B_META = 28,                        // [4]  loaders -> softmax: key metadata of tile t, t&3
    B_Q_FULL = 32,                      //      softmax -> issuer: Q of the row tile in TMEM
    B_O_FREE = 33,                      //      softmax -> issuer: epilogue finished reading O
    B_FINAL = 34,                       //      issuer -> teardown: every MMA complete
    NBAR = 35
};

// Per-key data of a key tile, by key pair p (keys 2p, 2p+1): what the
// softmax thread owning those keys reads in one 16-byte and one 8-byte load.
struct __align__(16) KeyMeta {
    float4 sl[BN / 2];                   // 2^8 sigma of both keys, log2 sigma of both (-inf = masked)
    float2 isig[BN / 2];                 // 1/sigma of both
};

static_assert(sizeof(KeyMeta) == kDsMetaBytes && BN == kDsTileKeys, "converted key metadata layout");

struct Shared {
    KeyMeta meta[4];                     // per key tile, ring of 4
    uint64_t bar[NBAR];
    uint32_t tmem_base;
    int32_t abort;
};

__device__ __forceinline__ uint32_t swz(int row, int chunk) {  // byte offset in a [rows][128 B] SW128 slice
    return static_cast<uint32_t>((row >> 3) * 1024 + (row & 7) * 128 + ((chunk ^ (row & 7)) << 4));
}

// Bounded wait, entered by every lane of the calling warp. A wait that runs
// out sets MLA_DEVERR_TIMEOUT and the sticky `abort` flag.
struct Wait {
    Shared *sh;
    int32_t *dev_err;
    __device__ bool operator()(int b, uint32_t parity) const {
        if (mbar_wait_cycles(smem_u32(&sh->bar[b]), parity, kWaitCycles)) return true;
        set_dev_err(dev_err, MLA_DEVERR_TIMEOUT);
        atomicExch(&sh->abort, 1);
        return false;
    }
};

// A dense work item is backed when each of its row tiles lies wholly inside both
// the device's and the host's count of rows; one that is not is skipped whole,
// before any setup. Out of line, so it shares no registers with the loops.
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

// Row tile description shared by all roles.
struct RowTile {
    int64_t grow0;      // first global query row (token*H + head)
    int nvalid;         // valid rows in the tile
    int n_ktiles;       // key tiles to visit
    int key_last;       // dense: last key position visible to any row
    int64_t tok;        // sparse: global token index
    int32_t qpos;       // sparse: position of the token (for index validation)
    int h0;             // sparse: first head of the tile
};

template <bool kSparse>
__device__ __forceinline__ RowTile make_tile(const AttnArgs &a, int b, int tile, int64_t sp_tok, int sp_h0) {
    RowTile rt{};
    if (kSparse) {
        rt.tok = sp_tok;
        rt.h0 = sp_h0;
        rt.grow0 = sp_tok * a.H + sp_h0;
        rt.nvalid = min(BM, a.H - sp_h0);
        const int q0 = __ldg(a.cu_seqlens + b);
        rt.qpos = __ldg(a.prefix_lens + b) + static_cast<int32_t>(sp_tok - q0);
        rt.n_ktiles = (a.topk + BN - 1) / BN;
        rt.key_last = rt.qpos;
    } else {
        const int q0 = __ldg(a.cu_seqlens + b), qn = __ldg(a.cu_seqlens + b + 1) - q0;
        const int P = __ldg(a.prefix_lens + b);
        const int rows = qn * a.H, r_lo = tile * BM;
        rt.grow0 = static_cast<int64_t>(q0) * a.H + r_lo;
        rt.nvalid = min(BM, rows - r_lo);
        rt.key_last = P + (r_lo + rt.nvalid - 1) / a.H;
        rt.n_ktiles = rt.key_last / BN + 1;
    }
    return rt;
}

// Last key position visible to query row `row` of the tile (-1: invalid row).
template <bool kSparse>
__device__ __forceinline__ int row_limit(const AttnArgs &a, const RowTile &rt, int b, int row) {
    if (row >= rt.nvalid) return -1;
    if (kSparse) return rt.qpos;
    const int r_lo = static_cast<int>(rt.grow0 - static_cast<int64_t>(__ldg(a.cu_seqlens + b)) * a.H);
    return __ldg(a.prefix_lens + b) + (r_lo + row) / a.H;
}

// Cache row of key k of key tile j (-1: no key) and its scale.
template <bool kSparse>
__device__ __forceinline__ int64_t key_row(const AttnArgs &a, const int32_t *bt, const RowTile &rt, int j, int k) {
    int64_t pos;
    if (kSparse) {
        const int idx = j * BN + k;
        pos = idx < a.topk ? static_cast<int64_t>(__ldg(a.idx + rt.tok * a.topk + idx)) : -1;
        if (pos < -1 || pos > rt.qpos) {
            set_dev_err(a.dev_err, MLA_DEVERR_BAD_INDEX);
            pos = -1;
        }
    } else {
        pos = static_cast<int64_t>(j) * BN + k;
        if (pos > rt.key_last) pos = -1;
    }
    return pos >= 0 ? cache_row(bt, a.max_blocks, a.num_blocks, pos, a.dev_err) : -1;
}

// A key row's four group scales (1 each for no key).
__device__ __forceinline__ float4 row_scales(const AttnArgs &a, int64_t row) {
    return row >= 0 ? __ldg(reinterpret_cast<const float4 *>(a.kv + row * kRow + kOffScales))
                    : make_float4(1.f, 1.f, 1.f, 1.f);
}
// The row's reference scale sigma (the largest of its group scales) and, per
// group, sigma_g / sigma as an f16 pair.
struct GroupRatios {
    float sig;
    uint32_t h[4];
};
__device__ __forceinline__ GroupRatios group_ratios(float4 sc) {
    GroupRatios g;
    g.sig = fmaxf(fmaxf(sc.x, sc.y), fmaxf(sc.z, sc.w));
    const float inv = 1.f / g.sig;
    g.h[0] = pack_half2(sc.x * inv, sc.x * inv);
    g.h[1] = pack_half2(sc.y * inv, sc.y * inv);
    g.h[2] = pack_half2(sc.z * inv, sc.z * inv);
    g.h[3] = pack_half2(sc.w * inv, sc.w * inv);
    return g;
}

__device__ __forceinline__ void write_meta(KeyMeta &m, int k, int64_t row, float sig) {
    float *sl = reinterpret_cast<float *>(&m.sl[k >> 1]);
    sl[k & 1] = sig * kCodeScale;
    sl[2 + (k & 1)] = row >= 0 ? __log2f(sig) : -INFINITY;
    reinterpret_cast<float *>(&m.isig[k >> 1])[k & 1] = 1.f / sig;
}

// Two e4m3 codes (bytes 0 and 2 of t, bytes 1 and 3 zero) -> f16x2 of code * 2^-8,
// exactly: an e4m3 code's exponent and mantissa fields, moved to bits 7..14,
// read as an f16 are the code's value times 2^-8 (normal and subnormal alike,
// since both formats have the same subnormal step relative to their bias);
// adding the sign bit to itself carries it from bit 14 to bit 15.
// The two NaN codes (0x7F, 0xFF) come out as +-480 * 2^-8; quantised caches
// never hold them.
__device__ __forceinline__ uint32_t f16x2_of_e4m3x2(uint32_t t) { return (t + (t & 0x00800080u)) << 7; }

// Converts NC 16-byte chunks (16 dims each, starting at chunk c0) of key k
// into the swizzled f16 slice at dst.
__device__ __forceinline__ uint32_t hmul2_bits(uint32_t x, uint32_t y) {
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(x), "r"(y));
    return r;
}
// 16 latent codes (one 16-byte chunk, dims 16i..16i+15 of a 64-dim slice) of key
// k -> f16 code * 2^-8 * ratio into the swizzled slice at dst.
__device__ __forceinline__ void store_codes(uint8_t *dst, int k, int i, const uint4 &r, uint32_t ratio) {
    uint32_t h[8];
    h[0] = f16x2_of_e4m3x2(__byte_perm(r.x, 0u, 0x4140u));
    h[1] = f16x2_of_e4m3x2(__byte_perm(r.x, 0u, 0x4342u));
    h[2] = f16x2_of_e4m3x2(__byte_perm(r.y, 0u, 0x4140u));
    h[3] = f16x2_of_e4m3x2(__byte_perm(r.y, 0u, 0x4342u));
    h[4] = f16x2_of_e4m3x2(__byte_perm(r.z, 0u, 0x4140u));
    h[5] = f16x2_of_e4m3x2(__byte_perm(r.z, 0u, 0x4342u));
    h[6] = f16x2_of_e4m3x2(__byte_perm(r.w, 0u, 0x4140u));
    h[7] = f16x2_of_e4m3x2(__byte_perm(r.w, 0u, 0x4342u));
#pragma unroll
    for (int u = 0; u < 8; ++u) h[u] = hmul2_bits(h[u], ratio);
    *reinterpret_cast<uint4 *>(dst + swz(k, 2 * i)) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4 *>(dst + swz(k, 2 * i + 1)) = make_uint4(h[4], h[5], h[6], h[7]);
}
// 16 bf16 RoPE values (two 16-byte chunks, dims 16i..16i+15) of key k -> f16 of
// value * 2^-8 / sigma into the swizzled RoPE slice at dst.
__device__ __forceinline__ void store_rope(uint8_t *dst, int k, int i, const uint4 (&r)[2], float scale) {
    uint32_t h[8];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        const __nv_bfloat162 *b = reinterpret_cast<const __nv_bfloat162 *>(&r[u]);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(b[e]);
            h[4 * u + e] = pack_half2(f.x * scale, f.y * scale);
        }
    }
    *reinterpret_cast<uint4 *>(dst + swz(k, 2 * i)) = make_uint4(h[0], h[1], h[2], h[3]);
    *reinterpret_cast<uint4 *>(dst + swz(k, 2 * i + 1)) = make_uint4(h[4], h[5], h[6], h[7]);
}
// The CTA's key tiles in visiting order: global index t -> (row tile, key tile).
struct Walk {
    int n0, total;      // key tiles of row tile 0, of both
    __device__ int r(int t) const { return t < n0 ? 0 : 1; }
    __device__ int j(int t) const { return t < n0 ? t : t - n0; }
};

// ---------------------------------------------------------------------------
// softmax-warp pieces
// ---------------------------------------------------------------------------
// Q rows ra, rb of the tile -> f16 (times a power-of-two row scale) in TMEM
// columns 0..287 of lane half 0 (16x256b layout: column group i holds dims
// 16i + 4tc .. +3 of this thread's rows); returns sm_scale*log2e / scale.
__device__ __forceinline__ void load_q_tmem(const AttnArgs &a, const RowTile &rt, uint32_t tq_addr, int ra, int rb,
                                            int tc, float &rs_a, float &rs_b) {
    const bool oka = ra < rt.nvalid, okb = rb < rt.nvalid;
    const __nv_bfloat16 *qa = a.q + (rt.grow0 + (oka ? ra : 0)) * kDqk + 4 * tc;
    const __nv_bfloat16 *qb = a.q + (rt.grow0 + (okb ? rb : 0)) * kDqk + 4 * tc;
    float mxa = 0.f, mxb = 0.f;
#pragma unroll 4
    for (int i = 0; i < 36; ++i) {
        const uint2 va = oka ? __ldg(reinterpret_cast<const uint2 *>(qa + 16 * i)) : make_uint2(0, 0);
        const uint2 vb = okb ? __ldg(reinterpret_cast<const uint2 *>(qb + 16 * i)) : make_uint2(0, 0);
        const __nv_bfloat162 *ha = reinterpret_cast<const __nv_bfloat162 *>(&va);
        const __nv_bfloat162 *hb = reinterpret_cast<const __nv_bfloat162 *>(&vb);
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const float2 fa = __bfloat1622float2(ha[e]), fb = __bfloat1622float2(hb[e]);
            mxa = fmaxf(mxa, fmaxf(fabsf(fa.x), fabsf(fa.y)));
            mxb = fmaxf(mxb, fmaxf(fabsf(fb.x), fabsf(fb.y)));
        }
    }
    mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, 1));
    mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, 1));
    mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, 2));
    mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, 2));
    int ea = 0, eb = 0;
    if (mxa > 0.f) frexpf(mxa, &ea);
    if (mxb > 0.f) frexpf(mxb, &eb);
    const float sa = mxa > 0.f ? ldexpf(1.f, 1 - ea) : 1.f, sb = mxb > 0.f ? ldexpf(1.f, 1 - eb) : 1.f;
    rs_a = a.sm_scale_log2 / sa;
    rs_b = a.sm_scale_log2 / sb;
#pragma unroll 1
    for (int g0 = 0; g0 < 36; g0 += 8) {
        uint32_t w[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int g = g0 + i;
            uint2 va = make_uint2(0, 0), vb = make_uint2(0, 0);
            if (g < 36) {
                if (oka) va = __ldg(reinterpret_cast<const uint2 *>(qa + 16 * g));
                if (okb) vb = __ldg(reinterpret_cast<const uint2 *>(qb + 16 * g));
            }
            const __nv_bfloat162 *ha = reinterpret_cast<const __nv_bfloat162 *>(&va);
            const __nv_bfloat162 *hb = reinterpret_cast<const __nv_bfloat162 *>(&vb);
            const float2 a0 = __bfloat1622float2(ha[0]), a1 = __bfloat1622float2(ha[1]);
            const float2 b0 = __bfloat1622float2(hb[0]), b1 = __bfloat1622float2(hb[1]);
            w[4 * i + 0] = pack_half2(a0.x * sa, a0.y * sa);
            w[4 * i + 1] = pack_half2(a1.x * sa, a1.y * sa);
            w[4 * i + 2] = pack_half2(b0.x * sb, b0.y * sb);
            w[4 * i + 3] = pack_half2(b1.x * sb, b1.y * sb);
        }
        if (g0 + 8 <= 36) tmem_st_16x256b_x8(tq_addr + 8 * g0, w);
        else tmem_st_16x256b_x4(tq_addr + 8 * g0, w);
    }
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
template <bool kSparse, bool kConv>
__global__ void __launch_bounds__(NT, 1) attn_kernel(const AttnArgs a, const int4 *__restrict__ work,
                                                    const __grid_constant__ CUtensorMap tmap_k) {
    extern __shared__ __align__(1024) uint8_t dsm[];
    __shared__ Shared sh;
    const uint32_t raw = smem_u32(dsm);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    uint8_t *sbase = dsm + pad;
    const uint32_t sbase_a = raw + pad;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // ----- the row tiles of this CTA -----
    int b = 0, tiles[2] = {-1, -1};
    int64_t sp_tok = 0;
    int sp_h0 = 0;
    if (kSparse) {
        sp_tok = a.tok_begin + blockIdx.x;
        sp_h0 = blockIdx.y * BM;
        int lo = 0, hi = a.batch - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (__ldg(a.cu_seqlens + mid) <= sp_tok) lo = mid; else hi = mid - 1;
        }
        b = lo;
        tiles[0] = 0;
    } else {
        const int4 it = work[blockIdx.x];
        b = it.x;
        tiles[0] = it.y;
        tiles[1] = it.z;
    }
    if (!kSparse && !dense_item_backed(a, b, tiles[0], tiles[1])) {
        // (filler items are reported by the kernel that wrote them)
        if (tid == 0 && tiles[0] >= 0) set_dev_err(a.dev_err, MLA_DEVERR_SEQ_MISMATCH);
        return;
    }
    const int n_rt = tiles[1] >= 0 ? 2 : 1;
    const int32_t *bt = a.block_table + static_cast<int64_t>(b) * a.max_blocks;
    Walk walk;
    walk.n0 = make_tile<kSparse>(a, b, tiles[0], sp_tok, sp_h0).n_ktiles;
    walk.total = walk.n0 + (n_rt > 1 ? make_tile<kSparse>(a, b, tiles[1], sp_tok, sp_h0).n_ktiles : 0);

    if (tid == 0) {
        for (int i = 0; i < NBAR; ++i) {
            uint32_t cnt = 1;
            if (i < B_FREE_PAIR || (i >= B_META && i < B_META + 4))
                cnt = kConv ? 1 : kLoaders;                                               // FULL_ROPE, FULL_PAIR, META
            if ((i >= B_S_FREE && i < B_S_FREE + 2) || (i >= B_P_FULL && i < B_P_FULL + 2) || i == B_Q_FULL ||
                i == B_O_FREE)
                cnt = 4;                                                                  // softmax warps
            mbar_init(smem_u32(&sh.bar[i]), cnt);
        }
        sh.abort = 0;
        mbar_fence_init();
    }
    if (warp == kIssuerWarp) {
        tmem_alloc(smem_u32(&sh.tmem_base), 512);
        tmem_relinquish();
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = sh.tmem_base;
    const Wait wait{&sh, a.dev_err};

    if (kConv && warp == 4) {
        // =================== TMA producer (converted rows) ===================
        if (lane == 0) {
            tma_prefetch_desc(&tmap_k);
            const int64_t cb = __ldg(a.conv_base + b);            // converted row of the sequence's key 0
            int armed_rope[2] = {-1, -1}, armed_meta[4] = {-1, -1, -1, -1}, armed_pair[kPairs];
#pragma unroll
            for (int p = 0; p < kPairs; ++p) armed_pair[p] = -1;
            bool ok = true;
            for (int t = 0; t < walk.total && ok; ++t) {
                const int rb = t & 1, j = walk.j(t);
                const int krow = static_cast<int>(cb + static_cast<int64_t>(j) * BN);
                // RoPE slot rb: free once QK of tile t-2 is complete
                if (t >= 2 && !(ok = wait(B_S_FULL + rb, ((t >> 1) - 1) & 1))) break;
                const uint32_t fr = smem_u32(&sh.bar[B_FULL_ROPE + rb]);
                mbar_expect_tx(fr, kSlot);
                tma_load_2d(sbase_a + kOffRope + rb * kSlot, &tmap_k, kDv, krow, fr);
                armed_rope[rb] = (t >> 1) & 1;
                // nope pairs; pair c of tile t uses slot pair (4t + c) mod 9
                for (int c = 0; c < 4; ++c) {
                    const int qn = 4 * t + c, p = qn % kPairs;
                    if (qn >= kPairs && !(ok = wait(B_FREE_PAIR + p, ((qn / kPairs) - 1) & 1))) break;
                    if (c == 0) {   // the tile's metadata (its ring slot was last read by the softmax of tile t-4)
                        const uint32_t fm = smem_u32(&sh.bar[B_META + (t & 3)]);
                        mbar_expect_tx(fm, static_cast<uint32_t>(sizeof(KeyMeta)));
                        bulk_load(smem_u32(&sh.meta[t & 3]),
                                  a.kmeta + (cb / BN + j) * static_cast<int64_t>(sizeof(KeyMeta)),
                                  static_cast<uint32_t>(sizeof(KeyMeta)), fm);
                        armed_meta[t & 3] = (t >> 2) & 1;
                    }
                    const uint32_t fp = smem_u32(&sh.bar[B_FULL_PAIR + p]);
                    mbar_expect_tx(fp, 2 * kSlot);
                    tma_load_2d(sbase_a + (2 * p) * kSlot, &tmap_k, 128 * c, krow, fp);
                    tma_load_2d(sbase_a + (2 * p + 1) * kSlot, &tmap_k, 128 * c + 64, krow, fp);
                    armed_pair[p] = (qn / kPairs) & 1;
                }
            }
            // drain: the last copy into every slot has landed
            bool drained = true;
            for (int i = 0; i < 2; ++i)
                if (armed_rope[i] >= 0)
                    drained = mbar_wait_cycles(smem_u32(&sh.bar[B_FULL_ROPE + i]), armed_rope[i], kWaitCycles) && drained;
            for (int i = 0; i < 4; ++i)
                if (armed_meta[i] >= 0)
                    drained = mbar_wait_cycles(smem_u32(&sh.bar[B_META + i]), armed_meta[i], kWaitCycles) && drained;
            for (int i = 0; i < kPairs; ++i)
                if (armed_pair[i] >= 0)
                    drained = mbar_wait_cycles(smem_u32(&sh.bar[B_FULL_PAIR + i]), armed_pair[i], kWaitCycles) && drained;
            if (!drained) set_dev_err(a.dev_err, MLA_DEVERR_TIMEOUT);
        }
        __syncwarp();
    } else if (!kConv && is_loader(warp)) {
        // =================== loaders ===================
        // Loader warp w covers keys 16w..16w+15 of a tile as two groups of 8;
        // lane l holds 16-byte chunk l%4 of one 64-dim slice row of key
        // 16w + 8g + l/4, so every warp-wide load reads 8 rows x 64 contiguous
        // bytes and every swizzled 16-byte store of 8 rows is conflict-free.
        // Tile t's raw bytes are in registers when iteration t starts; each
        // part is converted once its slot is free and the same part of tile t+1
        // is fetched right after.
        const int kq = 16 * loader_index(warp) + (lane >> 2), jc = lane & 3;   // key of group 0, chunk
        RowTile rt = make_tile<kSparse>(a, b, tiles[0], sp_tok, sp_h0);
        uint4 r_rope[2][2], r_s[4][4];         // [group][half], [pair][2 * half + group]
        float4 sc_cur[2];                      // the two keys' group scales
        int64_t row_cur[2];
        // pair c (slices 2c, 2c+1: dims 128c..128c+127) is group c of the row
        auto fetch = [&](const int64_t (&row)[2], int slice, uint4 *dst, int stride) {
#pragma unroll
            for (int g = 0; g < 2; ++g)
                dst[stride * g] = row[g] >= 0
                                      ? __ldg(reinterpret_cast<const uint4 *>(a.kv + row[g] * kRow + slice * 64) + jc)
                                      : make_uint4(0, 0, 0, 0);
        };
        auto fetch_rope = [&](const int64_t (&row)[2]) {   // bf16 dims 16jc..16jc+15: 32 bytes
#pragma unroll
            for (int g = 0; g < 2; ++g)
#pragma unroll
                for (int u = 0; u < 2; ++u)
                    r_rope[g][u] = row[g] >= 0 ? __ldg(reinterpret_cast<const uint4 *>(a.kv + row[g] * kRow +
                                                                                       kOffRopeBytes + 32 * jc) + u)
                                               : make_uint4(0, 0, 0, 0);
        };
#pragma unroll
        for (int g = 0; g < 2; ++g) {
            row_cur[g] = key_row<kSparse>(a, bt, rt, 0, kq + 8 * g);
            sc_cur[g] = row_scales(a, row_cur[g]);
        }
        fetch_rope(row_cur);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            fetch(row_cur, 2 * c, &r_s[c][0], 1);
            fetch(row_cur, 2 * c + 1, &r_s[c][2], 1);
        }
        bool ok = true;
        for (int t = 0; t < walk.total && ok; ++t) {
            const int rb = t & 1;
            const GroupRatios gr[2] = {group_ratios(sc_cur[0]), group_ratios(sc_cur[1])};
            // ---- RoPE slot rb: free once QK of tile t-2 is complete ----
            if (t >= 2 && !(ok = wait(B_S_FULL + rb, ((t >> 1) - 1) & 1))) break;
#pragma unroll
            for (int g = 0; g < 2; ++g)
                store_rope(sbase + kOffRope + rb * kSlot, kq + 8 * g, jc, r_rope[g], (1.f / kCodeScale) / gr[g].sig);
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&sh.bar[B_FULL_ROPE + rb]));
            // ---- the next tile's cache rows, group scales and RoPE bytes ----
            const bool more = t + 1 < walk.total;
            int64_t row_n[2] = {-1, -1};
            float4 sc_n[2] = {make_float4(1.f, 1.f, 1.f, 1.f), make_float4(1.f, 1.f, 1.f, 1.f)};
            if (more) {
                const int tn = t + 1;
                if (walk.r(tn) != walk.r(t)) rt = make_tile<kSparse>(a, b, tiles[walk.r(tn)], sp_tok, sp_h0);
#pragma unroll
                for (int g = 0; g < 2; ++g) {
                    row_n[g] = key_row<kSparse>(a, bt, rt, walk.j(tn), kq + 8 * g);
                    sc_n[g] = row_scales(a, row_n[g]);
                }
                fetch_rope(row_n);
            }
            // ---- nope pairs; pair c of tile t uses slot pair (4t + c) mod 9 ----
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int qn = 4 * t + c, p = qn % kPairs;
                if (qn >= kPairs && !(ok = wait(B_FREE_PAIR + p, ((qn / kPairs) - 1) & 1))) break;
                if (c == 0) {   // the tile's metadata (its ring slot was last read by the softmax of tile t-4)
                    if (jc == 0) {
                        write_meta(sh.meta[t & 3], kq, row_cur[0], gr[0].sig);
                        write_meta(sh.meta[t & 3], kq + 8, row_cur[1], gr[1].sig);
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&sh.bar[B_META + (t & 3)]));
                }
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int g = 0; g < 2; ++g)
                        store_codes(sbase + (2 * p + h) * kSlot, kq + 8 * g, jc, r_s[c][2 * h + g], gr[g].h[c]);
                fence_proxy_async();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&sh.bar[B_FULL_PAIR + p]));
                if (more) {
                    fetch(row_n, 2 * c, &r_s[c][0], 1);
                    fetch(row_n, 2 * c + 1, &r_s[c][2], 1);
                }
            }
            row_cur[0] = row_n[0];
            row_cur[1] = row_n[1];
            sc_cur[0] = sc_n[0];
            sc_cur[1] = sc_n[1];
        }
    } else if (warp >= 4) {
        // =================== MMA issuer (warp 7, lane 0); warps 10, 11 idle ===================
        // One thread runs the issue loop: issued warp-wide with a leader
        // predicate, the short M=64 MMAs become issue-bound (measured).
        if (warp == kIssuerWarp && lane == 0) {
            const uint32_t lead = 1u;
            const uint32_t id_qk = idesc_f16(BM, BN, false, false, false, false);
            const uint32_t id_pv = idesc_f16(BM, 128, false, false, false, true);
            // descriptors of the bases; an operand at byte offset x is the base plus x/16
            const uint64_t dk0 = sdesc(sbase_a, 16, 1024, kSw128);           // K-major key slices
            const uint64_t dv0 = sdesc(sbase_a, kSlot, 1024, kSw128);        // MN-major slot pairs (V)
            const uint64_t dp0 = sdesc(sbase_a + kOffP, 128, 1280, kSwNone); // P buffers
            bool ok = true;
            // QK(t): S buffer t&1 = Q K^T over slice 8 (RoPE), then pairs 0..3
            auto qk = [&](int t) -> bool {
                const int sb = t & 1;
                if (!wait(B_FULL_ROPE + sb, (t >> 1) & 1)) return false;
                if (t >= 2 && !wait(B_S_FREE + sb, ((t >> 1) - 1) & 1)) return false;
                fence_after_sync();
                const uint32_t d = tmem + kColS + BN * sb;
                {
                    const uint64_t db = dk0 + static_cast<uint64_t>((kOffRope + sb * kSlot) >> 4);
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_f16_ts_w(d, tmem + kColQ + 32 * 8 + 8 * ks, db + 2 * ks, id_qk, ks > 0 ? 1u : 0u, lead);
                }
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    const int qn = 4 * t + c, p = qn % kPairs;
                    if (!wait(B_FULL_PAIR + p, (qn / kPairs) & 1)) return false;
                    fence_after_sync();
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const int s = 2 * c + h;
                        const uint64_t db = dk0 + static_cast<uint64_t>(((2 * p + h) * kSlot) >> 4);
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks)
                            mma_f16_ts_w(d, tmem + kColQ + 32 * s + 8 * ks, db + 2 * ks, id_qk, 1u, lead);
                    }
                }
                mma_commit_w(smem_u32(&sh.bar[B_S_FULL + sb]), lead);
                return true;
            };
            // PV(t): O += P(t) V(t), four 128-dim chunks, each releasing its slot pair
            auto pv = [&](int t) -> bool {
                const int pb = t & 1, j = walk.j(t), r = walk.r(t);
                if (j == 0 && r > 0 && !wait(B_O_FREE, (r - 1) & 1)) return false;
                if (!wait(B_P_FULL + pb, (t >> 1) & 1)) return false;
                fence_after_sync();
                const uint64_t da = dp0 + static_cast<uint64_t>((pb * kPBuf) >> 4);
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    const int p = (4 * t + c) % kPairs;
                    const uint64_t dv = dv0 + static_cast<uint64_t>((2 * p * kSlot) >> 4);
                    const uint32_t d = tmem + kHalf1 + kColO + 128u * c;
#pragma unroll
                    for (int ks = 0; ks < BN / 16; ++ks)
                        mma_f16_ss_w(d, da + 16 * ks, dv + 128 * ks, id_pv, (j > 0 || ks > 0) ? 1u : 0u, lead);
                    mma_commit_w(smem_u32(&sh.bar[B_FREE_PAIR + p]), lead);
                }
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
        }
        __syncwarp();
    } else if (warp < 4) {
        // =================== softmax / correction (warps 0-3) ===================
        const int q = warp;                        // TMEM lane quadrant
        const int tq = lane >> 2, tc = lane & 3;
        const int ra = 16 * q + tq, rb = ra + 8;
        const uint32_t lane_lo = static_cast<uint32_t>(32 * q) << 16;
        const uint32_t lane_hi = lane_lo + kHalf1;
        uint8_t *pbuf = sbase + kOffP;
        // P word (row, keys 8i + 2tc, +1) lives at (row/8)*1280 + i*128 + (row%8)*16 + 4tc
        const uint32_t poff_a = static_cast<uint32_t>((ra >> 3) * 1280 + (ra & 7) * 16 + 4 * tc);
        const uint32_t poff_b = static_cast<uint32_t>((rb >> 3) * 1280 + (rb & 7) * 16 + 4 * tc);
        bool ok = true;
        RowTile rt = make_tile<kSparse>(a, b, tiles[0], sp_tok, sp_h0);
        float rs_a, rs_b;
        load_q_tmem(a, rt, tmem + lane_lo + kColQ, ra, rb, tc, rs_a, rs_b);
        tmem_st_wait();
        fence_before_sync();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sh.bar[B_Q_FULL]));
        int t = 0;
        for (int r = 0; r < n_rt && ok; ++r) {
            float m_a = -INFINITY, m_b = -INFINITY;  // reference maxima (log2 domain)
            float l_a = 0.f, l_b = 0.f;              // this thread's partial row sums (20 keys per tile)
            const int lim_a = row_limit<kSparse>(a, rt, b, ra), lim_b = row_limit<kSparse>(a, rt, b, rb);
            const int lim_min = min(lim_a, lim_b);
            for (int j = 0; j < rt.n_ktiles && ok; ++j, ++t) {
                const int sb = t & 1;
                if (!(ok = wait(B_META + (t & 3), (t >> 2) & 1))) break;
                if (!(ok = wait(B_S_FULL + sb, (t >> 1) & 1))) break;
                fence_after_sync();
                uint32_t sv[40];
                tmem_ld_16x256b_x8(tmem + lane_lo + kColS + BN * sb, sv);
                tmem_ld_16x256b_x2(tmem + lane_lo + kColS + BN * sb + 64, sv + 32);
                tmem_ld_wait();
                fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&sh.bar[B_S_FREE + sb]));
                // ---- logits u in the log2 domain and tile maxima; for j > 0 also P against
                // the current reference maxima (kept unless the tile raises one by > 2^8) ----
                const KeyMeta &meta = sh.meta[t & 3];
                const int key0 = kSparse ? 0 : j * BN;
                const bool full = kSparse ? (lim_min >= 0) : (key0 + BN - 1 <= lim_min);
                const float mu_a0 = m_a == -INFINITY ? 0.f : m_a, mu_b0 = m_b == -INFINITY ? 0.f : m_b;
                float mx_a = -INFINITY, mx_b = -INFINITY, lt_a = 0.f, lt_b = 0.f;
                uint32_t pk[20];
                auto logits = [&](auto with_p) {
#pragma unroll
                    for (int i = 0; i < BN / 8; ++i) {
                        const int k0 = 8 * i + 2 * tc;
                        const float4 m = meta.sl[4 * i + tc];     // keys k0, k0+1
                        float u0 = fmaf(__uint_as_float(sv[4 * i + 0]) * m.x, rs_a, m.z);
                        float u1 = fmaf(__uint_as_float(sv[4 * i + 1]) * m.y, rs_a, m.w);
                        float u2 = fmaf(__uint_as_float(sv[4 * i + 2]) * m.x, rs_b, m.z);
                        float u3 = fmaf(__uint_as_float(sv[4 * i + 3]) * m.y, rs_b, m.w);
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
                        mx_a = fmaxf(mx_a, fmaxf(u0, u1));
                        mx_b = fmaxf(mx_b, fmaxf(u2, u3));
                        if (decltype(with_p)::value) {
                            const float2 is = meta.isig[4 * i + tc];
                            const float p0 = fast_exp2(u0 - mu_a0), p1 = fast_exp2(u1 - mu_a0);
                            const float p2 = fast_exp2(u2 - mu_b0), p3 = fast_exp2(u3 - mu_b0);
                            lt_a = fmaf(p0, is.x, fmaf(p1, is.y, lt_a));
                            lt_b = fmaf(p2, is.x, fmaf(p3, is.y, lt_b));
                            pk[2 * i] = pack_half2(p0, p1);
                            pk[2 * i + 1] = pack_half2(p2, p3);
                        }
                    }
                };
                if (j > 0) logits(std::true_type{});
                else logits(std::false_type{});
                mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 1));
                mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 1));
                mx_a = fmaxf(mx_a, __shfl_xor_sync(0xffffffffu, mx_a, 2));
                mx_b = fmaxf(mx_b, __shfl_xor_sync(0xffffffffu, mx_b, 2));
                // ---- reference maxima: move (and O is rescaled) only when they grow by > 2^8 ----
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
                    // P (again) against the reference maxima now in force
                    const float mu_a = m_a == -INFINITY ? 0.f : m_a, mu_b = m_b == -INFINITY ? 0.f : m_b;
                    lt_a = 0.f;
                    lt_b = 0.f;
#pragma unroll
                    for (int i = 0; i < BN / 8; ++i) {
                        const float2 is = meta.isig[4 * i + tc];
                        const float p0 = fast_exp2(__uint_as_float(sv[4 * i + 0]) - mu_a);
                        const float p1 = fast_exp2(__uint_as_float(sv[4 * i + 1]) - mu_a);
                        const float p2 = fast_exp2(__uint_as_float(sv[4 * i + 2]) - mu_b);
                        const float p3 = fast_exp2(__uint_as_float(sv[4 * i + 3]) - mu_b);
                        lt_a = fmaf(p0, is.x, fmaf(p1, is.y, lt_a));
                        lt_b = fmaf(p2, is.x, fmaf(p3, is.y, lt_b));
                        pk[2 * i] = pack_half2(p0, p1);
                        pk[2 * i + 1] = pack_half2(p2, p3);
                    }
                }
                l_a = fmaf(l_a, al_a, lt_a);
                l_b = fmaf(l_b, al_b, lt_b);
                // ---- O rescale (rare): PV(t-1) must be complete, PV(t) is not yet issued ----
                if (any_resc) {
                    if (!(ok = wait(B_PV_DONE + ((t - 1) & 1), ((t - 1) >> 1) & 1))) break;
                    fence_after_sync();
#pragma unroll 1
                    for (int c0 = 0; c0 < 512; c0 += 64) {
                        uint32_t o[32];
                        tmem_ld_16x256b_x8(tmem + lane_hi + kColO + c0, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            o[4 * i + 0] = __float_as_uint(__uint_as_float(o[4 * i + 0]) * al_a);
                            o[4 * i + 1] = __float_as_uint(__uint_as_float(o[4 * i + 1]) * al_a);
                            o[4 * i + 2] = __float_as_uint(__uint_as_float(o[4 * i + 2]) * al_b);
                            o[4 * i + 3] = __float_as_uint(__uint_as_float(o[4 * i + 3]) * al_b);
                        }
                        tmem_st_16x256b_x8(tmem + lane_hi + kColO + c0, o);
                    }
                    tmem_st_wait();
                }
                // ---- P into smem buffer t&1 (its last reader, PV(t-2), must be complete) ----
                if (t >= 2 && !(ok = wait(B_PV_DONE + sb, ((t >> 1) - 1) & 1))) break;
                uint8_t *pw = pbuf + sb * kPBuf;
#pragma unroll
                for (int i = 0; i < BN / 8; ++i) {
                    *reinterpret_cast<uint32_t *>(pw + poff_a + 128 * i) = pk[2 * i];
                    *reinterpret_cast<uint32_t *>(pw + poff_b + 128 * i) = pk[2 * i + 1];
                }
                fence_proxy_async();
                fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&sh.bar[B_P_FULL + sb]));
            }
            if (!ok) break;
            // ---- the next row tile's Q (QK of this row tile is complete: its last S was read) ----
            const RowTile rt_done = rt;
            float rs_na = 0.f, rs_nb = 0.f;
            if (r + 1 < n_rt) {
                rt = make_tile<kSparse>(a, b, tiles[r + 1], sp_tok, sp_h0);
                load_q_tmem(a, rt, tmem + lane_lo + kColQ, ra, rb, tc, rs_na, rs_nb);
                tmem_st_wait();
                fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&sh.bar[B_Q_FULL]));
            }
            // ---- epilogue: O 2^8 / l to bf16, lse ----
            if (!(ok = wait(B_PV_DONE + ((t - 1) & 1), ((t - 1) >> 1) & 1))) break;
            fence_after_sync();
            l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
            l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
            l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
            l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);
            const bool va = lim_a >= 0, vb = lim_b >= 0;
            if (tc == 0 && a.lse) {
                if (va) a.lse[rt_done.grow0 + ra] = l_a > 0.f ? (m_a + __log2f(l_a)) * kLn2 : -INFINITY;
                if (vb) a.lse[rt_done.grow0 + rb] = l_b > 0.f ? (m_b + __log2f(l_b)) * kLn2 : -INFINITY;
            }
            const float ia = l_a > 0.f ? kCodeScale / l_a : 0.f, ib = l_b > 0.f ? kCodeScale / l_b : 0.f;
            __nv_bfloat16 *da = a.out + (rt_done.grow0 + ra) * kDv + 2 * tc;
            __nv_bfloat16 *db = a.out + (rt_done.grow0 + rb) * kDv + 2 * tc;
#pragma unroll 1
            for (int c0 = 0; c0 < 512; c0 += 64) {
                uint32_t o[32];
                tmem_ld_16x256b_x8(tmem + lane_hi + kColO + c0, o);
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
    if (warp == kIssuerWarp) {
        if (!mbar_wait_cycles(smem_u32(&sh.bar[B_FINAL]), 0, kWaitCycles)) set_dev_err(a.dev_err, MLA_DEVERR_TIMEOUT);
        fence_after_sync();
        tmem_dealloc(tmem, 512);
    }
}

// ---------------------------------------------------------------------------
// conversion of the dense keys: one thread per (converted row, 16-dim chunk);
// chunks 0..31 hold the latent codes, 32..35 the RoPE dims; chunk 0 also writes
// the row's entry of its tile's key metadata. The arithmetic is the loaders'
// (store_codes, store_rope, write_meta), so the f16 rows are the same bits.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) convert_kernel(const AttnArgs a, int64_t n_rows) {
    const int64_t gid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t row = gid / 36;
    const int ch = static_cast<int>(gid % 36);
    if (row >= n_rows) return;
    int lo = 0, hi = a.batch - 1;          // the sequence: the last b with conv_base[b] <= row
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(a.conv_base + mid) <= row) lo = mid; else hi = mid - 1;
    }
    const int b = lo;
    const int64_t pos = row - __ldg(a.conv_base + b);
    int64_t crow = -1;
    if (pos < __ldg(a.conv_ctx + b))
        crow = cache_row(a.block_table + static_cast<int64_t>(b) * a.max_blocks, a.max_blocks, a.num_blocks, pos,
                         a.dev_err);
    const GroupRatios gr = group_ratios(row_scales(a, crow));
    uint32_t h[8];
    if (ch < 32) {
        const uint4 r = crow >= 0 ? __ldg(reinterpret_cast<const uint4 *>(a.kv + crow * kRow) + ch)
                                  : make_uint4(0, 0, 0, 0);
        h[0] = f16x2_of_e4m3x2(__byte_perm(r.x, 0u, 0x4140u));
        h[1] = f16x2_of_e4m3x2(__byte_perm(r.x, 0u, 0x4342u));
        h[2] = f16x2_of_e4m3x2(__byte_perm(r.y, 0u, 0x4140u));
        h[3] = f16x2_of_e4m3x2(__byte_perm(r.y, 0u, 0x4342u));
        h[4] = f16x2_of_e4m3x2(__byte_perm(r.z, 0u, 0x4140u));
        h[5] = f16x2_of_e4m3x2(__byte_perm(r.z, 0u, 0x4342u));
        h[6] = f16x2_of_e4m3x2(__byte_perm(r.w, 0u, 0x4140u));
        h[7] = f16x2_of_e4m3x2(__byte_perm(r.w, 0u, 0x4342u));
        const uint32_t ratio = gr.h[ch >> 3];
#pragma unroll
        for (int u = 0; u < 8; ++u) h[u] = hmul2_bits(h[u], ratio);
    } else {
        const int i = ch - 32;
        uint4 r[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
        if (crow >= 0) {
            r[0] = __ldg(reinterpret_cast<const uint4 *>(a.kv + crow * kRow + kOffRopeBytes + 32 * i));
            r[1] = __ldg(reinterpret_cast<const uint4 *>(a.kv + crow * kRow + kOffRopeBytes + 32 * i) + 1);
        }
        const float scale = (1.f / kCodeScale) / gr.sig;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            const __nv_bfloat162 *bb = reinterpret_cast<const __nv_bfloat162 *>(&r[u]);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float2 f = __bfloat1622float2(bb[e]);
                h[4 * u + e] = pack_half2(f.x * scale, f.y * scale);
            }
        }
    }
    uint4 *dst = reinterpret_cast<uint4 *>(a.kconv + row * kDqk) + 2 * ch;
    dst[0] = make_uint4(h[0], h[1], h[2], h[3]);
    dst[1] = make_uint4(h[4], h[5], h[6], h[7]);
    if (ch == 0) write_meta(reinterpret_cast<KeyMeta *>(a.kmeta)[row / BN], static_cast<int>(row % BN), crow, gr.sig);
}

}  // namespace dsattn

cudaError_t launch_dense_ds(const AttnArgs &a, const int4 *work, int n_work, int64_t n_conv_rows,
                            const CUtensorMap &tmap_conv, cudaStream_t st) {
    cudaError_t e = cudaFuncSetAttribute(dsattn::attn_kernel<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         dsattn::kDynSmem);
    if (e != cudaSuccess) return e;
    if (n_work <= 0) return cudaSuccess;
    const int64_t threads = n_conv_rows * 36;
    dsattn::convert_kernel<<<static_cast<unsigned>((threads + 255) / 256), 256, 0, st>>>(a, n_conv_rows);
    dsattn::attn_kernel<false, true><<<n_work, dsattn::NT, dsattn::kDynSmem, st>>>(a, work, tmap_conv);
    return cudaGetLastError();
}

cudaError_t launch_sparse_ds(const AttnArgs &a, cudaStream_t st) {
    const int64_t n_tokens = a.tok_end - a.tok_begin;
    cudaError_t e =
        cudaFuncSetAttribute(dsattn::attn_kernel<true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, dsattn::kDynSmem);
    if (e != cudaSuccess) return e;
    const dim3 grid(static_cast<unsigned>(n_tokens), (a.H + dsattn::BM - 1) / dsattn::BM);
    CUtensorMap unused{};
    if (n_tokens > 0) dsattn::attn_kernel<true, false><<<grid, dsattn::NT, dsattn::kDynSmem, st>>>(a, nullptr, unused);
    return cudaGetLastError();
}

}  // namespace mla

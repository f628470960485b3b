// MLA prefill attention on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// One CTA owns a tile of 64 query rows (row = (token, head); for 64 heads one
// token) and streams the latent rows of the paged e4m3 cache 128 keys at a
// time. Per key tile:
//
//   S   = Q K^T          tcgen05.mma kind::f16, M=64 N=128, K=576, D in TMEM
//   u   = S*sigma*rowscale + log2(sigma)        (log2 domain, sigma folded in)
//   P   = 2^(u - m),  l += P / sigma             (m: running reference max)
//   O  += P V            tcgen05.mma M=64 N=256 (two Dv halves), A=P from TMEM
//
// and at the end out = O / l, lse = ln2 (m + log2 l).
//
// Why 64 rows: with the 512-wide value head an fp32 O for 128 rows fills all
// 512 TMEM columns, and a 128 x 576 f16 Q tile alone is 144 KB of shared
// memory. With 64 rows, O takes two lane-halves x 256 columns and Q 72 KB.
// M=64 MMAs run at half the M=128 rate on this part (2048 vs 4096 MAC/clk per
// SM, measured), so this kernel is capped at half the dense tensor peak.
//
// TMEM (M=64 layout: row r lives in lane 32*(r/16) + r%16 + 16*h; h = lane half)
//   cols   0..255 h=0 : O for value dims   0..255
//   cols   0..255 h=1 : O for value dims 256..511
//   cols 256..383 h=0 : S (128 keys)
//   cols 384..447 h=0 / h=1 : P (128 keys as f16 pairs), one copy per half
//
// Shared memory (1024-B aligned, 128B-swizzled K-major operand layouts)
//   Q  : 9 slices x [64 rows][64 dims] f16   (72 KB)
//   K  : 9 slices x [128 keys][64 dims] f16  (144 KB); slices 0..7 double as V
//        (MN-major B operand of PV), slice 8 holds the RoPE dims
//
// Warps: 0-3 softmax/correction (warp w owns TMEM lane quadrant w), 4-7
// loaders (Q prescale, e4m3 -> f16 conversion of K straight from global
// memory, per-key scales), 8 MMA issue. The K tile is single-buffered but
// recycled slice-group by slice-group: slice 8 is refilled as soon as QK has
// used it, slices 0-3 after the first PV half, slices 4-7 after the second.
// Every wait is bounded; a wait that runs out sets MLA_DEVERR_TIMEOUT and the
// CTA abandons its tile.
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace mla {
namespace tcattn {

using namespace tc;

constexpr int BM = 64;            // query rows per CTA tile
constexpr int BN = 128;           // keys per tile
constexpr int NSLICE = 9;         // 576 / 64
constexpr int NT = 288;           // 9 warps
constexpr int kQSlice = BM * 128;         // 8192 B
constexpr int kKSlice = BN * 128;         // 16384 B
constexpr int kSmemQ = NSLICE * kQSlice;  // 73728
constexpr int kSmemK = NSLICE * kKSlice;  // 147456
constexpr int kDynSmem = 1024 + kSmemQ + kSmemK;
constexpr long long kWaitCycles = 200000000LL;   // ~0.1 s: every wait here covers at most one tile of work
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only when the max grows by > 2^8

// TMEM columns
constexpr uint32_t kColO = 0, kColS = 256, kColP = 384;
constexpr uint32_t kHalf1 = 16u << 16;     // lane offset of the upper half

enum Bar {
    B_FULL_ROPE, B_FULL_A, B_FULL_B,    // loaders -> issuer: K slices converted (8 | 0-3 | 4-7)
    B_FREE_ROPE, B_FREE_A, B_FREE_B,    // issuer (MMA commit) -> loaders: slices consumed
    B_S_FULL,                           // issuer -> softmax: S ready
    B_S_FREE,                           // softmax -> issuer: S read out
    B_P_FULL,                           // softmax -> issuer: P written (and O rescaled)
    B_PV_DONE,                          // issuer -> softmax: PV of the tile complete
    B_Q_FULL,                           // loaders -> issuer: Q tile in smem
    B_O_FREE,                           // softmax -> issuer: epilogue finished reading O
    B_FINAL,                            // issuer -> all: every MMA of the CTA complete
    B_Q_FREE,                           // issuer -> loaders: last QK of a row tile complete (Q reusable)
    B_META0, B_META1,                   // loaders -> softmax: key metadata (and row data) of tile n, n&1
    NBAR
};

struct KeyMeta {
    float sig, lsig, isig, pad;          // sigma, log2 sigma (-inf = masked), 1/sigma
};

struct Shared {
    KeyMeta meta[4][BN];                 // per key tile, ring of 4
    float rowscale[2][BM];               // sm_scale*log2e / query prescale, per row tile parity
    int32_t rowlimit[2][BM];             // last visible position (dense); -1 = invalid row
    uint64_t bar[NBAR];
    uint32_t tmem_base;
    int32_t abort;
};

__device__ __forceinline__ uint32_t swz(int row, int chunk) {  // byte offset in a [rows][128 B] SW128 slice
    return static_cast<uint32_t>((row >> 3) * 1024 + (row & 7) * 128 + ((chunk ^ (row & 7)) << 4));
}

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

// ---------------------------------------------------------------------------
// loaders (warps 4-7): Q tile, per-key metadata, e4m3 -> f16 K slices
// ---------------------------------------------------------------------------
template <bool kSparse>
__device__ void load_q(const AttnArgs &a, Shared &sh, uint8_t *sq, const RowTile &rt, int b, int rt_par, int lt) {
    // lt in 0..127: two threads per row (row = lt/2), each 36 of the 72 16-B chunks;
    // pass 1 finds the row maximum, pass 2 re-reads (cache hits), scales and stores.
    const int row = lt >> 1, half = lt & 1;
    const bool ok = row < rt.nvalid;
    const uint4 *src = reinterpret_cast<const uint4 *>(a.q + (rt.grow0 + (ok ? row : 0)) * kDqk) + half * 36;
    float mx = 0.f;
    if (ok) {
#pragma unroll 6
        for (int i = 0; i < 36; ++i) {
            const uint4 v = __ldg(src + i);
            const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&v);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float2 f = __bfloat1622float2(h[j]);
                mx = fmaxf(mx, fmaxf(fabsf(f.x), fabsf(f.y)));
            }
        }
    }
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    int e = 0;
    if (mx > 0.f) frexpf(mx, &e);
    const float scale = mx > 0.f ? ldexpf(1.f, 1 - e) : 1.f;
#pragma unroll 6
    for (int i = 0; i < 36; ++i) {
        const int c = half * 36 + i;           // 16-B chunk of the row (8 dims)
        const int slice = c >> 3, chunk = c & 7;
        const uint4 v = ok ? __ldg(src + i) : make_uint4(0, 0, 0, 0);
        const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&v);
        uint32_t w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float2 f = __bfloat1622float2(h[j]);
            w[j] = pack_half2(f.x * scale, f.y * scale);
        }
        *reinterpret_cast<uint4 *>(sq + slice * kQSlice + swz(row, chunk)) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    if (half == 0) {
        sh.rowscale[rt_par][row] = a.sm_scale_log2 / scale;
        if (kSparse) {
            sh.rowlimit[rt_par][row] = ok ? rt.qpos : -1;
        } else {
            const int P = __ldg(a.prefix_lens + b);
            const int r_lo = static_cast<int>(rt.grow0 - static_cast<int64_t>(__ldg(a.cu_seqlens + b)) * a.H);
            sh.rowlimit[rt_par][row] = ok ? P + (r_lo + row) / a.H : -1;
        }
    }
}

// Metadata and cache row of key k (0..127) of key tile j.
template <bool kSparse>
__device__ __forceinline__ int64_t key_row(const AttnArgs &a, const int32_t *bt, const RowTile &rt, int j, int k,
                                           float &sig) {
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
    const int64_t row = pos >= 0 ? cache_row(bt, a.max_blocks, a.num_blocks, pos, a.dev_err) : -1;
    sig = row >= 0 ? __ldg(a.kv_scale + row) : 1.f;
    return row;
}

// Raw e4m3 bytes of slices s0..s0+NS-1 (64 dims each) of one cache row.
template <int NS>
__device__ __forceinline__ void fetch_slices(const uint8_t *kv, int64_t row, int s0, uint4 (&raw)[NS * 4]) {
#pragma unroll
    for (int s = 0; s < NS; ++s)
#pragma unroll
        for (int i = 0; i < 4; ++i)
            raw[4 * s + i] = row >= 0 ? __ldg(reinterpret_cast<const uint4 *>(kv + row * kDqk + (s0 + s) * 64) + i)
                                      : make_uint4(0, 0, 0, 0);
}
// e4m3 -> f16 (exact) into the swizzled K slices, key k.
template <int NS>
__device__ __forceinline__ void store_slices(uint8_t *sk, int k, int s0, const uint4 (&raw)[NS * 4]) {
#pragma unroll
    for (int s = 0; s < NS; ++s) {
        uint8_t *dst = sk + (s0 + s) * kKSlice;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint4 r = raw[4 * s + i];
            uint32_t h[8];
            e4m3x4_to_f16x4(r.x, h[0], h[1]);
            e4m3x4_to_f16x4(r.y, h[2], h[3]);
            e4m3x4_to_f16x4(r.z, h[4], h[5]);
            e4m3x4_to_f16x4(r.w, h[6], h[7]);
            *reinterpret_cast<uint4 *>(dst + swz(k, 2 * i)) = make_uint4(h[0], h[1], h[2], h[3]);
            *reinterpret_cast<uint4 *>(dst + swz(k, 2 * i + 1)) = make_uint4(h[4], h[5], h[6], h[7]);
        }
    }
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
template <bool kSparse>
__global__ void __launch_bounds__(NT, 1) attn_kernel(const AttnArgs a, const int4 *__restrict__ work) {
    extern __shared__ __align__(1024) uint8_t dsm[];
    __shared__ Shared sh;
    const uint32_t raw = smem_u32(dsm);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    uint8_t *sq = dsm + pad;
    uint8_t *sk = sq + kSmemQ;
    const uint32_t sq_a = raw + pad, sk_a = sq_a + kSmemQ;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // ----- the row tiles of this CTA -----
    int b = 0, tiles[2] = {-1, -1};
    int64_t sp_tok = 0;
    int sp_h0 = 0;
    if (kSparse) {
        sp_tok = blockIdx.x;
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
    const int n_rt = tiles[1] >= 0 ? 2 : 1;
    const int32_t *bt = a.block_table + static_cast<int64_t>(b) * a.max_blocks;

    if (tid == 0) {
        for (int i = 0; i < NBAR; ++i) {
            uint32_t cnt = 1;
            if (i == B_FULL_ROPE || i == B_FULL_A || i == B_FULL_B || i == B_Q_FULL || i == B_META0 || i == B_META1)
                cnt = 4;                                                                          // 4 loader warps
            if (i == B_S_FREE || i == B_P_FULL || i == B_O_FREE) cnt = 4;                      // 4 softmax warps
            mbar_init(smem_u32(&sh.bar[i]), cnt);
        }
        sh.abort = 0;
        mbar_fence_init();
    }
    if (warp == 8) {
        tmem_alloc(smem_u32(&sh.tmem_base), 512);
        tmem_relinquish();
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = sh.tmem_base;
    const Wait wait{&sh, a.dev_err};

    if (warp >= 4 && warp < 8) {
        // =================== loaders ===================
        const int lt = tid - 128;              // 0..127 = key index within a tile
        uint32_t ph_free_rope = 0, ph_free_a = 0, ph_free_b = 0, ph_q_free = 0;
        int ktile_global = 0;                  // key tiles loaded so far (meta ring index)
        for (int r = 0; r < n_rt; ++r) {
            const RowTile rt = make_tile<kSparse>(a, b, tiles[r], sp_tok, sp_h0);
            if (r > 0) {                       // Q is reusable once the last QK of the previous row tile is done
                if (!wait(B_Q_FREE, ph_q_free)) break;
                ph_q_free ^= 1;
            }
            load_q<kSparse>(a, sh, sq, rt, b, r & 1, lt);
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&sh.bar[B_Q_FULL]));
            bool ok = true;
            for (int j = 0; j < rt.n_ktiles && ok; ++j, ++ktile_global) {
                float sig;
                const int64_t row = key_row<kSparse>(a, bt, rt, j, lt, sig);
                const bool first = ktile_global == 0;
                KeyMeta &m = sh.meta[ktile_global & 3][lt];
                m.sig = sig;
                m.lsig = row >= 0 ? __log2f(sig) : -INFINITY;
                m.isig = 1.f / sig;
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&sh.bar[(ktile_global & 1) ? B_META1 : B_META0]));
                {   // slice 8 (RoPE dims): free once QK of the previous tile has used it
                    uint4 raw[4];
                    fetch_slices<1>(a.kv, row, 8, raw);
                    if (!first && !(ok = wait(B_FREE_ROPE, ph_free_rope))) break;
                    if (!first) ph_free_rope ^= 1;
                    store_slices<1>(sk, lt, 8, raw);
                    fence_proxy_async();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&sh.bar[B_FULL_ROPE]));
                }
#pragma unroll 1
                for (int g = 0; g < 2; ++g) {   // slices 0-3, then 4-7: free after the matching PV half
                    uint4 raw[16];
                    fetch_slices<4>(a.kv, row, 4 * g, raw);
                    if (!first) {
                        if (!(ok = wait(g ? B_FREE_B : B_FREE_A, g ? ph_free_b : ph_free_a))) break;
                        if (g) ph_free_b ^= 1; else ph_free_a ^= 1;
                    }
                    store_slices<4>(sk, lt, 4 * g, raw);
                    fence_proxy_async();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&sh.bar[g ? B_FULL_B : B_FULL_A]));
                }
            }
            if (!ok) break;
        }
    } else if (warp == 8) {
        // =================== MMA issuer ===================
        if (lane == 0) {
            const uint32_t id_qk = idesc_f16(BM, BN, false, false, false, false);
            const uint32_t id_pv = idesc_f16(BM, 256, false, false, false, true);
            uint32_t ph_full_rope = 0, ph_full_a = 0, ph_full_b = 0, ph_s_free = 0, ph_p_full = 0, ph_q_full = 0,
                     ph_o_free = 0;
            int ktile_global = 0;
            bool ok = true;
            for (int r = 0; r < n_rt && ok; ++r) {
                const RowTile rt = make_tile<kSparse>(a, b, tiles[r], sp_tok, sp_h0);
                ok = wait(B_Q_FULL, ph_q_full);
                ph_q_full ^= 1;
                fence_after_sync();
                for (int j = 0; j < rt.n_ktiles && ok; ++j, ++ktile_global) {
                    // ---- S = Q K^T, slice order 8, 0-3, 4-7 ----
                    if (!(ok = wait(B_FULL_ROPE, ph_full_rope))) break;
                    ph_full_rope ^= 1;
                    if (ktile_global > 0) {
                        if (!(ok = wait(B_S_FREE, ph_s_free))) break;
                        ph_s_free ^= 1;
                    }
                    fence_after_sync();
                    for (int s = 0; s < NSLICE && ok; ++s) {
                        const int slice = s == 0 ? 8 : s - 1;
                        if (s == 1) {
                            if (!(ok = wait(B_FULL_A, ph_full_a))) break;
                            ph_full_a ^= 1;
                            fence_after_sync();
                        }
                        if (s == 5) {
                            if (!(ok = wait(B_FULL_B, ph_full_b))) break;
                            ph_full_b ^= 1;
                            fence_after_sync();
                        }
#pragma unroll
                        for (int ks = 0; ks < 4; ++ks) {
                            const uint64_t da = sdesc(sq_a + slice * kQSlice + ks * 32, 16, 1024, kSw128);
                            const uint64_t db = sdesc(sk_a + slice * kKSlice + ks * 32, 16, 1024, kSw128);
                            mma_f16_ss(tmem + kColS, da, db, id_qk, (s > 0 || ks > 0) ? 1u : 0u);
                        }
                        if (s == 0) mma_commit(smem_u32(&sh.bar[B_FREE_ROPE]));
                    }
                    if (!ok) break;
                    mma_commit(smem_u32(&sh.bar[B_S_FULL]));
                    if (j + 1 == rt.n_ktiles) mma_commit(smem_u32(&sh.bar[B_Q_FREE]));
                    // ---- O += P V ----
                    if (j == 0 && r > 0) {
                        if (!(ok = wait(B_O_FREE, ph_o_free))) break;
                        ph_o_free ^= 1;
                    }
                    if (!(ok = wait(B_P_FULL, ph_p_full))) break;
                    ph_p_full ^= 1;
                    fence_after_sync();
#pragma unroll 1
                    for (int h = 0; h < 2; ++h) {
                        const uint32_t lane_off = h ? kHalf1 : 0u;
#pragma unroll
                        for (int ks = 0; ks < BN / 16; ++ks) {
                            const uint64_t dbv = sdesc(sk_a + (4 * h) * kKSlice + ks * 2048, kKSlice, 1024, kSw128);
                            mma_f16_ts(tmem + lane_off + kColO, tmem + lane_off + kColP + ks * 8, dbv, id_pv,
                                       (j > 0 || ks > 0) ? 1u : 0u);
                        }
                        mma_commit(smem_u32(&sh.bar[h ? B_FREE_B : B_FREE_A]));
                    }
                    mma_commit(smem_u32(&sh.bar[B_PV_DONE]));
                }
            }
            mma_commit(smem_u32(&sh.bar[B_FINAL]));
        }
        __syncwarp();
    } else {
        // =================== softmax / correction (warps 0-3) ===================
        const int q = warp;                        // TMEM lane quadrant
        const bool lo = lane < 16;                 // lower half: S, P_a, O_a ; upper: P_b, O_b
        const int row = 16 * q + (lane & 15);
        const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
        uint32_t ph_s_full = 0, ph_pv_done = 0, ph_meta[2] = {0, 0};
        int ktile_global = 0;
        bool ok = true;
        for (int r = 0; r < n_rt && ok; ++r) {
            const RowTile rt = make_tile<kSparse>(a, b, tiles[r], sp_tok, sp_h0);
            float m_ref = -INFINITY, l_sum = 0.f;
            float rs = 0.f;
            int lim = -1;
            for (int j = 0; j < rt.n_ktiles && ok; ++j, ++ktile_global) {
                if (!(ok = wait((ktile_global & 1) ? B_META1 : B_META0, ph_meta[ktile_global & 1]))) break;
                ph_meta[ktile_global & 1] ^= 1;
                if (!(ok = wait(B_S_FULL, ph_s_full))) break;
                ph_s_full ^= 1;
                fence_after_sync();
                if (j == 0) {
                    rs = sh.rowscale[r & 1][row];
                    lim = sh.rowlimit[r & 1][row];
                }
                // S row: lower-half threads keep keys 0..63, upper-half threads take keys 64..127
                // of the same row from the lower-half lane that holds them
                uint32_t sv[64];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t t[16];
                    tmem_ld16(tmem + lane_addr + kColS + 64 + 16 * c, t);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const uint32_t x = __shfl_sync(0xffffffffu, t[i], lane & 15);
                        if (!lo) sv[16 * c + i] = x;
                    }
                }
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    uint32_t t[16];
                    tmem_ld16(tmem + lane_addr + kColS + 16 * c, t);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        if (lo) sv[16 * c + i] = t[i];
                }
                fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&sh.bar[B_S_FREE]));
                // ---- logits in the log2 domain, tile max ----
                const KeyMeta *meta = sh.meta[ktile_global & 3] + (lo ? 0 : 64);
                const int key0 = (kSparse ? 0 : j * BN) + (lo ? 0 : 64);
                float mx = -INFINITY;
#pragma unroll
                for (int i = 0; i < 64; ++i) {
                    const float4 km = *reinterpret_cast<const float4 *>(&meta[i]);
                    const bool vis = kSparse ? lim >= 0 : (key0 + i <= lim);
                    const float u = vis ? fmaf(__uint_as_float(sv[i]) * km.x, rs, km.y) : -INFINITY;
                    sv[i] = __float_as_uint(u);
                    mx = fmaxf(mx, u);
                }
                mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
                // ---- reference max: moves (and O is rescaled) only when it grows by > 2^8 ----
                float alpha = 1.f;
                bool rescale = false;
                if (j == 0) {
                    m_ref = mx;
                } else if (mx > m_ref + kRescaleThreshold) {
                    alpha = fast_exp2(m_ref - mx);
                    m_ref = mx;
                    rescale = true;
                }
                const float mu = m_ref == -INFINITY ? 0.f : m_ref;
                float ls = 0.f;
                uint32_t pk[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const float p0 = fast_exp2(__uint_as_float(sv[2 * i]) - mu);
                    const float p1 = fast_exp2(__uint_as_float(sv[2 * i + 1]) - mu);
                    const float4 k0 = *reinterpret_cast<const float4 *>(&meta[2 * i]);
                    const float4 k1 = *reinterpret_cast<const float4 *>(&meta[2 * i + 1]);
                    ls = fmaf(p0, k0.z, fmaf(p1, k1.z, ls));
                    pk[i] = pack_half2(p0, p1);
                }
                ls += __shfl_xor_sync(0xffffffffu, ls, 16);
                l_sum = fmaf(l_sum, alpha, ls);
                // ---- the previous PV must be done before O is touched or P overwritten ----
                if (j > 0) {
                    if (!(ok = wait(B_PV_DONE, ph_pv_done))) break;
                    ph_pv_done ^= 1;
                    fence_after_sync();
                }
                if (__any_sync(0xffffffffu, rescale)) {
#pragma unroll 1
                    for (int c0 = 0; c0 < 256; c0 += 16) {
                        uint32_t o[16];
                        tmem_ld16(tmem + lane_addr + kColO + c0, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                        tmem_st16(tmem + lane_addr + kColO + c0, o);
                    }
                }
                // ---- P for all 128 keys into this thread's own lane (both halves hold a copy) ----
                uint32_t full[64];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const uint32_t other = __shfl_xor_sync(0xffffffffu, pk[i], 16);
                    full[i] = lo ? pk[i] : other;
                    full[32 + i] = lo ? other : pk[i];
                }
#pragma unroll
                for (int c0 = 0; c0 < 64; c0 += 16) {
                    uint32_t t[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) t[i] = full[c0 + i];
                    tmem_st16(tmem + lane_addr + kColP + c0, t);
                }
                tmem_st_wait();
                fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&sh.bar[B_P_FULL]));
            }
            if (!ok) break;
            // ---- epilogue: O / l to bf16, lse ----
            if (!(ok = wait(B_PV_DONE, ph_pv_done))) break;
            ph_pv_done ^= 1;
            fence_after_sync();
            const bool valid = row < rt.nvalid && lim >= 0;
            const float inv = l_sum > 0.f ? 1.f / l_sum : 0.f;
            __nv_bfloat16 *dst = a.out + (rt.grow0 + row) * kDv + (lo ? 0 : 256);
#pragma unroll 1
            for (int c0 = 0; c0 < 256; c0 += 32) {
                uint32_t o[32];
                tmem_ld32(tmem + lane_addr + kColO + c0, o);
                tmem_ld_wait();
                if (valid) {
                    uint4 *d4 = reinterpret_cast<uint4 *>(dst + c0);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        uint4 w;
                        w.x = pack_bf162(__uint_as_float(o[8 * i + 0]) * inv, __uint_as_float(o[8 * i + 1]) * inv);
                        w.y = pack_bf162(__uint_as_float(o[8 * i + 2]) * inv, __uint_as_float(o[8 * i + 3]) * inv);
                        w.z = pack_bf162(__uint_as_float(o[8 * i + 4]) * inv, __uint_as_float(o[8 * i + 5]) * inv);
                        w.w = pack_bf162(__uint_as_float(o[8 * i + 6]) * inv, __uint_as_float(o[8 * i + 7]) * inv);
                        d4[i] = w;
                    }
                }
            }
            if (valid && lo && a.lse)
                a.lse[rt.grow0 + row] = l_sum > 0.f ? (m_ref + __log2f(l_sum)) * kLn2 : -INFINITY;
            fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&sh.bar[B_O_FREE]));
        }
    }

    // ----- teardown: every MMA complete before TMEM is released -----
    __syncthreads();
    if (warp == 8) {
        if (!mbar_wait_cycles(smem_u32(&sh.bar[B_FINAL]), 0, kWaitCycles)) set_dev_err(a.dev_err, MLA_DEVERR_TIMEOUT);
        fence_after_sync();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace tcattn

cudaError_t launch_dense_tc(const AttnArgs &a, const int4 *work, int n_work, cudaStream_t st) {
    cudaError_t e =
        cudaFuncSetAttribute(tcattn::attn_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, tcattn::kDynSmem);
    if (e != cudaSuccess) return e;
    if (n_work > 0) tcattn::attn_kernel<false><<<n_work, tcattn::NT, tcattn::kDynSmem, st>>>(a, work);
    return cudaGetLastError();
}

cudaError_t launch_sparse_tc(const AttnArgs &a, int64_t n_tokens, cudaStream_t st) {
    cudaError_t e =
        cudaFuncSetAttribute(tcattn::attn_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, tcattn::kDynSmem);
    if (e != cudaSuccess) return e;
    dim3 grid(static_cast<unsigned>(n_tokens), (a.H + tcattn::BM - 1) / tcattn::BM);
    if (n_tokens > 0) tcattn::attn_kernel<true><<<grid, tcattn::NT, tcattn::kDynSmem, st>>>(a, nullptr);
    return cudaGetLastError();
}

}  // namespace mla

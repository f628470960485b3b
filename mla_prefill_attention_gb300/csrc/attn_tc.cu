// MLA prefill attention on the 5th-generation tensor cores (tcgen05 + TMEM).
//
// One CTA owns a tile of 64 query rows (row = (token, head); for 64 heads one
// token) and streams the latent rows of the paged e4m3 cache 128 keys at a
// time. Per key tile:
//
//   S   = Q K'^T         tcgen05.mma kind::f16, M=64 N=128, K=576, D in TMEM
//   u   = S*sigma'*rowscale + log2(sigma)       (log2 domain, sigma folded in)
//   P   = 2^(u - m),  l += P / sigma             (m: running reference max)
//   O  += P V'           tcgen05.mma M=64 N=256 (two Dv halves), A=P from TMEM
//
// and at the end out = 2^8 O / l, lse = ln2 (m + log2 l). K' and V' hold the
// e4m3 codes times 2^-8: the f16 bit pattern of that product is the code's own
// bits moved into place (see f16x2_of_e4m3x2), so dequantisation costs three
// integer operations per code pair and sigma' = 2^8 sigma restores the scale.
//
// Why 64 rows: with the 512-wide value head an fp32 O for 128 rows fills all
// 512 TMEM columns, and a 128 x 576 f16 Q tile alone is 144 KB of shared
// memory. With 64 rows, O takes two lane-halves x 256 columns and Q 72 KB.
// M=64 MMAs run at half the M=128 rate on this part (2048 vs 4096 MAC/clk per
// SM, measured), so this kernel is capped at half the dense tensor peak per
// clock.
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
// Warps: 0-3 softmax/correction (warp w owns TMEM lane quadrant w and reads S
// with the 16-lane shapes, so each thread holds two rows x 32 keys), 4-7
// loaders (one key per thread: the raw e4m3 bytes of the next key tile are
// fetched into registers while the current one is converted into the
// swizzled K slices), 8 MMA issue, 9-11 idle. Launched at 168 registers a
// thread, the softmax and loader warpgroups grow to 200 and 232 while the
// issuer's warpgroup shrinks to 56 (128 x (200 + 232 + 56) <= 384 x 168).
// The K tile is single-buffered but recycled
// slice-group by slice-group: slice 8 is refilled as soon as QK has used it
// (and the next tile's RoPE part of QK runs while the softmax works), slices
// 0-3 after the first PV half, slices 4-7 after the second. Every wait is
// bounded; a wait that runs out sets MLA_DEVERR_TIMEOUT and the CTA abandons
// its tile.
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
constexpr int NT = 384;           // 12 warps = 3 warpgroups
constexpr int kQSlice = BM * 128;         // 8192 B
constexpr int kKSlice = BN * 128;         // 16384 B
constexpr int kSmemQ = NSLICE * kQSlice;  // 73728
constexpr int kSmemK = NSLICE * kKSlice;  // 147456
constexpr int kDynSmem = 1024 + kSmemQ + kSmemK;
constexpr long long kWaitCycles = 200000000LL;   // ~0.1 s: every wait here covers at most one tile of work
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only when the max grows by > 2^8
constexpr float kCodeScale = 256.0f;       // K', V' hold code * 2^-8
constexpr uint32_t kRegsSoftmax = 200, kRegsLoader = 232, kRegsIssuer = 56;   // per-thread budgets after the split
static_assert(128 * (kRegsSoftmax + kRegsLoader + kRegsIssuer) <= NT * 168, "register split exceeds the launch pool");

// TMEM columns
constexpr uint32_t kColO = 0, kColS = 256, kColP = 384;
constexpr uint32_t kHalf1 = 16u << 16;     // lane offset of the upper half

enum Bar {
    B_FULL_ROPE, B_FULL_A, B_FULL_B,    // loaders -> issuer: K slices converted (8 | 0-3 | 4-7)
    B_FREE_A, B_FREE_B,                 // issuer (MMA commit) -> loaders: V slices consumed by PV
    B_S_FULL,                           // issuer -> softmax, loaders: QK complete (S ready, slice 8 and Q reusable)
    B_S_FREE,                           // softmax -> issuer: S read out
    B_P_FULL,                           // softmax -> issuer: P written (and O rescaled)
    B_PV_DONE,                          // issuer -> softmax: PV of the tile complete
    B_Q_FULL,                           // loaders -> issuer, softmax: Q tile and row data in smem
    B_O_FREE,                           // softmax -> issuer: epilogue finished reading O
    B_FINAL,                            // issuer -> all: every MMA of the CTA complete
    B_META0, B_META1,                   // loaders -> softmax: key metadata of tile n, n&1
    NBAR
};

struct __align__(16) KeyMeta {
    float sig, lsig, isig, pad;          // 2^8 sigma, log2 sigma (-inf = masked), 1/sigma
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

// Cache row of key k (0..127) of key tile j (-1: no key) and its scale.
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

__device__ __forceinline__ void write_meta(KeyMeta &m, int64_t row, float sig) {
    m.sig = sig * kCodeScale;
    m.lsig = row >= 0 ? __log2f(sig) : -INFINITY;
    m.isig = 1.f / sig;
}

// Raw e4m3 bytes of slices s0..s0+NS-1 (64 dims each) of one cache row.
template <int NS>
__device__ __forceinline__ void fetch_slices(const uint8_t *kv, int64_t row, int s0, uint4 *raw) {
#pragma unroll
    for (int s = 0; s < NS; ++s)
#pragma unroll
        for (int i = 0; i < 4; ++i)
            raw[4 * s + i] = row >= 0 ? __ldg(reinterpret_cast<const uint4 *>(kv + row * kDqk + (s0 + s) * 64) + i)
                                      : make_uint4(0, 0, 0, 0);
}

// Two e4m3 codes (bytes 0 and 2 of t, bytes 1 and 3 zero) -> f16x2 of code * 2^-8,
// exactly: an e4m3 code's exponent and mantissa fields, moved to bits 7..14,
// read as an f16 are the code's value times 2^-8 (normal and subnormal alike,
// since both formats have the same subnormal step relative to their bias);
// adding the sign bit to itself carries it from bit 14 to bit 15.
// The two NaN codes (0x7F, 0xFF) come out as +-480 * 2^-8; quantised caches
// never hold them.
__device__ __forceinline__ uint32_t f16x2_of_e4m3x2(uint32_t t) { return (t + (t & 0x00800080u)) << 7; }

template <int NS>
__device__ __forceinline__ void store_slices(uint8_t *sk, int k, int s0, const uint4 *raw) {
#pragma unroll
    for (int s = 0; s < NS; ++s) {
        uint8_t *dst = sk + (s0 + s) * kKSlice;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint4 r = raw[4 * s + i];
            uint32_t h[8];
            h[0] = f16x2_of_e4m3x2(__byte_perm(r.x, 0u, 0x4140u));
            h[1] = f16x2_of_e4m3x2(__byte_perm(r.x, 0u, 0x4342u));
            h[2] = f16x2_of_e4m3x2(__byte_perm(r.y, 0u, 0x4140u));
            h[3] = f16x2_of_e4m3x2(__byte_perm(r.y, 0u, 0x4342u));
            h[4] = f16x2_of_e4m3x2(__byte_perm(r.z, 0u, 0x4140u));
            h[5] = f16x2_of_e4m3x2(__byte_perm(r.z, 0u, 0x4342u));
            h[6] = f16x2_of_e4m3x2(__byte_perm(r.w, 0u, 0x4140u));
            h[7] = f16x2_of_e4m3x2(__byte_perm(r.w, 0u, 0x4342u));
            *reinterpret_cast<uint4 *>(dst + swz(k, 2 * i)) = make_uint4(h[0], h[1], h[2], h[3]);
            *reinterpret_cast<uint4 *>(dst + swz(k, 2 * i + 1)) = make_uint4(h[4], h[5], h[6], h[7]);
        }
    }
}

// (row tile, key tile) -> next (row tile, key tile) in the CTA's visiting order
struct Cursor {
    int r, j, n;        // row tile, key tile, key tiles of row tile r
};

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
        regs_inc<kRegsLoader>();
        // Tile t's raw bytes are in registers when iteration t starts; each
        // group is converted once its slots are free and the same group of
        // tile t+1 is fetched right after, a whole tile ahead of its use.
        const int lt = tid - 128;              // key index within a tile
        RowTile rt = make_tile<kSparse>(a, b, tiles[0], sp_tok, sp_h0);
        Cursor cur{0, 0, rt.n_ktiles};
        RowTile rt_next = rt;
        uint4 r_rope[4], r_a[16], r_b[16];
        float sig;
        int64_t row = key_row<kSparse>(a, bt, rt, 0, lt, sig);
        write_meta(sh.meta[0][lt], row, sig);
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sh.bar[B_META0]));
        fetch_slices<1>(a.kv, row, 8, r_rope);
        fetch_slices<4>(a.kv, row, 0, r_a);
        fetch_slices<4>(a.kv, row, 4, r_b);
        load_q<kSparse>(a, sh, sq, rt, b, 0, lt);
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&sh.bar[B_Q_FULL]));
        for (int t = 0;; ++t) {
            // ---- slice 8: free once the previous tile's QK is complete (that also frees Q) ----
            if (t > 0) {
                if (!wait(B_S_FULL, (t - 1) & 1)) break;
                if (cur.j == 0) {
                    load_q<kSparse>(a, sh, sq, rt, b, cur.r & 1, lt);
                    fence_proxy_async();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&sh.bar[B_Q_FULL]));
                }
            }
            store_slices<1>(sk, lt, 8, r_rope);
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&sh.bar[B_FULL_ROPE]));
            // ---- the next tile: metadata now, raw bytes group by group ----
            Cursor nxt = cur;
            bool more = true;
            if (++nxt.j == nxt.n) {
                nxt.j = 0;
                if (++nxt.r < n_rt) {
                    rt_next = make_tile<kSparse>(a, b, tiles[nxt.r], sp_tok, sp_h0);
                    nxt.n = rt_next.n_ktiles;
                } else {
                    more = false;
                }
            }
            int64_t row_n = -1;
            if (more) {
                row_n = key_row<kSparse>(a, bt, rt_next, nxt.j, lt, sig);
                write_meta(sh.meta[(t + 1) & 3][lt], row_n, sig);
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&sh.bar[((t + 1) & 1) ? B_META1 : B_META0]));
                fetch_slices<1>(a.kv, row_n, 8, r_rope);
            }
            // ---- slices 0-3, then 4-7: free after the matching half of the previous PV ----
            if (t > 0 && !wait(B_FREE_A, (t - 1) & 1)) break;
            store_slices<4>(sk, lt, 0, r_a);
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&sh.bar[B_FULL_A]));
            if (more) fetch_slices<4>(a.kv, row_n, 0, r_a);
            if (t > 0 && !wait(B_FREE_B, (t - 1) & 1)) break;
            store_slices<4>(sk, lt, 4, r_b);
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&sh.bar[B_FULL_B]));
            if (!more) break;
            fetch_slices<4>(a.kv, row_n, 4, r_b);
            cur = nxt;
            rt = rt_next;
        }
    } else if (warp >= 8) {
        // =================== MMA issuer (warp 8, lane 0) ===================
        regs_dec<kRegsIssuer>();
        if (warp == 8 && lane == 0) {
            const uint32_t id_qk = idesc_f16(BM, BN, false, false, false, false);
            const uint32_t id_pv = idesc_f16(BM, 256, false, false, false, true);
            // Descriptors of the operand bases; an operand at byte offset x is the base
            // descriptor plus x/16 (start-address field; shared addresses stay below 2^18).
            const uint64_t dq0 = sdesc(sq_a, 16, 1024, kSw128);
            const uint64_t dk0 = sdesc(sk_a, 16, 1024, kSw128);
            const uint64_t dv0 = sdesc(sk_a, kKSlice, 1024, kSw128);
            // QK over one 64-dim slice (4 MMAs of K=16)
            auto qk_slice = [&](int slice, bool first) {
                const uint64_t da = dq0 + static_cast<uint64_t>((slice * kQSlice) >> 4);
                const uint64_t db = dk0 + static_cast<uint64_t>((slice * kKSlice) >> 4);
#pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    mma_f16_ss(tmem + kColS, da + 2 * ks, db + 2 * ks, id_qk, (first && ks == 0) ? 0u : 1u);
            };
            int t = 0;
            bool rope_issued = false, ok = true;
            for (int r = 0; r < n_rt && ok; ++r) {
                const RowTile rt = make_tile<kSparse>(a, b, tiles[r], sp_tok, sp_h0);
                for (int j = 0; j < rt.n_ktiles && ok; ++j, ++t) {
                    // ---- S = Q K^T: slice 8 (unless already issued), then 0-3, 4-7 ----
                    if (!rope_issued) {
                        if (j == 0 && !(ok = wait(B_Q_FULL, r & 1))) break;
                        if (!(ok = wait(B_FULL_ROPE, t & 1))) break;
                        if (t > 0 && !(ok = wait(B_S_FREE, (t - 1) & 1))) break;
                        fence_after_sync();
                        qk_slice(8, true);
                    }
                    rope_issued = false;
                    if (!(ok = wait(B_FULL_A, t & 1))) break;
                    fence_after_sync();
#pragma unroll 1
                    for (int s = 0; s < 4; ++s) qk_slice(s, false);
                    if (!(ok = wait(B_FULL_B, t & 1))) break;
                    fence_after_sync();
#pragma unroll 1
                    for (int s = 4; s < 8; ++s) qk_slice(s, false);
                    mma_commit(smem_u32(&sh.bar[B_S_FULL]));
                    // ---- the next tile's RoPE slice while the softmax works on this one ----
                    if (j + 1 < rt.n_ktiles) {
                        if (!(ok = wait(B_FULL_ROPE, (t + 1) & 1))) break;
                        if (!(ok = wait(B_S_FREE, t & 1))) break;
                        fence_after_sync();
                        qk_slice(8, true);
                        rope_issued = true;
                    }
                    // ---- O += P V ----
                    if (j == 0 && r > 0) {
                        if (!(ok = wait(B_O_FREE, (r - 1) & 1))) break;
                    }
                    if (!(ok = wait(B_P_FULL, t & 1))) break;
                    fence_after_sync();
#pragma unroll 1
                    for (int h = 0; h < 2; ++h) {
                        const uint32_t lane_off = h ? kHalf1 : 0u;
                        const uint64_t dv = dv0 + static_cast<uint64_t>((4 * h * kKSlice) >> 4);
#pragma unroll
                        for (int ks = 0; ks < BN / 16; ++ks)
                            mma_f16_ts(tmem + lane_off + kColO, tmem + lane_off + kColP + ks * 8, dv + 128 * ks, id_pv,
                                       (j > 0 || ks > 0) ? 1u : 0u);
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
        regs_inc<kRegsSoftmax>();
        // S is read with the 16-lane shapes: thread t holds rows ra = 16q + t/4
        // and rb = ra + 8, keys 8i + 2(t%4) + {0,1} for i = 0..15.
        const int q = warp;                        // TMEM lane quadrant
        const int tq = lane >> 2, tc = lane & 3;
        const int ra = 16 * q + tq, rb = ra + 8;
        const uint32_t lane_addr = static_cast<uint32_t>(32 * q) << 16;
        int t = 0;
        bool ok = true;
        for (int r = 0; r < n_rt && ok; ++r) {
            const RowTile rt = make_tile<kSparse>(a, b, tiles[r], sp_tok, sp_h0);
            float m_a = -INFINITY, m_b = -INFINITY;  // reference maxima (log2 domain)
            float l_a = 0.f, l_b = 0.f;              // this thread's partial row sums (32 keys per tile)
            if (!(ok = wait(B_Q_FULL, r & 1))) break;
            const float rs_a = sh.rowscale[r & 1][ra], rs_b = sh.rowscale[r & 1][rb];
            const int lim_a = sh.rowlimit[r & 1][ra], lim_b = sh.rowlimit[r & 1][rb];
            const int lim_min = min(lim_a, lim_b);
            for (int j = 0; j < rt.n_ktiles && ok; ++j, ++t) {
                if (!(ok = wait((t & 1) ? B_META1 : B_META0, (t >> 1) & 1))) break;
                if (!(ok = wait(B_S_FULL, t & 1))) break;
                fence_after_sync();
                uint32_t sv[64];
                tmem_ld_16x256b_x8(tmem + lane_addr + kColS, sv);
                tmem_ld_16x256b_x8(tmem + lane_addr + kColS + 64, sv + 32);
                tmem_ld_wait();
                fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&sh.bar[B_S_FREE]));
                // ---- logits in the log2 domain, tile maxima ----
                const KeyMeta *meta = sh.meta[t & 3];
                const int key0 = kSparse ? 0 : j * BN;
                const bool full = kSparse ? (lim_min >= 0) : (key0 + BN - 1 <= lim_min);
                float mx_a = -INFINITY, mx_b = -INFINITY;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int k0 = 8 * i + 2 * tc;
                    const float4 m0 = *reinterpret_cast<const float4 *>(&meta[k0]);
                    const float4 m1 = *reinterpret_cast<const float4 *>(&meta[k0 + 1]);
                    float u0 = fmaf(__uint_as_float(sv[4 * i + 0]) * m0.x, rs_a, m0.y);
                    float u1 = fmaf(__uint_as_float(sv[4 * i + 1]) * m1.x, rs_a, m1.y);
                    float u2 = fmaf(__uint_as_float(sv[4 * i + 2]) * m0.x, rs_b, m0.y);
                    float u3 = fmaf(__uint_as_float(sv[4 * i + 3]) * m1.x, rs_b, m1.y);
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
                }
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
                const float mu_a = m_a == -INFINITY ? 0.f : m_a, mu_b = m_b == -INFINITY ? 0.f : m_b;
                l_a *= al_a;
                l_b *= al_b;
                uint32_t pk[32];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int k0 = 8 * i + 2 * tc;
                    const float i0 = meta[k0].isig, i1 = meta[k0 + 1].isig;
                    const float p0 = fast_exp2(__uint_as_float(sv[4 * i + 0]) - mu_a);
                    const float p1 = fast_exp2(__uint_as_float(sv[4 * i + 1]) - mu_a);
                    const float p2 = fast_exp2(__uint_as_float(sv[4 * i + 2]) - mu_b);
                    const float p3 = fast_exp2(__uint_as_float(sv[4 * i + 3]) - mu_b);
                    l_a = fmaf(p0, i0, fmaf(p1, i1, l_a));
                    l_b = fmaf(p2, i0, fmaf(p3, i1, l_b));
                    pk[2 * i] = pack_half2(p0, p1);
                    pk[2 * i + 1] = pack_half2(p2, p3);
                }
                // ---- the previous PV must be done before O is touched or P overwritten ----
                if (j > 0) {
                    if (!(ok = wait(B_PV_DONE, (t - 1) & 1))) break;
                    fence_after_sync();
                }
                if (__any_sync(0xffffffffu, resc)) {
                    // 32x32b view: lane L holds row 16q + L%16, half L/16; its factor lives in
                    // thread 4 (L%8) as row a (L%16 < 8) or row b
                    const int rr = lane & 15;
                    const float xa = __shfl_sync(0xffffffffu, al_a, 4 * (rr & 7));
                    const float xb = __shfl_sync(0xffffffffu, al_b, 4 * (rr & 7));
                    const float al = rr < 8 ? xa : xb;
#pragma unroll 1
                    for (int c0 = 0; c0 < 256; c0 += 16) {
                        uint32_t o[16];
                        tmem_ld16(tmem + lane_addr + kColO + c0, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 16; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * al);
                        tmem_st16(tmem + lane_addr + kColO + c0, o);
                    }
                }
                // ---- P into both lane halves (A operand of the two PV halves) ----
                tmem_st_16x128b_x16(tmem + lane_addr + kColP, pk);
                tmem_st_16x128b_x16(tmem + lane_addr + kHalf1 + kColP, pk);
                tmem_st_wait();
                fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(smem_u32(&sh.bar[B_P_FULL]));
            }
            if (!ok) break;
            // ---- epilogue: O 2^8 / l to bf16, lse ----
            if (!(ok = wait(B_PV_DONE, (t - 1) & 1))) break;
            fence_after_sync();
            l_a += __shfl_xor_sync(0xffffffffu, l_a, 1);
            l_b += __shfl_xor_sync(0xffffffffu, l_b, 1);
            l_a += __shfl_xor_sync(0xffffffffu, l_a, 2);
            l_b += __shfl_xor_sync(0xffffffffu, l_b, 2);
            if (tc == 0 && a.lse) {
                if (ra < rt.nvalid && lim_a >= 0)
                    a.lse[rt.grow0 + ra] = l_a > 0.f ? (m_a + __log2f(l_a)) * kLn2 : -INFINITY;
                if (rb < rt.nvalid && lim_b >= 0)
                    a.lse[rt.grow0 + rb] = l_b > 0.f ? (m_b + __log2f(l_b)) * kLn2 : -INFINITY;
            }
            const int rr = lane & 15, row = 16 * q + rr;
            const float ia = l_a > 0.f ? kCodeScale / l_a : 0.f, ib = l_b > 0.f ? kCodeScale / l_b : 0.f;
            const float xa = __shfl_sync(0xffffffffu, ia, 4 * (rr & 7));
            const float xb = __shfl_sync(0xffffffffu, ib, 4 * (rr & 7));
            const float inv = rr < 8 ? xa : xb;
            const bool valid = row < rt.nvalid && sh.rowlimit[r & 1][row] >= 0;
            __nv_bfloat16 *dst = a.out + (rt.grow0 + row) * kDv + (lane < 16 ? 0 : 256);
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

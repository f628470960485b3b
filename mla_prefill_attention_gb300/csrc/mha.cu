// Non-absorbed (MHA) MLA prefill for short prompts (tcgen05 kind::f16).
//
// GLM-5.3-Optimierungen Teil 2, section Ausprobieren: without the
// sparse_mla_force_mqa flag, prefill batches whose prompts fit within the
// top-k of 2,048 tokens take the dense MHA path. Per head h, with c_s the 512
// latent values and r_s the 64 RoPE values of cached token s (580-byte row:
// sigma_s * dec(codes)):
//
//   k_{s,h} = [ W_UK_h c_s ; r_s ]   (192 dims)      v_{s,h} = W_UV_h c_s   (128 dims)
//   out[t,h] = sum_s softmax_s(sm_scale q_{t,h} . k_{s,h}) v_{s,h},   s <= p(t)
//
// Two kernels.
//
// 1. Up-projection, one CTA per 128 cached rows of a sequence and a group of
//    heads: 256 threads decode the rows' e4m3 codes into bf16 (exact: an e4m3
//    value has 4 significant bits) straight into TMEM, the MMA's A operand; the
//    tensor core multiplies them by each half head's [128 x 512] slice of w_ukv
//    (TMA, 64-dim boxes through a 12-stage ring): D[row][n] = sum_d
//    dec(c)[row][d] W[h][n][d], M = 128 rows, N = 128 (the k rows, then the v
//    rows), K = 512, into one of two TMEM accumulators;
//    four epilogue warps (thread = row) scale by sigma_row and write f16 k and
//    v rows head-major, [H][R][128]. The first head group also writes the
//    RoPE dims, f16(sigma * dec(c)), as [R][64]. Rows past the context are
//    written as zeros (each sequence's rows are padded to 128). f16 keeps 11
//    significant bits of each up-projected value (bf16 would keep 8: its
//    rounding of the keys alone moved logits by ~1e-3 and outputs by up to
//    2.5e-2 of a row's RMS); the values must stay inside the f16 range.
//
// 2. Attention, one CTA per 128 new tokens of a sequence and one head (the
//    grid head-major: every tile of head 0 in longest-first order, then head 1,
//    ...; a head's keys and values, 0.5 KB a row, stay in L2 while its tiles run).
//    Each softmax thread reads its bf16 query row, converts it to f16 (values
//    below 2^-14 lose bits, so a query must lie inside the f16 range) and stores
//    it into TMEM, where the QK MMAs take their A operand; shared memory then
//    holds four K/V stages:
//      S  = Q K^T        M = 128 tokens, N = 64 keys, K = 192 (Q from TMEM; K in
//                        3 x 64-dim slices: two no-RoPE, one RoPE); S in one of two TMEM
//                        buffers so QK(t+1) runs during the softmax of tile t
//      P  = 2^(S*sm_scale*log2e - m)   in registers (a thread per query row),
//                        rounded to f16 into shared memory
//      O += P V          M = 128, N = 128 value dims, K = 64 keys (O in TMEM)
//    m is the row's running reference maximum; O and l are rescaled only when
//    a tile raises it by more than 8 (log2 units), so P stays below 2^8. l
//    sums the fp32 P. At the end out = O / l and lse = ln2 (m + log2 l).
//    Warps 0-3 softmax and epilogue (warp w owns TMEM lanes 32w..32w+31 =
//    query rows), 4 TMA producer, 5 MMA issuer (one thread).
//
// Every wait is bounded; one that runs out sets MLA_DEVERR_TIMEOUT and the
// CTA stops; before it exits, the producer waits for its copies and the issuer
// for its MMAs.
#include <cuda.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace mla {
namespace mha {

using namespace tc;

constexpr long long kWaitCycles = 200000000LL;

__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, int32_t *dev_err) {
    if (mbar_wait_cycles(smem_u32(bar), parity, kWaitCycles)) return true;
    set_dev_err(dev_err, MLA_DEVERR_TIMEOUT);
    return false;
}

// Two e4m3 codes (low byte first) as two bf16 values (exact).
__device__ __forceinline__ uint32_t bf16x2_of_e4m3x2(uint16_t two) {
    const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two), __NV_E4M3);
    const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&hr));
    return pack_bf162(f.x, f.y);
}

// ===========================================================================
// 1. up-projection
// ===========================================================================
constexpr int UP_ROWS = 128;
constexpr int UP_NT = 320;                       // warps 0-7 decode; then 0-3 epilogue, 8 producer, 9 issuer
constexpr int UP_WST = 12;                       // weight ring stages
constexpr int kUpW = 128 * 128;                  // one 64-dim slice of 128 weight rows (a head's k or v part): 16 KB
constexpr int kUpOffSig = UP_WST * kUpW;
constexpr int kUpSmem = 1024 + kUpOffSig + UP_ROWS * 4;
constexpr uint32_t kUpColA = 0, kUpColD = 256;   // TMEM: decoded rows (512 bf16 = 256 columns), two 128-column D
static_assert(kUpSmem <= 232448 - 256, "shared memory");

enum UpBar { U_W_FULL = 0, U_W_EMPTY = U_W_FULL + UP_WST, U_D_FULL = U_W_EMPTY + UP_WST, U_D_FREE = U_D_FULL + 2,
             U_FINAL = U_D_FREE + 2, U_NBAR };

// The decoded rows stay in TMEM as the A operand (lane = row, column c = latent
// dims 2c, 2c+1), so shared memory holds only the weight ring: twelve 16 KB
// slices in flight keep the tensor core fed across the round trip from L2. One
// unit of work is half a head (its 128 k rows or its 128 v rows): M = 128 rows,
// N = 128, K = 512, into one of two 128-column accumulators.
__global__ void __launch_bounds__(UP_NT, 1)
    up_kernel(const MhaArgs a, const int4 *__restrict__ work, const __grid_constant__ CUtensorMap tmap_w) {
    extern __shared__ __align__(1024) uint8_t dsm[];
    __shared__ uint64_t bar[U_NBAR];
    __shared__ uint32_t tmem_slot;
    const uint32_t raw = smem_u32(dsm);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    uint8_t *sbase = dsm + pad;
    const uint32_t sbase_a = raw + pad;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    const int n_hg = a.H / a.up_heads;
    const int4 it = work[blockIdx.x / n_hg];
    const int hg = blockIdx.x % n_hg;
    const int b = it.x, pos0 = it.y, ctx = it.w;
    const int64_t row0 = it.z;
    const int h0 = hg * a.up_heads, n_units = 2 * a.up_heads;
    float *sig = reinterpret_cast<float *>(sbase + kUpOffSig);

    if (tid == 0) {
        for (int i = 0; i < U_NBAR; ++i) mbar_init(smem_u32(&bar[i]), (i >= U_D_FREE && i < U_D_FREE + 2) ? 4u : 1u);
        mbar_fence_init();
    }
    if (warp == 9) {
        tmem_alloc(smem_u32(&tmem_slot), 512);
        tmem_relinquish();
    }
    if (warp == 8 && lane == 0) tma_prefetch_desc(&tmap_w);
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = tmem_slot;

    // ----- decode into TMEM: warp w holds rows 32(w&3)..+31 (its lane quadrant)
    // and latent dims 256(w>>2)..+255 (TMEM columns 128(w>>2)..+127) -----
    if (warp < 8) {
        const int q = warp & 3, half = warp >> 2, r = 32 * q + lane;
        const int pos = pos0 + r;
        int64_t cr = -1;
        if (pos < ctx) cr = cache_row(a.block_table + static_cast<int64_t>(b) * a.max_blocks, a.max_blocks,
                                      a.num_blocks, pos, a.dev_err);
        const float s = cr >= 0 ? __ldg(a.kv_scale + cr) : 0.f;
        if (half == 0) sig[r] = s;
        const uint8_t *src = a.kv + (cr >= 0 ? cr : 0) * kDqk;
        const uint32_t taddr = tmem + (static_cast<uint32_t>(32 * q) << 16) + kUpColA + 128u * half;
#pragma unroll 1
        for (int g = 0; g < 4; ++g) {                  // 64 latent dims = 32 TMEM columns per group
            uint32_t o[32];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const int d0 = 256 * half + 64 * g + 16 * c;
                uint4 raw16 = make_uint4(0u, 0u, 0u, 0u);
                if (cr >= 0) raw16 = __ldg(reinterpret_cast<const uint4 *>(src + d0));
                const uint32_t wv[4] = {raw16.x, raw16.y, raw16.z, raw16.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    o[8 * c + 2 * k] = bf16x2_of_e4m3x2(static_cast<uint16_t>(wv[k] & 0xFFFFu));
                    o[8 * c + 2 * k + 1] = bf16x2_of_e4m3x2(static_cast<uint16_t>(wv[k] >> 16));
                }
            }
            tmem_st32(taddr + 32u * g, o);
        }
        if (hg == 0) {      // the shared RoPE dims: 32 per thread
            uint4 rr[2] = {make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u)};
            if (cr >= 0) {
                rr[0] = __ldg(reinterpret_cast<const uint4 *>(src + kDv + 32 * half));
                rr[1] = __ldg(reinterpret_cast<const uint4 *>(src + kDv + 32 * half + 16));
            }
            uint32_t o[16];
#pragma unroll
            for (int qq = 0; qq < 2; ++qq) {
                const uint32_t wv[4] = {rr[qq].x, rr[qq].y, rr[qq].z, rr[qq].w};
#pragma unroll
                for (int k = 0; k < 4; ++k)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const uint16_t two = static_cast<uint16_t>(wv[k] >> (16 * e));
                        const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(two, __NV_E4M3);
                        const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&hr));
                        o[8 * qq + 2 * k + e] = pack_half2(s * f.x, s * f.y);
                    }
            }
            uint4 *dst = reinterpret_cast<uint4 *>(a.kr + (row0 + r) * kDr + 32 * half);
#pragma unroll
            for (int k = 0; k < 4; ++k) dst[k] = make_uint4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
        }
        tmem_st_wait();
    }
    fence_before_sync();
    __syncthreads();
    fence_after_sync();

    if (warp == 8) {
        // =================== TMA producer: each half head's weight slices ===================
        if (lane == 0) {
            int n = 0;
            bool ok = true;
            for (int u = 0; u < n_units && ok; ++u)
                for (int s = 0; s < 8 && ok; ++s, ++n) {
                    const int st = n % UP_WST;
                    if (n >= UP_WST && !(ok = wait_bar(&bar[U_W_EMPTY + st], ((n / UP_WST) - 1) & 1, a.dev_err))) break;
                    mbar_expect_tx(smem_u32(&bar[U_W_FULL + st]), kUpW);
                    tma_load_2d(sbase_a + st * kUpW, &tmap_w, 64 * s, (h0 + (u >> 1)) * 256 + 128 * (u & 1),
                                smem_u32(&bar[U_W_FULL + st]));
                }
            // drain: the last load of every stage has landed before the CTA exits
            for (int j = (n > UP_WST ? n - UP_WST : 0); j < n; ++j)
                if (!mbar_wait_cycles(smem_u32(&bar[U_W_FULL + j % UP_WST]), (j / UP_WST) & 1, kWaitCycles))
                    set_dev_err(a.dev_err, MLA_DEVERR_TIMEOUT);
        }
    } else if (warp == 9) {
        // =================== MMA issuer ===================
        if (lane == 0) {
            const uint32_t idesc = idesc_f16(128, 128, true, true, false, false);
            const uint64_t dw0 = sdesc(sbase_a, 16, 1024, kSw128);
            int n = 0;
            bool ok = true;
            for (int u = 0; u < n_units && ok; ++u) {
                const int db = u & 1;
                if (u >= 2 && !(ok = wait_bar(&bar[U_D_FREE + db], ((u >> 1) - 1) & 1, a.dev_err))) break;
                fence_after_sync();
                const uint32_t d = tmem + kUpColD + 128u * db;
                for (int s = 0; s < 8; ++s, ++n) {
                    const int st = n % UP_WST;
                    if (!(ok = wait_bar(&bar[U_W_FULL + st], (n / UP_WST) & 1, a.dev_err))) break;
                    fence_after_sync();
                    const uint64_t dw = dw0 + static_cast<uint64_t>((st * kUpW) >> 4);
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_f16_ts_w(d, tmem + kUpColA + 32u * s + 8u * ks, dw + 2 * ks, idesc, (s | ks) ? 1u : 0u, 1u);
                    mma_commit(smem_u32(&bar[U_W_EMPTY + st]));
                }
                if (ok) mma_commit(smem_u32(&bar[U_D_FULL + db]));
            }
            mma_commit(smem_u32(&bar[U_FINAL]));
        }
    } else if (warp < 4) {
        // =================== epilogue: thread = row ===================
        const int r = 32 * warp + lane;
        const float s = sig[r];
        const uint32_t lane_addr = static_cast<uint32_t>(32 * warp) << 16;
        for (int u = 0; u < n_units; ++u) {
            const int db = u & 1, h = h0 + (u >> 1);
            const bool got = wait_bar(&bar[U_D_FULL + db], (u >> 1) & 1, a.dev_err);
            if (!__all_sync(0xffffffffu, got)) break;
            fence_after_sync();
            __half *base = ((u & 1) ? a.v : a.kn) + (static_cast<int64_t>(h) * a.R + row0 + r) * kDvh;
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                uint32_t v[32];
                tmem_ld32(tmem + lane_addr + kUpColD + 128u * db + 32u * c, v);
                tmem_ld_wait();
                uint32_t o[16];
#pragma unroll
                for (int k = 0; k < 16; ++k)
                    o[k] = pack_half2(s * __uint_as_float(v[2 * k]), s * __uint_as_float(v[2 * k + 1]));
                uint4 *dst = reinterpret_cast<uint4 *>(base + 32 * c);
#pragma unroll
                for (int k = 0; k < 4; ++k) dst[k] = make_uint4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
            }
            fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bar[U_D_FREE + db]));
        }
    }

    __syncthreads();
    if (warp == 9) {
        if (!mbar_wait_cycles(smem_u32(&bar[U_FINAL]), 0, kWaitCycles)) set_dev_err(a.dev_err, MLA_DEVERR_TIMEOUT);
        fence_after_sync();
        tmem_dealloc(tmem, 512);
    }
}

// ===========================================================================
// 2. attention
// ===========================================================================
// paired f32 arithmetic (two IEEE operations per instruction) and a three-input max
__device__ __forceinline__ uint64_t pk2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ uint64_t pk2u(uint32_t lo, uint32_t hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
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
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
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

constexpr int AT_BM = 128;                    // query tokens per CTA
constexpr int AT_BN = 64;                     // keys per tile
constexpr int AT_ST = 4;                      // K/V ring stages
constexpr int AT_NT = 192;
constexpr int kKSlice = AT_BN * 128;          // 64 keys x 64 dims bf16: 8 KB
constexpr int kStage = 5 * kKSlice;           // no-RoPE 0, no-RoPE 1, RoPE, V 0, V 1
constexpr int kOffKV = 0;                     // the query tile lives in TMEM
constexpr int kOffP = kOffKV + AT_ST * kStage;
constexpr int kPBuf = AT_BM * AT_BN * 2;      // 16 KB
constexpr int kAtSmem = 1024 + kOffP + 2 * kPBuf;
constexpr float kRescale = 8.f;               // log2 units
constexpr uint32_t kColQ = 256;               // TMEM: S buffers 0..127, O 128..255, Q 256..351
constexpr uint32_t kAtTmemCols = 512;         // allocated and released as one (a power of two >= 352)
static_assert(kAtSmem <= 232448 - 256, "shared memory");

enum AtBar { A_Q_F16 = 0, A_KV_FULL, A_KV_EMPTY = A_KV_FULL + AT_ST, A_S_FULL = A_KV_EMPTY + AT_ST,
             A_S_FREE = A_S_FULL + 2, A_P_FULL = A_S_FREE + 2, A_PV_DONE = A_P_FULL + 2, A_FINAL = A_PV_DONE + 2,
             A_NBAR };

__global__ void __launch_bounds__(AT_NT, 1)
    attn_kernel(const MhaArgs a, const int4 *__restrict__ work, const __grid_constant__ CUtensorMap tmap_kn, const __grid_constant__ CUtensorMap tmap_kr,
                const __grid_constant__ CUtensorMap tmap_v) {
    extern __shared__ __align__(1024) uint8_t dsm[];
    __shared__ uint64_t bar[A_NBAR];
    __shared__ uint32_t tmem_slot;
    const uint32_t raw = smem_u32(dsm);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    uint8_t *sbase = dsm + pad;
    const uint32_t sbase_a = raw + pad;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // work item: {b, first new token in the sequence, its global index, valid rows},
    //            {prefix, key-row base, key tiles, -}; the grid runs head-major, so
    //            the CTAs in flight share one head's keys and values in L2
    const int n_items = static_cast<int>(gridDim.x) / a.H;
    const int item = blockIdx.x % n_items, h = blockIdx.x / n_items;
    const int4 w0 = work[2 * item], w1 = work[2 * item + 1];
    const int i0 = w0.y, n_valid = w0.w, P = w1.x, n_tiles = w1.z;
    const int64_t t0 = w0.z, kb = w1.y;

    if (tid == 0) {
        for (int i = 0; i < A_NBAR; ++i) {
            uint32_t cnt = 1;
            if ((i >= A_S_FREE && i < A_S_FREE + 2) || (i >= A_P_FULL && i < A_P_FULL + 2) || i == A_Q_F16) cnt = 4;
            mbar_init(smem_u32(&bar[i]), cnt);
        }
        mbar_fence_init();
    }
    if (warp == 5) {
        tmem_alloc(smem_u32(&tmem_slot), kAtTmemCols);
        tmem_relinquish();
    }
    if (warp == 4 && lane == 0) {
        tma_prefetch_desc(&tmap_kn);
        tma_prefetch_desc(&tmap_kr);
        tma_prefetch_desc(&tmap_v);
    }
    __syncthreads();
    fence_after_sync();
    const uint32_t tmem = tmem_slot;

    if (warp == 4) {
        // =================== TMA producer ===================
        if (lane == 0) {
            const int krow0 = static_cast<int>(static_cast<int64_t>(h) * a.R + kb);
            int t = 0;
            for (; t < n_tiles; ++t) {
                const int st = t % AT_ST;
                if (t >= AT_ST && !wait_bar(&bar[A_KV_EMPTY + st], ((t / AT_ST) - 1) & 1, a.dev_err)) break;
                const uint32_t sb = sbase_a + kOffKV + st * kStage, fb = smem_u32(&bar[A_KV_FULL + st]);
                mbar_expect_tx(fb, kStage);
                tma_load_2d(sb, &tmap_kn, 0, krow0 + AT_BN * t, fb);
                tma_load_2d(sb + kKSlice, &tmap_kn, 64, krow0 + AT_BN * t, fb);
                tma_load_2d(sb + 2 * kKSlice, &tmap_kr, 0, static_cast<int>(kb) + AT_BN * t, fb);
                tma_load_2d(sb + 3 * kKSlice, &tmap_v, 0, krow0 + AT_BN * t, fb);
                tma_load_2d(sb + 4 * kKSlice, &tmap_v, 64, krow0 + AT_BN * t, fb);
            }
            // drain: the last load of every stage has landed
            for (int j = (t > AT_ST ? t - AT_ST : 0); j < t; ++j)
                if (!mbar_wait_cycles(smem_u32(&bar[A_KV_FULL + j % AT_ST]), (j / AT_ST) & 1, kWaitCycles))
                    set_dev_err(a.dev_err, MLA_DEVERR_TIMEOUT);
        }
    } else if (warp == 5) {
        // =================== MMA issuer: QK(t+1) before PV(t) ===================
        if (lane == 0) {
            const uint32_t id_qk = idesc_f16(AT_BM, AT_BN, false, false, false, false);
            const uint32_t id_pv = idesc_f16(AT_BM, 128, false, false, false, true);
            const uint64_t dk0 = sdesc(sbase_a + kOffKV, 16, 1024, kSw128);
            const uint64_t dv0 = sdesc(sbase_a + kOffKV + 3 * kKSlice, kKSlice, 1024, kSw128);
            const uint64_t dp0 = sdesc(sbase_a + kOffP, 128, 1024, kSwNone);
            auto qk = [&](int t) -> bool {
                const int st = t % AT_ST, sb = t & 1;
                if (!wait_bar(&bar[A_KV_FULL + st], (t / AT_ST) & 1, a.dev_err)) return false;
                if (t >= 2 && !wait_bar(&bar[A_S_FREE + sb], ((t >> 1) - 1) & 1, a.dev_err)) return false;
                fence_after_sync();
                const uint32_t d = tmem + static_cast<uint32_t>(AT_BN * sb);
#pragma unroll
                for (int s = 0; s < 3; ++s) {
                    const uint64_t db = dk0 + static_cast<uint64_t>((st * kStage + s * kKSlice) >> 4);
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks)
                        mma_f16_ts_w(d, tmem + kColQ + 32u * s + 8u * ks, db + 2 * ks, id_qk, (s | ks) ? 1u : 0u, 1u);
                }
                mma_commit(smem_u32(&bar[A_S_FULL + sb]));
                return true;
            };
            auto pv = [&](int t) -> bool {
                const int st = t % AT_ST, pb = t & 1;
                if (!wait_bar(&bar[A_P_FULL + pb], (t >> 1) & 1, a.dev_err)) return false;
                fence_after_sync();
                const uint64_t da = dp0 + static_cast<uint64_t>((pb * kPBuf) >> 4);
                const uint64_t dv = dv0 + static_cast<uint64_t>((st * kStage) >> 4);
#pragma unroll
                for (int ks = 0; ks < AT_BN / 16; ++ks)
                    mma_f16_ss_w(tmem + 128u, da + 16 * ks, dv + 128 * ks, id_pv, (t | ks) ? 1u : 0u, 1u);
                mma_commit(smem_u32(&bar[A_KV_EMPTY + st]));
                mma_commit(smem_u32(&bar[A_PV_DONE + pb]));
                return true;
            };
            bool ok = n_tiles > 0 && wait_bar(&bar[A_Q_F16], 0, a.dev_err);
            if (ok) ok = qk(0);
            for (int t = 0; t < n_tiles && ok; ++t) {
                if (t + 1 < n_tiles && !(ok = qk(t + 1))) break;
                ok = pv(t);
            }
            mma_commit(smem_u32(&bar[A_FINAL]));
        }
    } else {
        // =================== softmax + epilogue: thread = query row ===================
        const int r = 32 * warp + lane;
        const int64_t pos = static_cast<int64_t>(P) + i0 + r;      // the row's position in its sequence
        const uint32_t lane_addr = static_cast<uint32_t>(32 * warp) << 16;
        const uint64_t scale2 = pk2(a.sm_scale_log2, a.sm_scale_log2);
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        uint8_t *prow = sbase + kOffP + (r >> 3) * 1024 + (r & 7) * 16;
        // the query row, converted to f16, into TMEM (lane = row, column c = dims
        // 2c, 2c+1): the QK MMAs read it from there. All 24 loads of the row go out
        // at once (one memory round trip); then each thread asks L2 for its row of the
        // CTA expected to follow on this SM, so that one finds its queries in L2.
        ok = n_tiles > 0;
        if (ok) {
            const bool have = t0 + r < a.total_q;
            const uint4 *src = reinterpret_cast<const uint4 *>(a.q + ((have ? t0 + r : 0) * a.H + h) * 192);
            uint4 xq[24];
#pragma unroll
            for (int c = 0; c < 24; ++c) xq[c] = have ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
            const int64_t nxt = static_cast<int64_t>(blockIdx.x) + a.ahead;
            if (a.ahead > 0 && nxt < gridDim.x) {
                const int item_n = static_cast<int>(nxt % n_items), h_n = static_cast<int>(nxt / n_items);
                const int4 wn = work[2 * item_n];
                if (r < wn.w && static_cast<int64_t>(wn.z) + r < a.total_q) {
                    const char *row = reinterpret_cast<const char *>(a.q + ((wn.z + r) * static_cast<int64_t>(a.H) + h_n) * 192);
#pragma unroll
                    for (int k = 0; k < 3; ++k) asm volatile("prefetch.global.L2 [%0];\n" ::"l"(row + 128 * k));
                }
            }
#pragma unroll
            for (int g = 0; g < 3; ++g) {                 // 64 dims = 32 TMEM columns per group
                uint32_t o[32];
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint4 x = xq[8 * g + c];
                    const uint32_t wv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&wv[k]));
                        o[4 * c + k] = pack_half2(f.x, f.y);
                    }
                }
                tmem_st32(tmem + lane_addr + kColQ + 32u * g, o);
            }
            tmem_st_wait();
            fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bar[A_Q_F16]));
        }
        for (int t = 0; t < n_tiles && ok; ++t) {
            const int sb = t & 1;
            ok = __all_sync(0xffffffffu, wait_bar(&bar[A_S_FULL + sb], (t >> 1) & 1, a.dev_err));
            if (!ok) break;
            fence_after_sync();
            uint32_t sv[64];
            tmem_ld32(tmem + lane_addr + static_cast<uint32_t>(AT_BN * sb), *reinterpret_cast<uint32_t(*)[32]>(sv));
            tmem_ld32(tmem + lane_addr + static_cast<uint32_t>(AT_BN * sb + 32),
                      *reinterpret_cast<uint32_t(*)[32]>(sv + 32));
            tmem_ld_wait();
            fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bar[A_S_FREE + sb]));
            // logits in log2 units, two per paired multiply; keys past the row's position
            // are masked (only tiles that reach past it need the compare)
            const int64_t k0 = static_cast<int64_t>(AT_BN) * t;
            uint64_t u2[32];
            float mx = -INFINITY;
#pragma unroll
            for (int k = 0; k < 32; ++k) u2[k] = mul2(pk2u(sv[2 * k], sv[2 * k + 1]), scale2);
            if (k0 + AT_BN - 1 > pos) {
#pragma unroll
                for (int k = 0; k < 32; ++k) {
                    float2 f = upk2(u2[k]);
                    if (k0 + 2 * k > pos) f.x = -INFINITY;
                    if (k0 + 2 * k + 1 > pos) f.y = -INFINITY;
                    u2[k] = pk2(f.x, f.y);
                }
            }
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                const float2 f = upk2(u2[k]);
                mx = max3(mx, f.x, f.y);
            }
            if (t == 0) {
                m = mx;
            } else {
                const bool need = mx > m + kRescale;
                if (__any_sync(0xffffffffu, need)) {
                    // O is rescaled in TMEM once PV(t-1) has finished with it
                    ok = __all_sync(0xffffffffu, wait_bar(&bar[A_PV_DONE + ((t - 1) & 1)], ((t - 1) >> 1) & 1, a.dev_err));
                    if (!ok) break;
                    fence_after_sync();
                    const float f = need ? fast_exp2(m - mx) : 1.f;
                    if (need) {
                        l *= f;
                        m = mx;
                    }
#pragma unroll 1
                    for (int c = 0; c < 4; ++c) {
                        uint32_t o[32];
                        tmem_ld32(tmem + lane_addr + 128u + 32u * c, o);
                        tmem_ld_wait();
#pragma unroll
                        for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * f);
                        tmem_st32(tmem + lane_addr + 128u + 32u * c, o);
                    }
                    tmem_st_wait();
                }
            }
            // P = 2^(u - m): fp32 into l, f16 into the P buffer of this tile
            uint32_t pw[32];
            uint64_t ls2 = 0;
            const uint64_t m2 = pk2(m, m);
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                const float2 d = upk2(sub2(u2[k], m2));
                const float p0 = fast_exp2(d.x), p1 = fast_exp2(d.y);
                const uint64_t pp = pk2(p0, p1);
                ls2 = k == 0 ? pp : add2(ls2, pp);
                pw[k] = pack_half2(p0, p1);
            }
            {
                const float2 f = upk2(ls2);
                l += f.x + f.y;
            }
            if (t >= 2) {       // PV(t-2) has read the buffer
                ok = __all_sync(0xffffffffu, wait_bar(&bar[A_PV_DONE + sb], ((t >> 1) - 1) & 1, a.dev_err));
                if (!ok) break;
            }
            uint8_t *pdst = prow + sb * kPBuf;
#pragma unroll
            for (int c = 0; c < 8; ++c)
                *reinterpret_cast<uint4 *>(pdst + c * 128) = make_uint4(pw[4 * c], pw[4 * c + 1], pw[4 * c + 2], pw[4 * c + 3]);
            fence_proxy_async();
            fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&bar[A_P_FULL + sb]));
        }
        // ----- epilogue -----
        if (ok && n_tiles > 0) {
            const int tl = n_tiles - 1;
            ok = __all_sync(0xffffffffu, wait_bar(&bar[A_PV_DONE + (tl & 1)], (tl >> 1) & 1, a.dev_err));
        }
        if (ok && n_tiles > 0) {
            fence_after_sync();
            const float inv = 1.f / l;
            const bool live = r < n_valid;
            __nv_bfloat16 *orow = a.out + ((t0 + r) * a.H + h) * kDvh;
            uint32_t ob[4][32];   // the row's 128 columns of O in one round trip
#pragma unroll
            for (int c = 0; c < 4; ++c) tmem_ld32(tmem + lane_addr + 128u + 32u * c, ob[c]);
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const uint32_t *o = ob[c];
                if (live) {
                    uint32_t w[16];
#pragma unroll
                    for (int k = 0; k < 16; ++k)
                        w[k] = pack_bf162(__uint_as_float(o[2 * k]) * inv, __uint_as_float(o[2 * k + 1]) * inv);
                    uint4 *dst = reinterpret_cast<uint4 *>(orow + 32 * c);
#pragma unroll
                    for (int k = 0; k < 4; ++k) dst[k] = make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
                }
            }
            if (live && a.lse) a.lse[(t0 + r) * a.H + h] = (m + log2f(l)) * kLn2;
        }
    }

    __syncthreads();
    if (warp == 5) {
        if (!mbar_wait_cycles(smem_u32(&bar[A_FINAL]), 0, kWaitCycles)) set_dev_err(a.dev_err, MLA_DEVERR_TIMEOUT);
        fence_after_sync();
        tmem_dealloc(tmem, kAtTmemCols);
    }
}

}  // namespace mha

cudaError_t launch_mha_up(const MhaArgs &a, const int4 *work, int n_work, const CUtensorMap &tmap_w, cudaStream_t st) {
    cudaError_t e = cudaFuncSetAttribute(mha::up_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, mha::kUpSmem);
    if (e != cudaSuccess) return e;
    const int64_t n_cta = static_cast<int64_t>(n_work) * (a.H / a.up_heads);
    if (n_cta > 0) mha::up_kernel<<<static_cast<unsigned>(n_cta), mha::UP_NT, mha::kUpSmem, st>>>(a, work, tmap_w);
    return cudaGetLastError();
}

cudaError_t launch_mha_attn(const MhaArgs &a, const int4 *work, int n_work, const CUtensorMap &tmap_kn, const CUtensorMap &tmap_kr, const CUtensorMap &tmap_v,
                            cudaStream_t st) {
    cudaError_t e = cudaFuncSetAttribute(mha::attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, mha::kAtSmem);
    if (e != cudaSuccess) return e;
    // one CTA per SM at a time (all of TMEM): the CTA that follows on an SM is about
    // an SM count further on in the grid
    int dev = 0, n_sm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    MhaArgs b = a;
    b.ahead = n_sm;
    const int64_t n_cta = static_cast<int64_t>(n_work) * a.H;
    if (n_cta > 0)
        mha::attn_kernel<<<static_cast<unsigned>(n_cta), mha::AT_NT, mha::kAtSmem, st>>>(b, work, tmap_kn,
                                                                                      tmap_kr, tmap_v);
    return cudaGetLastError();
}

}  // namespace mla

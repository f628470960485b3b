// Indexer scores on the 5th-generation tensor cores (tcgen05 kind::f8f6f4).
//
// score(t,s) = sigmaI_s * sum_h w[t,h] * max(0, q_{t,h} . k_s),   s <= position(t)
// (GLM-5.3 Teil 2, section "Warum nicht TP oder DP?": the indexer scores every
// earlier token to pick 2,048; footnote 3: an indexer key is 128 FP8 values
// plus a 4-byte scale.)
//
// One CTA scores 3 query tokens (x 64 heads) against a chunk of keys (2,048 to
// 32,768, chosen by the host), 128 keys at a time:
//
//   D[key][64 j + h] = k_key . q_{t_j,h}    tcgen05.mma e4m3 x e4m3 -> f32,
//                                           M = 128 keys, N = 192 = 3 tokens x 64
//                                           heads, K = 128 (4 steps of 32)
//
// so TMEM lane = key and each epilogue thread owns one key: the head sum
// sum_h w[t,h] max(0, D) is a per-thread loop over its own columns, with no
// cross-thread reduction. The products of the codes are exact in f32 and the
// sums are exact while they stay below 2^24 in units of the smallest product,
// which the integer-valued keys and queries of the indexer guarantee.
//
// Keys arrive by TMA: a 128-key tile starts at a multiple of 128 and so lies in
// one 256-token page, i.e. 128 contiguous rows of the paged key cache, copied
// with the 128-byte swizzle the MMA's K-major operand layout expects. The 3
// tokens' queries (192 rows) are one more TMA copy.
//
// Warps: 0-11 epilogue (warp w reads TMEM lane quadrant w%4 = keys 32(w%4)..+31
// of token w/4), 12 TMA producer, 13 MMA issue + TMEM owner. Key tiles go
// through a 6-stage ring; the accumulator is double-buffered in TMEM (2 x 192
// columns) so the MMA of tile i+1 overlaps the epilogue of tile i. Fourteen
// warps leave each thread 128 registers, enough for its token's 64 head weights
// (as 32 register pairs, loaded once), so the head sum reads no memory: per
// tile a thread takes its key's 64 values in four chunks of 16, the load of the
// next chunk in flight while one is reduced, and runs paired f32 FMAs
// (fma.rn.f32x2: two IEEE fmas, so the same result as scalar ones) with four
// independent accumulator pairs.
// Every wait is bounded and reports MLA_DEVERR_TIMEOUT.
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "tc.cuh"

namespace mla {
namespace idxtc {

using namespace tc;

constexpr int TOK = kIdxTokensPerCta;   // 3 query tokens per CTA
constexpr int KT = 128;                 // keys per tile
constexpr int STAGES = 6;
constexpr int kEpiWarps = 4 * TOK;      // tokens x 4 TMEM lane quadrants
constexpr int kDCols = 256;             // TMEM columns per accumulator buffer (TOK x 64 used)
constexpr int NT = 32 * (kEpiWarps + 2);
constexpr int kProducerWarp = kEpiWarps, kIssuerWarp = kEpiWarps + 1;
constexpr int kQBytes = TOK * kHidx * kDidx;       // 24 KB
constexpr int kTileBytes = KT * kDidx;             // 16 KB
constexpr int kDynSmem = 1024 + kQBytes + STAGES * kTileBytes;
constexpr long long kWaitCycles = 200000000LL;
static_assert(kIdxKeyChunkMin % KT == 0 && kPage % KT == 0, "key tiles must not straddle pages or chunks");

enum Bar {
    B_Q_FULL = 0,
    B_K_FULL = 1,                       // [STAGES]  TMA -> issuer
    B_K_EMPTY = B_K_FULL + STAGES,      // [STAGES]  issuer (commit) -> producer
    B_D_FULL = B_K_EMPTY + STAGES,      // [2]       issuer (commit) -> epilogue
    B_D_EMPTY = B_D_FULL + 2,           // [2]       epilogue (16 warps) -> issuer
    B_FINAL = B_D_EMPTY + 2,
    NBAR
};

struct Shared {
    uint64_t bar[NBAR];
    uint32_t tmem_base;
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
__device__ __forceinline__ float relu_bits(uint32_t x) { return fmaxf(__uint_as_float(x), 0.f); }

__device__ __forceinline__ bool wait_bar(Shared &sh, int32_t *dev_err, int b, uint32_t parity) {
    if (mbar_wait_cycles(smem_u32(&sh.bar[b]), parity, kWaitCycles)) return true;
    set_dev_err(dev_err, MLA_DEVERR_TIMEOUT);
    return false;
}

__global__ void __launch_bounds__(NT, 1)
    score_kernel(const IndexerArgs a, const int4 *__restrict__ work, const __grid_constant__ CUtensorMap tmap_k,
                 const __grid_constant__ CUtensorMap tmap_q) {
    extern __shared__ __align__(1024) uint8_t dsm[];
    __shared__ Shared sh;
    const uint32_t raw = smem_u32(dsm);
    const uint32_t pad = (1024u - (raw & 1023u)) & 1023u;
    const uint32_t sq = raw + pad, sk = sq + kQBytes;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    const int4 it = work[blockIdx.x];
    const int b = it.x, i0 = it.y, ntok = it.z;
    const int q0 = __ldg(a.cu_seqlens + b), P = __ldg(a.prefix_lens + b);
    const int32_t *bt = a.block_table + static_cast<int64_t>(b) * a.max_blocks;
    const int k_lo = it.w * a.key_chunk;
    const int k_hi = min(k_lo + a.key_chunk, P + i0 + ntok);        // exclusive
    const int n_tiles = (k_hi - k_lo + KT - 1) / KT;

    if (tid == 0) {
        for (int i = 0; i < NBAR; ++i) mbar_init(smem_u32(&sh.bar[i]), (i == B_D_EMPTY || i == B_D_EMPTY + 1) ? kEpiWarps : 1);
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

    if (warp == kProducerWarp) {
        // =================== TMA producer ===================
        if (lane == 0) {
            tma_prefetch_desc(&tmap_k);
            tma_prefetch_desc(&tmap_q);
            mbar_expect_tx(smem_u32(&sh.bar[B_Q_FULL]), kQBytes);
            tma_load_2d(sq, &tmap_q, 0, (q0 + i0) * kHidx, smem_u32(&sh.bar[B_Q_FULL]));
            for (int i = 0; i < n_tiles; ++i) {
                const int s = i % STAGES;
                if (i >= STAGES && !wait_bar(sh, a.dev_err, B_K_EMPTY + s, ((i / STAGES) - 1) & 1)) break;
                const int pos0 = k_lo + i * KT;
                const int page = pos0 / kPage;
                int blk = page < a.max_blocks ? __ldg(bt + page) : -1;
                if (blk < 0 || blk >= a.num_blocks) {   // reported; the epilogue masks these keys
                    set_dev_err(a.dev_err, MLA_DEVERR_BAD_PAGE);
                    blk = 0;
                }
                mbar_expect_tx(smem_u32(&sh.bar[B_K_FULL + s]), kTileBytes);
                tma_load_2d(sk + s * kTileBytes, &tmap_k, 0, blk * kPage + pos0 % kPage, smem_u32(&sh.bar[B_K_FULL + s]));
            }
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
        // =================== epilogue (warps 0-15) ===================
        const int quad = warp & 3, j = warp >> 2;                     // keys 32 quad.., token j
        const uint32_t lane_addr = static_cast<uint32_t>(32 * quad) << 16;
        const int kk = 32 * quad + lane;                              // key within the tile
        // the token's head weights, as pairs, for every tile of the chunk
        const float4 *wg = reinterpret_cast<const float4 *>(a.w + static_cast<int64_t>(q0 + i0 + min(j, ntok - 1)) *
                                                            a.w_stride);
        uint64_t wp[kHidx / 2];
#pragma unroll
        for (int h4 = 0; h4 < kHidx / 4; ++h4) {
            const float4 w4 = __ldg(wg + h4);
            wp[2 * h4] = pack2(w4.x, w4.y);
            wp[2 * h4 + 1] = pack2(w4.z, w4.w);
        }
        float *out_row = a.scores + static_cast<int64_t>(q0 + i0 + j) * a.score_stride;
        const int pos_hi = min(k_hi, P + i0 + j + 1);                 // causal bound of token j (exclusive)
        // The key scales go through a register pipeline: the page of tile i+3 and
        // the scale of tile i+2 are fetched while tile i is reduced, so the two
        // dependent global loads never sit on a tile's critical path. A tile lies
        // in one page; blk < 0 marks a bad page or a tile past the chunk.
        auto page_blk = [&](int i) -> int {
            if (i >= n_tiles) return -1;
            const int page = (k_lo + i * KT) / kPage;
            const int blk = page < a.max_blocks ? __ldg(bt + page) : -1;
            return blk;
        };
        auto key_ok = [&](int blk) { return blk >= 0 && blk < a.num_blocks; };
        auto key_sig = [&](int i, int blk) -> float {
            const int pos = k_lo + i * KT + kk;
            if (!key_ok(blk) || pos >= k_hi) return 0.f;
            return __ldg(a.ki_scale + static_cast<int64_t>(blk) * kPage + pos % kPage);
        };
        int blk0 = page_blk(0), blk1 = page_blk(1), blk2 = page_blk(2);
        float sig0 = key_sig(0, blk0), sig1 = key_sig(1, blk1);
        int blk3 = page_blk(3);
        for (int i = 0; i < n_tiles; ++i) {
            const int db = i & 1;
            const int pos = k_lo + i * KT + kk;
            const float sig = sig0;
            const bool ok_key = key_ok(blk0);
            sig0 = sig1;
            sig1 = key_sig(i + 2, blk2);
            blk0 = blk1;
            blk1 = blk2;
            blk2 = blk3;
            blk3 = page_blk(i + 4);
            if (!wait_bar(sh, a.dev_err, B_D_FULL + db, (i >> 1) & 1)) break;
            fence_after_sync();
            uint64_t acc[4] = {0, 0, 0, 0};
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
                for (int h4 = 0; h4 < 4; ++h4) {
                    const uint32_t *x = d[c & 1] + 4 * h4;
                    const int w2 = 8 * c + 2 * h4;
                    ffma2(acc[2 * (h4 & 1)], wp[w2], pack2(relu_bits(x[0]), relu_bits(x[1])));
                    ffma2(acc[2 * (h4 & 1) + 1], wp[w2 + 1], pack2(relu_bits(x[2]), relu_bits(x[3])));
                }
                if (c < 3) tmem_ld_wait();
                if (c == 2) {      // every column read: the buffer goes back to the MMA
                    fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(smem_u32(&sh.bar[B_D_EMPTY + db]));
                }
            }
            const float sc = (sum2(acc[0]) + sum2(acc[1])) + (sum2(acc[2]) + sum2(acc[3]));
            if (j < ntok && pos < pos_hi) out_row[pos] = ok_key ? sig * sc : -INFINITY;
        }
    }

    // ----- teardown -----
    __syncthreads();
    if (warp == kIssuerWarp) {
        if (!mbar_wait_cycles(smem_u32(&sh.bar[B_FINAL]), 0, kWaitCycles)) set_dev_err(a.dev_err, MLA_DEVERR_TIMEOUT);
        fence_after_sync();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace idxtc

cudaError_t launch_indexer_scores_tc(const IndexerArgs &a, const int4 *work, int n_work, const CUtensorMap &tmap_k,
                                     const CUtensorMap &tmap_q, cudaStream_t st) {
    cudaError_t e = cudaFuncSetAttribute(idxtc::score_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         idxtc::kDynSmem);
    if (e != cudaSuccess) return e;
    if (n_work > 0) idxtc::score_kernel<<<n_work, idxtc::NT, idxtc::kDynSmem, st>>>(a, work, tmap_k, tmap_q);
    return cudaGetLastError();
}

}  // namespace mla

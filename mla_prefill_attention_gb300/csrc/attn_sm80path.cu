// MLA prefill attention, first correct path: warp-level mma.sync (f16 in,
// fp32 accumulate) on sm_103a. One CTA computes a tile of 64 query rows
// (row = (token, head) of one sequence) against the latent rows of the paged
// e4m3 cache, 64 keys at a time:
//
//   S    = Q K^T over 576 dims (latent 512 + RoPE 64)         [64 x 64]
//   u    = S * sigma_key * rowscale + log2(sigma_key)          (log2 domain)
//   P'   = 2^(u - M),  M = running max of u;  l += P' / sigma_key
//   O   += P' V over 512 dims (V = first 512 dims of the same K tile)
//   out  = O / l,  lse = ln2 * (M + log2 l)
//
// Because P' = 2^(logit*log2e - M) * sigma_key, the per-token cache scale
// is folded into the exponent (no pass over K or V applies it) and P' <= 1.
// The query row is prescaled by a power of two so that its largest entry is
// in [1, 2); e4m3 codes convert to f16 exactly, so the only roundings before
// the fp32 accumulators are that of bf16 -> f16 for entries far below the row
// maximum and that of P' to f16.
//
// Warp w of 8: row group rg = w & 3 (16 rows), half kh = w >> 2. For QK the
// halves split the 64 keys (32 each); for PV they split the 512 value dims
// (256 each). The two warps of a row group exchange row maxima and P' through
// shared memory behind a 64-thread named barrier.
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"

namespace mla {
namespace sm80path {

constexpr int BM = 64, BN = 64, NT = 256;
constexpr int kRowBytes = kDqk * 2;                  // 1152 B per f16 row
constexpr int kSQ = BM * kRowBytes;                  // 73728
constexpr int kSK = BN * kRowBytes;                  // 73728
constexpr int kSP = BM * BN * 2;                     // 8192
constexpr int kSK8 = BN * kDqk;                      // 36864
constexpr int kChunks8 = kDqk / 16;                  // 36 16-byte chunks per fp8 row

struct Smem {
    alignas(128) uint8_t q[kSQ];
    alignas(128) uint8_t k[kSK];
    alignas(128) uint8_t p[kSP];
    alignas(128) uint8_t k8[kSK8];
    int64_t krow[2][BN];       // cache row (page*256+slot) per key, -1 = masked
    int32_t kpos[2][BN];       // key position, -1 = masked
    float ksig[2][BN];         // sigma (per-token cache scale)
    float klsig[2][BN];        // log2(sigma)
    float kisig[2][BN];        // 1/sigma
    float rowscale[BM];        // sm_scale*log2e / (query prescale)
    int32_t rowlimit[BM];      // last visible position (dense), -1 = row invalid
    float redmax[2][BM];
    float redsum[2][BM];
};

__device__ __forceinline__ uint32_t sw1152(uint32_t base, int row, int chunk) {
    return base + row * kRowBytes + ((chunk ^ (row & 7)) << 4);
}
__device__ __forceinline__ uint32_t sw128(uint32_t base, int row, int chunk) {
    return base + row * 128 + ((chunk ^ (row & 7)) << 4);
}
__device__ __forceinline__ void pair_sync(int rg) {
    asm volatile("bar.sync %0, 64;\n" ::"r"(rg + 1));
}

// Load 64 query rows (global rows grow0 + r, r < nvalid) into smem as f16,
// each row prescaled by 2^k so that max|q| lands in [1, 2).
__device__ void load_q(Smem &sm, const __nv_bfloat16 *q, int64_t grow0, int nvalid, float sm_scale_log2) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t sq = smem_u32(sm.q);
    for (int r = warp; r < BM; r += NT / 32) {
        uint4 v[3];
        float mx = 0.f;
        const bool ok = r < nvalid;
        const uint4 *src = reinterpret_cast<const uint4 *>(q + (grow0 + r) * kDqk);
#pragma unroll
        for (int i = 0; i < 3; ++i) {
            const int c = lane + 32 * i;
            v[i] = make_uint4(0, 0, 0, 0);
            if (ok && c < kDqk / 8) v[i] = __ldg(src + c);
            const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&v[i]);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float2 f = __bfloat1622float2(h[j]);
                mx = fmaxf(mx, fmaxf(fabsf(f.x), fabsf(f.y)));
            }
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        int e = 0;
        if (mx > 0.f) frexpf(mx, &e);
        const float scale = mx > 0.f ? ldexpf(1.f, 1 - e) : 1.f;
#pragma unroll
        for (int i = 0; i < 3; ++i) {
            const int c = lane + 32 * i;
            if (c >= kDqk / 8) continue;
            const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&v[i]);
            uint4 o;
            uint32_t *ow = reinterpret_cast<uint32_t *>(&o);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float2 f = __bfloat1622float2(h[j]);
                ow[j] = pack_half2(f.x * scale, f.y * scale);
            }
            asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(sw1152(sq, r, c)), "r"(o.x), "r"(o.y),
                         "r"(o.z), "r"(o.w));
        }
        if (lane == 0) sm.rowscale[r] = sm_scale_log2 / scale;
    }
}

// Key metadata of one tile (threads 0..63): position -> cache row, scale.
template <bool kSparse>
__device__ void key_meta(Smem &sm, int buf, const AttnArgs &a, const int32_t *bt, int key0, int key_last,
                         const int32_t *idx_row, int32_t qpos_limit) {
    const int k = threadIdx.x;
    if (k >= BN) return;
    int64_t pos;
    if (kSparse) {
        const int j = key0 + k;
        pos = j < a.topk ? static_cast<int64_t>(__ldg(idx_row + j)) : -1;
        if (pos < -1 || pos > qpos_limit) {
            set_dev_err(a.dev_err, MLA_DEVERR_BAD_INDEX);
            pos = -1;
        }
    } else {
        pos = key0 + k;
        if (pos > key_last) pos = -1;
    }
    int64_t row = pos >= 0 ? cache_row(bt, a.max_blocks, a.num_blocks, pos, a.dev_err) : -1;
    if (row < 0) pos = -1;
    float sig = row >= 0 ? __ldg(a.kv_scale + row) : 1.f;
    sm.krow[buf][k] = row;
    sm.kpos[buf][k] = static_cast<int32_t>(pos);
    sm.ksig[buf][k] = sig;
    sm.klsig[buf][k] = __log2f(sig);
    sm.kisig[buf][k] = 1.f / sig;
}

__device__ __forceinline__ void issue_k8(Smem &sm, int buf, const uint8_t *kv) {
    const uint32_t s8 = smem_u32(sm.k8);
#pragma unroll
    for (int i = 0; i < (BN * kChunks8) / NT; ++i) {
        const int c = threadIdx.x + NT * i;
        const int key = c / kChunks8, part = c % kChunks8;
        const int64_t row = sm.krow[buf][key];
        const uint8_t *src = kv + (row >= 0 ? row : 0) * kDqk + part * 16;
        cp_async16(s8 + key * kDqk + part * 16, src, row >= 0 ? 16 : 0);
    }
    cp_async_commit();
}

__device__ __forceinline__ void convert_k(Smem &sm) {
    const uint32_t sk = smem_u32(sm.k);
#pragma unroll
    for (int i = 0; i < (BN * kChunks8) / NT; ++i) {
        const int c = threadIdx.x + NT * i;
        const int key = c / kChunks8, part = c % kChunks8;
        const uint4 v = *reinterpret_cast<const uint4 *>(sm.k8 + key * kDqk + part * 16);
        uint32_t h[8];
        e4m3x4_to_f16x4(v.x, h[0], h[1]);
        e4m3x4_to_f16x4(v.y, h[2], h[3]);
        e4m3x4_to_f16x4(v.z, h[4], h[5]);
        e4m3x4_to_f16x4(v.w, h[6], h[7]);
        asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(sw1152(sk, key, 2 * part)), "r"(h[0]),
                     "r"(h[1]), "r"(h[2]), "r"(h[3]));
        asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(sw1152(sk, key, 2 * part + 1)), "r"(h[4]),
                     "r"(h[5]), "r"(h[6]), "r"(h[7]));
    }
}

// One 64-row tile over n_tiles key tiles. Rows with rowlimit < 0 are invalid.
template <bool kSparse>
__device__ void attend_tile(Smem &sm, const AttnArgs &a, const int32_t *bt, int64_t grow0, int nvalid,
                            int key_last, int n_ktiles, const int32_t *idx_row, int32_t qpos_limit) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rg = warp & 3, kh = warp >> 2, g = lane >> 2, t4 = lane & 3;
    const int r0 = 16 * rg + g, r1 = r0 + 8;
    const uint32_t sq = smem_u32(sm.q), sk = smem_u32(sm.k), sp = smem_u32(sm.p);

    load_q(sm, a.q, grow0, nvalid, a.sm_scale_log2);
    key_meta<kSparse>(sm, 0, a, bt, 0, key_last, idx_row, qpos_limit);
    __syncthreads();
    issue_k8(sm, 0, a.kv);

    float o[32][4];
#pragma unroll
    for (int i = 0; i < 32; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    const float rs0 = sm.rowscale[r0], rs1 = sm.rowscale[r1];
    const int lim0 = sm.rowlimit[r0], lim1 = sm.rowlimit[r1];

    for (int j = 0; j < n_ktiles; ++j) {
        const int buf = j & 1;
        cp_async_wait<0>();
        __syncthreads();
        convert_k(sm);
        if (j + 1 < n_ktiles) key_meta<kSparse>(sm, buf ^ 1, a, bt, (j + 1) * BN, key_last, idx_row, qpos_limit);
        __syncthreads();
        if (j + 1 < n_ktiles) issue_k8(sm, buf ^ 1, a.kv);

        // ---- S = Q K^T for rows 16rg..+16, keys 32kh..+32 ----
        float s[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll 4
        for (int ks = 0; ks < kDqk / 16; ++ks) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4(sw1152(sq, 16 * rg + (lane & 15), 2 * ks + (lane >> 4)), a0, a1, a2, a3);
#pragma unroll
            for (int np = 0; np < 2; ++np) {
                const int key = 32 * kh + 16 * np + (lane & 7) + ((lane >> 4) << 3);
                uint32_t b0, b1, b2, b3;
                ldsm_x4(sw1152(sk, key, 2 * ks + ((lane >> 3) & 1)), b0, b1, b2, b3);
                mma_f16_16816(s[2 * np], a0, a1, a2, a3, b0, b1);
                mma_f16_16816(s[2 * np + 1], a0, a1, a2, a3, b2, b3);
            }
        }

        // ---- online softmax in the log2 domain, sigma folded into u ----
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int kk = 32 * kh + 8 * nt + 2 * t4 + e;
                const int pos = sm.kpos[buf][kk];
                const float ls = sm.klsig[buf][kk], sg = sm.ksig[buf][kk];
                const bool ok0 = pos >= 0 && (kSparse || pos <= lim0) && lim0 >= 0;
                const bool ok1 = pos >= 0 && (kSparse || pos <= lim1) && lim1 >= 0;
                s[nt][e] = ok0 ? fmaf(s[nt][e] * sg, rs0, ls) : -INFINITY;
                s[nt][2 + e] = ok1 ? fmaf(s[nt][2 + e] * sg, rs1, ls) : -INFINITY;
                mx0 = fmaxf(mx0, s[nt][e]);
                mx1 = fmaxf(mx1, s[nt][2 + e]);
            }
        }
#pragma unroll
        for (int o2 = 1; o2 <= 2; o2 <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o2));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o2));
        }
        if (t4 == 0) {
            sm.redmax[kh][r0] = mx0;
            sm.redmax[kh][r1] = mx1;
        }
        pair_sync(rg);
        mx0 = fmaxf(mx0, sm.redmax[kh ^ 1][r0]);
        mx1 = fmaxf(mx1, sm.redmax[kh ^ 1][r1]);
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        const float mu0 = mn0 == -INFINITY ? 0.f : mn0, mu1 = mn1 == -INFINITY ? 0.f : mn1;
        const float al0 = fast_exp2(m0 - mu0), al1 = fast_exp2(m1 - mu1);
        m0 = mn0;
        m1 = mn1;
        float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
            const int kk = 32 * kh + 8 * nt + 2 * t4;
            const float is0 = sm.kisig[buf][kk], is1 = sm.kisig[buf][kk + 1];
            const float p00 = fast_exp2(s[nt][0] - mu0), p01 = fast_exp2(s[nt][1] - mu0);
            const float p10 = fast_exp2(s[nt][2] - mu1), p11 = fast_exp2(s[nt][3] - mu1);
            ps0 = fmaf(p00, is0, fmaf(p01, is1, ps0));
            ps1 = fmaf(p10, is0, fmaf(p11, is1, ps1));
            const uint32_t w0 = pack_half2(p00, p01), w1 = pack_half2(p10, p11);
            const uint32_t ad0 = sw128(sp, r0, kk >> 3) + (kk & 7) * 2;
            const uint32_t ad1 = sw128(sp, r1, kk >> 3) + (kk & 7) * 2;
            asm volatile("st.shared.b32 [%0], %1;\n" ::"r"(ad0), "r"(w0));
            asm volatile("st.shared.b32 [%0], %1;\n" ::"r"(ad1), "r"(w1));
        }
        l0 = fmaf(l0, al0, ps0);
        l1 = fmaf(l1, al1, ps1);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            o[i][0] *= al0;
            o[i][1] *= al0;
            o[i][2] *= al1;
            o[i][3] *= al1;
        }
        pair_sync(rg);

        // ---- O[16 rows, dims 256kh..+256] += P' V ----
#pragma unroll
        for (int ks = 0; ks < BN / 16; ++ks) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4(sw128(sp, 16 * rg + (lane & 15), 2 * ks + (lane >> 4)), a0, a1, a2, a3);
            const int key = 16 * ks + (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
            for (int np = 0; np < 16; ++np) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(sw1152(sk, key, 32 * kh + 2 * np + (lane >> 4)), b0, b1, b2, b3);
                mma_f16_16816(o[2 * np], a0, a1, a2, a3, b0, b1);
                mma_f16_16816(o[2 * np + 1], a0, a1, a2, a3, b2, b3);
            }
        }
    }

    // ---- epilogue: l over both key halves, O / l, lse ----
#pragma unroll
    for (int o2 = 1; o2 <= 2; o2 <<= 1) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, o2);
        l1 += __shfl_xor_sync(0xffffffffu, l1, o2);
    }
    if (t4 == 0) {
        sm.redsum[kh][r0] = l0;
        sm.redsum[kh][r1] = l1;
    }
    __syncthreads();
    const float L0 = sm.redsum[0][r0] + sm.redsum[1][r0];
    const float L1 = sm.redsum[0][r1] + sm.redsum[1][r1];
    const float inv0 = L0 > 0.f ? 1.f / L0 : 0.f, inv1 = L1 > 0.f ? 1.f / L1 : 0.f;
    const bool v0 = r0 < nvalid && lim0 >= 0, v1 = r1 < nvalid && lim1 >= 0;
    __nv_bfloat16 *out0 = a.out + (grow0 + r0) * kDv + 256 * kh + 2 * t4;
    __nv_bfloat16 *out1 = a.out + (grow0 + r1) * kDv + 256 * kh + 2 * t4;
#pragma unroll
    for (int nt = 0; nt < 32; ++nt) {
        if (v0) *reinterpret_cast<uint32_t *>(out0 + 8 * nt) = pack_bf162(o[nt][0] * inv0, o[nt][1] * inv0);
        if (v1) *reinterpret_cast<uint32_t *>(out1 + 8 * nt) = pack_bf162(o[nt][2] * inv1, o[nt][3] * inv1);
    }
    if (a.lse && kh == 0 && t4 == 0) {
        if (v0) a.lse[grow0 + r0] = L0 > 0.f ? (m0 + __log2f(L0)) * kLn2 : -INFINITY;
        if (v1) a.lse[grow0 + r1] = L1 > 0.f ? (m1 + __log2f(L1)) * kLn2 : -INFINITY;
    }
    __syncthreads();   // smem reused by the next tile of this CTA
}

__device__ __forceinline__ int find_seq(const int32_t *cu, int batch, int64_t t) {
    int lo = 0, hi = batch - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(cu + mid) <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Dense: work item = (sequence, row tile a, row tile b or -1).
__global__ void __launch_bounds__(NT, 1) dense_kernel(const AttnArgs a, const int4 *__restrict__ work) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    Smem &sm = *reinterpret_cast<Smem *>(smem_raw);
    const int4 it = work[blockIdx.x];
    const int b = it.x;
    const int q0 = __ldg(a.cu_seqlens + b), qn = __ldg(a.cu_seqlens + b + 1) - q0;
    const int P = __ldg(a.prefix_lens + b);
    const int32_t *bt = a.block_table + static_cast<int64_t>(b) * a.max_blocks;
    const int rows = qn * a.H;
    for (int w = 0; w < 2; ++w) {
        const int tile = w == 0 ? it.y : it.z;
        if (tile < 0) continue;
        const int r_lo = tile * BM;
        const int nvalid = min(BM, rows - r_lo);
        if (threadIdx.x < BM) {
            const int r = r_lo + threadIdx.x;
            sm.rowlimit[threadIdx.x] = threadIdx.x < nvalid ? P + r / a.H : -1;
        }
        const int key_last = P + (r_lo + nvalid - 1) / a.H;
        const int nk = key_last / BN + 1;
        __syncthreads();
        attend_tile<false>(sm, a, bt, static_cast<int64_t>(q0) * a.H + r_lo, nvalid, key_last, nk, nullptr, 0);
    }
}

// Sparse: one CTA per (token, block of 64 heads).
__global__ void __launch_bounds__(NT, 1) sparse_kernel(const AttnArgs a) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    Smem &sm = *reinterpret_cast<Smem *>(smem_raw);
    const int64_t t = blockIdx.x;
    const int h0 = blockIdx.y * BM;
    const int b = find_seq(a.cu_seqlens, a.batch, t);
    const int64_t qpos = static_cast<int64_t>(__ldg(a.prefix_lens + b)) + (t - __ldg(a.cu_seqlens + b));
    const int32_t *bt = a.block_table + static_cast<int64_t>(b) * a.max_blocks;
    const int nvalid = min(BM, a.H - h0);
    if (threadIdx.x < BM) sm.rowlimit[threadIdx.x] = threadIdx.x < nvalid ? static_cast<int32_t>(qpos) : -1;
    __syncthreads();
    attend_tile<true>(sm, a, bt, t * a.H + h0, nvalid, 0, (a.topk + BN - 1) / BN,
                      a.idx + t * a.topk, static_cast<int32_t>(qpos));
}

}  // namespace sm80path

cudaError_t launch_dense_sm80path(const AttnArgs &a, const int4 *work, int n_work, cudaStream_t st) {
    const int smem = sizeof(sm80path::Smem);
    cudaError_t e = cudaFuncSetAttribute(sm80path::dense_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (n_work > 0) sm80path::dense_kernel<<<n_work, sm80path::NT, smem, st>>>(a, work);
    return cudaGetLastError();
}

cudaError_t launch_sparse_sm80path(const AttnArgs &a, int64_t n_tokens, cudaStream_t st) {
    const int smem = sizeof(sm80path::Smem);
    cudaError_t e = cudaFuncSetAttribute(sm80path::sparse_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    dim3 grid(static_cast<unsigned>(n_tokens), (a.H + sm80path::BM - 1) / sm80path::BM);
    if (n_tokens > 0) sm80path::sparse_kernel<<<grid, sm80path::NT, smem, st>>>(a);
    return cudaGetLastError();
}

}  // namespace mla

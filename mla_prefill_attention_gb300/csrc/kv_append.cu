// Cache write of the new tokens, the step before attention (sm_103a).
//
// Each new token's latent row (576 bf16: 512 latent + 64 RoPE dims) and,
// optionally, its indexer key (128 bf16) are quantised to e4m3 with one fp32
// scale per token and row, and stored at the token's position through the
// block table ("More throughput from fewer GPUs", section System architecture:
// FP8 KV cache, one latent row per token; section KV hand-off and caching:
// 256-token chunks; GLM-5.3 Teil 2, footnote 3: indexer keys are 128 FP8
// values plus a 4-byte scale).
//
//   scale = max(amax / 448, 2^-126), amax = max |x| over the row; 1 if amax = 0
//   code  = cvt.rn.satfinite.e4m3(x * (1 / scale))
// with the division, reciprocal and product each one IEEE binary32 operation
// (rounded to nearest even), so every code is fixed by the definition; the
// floor at the smallest normal value keeps the reciprocal finite.
//
// Pure streaming work (2,120 bytes moved per token with the indexer key): one
// warp per token, 16-byte loads, 8-byte code stores, the row maximum reduced
// on the bf16 magnitude bits (a token's two maxima packed in one word, so one
// shuffle chain serves both).
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"

namespace mla {
namespace app {

constexpr int kWarps = 8;   // tokens per CTA, one per warp

// Pairwise maxima of the magnitudes of eight bf16 values (sign bits cleared):
// two 16-bit maxima in one word. bf16 magnitude order equals the order of
// these bit patterns for every non-NaN value.
__device__ __forceinline__ uint32_t mag8(const uint4 &v) {
    const uint32_t m = 0x7fff7fffu;
    return __vmaxu2(__vmaxu2(v.x & m, v.y & m), __vmaxu2(v.z & m, v.w & m));
}

__device__ __forceinline__ uint32_t fold16(uint32_t m) { return max(m & 0xffffu, m >> 16); }

__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Two bf16 in one word -> the IEEE binary32 products with inv -> two e4m3 codes
__device__ __forceinline__ uint32_t quant2(uint32_t w, float inv) {
    return e4m3x2(__fmul_rn(__uint_as_float(w << 16), inv), __fmul_rn(__uint_as_float(w & 0xffff0000u), inv));
}

__device__ __forceinline__ uint2 quant8(const uint4 &v, float inv) {
    return make_uint2(quant2(v.x, inv) | (quant2(v.y, inv) << 16), quant2(v.z, inv) | (quant2(v.w, inv) << 16));
}

__device__ __forceinline__ float scale_of(uint32_t mag) {
    const float amax = __uint_as_float(mag << 16);
    return amax > 0.f ? fmaxf(__fdiv_rn(amax, 448.f), 0x1p-126f) : 1.f;
}

// One token's rows as this lane holds them: the latent row is 72 chunks of 8
// bf16 (lanes 0..31 take chunks lane and 32 + lane, lanes 0..7 also 64 +
// lane); the indexer key's 16 chunks go to lanes 8..23, which hold one latent
// chunk fewer.
struct TokenRows {
    uint4 v0, v1, v2, k0;
    int64_t row;   // cache row, -1 if the token's page is invalid
};

__device__ __forceinline__ TokenRows load_token(const AppendArgs &a, int64_t t, int lane, bool has_k) {
    TokenRows r;
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    r.v2 = r.k0 = z;
    const uint4 *lat = reinterpret_cast<const uint4 *>(a.latent) + t * (kDqk / 8);
    r.v0 = __ldg(lat + lane);
    r.v1 = __ldg(lat + 32 + lane);
    if (lane < 8) r.v2 = __ldg(lat + 64 + lane);
    if (has_k) r.k0 = __ldg(reinterpret_cast<const uint4 *>(a.kidx) + t * (kDidx / 8) + (lane - 8));
    const int b = find_seq(a.cu_seqlens, a.batch, t);
    const int64_t pos = __ldg(a.prefix_lens + b) + (t - __ldg(a.cu_seqlens + b));
    r.row = cache_row(a.block_table + static_cast<int64_t>(b) * a.max_blocks, a.max_blocks, a.num_blocks, pos,
                      lane == 0 ? a.dev_err : nullptr);
    return r;
}

// Both rows' maxima over the warp: latent in the high half-word, key in the low.
__device__ __forceinline__ uint32_t row_maxima(const TokenRows &r) {
    uint32_t m = (fold16(__vmaxu2(__vmaxu2(mag8(r.v0), mag8(r.v1)), mag8(r.v2))) << 16) | fold16(mag8(r.k0));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = __vmaxu2(m, __shfl_xor_sync(0xffffffffu, m, off));
    return m;
}

__device__ __forceinline__ void store_token(const AppendArgs &a, const TokenRows &r, int lane, bool has_k, float sl,
                                            float il, float sk, float ik) {
    if (r.row < 0) return;   // the same for every lane of the warp
    uint2 *dst = reinterpret_cast<uint2 *>(a.kv + r.row * kDqk);
    dst[lane] = quant8(r.v0, il);
    dst[32 + lane] = quant8(r.v1, il);
    if (lane < 8) dst[64 + lane] = quant8(r.v2, il);
    if (lane == 0) a.kv_scale[r.row] = sl;
    if (has_k) {
        reinterpret_cast<uint2 *>(a.ki + r.row * kDidx)[lane - 8] = quant8(r.k0, ik);
        if (lane == 8) a.ki_scale[r.row] = sk;
    }
}

// One token per warp; the two rows' scales and reciprocals come out of one
// pass of the division and reciprocal code (lane 0 computes the latent row's,
// lane 1 the key's) and are broadcast by shuffles.
__global__ void __launch_bounds__(kWarps * 32) kv_append_kernel(AppendArgs a) {
    const int lane = threadIdx.x & 31;
    const int64_t t = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
    if (t >= a.n_tokens) return;
    const bool has_k = a.kidx != nullptr && lane >= 8 && lane < 8 + kDidx / 8;
    const TokenRows r = load_token(a, t, lane, has_k);
    const uint32_t m = row_maxima(r);
    const float s = scale_of((lane & 1) ? (m & 0xffffu) : (m >> 16));
    const float inv = __frcp_rn(s);
    store_token(a, r, lane, has_k, __shfl_sync(0xffffffffu, s, 0), __shfl_sync(0xffffffffu, inv, 0),
                __shfl_sync(0xffffffffu, s, 1), __shfl_sync(0xffffffffu, inv, 1));
}

}  // namespace app

cudaError_t launch_kv_append(const AppendArgs &a, cudaStream_t st) {
    if (a.n_tokens <= 0) return cudaSuccess;
    const int64_t grid = (a.n_tokens + app::kWarps - 1) / app::kWarps;
    app::kv_append_kernel<<<static_cast<unsigned>(grid), app::kWarps * 32, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace mla

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
// Pure streaming work (2,120 bytes moved per token with the indexer key): four
// tokens per warp, 16-byte loads, 8-byte code stores, the row maximum reduced
// on the bf16 magnitude bits (a token's two maxima packed in one word, so one
// shuffle chain serves both).
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"

namespace mla {
namespace app {

constexpr int kWarps = 8;          // warps per CTA
constexpr int kTokensPerWarp = 4;

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

// Four tokens per warp, eight lanes per token: lane 8u + i takes chunks i, i+8,
// ..., i+80 of token u's 88 chunks of 8 values (72 latent, then 16 key), i.e.
// nine latent chunks and two key chunks, so every lane has work and each load
// instruction covers four 128-byte runs.
constexpr int kLatChunks = kDqk / 8, kKeyChunks = kDidx / 8;   // 72, 16
constexpr int kLatPerLane = kLatChunks / 8, kKeyPerLane = kKeyChunks / 8;   // 9, 2

__global__ void __launch_bounds__(kWarps * 32) kv_append_kernel(AppendArgs a) {
    const int lane = threadIdx.x & 31, u = lane >> 3, i8 = lane & 7;
    const int64_t t = (static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5)) * kTokensPerWarp + u;
    const bool live = t < a.n_tokens;
    const bool has_k = a.kidx != nullptr;
    const uint4 z = make_uint4(0u, 0u, 0u, 0u);
    uint4 lv[kLatPerLane], kv4[kKeyPerLane];
    const uint4 *lat = reinterpret_cast<const uint4 *>(a.latent) + (live ? t : 0) * kLatChunks + i8;
    const uint4 *key = has_k ? reinterpret_cast<const uint4 *>(a.kidx) + (live ? t : 0) * kKeyChunks + i8 : nullptr;
#pragma unroll
    for (int m = 0; m < kLatPerLane; ++m) lv[m] = live ? __ldg(lat + 8 * m) : z;
#pragma unroll
    for (int m = 0; m < kKeyPerLane; ++m) kv4[m] = live && has_k ? __ldg(key + 8 * m) : z;

    int64_t row = -1;
    if (live) {
        const int b = find_seq(a.cu_seqlens, a.batch, t);
        const int64_t pos = __ldg(a.prefix_lens + b) + (t - __ldg(a.cu_seqlens + b));
        row = cache_row(a.block_table + static_cast<int64_t>(b) * a.max_blocks, a.max_blocks, a.num_blocks, pos,
                        i8 == 0 ? a.dev_err : nullptr);
    }
    // both rows' maxima over the token's eight lanes: latent high half-word, key low
    uint32_t ml = 0, mk = 0;
#pragma unroll
    for (int m = 0; m < kLatPerLane; ++m) ml = __vmaxu2(ml, mag8(lv[m]));
#pragma unroll
    for (int m = 0; m < kKeyPerLane; ++m) mk = __vmaxu2(mk, mag8(kv4[m]));
    uint32_t mx = (fold16(ml) << 16) | fold16(mk);
#pragma unroll
    for (int off = 4; off > 0; off >>= 1) mx = __vmaxu2(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    // one pass of the division and reciprocal code for the warp's eight rows: lane
    // 8u takes token u's latent row, lane 8u + 1 its key
    const float s = scale_of((i8 & 1) ? (mx & 0xffffu) : (mx >> 16));
    const float inv = __frcp_rn(s);
    const float sl = __shfl_sync(0xffffffffu, s, 8 * u), il = __shfl_sync(0xffffffffu, inv, 8 * u);
    const float sk = __shfl_sync(0xffffffffu, s, 8 * u + 1), ik = __shfl_sync(0xffffffffu, inv, 8 * u + 1);
    if (row < 0) return;   // the same for the token's eight lanes; the shuffles are done
    uint2 *dl = reinterpret_cast<uint2 *>(a.kv + row * kDqk) + i8;
#pragma unroll
    for (int m = 0; m < kLatPerLane; ++m) dl[8 * m] = quant8(lv[m], il);
    if (i8 == 0) a.kv_scale[row] = sl;
    if (has_k) {
        uint2 *dk = reinterpret_cast<uint2 *>(a.ki + row * kDidx) + i8;
#pragma unroll
        for (int m = 0; m < kKeyPerLane; ++m) dk[8 * m] = quant8(kv4[m], ik);
        if (i8 == 0) a.ki_scale[row] = sk;
    }
}

}  // namespace app

cudaError_t launch_kv_append(const AppendArgs &a, cudaStream_t st) {
    if (a.n_tokens <= 0) return cudaSuccess;
    const int64_t per_cta = app::kWarps * app::kTokensPerWarp;
    const int64_t grid = (a.n_tokens + per_cta - 1) / per_cta;
    app::kv_append_kernel<<<static_cast<unsigned>(grid), app::kWarps * 32, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace mla

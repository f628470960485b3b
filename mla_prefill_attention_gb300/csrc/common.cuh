// Shared device helpers of the MLA prefill kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "../../include/mla.h"

namespace mla {

constexpr int kPage = 256;     // tokens per KV page
constexpr int kDqk = 576;      // latent 512 + RoPE 64
constexpr int kDv = 512;
constexpr int kDidx = 128;     // indexer head dim
constexpr int kHidx = 64;      // indexer heads
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t pack_half2(float x, float y) {
    __half2 h = __floats2half2_rn(x, y);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ uint32_t pack_bf162(float x, float y) {
    __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
    return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void set_dev_err(int32_t *dev_err, int bit) {
    if (dev_err) atomicOr(dev_err, bit);
}

// Sequence of global new-token t: the last b with cu[b] <= t (cu non-decreasing,
// so sequences without new tokens are passed over).
__device__ __forceinline__ int find_seq(const int32_t *cu, int batch, int64_t t) {
    int lo = 0, hi = batch - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(cu + mid) <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// Physical cache row of position s of the sequence whose block-table row is bt;
// -1 (and an error bit) if the page id is outside [0, num_blocks).
__device__ __forceinline__ int64_t cache_row(const int32_t *bt, int32_t max_blocks, int32_t num_blocks, int64_t s,
                                             int32_t *dev_err) {
    int64_t blk = s / kPage;
    if (blk >= max_blocks) {
        set_dev_err(dev_err, MLA_DEVERR_BAD_PAGE);
        return -1;
    }
    int32_t page = __ldg(bt + blk);
    if (page < 0 || page >= num_blocks) {
        set_dev_err(dev_err, MLA_DEVERR_BAD_PAGE);
        return -1;
    }
    return static_cast<int64_t>(page) * kPage + (s % kPage);
}

}  // namespace mla

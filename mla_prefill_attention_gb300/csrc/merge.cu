// Merge of partial attention results over disjoint key sets (sm_103a).
//
// When a query's keys are split (GLM-5.3 Teil 2, section "DCP: Sharding auch
// des KV-Caches": every GPU attends over its own shard of the cache and the
// partial results are combined through their log-sum-exp), part i gives the
// softmax-weighted mean o_i over its keys and lse_i = ln(sum of exp(logit)).
// Attention over the union is
//   lse = ln sum_i exp(lse_i),   out = sum_i exp(lse_i - lse) * o_i
// computed here as m = max_i lse_i, w_i = exp(lse_i - m), out = sum w_i o_i /
// sum w_i, lse = m + ln(sum w_i). A part with lse_i = -inf has w_i = 0; a row
// whose parts are all empty gets out = 0, lse = -inf.
//
// Streaming work: one warp per 512-value row, two 16-byte loads per lane and
// part (the part count is a template parameter, so only live parts hold
// registers), fp32 arithmetic, one rounding to bf16 at the end.
#include <cuda_runtime.h>
#include <math.h>

#include "common.cuh"
#include "kernels.h"

namespace mla {
namespace mrg {

constexpr int kWarps = 8;   // rows per CTA

__device__ __forceinline__ void acc8(float *acc, const uint4 &v, float w) {
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        acc[2 * j] = fmaf(w, __uint_as_float(u[j] << 16), acc[2 * j]);
        acc[2 * j + 1] = fmaf(w, __uint_as_float(u[j] & 0xffff0000u), acc[2 * j + 1]);
    }
}

__device__ __forceinline__ uint4 pack8(const float *acc, float inv) {
    return make_uint4(pack_bf162(acc[0] * inv, acc[1] * inv), pack_bf162(acc[2] * inv, acc[3] * inv),
                      pack_bf162(acc[4] * inv, acc[5] * inv), pack_bf162(acc[6] * inv, acc[7] * inv));
}

template <int N>
__global__ void __launch_bounds__(kWarps * 32) merge_kernel(MergeArgs a) {
    const int lane = threadIdx.x & 31;
    const int64_t r = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
    if (r >= a.rows) return;
    float l[N];
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < N; ++i) {
        l[i] = __ldg(a.lses[i] + r);
        m = fmaxf(m, l[i]);
    }
    uint4 *dst = a.out + r * (kDv / 8);
    if (m == -INFINITY) {
        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
        dst[lane] = z;
        dst[32 + lane] = z;
        if (lane == 0 && a.lse) a.lse[r] = -INFINITY;
        return;
    }
    uint4 v[N][2];
#pragma unroll
    for (int i = 0; i < N; ++i)
        if (l[i] != -INFINITY) {
            const uint4 *src = a.outs[i] + r * (kDv / 8);
            v[i][0] = __ldg(src + lane);
            v[i][1] = __ldg(src + 32 + lane);
        }
    float acc0[8] = {}, acc1[8] = {}, wsum = 0.f;
#pragma unroll
    for (int i = 0; i < N; ++i)
        if (l[i] != -INFINITY) {
            const float w = expf(l[i] - m);
            wsum += w;
            acc8(acc0, v[i][0], w);
            acc8(acc1, v[i][1], w);
        }
    const float inv = 1.f / wsum;
    dst[lane] = pack8(acc0, inv);
    dst[32 + lane] = pack8(acc1, inv);
    if (lane == 0 && a.lse) a.lse[r] = m + logf(wsum);
}

}  // namespace mrg

cudaError_t launch_merge(const MergeArgs &a, cudaStream_t st) {
    if (a.rows <= 0) return cudaSuccess;
    const int64_t grid = (a.rows + mrg::kWarps - 1) / mrg::kWarps;
    const dim3 g(static_cast<unsigned>(grid)), b(mrg::kWarps * 32);
    switch (a.n_parts) {
    case 1: mrg::merge_kernel<1><<<g, b, 0, st>>>(a); break;
    case 2: mrg::merge_kernel<2><<<g, b, 0, st>>>(a); break;
    case 3: mrg::merge_kernel<3><<<g, b, 0, st>>>(a); break;
    case 4: mrg::merge_kernel<4><<<g, b, 0, st>>>(a); break;
    case 5: mrg::merge_kernel<5><<<g, b, 0, st>>>(a); break;
    case 6: mrg::merge_kernel<6><<<g, b, 0, st>>>(a); break;
    case 7: mrg::merge_kernel<7><<<g, b, 0, st>>>(a); break;
    case 8: mrg::merge_kernel<8><<<g, b, 0, st>>>(a); break;
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace mla

// Allocation-free variant of the dense entry point (mla_prefill_dense_static).
//
// Who needs it: code that is handed only its input and output buffers and may
// not allocate device memory itself. Examples are a plugin running inside a
// host framework that owns the whole device memory pool and offers no
// workspace hook, and latency-critical callers that must not hit the implicit
// device synchronisation of cudaMalloc/cudaFree.
//
// What differs from mla_prefill_dense: the work list (one 16-byte item per
// pair of row tiles) is not placed in a caller workspace. It lives in the
// file-scope device array below, which every GPU that loads this library
// keeps until the process exits, and it is built on the GPU by a one-CTA
// kernel rather than uploaded from the host. Items follow sequence order (the
// workspace entry point also sorts them by cost). The attention kernel itself
// is the same one mla_prefill_dense launches.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/mla.h"
#include "kernels.h"

namespace {

constexpr int kBM = 64;           // query rows per tile, as in the dense kernel
constexpr int kMaxDevices = 64;

static __device__ __align__(256) int4 g_dense_static_work[MLA_DENSE_STATIC_MAX_WORK_ITEMS];

std::mutex g_mu;
int4 *g_work_ptr[kMaxDevices] = {};

// Address of g_dense_static_work on the current device, looked up once per
// device (the host-side symbol is only a stand-in, never a device address).
cudaError_t static_work_ptr(int4 **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_work_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_dense_static_work);
        if (e != cudaSuccess) return e;
        g_work_ptr[dev] = static_cast<int4 *>(p);
    }
    *out = g_work_ptr[dev];
    return cudaSuccess;
}

// One CTA: sequences in chunks of blockDim; a block-wide scan over the pair
// counts gives each sequence its first item, then each thread writes the items
// of its own sequence: (b, tile i, tile n-1-i or -1). Exactly n_items entries
// are written (the count the host derived from its mirror of cu_seqlens):
// items past the device count become empty (tile -1, which the attention
// kernel skips), so no entry left over from an earlier call is ever read. If
// the device count differs from n_items (the device cu_seqlens disagrees with
// its host mirror) MLA_DEVERR_SEQ_MISMATCH is set; items past n_items are
// dropped.
__global__ void build_pairs_kernel(const int32_t *__restrict__ cu, int32_t batch, int32_t H, int4 *work,
                                   int32_t n_items, int32_t *dev_err) {
    __shared__ int32_t scan[1024];
    __shared__ int32_t base;
    if (threadIdx.x == 0) base = 0;
    __syncthreads();
    for (int c0 = 0; c0 < batch; c0 += blockDim.x) {
        const int b = c0 + threadIdx.x;
        int32_t tiles = 0, pairs = 0;
        if (b < batch) {
            const int64_t rows = static_cast<int64_t>(cu[b + 1] - cu[b]) * H;
            tiles = static_cast<int32_t>((rows + kBM - 1) / kBM);
            pairs = (tiles + 1) / 2;
        }
        scan[threadIdx.x] = pairs;
        __syncthreads();
        for (int o = 1; o < static_cast<int>(blockDim.x); o <<= 1) {
            const int32_t v = threadIdx.x >= static_cast<unsigned>(o) ? scan[threadIdx.x - o] : 0;
            __syncthreads();
            scan[threadIdx.x] += v;
            __syncthreads();
        }
        const int32_t first = base + scan[threadIdx.x] - pairs;
        for (int32_t i = 0; i < pairs && first + i < n_items; ++i) {
            const int32_t j = tiles - 1 - i;
            work[first + i] = make_int4(b, i, j != i ? j : -1, 0);
        }
        __syncthreads();
        if (threadIdx.x == blockDim.x - 1) base += scan[threadIdx.x];
        __syncthreads();
    }
    for (int32_t i = base + threadIdx.x; i < n_items; i += blockDim.x) work[i] = make_int4(0, -1, -1, 0);
    if (threadIdx.x == 0 && base != n_items && dev_err) atomicOr(dev_err, MLA_DEVERR_SEQ_MISMATCH);
}

}  // namespace

namespace mla {
// Shared with mla_api.cu: argument checks and error reporting of the C ABI.
mla_status_t check_dense_args(const mla_seqs_t *seqs, const void *q, int32_t H, const uint8_t *kv,
                              const float *kv_scale, const void *out, const float *lse, float sm_scale);
mla_status_t report(mla_status_t s, const char *msg);
AttnArgs make_attn_args(const mla_seqs_t *s, const void *q, int32_t H, const uint8_t *kv, const float *kv_scale,
                        float sm_scale, void *out, float *lse, int32_t *dev_err);
}  // namespace mla

extern "C" mla_status_t mla_prefill_dense_static(const mla_seqs_t *seqs, const void *q_bf16, int32_t num_heads,
                                                 const uint8_t *kv_e4m3, const float *kv_scale, float sm_scale,
                                                 void *out_bf16, float *lse, int32_t *dev_err,
                                                 cudaStream_t stream) {
    mla_status_t st = mla::check_dense_args(seqs, q_bf16, num_heads, kv_e4m3, kv_scale, out_bf16, lse, sm_scale);
    if (st != MLA_OK) return st;
    int64_t items = 0;
    for (int b = 0; b < seqs->batch; ++b) {
        const int64_t rows =
            static_cast<int64_t>(seqs->cu_seqlens_q_host[b + 1] - seqs->cu_seqlens_q_host[b]) * num_heads;
        items += ((rows + kBM - 1) / kBM + 1) / 2;
    }
    if (items == 0) return MLA_OK;
    if (items > MLA_DENSE_STATIC_MAX_WORK_ITEMS)
        return mla::report(MLA_ERR_UNSUPPORTED,
                           "mla_prefill_dense_static: batch needs more work items than its fixed device array "
                           "holds (MLA_DENSE_STATIC_MAX_WORK_ITEMS); split the batch or use mla_prefill_dense");
    int4 *work = nullptr;
    cudaError_t e = static_work_ptr(&work);
    if (e != cudaSuccess) return mla::report(MLA_ERR_CUDA, cudaGetErrorString(e));
    build_pairs_kernel<<<1, 1024, 0, stream>>>(seqs->cu_seqlens_q, seqs->batch, num_heads, work,
                                               static_cast<int32_t>(items), dev_err);
    if ((e = cudaGetLastError()) != cudaSuccess) return mla::report(MLA_ERR_CUDA, cudaGetErrorString(e));
    const mla::AttnArgs a =
        mla::make_attn_args(seqs, q_bf16, num_heads, kv_e4m3, kv_scale, sm_scale, out_bf16, lse, dev_err);
    CUtensorMap tmap_kv;
    if (!mla::encode_kv_tmap(&tmap_kv, kv_e4m3, seqs->num_blocks))
        return mla::report(MLA_ERR_CUDA, "tensor map encoding for the latent cache failed");
    e = mla::launch_dense_f8(a, work, static_cast<int>(items), tmap_kv, stream);
    if (e != cudaSuccess) return mla::report(MLA_ERR_CUDA, cudaGetErrorString(e));
    return MLA_OK;
}

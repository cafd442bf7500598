// Channel selection (Prox technical summary, Stage 1 "Mask Generation": the magnitude
// ranking of s~ gives the binary channel mask m_s; the abstract: the mask needs only the
// ranking of the entries, not their values).
//
// topk_kernel   one block per token. The salience values are non-negative fp32, so their
//               bit patterns order like the values and a 4-pass 8-bit radix select finds
//               the k-th largest key T and how many keys equal to T belong to the top k.
//               One scan in index order then emits the mask as ascending channel indices,
//               giving equal values to the lower index.
// union_kernel  batch path: the tile's per-token masks are merged into one ascending list
//               of channels and a bit mask per entry telling which tokens selected it, so
//               Stage 2 reads each selected row once for the whole tile.
#include "prox_kernels.cuh"

namespace prox {

constexpr int kTopkThreads = 1024;

__global__ void __launch_bounds__(kTopkThreads)
topk_kernel(const float* __restrict__ sigma, int F, int k, int32_t* __restrict__ idx) {
    extern __shared__ __align__(16) unsigned char smem[];
    uint32_t* keys = reinterpret_cast<uint32_t*>(smem);
    __shared__ int hist[256], sel[4], scan[32];
    const int b = blockIdx.x;
    grid_dep_wait();
    const float* sg = sigma + static_cast<size_t>(b) * F;
    for (int i = threadIdx.x; i < F; i += kTopkThreads) keys[i] = __float_as_uint(sg[i]);
    __syncthreads();
    uint32_t T;
    int take;
    block_radix_select<kTopkThreads>(keys, F, k, hist, sel, T, take);
    block_compact_topk<kTopkThreads>(keys, F, T, take, idx + static_cast<size_t>(b) * k, k, scan);
    grid_dep_launch();
}

__global__ void __launch_bounds__(kTopkThreads)
union_kernel(const int32_t* __restrict__ idx, int nb, int k, int F, int32_t* __restrict__ ulist,
             uint32_t* __restrict__ ubits, int* __restrict__ count, int* __restrict__ status) {
    extern __shared__ __align__(16) unsigned char smem[];
    uint32_t* bits = reinterpret_cast<uint32_t*>(smem);
    __shared__ int scan[32];
    const int tid = threadIdx.x;
    grid_dep_wait();
    for (int i = tid; i < F; i += kTopkThreads) bits[i] = 0u;
    __syncthreads();
    for (int b = 0; b < nb; ++b)
        for (int r = tid; r < k; r += kTopkThreads) {
            const int j = idx[static_cast<size_t>(b) * k + r];
            if (j >= 0 && j < F)
                atomicOr(&bits[j], 1u << b);
            else if (status)
                set_status(status, PROX_ERR_BOUNDS);
        }
    __syncthreads();
    const int per = (F + kTopkThreads - 1) / kTopkThreads;
    const int lo = min(F, tid * per), hi = min(F, lo + per);
    int cnt = 0;
    for (int i = lo; i < hi; ++i) cnt += bits[i] != 0u;
    int total;
    int pos = block_exclusive_scan<kTopkThreads>(cnt, scan, total);
    for (int i = lo; i < hi; ++i) {
        if (bits[i]) {
            ulist[pos] = i;
            ubits[pos] = bits[i];
            ++pos;
        }
    }
    if (tid == 0) *count = total;
    grid_dep_launch();
}

int launch_topk(const float* sigma_tile, int F, int nb, int k, int32_t* idx_tile, cudaStream_t s) {
    const size_t smem = static_cast<size_t>(F) * 4;
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(reinterpret_cast<const void*>(topk_kernel),
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
        return PROX_ERR_CUDA;
    topk_kernel<<<nb, kTopkThreads, smem, s>>>(sigma_tile, F, k, idx_tile);
    return cudaGetLastError() == cudaSuccess ? PROX_OK : PROX_ERR_CUDA;
}

int launch_union(const int32_t* idx_tile, int nb, int k, int F, int32_t* ulist, uint32_t* ubits,
                 int* count, int* status, cudaStream_t s) {
    const size_t smem = static_cast<size_t>(F) * 4;
    if (smem > 48 * 1024 &&
        cudaFuncSetAttribute(reinterpret_cast<const void*>(union_kernel),
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
        return PROX_ERR_CUDA;
    union_kernel<<<1, kTopkThreads, smem, s>>>(idx_tile, nb, k, F, ulist, ubits, count, status);
    return cudaGetLastError() == cudaSuccess ? PROX_OK : PROX_ERR_CUDA;
}

}  // namespace prox

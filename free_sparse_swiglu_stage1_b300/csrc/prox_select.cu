// Channel selection (Prox technical summary, Stage 1 "Mask Generation": the magnitude
// ranking of s~ gives the binary channel mask m_s; the abstract: the mask needs only the
// ranking of the entries, not their values).
//
// topk_kernel   one block per token. The salience values are non-negative fp32, so their
//               bit patterns order like the values and a three-pass radix select (11, 11
//               and 9 bits) finds the k-th largest key T and how many keys equal to T belong
//               to the top k; the first pass's histogram comes ready from Stage 1, so only
//               the candidates of one bin are scanned again. One scan in index order then
//               emits the mask as ascending channel indices, giving equal values to the
//               lower index.
//               With a channel bitmap given, each block also ORs its token's bit into the
//               word of every channel it selected (the tensor-core Stage 2 reads it).
// union_kernel  CUDA-core batch path: the tile's per-token masks are merged into one
//               ascending list of channels and a bit mask per entry telling which tokens
//               selected it, so Stage 2 reads each selected row once for the whole tile.
// mask_bits_kernel  the bitmap of given masks (for the tensor-core Stage 2).
#include "prox_kernels.cuh"

namespace prox {

constexpr int kTopkThreads = 1024;

template <int NT, int RUN>
__global__ void __launch_bounds__(NT)
topk_kernel(const float* __restrict__ sigma, int F, int k, int32_t* __restrict__ idx,
            const int* __restrict__ ghist, uint32_t* __restrict__ bits, long long spin,
            int* __restrict__ status) {
    extern __shared__ __align__(128) unsigned char smem[];
    uint32_t* keys = reinterpret_cast<uint32_t*>(smem);   // [F] salience bits (all >= 0)
    __shared__ __align__(128) int hist[2 * 2048];
    __shared__ int wsum[NT / 32 + 4];
    __shared__ __align__(8) uint64_t bar;
    const int b = blockIdx.x, tid = threadIdx.x;
    if (tid == 0) {
        mbar_init(&bar, 1);
        mbar_init_fence();
    }
    __syncthreads();
    grid_dep_wait();
    grid_dep_launch();
    // the token's salience row and its first-pass histogram, each one bulk copy
    if (tid == 0) {
        mbar_arrive_expect_tx(&bar, static_cast<uint32_t>(F) * 4 + 2048 * 4);
        bulk_g2s(keys, sigma + static_cast<size_t>(b) * F, static_cast<uint32_t>(F) * 4, &bar);
        bulk_g2s(hist, ghist + static_cast<size_t>(b) * 2048, 2048 * 4, &bar);
    }
    if (!__syncthreads_and(mbar_wait(&bar, 0u, spin, status))) {
        // nothing usable arrived: leave the mask unwritten; the status word says why
        return;
    }
    uint32_t T;
    int take, eq_total;
    block_select_kth<NT, RUN>(keys, F, k, hist, wsum, T, take, eq_total, nullptr, true);
    uint64_t mine;
    const int cnt = block_take_topk<NT, RUN>(keys, F, T, take, eq_total, wsum, mine);
    int total;
    int pos = block_exclusive_scan<NT>(cnt, wsum, total);   // ends with a barrier: keys are free
    // the mask is assembled in shared memory (over the keys) and written out coalesced
    int32_t* s_idx = reinterpret_cast<int32_t*>(keys);
    const int lo = tid * RUN;
#pragma unroll
    for (int i = 0; i < RUN; ++i)
        if (((mine >> i) & 1ull) && pos < k) s_idx[pos++] = lo + i;
    __syncthreads();
    int32_t* out = idx + static_cast<size_t>(b) * k;
    for (int i = tid; i < k; i += NT) out[i] = s_idx[i];
    if (bits)   // the batch's channel bitmap for the tensor-core Stage 2
        for (int i = tid; i < k; i += NT) atomicOr(&bits[s_idx[i]], 1u << b);
}

// bits[j] |= 1 << b for every channel j of index row b; grid (chunks of the rows, B).
__global__ void __launch_bounds__(256)
mask_bits_kernel(const int32_t* __restrict__ idx, int k, int F, uint32_t* __restrict__ bits,
                 int* __restrict__ status) {
    grid_dep_wait();
    grid_dep_launch();
    const int b = blockIdx.y;
    for (int i = blockIdx.x * 256 + threadIdx.x; i < k; i += gridDim.x * 256) {
        const int j = idx[static_cast<size_t>(b) * k + i];
        if (j >= 0 && j < F)
            atomicOr(&bits[j], 1u << b);
        else if (status)
            set_status(status, PROX_ERR_BOUNDS);
    }
}

__global__ void __launch_bounds__(kTopkThreads)
union_kernel(const int32_t* __restrict__ idx, int nb, int k, int F, int32_t* __restrict__ ulist,
             uint32_t* __restrict__ ubits, int* __restrict__ count, int* __restrict__ status) {
    extern __shared__ __align__(128) unsigned char smem[];
    uint32_t* bits = reinterpret_cast<uint32_t*>(smem);
    __shared__ int wsum[kTopkThreads / 32 + 4];
    const int tid = threadIdx.x;
    grid_dep_wait();
    grid_dep_launch();
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
    int pos = block_exclusive_scan<kTopkThreads>(cnt, wsum, total);
    for (int i = lo; i < hi; ++i) {
        if (bits[i]) {
            ulist[pos] = i;
            ubits[pos] = bits[i];
            ++pos;
        }
    }
    if (tid == 0) *count = total;
}

template <int NT, int RUN>
static int launch_topk_t(const float* sigma, int F, int B, int k, int32_t* idx,
                         const int* ghist, uint32_t* bits, int* status, cudaStream_t s) {
    const size_t smem = static_cast<size_t>(F) * 4;
    auto fn = topk_kernel<NT, RUN>;
    if (ensure_dynamic_smem(reinterpret_cast<const void*>(fn), smem) != PROX_OK) return PROX_ERR_CUDA;
    return launch_pdl(fn, dim3(B), dim3(NT), smem, s, sigma, F, k, idx, ghist, bits,
                      kDefaultSpinCycles, status);
}

int launch_topk(const float* sigma, int F, int B, int k, int32_t* idx, const int* ghist,
                uint32_t* bits, int* status, cudaStream_t s) {
    switch (select_run(F, 1024)) {
        case 4: return launch_topk_t<1024, 4>(sigma, F, B, k, idx, ghist, bits, status, s);
        case 8: return launch_topk_t<1024, 8>(sigma, F, B, k, idx, ghist, bits, status, s);
        case 16: return launch_topk_t<1024, 16>(sigma, F, B, k, idx, ghist, bits, status, s);
        case 32: return launch_topk_t<1024, 32>(sigma, F, B, k, idx, ghist, bits, status, s);
        case 64: return launch_topk_t<1024, 64>(sigma, F, B, k, idx, ghist, bits, status, s);
        default: return PROX_ERR_UNSUPPORTED;
    }
}

int launch_mask_bits(const int32_t* idx, int B, int k, int F, uint32_t* bits, int* status,
                     cudaStream_t s) {
    int chunks = (k + 255) / 256;
    if (chunks > 16) chunks = 16;
    return launch_pdl(mask_bits_kernel, dim3(chunks, B), dim3(256), 0, s, idx, k, F, bits, status);
}

int launch_union(const int32_t* idx_tile, int nb, int k, int F, int32_t* ulist, uint32_t* ubits,
                 int* count, int* status, cudaStream_t s) {
    const size_t smem = static_cast<size_t>(F) * 4;
    if (ensure_dynamic_smem(reinterpret_cast<const void*>(union_kernel), smem) != PROX_OK) return PROX_ERR_CUDA;
    return launch_pdl(union_kernel, dim3(1), dim3(kTopkThreads), smem, s, idx_tile, nb, k, F, ulist,
                      ubits, count, status);
}

}  // namespace prox

// Small kernels around the path: the unit-gain RMSNorm between stacked layers, an index
// fill for the all-channels mask, and the bounded-wait probe used to test timeouts.
#include <atomic>
#include <cstdio>
#include <map>
#include <mutex>
#include <utility>

#include "prox_kernels.cuh"

namespace prox {

namespace {
thread_local char g_last_cuda_error[256] = "none";
}

int cuda_fail(cudaError_t err, const char* what) {
    snprintf(g_last_cuda_error, sizeof(g_last_cuda_error), "%s: %s (%s)", what,
             cudaGetErrorName(err), cudaGetErrorString(err));
    return PROX_ERR_CUDA;
}

const char* last_cuda_error() { return g_last_cuda_error; }

namespace {
std::atomic<uint64_t> g_launches{0};
}

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }
uint64_t launch_count() { return g_launches.load(std::memory_order_relaxed); }

int ensure_dynamic_smem(const void* fn, size_t bytes) {
    static std::mutex mu;
    static std::map<std::pair<const void*, int>, size_t> done;
    int dev = 0;
    if (cuda_ok(cudaGetDevice(&dev), "cudaGetDevice") != PROX_OK) return PROX_ERR_CUDA;
    std::lock_guard<std::mutex> lock(mu);
    size_t& have = done[std::make_pair(fn, dev)];
    if (bytes <= have && have != 0) return PROX_OK;
    const cudaError_t err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 static_cast<int>(bytes));
    if (err != cudaSuccess) return cuda_fail(err, "raising a kernel's shared-memory limit");
    have = bytes;
    return PROX_OK;
}

// x_out[b][:] = y[b][:] / sqrt(mean(y[b]^2) + eps); one block per row, fixed-order sum.
__global__ void __launch_bounds__(256)
rmsnorm_kernel(const float* __restrict__ y, float* __restrict__ x_out, int d, float eps) {
    __shared__ float part[8];
    __shared__ float scale;
    const float* yr = y + static_cast<size_t>(blockIdx.x) * d;
    float* xr = x_out + static_cast<size_t>(blockIdx.x) * d;
    grid_dep_wait();
    grid_dep_launch();
    float s = 0.f;
    for (int i = threadIdx.x; i < d; i += 256) s = fmaf(yr[i], yr[i], s);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = s;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = 0.f;
        for (int w = 0; w < 8; ++w) t += part[w];
        scale = sqrtf(t / static_cast<float>(d) + eps);
    }
    __syncthreads();
    const float r = scale;
    for (int i = threadIdx.x; i < d; i += 256) xr[i] = yr[i] / r;
}

__global__ void iota_kernel(int32_t* __restrict__ out, int n, int rows) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n * rows) out[i] = i % n;
}

// Waits on a barrier that nothing completes; gives up after spin_cycles and records
// PROX_ERR_TIMEOUT. Exercises the same bounded wait the pipelined kernels use.
__global__ void wait_probe_kernel(int* __restrict__ status, long long spin_cycles) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        mbar_init_fence();
    }
    __syncthreads();
    if (threadIdx.x == 0) (void)mbar_wait(&bar, 0u, spin_cycles, status);
}

int launch_rmsnorm(const float* y, float* x_out, int batch, int d, float eps, cudaStream_t s) {
    rmsnorm_kernel<<<batch, 256, 0, s>>>(y, x_out, d, eps);
    const int rc = cuda_ok(cudaGetLastError(), "rmsnorm launch");
    if (rc == PROX_OK) count_launch();
    return rc;
}

int launch_iota(int32_t* out, int n, int rows, cudaStream_t s) {
    const int total = n * rows;
    iota_kernel<<<(total + 255) / 256, 256, 0, s>>>(out, n, rows);
    const int rc = cuda_ok(cudaGetLastError(), "index fill launch");
    if (rc == PROX_OK) count_launch();
    return rc;
}

int launch_wait_probe(int* status, long long spin_cycles, cudaStream_t s) {
    wait_probe_kernel<<<1, 32, 0, s>>>(status, spin_cycles);
    const int rc = cuda_ok(cudaGetLastError(), "wait probe launch");
    if (rc == PROX_OK) count_launch();
    return rc;
}

}  // namespace prox

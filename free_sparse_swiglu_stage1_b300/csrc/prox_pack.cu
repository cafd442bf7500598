// Offline packing of one SwiGLU FFN layer (Prox technical summary, Stage 1 "Input Sparsity &
// Quantization": INT4 proxy weights for the gate and up projections; Stage 2 "Exact
// Projections": the original bf16 weights of the selected channels).
//
//  pack_proxy_kernel      W_gate, W_up [F][d] bf16 -> codes [d][F] (gate nibble | up nibble
//                         << 4, each q + 8) and scales [d/128][F] (fp16 gate | fp16 up << 16).
//                         One block per (128-channel block, group): each thread quantizes
//                         one channel's 128 inputs into a shared tile, and the tile is
//                         written out input-major, one contiguous 128-byte run per input.
//  pack_rows_*_kernel     rows [F][3][d] bf16: W_gate[j,:], W_up[j,:], W_down[:,j] per
//                         channel; W_down is transposed through 32x32 shared tiles.
//  pack_fp8_*_kernel      the FP8 format's rows [F][3 d + 16] bytes: per channel the E4M3
//                         codes of W_gate[j,:], W_up[j,:], W_down[:,j], then their fp32
//                         scales (s = max |w| / 448, code = e4m3(w / s), round to nearest
//                         even, saturating) and a zero.
#include "prox_kernels.cuh"

namespace prox {

__global__ void __launch_bounds__(128)
pack_proxy_kernel(const uint16_t* __restrict__ w_gate, const uint16_t* __restrict__ w_up,
                  int d, int F, uint8_t* __restrict__ codes, uint32_t* __restrict__ scales) {
    __shared__ uint8_t tile[128][128 + 4];
    const int t = threadIdx.x;
    const int j = blockIdx.x * 128 + t;
    const int g = blockIdx.y;
    if (j < F) {
        uint32_t sbits = 0;
#pragma unroll 1
        for (int p = 0; p < 2; ++p) {
            const uint16_t* row = (p == 0 ? w_gate : w_up) + static_cast<size_t>(j) * d + g * 128;
            float a = 0.f;
            for (int i = 0; i < 128; i += 8) {
                const uint4 v = *reinterpret_cast<const uint4*>(row + i);
                const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int m = 0; m < 4; ++m)
                    a = fmaxf(a, fmaxf(fabsf(bf16lo(w4[m])), fabsf(bf16hi(w4[m]))));
            }
            // sw = fp16(fp32(a) / 7); q = clamp(rint(w / sw), -7, 7); q = 0 when sw == 0
            const __half sw = __float2half_rn(__fdiv_rn(a, 7.0f));
            const float swf = __half2float(sw);
            for (int i = 0; i < 128; i += 8) {
                const uint4 v = *reinterpret_cast<const uint4*>(row + i);
                const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    const float w = (m & 1) ? bf16hi(w4[m >> 1]) : bf16lo(w4[m >> 1]);
                    float q = 0.f;
                    if (swf != 0.f) q = fminf(7.f, fmaxf(-7.f, rintf(__fdiv_rn(w, swf))));
                    const uint32_t nib = static_cast<uint32_t>(static_cast<int>(q) + 8);
                    if (p == 0)
                        tile[i + m][t] = static_cast<uint8_t>(nib);
                    else
                        tile[i + m][t] = static_cast<uint8_t>(tile[i + m][t] | (nib << 4));
                }
            }
            sbits |= static_cast<uint32_t>(__half_as_ushort(sw)) << (16 * p);
        }
        scales[static_cast<size_t>(g) * F + j] = sbits;
    }
    __syncthreads();
    if (j < F) {
        for (int i = 0; i < 128; ++i)
            codes[static_cast<size_t>(g * 128 + i) * F + j] = tile[i][t];
    }
}

__global__ void __launch_bounds__(256)
pack_rows_gate_up_kernel(const uint16_t* __restrict__ w_gate, const uint16_t* __restrict__ w_up,
                         int d, uint16_t* __restrict__ rows) {
    const int j = blockIdx.x;   // one block per channel, 16-byte copies
    const uint4* sg = reinterpret_cast<const uint4*>(w_gate + static_cast<size_t>(j) * d);
    const uint4* su = reinterpret_cast<const uint4*>(w_up + static_cast<size_t>(j) * d);
    uint4* dst = reinterpret_cast<uint4*>(rows + static_cast<size_t>(j) * 3 * d);
    const int n = d / 8;
    for (int c = threadIdx.x; c < n; c += blockDim.x) {
        dst[c] = sg[c];
        dst[n + c] = su[c];
    }
}

__global__ void __launch_bounds__(1024)
pack_rows_down_kernel(const uint16_t* __restrict__ w_down, int d, int F,
                      uint16_t* __restrict__ rows) {
    __shared__ uint16_t tile[32][33];   // rows[j][2][i] = W_down[i][j]
    const int j0 = blockIdx.x * 32, i0 = blockIdx.y * 32;
    const int tx = threadIdx.x, ty = threadIdx.y;
    if (i0 + ty < d && j0 + tx < F) tile[ty][tx] = w_down[static_cast<size_t>(i0 + ty) * F + j0 + tx];
    __syncthreads();
    const int jj = j0 + ty, ii = i0 + tx;
    if (jj < F && ii < d) rows[(static_cast<size_t>(jj) * 3 + 2) * d + ii] = tile[tx][ty];
}

// E4M3 code of v (IEEE binary32): round to nearest even, saturating at +-448
__device__ __forceinline__ uint8_t to_e4m3(float v) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.f), "f"(v));
    return static_cast<uint8_t>(r & 0xFFu);   // the second source lands in the low byte
}

// one block per channel: the E4M3 codes and scales of W_gate[j,:] and W_up[j,:]
__global__ void __launch_bounds__(256)
pack_fp8_gate_up_kernel(const uint16_t* __restrict__ w_gate, const uint16_t* __restrict__ w_up,
                        int d, size_t row_bytes, uint8_t* __restrict__ rows8) {
    __shared__ float red[8];
    const int j = blockIdx.x, tid = threadIdx.x;
    uint8_t* run = rows8 + static_cast<size_t>(j) * row_bytes;
    for (int p = 0; p < 2; ++p) {
        const uint16_t* w = (p == 0 ? w_gate : w_up) + static_cast<size_t>(j) * d;
        float a = 0.f;
        for (int i = tid; i < d; i += 256) a = fmaxf(a, fabsf(__uint_as_float(static_cast<uint32_t>(w[i]) << 16)));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
        if ((tid & 31) == 0) red[tid >> 5] = a;
        __syncthreads();
        float amax = 0.f;
        for (int k = 0; k < 8; ++k) amax = fmaxf(amax, red[k]);
        const float sc = __fdiv_rn(amax, 448.0f);
        for (int i = tid; i < d; i += 256) {
            const float v = __uint_as_float(static_cast<uint32_t>(w[i]) << 16);
            run[static_cast<size_t>(p) * d + i] = sc != 0.f ? to_e4m3(__fdiv_rn(v, sc)) : 0;
        }
        if (tid == 0) reinterpret_cast<float*>(run + 3 * static_cast<size_t>(d))[p] = sc;
        __syncthreads();   // red is rewritten for the next row
    }
    if (tid == 0) reinterpret_cast<float*>(run + 3 * static_cast<size_t>(d))[3] = 0.f;
}

// one thread per channel j: the scale of W_down[:, j] (max over the column, coalesced rows)
__global__ void __launch_bounds__(256)
pack_fp8_down_scale_kernel(const uint16_t* __restrict__ w_down, int d, int F, size_t row_bytes,
                           uint8_t* __restrict__ rows8) {
    const int j = blockIdx.x * 256 + threadIdx.x;
    if (j >= F) return;
    float a = 0.f;
    for (int i = 0; i < d; ++i)
        a = fmaxf(a, fabsf(__uint_as_float(static_cast<uint32_t>(w_down[static_cast<size_t>(i) * F + j]) << 16)));
    reinterpret_cast<float*>(rows8 + static_cast<size_t>(j) * row_bytes + 3 * static_cast<size_t>(d))[2] =
        __fdiv_rn(a, 448.0f);
}

// the codes of W_down[:, j] through 32x32 shared tiles (after the scales are written)
__global__ void __launch_bounds__(1024)
pack_fp8_down_kernel(const uint16_t* __restrict__ w_down, int d, int F, size_t row_bytes,
                     uint8_t* __restrict__ rows8) {
    __shared__ float tile[32][33];
    const int j0 = blockIdx.x * 32, i0 = blockIdx.y * 32;
    const int tx = threadIdx.x, ty = threadIdx.y;
    if (i0 + ty < d && j0 + tx < F)
        tile[ty][tx] = __uint_as_float(static_cast<uint32_t>(w_down[static_cast<size_t>(i0 + ty) * F + j0 + tx]) << 16);
    __syncthreads();
    const int jj = j0 + ty, ii = i0 + tx;
    if (jj < F && ii < d) {
        uint8_t* run = rows8 + static_cast<size_t>(jj) * row_bytes;
        const float sc = reinterpret_cast<const float*>(run + 3 * static_cast<size_t>(d))[2];
        run[2 * static_cast<size_t>(d) + ii] = sc != 0.f ? to_e4m3(__fdiv_rn(tile[tx][ty], sc)) : 0;
    }
}

int launch_pack(const uint16_t* w_gate, const uint16_t* w_up, const uint16_t* w_down, int d,
                int F, const PackedLayout& L, uint8_t* base, cudaStream_t s) {
    uint8_t* codes = base + L.codes_off;
    uint32_t* scales = reinterpret_cast<uint32_t*>(base + L.scales_off);
    pack_proxy_kernel<<<dim3((F + 127) / 128, d / 128), 128, 0, s>>>(w_gate, w_up, d, F, codes,
                                                                     scales);
    if (L.format == PROX_FORMAT_FP8) {
        uint8_t* rows8 = base + L.rows_off;
        pack_fp8_gate_up_kernel<<<F, 256, 0, s>>>(w_gate, w_up, d, L.row_bytes, rows8);
        pack_fp8_down_scale_kernel<<<(F + 255) / 256, 256, 0, s>>>(w_down, d, F, L.row_bytes, rows8);
        pack_fp8_down_kernel<<<dim3((F + 31) / 32, (d + 31) / 32), dim3(32, 32), 0, s>>>(
            w_down, d, F, L.row_bytes, rows8);
    } else {
        uint16_t* rows = reinterpret_cast<uint16_t*>(base + L.rows_off);
        pack_rows_gate_up_kernel<<<F, 256, 0, s>>>(w_gate, w_up, d, rows);
        pack_rows_down_kernel<<<dim3((F + 31) / 32, (d + 31) / 32), dim3(32, 32), 0, s>>>(w_down, d,
                                                                                        F, rows);
    }
    const int rc = cuda_ok(cudaGetLastError(), "packing launch");
    if (rc == PROX_OK)
        for (int i = 0; i < (L.format == PROX_FORMAT_FP8 ? 4 : 3); ++i) count_launch();
    return rc;
}

}  // namespace prox

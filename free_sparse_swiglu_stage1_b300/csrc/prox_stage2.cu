// Prox Stage 2 ("Exact Sparse Computation" in the technical summary): for the selected
// channels only, exact gate and up projections from the bf16 weights, s = SiLU(g) * u, and
// the down projection over the same channels ("all three projections" sparse, abstract).
//
// stage2_kernel (one block per SM, persistent over a contiguous run of the channel list)
//   The packed rows put W_gate[j,:], W_up[j,:] and W_down[:,j] of channel j in one
//   contiguous 6*d-byte run, so a selected channel is ONE bulk copy (cp.async.bulk with an
//   mbarrier transaction count) from HBM into a shared-memory stage. One producer thread
//   keeps up to `nstage` channels in flight; the consumer warps own fixed 16-byte column
//   chunks, keep their activations x and their slice of the partial output y in
//   registers, and per batch of C channels
//     1. form the partial dot products of the gate and up rows with x,
//     2. reduce them across the block (warp butterfly, then a fixed-order sum of the warp
//        partials through shared memory),
//     3. s = SiLU(g) * u, zeroed for tokens that did not select the channel (batch path),
//     4. y += s * W_down[:, j] on their columns, then release the stages.
//   Every wait is bounded; a wait that runs out records PROX_ERR_TIMEOUT, the consumers
//   leave together (barrier with an OR reduction), and the producer drains its copies.
// reduce_kernel
//   Sums the per-block partial outputs in a fixed order, so y is bit-reproducible.
// The dense baseline is the same kernel over every channel (list == nullptr).
#include "prox_kernels.cuh"

namespace prox {

__device__ __forceinline__ int bar_red_or(int id, int n, int pred) {
    int r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.s32 q, %1, 0;\n\t"
        "bar.red.or.pred p, %2, %3, q;\n\t"
        "selp.s32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"(pred), "r"(id), "r"(n)
        : "memory");
    return r;
}

__device__ __forceinline__ void bar_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

__device__ __forceinline__ float dot8(const float (&x)[8], uint4 w) {
    float a = x[0] * bf16lo(w.x);
    a = fmaf(x[1], bf16hi(w.x), a);
    a = fmaf(x[2], bf16lo(w.y), a);
    a = fmaf(x[3], bf16hi(w.y), a);
    a = fmaf(x[4], bf16lo(w.z), a);
    a = fmaf(x[5], bf16hi(w.z), a);
    a = fmaf(x[6], bf16lo(w.w), a);
    a = fmaf(x[7], bf16hi(w.w), a);
    return a;
}

__device__ __forceinline__ void axpy8(float (&y)[8], float s, uint4 w) {
    y[0] = fmaf(s, bf16lo(w.x), y[0]);
    y[1] = fmaf(s, bf16hi(w.x), y[1]);
    y[2] = fmaf(s, bf16lo(w.y), y[2]);
    y[3] = fmaf(s, bf16hi(w.y), y[3]);
    y[4] = fmaf(s, bf16lo(w.z), y[4]);
    y[5] = fmaf(s, bf16hi(w.z), y[5]);
    y[6] = fmaf(s, bf16lo(w.w), y[6]);
    y[7] = fmaf(s, bf16hi(w.w), y[7]);
}

template <int TB, int CPT, int C>
__global__ void __launch_bounds__(TB == 4 ? 288 : 544)
stage2_kernel(const uint16_t* __restrict__ rows, int d, int F, const float* __restrict__ x, int nb,
              const int32_t* __restrict__ list, const uint32_t* __restrict__ lbits,
              const int* __restrict__ count_dev, int count_host, float* __restrict__ ypart,
              int nstage, long long spin, int* __restrict__ status) {
    extern __shared__ __align__(128) unsigned char smem[];
    constexpr int V = 2 * C * TB;
    const int NT = blockDim.x - 32, NW = NT >> 5;
    const uint32_t stage_bytes = 6u * static_cast<uint32_t>(d);
    unsigned char* stages = smem;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(nstage) * stage_bytes);
    uint64_t* empty = full + nstage;
    float* red = reinterpret_cast<float*>(empty + nstage);   // [2][NW][V]
    float* ssm = red + 2 * NW * V;                           // [2][C*TB]
    volatile int* abort_flag = reinterpret_cast<volatile int*>(ssm + 2 * C * TB);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    if (tid == 0) {
        for (int i = 0; i < nstage; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], NW);
        }
        *abort_flag = 0;
        mbar_init_fence();
    }
    __syncthreads();
    grid_dep_wait();   // the channel list and the activations come from earlier kernels

    const int n = count_dev ? *count_dev : count_host;
    const int P = gridDim.x;
    const int e0 = static_cast<int>(static_cast<long long>(n) * blockIdx.x / P);
    const int e1 = static_cast<int>(static_cast<long long>(n) * (blockIdx.x + 1) / P);

    if (warp == NW) {
        // ---------------------------------------------------------------- producer
        if (lane == 0) {
            int it = 0;
            for (int e = e0; e < e1; ++e, ++it) {
                const int st = it % nstage;
                if (it >= nstage &&
                    !mbar_wait(&empty[st], static_cast<uint32_t>((it / nstage) - 1) & 1u, spin, status)) {
                    *abort_flag = 1;
                    break;
                }
                if (*abort_flag) break;
                int j = list ? list[e] : e;
                if (j < 0 || j >= F) {
                    set_status(status, PROX_ERR_BOUNDS);
                    j = 0;
                }
                mbar_arrive_expect_tx(&full[st], stage_bytes);
                bulk_g2s(stages + static_cast<size_t>(st) * stage_bytes,
                         rows + static_cast<size_t>(j) * 3 * d, stage_bytes, &full[st]);
            }
            if (*abort_flag) {
                // copies still in flight must land before the block's shared memory is freed
                for (int t = it > nstage ? it - nstage : 0; t < it; ++t)
                    mbar_wait(&full[t % nstage], static_cast<uint32_t>(t / nstage) & 1u, spin, status);
            }
        }
        return;
    }

    // -------------------------------------------------------------------- consumers
    const int nchunk = d >> 3;
    float xr[TB][CPT][8], yr[TB][CPT][8];
#pragma unroll
    for (int c = 0; c < CPT; ++c) {
        const int q = c * NT + tid;
#pragma unroll
        for (int b = 0; b < TB; ++b) {
            float4 a = make_float4(0.f, 0.f, 0.f, 0.f), bb = a;
            if (b < nb && q < nchunk) {
                const float4* src = reinterpret_cast<const float4*>(x + static_cast<size_t>(b) * d + q * 8);
                a = src[0];
                bb = src[1];
            }
            xr[b][c][0] = a.x; xr[b][c][1] = a.y; xr[b][c][2] = a.z; xr[b][c][3] = a.w;
            xr[b][c][4] = bb.x; xr[b][c][5] = bb.y; xr[b][c][6] = bb.z; xr[b][c][7] = bb.w;
#pragma unroll
            for (int m = 0; m < 8; ++m) yr[b][c][m] = 0.f;
        }
    }

    int buf = 0;
    for (int eb = e0; eb < e1; eb += C) {
        const int cn = min(C, e1 - eb);
        float vals[V];
        bool ok = true;
#pragma unroll
        for (int cb = 0; cb < C; ++cb) {
            float gp[TB], up[TB];
#pragma unroll
            for (int b = 0; b < TB; ++b) gp[b] = up[b] = 0.f;
            if (cb < cn) {
                const int it = eb + cb - e0;
                const int st = it % nstage;
                ok = ok && mbar_wait(&full[st], static_cast<uint32_t>(it / nstage) & 1u, spin, status);
                const uint16_t* sb = reinterpret_cast<const uint16_t*>(stages + static_cast<size_t>(st) * stage_bytes);
#pragma unroll
                for (int c = 0; c < CPT; ++c) {
                    const int q = c * NT + tid;
                    if (q < nchunk) {
                        const uint4 wg = *reinterpret_cast<const uint4*>(sb + q * 8);
                        const uint4 wu = *reinterpret_cast<const uint4*>(sb + d + q * 8);
#pragma unroll
                        for (int b = 0; b < TB; ++b) {
                            gp[b] += dot8(xr[b][c], wg);
                            up[b] += dot8(xr[b][c], wu);
                        }
                    }
                }
            }
#pragma unroll
            for (int b = 0; b < TB; ++b) {
                vals[(cb * TB + b) * 2] = gp[b];
                vals[(cb * TB + b) * 2 + 1] = up[b];
            }
        }
#pragma unroll
        for (int v = 0; v < V; ++v)
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) vals[v] += __shfl_xor_sync(0xffffffffu, vals[v], o);
        if (lane == 0) {
#pragma unroll
            for (int v = 0; v < V; ++v) red[(buf * NW + warp) * V + v] = vals[v];
        }
        if (bar_red_or(1, NT, !ok)) {
            if (tid == 0) *abort_flag = 1;
            break;
        }
        if (tid < C * TB) {
            const int cb = tid / TB, b = tid % TB;
            float g = 0.f, u = 0.f;
            for (int w2 = 0; w2 < NW; ++w2) {
                g += red[(buf * NW + w2) * V + 2 * tid];
                u += red[(buf * NW + w2) * V + 2 * tid + 1];
            }
            float sv = 0.f;
            if (cb < cn && b < nb) {
                const uint32_t bits = lbits ? lbits[eb + cb] : 0xffffffffu;
                if ((bits >> b) & 1u) sv = silu_f(g) * u;
            }
            ssm[buf * C * TB + tid] = sv;
        }
        bar_sync(1, NT);
#pragma unroll
        for (int cb = 0; cb < C; ++cb) {
            if (cb < cn) {
                const int it = eb + cb - e0;
                const int st = it % nstage;
                const uint16_t* sb = reinterpret_cast<const uint16_t*>(stages + static_cast<size_t>(st) * stage_bytes);
                float sv[TB];
#pragma unroll
                for (int b = 0; b < TB; ++b) sv[b] = ssm[buf * C * TB + cb * TB + b];
#pragma unroll
                for (int c = 0; c < CPT; ++c) {
                    const int q = c * NT + tid;
                    if (q < nchunk) {
                        const uint4 wd = *reinterpret_cast<const uint4*>(sb + 2 * d + q * 8);
#pragma unroll
                        for (int b = 0; b < TB; ++b) axpy8(yr[b][c], sv[b], wd);
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) {
            for (int cb = 0; cb < cn; ++cb) mbar_arrive(&empty[(eb + cb - e0) % nstage]);
        }
        buf ^= 1;
    }

    float* yp = ypart + static_cast<size_t>(blockIdx.x) * TB * d;
#pragma unroll
    for (int c = 0; c < CPT; ++c) {
        const int q = c * NT + tid;
        if (q < nchunk) {
#pragma unroll
            for (int b = 0; b < TB; ++b) {
                float4* dst = reinterpret_cast<float4*>(yp + static_cast<size_t>(b) * d + q * 8);
                dst[0] = make_float4(yr[b][c][0], yr[b][c][1], yr[b][c][2], yr[b][c][3]);
                dst[1] = make_float4(yr[b][c][4], yr[b][c][5], yr[b][c][6], yr[b][c][7]);
            }
        }
    }
    grid_dep_launch();
}

// y[b][:] = sum over blocks p (fixed order) of ypart[p][b][:]
__global__ void __launch_bounds__(256)
reduce_kernel(const float4* __restrict__ ypart, int P, int TB, int d, float4* __restrict__ y) {
    __shared__ float4 sm[8][32];
    const int cx = threadIdx.x & 31, pg = threadIdx.x >> 5;
    const int n4 = d >> 2;
    const int col = blockIdx.x * 32 + cx;
    const int b = blockIdx.y;
    grid_dep_wait();
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (col < n4) {
        for (int p = pg; p < P; p += 8) {
            const float4 v = __ldcg(&ypart[(static_cast<size_t>(p) * TB + b) * n4 + col]);
            acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
        }
    }
    sm[pg][cx] = acc;
    __syncthreads();
    if (pg == 0 && col < n4) {
        float4 t = sm[0][cx];
#pragma unroll
        for (int g = 1; g < 8; ++g) {
            t.x += sm[g][cx].x; t.y += sm[g][cx].y; t.z += sm[g][cx].z; t.w += sm[g][cx].w;
        }
        y[static_cast<size_t>(b) * n4 + col] = t;
    }
    grid_dep_launch();
}

template <int TB, int CPT, int C>
static int launch_stage2_t(const uint16_t* rows, int d, int F, const float* x, int nb,
                           const int32_t* list, const uint32_t* lbits, const int* count_dev,
                           int count_host, float* ypart, int nstage, int P, int* status,
                           cudaStream_t s) {
    const int NT = stage2_consumers(d);
    const int NW = NT / 32;
    const size_t smem = static_cast<size_t>(nstage) * 6 * d + 2 * nstage * sizeof(uint64_t) +
                        (2 * NW * 2 * C * TB + 2 * C * TB) * sizeof(float) + 16;
    auto fn = stage2_kernel<TB, CPT, C>;
    if (cudaFuncSetAttribute(reinterpret_cast<const void*>(fn),
                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem)) != cudaSuccess)
        return PROX_ERR_CUDA;
    fn<<<P, NT + 32, smem, s>>>(rows, d, F, x, nb, list, lbits, count_dev, count_host, ypart,
                                nstage, kDefaultSpinCycles, status);
    return cudaGetLastError() == cudaSuccess ? PROX_OK : PROX_ERR_CUDA;
}

template <int TB, int CPT>
static int launch_stage2_c(int C, const uint16_t* rows, int d, int F, const float* x, int nb,
                           const int32_t* list, const uint32_t* lbits, const int* count_dev,
                           int count_host, float* ypart, int nstage, int P, int* status,
                           cudaStream_t s) {
    if (C >= 4)
        return launch_stage2_t<TB, CPT, 4>(rows, d, F, x, nb, list, lbits, count_dev, count_host,
                                           ypart, nstage, P, status, s);
    if (C >= 2)
        return launch_stage2_t<TB, CPT, 2>(rows, d, F, x, nb, list, lbits, count_dev, count_host,
                                           ypart, nstage, P, status, s);
    return launch_stage2_t<TB, CPT, 1>(rows, d, F, x, nb, list, lbits, count_dev, count_host,
                                       ypart, nstage, P, status, s);
}

template <int TB>
static int launch_stage2_cpt(int cpt, int C, const uint16_t* rows, int d, int F, const float* x,
                             int nb, const int32_t* list, const uint32_t* lbits,
                             const int* count_dev, int count_host, float* ypart, int nstage,
                             int P, int* status, cudaStream_t s) {
    if (cpt == 1)
        return launch_stage2_c<TB, 1>(C, rows, d, F, x, nb, list, lbits, count_dev, count_host,
                                      ypart, nstage, P, status, s);
    if (cpt == 2)
        return launch_stage2_c<TB, 2>(C, rows, d, F, x, nb, list, lbits, count_dev, count_host,
                                      ypart, nstage, P, status, s);
    return launch_stage2_c<TB, 4>(C, rows, d, F, x, nb, list, lbits, count_dev, count_host, ypart,
                                  nstage, P, status, s);
}

int launch_stage2(const uint8_t* packed, const PackedLayout& L, int d, int F, const float* x_tile,
                  int nb, const int32_t* list, const uint32_t* lbits, const int* count_dev,
                  int count_host, float* y_tile, uint8_t* ws, const WsLayout& W, int sms,
                  cudaStream_t s) {
    const uint16_t* rows = reinterpret_cast<const uint16_t*>(packed + L.rows_off);
    float* ypart = reinterpret_cast<float*>(ws + W.ypart);
    int* status = &reinterpret_cast<Control*>(ws + W.control)->status;
    const int nstage = stage2_nstage(d);
    const int C = stage2_batch(nstage);
    const int cpt = stage2_cpt(d);
    const int TB = nb <= 1 ? 1 : (nb <= 2 ? 2 : 4);
    const int P = W.P < sms ? W.P : sms;
    int rc;
    if (TB == 1)
        rc = launch_stage2_cpt<1>(cpt, C, rows, d, F, x_tile, nb, list, lbits, count_dev,
                                  count_host, ypart, nstage, P, status, s);
    else if (TB == 2)
        rc = launch_stage2_cpt<2>(cpt, C, rows, d, F, x_tile, nb, list, lbits, count_dev,
                                  count_host, ypart, nstage, P, status, s);
    else
        rc = launch_stage2_cpt<4>(cpt, C, rows, d, F, x_tile, nb, list, lbits, count_dev,
                                  count_host, ypart, nstage, P, status, s);
    if (rc != PROX_OK) return rc;
    const int n4 = d / 4;
    reduce_kernel<<<dim3((n4 + 31) / 32, nb), 256, 0, s>>>(reinterpret_cast<const float4*>(ypart), P,
                                                          TB, d, reinterpret_cast<float4*>(y_tile));
    return cudaGetLastError() == cudaSuccess ? PROX_OK : PROX_ERR_CUDA;
}

}  // namespace prox

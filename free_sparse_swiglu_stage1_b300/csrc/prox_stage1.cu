// Prox Stage 1 ("Lightweight Proxy Construction" in the technical summary): input sparsity,
// INT4 proxy projections of W_gate and W_up over the kept inputs only, and the salience
// |SiLU(g~) * u~| of every intermediate channel.
//
// input_quant_kernel (one block per tile of tokens)
//   For each token: radix-select the k_in largest |x_i| (ties to the lower index), then per
//   group of 128 inputs sx = max|x_hat| / 127 and qx = clamp(rint(x_hat / sx), -127, 127)
//   in binary32. The union of the tile's kept inputs becomes an ascending row list; each
//   row carries its tokens' int8 codes packed in one 32-bit word, and gstart[g] marks where
//   group g starts in the list.
//
// stage1_kernel (grid: 128-channel blocks x S slices of the row list, 8 warps per block)
//   The "fused split-N" design: a block owns 128 channels and a slice of the kept rows;
//   a kept input is one contiguous 128-byte run of codes (gate | up nibbles of 128
//   channels), read by one warp with one 32-bit load per lane, so rejected inputs cost
//   no bytes. Lane l owns channels 4l..4l+3 of both projections.
//   The int4 x int8 products are accumulated exactly in two 16-bit lanes of a 32-bit
//   register: the nibble pairs (0,4), (1,5), (2,6), (3,7) of a code word are isolated with
//   one mask each and multiplied by the activation code in a single integer multiply-add.
//   With codes in [0, 15] and |qx| <= 127, sixteen rows fit in a signed 16-bit lane
//   (16 * 15 * 127 = 30480 < 32768); every 16 rows the lanes are moved into int32
//   accumulators. Codes are stored as q + 8, so the group result is corrected by
//   -8 * sum(qx) over the same rows, which keeps every integer exact.
//   At each group end the exact integer A is scaled by sx * sw and added to a double-float
//   (hi, lo) sum, so g~ and u~ carry about 44 significant bits before the final fp32
//   rounding. Warps, then row slices, are combined in a fixed order (the last block to
//   finish a channel block does the final sum), so the result is deterministic.
#include "prox_kernels.cuh"

namespace prox {

constexpr int kSelThreads = 1024;
constexpr int kS1Threads = 256;
constexpr int kS1Warps = kS1Threads / 32;
constexpr int kRowsPerFlush = 16;

__global__ void __launch_bounds__(kSelThreads)
input_quant_kernel(const float* __restrict__ x, int d, int nb, int TB, int k_in,
                   int* __restrict__ rows, uint32_t* __restrict__ qxt, float* __restrict__ sx_ws,
                   int* __restrict__ gstart, int8_t* __restrict__ dbg_qx,
                   float* __restrict__ dbg_sx) {
    extern __shared__ __align__(16) unsigned char smem[];
    float* xs = reinterpret_cast<float*>(smem);
    uint32_t* keys = reinterpret_cast<uint32_t*>(xs + d);
    int8_t* qx8 = reinterpret_cast<int8_t*>(keys + d);
    uint8_t* kflag = reinterpret_cast<uint8_t*>(qx8 + TB * d);
    __shared__ int hist[256], sel[4], scan[32];
    constexpr int NT = kSelThreads, NW = NT / 32;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = d >> 7;
    const int per = (d + NT - 1) / NT;
    const int lo = min(d, tid * per), hi = min(d, lo + per);

    grid_dep_wait();
    for (int i = tid; i < d; i += NT) kflag[i] = 0;
    for (int i = tid; i < TB * d; i += NT) qx8[i] = 0;
    __syncthreads();

    for (int b = 0; b < nb; ++b) {
        for (int i = tid; i < d; i += NT) {
            const float v = x[static_cast<size_t>(b) * d + i];
            xs[i] = v;
            keys[i] = __float_as_uint(v) & 0x7fffffffu;
        }
        __syncthreads();
        uint32_t T;
        int take;
        block_radix_select<NT>(keys, d, k_in, hist, sel, T, take);
        // mark the kept inputs, walking contiguous runs so equal keys go to lower indices
        int eq = 0;
        for (int i = lo; i < hi; ++i) eq += keys[i] == T;
        int eq_total;
        int e = block_exclusive_scan<NT>(eq, scan, eq_total);
        for (int i = lo; i < hi; ++i) {
            const uint32_t kk = keys[i];
            bool keep = kk > T;
            if (kk == T) { keep = e < take; ++e; }
            if (keep) kflag[i] |= static_cast<uint8_t>(1u << b);
        }
        __syncthreads();
        // per-group scale and int8 codes of the kept inputs
        for (int g = warp; g < G; g += NW) {
            float xv[4];
            bool kp[4];
            float m = 0.f;
#pragma unroll
            for (int mm = 0; mm < 4; ++mm) {
                const int i = g * 128 + lane * 4 + mm;
                xv[mm] = xs[i];
                kp[mm] = (kflag[i] >> b) & 1;
                if (kp[mm]) m = fmaxf(m, fabsf(xv[mm]));
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
            const float sxg = __fdiv_rn(m, 127.0f);
#pragma unroll
            for (int mm = 0; mm < 4; ++mm) {
                const int i = g * 128 + lane * 4 + mm;
                float q = 0.f;
                if (kp[mm] && sxg != 0.f)
                    q = fminf(127.f, fmaxf(-127.f, rintf(__fdiv_rn(xv[mm], sxg))));
                const int8_t qi = static_cast<int8_t>(static_cast<int>(q));
                qx8[b * d + i] = qi;
                if (dbg_qx) dbg_qx[static_cast<size_t>(b) * d + i] = qi;
            }
            if (lane == 0) {
                sx_ws[b * G + g] = sxg;
                if (dbg_sx) dbg_sx[b * G + g] = sxg;
            }
        }
        __syncthreads();
    }
    for (int i = tid; i < (TB - nb) * G; i += NT) sx_ws[nb * G + i] = 0.f;

    // ascending union of the kept inputs, with the tile's codes packed per row
    int cnt = 0;
    for (int i = lo; i < hi; ++i) cnt += kflag[i] != 0;
    int total;
    int pos = block_exclusive_scan<NT>(cnt, scan, total);
    for (int i = lo; i < hi; ++i) {
        if ((i & 127) == 0) gstart[i >> 7] = pos;
        if (kflag[i]) {
            uint32_t w = 0;
            for (int b = 0; b < TB; ++b)
                w |= static_cast<uint32_t>(static_cast<uint8_t>(qx8[b * d + i])) << (8 * b);
            rows[pos] = i;
            qxt[pos] = w;
            ++pos;
        }
    }
    if (tid == 0) {
        gstart[G] = total;
        gstart[G + 1] = total;
    }
    grid_dep_launch();
}

// Moves the two signed 16-bit lanes of a packed accumulator into int32 sums.
__device__ __forceinline__ void unpack_lanes(uint32_t p, int& lo_acc, int& hi_acc) {
    const int lo = static_cast<int>(static_cast<int16_t>(p & 0xFFFFu));
    const int hi = static_cast<int>(p - static_cast<uint32_t>(lo)) >> 16;
    lo_acc += lo;
    hi_acc += hi;
}

template <int TB>
__global__ void __launch_bounds__(kS1Threads)
stage1_kernel(const uint8_t* __restrict__ codes, const uint32_t* __restrict__ scales, int d, int F,
              const int* __restrict__ rows, const uint32_t* __restrict__ qxt,
              const float* __restrict__ sx, const int* __restrict__ gstart, int S, int nb,
              float2* __restrict__ part, int* __restrict__ cnt, float* __restrict__ sigma,
              int32_t* __restrict__ dbg_gate, int32_t* __restrict__ dbg_up, int* __restrict__ status) {
    extern __shared__ __align__(16) unsigned char smem[];
    DF* red = reinterpret_cast<DF*>(smem);                        // [warps][TB][8][32]
    float* gu = reinterpret_cast<float*>(smem);                   // [TB][8][32] (reused)
    __shared__ int last_flag;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = d >> 7;
    const int blk = blockIdx.x, s = blockIdx.y;
    const int j0 = blk * 128 + lane * 4;
    const bool valid = j0 < F;

    grid_dep_wait();
    const int nrows = gstart[G];
    const int ra = static_cast<int>(static_cast<long long>(nrows) * s / S);
    const int rb = static_cast<int>(static_cast<long long>(nrows) * (s + 1) / S);
    const int m = rb - ra;
    const int wa = ra + static_cast<int>(static_cast<long long>(m) * warp / kS1Warps);
    const int wb = ra + static_cast<int>(static_cast<long long>(m) * (warp + 1) / kS1Warps);
    const uint8_t* cbase = codes + (valid ? j0 : 0);

    DF acc[TB][8];
#pragma unroll
    for (int b = 0; b < TB; ++b)
#pragma unroll
        for (int v = 0; v < 8; ++v) acc[b][v] = DF{0.f, 0.f};

    int r = wa;
    while (r < wb) {
        const int g = rows[r] >> 7;
        const int gend = min(wb, gstart[g + 1]);
        if (g >= G || gend <= r) {   // inconsistent row list: record it, never spin
            if (lane == 0) set_status(status, PROX_ERR_BOUNDS);
            break;
        }
        int A[TB][8];
        int qs[TB];
#pragma unroll
        for (int b = 0; b < TB; ++b) {
            qs[b] = 0;
#pragma unroll
            for (int v = 0; v < 8; ++v) A[b][v] = 0;
        }
        for (int c = r; c < gend; c += kRowsPerFlush) {
            const int n = min(kRowsPerFlush, gend - c);
            int myrow = 0;
            uint32_t myq = 0;
            if (lane < n) {
                myrow = rows[c + lane];
                myq = qxt[c + lane];
            }
            uint32_t w[kRowsPerFlush];
#pragma unroll
            for (int u = 0; u < kRowsPerFlush; ++u) {
                const int ri = __shfl_sync(0xffffffffu, myrow, u);
                w[u] = (u < n && valid)
                           ? __ldg(reinterpret_cast<const uint32_t*>(cbase + static_cast<size_t>(ri) * F))
                           : 0u;
            }
            uint32_t P[TB][4];
#pragma unroll
            for (int b = 0; b < TB; ++b)
#pragma unroll
                for (int k = 0; k < 4; ++k) P[b][k] = 0u;
#pragma unroll
            for (int u = 0; u < kRowsPerFlush; ++u) {
                const uint32_t qq = __shfl_sync(0xffffffffu, myq, u);
                const uint32_t e0 = w[u] & 0x000F000Fu;          // gate c0 | gate c2
                const uint32_t e1 = (w[u] >> 4) & 0x000F000Fu;   // up   c0 | up   c2
                const uint32_t e2 = (w[u] >> 8) & 0x000F000Fu;   // gate c1 | gate c3
                const uint32_t e3 = (w[u] >> 12) & 0x000F000Fu;  // up   c1 | up   c3
#pragma unroll
                for (int b = 0; b < TB; ++b) {
                    const int q = static_cast<int>(static_cast<int8_t>(qq >> (8 * b)));
                    const uint32_t uq = static_cast<uint32_t>(q);
                    P[b][0] += e0 * uq;
                    P[b][1] += e1 * uq;
                    P[b][2] += e2 * uq;
                    P[b][3] += e3 * uq;
                    qs[b] += q;
                }
            }
#pragma unroll
            for (int b = 0; b < TB; ++b) {
                unpack_lanes(P[b][0], A[b][0], A[b][2]);
                unpack_lanes(P[b][1], A[b][4], A[b][6]);
                unpack_lanes(P[b][2], A[b][1], A[b][3]);
                unpack_lanes(P[b][3], A[b][5], A[b][7]);
            }
        }
        // group end: A - 8*sum(qx) is the exact integer proxy product over these rows
        if (valid) {
            const uint4 sw4 = __ldg(reinterpret_cast<const uint4*>(scales + static_cast<size_t>(g) * F + j0));
            const uint32_t swv[4] = {sw4.x, sw4.y, sw4.z, sw4.w};
#pragma unroll
            for (int b = 0; b < TB; ++b) {
                const float sxb = sx[b * G + g];
#pragma unroll
                for (int c4 = 0; c4 < 4; ++c4) {
                    const int ag = A[b][c4] - 8 * qs[b];
                    const int au = A[b][4 + c4] - 8 * qs[b];
                    const float swg = __half2float(__ushort_as_half(static_cast<unsigned short>(swv[c4] & 0xFFFFu)));
                    const float swu = __half2float(__ushort_as_half(static_cast<unsigned short>(swv[c4] >> 16)));
                    acc[b][c4] = df_add(acc[b][c4], df_scaled_int(sxb, swg, ag));
                    acc[b][4 + c4] = df_add(acc[b][4 + c4], df_scaled_int(sxb, swu, au));
                    if (dbg_gate && b < nb) atomicAdd(&dbg_gate[(static_cast<size_t>(b) * G + g) * F + j0 + c4], ag);
                    if (dbg_up && b < nb) atomicAdd(&dbg_up[(static_cast<size_t>(b) * G + g) * F + j0 + c4], au);
                }
            }
        }
        r = gend;
    }

    // combine the 8 warps in a fixed order
#pragma unroll
    for (int b = 0; b < TB; ++b)
#pragma unroll
        for (int v = 0; v < 8; ++v) red[((warp * TB + b) * 8 + v) * 32 + lane] = acc[b][v];
    __syncthreads();
    {
        const int v = warp;   // 8 warps <-> 8 values (gate c0..c3, up c0..c3)
        const int j = j0 + (v & 3);
#pragma unroll
        for (int b = 0; b < TB; ++b) {
            DF t = red[((0 * TB + b) * 8 + v) * 32 + lane];
            for (int w2 = 1; w2 < kS1Warps; ++w2) t = df_add(t, red[((w2 * TB + b) * 8 + v) * 32 + lane]);
            if (valid)
                part[((static_cast<size_t>(s) * TB + b) * F + j) * 2 + (v >> 2)] = make_float2(t.hi, t.lo);
        }
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) last_flag = atomicAdd(&cnt[blk], 1) == S - 1;
    __syncthreads();
    if (!last_flag) {
        grid_dep_launch();
        return;
    }
    __threadfence();
    {
        const int v = warp;
        const int j = j0 + (v & 3);
#pragma unroll
        for (int b = 0; b < TB; ++b) {
            DF t{0.f, 0.f};
            if (valid) {
                for (int s2 = 0; s2 < S; ++s2) {
                    const float2 p = __ldcg(&part[((static_cast<size_t>(s2) * TB + b) * F + j) * 2 + (v >> 2)]);
                    t = df_add(t, DF{p.x, p.y});
                }
            }
            gu[(b * 8 + v) * 32 + lane] = t.hi + t.lo;
        }
    }
    __syncthreads();
    if (warp < 4 && valid) {
        const int j = j0 + warp;
        for (int b = 0; b < nb; ++b) {
            const float gt = gu[(b * 8 + warp) * 32 + lane];
            const float ut = gu[(b * 8 + 4 + warp) * 32 + lane];
            sigma[static_cast<size_t>(b) * F + j] = fabsf(silu_f(gt) * ut);
        }
    }
    if (tid == 0) cnt[blk] = 0;
    grid_dep_launch();
}

static int set_smem(const void* fn, size_t bytes) {
    if (bytes <= 48 * 1024) return PROX_OK;
    return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                static_cast<int>(bytes)) == cudaSuccess
               ? PROX_OK
               : PROX_ERR_CUDA;
}

int launch_input_quant(const float* x, int d, int nb, int k_in, uint8_t* ws, const WsLayout& W,
                       int8_t* dbg_qx, float* dbg_sx, cudaStream_t s) {
    const size_t smem = static_cast<size_t>(d) * 9 + static_cast<size_t>(W.TB) * d;
    if (set_smem(reinterpret_cast<const void*>(input_quant_kernel), smem) != PROX_OK) return PROX_ERR_CUDA;
    input_quant_kernel<<<1, kSelThreads, smem, s>>>(
        x, d, nb, W.TB, k_in, reinterpret_cast<int*>(ws + W.rows),
        reinterpret_cast<uint32_t*>(ws + W.qxt), reinterpret_cast<float*>(ws + W.sx),
        reinterpret_cast<int*>(ws + W.gstart), dbg_qx, dbg_sx);
    return cudaGetLastError() == cudaSuccess ? PROX_OK : PROX_ERR_CUDA;
}

template <int TB>
static int launch_stage1_t(const uint8_t* packed, const PackedLayout& L, int d, int F, int nb,
                           int S, uint8_t* ws, const WsLayout& W, float* sigma_tile,
                           int32_t* dbg_gate, int32_t* dbg_up, cudaStream_t s) {
    const size_t smem = static_cast<size_t>(kS1Warps) * TB * 8 * 32 * sizeof(DF);
    auto fn = stage1_kernel<TB>;
    if (set_smem(reinterpret_cast<const void*>(fn), smem) != PROX_OK) return PROX_ERR_CUDA;
    fn<<<dim3(W.nblk, S), kS1Threads, smem, s>>>(
        packed + L.codes_off, reinterpret_cast<const uint32_t*>(packed + L.scales_off), d, F,
        reinterpret_cast<const int*>(ws + W.rows), reinterpret_cast<const uint32_t*>(ws + W.qxt),
        reinterpret_cast<const float*>(ws + W.sx), reinterpret_cast<const int*>(ws + W.gstart), S,
        nb, reinterpret_cast<float2*>(ws + W.s1part), reinterpret_cast<int*>(ws + W.s1_cnt),
        sigma_tile, dbg_gate, dbg_up, &reinterpret_cast<Control*>(ws + W.control)->status);
    return cudaGetLastError() == cudaSuccess ? PROX_OK : PROX_ERR_CUDA;
}

int launch_stage1(const uint8_t* packed, const PackedLayout& L, int d, int F, int nb, int k_in,
                  uint8_t* ws, const WsLayout& W, float* sigma_tile, int32_t* dbg_gate,
                  int32_t* dbg_up, int sms, cudaStream_t s) {
    const int nrows_est = nb * k_in < d ? nb * k_in : d;
    int S = stage1_splits(W.nblk, nrows_est, sms);
    if (S > W.S_max) S = W.S_max;
    // the narrowest instantiation that holds the tile's tokens
    if (nb <= 1) return launch_stage1_t<1>(packed, L, d, F, nb, S, ws, W, sigma_tile, dbg_gate, dbg_up, s);
    if (nb <= 2) return launch_stage1_t<2>(packed, L, d, F, nb, S, ws, W, sigma_tile, dbg_gate, dbg_up, s);
    return launch_stage1_t<4>(packed, L, d, F, nb, S, ws, W, sigma_tile, dbg_gate, dbg_up, s);
}

}  // namespace prox

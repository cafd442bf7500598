// Prox Stage 1 ("Lightweight Proxy Construction" in the technical summary): input sparsity,
// INT4 proxy projections of W_gate and W_up over the kept inputs only, and the salience
// |SiLU(g~) * u~| of every intermediate channel.
//
// input_quant_kernel (one block of 1024 threads per tile of tokens)
//   For each token: a three-pass radix select finds the k_in-th largest |x_i| (ties to the
//   lower index); then per group of 128 inputs sx = max|x_hat| / 127 and
//   qx = clamp(rint(x_hat / sx), -127, 127) in binary32. Per group, the inputs any token of
//   the tile kept are listed in ascending order (padded to a multiple of 4 with copies of the
//   last one, whose codes are 0) with every token's int8 codes; no global compaction is
//   needed, since each group's list has a fixed place.
//
// stage1_kernel (grid: channel tiles x slices of consecutive groups x token tiles, 8 warps
// per block)
//   The "fused split-N" design: a block owns a tile of 32 * CPL channels and the kept rows
//   of a few groups; a kept input is one contiguous run of CPL bytes per lane (gate | up
//   nibbles of CPL channels), so rejected inputs cost no bytes and a warp reads a row with
//   one wide load per lane. The rows are taken four at a time (a quad never crosses a
//   group): the four loaded words of each 4-channel column are transposed with byte
//   permutes, so each channel's codes of the four rows sit in one word, and one dp4a per
//   channel and projection multiplies them by the four rows' int8 codes. Gate codes enter as
//   bytes q + 8 in [1, 15], up codes as 16 * (q + 8), and one more dp4a accumulates 8 * sum(qx)
//   of the rows, so A = sum(q * qx) is recovered exactly per group in int32.
//   At each group end the exact integer A is scaled by sx * sw and added to a double-float
//   (hi, lo) sum in shared memory, so g~ and u~ carry about 44 significant bits before the
//   final fp32 rounding. Warps, then group slices, are combined in a fixed order (the last
//   block to finish a channel tile does the final sum and the salience), so the result is
//   deterministic. That block also counts the salience's top 11 bits into a histogram the
//   top-k starts from.
#include <cooperative_groups.h>

#include "prox_kernels.cuh"

namespace prox {

constexpr int kSelThreads = 1024;
constexpr int kS1Threads = 256;
constexpr int kS1Warps = kS1Threads / 32;

// Input selection and activation codes (see the file comment); block z handles token tile z
// (tokens z*TB .. z*TB + nb - 1 of the B). Thread t owns the run of inputs
// [t*RUN, t*RUN + RUN), RUN a power of two in [4, 16], so a run lies inside one group of 128
// and a group's runs are 128/RUN aligned lanes of one warp. Outputs per tile: grows [G][128],
// gcnt [G], gq [G + 1], gqx [TB][G][128] (TBs rows written: the Stage-1 kernel's token
// width), sx [TB][G]; clears the tile's ghist [TB][2048] and, in block 0, zbits [F] if given.
template <int RUN>
__global__ void __launch_bounds__(kSelThreads)
input_quant_kernel(const float* __restrict__ x, int d, int B, int TB, int TBs, int k_in,
                   int* __restrict__ grows, int* __restrict__ gcnt, int* __restrict__ gq,
                   int8_t* __restrict__ gqx, float* __restrict__ sx_ws, int* __restrict__ ghist,
                   uint32_t* __restrict__ zbits, int F, uint16_t* __restrict__ qxh,
                   int8_t* __restrict__ dbg_qx, float* __restrict__ dbg_sx, int lists) {
    extern __shared__ __align__(16) unsigned char smem[];
    uint32_t* keys = reinterpret_cast<uint32_t*>(smem);                 // [d]
    int8_t* qx8 = reinterpret_cast<int8_t*>(keys + d);                   // [TB][d]
    __shared__ int hist[2 * 2048];
    __shared__ int wsum[kSelThreads / 32 + 4];
    __shared__ int s_gq[128];   // quads per group
    constexpr int NT = kSelThreads;
    constexpr int tpg = 128 / RUN;                 // threads per group (8 .. 32)
    const int tid = threadIdx.x;
    const int G = d >> 7;
    const int lo = min(d, tid * RUN), hi = min(d, lo + RUN);
    const int g_mine = lo >> 7;
    const bool active = lo < hi;
    const int gl = tid & (tpg - 1);                // this thread's place among its group's
    const int z = blockIdx.x, t0 = z * TB;
    const int nb = min(TB, B - t0);
    x += static_cast<size_t>(t0) * d;
    grows += static_cast<size_t>(z) * d;
    gcnt += static_cast<size_t>(z) * G;
    gq += static_cast<size_t>(z) * (G + 1);
    gqx += static_cast<size_t>(z) * TB * d;
    sx_ws += static_cast<size_t>(z) * TB * G;
    ghist += static_cast<size_t>(z) * TB * 2048;
    if (dbg_qx) dbg_qx += static_cast<size_t>(t0) * d;
    if (dbg_sx) dbg_sx += static_cast<size_t>(t0) * G;

    grid_dep_wait();
    grid_dep_launch();
    for (int i = tid; i < TB * 512; i += NT)   // filled by Stage 1 for the top-k
        reinterpret_cast<int4*>(ghist)[i] = make_int4(0, 0, 0, 0);
    if (zbits && z == 0)   // the batch's channel bitmap, filled by the top-k
        for (int i = tid; i < F; i += NT) zbits[i] = 0u;
    if (qxh && z == 0)     // dense f16 codes: rows past the batch stay zero
        for (int i = B * d + tid; i < kTcMaxTokens * d; i += NT) qxh[i] = 0;
    uint64_t any = 0ull;
    for (int b = 0; b < nb; ++b) {
        float xv[RUN];
#pragma unroll
        for (int e4 = 0; e4 < RUN / 4; ++e4) {
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (active) v = *reinterpret_cast<const float4*>(x + static_cast<size_t>(b) * d + lo + e4 * 4);
            xv[e4 * 4] = v.x; xv[e4 * 4 + 1] = v.y; xv[e4 * 4 + 2] = v.z; xv[e4 * 4 + 3] = v.w;
            if (active) {
                uint4 kk;
                kk.x = __float_as_uint(v.x) & 0x7fffffffu;
                kk.y = __float_as_uint(v.y) & 0x7fffffffu;
                kk.z = __float_as_uint(v.z) & 0x7fffffffu;
                kk.w = __float_as_uint(v.w) & 0x7fffffffu;
                *reinterpret_cast<uint4*>(keys + lo + e4 * 4) = kk;
            }
        }
        __syncthreads();
        uint32_t T;
        int take, eq_total;
        block_select_kth<NT, RUN>(keys, d, k_in, hist, wsum, T, take, eq_total);
        uint64_t mine;
        block_take_topk<NT, RUN>(keys, d, T, take, eq_total, wsum, mine);
        any |= mine;
        // per-group scale over the group's aligned lanes
        float m = 0.f;
#pragma unroll
        for (int e = 0; e < RUN; ++e)
            if ((mine >> e) & 1ull) m = fmaxf(m, fabsf(xv[e]));
        for (int o = tpg >> 1; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        const float sxg = __fdiv_rn(m, 127.0f);
        uint32_t qw[RUN / 4];
#pragma unroll
        for (int e4 = 0; e4 < RUN / 4; ++e4) qw[e4] = 0u;
#pragma unroll
        for (int e = 0; e < RUN; ++e) {
            float q = 0.f;
            if (((mine >> e) & 1ull) && sxg != 0.f)
                q = fminf(127.f, fmaxf(-127.f, rintf(__fdiv_rn(xv[e], sxg))));
            const uint32_t qb = static_cast<uint32_t>(static_cast<uint8_t>(static_cast<int8_t>(static_cast<int>(q))));
            qw[e >> 2] |= qb << (8 * (e & 3));
        }
        if (active) {
            if (qxh) {
                uint16_t* qh = qxh + static_cast<size_t>(t0 + b) * d + lo;
#pragma unroll
                for (int e = 0; e < RUN; ++e)
                    qh[e] = __half_as_ushort(__int2half_rn(static_cast<int>(static_cast<int8_t>(qw[e >> 2] >> (8 * (e & 3))))));
            }
#pragma unroll
            for (int e4 = 0; e4 < RUN / 4; ++e4) {
                *reinterpret_cast<uint32_t*>(qx8 + b * d + lo + e4 * 4) = qw[e4];
                if (dbg_qx)
                    *reinterpret_cast<uint32_t*>(dbg_qx + static_cast<size_t>(b) * d + lo + e4 * 4) = qw[e4];
            }
            if (gl == 0) {
                sx_ws[b * G + g_mine] = sxg;
                if (dbg_sx) dbg_sx[b * G + g_mine] = sxg;
            }
        }
        __syncthreads();   // keys are rewritten for the next token
    }
    for (int i = tid; i < (TB - nb) * G; i += NT) sx_ws[nb * G + i] = 0.f;
    if (!lists) return;   // the tensor-core Stage 1 reads the dense codes only

    // per group: the inputs any token kept, ascending, then padding to a multiple of 4
    const int cnt = __popcll(any);
    int incl = cnt;
    for (int o = 1; o < tpg; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o, tpg);
        if (gl >= o) incl += y;
    }
    const int n_g = __shfl_sync(0xffffffffu, incl, tpg - 1, tpg);
    int last = -1;
#pragma unroll
    for (int e = 0; e < RUN; ++e)
        if ((any >> e) & 1ull) last = lo + e;
    for (int o = tpg >> 1; o > 0; o >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
    if (active) {
        int* rows_g = grows + g_mine * 128;
        int p = incl - cnt;
#pragma unroll
        for (int e = 0; e < RUN; ++e) {
            if ((any >> e) & 1ull) {
                const int i = lo + e;
                rows_g[p] = i;
                for (int b = 0; b < TBs; ++b)
                    gqx[(static_cast<size_t>(b) * G + g_mine) * 128 + p] = b < nb ? qx8[b * d + i] : 0;
                ++p;
            }
        }
        if (gl == tpg - 1) {
            const int padded = (n_g + 3) & ~3;
            for (int q = n_g; q < padded; ++q) {
                rows_g[q] = last;
                for (int b = 0; b < TBs; ++b) gqx[(static_cast<size_t>(b) * G + g_mine) * 128 + q] = 0;
            }
            gcnt[g_mine] = padded;
            s_gq[g_mine] = padded >> 2;
        }
    }
    // quad offsets of the groups (exclusive sums of the padded counts / 4), for Stage 1
    __syncthreads();
    if (tid < 32) {
        int c4v[4], loc = 0;
#pragma unroll
        for (int m4 = 0; m4 < 4; ++m4) {
            const int g = tid * 4 + m4;
            c4v[m4] = g < G ? s_gq[g] : 0;
            loc += c4v[m4];
        }
        int incl = loc;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (tid >= o) incl += y;
        }
        int run = incl - loc;
#pragma unroll
        for (int m4 = 0; m4 < 4; ++m4) {
            const int g = tid * 4 + m4;
            if (g < G) gq[g] = run;
            run += c4v[m4];
        }
        if (tid == 31) gq[G] = incl;
    }
}

// dp4a with unsigned bytes in a and signed bytes in b
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    int r;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
    return r;
}

// CPL bytes of codes (CPL/4 words) of one row for one lane
template <int CPL>
__device__ __forceinline__ void load_codes(uint32_t (&w)[CPL / 4], const uint8_t* p, bool ok) {
    if constexpr (CPL == 16) {
        const uint4 v = ok ? __ldg(reinterpret_cast<const uint4*>(p)) : make_uint4(0u, 0u, 0u, 0u);
        w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
    } else if constexpr (CPL == 8) {
        const uint2 v = ok ? __ldg(reinterpret_cast<const uint2*>(p)) : make_uint2(0u, 0u);
        w[0] = v.x; w[1] = v.y;
    } else {
        w[0] = ok ? __ldg(reinterpret_cast<const uint32_t*>(p)) : 0u;
    }
}

template <int TB, int CPL>
__global__ void __launch_bounds__(kS1Threads, 2)
stage1_kernel(const uint8_t* __restrict__ codes, const uint32_t* __restrict__ scales, int d, int F,
              const int* __restrict__ grows, const int* __restrict__ gq,
              const int8_t* __restrict__ gqx, const float* __restrict__ sx, int gps, int S,
              int B, float* __restrict__ sigma, int* __restrict__ ghist,
              int32_t* __restrict__ dbg_gate, int32_t* __restrict__ dbg_up,
              int* __restrict__ status) {
    constexpr int NV = 2 * CPL * TB;       // values per lane: (token, channel, projection)
    constexpr int NWC = CPL / 4;           // code words per lane and row
    constexpr int TILE = 32 * CPL;         // channels per block
    extern __shared__ __align__(16) unsigned char smem[];
    int* s_A = reinterpret_cast<int*>(smem);                               // [gps][NV][32]
    uint32_t* s_sc = reinterpret_cast<uint32_t*>(s_A + gps * NV * 32);     // [gps][TILE]
    int* s_rows = reinterpret_cast<int*>(s_sc + gps * TILE);               // [gps][128]
    uint32_t* s_qx = reinterpret_cast<uint32_t*>(s_rows + gps * 128);      // [TB][gps][32]
    float* s_sx = reinterpret_cast<float*>(s_qx + TB * gps * 32);          // [TB][gps]
    int* s_qs = reinterpret_cast<int*>(s_sx + TB * gps);                   // [gps + 1] quad starts
    __shared__ DF s_part[NV * 32];   // this slice's double-float sums, read by the whole cluster
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int tile = blockIdx.x, s = blockIdx.y, z = blockIdx.z;
    const int G = d >> 7;
    const int g0 = s * gps, ng = min(gps, G - g0);
    // token tile z: tokens z*TB .. z*TB + nb - 1
    const int nb = min(TB, B - z * TB);
    grows += static_cast<size_t>(z) * d;
    gq += static_cast<size_t>(z) * (G + 1);
    gqx += static_cast<size_t>(z) * TB * d;
    sx += static_cast<size_t>(z) * TB * G;
    ghist += static_cast<size_t>(z) * TB * 2048;
    sigma += static_cast<size_t>(z) * TB * F;
    if (dbg_gate) dbg_gate += static_cast<size_t>(z) * TB * G * F;
    if (dbg_up) dbg_up += static_cast<size_t>(z) * TB * G * F;
    const int c0 = tile * TILE + lane * CPL;          // this lane's first channel
    const bool valid = c0 < F;                        // F % 16 == 0: all CPL channels or none
    const uint8_t* cbase = codes + (valid ? c0 : 0);

    // the packed weights do not depend on earlier kernels: stage this tile's scales first
    for (int i = tid; i < ng * (TILE / 4); i += kS1Threads) {
        const int gl = i / (TILE / 4), c4 = i - gl * (TILE / 4);
        const int ch = tile * TILE + 4 * c4;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (ch < F) v = __ldg(reinterpret_cast<const uint4*>(scales + static_cast<size_t>(g0 + gl) * F + ch));
        reinterpret_cast<uint4*>(s_sc)[gl * (TILE / 4) + c4] = v;
    }
    for (int i = tid; i < ng * NV * 32 / 4; i += kS1Threads)
        reinterpret_cast<int4*>(s_A)[i] = make_int4(0, 0, 0, 0);
    grid_dep_wait();
    grid_dep_launch();
    for (int i = tid; i < ng * 32; i += kS1Threads)
        reinterpret_cast<int4*>(s_rows)[i] = __ldcg(reinterpret_cast<const int4*>(grows + g0 * 128) + i);
    for (int i = tid; i < TB * ng * 32; i += kS1Threads) {
        const int b = i / (ng * 32), r = i - b * (ng * 32);
        s_qx[b * gps * 32 + r] = __ldcg(reinterpret_cast<const uint32_t*>(gqx + (static_cast<size_t>(b) * G + g0) * 128) + r);
    }
    for (int i = tid; i < TB * ng; i += kS1Threads) {
        const int b = i / ng, gl = i - b * ng;
        s_sx[b * gps + gl] = __ldcg(sx + b * G + g0 + gl);
    }
    for (int i = tid; i <= ng; i += kS1Threads) s_qs[i] = __ldcg(gq + g0 + i);
    __syncthreads();
    // quad starts relative to the slice; a group holds at most 32 quads
    int qv = 0, qprev = 0;
    if (tid <= ng) {
        qv = s_qs[tid] - s_qs[0];
        qprev = tid > 0 ? s_qs[tid - 1] - s_qs[0] : 0;
    }
    __syncthreads();
    if (tid <= ng) {
        if (qv < qprev || qv - qprev > 32 || qv > 32 * tid) {
            set_status(status, PROX_ERR_BOUNDS);
            qv = qprev;
        }
        s_qs[tid] = qv;
    }
    __syncthreads();
    // this warp's quads of the slice
    const int Q = s_qs[ng];
    const int qa = static_cast<int>(static_cast<long long>(Q) * warp / kS1Warps);
    const int qb = static_cast<int>(static_cast<long long>(Q) * (warp + 1) / kS1Warps);

    int gl = 0;
    while (gl + 1 < ng && s_qs[gl + 1] <= qa) ++gl;
    auto load_quad = [&](uint32_t (&w)[4][NWC], int q, int g) {
        int4 r4 = *reinterpret_cast<const int4*>(s_rows + g * 128 + 4 * (q - s_qs[g]));
        if (static_cast<unsigned>(r4.x) >= static_cast<unsigned>(d) || static_cast<unsigned>(r4.y) >= static_cast<unsigned>(d) ||
            static_cast<unsigned>(r4.z) >= static_cast<unsigned>(d) || static_cast<unsigned>(r4.w) >= static_cast<unsigned>(d)) {
            set_status(status, PROX_ERR_BOUNDS);   // a row outside the layer: read row 0 instead
            r4 = make_int4(0, 0, 0, 0);
        }
        load_codes<CPL>(w[0], cbase + static_cast<size_t>(r4.x) * F, valid);
        load_codes<CPL>(w[1], cbase + static_cast<size_t>(r4.y) * F, valid);
        load_codes<CPL>(w[2], cbase + static_cast<size_t>(r4.z) * F, valid);
        load_codes<CPL>(w[3], cbase + static_cast<size_t>(r4.w) * F, valid);
    };
    int ag[TB][CPL], au[TB][CPL], corr[TB];
#pragma unroll
    for (int b = 0; b < TB; ++b) {
        corr[b] = 0;
#pragma unroll
        for (int c = 0; c < CPL; ++c) ag[b][c] = au[b][c] = 0;
    }
    // multiply one quad: transpose each 4-channel column of the four rows, one dp4a per
    // channel and projection (gate nibbles as bytes 0..15, up nibbles as 16 * 0..15); at the
    // end of this warp's part of a group, add the exact integers A = sum((q + 8) qx) -
    // 8 sum(qx) to the block's per-group sums (integer adds, so their order does not matter)
    auto step = [&](const uint32_t (&w)[4][NWC], int q, int gcur, int gnext, bool last) {
        const int qo = q - s_qs[gcur];
#pragma unroll
        for (int b = 0; b < TB; ++b) {
            const uint32_t q4 = s_qx[(b * gps + gcur) * 32 + qo];
            corr[b] = dp4a_us(0x08080808u, q4, corr[b]);
#pragma unroll
            for (int wcol = 0; wcol < NWC; ++wcol) {
                const uint32_t w0 = w[0][wcol], w1 = w[1][wcol], w2 = w[2][wcol], w3 = w[3][wcol];
                const uint32_t a = __byte_perm(w0, w1, 0x5140), bq = __byte_perm(w2, w3, 0x5140);
                const uint32_t cq = __byte_perm(w0, w1, 0x7362), dq = __byte_perm(w2, w3, 0x7362);
                const uint32_t t[4] = {__byte_perm(a, bq, 0x5410), __byte_perm(a, bq, 0x7632),
                                       __byte_perm(cq, dq, 0x5410), __byte_perm(cq, dq, 0x7632)};
#pragma unroll
                for (int ch = 0; ch < 4; ++ch) {
                    ag[b][4 * wcol + ch] = dp4a_us(t[ch] & 0x0F0F0F0Fu, q4, ag[b][4 * wcol + ch]);
                    au[b][4 * wcol + ch] = dp4a_us(t[ch] & 0xF0F0F0F0u, q4, au[b][4 * wcol + ch]);
                }
            }
        }
        if (last || gnext != gcur) {
            int* A = s_A + gcur * NV * 32 + lane;
#pragma unroll
            for (int b = 0; b < TB; ++b) {
#pragma unroll
                for (int ch = 0; ch < CPL; ++ch) {
                    const int v = (b * CPL + ch) * 2;
                    atomicAdd(&A[v * 32], ag[b][ch] - corr[b]);
                    atomicAdd(&A[(v + 1) * 32], (au[b][ch] >> 4) - corr[b]);
                    ag[b][ch] = au[b][ch] = 0;
                }
                corr[b] = 0;
            }
        }
    };
    if constexpr (CPL == 16) {
        // 16-byte loads: two quads in flight keep enough bytes in flight
        uint32_t wa[4][NWC], wb[4][NWC];
        if (qa < qb) load_quad(wa, qa, gl);
        for (int q = qa; q < qb; q += 2) {
            // quad q is in wa; load quad q + 1 into wb, then q + 2 into wa after q is done
            int g1 = gl;
            if (q + 1 < qb) {
                while (g1 + 1 < ng && s_qs[g1 + 1] <= q + 1) ++g1;
                load_quad(wb, q + 1, g1);
            }
            step(wa, q, gl, g1, q + 1 == qb);
            if (q + 1 >= qb) break;
            int g2 = g1;
            if (q + 2 < qb) {
                while (g2 + 1 < ng && s_qs[g2 + 1] <= q + 2) ++g2;
                load_quad(wa, q + 2, g2);
            }
            step(wb, q + 1, g1, g2, q + 2 == qb);
            gl = g2;
        }
    } else {
        // narrower loads: a ring of kQ quads in flight; slot j holds quads j, j + kQ, ...
        constexpr int kQ = 4;
        uint32_t wr[kQ][4][NWC];
        int gs[kQ];   // group of the quad in each slot
        int gt = gl;  // group of the last quad loaded
#pragma unroll
        for (int j = 0; j < kQ; ++j) {
            gs[j] = gt;
            if (qa + j < qb) {
                while (gt + 1 < ng && s_qs[gt + 1] <= qa + j) ++gt;
                gs[j] = gt;
                load_quad(wr[j], qa + j, gt);
            }
        }
        for (int q0 = qa; q0 < qb; q0 += kQ) {
#pragma unroll
            for (int j = 0; j < kQ; ++j) {
                const int q = q0 + j;
                if (q >= qb) break;
                // slot j + 1 (mod kQ) holds quad q + 1 when there is one
                step(wr[j], q, gs[j], q + 1 < qb ? gs[(j + 1) % kQ] : gs[j], q + 1 == qb);
                const int qn = q + kQ;
                if (qn < qb) {
                    while (gt + 1 < ng && s_qs[gt + 1] <= qn) ++gt;
                    gs[j] = gt;
                    load_quad(wr[j], qn, gt);
                }
            }
        }
    }
    __syncthreads();

    // per (value, lane): the slice's groups in order, each scaled by sx * sw, summed as a
    // double-float; then this slice's partial sums go to global memory. Each thread carries
    // its NV * 32 / 256 entries side by side, so their dependent chains overlap.
    constexpr int EPT = NV * 32 / kS1Threads;   // 4
    DF t[EPT];
    int ve[EPT], lne[EPT];
#pragma unroll
    for (int k = 0; k < EPT; ++k) {
        const int e = tid + k * kS1Threads;
        ve[k] = e >> 5;
        lne[k] = e & 31;
        t[k] = DF{0.f, 0.f};
    }
    for (int g = 0; g < ng; ++g) {
#pragma unroll
        for (int k = 0; k < EPT; ++k) {
            const int v = ve[k], ln = lne[k];
            const int b = v / (2 * CPL), ch = (v >> 1) % CPL, proj = v & 1;
            const int A = s_A[(g * NV + v) * 32 + ln];
            const uint32_t swv = s_sc[g * TILE + ln * CPL + ch];
            const float sw = __half2float(__ushort_as_half(static_cast<unsigned short>(proj ? swv >> 16 : swv & 0xFFFFu)));
            t[k] = df_add(t[k], df_scaled_int(s_sx[b * gps + g], sw, A));
            int32_t* dbg = proj ? dbg_up : dbg_gate;
            const int c = tile * TILE + ln * CPL + ch;
            if (dbg && b < nb && c < F) dbg[(static_cast<size_t>(b) * G + g0 + g) * F + c] = A;
        }
    }
#pragma unroll
    for (int k = 0; k < EPT; ++k) s_part[tid + k * kS1Threads] = t[k];

    // the S slices of this tile are one cluster: after the cluster barrier, rank r adds the
    // slices' sums in order for its share of the tile's (token, channel) pairs, through
    // distributed shared memory, and writes their salience and histogram counts
    namespace cg = cooperative_groups;
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();
    const int npairs = TB * TILE;
    const int r = static_cast<int>(cluster.block_rank());
    const int pa = npairs * r / S, pb = npairs * (r + 1) / S;
    for (int pr = pa + tid; pr < pb; pr += kS1Threads) {
        const int b = pr / TILE, cl = pr - b * TILE;
        const int c = tile * TILE + cl;
        const int ln = cl / CPL, ch = cl - ln * CPL;
        const int eg = ((b * CPL + ch) * 2) * 32 + ln;   // gate entry; up entry is eg + 32
        if (b < nb && c < F) {
            DF tg{0.f, 0.f}, tu{0.f, 0.f};
            for (int s2 = 0; s2 < S; ++s2) {
                const DF* rp = cluster.map_shared_rank(s_part, s2);
                tg = df_add(tg, rp[eg]);
                tu = df_add(tu, rp[eg + 32]);
            }
            const float sg = fabsf(silu_f(tg.hi + tg.lo) * (tu.hi + tu.lo));
            sigma[static_cast<size_t>(b) * F + c] = sg;
            atomicAdd(&ghist[b * 2048 + (__float_as_uint(sg) >> 20)], 1);
        }
    }
    cluster.sync();   // no block leaves while another still reads its shared memory
}

int launch_input_quant(const float* x, int d, int F, int B, int k_in, uint8_t* ws,
                       const WsLayout& W, uint32_t* zbits, bool dense_codes, int8_t* dbg_qx,
                       float* dbg_sx, cudaStream_t s) {
    if (dense_codes && (W.BPtc == 0 || B > kTcMaxTokens)) return PROX_ERR_UNSUPPORTED;
    // with dense codes (the tensor-core Stage 1) every token is a block of its own and no
    // per-tile kept-row lists are built; the per-token outputs (sx [B][G], ghist [B][2048]) keep
    // their places, the tiles being consecutive tokens
    const int TB = dense_codes ? 1 : W.TB;
    const size_t smem = static_cast<size_t>(d) * 4 + static_cast<size_t>(TB) * d;
    const int run = select_run(d, kSelThreads);   // d <= 16384: at most 16
    if (run > 16) return PROX_ERR_UNSUPPORTED;
    auto fn = run <= 4 ? input_quant_kernel<4> : (run <= 8 ? input_quant_kernel<8> : input_quant_kernel<16>);
    if (ensure_dynamic_smem(reinterpret_cast<const void*>(fn), smem) != PROX_OK) return PROX_ERR_CUDA;
    const int ntiles = (B + TB - 1) / TB;
    return launch_pdl(fn, dim3(ntiles), dim3(kSelThreads), smem, s, x, d, B, TB,
                      stage1_width(B, TB), k_in, reinterpret_cast<int*>(ws + W.grows),
                      reinterpret_cast<int*>(ws + W.gcnt), reinterpret_cast<int*>(ws + W.gq),
                      reinterpret_cast<int8_t*>(ws + W.gqx), reinterpret_cast<float*>(ws + W.sx),
                      reinterpret_cast<int*>(ws + W.ghist), zbits, F,
                      dense_codes ? reinterpret_cast<uint16_t*>(ws + W.qxh) : nullptr, dbg_qx,
                      dbg_sx, dense_codes ? 0 : 1);
}

template <int TB, int CPL>
static int launch_stage1_t(const uint8_t* packed, const PackedLayout& L, int d, int F, int B,
                           const Stage1Plan& pl, uint8_t* ws, const WsLayout& W, float* sigma,
                           int32_t* dbg_gate, int32_t* dbg_up, cudaStream_t s) {
    constexpr int NV = 2 * CPL * TB;
    constexpr int TILE = 32 * CPL;
    const size_t smem = static_cast<size_t>(pl.gps) * NV * 32 * 4 +
                        static_cast<size_t>(pl.gps) * TILE * 4 + static_cast<size_t>(pl.gps) * 128 * 4 +
                        static_cast<size_t>(TB) * pl.gps * 128 + static_cast<size_t>(TB) * pl.gps * 4 +
                        static_cast<size_t>(pl.gps + 1) * 4;
    auto fn = stage1_kernel<TB, CPL>;
    if (ensure_dynamic_smem(reinterpret_cast<const void*>(fn), smem) != PROX_OK) return PROX_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(pl.tiles, pl.S, (B + TB - 1) / TB);   // z: token tiles
    cfg.blockDim = dim3(kS1Threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;   // the S slices of a tile
    attr[1].val.clusterDim.x = 1;
    attr[1].val.clusterDim.y = pl.S;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    const cudaError_t err = cudaLaunchKernelEx(
        &cfg, fn, L.codes(packed), L.scales(packed), d, F,
        static_cast<const int*>(reinterpret_cast<const int*>(ws + W.grows)),
        static_cast<const int*>(reinterpret_cast<const int*>(ws + W.gq)),
        static_cast<const int8_t*>(reinterpret_cast<const int8_t*>(ws + W.gqx)),
        static_cast<const float*>(reinterpret_cast<const float*>(ws + W.sx)), pl.gps, pl.S, B,
        sigma, reinterpret_cast<int*>(ws + W.ghist), dbg_gate, dbg_up,
        &reinterpret_cast<Control*>(ws + W.control)->status);
    if (err != cudaSuccess) return cuda_fail(err, "Stage-1 cluster launch");
    count_launch();
    return PROX_OK;
}

int launch_stage1(const uint8_t* packed, const PackedLayout& L, int d, int F, int B, uint8_t* ws,
                  const WsLayout& W, float* sigma, int32_t* dbg_gate, int32_t* dbg_up, int sms,
                  cudaStream_t s) {
    const int TB = stage1_width(B, W.TB);
    const Stage1Plan pl = stage1_plan(d, F, TB, sms);
    if (TB == 1) return launch_stage1_t<1, 16>(packed, L, d, F, B, pl, ws, W, sigma, dbg_gate, dbg_up, s);
    if (TB == 2) return launch_stage1_t<2, 8>(packed, L, d, F, B, pl, ws, W, sigma, dbg_gate, dbg_up, s);
    return launch_stage1_t<4, 4>(packed, L, d, F, B, pl, ws, W, sigma, dbg_gate, dbg_up, s);
}

}  // namespace prox

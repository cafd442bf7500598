// Prox Stage 2 ("Exact Sparse Computation" in the technical summary): for the selected
// channels only, exact gate and up projections from the bf16 weights, s = SiLU(g) * u, and
// the down projection over the same channels ("all three projections" sparse, abstract).
//
// stage2_kernel (one block per SM, persistent over a contiguous run of the channel list)
//   The packed rows put W_gate[j,:], W_up[j,:] and W_down[:,j] of channel j in one
//   contiguous 6*d-byte run, so a selected channel is ONE bulk copy (cp.async.bulk with an
//   mbarrier transaction count) from HBM into a shared-memory stage. The block's slice of
//   the channel list is staged in shared memory first, then a power-of-two ring of stages
//   is kept in flight.
//   The warps form NG independent groups (4, 2 or 1); group g takes every NG-th channel of
//   the block's slice, keeps a full partial output y of its own, and issues the copies
//   into its own ring slots (NG divides the ring size, so channel it + nstage reuses the
//   slot of channel it within the same group). Within a
//   group each thread owns CPT fixed 16-byte column chunks and keeps their activations x
//   and partial outputs y in registers. Per channel a group
//     1. forms the partial dot products of the gate and up rows with x (packed f32x2 FMAs),
//     2. reduces them across each warp (reduce-scatter butterfly), writes the warp sums to
//        shared memory and meets at a barrier of its own warps only,
//     3. every warp adds the group's warp sums in a fixed order and forms s = SiLU(g) * u,
//        zeroed for tokens that did not select the channel (batch path),
//     4. y += s * W_down[:, j] on its columns; the slot is refilled at the group's next
//        barrier, when every warp of the group is past it.
//   The groups run unsynchronised, so one group's barrier latency hides behind another's
//   arithmetic. At the end the groups' partial outputs are added in a fixed order.
//   Every wait is bounded; a wait that runs out records PROX_ERR_TIMEOUT, the group leaves
//   together (barrier with an OR reduction), and its leader drains the copies it issued.
// reduce_kernel
//   Sums the per-block partial outputs in a fixed order, so y is bit-reproducible.
// The dense baseline is the same kernel over every channel (list == nullptr).
#include "prox_kernels.cuh"

namespace prox {

constexpr int kS2MaxConsumers = 512;

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

// c + a * b on two fp32 lanes at once
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rb, {%4, %5};\n\t"
        "mov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rc, ra, rb, rc;\n\t"
        "mov.b64 {%0, %1}, rc;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

// the two bf16 of a 32-bit word (element 0 in the low half) as fp32
__device__ __forceinline__ float2 bf16x2_f32(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// acc += x[0..7] * w[0..7] elementwise on lane pairs
__device__ __forceinline__ float2 dot8x2(const float2 (&x)[4], uint4 w, float2 acc) {
    acc = ffma2(x[0], bf16x2_f32(w.x), acc);
    acc = ffma2(x[1], bf16x2_f32(w.y), acc);
    acc = ffma2(x[2], bf16x2_f32(w.z), acc);
    acc = ffma2(x[3], bf16x2_f32(w.w), acc);
    return acc;
}

__device__ __forceinline__ void axpy8x2(float2 (&y)[4], float2 s, uint4 w) {
    y[0] = ffma2(s, bf16x2_f32(w.x), y[0]);
    y[1] = ffma2(s, bf16x2_f32(w.y), y[1]);
    y[2] = ffma2(s, bf16x2_f32(w.z), y[2]);
    y[3] = ffma2(s, bf16x2_f32(w.w), y[3]);
}

template <int V>
struct Log2 {
    static constexpr int value = V <= 1 ? 0 : 1 + Log2<V / 2>::value;
};
template <>
struct Log2<1> {
    static constexpr int value = 0;
};

// Warp-wide sums of V values (V a power of two, <= 32) with V - 1 + (5 - log2 V) shuffles:
// at each halving step a lane keeps one half of its values and adds its partner's copy of
// that half. Afterwards lane L holds the sum of value index L >> (5 - log2 V).
template <int V>
__device__ __forceinline__ float warp_reduce_scatter(float (&v)[V], int lane) {
    constexpr int LV = Log2<V>::value;
#pragma unroll
    for (int lvl = 0; lvl < LV; ++lvl) {
        const int off = 16 >> lvl;
        const int half = V >> (lvl + 1);
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const float send = upper ? v[i] : v[i + half];
            const float keep = upper ? v[i + half] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
    }
    float r = v[0];
#pragma unroll
    for (int off = 16 >> LV; off > 0; off >>= 1) r += __shfl_xor_sync(0xffffffffu, r, off);
    return r;
}

// The top-k channel selection at the front of the single-token Stage-2 kernel (every block
// does it redundantly, so no separate kernel and no index round trip is needed). Stage 1
// leaves the salience sigma[F] and a histogram of its bits 30..20 (ghist[2048]).
//  1. From the histogram, the bin b1 holding the k-th largest key: every channel in a higher
//     bin is selected for sure. Each thread owns KRUN consecutive channels (keys held in
//     registers); a block scan gives the sure channels' positions in ascending order, and
//     this block takes the slice [S*blk/P, S*(blk+1)/P) of them (S = number of sure ones).
//  2. `start(nsure)` is called, so copies of the sure channels begin.
//  3. Two more radix passes over the keys in bin b1 find the exact k-th key T and how many
//     keys equal to T are taken (lowest channel first); the winners of bin b1, in ascending
//     order, are split over the blocks in the same way and appended to this block's list.
// Returns this block's channel count. The union of the blocks' lists is the top-k set of
// the ranking rule (largest salience first, equal values to the lower channel index).
// If dbg_sel is not null, the sure channels are also written to dbg_sel[0, S) and the winners
// to dbg_sel[S, k), each in ascending order (a test hook).
template <int KRUN, typename Start>
__device__ int select_channels(const float* __restrict__ sigma, const int* __restrict__ ghist, int F,
                               int k, int* s_list, uint32_t* s_bits, int* hist, int* wsum,
                               unsigned char* scratch, uint64_t* bar, long long spin,
                               int* status, int32_t* dbg_sel, Start start) {
    constexpr int NT = kS2MaxConsumers;
    constexpr int NW = NT / 32;
    const int tid = threadIdx.x;
    const int P = gridDim.x, blk = blockIdx.x;
    int* sel = wsum + NW;
    int* s_cnt = sel + 3;
    // 1. the salience row (into the not yet used stage memory) and the first-pass histogram,
    //    one bulk copy each, then the bin of the k-th largest key
    if (tid == 0) {
        mbar_arrive_expect_tx(bar, static_cast<uint32_t>(F) * 4 + 2048 * 4);
        bulk_g2s(scratch, sigma, static_cast<uint32_t>(F) * 4, bar);
        bulk_g2s(hist, ghist, 2048 * 4, bar);
    }
    for (int i = tid; i < 2048; i += NT) hist[2048 + i] = 0;
    const int lo = tid * KRUN;
    const int nv = lo < F ? (F - lo < KRUN ? F - lo : KRUN) : 0;
    // every thread decides the same way (a wait can run out for some threads only)
    if (!__syncthreads_and(mbar_wait(bar, 0u, spin, status))) {
        // nothing usable arrived (the status word says why): this block takes no channels
        return 0;
    }
    uint32_t key[KRUN];
#pragma unroll
    for (int i4 = 0; i4 < KRUN / 4; ++i4) {
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (4 * i4 < nv) v = *reinterpret_cast<const uint4*>(scratch + 4 * (lo + 4 * i4));
        key[4 * i4] = v.x & 0x7fffffffu;
        key[4 * i4 + 1] = v.y & 0x7fffffffu;
        key[4 * i4 + 2] = v.z & 0x7fffffffu;
        key[4 * i4 + 3] = v.w & 0x7fffffffu;
    }
    block_find_bin<NT>(hist, 2048, k, wsum, sel);   // its barriers also free the stage memory
    const uint32_t b1 = static_cast<uint32_t>(sel[0]);
    const int above = sel[1];
    // sure channels: bins above b1
    int cnt = 0;
#pragma unroll
    for (int e = 0; e < KRUN; ++e) cnt += (e < nv && (key[e] >> 20) > b1);
    int total;
    int pos = block_exclusive_scan<NT>(cnt, wsum, total);
    if (tid == 0 && total != above) set_status(status, PROX_ERR_BOUNDS);   // histogram mismatch
    const int s0 = static_cast<int>(static_cast<long long>(total) * blk / P);
    const int s1 = static_cast<int>(static_cast<long long>(total) * (blk + 1) / P);
#pragma unroll
    for (int e = 0; e < KRUN; ++e) {
        if (e < nv && (key[e] >> 20) > b1) {
            if (pos >= s0 && pos < s1 && pos - s0 < kStage2ListMax) {
                s_list[pos - s0] = lo + e;
                s_bits[pos - s0] = 0xffffffffu;
                if (dbg_sel) dbg_sel[pos] = lo + e;
            }
            ++pos;
        }
    }
    const int nsure = min(s1 - s0, kStage2ListMax);
    __syncthreads();
    start(nsure);
    // 3. the exact threshold inside bin b1 (two passes of 11 and 9 bits over its keys)
    uint32_t prefix = b1 << 20, pmask = 0x7FFu << 20;
    int remaining = k - above;
    int eq_total = 0;
#pragma unroll 1
    for (int p = 1; p < 3; ++p) {
        const int shift = p == 1 ? 9 : 0;
        const int nbins = p == 1 ? 2048 : 512;
        const uint32_t dmask = static_cast<uint32_t>(nbins - 1);
        int* h = hist + (p & 1) * 2048;
#pragma unroll
        for (int e = 0; e < KRUN; ++e)
            if (e < nv && (key[e] & pmask) == prefix) atomicAdd(&h[(key[e] >> shift) & dmask], 1);
        if (p == 1)
            for (int i = tid; i < 2048; i += NT) hist[i] = 0;   // buffer for the last pass
        __syncthreads();
        block_find_bin<NT>(h, nbins, remaining, wsum, sel);
        remaining -= sel[1];
        eq_total = sel[2];
        prefix |= static_cast<uint32_t>(sel[0]) << shift;
        pmask |= dmask << shift;
    }
    const uint32_t T = prefix;
    const int take_eq = remaining;
    __syncthreads();   // sel is free again
    // winners of bin b1: keys above T, and the first take_eq keys equal to T
    int e_rank = 0;
    if (take_eq != eq_total) {
        int eq = 0;
#pragma unroll
        for (int e = 0; e < KRUN; ++e) eq += (e < nv && key[e] == T);
        int eq_all;
        e_rank = block_exclusive_scan<NT>(eq, wsum, eq_all);
    }
    uint64_t win = 0ull;
    int wc = 0;
#pragma unroll
    for (int e = 0; e < KRUN; ++e) {
        if (e < nv && (key[e] >> 20) == b1) {
            bool t = key[e] > T;
            if (key[e] == T) {
                t = e_rank < take_eq;
                ++e_rank;
            }
            if (t) {
                win |= 1ull << e;
                ++wc;
            }
        }
    }
    int wtotal;
    int wpos = block_exclusive_scan<NT>(wc, wsum, wtotal);
    if (tid == 0 && wtotal != k - above) set_status(status, PROX_ERR_BOUNDS);
    const int w0 = static_cast<int>(static_cast<long long>(wtotal) * blk / P);
    const int w1 = static_cast<int>(static_cast<long long>(wtotal) * (blk + 1) / P);
#pragma unroll
    for (int e = 0; e < KRUN; ++e) {
        if ((win >> e) & 1ull) {
            const int at = nsure + wpos - w0;
            if (wpos >= w0 && wpos < w1 && at < kStage2ListMax) {
                s_list[at] = lo + e;
                s_bits[at] = 0xffffffffu;
                if (dbg_sel) dbg_sel[total + wpos] = lo + e;
            }
            ++wpos;
        }
    }
    if (tid == 0) *s_cnt = min(nsure + (w1 - w0), kStage2ListMax);
    __syncthreads();
    return *s_cnt;
}

template <int TB, int CPT, int KRUN>
__global__ void __launch_bounds__(kS2MaxConsumers, 1)
stage2_kernel(const uint16_t* __restrict__ rows, int d, int F, const float* __restrict__ x, int nb,
              const int32_t* __restrict__ list, const uint32_t* __restrict__ lbits,
              const int* __restrict__ count_dev, int count_host, const float* __restrict__ sigma,
              const int* __restrict__ ghist, int ksel, int32_t* __restrict__ dbg_sel,
              float* __restrict__ ypart, int nstage_log2, int NG, long long spin,
              int* __restrict__ status) {
    extern __shared__ __align__(128) unsigned char smem[];
    constexpr int V = 2 * TB;
    constexpr int LV = Log2<V>::value;
    const int NT = blockDim.x, NW = NT >> 5;
    const int WPG = NW / NG, GT = WPG * 32;
    const int nstage = 1 << nstage_log2, smask = nstage - 1;
    const uint32_t stage_bytes = 6u * static_cast<uint32_t>(d);
    unsigned char* stages = smem;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + static_cast<size_t>(nstage) * stage_bytes);
    int* s_list = reinterpret_cast<int*>(full + nstage);              // [kStage2ListMax]
    uint32_t* s_bits = reinterpret_cast<uint32_t*>(s_list + kStage2ListMax);
    float* red = reinterpret_cast<float*>(s_bits + kStage2ListMax);    // [NG][2][V][WPG]
    int* s_hist = reinterpret_cast<int*>(red + NG * 2 * V * WPG);     // [2][2048] (select mode)
    int* s_wsum = s_hist + (KRUN ? 2 * 2048 : 0);                      // [NW + 4]
    uint64_t* s_selbar = reinterpret_cast<uint64_t*>(s_wsum + (KRUN ? NW + 4 : 0));
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int P = gridDim.x;

    if (tid == 0) {
        for (int i = 0; i < nstage; ++i) mbar_init(&full[i], 1);
        if (KRUN > 0) mbar_init(s_selbar, 1);
        mbar_init_fence();
    }
    __syncthreads();
    grid_dep_wait();   // the channel list (or the salience), the activations: earlier kernels
    grid_dep_launch();

    // Group gi consumes channels gi, gi + NG, ...; since NG divides the ring size, its
    // channels always land in its own ring slots, and its leader refills a slot as soon as the
    // whole group is past the channel that used it.
    const int gi = warp / WPG, gw = warp - gi * WPG, gtid = tid - gi * GT;
    const bool leader = gtid == 0;
    int next_issue = gi;   // next channel this group copies in
    auto issue = [&](int it) {
        const int st = it & smask;
        mbar_arrive_expect_tx(&full[st], stage_bytes);
        bulk_g2s(stages + static_cast<size_t>(st) * stage_bytes,
                 rows + static_cast<size_t>(s_list[it]) * 3 * d, stage_bytes, &full[st]);
    };

    int nloc;
    if constexpr (KRUN > 0) {
        nloc = select_channels<KRUN>(sigma, ghist, F, ksel, s_list, s_bits, s_hist, s_wsum, stages,
                                     s_selbar, spin, status, dbg_sel, [&](int nsure) {
                                         // copies of the sure channels start before the
                                         // boundary bin is resolved
                                         if (leader)
                                             for (; next_issue < nsure && next_issue < nstage;
                                                  next_issue += NG)
                                                 issue(next_issue);
                                     });
    } else {
        const int n = count_dev ? *count_dev : count_host;
        const int e0 = static_cast<int>(static_cast<long long>(n) * blockIdx.x / P);
        nloc = static_cast<int>(static_cast<long long>(n) * (blockIdx.x + 1) / P) - e0;
        if (nloc > kStage2ListMax) {   // the host sizes the grid so this cannot happen
            if (tid == 0) set_status(status, PROX_ERR_BOUNDS);
            nloc = kStage2ListMax;
        }
        for (int i = tid; i < nloc; i += NT) {
            int j = list ? list[e0 + i] : e0 + i;
            if (j < 0 || j >= F) {
                set_status(status, PROX_ERR_BOUNDS);
                j = 0;
            }
            s_list[i] = j;
            s_bits[i] = lbits ? lbits[e0 + i] : 0xffffffffu;
        }
        __syncthreads();
    }
    if (leader)
        for (; next_issue < nloc && next_issue < nstage; next_issue += NG) issue(next_issue);

    const int nchunk = d >> 3;
    float2 xr[TB][CPT][4], yr[TB][CPT][4];
#pragma unroll
    for (int c = 0; c < CPT; ++c) {
        const int q = c * GT + gtid;
#pragma unroll
        for (int b = 0; b < TB; ++b) {
            float4 a = make_float4(0.f, 0.f, 0.f, 0.f), bb = a;
            if (b < nb && q < nchunk) {
                const float4* src = reinterpret_cast<const float4*>(x + static_cast<size_t>(b) * d + q * 8);
                a = src[0];
                bb = src[1];
            }
            xr[b][c][0] = make_float2(a.x, a.y);
            xr[b][c][1] = make_float2(a.z, a.w);
            xr[b][c][2] = make_float2(bb.x, bb.y);
            xr[b][c][3] = make_float2(bb.z, bb.w);
#pragma unroll
            for (int m = 0; m < 4; ++m) yr[b][c][m] = make_float2(0.f, 0.f);
        }
    }

    float* gred = red + gi * 2 * V * WPG;
    bool broke = false;
    int slot = 0, it = gi;
    for (; it < nloc; it += NG, slot ^= 1) {
        const int st = it & smask;
        const bool ok = mbar_wait(&full[st], static_cast<uint32_t>(it >> nstage_log2) & 1u, spin, status);
        const uint16_t* sb = reinterpret_cast<const uint16_t*>(stages + static_cast<size_t>(st) * stage_bytes);
        float2 ga[TB], ua[TB];
#pragma unroll
        for (int b = 0; b < TB; ++b) ga[b] = ua[b] = make_float2(0.f, 0.f);
        if (ok) {
#pragma unroll
            for (int c = 0; c < CPT; ++c) {
                const int q = c * GT + gtid;
                if (q < nchunk) {
                    const uint4 wg = *reinterpret_cast<const uint4*>(sb + q * 8);
                    const uint4 wu = *reinterpret_cast<const uint4*>(sb + d + q * 8);
#pragma unroll
                    for (int b = 0; b < TB; ++b) {
                        ga[b] = dot8x2(xr[b][c], wg, ga[b]);
                        ua[b] = dot8x2(xr[b][c], wu, ua[b]);
                    }
                }
            }
        }
        float v[V];
#pragma unroll
        for (int b = 0; b < TB; ++b) {
            v[2 * b] = ga[b].x + ga[b].y;
            v[2 * b + 1] = ua[b].x + ua[b].y;
        }
        const float r = warp_reduce_scatter<V>(v, lane);
        if ((lane & ((32 >> LV) - 1)) == 0) gred[(slot * V + (lane >> (5 - LV))) * WPG + gw] = r;
        if (bar_red_or(1 + gi, GT, !ok)) {
            broke = true;
            break;
        }
        // every warp of the group is past channel it - NG: its slot takes the next copy
        if (leader && it - NG >= 0 && next_issue < nloc) {
            issue(next_issue);
            next_issue += NG;
        }
        float2 sv[TB];
#pragma unroll
        for (int b = 0; b < TB; ++b) {
            float g = 0.f, u = 0.f;
            for (int w2 = 0; w2 < WPG; ++w2) {
                g += gred[(slot * V + 2 * b) * WPG + w2];
                u += gred[(slot * V + 2 * b + 1) * WPG + w2];
            }
            const float s_val = (b < nb && ((s_bits[it] >> b) & 1u)) ? silu_f(g) * u : 0.f;
            sv[b] = make_float2(s_val, s_val);
        }
#pragma unroll
        for (int c = 0; c < CPT; ++c) {
            const int q = c * GT + gtid;
            if (q < nchunk) {
                const uint4 wd = *reinterpret_cast<const uint4*>(sb + 2 * d + q * 8);
#pragma unroll
                for (int b = 0; b < TB; ++b) axpy8x2(yr[b][c], sv[b], wd);
            }
        }
    }
    if (broke && leader) {
        // copies this group issued but did not consume must land before shared memory is freed
        for (int t = it; t < next_issue; t += NG)
            mbar_wait(&full[t & smask], static_cast<uint32_t>(t >> nstage_log2) & 1u, spin, status);
    }

    // add the groups' partial outputs in a fixed order; the stage buffers are free once every
    // group finished normally (each issued copy was then waited for), so they serve as scratch,
    // and after an abort the partial output is left unsummed (the status says why)
    const bool any_broke = bar_red_or(6, NT, broke) != 0;
    float* yp = ypart + static_cast<size_t>(blockIdx.x) * TB * d;
    if (NG == 1 || any_broke) {
#pragma unroll
        for (int c = 0; c < CPT; ++c) {
            const int q = c * GT + gtid;
            if (q < nchunk && gi == 0) {
#pragma unroll
                for (int b = 0; b < TB; ++b) {
                    float4* dst = reinterpret_cast<float4*>(yp + static_cast<size_t>(b) * d + q * 8);
                    dst[0] = make_float4(yr[b][c][0].x, yr[b][c][0].y, yr[b][c][1].x, yr[b][c][1].y);
                    dst[1] = make_float4(yr[b][c][2].x, yr[b][c][2].y, yr[b][c][3].x, yr[b][c][3].y);
                }
            }
        }
    } else {
        float* scratch = reinterpret_cast<float*>(stages);   // [NG][TB][d]
#pragma unroll
        for (int c = 0; c < CPT; ++c) {
            const int q = c * GT + gtid;
            if (q < nchunk) {
#pragma unroll
                for (int b = 0; b < TB; ++b) {
                    float4* dst = reinterpret_cast<float4*>(scratch + (static_cast<size_t>(gi) * TB + b) * d + q * 8);
                    dst[0] = make_float4(yr[b][c][0].x, yr[b][c][0].y, yr[b][c][1].x, yr[b][c][1].y);
                    dst[1] = make_float4(yr[b][c][2].x, yr[b][c][2].y, yr[b][c][3].x, yr[b][c][3].y);
                }
            }
        }
        bar_sync(6, NT);
        const int n4 = TB * d / 4;
        for (int i = tid; i < n4; i += NT) {
            float4 t = reinterpret_cast<const float4*>(scratch)[i];
            for (int g2 = 1; g2 < NG; ++g2) {
                const float4 u = reinterpret_cast<const float4*>(scratch + static_cast<size_t>(g2) * TB * d)[i];
                t.x += u.x; t.y += u.y; t.z += u.z; t.w += u.w;
            }
            reinterpret_cast<float4*>(yp)[i] = t;
        }
    }
}

// y[b][:] = sum over blocks p (fixed order) of ypart[p][b][:]. A block covers 8 float4
// columns; its 32 row groups each add every 32nd partial, then the groups are added in order.
__global__ void __launch_bounds__(256)
reduce_kernel(const float4* __restrict__ ypart, int P, int TB, int d, float4* __restrict__ y) {
    __shared__ float4 sm[32][8];
    const int cx = threadIdx.x & 7, pg = threadIdx.x >> 3;
    const int n4 = d >> 2;
    const int col = blockIdx.x * 8 + cx;
    const int b = blockIdx.y;
    grid_dep_wait();
    grid_dep_launch();
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (col < n4) {
        for (int p = pg; p < P; p += 32) {
            const float4 v = __ldcg(&ypart[(static_cast<size_t>(p) * TB + b) * n4 + col]);
            acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
        }
    }
    sm[pg][cx] = acc;
    __syncthreads();
    if (pg == 0 && col < n4) {
        float4 t = sm[0][cx];
#pragma unroll 8
        for (int g = 1; g < 32; ++g) {
            t.x += sm[g][cx].x; t.y += sm[g][cx].y; t.z += sm[g][cx].z; t.w += sm[g][cx].w;
        }
        y[static_cast<size_t>(b) * n4 + col] = t;
    }
}

// Consumer layout of the Stage-2 kernel for a row length and token tile: NG groups of WPG
// warps, CPT 16-byte chunks per thread, with CPT * TB <= 4 so x and y fit in registers.
struct S2Shape {
    int NG, WPG, CPT;
};
static S2Shape stage2_shape(int d, int TB) {
    const int nchunk = d / 8;
    const int nstage = 1 << stage2_nstage_log2(d);
    for (int NG = 4; NG >= 1; NG >>= 1) {
        if (nstage < 2 * NG) continue;   // each group needs two ring slots of its own
        int WPG = 16 / NG;
        const int need = (nchunk + 31) / 32;
        if (WPG > need) WPG = need;
        const int CPT = (nchunk + 32 * WPG - 1) / (32 * WPG);
        if (CPT * TB <= 4) return S2Shape{NG, WPG, CPT};
    }
    return S2Shape{0, 0, 0};
}

static size_t stage2_smem_bytes(int d, int TB, const S2Shape& sh, bool select) {
    const int nstage = 1 << stage2_nstage_log2(d);
    const int NW = sh.NG * sh.WPG;
    return static_cast<size_t>(nstage) * 6 * d + nstage * sizeof(uint64_t) +
           2 * kStage2ListMax * sizeof(int) +
           static_cast<size_t>(sh.NG) * 2 * 2 * TB * sh.WPG * sizeof(float) +
           (select ? (2 * 2048 + NW + 4) * sizeof(int) + 2 * sizeof(uint64_t) : 0);
}

template <int TB, int CPT, int KRUN>
static int launch_stage2_t(const uint16_t* rows, int d, int F, const float* x, int nb,
                           const int32_t* list, const uint32_t* lbits, const int* count_dev,
                           int count_host, const float* sigma, const int* ghist, int ksel,
                           int32_t* dbg_sel, float* ypart, int P, const S2Shape& sh, int* status,
                           cudaStream_t s) {
    const size_t smem = stage2_smem_bytes(d, TB, sh, KRUN > 0);
    auto fn = stage2_kernel<TB, CPT, KRUN>;
    if (ensure_dynamic_smem(reinterpret_cast<const void*>(fn), smem) != PROX_OK) return PROX_ERR_CUDA;
    const int NT = sh.NG * sh.WPG * 32;
    return launch_pdl(fn, dim3(P), dim3(NT), smem, s, rows, d, F, x, nb, list, lbits, count_dev,
                      count_host, sigma, ghist, ksel, dbg_sel, ypart, stage2_nstage_log2(d),
                      sh.NG, kDefaultSpinCycles, status);
}

int launch_reduce_partials(const float* ypart, int P, int TB, int d, int nb, float* y_tile,
                           cudaStream_t s) {
    const int n4 = d / 4;
    return launch_pdl(reduce_kernel, dim3((n4 + 7) / 8, nb), dim3(256), 0, s,
                      reinterpret_cast<const float4*>(ypart), P, TB, d,
                      reinterpret_cast<float4*>(y_tile));
}

int launch_stage2(const uint8_t* packed, const PackedLayout& L, int d, int F, const float* x_tile,
                  int nb, const int32_t* list, const uint32_t* lbits, const int* count_dev,
                  int count_host, float* y_tile, uint8_t* ws, const WsLayout& W, int sms,
                  cudaStream_t s) {
    const uint16_t* rows = reinterpret_cast<const uint16_t*>(L.rows(packed));
    float* ypart = reinterpret_cast<float*>(ws + W.ypart);
    int* status = &reinterpret_cast<Control*>(ws + W.control)->status;
    const int TB = nb <= 1 ? 1 : (nb <= 2 ? 2 : 4);
    const S2Shape sh = stage2_shape(d, TB);
    int P = stage2_blocks(F, sms);
    if (P > W.P) P = W.P;
    int rc = PROX_ERR_UNSUPPORTED;
#define PROX_S2(tb, cp)                                                                          \
    if (TB == tb && sh.CPT == cp)                                                                \
        rc = launch_stage2_t<tb, cp, 0>(rows, d, F, x_tile, nb, list, lbits, count_dev,          \
                                        count_host, nullptr, nullptr, 0, nullptr, ypart, P, sh,   \
                                        status, s);
    PROX_S2(1, 1)
    PROX_S2(1, 2)
    PROX_S2(1, 3)
    PROX_S2(1, 4)
    PROX_S2(2, 1)
    PROX_S2(2, 2)
    PROX_S2(4, 1)
#undef PROX_S2
    if (rc != PROX_OK) return rc;
    return launch_reduce_partials(ypart, P, TB, d, nb, y_tile, s);
}

bool stage2_select_supported(int d, int F) {
    const S2Shape sh = stage2_shape(d, 1);
    return sh.NG * sh.WPG * 32 == kS2MaxConsumers && F <= 64 * kS2MaxConsumers;
}

int launch_stage2_select(const uint8_t* packed, const PackedLayout& L, int d, int F,
                         const float* x, const float* sigma, const int* ghist, int k, float* y,
                         int32_t* dbg_sel, uint8_t* ws, const WsLayout& W, int sms,
                         cudaStream_t s) {
    if (!stage2_select_supported(d, F)) return PROX_ERR_UNSUPPORTED;
    const uint16_t* rows = reinterpret_cast<const uint16_t*>(L.rows(packed));
    float* ypart = reinterpret_cast<float*>(ws + W.ypart);
    int* status = &reinterpret_cast<Control*>(ws + W.control)->status;
    const S2Shape sh = stage2_shape(d, 1);
    int P = stage2_blocks(F, sms);
    if (P > W.P) P = W.P;
    const bool wide = F > 32 * kS2MaxConsumers;
    int rc = PROX_ERR_UNSUPPORTED;
#define PROX_S2S(cp)                                                                             \
    if (sh.CPT == cp)                                                                            \
        rc = wide ? launch_stage2_t<1, cp, 64>(rows, d, F, x, 1, nullptr, nullptr, nullptr, 0,   \
                                               sigma, ghist, k, dbg_sel, ypart, P, sh, status, s) \
                  : launch_stage2_t<1, cp, 32>(rows, d, F, x, 1, nullptr, nullptr, nullptr, 0,   \
                                               sigma, ghist, k, dbg_sel, ypart, P, sh, status, s);
    PROX_S2S(1)
    PROX_S2S(2)
    PROX_S2S(3)
    PROX_S2S(4)
#undef PROX_S2S
    if (rc != PROX_OK) return rc;
    return launch_reduce_partials(ypart, P, 1, d, 1, y, s);
}

}  // namespace prox

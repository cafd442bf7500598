// The fused single-token kernel (see prox_fused.cu for what it computes) and the host-side
// shape rules shared by its two translation units.
#pragma once

#include <type_traits>

#include "prox_kernels.cuh"

namespace prox {

// Everything the two translation units of the fused kernel share (prox_fused.cu: bf16 rows
// and the launch code; prox_fused_fp8.cu: FP8 rows).
namespace fused_detail {

constexpr int NT = kFusedThreads;
constexpr int NW = NT / 32;
constexpr int kListMax = 1024;   // channels one block may own in Stage 2
constexpr int kTileUnit = 8;     // Stage-1 tiles are whole units of 8 chunks of 16 channels
constexpr int kTopkKeysOff = 2 * 2048 * 4;   // the layer's salience keys, after two histograms
constexpr int kCandCap = 4096;               // boundary-bin candidates ranked on their own
constexpr int kTopkBar = 16;                 // mbarrier of the top-k's copies (ring: 0..15)

struct FusedParams {
    const uint8_t* codes;
    const uint32_t* scales;
    const uint16_t* rows;        // Stage-2 rows (bf16), or the FP8 rows' bytes
    size_t row_bytes;            // bytes of one channel's run (6 d bf16, 3 d + 16 FP8)
    const float* x;
    int d, F, k, k_in, mode;
    const int32_t* idx_in;
    int32_t* idx;
    float* sigma;
    float* ypart;
    float* y;
    FusedControl* ctl;
    int* status;
    long long spin;
    int region_bytes, nstage_log2, NG, WPG, CPT;
    int write_idx;   // also store the mask into idx (the caller asked for it)
    int prefetch_codes;   // ask L2 for the likely-kept proxy rows during the input selection
    int scales_smem;      // the tile's group scales are copied into shared memory at the start
    int8_t* dbg_qx;
    float* dbg_sx;
    int32_t* dbg_gate;
    int32_t* dbg_up;
};

// ------------------------------------------------------------------ small helpers

// 16 read-only bytes.
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
    return __ldg(reinterpret_cast<const uint4*>(p));
}

__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}


__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    int r;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
    return r;
}

__device__ __forceinline__ int named_bar_or(int id, int n, int pred) {
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

__device__ __forceinline__ float2 bf16x2_f32(uint32_t w) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// The four E4M3 codes of w (byte k = element k) as fp32 values, exactly: the hardware
// conversion to f16 pairs (every E4M3 value is an f16 value), then to fp32.
__device__ __forceinline__ void e4m3x4_f32(uint32_t w, float2& e01, float2& e23) {
    uint32_t h01, h23;
    asm("{\n\t.reg .b16 lo, hi;\n\t"
        "mov.b32 {lo, hi}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, lo;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, hi;\n\t}"
        : "=r"(h01), "=r"(h23)
        : "r"(w));
    e01 = __half22float2(*reinterpret_cast<const __half2*>(&h01));
    e23 = __half22float2(*reinterpret_cast<const __half2*>(&h23));
}

// Grid-wide barrier in two halves, so a block can do independent work between arriving and
// waiting. The workspace's arrival counter only grows, and every launch's barriers are complete
// when it ends, so at a launch's start the counter is a multiple of P (the grid size) up to the
// arrivals of this launch's first barrier: grid_base reads it once per block (thread 0, early
// in the launch, before its first arrival) and rounds down to that multiple; the launch's i-th barrier (i from 1) is complete once
// the counter reaches base + i P. grid_arrive: every thread of the block calls it after its
// writes; thread 0 adds one with a release reduction (no round trip; after a block barrier, so
// it publishes the whole block's writes). grid_wait: thread 0 waits, bounded, with acquire
// loads, then the block meets, so the block sees every block's writes made before their
// arrival. A wait that runs out records PROX_ERR_TIMEOUT and returns false.
static __device__ unsigned long long grid_base(GridBarrier* b) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(&b->arrived) : "memory");
    const unsigned long long P = gridDim.x;
    return v / P * P;
}

static __device__ void grid_arrive(GridBarrier* b) {
    __syncthreads();
    if (threadIdx.x == 0)
        asm volatile("red.release.gpu.global.add.u64 [%0], 1;" ::"l"(&b->arrived) : "memory");
}

static __device__ bool grid_wait(GridBarrier* b, unsigned long long target, int* s_flag, long long spin,
                          int* status) {
    if (threadIdx.x == 0) {
        int ok = 1;
        unsigned long long v;
        const long long t0 = clock64();
        while (true) {
            asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(&b->arrived) : "memory");
            if (v >= target) break;
            if (clock64() - t0 > spin) {
                set_status(status, PROX_ERR_TIMEOUT);
                ok = 0;
                break;
            }
        }
        *s_flag = ok;
    }
    __syncthreads();
    return *s_flag != 0;
}

static __device__ bool grid_barrier(GridBarrier* b, unsigned long long target, int* s_flag,
                             long long spin, int* status) {
    grid_arrive(b);
    return grid_wait(b, target, s_flag, spin, status);
}

// ------------------------------------------------------------------ 1. input selection

// Thread t owns inputs [t RUN, t RUN + RUN) (RUN a power of two; a run lies in one group and a
// group's runs are 128 / RUN aligned lanes of one warp). Writes per group g: s_rows[g][*] the
// kept inputs ascending (padded), s_qx[g][*] their codes, s_nq[g] the padded count / 4,
// s_sx[g] the activation scale.
template <int RUN>
__device__ void select_inputs(const FusedParams& p, uint32_t* keys, int* hist, int* wsum,
                              int16_t* s_rows, int8_t* s_qx, int* s_nq, float* s_sx) {
    constexpr int tpg = 128 / RUN;
    const int d = p.d, tid = threadIdx.x;
    const int lo = min(d, tid * RUN), hi = min(d, lo + RUN);
    const bool active = lo < hi;
    const int g = lo >> 7, gl = tid & (tpg - 1);
    float xv[RUN];
#pragma unroll
    for (int e4 = 0; e4 < RUN / 4; ++e4) {
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (active) v = __ldg(reinterpret_cast<const float4*>(p.x + lo) + e4);
        xv[4 * e4] = v.x;
        xv[4 * e4 + 1] = v.y;
        xv[4 * e4 + 2] = v.z;
        xv[4 * e4 + 3] = v.w;
        if (active)
            reinterpret_cast<uint4*>(keys)[key_quad<RUN, true>(tid, e4)] =
                make_uint4(__float_as_uint(v.x) & 0x7fffffffu, __float_as_uint(v.y) & 0x7fffffffu,
                           __float_as_uint(v.z) & 0x7fffffffu, __float_as_uint(v.w) & 0x7fffffffu);
    }
    // first radix pass here (counts of the keys' bits 30..20): inputs in bins at or above the
    // bin of the k_in-th largest are a superset of the kept ones, so each block can already ask
    // L2 for its share of those proxy rows (rows blk, blk + P, ...) while the selection finishes
    // and HBM would otherwise idle; a hint only
    for (int i = tid; i < 2048; i += NT) hist[i] = 0;
    __syncthreads();
    if (active)
#pragma unroll
        for (int e = 0; e < RUN; ++e) atomicAdd(&hist[(__float_as_uint(xv[e]) & 0x7fffffffu) >> 20], 1);
    __syncthreads();
    if (p.prefetch_codes) {
        int* sel = wsum + NW;
        block_find_bin<NT>(hist, 2048, p.k_in, wsum, sel);
        const uint32_t b1 = static_cast<uint32_t>(sel[0]);
        const int r = blockIdx.x + tid * gridDim.x;
        if (r < d && ((__float_as_uint(__ldg(p.x + r)) & 0x7fffffffu) >> 20) >= b1)
            prefetch_l2(p.codes + static_cast<size_t>(r) * p.F, static_cast<uint32_t>(p.F));
    }
    uint32_t T;
    int take, eq_total;
    block_select_kth<NT, RUN, true>(keys, d, p.k_in, hist, wsum, T, take, eq_total, nullptr, true,
                                    p.prefetch_codes != 0);
    uint64_t mine;
    block_take_topk<NT, RUN, true>(keys, d, T, take, eq_total, wsum, mine);
    // the group's scale: its largest kept magnitude / 127
    float m = 0.f;
#pragma unroll
    for (int e = 0; e < RUN; ++e)
        if ((mine >> e) & 1ull) m = fmaxf(m, fabsf(xv[e]));
#pragma unroll
    for (int o = tpg >> 1; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float sxg = __fdiv_rn(m, 127.0f);
    int8_t q8[RUN];
#pragma unroll
    for (int e = 0; e < RUN; ++e) {
        float q = 0.f;
        if (((mine >> e) & 1ull) && sxg != 0.f)
            q = fminf(127.f, fmaxf(-127.f, rintf(__fdiv_rn(xv[e], sxg))));
        q8[e] = static_cast<int8_t>(static_cast<int>(q));
    }
    // the group's kept inputs in ascending order: an inclusive scan over its lanes
    const int cnt = __popcll(mine);
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < tpg; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o, tpg);
        if (gl >= o) incl += y;
    }
    const int n_g = __shfl_sync(0xffffffffu, incl, tpg - 1, tpg);
    int last = -1;
#pragma unroll
    for (int e = 0; e < RUN; ++e)
        if ((mine >> e) & 1ull) last = lo + e;
#pragma unroll
    for (int o = tpg >> 1; o > 0; o >>= 1) last = max(last, __shfl_xor_sync(0xffffffffu, last, o));
    if (active) {
        int pos = incl - cnt;
#pragma unroll
        for (int e = 0; e < RUN; ++e) {
            if ((mine >> e) & 1ull) {
                s_rows[g * 128 + pos] = static_cast<int16_t>(lo + e);
                s_qx[g * 128 + pos] = q8[e];
                ++pos;
            }
        }
        if (gl == tpg - 1) {
            const int padded = (n_g + 3) & ~3;
            for (int q = n_g; q < padded; ++q) {
                s_rows[g * 128 + q] = static_cast<int16_t>(last);
                s_qx[g * 128 + q] = 0;
            }
            s_nq[g] = padded >> 2;
            s_sx[g] = sxg;
        }
        if (blockIdx.x == 0) {
            if (p.dbg_qx)
#pragma unroll
                for (int e = 0; e < RUN; ++e) p.dbg_qx[lo + e] = q8[e];
            if (p.dbg_sx && gl == 0) p.dbg_sx[g] = sxg;
        }
    }
}

// ------------------------------------------------------------------ 2. Stage-1 proxy GEMV

constexpr int kARow = 33;   // ints per (group, chunk) row of s_A: 32 values + 1 (bank spread)

// Tasks are (group g, part h) for h < H: the quads [nq h / H, nq (h + 1) / H) of group g, for
// every chunk of the tile. Lane l = gs CW + c of warp w serves task slot w GS + gs (GS =
// 32 / CW) for chunk c (16 channels), the slots looping over the tasks; a lane streams its
// task's quads with kDepth quads of loads in flight, then adds its exact group sums into
// s_A[(g CW + c) kARow + v], v = 2 ch + proj, with shared-memory atomics (the parts of a group
// meet there; integer adds, so their order does not matter). s_A must be zero on entry.
template <int CW>
__device__ void proxy_gemv(const FusedParams& p, int c0, int nch, const int16_t* s_rows,
                           const int8_t* s_qx, const int* s_nq, int* s_A) {
    constexpr int GS = 32 / CW;
    constexpr int kDepth = 3;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int c = lane & (CW - 1), gs = lane / CW;
    const bool act = c < nch;
    const size_t F = static_cast<size_t>(p.F);
    const uint8_t* cb = p.codes + c0 + 16 * (act ? c : 0);
    const int G = p.d >> 7;
    const int slots = NW * GS;
    int H = slots / G;
    H = H < 1 ? 1 : (H > 16 ? 16 : H);
    const int ntask = G * H;
    for (int task = warp * GS + gs; task < ntask; task += slots) {
        const int g = task / H, h = task - g * H;
        const int nq = s_nq[g];
        const int qa = nq * h / H, qb = nq * (h + 1) / H;
        const int16_t* rows = s_rows + g * 128;
        const uint32_t* qxw = reinterpret_cast<const uint32_t*>(s_qx + g * 128);
        int ag[16], au[16], corr = 0;
#pragma unroll
        for (int i = 0; i < 16; ++i) ag[i] = au[i] = 0;
        auto load = [&](uint4 (&w)[4], int q) {
            const short4 r = *reinterpret_cast<const short4*>(rows + 4 * q);
            if (act) {
                w[0] = ld_stream16(cb + static_cast<size_t>(r.x) * F);
                w[1] = ld_stream16(cb + static_cast<size_t>(r.y) * F);
                w[2] = ld_stream16(cb + static_cast<size_t>(r.z) * F);
                w[3] = ld_stream16(cb + static_cast<size_t>(r.w) * F);
            } else {
#pragma unroll
                for (int i = 0; i < 4; ++i) w[i] = make_uint4(0u, 0u, 0u, 0u);
            }
        };
        auto step = [&](const uint4 (&w)[4], int q) {
            const uint32_t q4 = qxw[q];
            corr = dp4a_us(0x08080808u, q4, corr);
#pragma unroll
            for (int wc = 0; wc < 4; ++wc) {
                const uint32_t w0 = wc == 0 ? w[0].x : wc == 1 ? w[0].y : wc == 2 ? w[0].z : w[0].w;
                const uint32_t w1 = wc == 0 ? w[1].x : wc == 1 ? w[1].y : wc == 2 ? w[1].z : w[1].w;
                const uint32_t w2 = wc == 0 ? w[2].x : wc == 1 ? w[2].y : wc == 2 ? w[2].z : w[2].w;
                const uint32_t w3 = wc == 0 ? w[3].x : wc == 1 ? w[3].y : wc == 2 ? w[3].z : w[3].w;
                const uint32_t a = __byte_perm(w0, w1, 0x5140), b = __byte_perm(w2, w3, 0x5140);
                const uint32_t cc = __byte_perm(w0, w1, 0x7362), dd = __byte_perm(w2, w3, 0x7362);
                const uint32_t t[4] = {__byte_perm(a, b, 0x5410), __byte_perm(a, b, 0x7632),
                                       __byte_perm(cc, dd, 0x5410), __byte_perm(cc, dd, 0x7632)};
#pragma unroll
                for (int ch = 0; ch < 4; ++ch) {
                    ag[4 * wc + ch] = dp4a_us(t[ch] & 0x0F0F0F0Fu, q4, ag[4 * wc + ch]);
                    au[4 * wc + ch] = dp4a_us(t[ch] & 0xF0F0F0F0u, q4, au[4 * wc + ch]);
                }
            }
        };
        uint4 w[kDepth][4];
#pragma unroll
        for (int j = 0; j < kDepth; ++j)
            if (qa + j < qb) load(w[j], qa + j);
        for (int q0 = qa; q0 < qb; q0 += kDepth) {
#pragma unroll
            for (int j = 0; j < kDepth; ++j) {
                const int q = q0 + j;
                if (q < qb) {
                    step(w[j], q);
                    if (q + kDepth < qb) load(w[j], q + kDepth);
                }
            }
        }
        if (act && qa < qb) {
            int* dst = s_A + (g * CW + c) * kARow;
#pragma unroll
            for (int ch = 0; ch < 16; ++ch) {
                atomicAdd(dst + 2 * ch, ag[ch] - corr);
                atomicAdd(dst + 2 * ch + 1, (au[ch] >> 4) - corr);
            }
        }
    }
}

// ------------------------------------------------------------------ 3. salience

// Thread (part, jl): channel jl of the tile over the part-th of the groups; the parts' double-
// float sums are then added in part order. Writes sigma, the tile's keys and (if hist) its
// counts per bin of bits 30..20 into s_hist. The group scales come from s_sc ([G][nchan], the
// tile's copy) when given, else from global memory.
template <int CW>
__device__ void salience(const FusedParams& p, int c0, int nch, const int* s_A, const float* s_sx,
                         float4* s_part, uint32_t* s_key, int* s_hist, bool hist,
                         const uint32_t* s_sc) {
    constexpr int NCH = 16 * CW;
    constexpr int PARTS = NT / NCH;
    const int tid = threadIdx.x, jl = tid % NCH, part = tid / NCH;
    const int G = p.d >> 7;
    const int ga = G * part / PARTS, gb = G * (part + 1) / PARTS;
    const int nchan = 16 * nch;
    DF tg{0.f, 0.f}, tu{0.f, 0.f};
    if (jl < nchan) {
        const int c = jl >> 4, ch = jl & 15;
        const int j = c0 + jl;
        for (int g0 = ga; g0 < gb; g0 += 8) {
            uint32_t sw8[8];   // eight groups' scales in flight at once
#pragma unroll
            for (int i = 0; i < 8; ++i)
                sw8[i] = g0 + i >= gb ? 0u
                         : s_sc ? s_sc[(g0 + i) * nchan + jl]   // the tile's scales, [G][nchan]
                                : __ldg(p.scales + static_cast<size_t>(g0 + i) * p.F + j);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int g = g0 + i;
                if (g < gb) {
                    const int* a = s_A + (g * CW + c) * kARow + 2 * ch;
                    const int Ag = a[0], Au = a[1];
                    const float sx = s_sx[g];
                    const float swg = __half2float(__ushort_as_half(static_cast<unsigned short>(sw8[i] & 0xFFFFu)));
                    const float swu = __half2float(__ushort_as_half(static_cast<unsigned short>(sw8[i] >> 16)));
                    tg = df_add(tg, df_scaled_int(sx, swg, Ag));
                    tu = df_add(tu, df_scaled_int(sx, swu, Au));
                    if (p.dbg_gate) p.dbg_gate[static_cast<size_t>(g) * p.F + j] = Ag;
                    if (p.dbg_up) p.dbg_up[static_cast<size_t>(g) * p.F + j] = Au;
                }
            }
        }
    }
    s_part[part * NCH + jl] = make_float4(tg.hi, tg.lo, tu.hi, tu.lo);
    __syncthreads();
    if (tid < nchan) {
        float4 a = s_part[tid];
        DF g2{a.x, a.y}, u2{a.z, a.w};
#pragma unroll
        for (int q = 1; q < PARTS; ++q) {
            const float4 b = s_part[q * NCH + tid];
            g2 = df_add(g2, DF{b.x, b.y});
            u2 = df_add(u2, DF{b.z, b.w});
        }
        const float sg = fabsf(silu_f(g2.hi + g2.lo) * (u2.hi + u2.lo));
        p.sigma[c0 + tid] = sg;
        s_key[tid] = __float_as_uint(sg);
        if (hist) atomicAdd(&s_hist[__float_as_uint(sg) >> 20], 1);
    }
}

// ------------------------------------------------------------------ 4. top-k

__device__ __forceinline__ int warp_sum(int v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Run by one whole warp: over the nbins (<= 256) bins of h taken from the highest down, the
// bin holding the remaining-th key (1 <= remaining <= the bins' total). sel[0] = the bin,
// sel[1] = keys in higher bins, sel[2] = the bin's count.
__device__ __forceinline__ void warp_find_digit(const int* h, int nbins, int remaining, int* sel) {
    const int lane = threadIdx.x & 31;
    int c[8], local = 0;
#pragma unroll
    for (int m = 0; m < 8; ++m) {
        const int r = lane * 8 + m;   // rank of the bin from the top
        c[m] = r < nbins ? h[nbins - 1 - r] : 0;
        local += c[m];
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    int run = incl - local;
    if (run < remaining && incl >= remaining) {
#pragma unroll
        for (int m = 0; m < 8; ++m) {
            if (run < remaining && run + c[m] >= remaining) {
                sel[0] = nbins - 1 - (lane * 8 + m);
                sel[1] = run;
                sel[2] = c[m];
            }
            run += c[m];
        }
    }
}

// Among the keys of a[0, n) whose bits 31..20 equal b1, taken in index order, marks the rem
// largest in the channel bitmap wbits (equal keys go to the lower index; ch[i] is a[i]'s
// channel, or i itself if ch is null). With cnt, a is a list of segments of `seg` slots and
// only the first cnt[w] slots of segment w hold keys. Radix passes of 8, 8 and 4 bits over bits 19..0; once
// the digit holding the rem-th key is taken whole, the passes stop there. dh: 256 ints.
static __device__ void rank_boundary(const uint32_t* a, const uint16_t* ch, int n, uint32_t b1, int rem,
                              uint32_t* wbits, int* dh, int* wsum, int* sel, const int* cnt = nullptr,
                              int seg = 0) {
    // slot i of a segmented list is live if it lies within its segment's count
    auto live = [&](int i) { return !cnt || (i % seg) < cnt[i / seg]; };
    const int tid = threadIdx.x;
    uint32_t P = b1;   // the key bits fixed so far: bits 31..s
    int s = 20;
    bool take_all = false;
    for (int pass = 0; pass < 3 && !take_all; ++pass) {
        const int sh = pass == 0 ? 12 : (pass == 1 ? 4 : 0);
        const int nbins = 1 << (s - sh);
        for (int i = tid; i < 256; i += NT) dh[i] = 0;
        __syncthreads();
        for (int i = tid; i < n; i += NT) {
            const uint32_t key = a[i];
            if (live(i) && (key >> s) == P) atomicAdd(&dh[(key >> sh) & (nbins - 1)], 1);
        }
        __syncthreads();
        if (tid < 32) warp_find_digit(dh, nbins, rem, sel);
        __syncthreads();
        rem -= sel[1];
        P = (P << (s - sh)) | static_cast<uint32_t>(sel[0]);
        take_all = sel[2] == rem;
        s = sh;
    }
    // winners: above P at bit s; equal to it: all of them, or (ties of whole keys) the first rem
    if (take_all) {
        for (int i = tid; i < n; i += NT) {
            const uint32_t key = a[i];
            if (live(i) && (key >> 20) == b1 && (key >> s) >= P) {
                const int c = ch ? ch[i] : i;
                atomicOr(&wbits[c >> 5], 1u << (c & 31));
            }
        }
        return;
    }
    const int R = (n + NT - 1) / NT;
    const int lo = tid * R < n ? tid * R : n, hi = lo + R < n ? lo + R : n;
    int eq = 0;
    for (int i = lo; i < hi; ++i) eq += live(i) && a[i] == P;
    int eq_all;
    int r = block_exclusive_scan<NT>(eq, wsum, eq_all);
    for (int i = lo; i < hi; ++i) {
        if (!live(i)) continue;
        const uint32_t key = a[i];
        bool win = (key >> 20) == b1 && key > P;
        if (key == P) win = r++ < rem;
        if (win) {
            const int c = ch ? ch[i] : i;
            atomicOr(&wbits[c >> 5], 1u << (c & 31));
        }
    }
}

// Shared memory of the top-k inside the region (bytes from its start).
constexpr int kTopkDigitsOff = 2048 * 4;   // the 256 digit counts, after the layer histogram
inline __host__ __device__ size_t topk_region_bytes(int F) {
    return kTopkKeysOff + static_cast<size_t>(F) * 4 + static_cast<size_t>(kCandCap) * 6 +
           static_cast<size_t>(F / 32) * 4 + 2 * NW * 4;
}

// The layer's top-k, taken by every block on its own from the salience and the histogram in
// global memory (one bulk copy of each). Channels in bins above b1, the bin of the k-th largest
// key, are taken for sure; the candidates of bin b1 are collected in channel order and ranked
// among themselves (rank_boundary marks the winners in a channel bitmap). Writes the block's
// slice [e0, e0 + nloc) of the ascending mask to s_list (and to p.idx if asked). Warp w reads
// the keys' quads [F/4 w / NW, F/4 (w + 1) / NW), lanes on consecutive quads; the passes over
// the keys are branch-free (a quad's four channels share one bitmap word).
static __device__ void layer_topk(const FusedParams& p, unsigned char* region, uint64_t* kbar,
                                  int* wsum, int* sel, int* s_list, int e0, int nloc) {
    const int F = p.F, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int* h2 = reinterpret_cast<int*>(region);                                     // [2048]
    int* dh = reinterpret_cast<int*>(region + kTopkDigitsOff);                    // [256]
    uint32_t* keys = reinterpret_cast<uint32_t*>(region + kTopkKeysOff);          // [F]
    uint32_t* ck = keys + F;                                                      // [kCandCap]
    uint16_t* cch = reinterpret_cast<uint16_t*>(ck + kCandCap);                   // [kCandCap]
    uint32_t* wbits = reinterpret_cast<uint32_t*>(cch + kCandCap);                // [F / 32]
    int* wa = reinterpret_cast<int*>(wbits + (F >> 5));                           // [2 NW]
    if (tid == 0) {
        mbar_arrive_expect_tx(kbar, static_cast<uint32_t>(F) * 4u + 2048u * 4u);
        bulk_g2s(keys, p.sigma, static_cast<uint32_t>(F) * 4u, kbar);
        bulk_g2s(h2, p.ctl->hist, 2048u * 4u, kbar);
    }
    for (int i = tid; i < (F >> 5); i += NT) wbits[i] = 0u;
    mbar_wait(kbar, 0u, p.spin, p.status);
    block_find_bin<NT>(h2, 2048, p.k, wsum, sel);
    const uint32_t b1 = static_cast<uint32_t>(sel[0]);
    const int rem = p.k - sel[1], nb1 = sel[2];
    const bool whole = nb1 == rem;   // every key of bin b1 is taken
    const int nq = F >> 2;
    const int qa = nq * warp / NW, qb = nq * (warp + 1) / NW;
    const uint4* k4p = reinterpret_cast<const uint4*>(keys);
    // pass 1: each warp counts its sure keys (bins above b1) and lists its candidates (bin b1)
    // in channel order in its own segment of the candidate area (ballots give the places)
    constexpr int seg = kCandCap / NW;
    const uint32_t lt = (1u << lane) - 1u;
    int ns = 0, nc = 0;
    for (int q0 = qa; q0 < qb; q0 += 32) {
        const int q = q0 + lane;
        const bool valid = q < qb;
        const uint4 v = valid ? k4p[q] : make_uint4(0u, 0u, 0u, 0u);
        const uint32_t kk[4] = {v.x, v.y, v.z, v.w};
        bool f[4];
        uint32_t m[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            ns += valid && (kk[e] >> 20) > b1;
            f[e] = valid && (kk[e] >> 20) == b1;
            m[e] = __ballot_sync(0xffffffffu, f[e]);
        }
        int pos = nc + __popc(m[0] & lt) + __popc(m[1] & lt) + __popc(m[2] & lt) + __popc(m[3] & lt);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            if (f[e] && pos < seg) {
                ck[warp * seg + pos] = kk[e];
                cch[warp * seg + pos] = static_cast<uint16_t>(4 * q + e);
            }
            pos += f[e];
        }
        nc += __popc(m[0]) + __popc(m[1]) + __popc(m[2]) + __popc(m[3]);
    }
    ns = warp_sum(ns);
    if (lane == 0) {
        wa[warp] = nc;
        wa[NW + warp] = ns;
    }
    __syncthreads();
    if (!whole) {
        bool listed = true;   // every warp's candidates fit its segment
        for (int w = 0; w < NW; ++w) listed = listed && wa[w] <= seg;
        if (listed) {
            rank_boundary(ck, cch, NW * seg, b1, rem, wbits, dh, wsum, sel, wa, seg);
        } else {
            rank_boundary(keys, nullptr, F, b1, rem, wbits, dh, wsum, sel);   // many near-equal keys
        }
        __syncthreads();
    }
    // each warp's taken count: its sure keys plus its winners (or its whole bin-b1 share)
    int won = wa[warp];
    if (!whole) {
        const int c0 = 4 * qa, c1 = 4 * qb;   // the warp's channels [c0, c1)
        int n = 0;
        for (int wd = (c0 >> 5) + lane; wd <= ((c1 - 1) >> 5); wd += 32) {
            uint32_t m = wbits[wd];
            const int lo = wd * 32;
            if (lo < c0) m &= ~0u << (c0 - lo);
            if (lo + 32 > c1) m &= (c1 - lo) >= 32 ? ~0u : ((1u << (c1 - lo)) - 1u);
            n += __popc(m);
        }
        won = warp_sum(n);
    }
    __syncthreads();   // every warp has read wa[warp]
    if (lane == 0) wa[warp] = wa[NW + warp] + won;
    __syncthreads();
    int base = 0, total = 0;
    for (int w = 0; w < NW; ++w) {
        const int v = wa[w];
        base += w < warp ? v : 0;
        total += v;
    }
    if (tid == 0 && total != p.k) set_status(p.status, PROX_ERR_BOUNDS);
    // pass 3: every taken channel's place in the ascending mask (ballots give the places)
    const uint32_t all_b1 = whole ? 0xFu : 0u;
    for (int q0 = qa; q0 < qb; q0 += 32) {
        const int q = q0 + lane;
        uint32_t tm = 0u;   // bit e: channel 4 q + e is taken
        if (q < qb) {
            const uint4 v = k4p[q];
            const uint32_t wb = ((wbits[q >> 3] >> ((4 * q) & 31)) | all_b1) & 0xFu;
            const uint32_t b[4] = {v.x >> 20, v.y >> 20, v.z >> 20, v.w >> 20};
#pragma unroll
            for (int e = 0; e < 4; ++e)
                tm |= static_cast<uint32_t>((b[e] > b1) | ((b[e] == b1) & ((wb >> e) & 1u))) << e;
        }
        uint32_t m[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) m[e] = __ballot_sync(0xffffffffu, (tm >> e) & 1u);
        int pos = base + __popc(m[0] & lt) + __popc(m[1] & lt) + __popc(m[2] & lt) + __popc(m[3] & lt);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            if (((tm >> e) & 1u) && pos >= e0 && pos < e0 + nloc) {
                s_list[pos - e0] = 4 * q + e;
                if (p.write_idx) p.idx[pos] = 4 * q + e;
            }
            pos += (tm >> e) & 1u;
        }
        base += __popc(m[0]) + __popc(m[1]) + __popc(m[2]) + __popc(m[3]);
    }
}

// ------------------------------------------------------------------ 5. Stage 2

struct S2Smem {
    unsigned char* stages;
    uint64_t* full;
    float* red;
};

// Stage 2 over s_list[0, nloc) for one token; the block's partial output to ypart_blk [d].
// Warps [0, NG WPG) form NG groups; group gi consumes channels gi, gi + NG, ... and owns the
// ring slots they land in (NG divides the ring size). Threads beyond the groups only join
// the block-wide steps.
template <int CPTMAX, bool FP8>
__device__ void stage2(const FusedParams& p, const int* s_list, int nloc, const S2Smem& sm,
                       float* ypart_blk) {
    const int d = p.d, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int NG = p.NG, WPG = p.WPG, CPT = p.CPT, GT = WPG * 32;
    const int nstage = 1 << p.nstage_log2, smask = nstage - 1;
    const uint32_t stage_bytes = static_cast<uint32_t>(p.row_bytes);
    const int gi = warp / WPG, gw = warp - gi * WPG, gtid = tid - gi * GT;
    const bool member = gi < NG;
    const bool leader = member && gtid == 0;
    const int nchunk = d >> 3;
    int next_issue = gi;
    auto issue = [&](int it) {
        const int st = it & smask;
        mbar_arrive_expect_tx(&sm.full[st], stage_bytes);
        bulk_g2s(sm.stages + static_cast<size_t>(st) * stage_bytes,
                 reinterpret_cast<const unsigned char*>(p.rows) + static_cast<size_t>(s_list[it]) * p.row_bytes,
                 stage_bytes, &sm.full[st]);
    };
    if (leader)
        for (; next_issue < nloc && next_issue < nstage; next_issue += NG) issue(next_issue);

    float2 xr[CPTMAX][4], yr[CPTMAX][4];
#pragma unroll
    for (int c = 0; c < CPTMAX; ++c) {
        const int q = c * GT + gtid;
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
        if (member && c < CPT && q < nchunk) {
            const float4* src = reinterpret_cast<const float4*>(p.x + q * 8);
            a = __ldg(src);
            b = __ldg(src + 1);
        }
        xr[c][0] = make_float2(a.x, a.y);
        xr[c][1] = make_float2(a.z, a.w);
        xr[c][2] = make_float2(b.x, b.y);
        xr[c][3] = make_float2(b.z, b.w);
#pragma unroll
        for (int m = 0; m < 4; ++m) yr[c][m] = make_float2(0.f, 0.f);
    }

    bool broke = false;
    int it = gi, slot = 0;
    if (member) {
        float* gred = sm.red + gi * 2 * 2 * WPG;
        for (; it < nloc; it += NG, slot ^= 1) {
            const int st = it & smask;
            const bool ok = mbar_wait(&sm.full[st], static_cast<uint32_t>(it >> p.nstage_log2) & 1u,
                                      p.spin, p.status);
            const uint16_t* sb =
                reinterpret_cast<const uint16_t*>(sm.stages + static_cast<size_t>(st) * stage_bytes);
            float2 ga = make_float2(0.f, 0.f), ua = ga;
            const unsigned char* sb8 = reinterpret_cast<const unsigned char*>(sb);
            if (ok) {
#pragma unroll
                for (int c = 0; c < CPTMAX; ++c) {
                    const int q = c * GT + gtid;
                    if (c < CPT && q < nchunk) {
                        if constexpr (FP8) {
                            const uint2 wg = *reinterpret_cast<const uint2*>(sb8 + q * 8);
                            const uint2 wu = *reinterpret_cast<const uint2*>(sb8 + d + q * 8);
                            float2 e0, e1, e2, e3;
                            e4m3x4_f32(wg.x, e0, e1);
                            e4m3x4_f32(wg.y, e2, e3);
                            ga = ffma2(xr[c][0], e0, ga);
                            ga = ffma2(xr[c][1], e1, ga);
                            ga = ffma2(xr[c][2], e2, ga);
                            ga = ffma2(xr[c][3], e3, ga);
                            e4m3x4_f32(wu.x, e0, e1);
                            e4m3x4_f32(wu.y, e2, e3);
                            ua = ffma2(xr[c][0], e0, ua);
                            ua = ffma2(xr[c][1], e1, ua);
                            ua = ffma2(xr[c][2], e2, ua);
                            ua = ffma2(xr[c][3], e3, ua);
                        } else {
                            const uint4 wg = *reinterpret_cast<const uint4*>(sb + q * 8);
                            const uint4 wu = *reinterpret_cast<const uint4*>(sb + d + q * 8);
                            ga = ffma2(xr[c][0], bf16x2_f32(wg.x), ga);
                            ga = ffma2(xr[c][1], bf16x2_f32(wg.y), ga);
                            ga = ffma2(xr[c][2], bf16x2_f32(wg.z), ga);
                            ga = ffma2(xr[c][3], bf16x2_f32(wg.w), ga);
                            ua = ffma2(xr[c][0], bf16x2_f32(wu.x), ua);
                            ua = ffma2(xr[c][1], bf16x2_f32(wu.y), ua);
                            ua = ffma2(xr[c][2], bf16x2_f32(wu.z), ua);
                            ua = ffma2(xr[c][3], bf16x2_f32(wu.w), ua);
                        }
                    }
                }
            }
            // gate sum to lanes 0-15, up sum to lanes 16-31, then across the warp
            float gsum = ga.x + ga.y, usum = ua.x + ua.y;
            {
                const bool upper = (lane & 16) != 0;
                const float send = upper ? gsum : usum;
                float r = (upper ? usum : gsum) + __shfl_xor_sync(0xffffffffu, send, 16);
#pragma unroll
                for (int off = 8; off > 0; off >>= 1) r += __shfl_xor_sync(0xffffffffu, r, off);
                if ((lane & 15) == 0) gred[(slot * 2 + (lane >> 4)) * WPG + gw] = r;
            }
            if (named_bar_or(1 + gi, GT, !ok)) {
                broke = true;
                break;
            }
            // every warp of the group is past channel it - NG: its slot takes the next copy
            if (leader && it - NG >= 0 && next_issue < nloc) {
                issue(next_issue);
                next_issue += NG;
            }
            float g = 0.f, u = 0.f;
            for (int w2 = 0; w2 < WPG; ++w2) {
                g += gred[(slot * 2) * WPG + w2];
                u += gred[(slot * 2 + 1) * WPG + w2];
            }
            float coef;
            if constexpr (FP8) {   // the rows' scales follow the codes
                const float4 sc = *reinterpret_cast<const float4*>(sb8 + 3 * d);
                g *= sc.x;
                u *= sc.y;
                coef = silu_f(g) * u * sc.z;
            } else {
                coef = silu_f(g) * u;
            }
            const float2 s2 = make_float2(coef, coef);
#pragma unroll
            for (int c = 0; c < CPTMAX; ++c) {
                const int q = c * GT + gtid;
                if (c < CPT && q < nchunk) {
                    if constexpr (FP8) {
                        const uint2 wd = *reinterpret_cast<const uint2*>(sb8 + 2 * d + q * 8);
                        float2 e0, e1, e2, e3;
                        e4m3x4_f32(wd.x, e0, e1);
                        e4m3x4_f32(wd.y, e2, e3);
                        yr[c][0] = ffma2(s2, e0, yr[c][0]);
                        yr[c][1] = ffma2(s2, e1, yr[c][1]);
                        yr[c][2] = ffma2(s2, e2, yr[c][2]);
                        yr[c][3] = ffma2(s2, e3, yr[c][3]);
                    } else {
                        const uint4 wd = *reinterpret_cast<const uint4*>(sb + 2 * d + q * 8);
                        yr[c][0] = ffma2(s2, bf16x2_f32(wd.x), yr[c][0]);
                        yr[c][1] = ffma2(s2, bf16x2_f32(wd.y), yr[c][1]);
                        yr[c][2] = ffma2(s2, bf16x2_f32(wd.z), yr[c][2]);
                        yr[c][3] = ffma2(s2, bf16x2_f32(wd.w), yr[c][3]);
                    }
                }
            }
        }
        if (broke && leader) {
            // copies this group issued but did not consume must land before the ring is reused
            for (int t = it; t < next_issue; t += NG)
                mbar_wait(&sm.full[t & smask], static_cast<uint32_t>(t >> p.nstage_log2) & 1u,
                          p.spin, p.status);
        }
    }
    // the groups' partial outputs added in group order (through the ring, now idle)
    const bool any_broke = named_bar_or(6, NT, broke) != 0;
    float* scratch = reinterpret_cast<float*>(sm.stages);   // [NG][d]
    if (!any_broke && member) {
#pragma unroll
        for (int c = 0; c < CPTMAX; ++c) {
            const int q = c * GT + gtid;
            if (c < CPT && q < nchunk) {
                float4* dst = reinterpret_cast<float4*>(scratch + static_cast<size_t>(gi) * d + q * 8);
                dst[0] = make_float4(yr[c][0].x, yr[c][0].y, yr[c][1].x, yr[c][1].y);
                dst[1] = make_float4(yr[c][2].x, yr[c][2].y, yr[c][3].x, yr[c][3].y);
            }
        }
    }
    __syncthreads();
    for (int i = tid; i < d / 4; i += NT) {
        float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
        if (!any_broke) {
            t = reinterpret_cast<const float4*>(scratch)[i];
            for (int g2 = 1; g2 < NG; ++g2) {
                const float4 u = reinterpret_cast<const float4*>(scratch + static_cast<size_t>(g2) * d)[i];
                t.x += u.x;
                t.y += u.y;
                t.z += u.z;
                t.w += u.w;
            }
        }
        reinterpret_cast<float4*>(ypart_blk)[i] = t;
    }
}

// ------------------------------------------------------------------ the kernel

template <int RUN, int CW, int CPTMAX, bool FP8>
__global__ void __launch_bounds__(NT, 1) fused_token_kernel(const FusedParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    const int tid = threadIdx.x, blk = blockIdx.x, P = gridDim.x;
    const int d = p.d, F = p.F, G = d >> 7;
    const int nstage = 1 << p.nstage_log2;
    // fixed part after the shared region (see fused_smem_bytes)
    unsigned char* region = smem;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.region_bytes);          // [24]
    int* s_list = reinterpret_cast<int*>(full + 24);                               // [kListMax]
    float* red = reinterpret_cast<float*>(s_list + kListMax);                      // [256]
    int* wsum = reinterpret_cast<int*>(red + 256);                                 // [NW + 8]
    int* sel = wsum + NW;                                                          // [3] + misc
    int* s_flag = sel + 4;
    uint32_t* s_key = reinterpret_cast<uint32_t*>(wsum + NW + 8);                 // [tile]
    float* s_sx = reinterpret_cast<float*>(s_key + kFusedTileMax);                 // [G <= 64]
    int* s_nq = reinterpret_cast<int*>(s_sx + 64);                                 // [G <= 64]
    // phase buffers inside the region
    const int sizeA = G * CW * kARow * 4;
    const int offP1 = max(sizeA, 4 * d + 2 * 2048 * 4);
    uint32_t* keys = reinterpret_cast<uint32_t*>(region);                          // phase 1
    int* hist = reinterpret_cast<int*>(region + 4 * d);                            // phase 1
    int* s_A = reinterpret_cast<int*>(region);                                     // phase 2-3
    int16_t* s_rows = reinterpret_cast<int16_t*>(region + offP1);                  // phase 1-2
    int8_t* s_qx = reinterpret_cast<int8_t*>(region + offP1 + G * 128 * 2);        // phase 1-2
    float4* s_part = reinterpret_cast<float4*>(region + offP1);                    // phase 3
    int* s_hist = reinterpret_cast<int*>(region + offP1 + NT * 16);                // phase 3
    const int offSc = offP1 + max(G * 128 * 3, NT * 16 + 2048 * 4);
    uint32_t* s_sc = reinterpret_cast<uint32_t*>(region + offSc);                  // phases 1-3

    if (tid == 0) {
        for (int i = 0; i < nstage; ++i) mbar_init(&full[i], 1);
        mbar_init(&full[kTopkBar], 1);
        mbar_init_fence();
    }
    // this block's Stage-1 tile: chunks [ca, cb) of 16 channels, whole units of kTileUnit
    // chunks (128 channels, so every row piece a block reads is a whole 128-byte line)
    const int nchunks = F >> 4;
    const int nunits = (nchunks + kTileUnit - 1) / kTileUnit;
    const int ca = min(nchunks, kTileUnit * (nunits * blk / P));
    const int cb = min(nchunks, kTileUnit * (nunits * (blk + 1) / P));
    const int c0 = 16 * ca, nch = cb - ca, nchan = 16 * nch;
    const bool stage1 = (p.mode & kFusedStage1) != 0;
    const bool select = (p.mode & kFusedSelect) != 0;
    if (stage1 && nch > 0) {
        // the tile's scales, needed after the GEMV: copied into shared memory (16-byte
        // cp.async pieces, waited for before the salience), or hinted into L2
        if (p.scales_smem) {
            const int per_row = nch * 4;   // 16-byte pieces of one group's nchan scales
            const uint32_t dst0 = static_cast<uint32_t>(__cvta_generic_to_shared(s_sc));
            for (int i = tid; i < G * per_row; i += NT) {
                const int g = i / per_row, c = i - g * per_row;
                asm volatile("cp.async.cg.shared.global [%0], [%1], 16;"
                             :: "r"(dst0 + static_cast<uint32_t>((g * nchan + 4 * c) * 4)),
                                "l"(p.scales + static_cast<size_t>(g) * F + c0 + 4 * c) : "memory");
            }
            asm volatile("cp.async.commit_group;" ::: "memory");
        } else if (tid < G) {
            prefetch_l2(p.scales + static_cast<size_t>(tid) * F + c0, static_cast<uint32_t>(nch) * 64u);
        }
    }
    __syncthreads();

    int nloc = 0;
    // the launch's barrier i completes at base + i P; only thread 0 waits, so only it reads the
    // base, here, while the first loads of x are in flight (long before its first arrival)
    const unsigned long long bar_base = tid == 0 ? grid_base(&p.ctl->bar) : 0ull;
    int bars = 0;      // grid barriers of this launch so far
    if (stage1) {
        select_inputs<RUN>(p, keys, hist, wsum, s_rows, s_qx, s_nq, s_sx);
        __syncthreads();
        for (int i = tid; i < G * CW * kARow; i += NT) s_A[i] = 0;   // over the dead keys
        __syncthreads();
        proxy_gemv<CW>(p, c0, nch, s_rows, s_qx, s_nq, s_A);
        __syncthreads();
        for (int i = tid; i < 2048; i += NT) s_hist[i] = 0;
        __syncthreads();
        if (p.scales_smem) asm volatile("cp.async.wait_all;" ::: "memory");
        __syncthreads();
        salience<CW>(p, c0, nch, s_A, s_sx, s_part, s_key, s_hist, select,
                     p.scales_smem ? s_sc : nullptr);
        __syncthreads();
        if (select) {
            for (int i = tid; i < 2048; i += NT)
                if (s_hist[i]) atomicAdd(&p.ctl->hist[i], s_hist[i]);
            grid_arrive(&p.ctl->bar);   // (1) arrive; wait below
        }
        if (select && (p.mode & kFusedStage2) && nchan > 0) {
            // while the mask is being agreed on, bring the rows of the tile's M most salient
            // channels (M = 60% of the tile's expected share of the mask) into L2, so HBM keeps
            // streaming; a hint only. A channel's rank in its tile is counted directly.
            const int M = static_cast<int>(0.6 * static_cast<double>(p.k) * nchan / F);
            if (tid < nchan && M >= 1) {
                const uint32_t key = s_key[tid];
                int above = 0;
                for (int j = 0; j < nchan; ++j) {
                    const uint32_t kj = s_key[j];
                    above += kj > key || (kj == key && j < tid);
                }
                if (above < M)
                    prefetch_l2(reinterpret_cast<const unsigned char*>(p.rows) + static_cast<size_t>(c0 + tid) * p.row_bytes,
                                static_cast<uint32_t>(p.row_bytes));
            }
        }
    }

    if (select) {
        // every block takes the whole top-k itself and keeps the slice [e0, e1) of the
        // ascending mask that is its Stage-2 share (writing that slice of the mask out as well)
        grid_wait(&p.ctl->bar, bar_base + static_cast<unsigned long long>(++bars) * P, s_flag, p.spin,
                  p.status);   // (1) salience complete
        const int e0 = static_cast<int>(static_cast<long long>(p.k) * blk / P);
        const int e1 = static_cast<int>(static_cast<long long>(p.k) * (blk + 1) / P);
        nloc = min(e1 - e0, kListMax);
        layer_topk(p, region, full + kTopkBar, wsum, sel, s_list, e0, nloc);
        __syncthreads();
        if (!(p.mode & kFusedStage2) && tid == 0) {
            // no later barrier: the last block to have read the histogram clears it
            if (atomicAdd(&p.ctl->readers, 1u) == static_cast<unsigned>(P) - 1) {
                for (int i = 0; i < 2048; ++i) p.ctl->hist[i] = 0;
                p.ctl->readers = 0u;
            }
        }
    } else if (p.mode & (kFusedDense | kFusedGiven)) {
        const int n = (p.mode & kFusedDense) ? F : p.k;
        const int e0 = static_cast<int>(static_cast<long long>(n) * blk / P);
        nloc = static_cast<int>(static_cast<long long>(n) * (blk + 1) / P) - e0;
        if (nloc > kListMax) {   // the host sizes the grid so this cannot happen
            if (tid == 0) set_status(p.status, PROX_ERR_BOUNDS);
            nloc = kListMax;
        }
        for (int i = tid; i < nloc; i += NT) {
            int j = (p.mode & kFusedDense) ? e0 + i : p.idx_in[e0 + i];
            if (j < 0 || j >= F) {
                set_status(p.status, PROX_ERR_BOUNDS);
                j = 0;
            }
            s_list[i] = j;
        }
    }

    if (p.mode & kFusedStage2) {
        __syncthreads();
        S2Smem sm{region, full, red};
        stage2<CPTMAX, FP8>(p, s_list, nloc, sm, p.ypart + static_cast<size_t>(blk) * d);
        grid_barrier(&p.ctl->bar, bar_base + static_cast<unsigned long long>(++bars) * P, s_flag,
                     p.spin, p.status);   // (2) partials written
        if (select) {   // every block read the histogram before its Stage 2: clear a share
            const int a = 2048 * blk / P, b = 2048 * (blk + 1) / P;
            for (int i = a + tid; i < b; i += NT) p.ctl->hist[i] = 0;
        }
        // block blk adds columns [n4 blk / P, n4 (blk + 1) / P) (float4 units) over all blocks
        const int n4 = d >> 2;
        const int q0 = static_cast<int>(static_cast<long long>(n4) * blk / P);
        const int q1 = static_cast<int>(static_cast<long long>(n4) * (blk + 1) / P);
        float4* s_red = reinterpret_cast<float4*>(region);   // [32][16]
        const int col = tid & 15, ps = tid >> 4;             // 16 columns x 32 partial slices
        for (int cbase = q0; cbase < q1; cbase += 16) {
            const int cc = cbase + col;
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
            if (cc < q1) {
                // every load of the thread's partial rows in flight at once, then added in order
                constexpr int kRows = kFusedMaxBlocks / 32;
                float4 v[kRows];
#pragma unroll
                for (int j = 0; j < kRows; ++j) {
                    const int pp = ps + 32 * j;
                    v[j] = pp < P ? __ldcg(reinterpret_cast<const float4*>(p.ypart + static_cast<size_t>(pp) * d) + cc)
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
                }
#pragma unroll
                for (int j = 0; j < kRows; ++j) {
                    acc.x += v[j].x;
                    acc.y += v[j].y;
                    acc.z += v[j].z;
                    acc.w += v[j].w;
                }
            }
            s_red[ps * 16 + col] = acc;
            __syncthreads();
            if (ps == 0 && cc < q1) {
                float4 t = s_red[col];
                for (int q = 1; q < 32; ++q) {
                    const float4 u = s_red[q * 16 + col];
                    t.x += u.x;
                    t.y += u.y;
                    t.z += u.z;
                    t.w += u.w;
                }
                reinterpret_cast<float4*>(p.y)[cc] = t;
            }
            __syncthreads();
        }
    }
}

// ------------------------------------------------------------------ host-side shape

struct FusedShape {
    int RUN, CW, CPTMAX, NG, WPG, CPT, nstage_log2;
    bool scales_smem;
    size_t region, smem;
};

// shared memory after the region: barriers, the Stage-2 list, reductions, the tile's keys,
// scales and quad counts (the carve at the top of the kernel)
constexpr size_t kFixedSmem = 24 * 8 + kListMax * 4 + 256 * 4 + (NW + 8) * 4 + kFusedTileMax * 4 +
                              64 * 4 * 2;
constexpr size_t kMaxSmem = 227 * 1024;

// Stage-2 consumer layout for one token: NG groups of WPG warps (at most 16 warps), CPT
// 16-byte chunks of the row per thread, two ring slots per group at least.
// ring stages of row_bytes each: a power of two (2 .. 16) within the shared-memory budget
inline int fused_nstage_log2(size_t row_bytes) {
    int lg = 1;
    while (lg < 4 && (row_bytes << (lg + 1)) <= kStage2SmemBudget) ++lg;
    return lg;
}

inline bool fused_shape(int d, int F, int sms, FusedShape& s, size_t row_bytes) {
    if (d < 128 || d > 8192 || d % 128 || F < 32 || F % 32) return false;
    if (sms < 1 || sms > kFusedMaxBlocks) return false;
    const int nchunks = F / 16;
    const int nunits = (nchunks + kTileUnit - 1) / kTileUnit;
    const int nch_max = kTileUnit * ((nunits + sms - 1) / sms);
    if (nch_max > 16) return false;
    if ((F + sms - 1) / sms > kListMax) return false;
    s.RUN = select_run(d, NT);
    if (s.RUN > 16) return false;
    s.CW = nch_max <= 4 ? 4 : (nch_max <= 8 ? 8 : 16);
    s.nstage_log2 = fused_nstage_log2(row_bytes);
    const int nstage = 1 << s.nstage_log2;
    const int nchunk = d / 8;
    s.NG = 0;
    for (int NG = 4; NG >= 1; NG >>= 1) {
        if (nstage < 2 * NG) continue;
        int WPG = 16 / NG;
        const int need = (nchunk + 31) / 32;
        if (WPG > need) WPG = need;
        const int CPT = (nchunk + 32 * WPG - 1) / (32 * WPG);
        if (CPT <= 4) {
            s.NG = NG;
            s.WPG = WPG;
            s.CPT = CPT;
            break;
        }
    }
    if (s.NG == 0) return false;
    s.CPTMAX = s.RUN <= 4 ? 2 : 4;
    if (s.CPT > s.CPTMAX) return false;
    const int G = d / 128;
    const size_t sizeA = static_cast<size_t>(G) * s.CW * kARow * 4;
    size_t offP1 = static_cast<size_t>(4) * d + 2 * 2048 * 4;
    if (sizeA > offP1) offP1 = sizeA;
    size_t p1 = static_cast<size_t>(G) * 128 * 3;              // rows (int16) + codes
    const size_t p3 = static_cast<size_t>(NT) * 16 + 2048 * 4;  // parts + histogram
    if (p3 > p1) p1 = p3;
    size_t region = offP1 + p1;
    const size_t p4 = topk_region_bytes(F);
    if (p4 > region) region = p4;
    // the tile's group scales [G][16 CW] during Stage 1, after the phase buffers
    const size_t sc_end = offP1 + p1 + static_cast<size_t>(G) * 16 * s.CW * 4;
    if (sc_end > region && align_up(sc_end, 128) + kFixedSmem <= kMaxSmem) region = sc_end;
    s.scales_smem = sc_end <= region;
    const size_t ring = static_cast<size_t>(nstage) * row_bytes;
    if (ring > region) region = ring;
    const size_t scratch = static_cast<size_t>(s.NG) * d * 4 > 32 * 16 * 16
                               ? static_cast<size_t>(s.NG) * d * 4 : 32 * 16 * 16;   // Stage-2 end
    if (scratch > region) region = scratch;
    s.region = align_up(region, 128);
    s.smem = s.region + kFixedSmem;
    return s.smem <= kMaxSmem;
}

using FusedFn = void (*)(const FusedParams);

// the instantiations of one row format (each in its own translation unit)
FusedFn fused_fn_bf16(const FusedShape& s);
FusedFn fused_fn_fp8(const FusedShape& s);

}  // namespace fused_detail
}  // namespace prox

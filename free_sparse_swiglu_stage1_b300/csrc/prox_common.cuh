// Device helpers shared by the Prox kernels: status word, bounded waits, mbarrier and bulk
// copy wrappers (inline PTX for sm_103a), bf16 unpacking, block-level scans and the
// block radix select used for both top-k selections of the method.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>

#include "../../include/prox.h"

namespace prox {

// ---------------------------------------------------------------------------------------
// Workspace control block (first bytes of every workspace)
// ---------------------------------------------------------------------------------------
struct Control {
    int      status;          // first device-side error code, 0 when fine
    int      pad0;
    long long spin_limit;     // cycles a bounded wait may spin before giving up
    int      union_count;     // size of the batch union (device-side result)
    int      pad1[3];
};
static_assert(sizeof(Control) <= 256, "control block");

constexpr long long kDefaultSpinCycles = 4000000000LL;   // about two seconds at 2 GHz

__device__ __forceinline__ void set_status(int* status, int code) {
    atomicCAS(status, 0, code);
}

// ---------------------------------------------------------------------------------------
// mbarrier and bulk-copy wrappers
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Waits for the phase with the given parity to complete, for at most `limit` cycles.
// Returns false (and records PROX_ERR_TIMEOUT) if the wait ran out.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, long long limit,
                                          int* status) {
    if (mbar_try_wait(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_try_wait(bar, parity)) {
        if (clock64() - t0 > limit) {
            set_status(status, PROX_ERR_TIMEOUT);
            return false;
        }
    }
    return true;
}

// One bulk copy global -> this CTA's shared memory, completing on `bar` with tx bytes.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// Programmatic dependent launch: wait for the previous grid's results / let the next grid
// start its prologue. Both are no-ops when the launch carried no such dependency.
__device__ __forceinline__ void grid_dep_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_dep_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------------------
// bf16 helpers
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// ---------------------------------------------------------------------------------------
// Double-float (hi, lo) accumulation with FMA-exact products
// ---------------------------------------------------------------------------------------
struct DF {
    float hi, lo;
};

__device__ __forceinline__ DF df_add(DF a, DF b) {
    const float s = a.hi + b.hi;
    const float bb = s - a.hi;
    float e = (a.hi - (s - bb)) + (b.hi - bb);
    e += a.lo + b.lo;
    const float hi = s + e;
    return DF{hi, e - (hi - s)};
}

// (p * q) * n as a double-float, with p, q binary32 and n an integer below 2^24 in size.
// p*q is split exactly by FMA; the (hi part) * n product too; the low part's product is
// rounded once, which is far below the precision the salience needs.
// The same with the integer given as a float that holds it exactly.
__device__ __forceinline__ DF df_scaled(float p, float q, float nf) {
    const float ph = __fmul_rn(p, q);
    const float pl = __fmaf_rn(p, q, -ph);
    const float th = __fmul_rn(ph, nf);
    const float tl = __fmaf_rn(ph, nf, -th) + __fmul_rn(pl, nf);
    const float hi = th + tl;
    return DF{hi, tl - (hi - th)};
}
__device__ __forceinline__ DF df_scaled_int(float p, float q, int n) {
    return df_scaled(p, q, static_cast<float>(n));
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + expf(-z)); }

// ---------------------------------------------------------------------------------------
// Block-level helpers (all threads of the block must call them)
// ---------------------------------------------------------------------------------------

// Exclusive prefix sum over the block in thread order; `total` receives the block sum.
// `wsum` is NT/32 ints of shared memory. Two barriers; the caller may reuse wsum only after
// another barrier.
template <int NT>
__device__ __forceinline__ int block_exclusive_scan(int v, int* wsum, int& total) {
    constexpr int NW = NT / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    const int wv = lane < NW ? wsum[lane] : 0;
    int before = lane < warp ? wv : 0;
    int all = wv;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        before += __shfl_xor_sync(0xffffffffu, before, o);
        all += __shfl_xor_sync(0xffffffffu, all, o);
    }
    total = all;
    __syncthreads();
    return before + x - v;
}

// Length of the contiguous run of keys each thread owns in the block-wide selections: a
// power of two, at least 4 (so runs are read as 16-byte vectors).
__host__ __device__ inline int select_run(int n, int nt) {
    const int need = (n + nt - 1) / nt;
    int r = 4;
    while (r < need) r <<= 1;
    return r;
}

// The uint4 slot that holds the i4-th group of 4 keys of thread t's run of RUN keys. Plain:
// t * RUN / 4 + i4 (runs contiguous). Swizzled (SWZ): the slot inside the run is XORed with a
// function of t chosen so that the threads of a warp reading their i4-th groups at once touch
// different bank groups (contiguous runs of 32 or more bytes per thread otherwise conflict).
template <int RUN, bool SWZ>
__device__ __forceinline__ int key_quad(int t, int i4) {
    constexpr int R4 = RUN / 4;
    if constexpr (!SWZ || R4 == 1) {
        return t * R4 + i4;
    } else {
        const int s = R4 >= 8 ? (t & 7) : ((t * R4 / 8) & (R4 - 1));
        return t * R4 + (i4 ^ s);
    }
}

// Over the bins of histogram h taken in descending order, finds the bin where the running
// count reaches `remaining` (1 <= remaining <= total). Writes sel[0] = that bin, sel[1] = the
// count in the bins above it, sel[2] = the count in the bin. nbins <= 2048, a multiple of NT
// or at most NT. Two barriers; every thread calls it; sel and wsum are shared memory
// (wsum NT/32 ints, sel 3 ints), read sel only after the call.
template <int NT>
__device__ __forceinline__ void block_find_bin(const int* h, int nbins, int remaining, int* wsum,
                                               int* sel) {
    constexpr int NW = NT / 32;
    constexpr int BPT = 2048 / NT > 0 ? 2048 / NT : 1;   // bins per thread at most
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int cnt[BPT], local = 0;
#pragma unroll
    for (int m = 0; m < BPT; ++m) {
        const int r = tid * BPT + m;
        cnt[m] = r < nbins ? h[nbins - 1 - r] : 0;
        local += cnt[m];
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    int before = (lane < warp && lane < NW) ? wsum[lane] : 0;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) before += __shfl_xor_sync(0xffffffffu, before, o);
    const int excl = before + incl - local;
    if (excl < remaining && excl + local >= remaining) {
        int runc = excl;
#pragma unroll
        for (int m = 0; m < BPT; ++m) {
            if (runc < remaining && runc + cnt[m] >= remaining) {
                sel[0] = nbins - 1 - (tid * BPT + m);
                sel[1] = runc;
                sel[2] = cnt[m];
            }
            runc += cnt[m];
        }
    }
    __syncthreads();
}

// Radix select over n keys (bit 31 clear, n a multiple of 4) held in shared memory, in up to
// three passes of 11, 11 and 9 bits. Thread t scans the run [t*RUN, t*RUN + RUN). Finds T, the
// k-th largest key (1 <= k <= n); take_eq, how many keys equal to T belong to the top k when
// ties go to the lowest indices; and eq_total, how many keys equal T. If a pass finds that the
// bin holding the k-th key is taken whole, it stops there: T is then the bin's lowest value
// and take_eq = eq_total = 2^30, so "key > T, or key == T" selects exactly the top k. `hist` is 2 * 2048 ints and
// `wsum` NT/32 + 4 ints of shared memory. If hist0 is not null it holds the first pass's
// 2048-bin histogram of the keys' bits 30..20 (built by whoever produced the keys), and that
// pass only reads it.
// If hist_ready, hist[0, 2048) already holds that first-pass histogram in shared memory; if
// also bin_ready, wsum[NT/32 ..] already holds block_find_bin's result for it (k-th key).
template <int NT, int RUN, bool SWZ = false>
__device__ void block_select_kth(const uint32_t* keys, int n, int k, int* hist, int* wsum,
                                 uint32_t& T, int& take_eq, int& eq_total,
                                 const int* hist0 = nullptr, bool hist_ready = false,
                                 bool bin_ready = false) {
    constexpr int NW = NT / 32;
    const int tid = threadIdx.x;
    const int lo = tid * RUN;
    const int nv = lo < n ? (n - lo < RUN ? n - lo : RUN) : 0;   // keys in this thread's run
    int* sel = wsum + NW;
    uint32_t prefix = 0, pmask = 0;
    int remaining = k;
    if (!hist_ready) {
        for (int i = tid; i < 2048; i += NT) hist[i] = hist0 ? __ldcg(hist0 + i) : 0;
        __syncthreads();
    }
    const bool first_ready = hist_ready || hist0;
#pragma unroll 1
    for (int p = 0; p < 3; ++p) {
        const int shift = p == 0 ? 20 : (p == 1 ? 9 : 0);
        const int nbins = p == 2 ? 512 : 2048;
        const uint32_t dmask = static_cast<uint32_t>(nbins - 1);
        int* h = hist + (p & 1) * 2048;
        if (p > 0 || !first_ready) {
#pragma unroll
            for (int i4 = 0; i4 < RUN / 4; ++i4) {
                if (4 * i4 < nv) {
                    const uint4 kk = reinterpret_cast<const uint4*>(keys)[key_quad<RUN, SWZ>(tid, i4)];
                    const uint32_t k4[4] = {kk.x, kk.y, kk.z, kk.w};
#pragma unroll
                    for (int m = 0; m < 4; ++m)
                        if ((k4[m] & pmask) == prefix) atomicAdd(&h[(k4[m] >> shift) & dmask], 1);
                }
            }
        }
        if (p < 2) {   // clear the other buffer for the next pass
            int* h2 = hist + ((p + 1) & 1) * 2048;
            for (int i = tid; i < 2048; i += NT) h2[i] = 0;
        }
        __syncthreads();
        if (p > 0 || !bin_ready) block_find_bin<NT>(h, nbins, remaining, wsum, sel);
        const uint32_t dig = static_cast<uint32_t>(sel[0]);
        remaining -= sel[1];
        eq_total = sel[2];
        prefix |= dig << shift;
        pmask |= dmask << shift;
        if (p < 2 && eq_total == remaining) {
            // the whole bin is taken: every key >= the bin's lowest value is in the top k
            T = prefix;
            take_eq = eq_total = 1 << 30;
            __syncthreads();
            return;
        }
    }
    T = prefix;
    take_eq = remaining;
    __syncthreads();   // sel and wsum are free again
}

// Marks the top k given (T, take_eq, eq_total) from block_select_kth: a key is taken if it
// is above T, or equal to T and among the first take_eq equal keys in index order. Thread t
// owns the run [t*RUN, t*RUN + RUN) (RUN <= 64); `take` receives one bit per element of the
// run. Returns the number taken in the run. `wsum` as for the scan.
template <int NT, int RUN, bool SWZ = false>
__device__ __forceinline__ int block_take_topk(const uint32_t* keys, int n, uint32_t T,
                                               int take_eq, int eq_total, int* wsum,
                                               uint64_t& take) {
    const int lo = static_cast<int>(threadIdx.x) * RUN;
    const int nv = lo < n ? (n - lo < RUN ? n - lo : RUN) : 0;
    int e = 0;
    if (take_eq != eq_total) {   // only a partial tie needs the rank of equal keys
        int eq = 0;
#pragma unroll
        for (int i = 0; i < RUN; ++i)
            if (i < nv) eq += keys[4 * key_quad<RUN, SWZ>(threadIdx.x, i >> 2) + (i & 3)] == T;
        int eq_all;
        e = block_exclusive_scan<NT>(eq, wsum, eq_all);
    }
    take = 0ull;
    int cnt = 0;
#pragma unroll
    for (int i4 = 0; i4 < RUN / 4; ++i4) {
        if (4 * i4 < nv) {
            const uint4 kk = reinterpret_cast<const uint4*>(keys)[key_quad<RUN, SWZ>(threadIdx.x, i4)];
            const uint32_t k4[4] = {kk.x, kk.y, kk.z, kk.w};
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                bool t = k4[m] > T;
                if (k4[m] == T) {
                    t = e < take_eq;
                    ++e;
                }
                if (t) {
                    take |= 1ull << (4 * i4 + m);
                    ++cnt;
                }
            }
        }
    }
    return cnt;
}

}  // namespace prox

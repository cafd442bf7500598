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
__device__ __forceinline__ DF df_scaled_int(float p, float q, int n) {
    const float ph = __fmul_rn(p, q);
    const float pl = __fmaf_rn(p, q, -ph);
    const float nf = static_cast<float>(n);
    const float th = __fmul_rn(ph, nf);
    const float tl = __fmaf_rn(ph, nf, -th) + __fmul_rn(pl, nf);
    const float hi = th + tl;
    return DF{hi, tl - (hi - th)};
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + expf(-z)); }

// ---------------------------------------------------------------------------------------
// Block-level helpers (all threads of the block must call them)
// ---------------------------------------------------------------------------------------
template <int NT>
__device__ __forceinline__ int block_exclusive_scan(int v, int* smem_warp, int& total) {
    constexpr int NW = NT / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) smem_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = lane < NW ? smem_warp[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < NW) smem_warp[lane] = w;   // inclusive warp totals
    }
    __syncthreads();
    const int before = warp > 0 ? smem_warp[warp - 1] : 0;
    total = smem_warp[NW - 1];
    __syncthreads();
    return before + x - v;
}

// Radix select over n uint32 keys held in shared memory: finds T, the k-th largest key,
// and how many keys equal to T belong to the top k (take_eq >= 1) when the ties among them
// are given to the lowest indices. 1 <= k <= n. `hist` is 256 ints of shared memory,
// `sel` 4 ints of shared memory.
template <int NT>
__device__ void block_radix_select(const uint32_t* keys, int n, int k, int* hist, int* sel,
                                   uint32_t& T, int& take_eq) {
    const int tid = threadIdx.x, lane = tid & 31;
    uint32_t prefix = 0, pmask = 0;
    int remaining = k;
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int b = tid; b < 256; b += NT) hist[b] = 0;
        __syncthreads();
        for (int base = 0; base < n; base += NT) {
            const int i = base + tid;
            const bool act = i < n && ((keys[i] & pmask) == prefix);
            const unsigned amask = __ballot_sync(0xffffffffu, act);
            if (act) {
                const int dig = (keys[i] >> shift) & 255;
                const unsigned peers = __match_any_sync(amask, dig);
                if (lane == __ffs(peers) - 1) atomicAdd(&hist[dig], __popc(peers));
            }
        }
        __syncthreads();
        if (tid < 32) {
            // lane L owns digits 255-8L .. 248-8L (descending); find the digit where the
            // running count from the top reaches `remaining`
            int cnt[8], s = 0;
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                cnt[m] = hist[255 - 8 * lane - m];
                s += cnt[m];
            }
            int incl = s;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            const int excl = incl - s;
            if (excl < remaining && incl >= remaining) {
                int run = excl;
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    if (run < remaining && run + cnt[m] >= remaining) {
                        sel[0] = 255 - 8 * lane - m;
                        sel[1] = run;
                    }
                    run += cnt[m];
                }
            }
        }
        __syncthreads();
        const int dig = sel[0];
        remaining -= sel[1];
        prefix |= static_cast<uint32_t>(dig) << shift;
        pmask |= 255u << shift;
        __syncthreads();
    }
    T = prefix;
    take_eq = remaining;
}

// Writes, in ascending index order, every i with keys[i] > T plus the first take_eq
// indices with keys[i] == T. Each thread scans a contiguous run of indices.
// Never writes more than max_out entries. Returns the number selected (== k).
// `scan_smem` is NT/32 ints of shared memory.
template <int NT>
__device__ int block_compact_topk(const uint32_t* keys, int n, uint32_t T, int take_eq,
                                  int32_t* out, int max_out, int* scan_smem) {
    const int tid = threadIdx.x;
    const int per = (n + NT - 1) / NT;
    const int lo = min(n, tid * per), hi = min(n, lo + per);
    int eq = 0;
    for (int i = lo; i < hi; ++i) eq += keys[i] == T;
    int eq_total;
    int eq_before = block_exclusive_scan<NT>(eq, scan_smem, eq_total);
    int cnt = 0;
    {
        int e = eq_before;
        for (int i = lo; i < hi; ++i) {
            const uint32_t kk = keys[i];
            if (kk > T) ++cnt;
            else if (kk == T) { cnt += e < take_eq; ++e; }
        }
    }
    int total;
    int pos = block_exclusive_scan<NT>(cnt, scan_smem, total);
    int e = eq_before;
    for (int i = lo; i < hi; ++i) {
        const uint32_t kk = keys[i];
        bool take = kk > T;
        if (kk == T) { take = e < take_eq; ++e; }
        if (take && pos < max_out) out[pos++] = i;
    }
    return total;
}

}  // namespace prox

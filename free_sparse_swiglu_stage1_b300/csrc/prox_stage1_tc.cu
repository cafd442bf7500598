// Stage 1 of a batch of tokens on the tensor cores (tcgen05, sm_103a).
//
// Method: Stage 1 of the Prox FFN (technical summary, Stage 1 "Proxy Activation" and "Mask
// Generation"): per token, the INT4 proxies of W_gate and W_up multiply the int8 codes of the
// kept inputs; per group g of 128 inputs the exact integer A[g, j] = sum q[j, i] qx[i] is
// scaled by sx[g] sw[g, j], and the salience is |SiLU(g~_j) u~_j|.
//
// For a batch the proxy GEMV is a contraction over the batch: with the codes taken as f16
// (q in [-7, 7], qx in [-127, 127], both exact) the tensor cores form the per-group sums of
// products with fp32 accumulation, which is exact here (|A| <= 128 * 7 * 127 < 2^24), so
// A[g, j] is the same integer the CUDA-core kernel forms with dp4a. The activations are dense:
// a dropped input has qx = 0 (at a batch's union of kept inputs, most rows are read anyway).
//
// Work split: one CTA per SM owns a window of about F / P consecutive channels, split into
// M-tiles of at most 112 channels (one 128-channel TMA box from a 16-byte aligned start).
// Per M-tile and group, two stages of 64 inputs:
//   warp 0        TMA: the codes tile [64 inputs][128 channels] (bytes, input-major as packed)
//                 and the activation tile [16 tokens][64 inputs] (f16, 128-byte swizzle);
//   warps 1..8    unpack the nibbles into two f16 A operands (gate, up) in the MN-major
//                 128-byte-swizzled layout (channels contiguous), 16 codes per thread-copy;
//   warps 9, 10   MMAs D_gate, D_up [128 channels x 16 tokens] += A . qx^T (K = 64 per stage),
//                 one issuing thread per projection; the group's accumulators alternate between
//                 two tensor-memory buffers;
//   warps 11..18  per group, read the exact integers of their channel (one TMEM lane per
//                 thread; two warps per lane quarter, 8 tokens each), scale them by sx sw into
//                 double-float sums (the same arithmetic as the CUDA-core kernel, groups in
//                 ascending order); after the last group write the salience and count its top
//                 11 bits into the top-k's histogram.
// Every wait is bounded (PROX_ERR_TIMEOUT), copies are drained and tensor memory freed.
#include "prox_tc.cuh"

namespace prox {

namespace {

constexpr int kUnpackers = 256;                      // warps 1..8
constexpr int kMmaWarp = 9;                          // gate MMAs (and tensor memory)
constexpr int kMmaWarpUp = 10;                       // up MMAs
constexpr int kEpilogue = 256;                       // warps 11..18: two per TMEM lane quarter
constexpr int kThreads = 32 + kUnpackers + 64 + kEpilogue;   // 608
constexpr int kCodeSlots = 6;
constexpr uint32_t kCodeBytes = 64 * 128;            // 64 inputs x 128 channels
constexpr uint32_t kQxBytes = 16 * 128;              // 16 tokens x 64 inputs, f16
constexpr uint32_t kCodeSlot = kCodeBytes + kQxBytes;
constexpr int kASlots = 3;
constexpr uint32_t kAProj = 16 * 1024;               // one projection: 2 MN-atoms x 8 K-groups
constexpr uint32_t kASlot = 2 * kAProj;
constexpr int kWin = 112;                            // channels of an M-tile
constexpr uint32_t kTmemCols = 64;                   // 2 buffers x (gate 16 | up 16)
constexpr int kTokens = 16;

// barrier indices
constexpr int kCFull = 0, kCEmpty = kCodeSlots, kAFull = 2 * kCodeSlots,
              kAEmpty = kAFull + kASlots, kDFull = kAEmpty + kASlots, kDEmpty = kDFull + 2,
              kDone = kDEmpty + 2, kNumBars = kDone + 2;

struct S1Smem {
    uint32_t code, a, sx, bars, misc, total;
};
__host__ __device__ inline S1Smem s1_smem_layout(int G) {
    S1Smem L;
    uint32_t o = 0;
    L.code = o;
    o += kCodeSlots * kCodeSlot;
    L.a = o;
    o += kASlots * kASlot;
    L.sx = o;
    o += static_cast<uint32_t>(kTokens * G) * 4;
    o = (o + 7u) & ~7u;
    L.bars = o;
    o += kNumBars * 8;
    L.misc = o;
    o += 16;
    L.total = o + 1024;
    return L;
}

// four code bytes (channels c..c+3 of one input) -> f16 pairs of the gate and up codes q - 8
__device__ __forceinline__ void unpack4(uint32_t w, uint32_t& g01, uint32_t& g23, uint32_t& u01,
                                        uint32_t& u23) {
    const uint32_t lo = __byte_perm(w, 0u, 0x4140);   // 16-bit lanes: byte 0, byte 1
    const uint32_t hi = __byte_perm(w, 0u, 0x4342);   // byte 2, byte 3
    // 0x6400 | n is f16 1024 + n; subtracting 1032 leaves n - 8 exactly
    const __half2 off = __halves2half2(__ushort_as_half(0x6408), __ushort_as_half(0x6408));
    auto cv = [&](uint32_t v) {
        const __half2 h = __hsub2(*reinterpret_cast<const __half2*>(&v), off);
        return *reinterpret_cast<const uint32_t*>(&h);
    };
    g01 = cv((lo & 0x000F000Fu) | 0x64006400u);
    g23 = cv((hi & 0x000F000Fu) | 0x64006400u);
    u01 = cv(((lo >> 4) & 0x000F000Fu) | 0x64006400u);
    u23 = cv(((hi >> 4) & 0x000F000Fu) | 0x64006400u);
}

__global__ void __launch_bounds__(kThreads, 1)
stage1_tc_kernel(const __grid_constant__ CUtensorMap tm_codes, const __grid_constant__ CUtensorMap tm_qx,
                 const uint32_t* __restrict__ scales, const float* __restrict__ sx, int d, int F,
                 int B, float* __restrict__ sigma, int* __restrict__ ghist,
                 int32_t* __restrict__ dbg_gate, int32_t* __restrict__ dbg_up, long long spin,
                 int* status) {
    constexpr uint32_t kIdesc = mma_idesc(128, kTokens, 1, 0, kFmtF16);
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const int G = d >> 7;
    const S1Smem SL = s1_smem_layout(G);
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    unsigned char* sbase = smem_raw + (base - raw);
    float* s_sx = reinterpret_cast<float*>(sbase + SL.sx);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sbase + SL.bars);
    uint32_t* misc = reinterpret_cast<uint32_t*>(sbase + SL.misc);   // [0] tmem, [1] issued, [2] consumed
    const uint32_t code0 = base + SL.code, a0 = base + SL.a;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int P = gridDim.x;
    const int c_lo = static_cast<int>(static_cast<long long>(F) * blockIdx.x / P);
    const int c_hi = static_cast<int>(static_cast<long long>(F) * (blockIdx.x + 1) / P);
    const int nmt = (c_hi - c_lo + kWin - 1) / kWin;
    const int total = nmt * G * 2;   // stages

    if (tid == 0) {
        for (int i = 0; i < kCodeSlots; ++i) {
            mbar_init(&bars[kCFull + i], 1);
            mbar_init(&bars[kCEmpty + i], kUnpackers / 32 + 2);
        }
        for (int i = 0; i < kASlots; ++i) {
            mbar_init(&bars[kAFull + i], kUnpackers / 32);
            mbar_init(&bars[kAEmpty + i], 2);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars[kDFull + i], 2);
            mbar_init(&bars[kDEmpty + i], kEpilogue / 32);
            mbar_init(&bars[kDone + i], 1);
        }
        mbar_init_fence();
        misc[1] = 0;
        misc[2] = 0;
        asm volatile("prefetch.tensormap [%0];" ::"l"(&tm_codes) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(&tm_qx) : "memory");
    }
    if (warp == kMmaWarp) tmem_alloc(&misc[0], kTmemCols);

    grid_dep_wait();
    grid_dep_launch();
    for (int i = tid; i < kTokens * G; i += kThreads) {
        const int b = i / G;
        s_sx[i] = b < B ? sx[i] : 0.f;   // sx [B][G] (token tiles are consecutive)
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];

    if (total > 0 && warp == 0 && lane == 0) {
        // ---------------------------------------------------------------- TMA copies
        uint32_t s = 0;
        for (; s < static_cast<uint32_t>(total); ++s) {
            const int c = s % kCodeSlots;
            if (s >= kCodeSlots &&
                !mbar_wait(&bars[kCEmpty + c], ((s / kCodeSlots) - 1) & 1, spin, status))
                break;
            const int j = s >> 1, h = s & 1, mt = j / G, g = j - mt * G;
            const int x0 = (c_lo + mt * kWin) & ~15;
            const int row = g * 128 + h * 64;
            const uint32_t dst = code0 + c * kCodeSlot;
            mbar_arrive_expect_tx(&bars[kCFull + c], kCodeSlot);
            tma_tile_2d(dst, &tm_codes, x0, row, &bars[kCFull + c]);
            tma_tile_2d(dst + kCodeBytes, &tm_qx, row, 0, &bars[kCFull + c]);
        }
        misc[1] = s;
    } else if (total > 0 && warp >= 1 && warp <= kUnpackers / 32) {
        // ---------------------------------------------------------------- unpack codes
        const int ut = tid - 32;
        for (int s = 0; s < total; ++s) {
            const int c = s % kCodeSlots, a = s % kASlots;
            if (!mbar_wait(&bars[kCFull + c], (s / kCodeSlots) & 1, spin, status)) break;
            if (s >= kASlots && !mbar_wait(&bars[kAEmpty + a], ((s / kASlots) - 1) & 1, spin, status))
                break;
            const unsigned char* cs = sbase + SL.code + c * kCodeSlot;
            unsigned char* as = sbase + SL.a + a * kASlot;
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int piece = ut + k * kUnpackers;   // 512 pieces of 16 codes
                const int r = piece >> 3, cc = piece & 7;
                const uint4 w = *reinterpret_cast<const uint4*>(cs + r * 128 + cc * 16);
                uint4 g0, g1, u0, u1;
                unpack4(w.x, g0.x, g0.y, u0.x, u0.y);
                unpack4(w.y, g0.z, g0.w, u0.z, u0.w);
                unpack4(w.z, g1.x, g1.y, u1.x, u1.y);
                unpack4(w.w, g1.z, g1.w, u1.z, u1.w);
                // MN-major atom (channels 64 * (cc / 4) .., inputs 8 * (r / 8) ..), line r % 8
                const int line = r & 7, j0 = (cc & 3) * 2;
                unsigned char* at = as + (cc >> 2) * 8192 + (r >> 3) * 1024 + line * 128;
                *reinterpret_cast<uint4*>(at + ((j0 ^ line) << 4)) = g0;
                *reinterpret_cast<uint4*>(at + (((j0 + 1) ^ line) << 4)) = g1;
                *reinterpret_cast<uint4*>(at + kAProj + ((j0 ^ line) << 4)) = u0;
                *reinterpret_cast<uint4*>(at + kAProj + (((j0 + 1) ^ line) << 4)) = u1;
            }
            fence_smem_async();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&bars[kAFull + a]);
                mbar_arrive(&bars[kCEmpty + c]);
            }
        }
    } else if (total > 0 && (warp == kMmaWarp || warp == kMmaWarpUp) && lane == 0) {
        // ---------------------------------------------------------------- MMA issue
        // one thread issues the gate MMAs, another the up MMAs (separate accumulators)
        const int proj = warp == kMmaWarpUp;
        int s = 0;
        bool ok = true;
        for (; ok && s < total; ++s) {
            const int c = s % kCodeSlots, a = s % kASlots;
            const int j = s >> 1, h = s & 1, buf = j & 1;
            if (h == 0 && j >= 2 &&
                !mbar_wait(&bars[kDEmpty + buf], ((j >> 1) - 1) & 1, spin, status)) {
                ok = false;
                break;
            }
            if (!mbar_wait(&bars[kCFull + c], (s / kCodeSlots) & 1, spin, status) ||
                !mbar_wait(&bars[kAFull + a], (s / kASlots) & 1, spin, status)) {
                ok = false;
                break;
            }
            fence_smem_async();   // the A operands are ordinary shared-memory writes
            tc_fence_after();
            const uint32_t as = a0 + a * kASlot, qs = code0 + c * kCodeSlot + kCodeBytes;
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                const uint64_t bq = smem_desc(qs + ks * 32, 16, 1024, kLayoutSw128);
                mma_f16(tmem + buf * 32 + proj * 16,
                        smem_desc(as + proj * kAProj + ks * 2048, 8192, 1024, kLayoutSw128), bq,
                        kIdesc, (h | ks) != 0);
            }
            mma_commit(&bars[kAEmpty + a]);
            mma_commit(&bars[kCEmpty + c]);
            if (h == 1) mma_commit(&bars[kDFull + buf]);
        }
        if (proj == 0) misc[2] = s;
        mma_commit(&bars[kDone + proj]);
        mbar_wait(&bars[kDone + proj], 0, spin, status);
    } else if (total > 0 && warp > kMmaWarpUp) {
        // ---------------------------------------------------------------- scale and combine
        const int q = warp & 3;
        const int t0 = ((warp - kMmaWarpUp - 1) >> 2) * 8;   // this warp's 8 tokens
        const int m = q * 32 + lane;
        const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
        bool ok = true;
        for (int mt = 0; ok && mt < nmt; ++mt) {
            const int w0 = c_lo + mt * kWin, w1 = min(c_hi, w0 + kWin);
            const int c = (w0 & ~15) + m;
            const bool valid = c >= w0 && c < w1;
            DF tg[8], tu[8];
#pragma unroll
            for (int b = 0; b < 8; ++b) tg[b] = tu[b] = DF{0.f, 0.f};
            uint32_t swn = valid ? __ldg(scales + c) : 0u;
            for (int g = 0; g < G; ++g) {
                const int j = mt * G + g, buf = j & 1;
                const uint32_t sw = swn;
                if (valid && g + 1 < G) swn = __ldg(scales + static_cast<size_t>(g + 1) * F + c);
                if (!mbar_wait(&bars[kDFull + buf], (j >> 1) & 1, spin, status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                float vg[8], vu[8];
                tmem_ld8x2(tmem + lane_off + buf * 32 + t0, tmem + lane_off + buf * 32 + 16 + t0,
                           vg, vu);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars[kDEmpty + buf]);
                const float swg = __half2float(__ushort_as_half(static_cast<unsigned short>(sw & 0xFFFFu)));
                const float swu = __half2float(__ushort_as_half(static_cast<unsigned short>(sw >> 16)));
#pragma unroll
                for (int b = 0; b < 8; ++b) {
                    // the accumulators hold exact integers
                    const float sxb = s_sx[(t0 + b) * G + g];
                    tg[b] = df_add(tg[b], df_scaled(sxb, swg, vg[b]));
                    tu[b] = df_add(tu[b], df_scaled(sxb, swu, vu[b]));
                    if (valid && t0 + b < B) {
                        const size_t o = (static_cast<size_t>(t0 + b) * G + g) * F + c;
                        if (dbg_gate) dbg_gate[o] = __float2int_rn(vg[b]);
                        if (dbg_up) dbg_up[o] = __float2int_rn(vu[b]);
                    }
                }
            }
            if (ok && valid) {
#pragma unroll
                for (int b = 0; b < 8; ++b) {
                    if (t0 + b < B) {
                        const float sg = fabsf(silu_f(tg[b].hi + tg[b].lo) * (tu[b].hi + tu[b].lo));
                        sigma[static_cast<size_t>(t0 + b) * F + c] = sg;
                        atomicAdd(&ghist[(t0 + b) * 2048 + (__float_as_uint(sg) >> 20)], 1);
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
        // copies that were issued but not consumed (only after a timeout) land before the end
        const uint32_t issued = misc[1], consumed = misc[2];
        for (uint32_t s = consumed; s < issued; ++s)
            mbar_wait(&bars[kCFull + s % kCodeSlots], (s / kCodeSlots) & 1, spin, status);
    }
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_free(tmem, kTmemCols);
    }
}

}  // namespace

bool stage1_tc_supported(int d, int F, int B, int sms) {
    (void)d;
    return B >= 2 && B <= kTokens && F >= 16 && sms > 0;
}

int launch_stage1_tc(const uint8_t* packed, const PackedLayout& L, int d, int F, int B,
                     uint8_t* ws, const WsLayout& W, float* sigma, int32_t* dbg_gate,
                     int32_t* dbg_up, int sms, cudaStream_t s) {
    if (!stage1_tc_supported(d, F, B, sms) || W.BPtc == 0) return PROX_ERR_UNSUPPORTED;
    const int G = d / 128;
    const uint16_t* qxh = reinterpret_cast<const uint16_t*>(ws + W.qxh);
    CUtensorMap tm_codes, tm_qx;
    if (encode_map_2d(&tm_codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, L.codes(packed), F, d, F, 128, 64,
                      CU_TENSOR_MAP_SWIZZLE_NONE) != PROX_OK)
        return PROX_ERR_CUDA;
    if (encode_map_2d(&tm_qx, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, qxh, d, kTokens,
                      static_cast<uint64_t>(2) * d, 64, kTokens, CU_TENSOR_MAP_SWIZZLE_128B) != PROX_OK)
        return PROX_ERR_CUDA;
    const size_t smem = s1_smem_layout(G).total;
    if (ensure_dynamic_smem(reinterpret_cast<const void*>(stage1_tc_kernel), smem) != PROX_OK)
        return PROX_ERR_CUDA;
    return launch_pdl(stage1_tc_kernel, dim3(sms), dim3(kThreads), smem, s, tm_codes, tm_qx,
                      L.scales(packed),
                      reinterpret_cast<const float*>(ws + W.sx), d, F, B, sigma,
                      reinterpret_cast<int*>(ws + W.ghist), dbg_gate, dbg_up, kDefaultSpinCycles,
                      &reinterpret_cast<Control*>(ws + W.control)->status);
}

}  // namespace prox

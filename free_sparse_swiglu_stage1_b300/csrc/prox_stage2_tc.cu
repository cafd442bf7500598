// Stage 2 of a batch of tokens on the fifth-generation tensor cores (tcgen05, sm_103a).
//
// Method: Stage 2 of the Prox FFN ("Prox: two-stage sparse SwiGLU FFN" pages, Stage 2: the
// selected channels' gate and up rows are multiplied exactly, SiLU(g) * u is formed, and only
// the matching rows of W_down^T contribute to y). With a batch, the selected set is the union
// U of the tokens' masks and each token keeps only its own channels:
//     y_b = sum over j in U with j in M_b of SiLU(x_b . Wg[j]) (x_b . Wu[j]) W_down^T[j].
// For a batch of 2 to 16 tokens the two gathered projections are dense contractions over
// the batch, so they run as tcgen05 MMAs (bf16 operands, fp32 accumulation in tensor memory).
//
// Precision: x and h = SiLU(g) u are fp32 on the CUDA-core path. Here each is split into a
// bf16 pair hi + lo (hi = bf16(v), lo = bf16(v - hi)), which represents v to about 2^-17 of
// its size; the pair occupies two columns of the MMA's N dimension (N = 2 * BP for BP padded
// tokens) and the two halves of the accumulator are added in fp32 afterwards. The weights are
// bf16 already. Products are exact in fp32 and accumulate in fp32.
//
// Work split: one CTA per SM owns the selected channels (nonzero words of the batch's channel
// bitmap) in a contiguous range of about F / P channels (at most kTcListMax). Eight warps
// copy, the next warp issues the MMAs, the last four read the accumulators.
//   Copies, two modes chosen per block from the union's density in its window:
//     tiles (density above 3/4): the whole window of consecutive channels is copied with TMA
//       2-D tiles of BH rows x 128 bytes, which land in the 128-byte-swizzled canonical layouts
//       directly; unselected channels get h = 0.
//     gather: the selected rows are brought in by 16-byte cp.async copies from 256 threads
//       (eight per 128-byte row piece, so each warp copy covers four whole pieces), written
//       straight to their place in the same layouts; each thread's copies complete on the
//       stage's mbarrier (cp.async.mbarrier.arrive.noinc).
//     Measured on this part: TMA tile::gather4 copies of four 128-byte row pieces stream at
//     about 1.9 TB/s and the cp.async gather at up to about 4.9 TB/s; whole tiles stream
//     like any TMA operand load.
//   Phase A, per M-tile of 128 of the slice's channels: D_gate, D_up [128 x N] accumulate over
//     d in stages of 64 inputs. The A operand is 128 gathered channel rows x 128 bytes in the
//     K-major layout; the B operand is the [N x 64] slice of the split activations (one TMA
//     tile copy).
//   Epilogue A: a thread owns one channel (one TMEM lane), forms h for every token (zero where
//     the token did not select the channel) and writes the hi/lo pair into the B operand of
//     phase B (K-major, no swizzle, resident in shared memory for the whole slice).
//   Phase B, per tile of 128 outputs: D_y [128 x N] = W_down^T[slice, tile]^T . h, with the
//     W_down^T rows copied the same way into the MN-major layout (outputs contiguous; the two
//     64-output halves 16 KB apart, groups of 8 channels 1 KB apart), K = the slice's
//     channels in steps of 16.
//   Epilogue B: y_b = D_y[:, b] + D_y[:, BP + b] is stored as the block's partial output
//     ypart[block][b][tile]; a fixed-order reduction over blocks follows (bit-reproducible).
// Every wait is bounded; a wait that runs out records PROX_ERR_TIMEOUT and the roles leave
// their loops; copies still in flight are drained (bounded) and tensor memory is freed.
#include "prox_tc.cuh"

namespace prox {

namespace {

constexpr int kTcProducers = 256;           // warps 0..7 copy
constexpr int kTcMmaWarp = kTcProducers / 32;   // then one MMA warp, then four epilogue warps
constexpr int kTcThreads = kTcProducers + 32 + 128;
constexpr int kTcSlots = 5;                 // ring of stage buffers
constexpr uint32_t kTcSlotBytes = 36 * 1024;
constexpr uint32_t kTcUpOff = 16 * 1024;    // phase-A slot: gate rows | up rows | activations
constexpr uint32_t kTcXOff = 32 * 1024;
constexpr uint32_t kTcTmemCols = 256;       // A accumulators 2 x 64 columns, D_y 2 x 32
constexpr uint32_t kTcHSbo = kTcListMax * 16;   // h operand: bytes between 8-row groups

__device__ __forceinline__ uint16_t bf16_bits(float v) {
    return __bfloat16_as_ushort(__float2bfloat16_rn(v));
}

// ------------------------------------------------------------------ the kernel
struct TcSmem {
    uint32_t slots, hop, ch, bits, bars, misc, total;
};
__host__ __device__ inline TcSmem tc_smem_layout(int BP) {
    TcSmem L;
    uint32_t o = 0;
    L.slots = o;
    o += kTcSlots * kTcSlotBytes;
    L.hop = o;
    o += static_cast<uint32_t>(2 * BP / 8) * kTcHSbo;
    L.ch = o;
    o += kTcListMax * 4;
    L.bits = o;
    o += kTcListMax * 4;
    L.bars = o;
    o += (2 * kTcSlots + 9) * 8;
    L.misc = o;
    o += 64;
    L.total = o + 1024;   // room to align the base to 1024 bytes
    return L;
}

// Barrier indices inside the barrier array.
constexpr int kBarFull = 0, kBarEmpty = kTcSlots, kBarAFull = 2 * kTcSlots,
              kBarAEmpty = kBarAFull + 2, kBarBFull = kBarAEmpty + 2, kBarBEmpty = kBarBFull + 2,
              kBarH = kBarBEmpty + 2, kBarDone = kBarH + 1;

template <int BP>
__global__ void __launch_bounds__(kTcThreads, 1)
stage2_tc_kernel(const uint16_t* __restrict__ rows_g, const __grid_constant__ CUtensorMap tm_rows,
                 const __grid_constant__ CUtensorMap tm_x, int BH, int d, int F, int nb,
                 const uint32_t* __restrict__ ubits, float* __restrict__ ypart, long long spin,
                 int* status) {
    constexpr int N = 2 * BP;
    constexpr uint32_t kIdescA = mma_idesc(128, N, 0, 0, kFmtBf16);
    constexpr uint32_t kIdescB = mma_idesc(128, N, 1, 0, kFmtBf16);
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const TcSmem SL = tc_smem_layout(BP);
    const uint32_t raw = smem_addr(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    unsigned char* sbase = smem_raw + (base - raw);
    int32_t* s_ch = reinterpret_cast<int32_t*>(sbase + SL.ch);
    uint32_t* s_bits = reinterpret_cast<uint32_t*>(sbase + SL.bits);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sbase + SL.bars);
    // misc: [0] tensor-memory address, [1] stages issued, [2] stages consumed, [3] channels
    uint32_t* misc = reinterpret_cast<uint32_t*>(sbase + SL.misc);
    const uint32_t slot0 = base + SL.slots, hop = base + SL.hop;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int i = 0; i < kTcSlots; ++i) {
            mbar_init(&bars[kBarFull + i], kTcProducers + 1);
            mbar_init(&bars[kBarEmpty + i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars[kBarAFull + i], 1);
            mbar_init(&bars[kBarAEmpty + i], 4);
            mbar_init(&bars[kBarBFull + i], 1);
            mbar_init(&bars[kBarBEmpty + i], 4);
        }
        mbar_init(&bars[kBarH], 4);
        mbar_init(&bars[kBarDone], 1);
        mbar_init_fence();
        misc[1] = 0;
        misc[2] = 0;
        asm volatile("prefetch.tensormap [%0];" ::"l"(&tm_x) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(&tm_rows) : "memory");
    }
    // rows a tile copy does not cover must read as zeros (their h is zero too)
    for (uint32_t i = tid; i < kTcSlots * kTcSlotBytes / 16; i += kTcThreads)
        reinterpret_cast<int4*>(sbase + SL.slots)[i] = make_int4(0, 0, 0, 0);
    fence_smem_async();
    if (warp == kTcMmaWarp) {
        tmem_alloc(&misc[0], kTcTmemCols);
    }

    grid_dep_wait();
    grid_dep_launch();

    // this block's slice of the union: the selected channels among [c_lo, c_hi)
    const int P = gridDim.x;
    const int c_lo = static_cast<int>(static_cast<long long>(F) * blockIdx.x / P);
    const int c_hi = static_cast<int>(static_cast<long long>(F) * (blockIdx.x + 1) / P);
    const uint32_t all_bits = nb >= 32 ? 0xFFFFFFFFu : ((1u << nb) - 1u);
    if (warp == 0) {
        int n = 0;
        for (int c = c_lo; c < c_hi; c += 32) {
            const int ch = c + lane;
            uint32_t bt = 0u;
            if (ch < c_hi) bt = ubits ? (ubits[ch] & all_bits) : all_bits;
            const uint32_t m = __ballot_sync(0xffffffffu, bt != 0u);
            const int pos = n + __popc(m & ((1u << lane) - 1u));
            if (bt != 0u && pos < kTcListMax) {
                s_ch[pos] = ch;
                s_bits[pos] = bt;
            }
            n += __popc(m);
        }
        if (lane == 0) misc[3] = static_cast<uint32_t>(n);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    int cb = static_cast<int>(misc[3]);
    if (cb > kTcListMax) {
        if (tid == 0) set_status(status, PROX_ERR_BOUNDS);
        cb = 0;
    }
    // Copy mode: a window whose union density is above 3/4 is copied whole with TMA tiles of
    // BH consecutive rows (the unselected channels get h = 0); otherwise the selected rows
    // are gathered by the cp.async threads. M-tile / K-chunk i holds rows_of(i) rows.
    const int R = c_hi - c_lo;
    const bool tiles = BH > 0 && cb * 4 > R * 3;
    const int nmt = tiles ? (R + BH - 1) / BH : (cb + 127) >> 7;
    auto rows_of = [&](int i) { return tiles ? BH : min(128, cb - i * 128); };
    if (tiles) {
        // per-row-slot token bits of the window: slot i * 128 + m is channel c_lo + i * BH + m
        __syncthreads();
        for (int j = tid; j < nmt * 128; j += kTcThreads) {
            const int i = j >> 7, m = j & 127, c = c_lo + i * BH + m;
            uint32_t bt = 0u;
            if (m < BH && c < c_hi) bt = ubits ? (ubits[c] & all_bits) : all_bits;
            s_bits[j] = bt;
        }
    } else if (cb > 0) {
        // padding rows repeat the last channel (finite data; their h is zero)
        for (int i = cb + tid; i < ((cb + 15) & ~15); i += kTcThreads) {
            s_ch[i] = s_ch[cb - 1];
            s_bits[i] = 0u;
        }
    }
    __syncthreads();
    const uint32_t tmem = misc[0];
    const int nka = d >> 6;                // phase-A stages per M-tile
    const int ntile = d >> 7;              // phase-B output tiles

    if (cb > 0 && tid < kTcProducers) {
        // ---------------------------------------------------------------- copies
        // gather mode: thread p copies 16-byte chunk (p % 8) of row pieces p / 8,
        // p / 8 + kTcProducers / 8, ...; tile mode: thread 0 issues the TMA tile copies.
        // Every producer thread arrives once per stage.
        const size_t pitch = static_cast<size_t>(3) * d;   // elements per packed channel run
        const int chunk = tid & 7;
        uint32_t it = 0;
        bool ok = true;
        for (int mt = 0; ok && mt < nmt; ++mt) {
            const int rows = rows_of(mt);
            for (int kc = 0; kc < nka; ++kc, ++it) {
                const int slot = it % kTcSlots;
                if (it >= kTcSlots &&
                    !mbar_wait(&bars[kBarEmpty + slot], ((it / kTcSlots) - 1) & 1, spin, status)) {
                    ok = false;
                    break;
                }
                const uint32_t sb = slot0 + slot * kTcSlotBytes;
                uint64_t* fb = &bars[kBarFull + slot];
                if (tid == 0) {
                    mbar_arrive_expect_tx(fb, N * 128u + (tiles ? 256u * BH : 0u));
                    tma_tile_2d(sb + kTcXOff, &tm_x, kc * 64, 0, fb);
                    if (tiles) {
                        const int row = c_lo + mt * BH;
                        tma_tile_2d(sb, &tm_rows, kc * 64, row, fb);
                        tma_tile_2d(sb + kTcUpOff, &tm_rows, d + kc * 64, row, fb);
                    }
                }
                if (!tiles) {
                    // gate pieces (proj 0) then up pieces (proj 1) of the M-tile's rows
                    for (int i = tid >> 3; i < 2 * rows; i += kTcProducers / 8) {
                        const int proj = i >= rows, r = i - proj * rows;
                        const uint16_t* src = rows_g + s_ch[mt * 128 + r] * pitch + proj * d +
                                              kc * 64 + chunk * 8;
                        const uint32_t dst = sb + proj * kTcUpOff + (r >> 3) * 1024 +
                                             (r & 7) * 128 + ((chunk ^ (r & 7)) << 4);
                        cp_async16(dst, src);
                    }
                }
                cp_async_arrive(fb);
            }
        }
        for (int t = 0; ok && t < ntile; ++t) {
            for (int kc = 0; kc < nmt; ++kc, ++it) {
                const int rows = rows_of(kc);
                const int r16 = (rows + 15) & ~15;
                const int slot = it % kTcSlots;
                if (it >= kTcSlots &&
                    !mbar_wait(&bars[kBarEmpty + slot], ((it / kTcSlots) - 1) & 1, spin, status)) {
                    ok = false;
                    break;
                }
                const uint32_t sb = slot0 + slot * kTcSlotBytes;
                uint64_t* fb = &bars[kBarFull + slot];
                // W_down^T row pieces of 64 outputs in MN-major atoms (8 channels x 128 bytes):
                // output half h at h * 16 KB, channel group g at g * 1 KB
                if (tid == 0) {
                    mbar_arrive_expect_tx(fb, tiles ? 256u * BH : 0u);
                    if (tiles) {
                        const int row = c_lo + kc * BH;
                        tma_tile_2d(sb, &tm_rows, 2 * d + t * 128, row, fb);
                        tma_tile_2d(sb + kTcUpOff, &tm_rows, 2 * d + t * 128 + 64, row, fb);
                    }
                }
                if (!tiles) {
                    for (int i = tid >> 3; i < 2 * r16; i += kTcProducers / 8) {
                        const int half = i & 1, r = i >> 1;
                        const uint16_t* src = rows_g + s_ch[kc * 128 + r] * pitch + 2 * d +
                                              t * 128 + half * 64 + chunk * 8;
                        const uint32_t dst = sb + half * kTcUpOff + (r >> 3) * 1024 +
                                             (r & 7) * 128 + ((chunk ^ (r & 7)) << 4);
                        cp_async16(dst, src);
                    }
                }
                cp_async_arrive(fb);
            }
        }
        cp_async_wait_all();
        if (tid == 0) misc[1] = it;
    } else if (cb > 0 && warp == kTcMmaWarp && lane == 0) {
        // ---------------------------------------------------------------- MMA issue
        uint32_t it = 0;
        bool ok = true;
        for (int mt = 0; ok && mt < nmt; ++mt) {
            const int buf = mt & 1;
            if (mt >= 2 && !mbar_wait(&bars[kBarAEmpty + buf], ((mt >> 1) - 1) & 1, spin, status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t dg = tmem + buf * 64, du = dg + 32;
            for (int kc = 0; kc < nka; ++kc, ++it) {
                const int slot = it % kTcSlots;
                if (!mbar_wait(&bars[kBarFull + slot], (it / kTcSlots) & 1, spin, status)) {
                    ok = false;
                    break;
                }
                fence_smem_async();   // the copies are ordinary shared-memory writes
                tc_fence_after();
                const uint32_t sb = slot0 + slot * kTcSlotBytes;
#pragma unroll
                for (int ks = 0; ks < 4; ++ks) {
                    const uint64_t bx = smem_desc(sb + kTcXOff + ks * 32, 16, 1024, kLayoutSw128);
                    const uint32_t acc = (kc | ks) != 0;
                    mma_f16(dg, smem_desc(sb + ks * 32, 16, 1024, kLayoutSw128), bx, kIdescA, acc);
                    mma_f16(du, smem_desc(sb + kTcUpOff + ks * 32, 16, 1024, kLayoutSw128), bx,
                             kIdescA, acc);
                }
                mma_commit(&bars[kBarEmpty + slot]);
            }
            if (ok) mma_commit(&bars[kBarAFull + buf]);
        }
        if (ok && !mbar_wait(&bars[kBarH], 0, spin, status)) ok = false;
        tc_fence_after();
        for (int t = 0; ok && t < ntile; ++t) {
            const int buf = t & 1;
            if (t >= 2 && !mbar_wait(&bars[kBarBEmpty + buf], ((t >> 1) - 1) & 1, spin, status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t dy = tmem + 128 + buf * 32;
            for (int kc = 0; kc < nmt; ++kc, ++it) {
                const int r16 = (rows_of(kc) + 15) & ~15;
                const int slot = it % kTcSlots;
                if (!mbar_wait(&bars[kBarFull + slot], (it / kTcSlots) & 1, spin, status)) {
                    ok = false;
                    break;
                }
                fence_smem_async();
                tc_fence_after();
                const uint32_t sb = slot0 + slot * kTcSlotBytes;
                for (int ks = 0; ks < r16 / 16; ++ks) {
                    const uint64_t a = smem_desc(sb + ks * 2048, kTcUpOff, 1024, kLayoutSw128);
                    const uint64_t b =
                        smem_desc(hop + (kc * 16 + ks * 2) * 128, 128, kTcHSbo, kLayoutNone);
                    mma_f16(dy, a, b, kIdescB, (kc | ks) != 0);
                }
                mma_commit(&bars[kBarEmpty + slot]);
            }
            if (ok) mma_commit(&bars[kBarBFull + buf]);
        }
        misc[2] = it;
        // every MMA this thread issued has finished before tensor memory is freed
        mma_commit(&bars[kBarDone]);
        mbar_wait(&bars[kBarDone], 0, spin, status);
    } else if (cb > 0 && warp > kTcMmaWarp) {
        // ---------------------------------------------------------------- epilogue
        const int q = warp & 3;               // TMEM lane quarter this warp may read
        const int m = q * 32 + lane;          // accumulator row of this thread
        const uint32_t lane_off = static_cast<uint32_t>(q * 32) << 16;
        bool ok = true;
        for (int mt = 0; ok && mt < nmt; ++mt) {
            const int buf = mt & 1;
            if (!mbar_wait(&bars[kBarAFull + buf], (mt >> 1) & 1, spin, status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            float g[N], u[N];
#pragma unroll
            for (int c = 0; c < N; c += 16) {
                tmem_ld16(tmem + lane_off + buf * 64 + c, g + c);
                tmem_ld16(tmem + lane_off + buf * 64 + 32 + c, u + c);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[kBarAEmpty + buf]);
            const int cl = mt * 128 + m;
            if (m < ((rows_of(mt) + 15) & ~15)) {
                const uint32_t bt = s_bits[cl];
                unsigned char* hp = sbase + SL.hop + (cl >> 3) * 128 + (cl & 7) * 2;
#pragma unroll
                for (int b = 0; b < BP; ++b) {
                    const float gg = g[b] + g[BP + b];
                    const float uu = u[b] + u[BP + b];
                    const float h = ((bt >> b) & 1u) ? silu_f(gg) * uu : 0.f;
                    const float hi = __bfloat162float(__float2bfloat16_rn(h));
                    const int nh = b, nl = BP + b;
                    *reinterpret_cast<uint16_t*>(hp + (nh & 7) * 16 + (nh >> 3) * kTcHSbo) =
                        bf16_bits(hi);
                    *reinterpret_cast<uint16_t*>(hp + (nl & 7) * 16 + (nl >> 3) * kTcHSbo) =
                        bf16_bits(h - hi);
                }
            }
        }
        fence_smem_async();
        __syncwarp();
        if (ok && lane == 0) mbar_arrive(&bars[kBarH]);
        for (int t = 0; ok && t < ntile; ++t) {
            const int buf = t & 1;
            if (!mbar_wait(&bars[kBarBFull + buf], (t >> 1) & 1, spin, status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            float v[N];
#pragma unroll
            for (int c = 0; c < N; c += 16) tmem_ld16(tmem + lane_off + 128 + buf * 32 + c, v + c);
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars[kBarBEmpty + buf]);
            float* yp = ypart + static_cast<size_t>(blockIdx.x) * BP * d + t * 128 + m;
#pragma unroll
            for (int b = 0; b < BP; ++b)
                if (b < nb) yp[static_cast<size_t>(b) * d] = v[b] + v[BP + b];
        }
    }
    if (cb == 0) {
        // an empty slice contributes zeros
        for (int i = tid; i < nb * d; i += kTcThreads)
            ypart[static_cast<size_t>(blockIdx.x) * BP * d + i] = 0.f;
    }

    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
        // copies that no MMA consumed (only after a timeout) must land before the block ends
        const uint32_t issued = misc[1], consumed = misc[2];
        for (uint32_t it = consumed; it < issued; ++it)
            mbar_wait(&bars[kBarFull + it % kTcSlots], (it / kTcSlots) & 1, spin, status);
    }
    __syncthreads();
    if (warp == kTcMmaWarp) {
        tc_fence_after();
        tmem_free(tmem, kTcTmemCols);
    }
}

// x [nb][d] fp32 -> xhl [2 BP][d] bf16: rows 0..BP-1 hold bf16(x), rows BP..2BP-1 the
// remainder bf16(x - bf16(x)); rows of tokens nb..BP-1 are zero.
__global__ void __launch_bounds__(256)
split_x_kernel(const float* __restrict__ x, int nb, int d, int BP, uint16_t* __restrict__ xhl) {
    grid_dep_wait();
    grid_dep_launch();
    const int total = BP * d;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
        const float v = i < nb * d ? x[i] : 0.f;
        const float hi = __bfloat162float(__float2bfloat16_rn(v));
        xhl[i] = bf16_bits(hi);
        xhl[total + i] = bf16_bits(v - hi);
    }
}

// ------------------------------------------------------------------ host side
template <int BP>
int launch_tc_t(const uint16_t* rows, const CUtensorMap& tm_rows, const CUtensorMap& tm_x, int BH,
                int d, int F, int nb, const uint32_t* bits, float* ypart, int P, int* status,
                cudaStream_t s) {
    const size_t smem = tc_smem_layout(BP).total;
    auto fn = stage2_tc_kernel<BP>;
    if (ensure_dynamic_smem(reinterpret_cast<const void*>(fn), smem) != PROX_OK) return PROX_ERR_CUDA;
    return launch_pdl(fn, dim3(P), dim3(kTcThreads), smem, s, rows, tm_rows, tm_x, BH, d, F, nb,
                      bits, ypart, kDefaultSpinCycles, status);
}

}  // namespace

bool stage2_tc_supported(int d, int F, int nb, int sms) {
    return nb >= 1 && nb <= kTcMaxTokens && d % 128 == 0 &&
           static_cast<long long>(tc_blocks(F, sms)) * kTcListMax >= F;
}

int launch_stage2_tc(const uint8_t* packed, const PackedLayout& L, int d, int F, const float* x,
                     int nb, const uint32_t* bits, float* y, uint8_t* ws, const WsLayout& W,
                     int sms, cudaStream_t s) {
    if (!stage2_tc_supported(d, F, nb, sms) || W.BPtc < nb) return PROX_ERR_UNSUPPORTED;
    const int BP = W.BPtc;
    const int P = tc_blocks(F, sms);
    uint16_t* xhl = reinterpret_cast<uint16_t*>(ws + W.xhl);
    float* ypart = reinterpret_cast<float*>(ws + W.ypart);
    int* status = &reinterpret_cast<Control*>(ws + W.control)->status;
    const uint16_t* rows = reinterpret_cast<const uint16_t*>(L.rows(packed));
    // tile copies: a block's window of at most ceil(F / P) channels in nmt tiles of BH rows
    const int rmax = (F + P - 1) / P;
    const int nmt = (rmax + 127) / 128;
    const int BH = (rmax + nmt - 1) / nmt;
    CUtensorMap tm_rows, tm_x;
    if (encode_map_2d(&tm_rows, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rows, static_cast<uint64_t>(3) * d,
                      F, static_cast<uint64_t>(6) * d, 64, BH, CU_TENSOR_MAP_SWIZZLE_128B) != PROX_OK)
        return PROX_ERR_CUDA;
    if (encode_map_2d(&tm_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, xhl, d, 2 * BP,
                      static_cast<uint64_t>(2) * d, 64, 2 * BP, CU_TENSOR_MAP_SWIZZLE_128B) != PROX_OK)
        return PROX_ERR_CUDA;
    const int total = BP * d;
    int rc = launch_pdl(split_x_kernel, dim3((total + 1023) / 1024), dim3(256), 0, s, x, nb, d, BP,
                        xhl);
    if (rc != PROX_OK) return rc;
    rc = BP == 16 ? launch_tc_t<16>(rows, tm_rows, tm_x, BH, d, F, nb, bits, ypart, P, status, s)
                  : launch_tc_t<8>(rows, tm_rows, tm_x, BH, d, F, nb, bits, ypart, P, status, s);
    if (rc != PROX_OK) return rc;
    return launch_reduce_partials(ypart, P, BP, d, nb, y, s);
}

}  // namespace prox

// The whole single-token Prox path in one persistent launch (technical summary,
// "Methodology: The Prox Framework": Stage 1 "Lightweight Proxy Construction", then Stage 2
// "Exact Sparse Computation"; "Hardware Implementation": the fused split-N Stage-1 kernel and
// the fused output-sparse Stage-2 kernel).
//
// fused_token_kernel: one block of 512 threads per SM, all blocks resident at once (launched
// cooperatively), so the steps that exchange data between blocks meet at grid-wide barriers
// inside the kernel instead of at kernel boundaries. Block p:
//  1. Input selection, redundantly in every block: a radix select of the k_in largest |x_i|
//     (ties to the lower index) over x in shared memory; after its first pass the rows that may
//     be kept are hinted into L2 (each block its share); per group of 128 inputs the int8
//     activation codes qx = clamp(rint(x / sx), -127, 127), sx = max|kept x| / 127 (binary32)
//     and the ascending list of kept inputs, padded to a multiple of 4 with code-0 copies.
//  2. Stage-1 proxy GEMV for the block's tile of 16-channel chunks (whole 128-channel units,
//     all groups): each lane owns one chunk (16 channels, one 16-byte load per kept input row),
//     the lanes of a warp that share a chunk split the group's row quads, the four loaded words
//     of a 4-channel column are byte-transposed so one dp4a per channel and projection
//     multiplies a channel's four row codes by the rows' activation codes (gate codes as bytes
//     q + 8, up codes as 16 (q + 8), one more dp4a for 8 sum(qx)), so the group sums
//     A = sum q qx are exact int32, added across warps with shared-memory integer atomics.
//  3. Salience: sum over groups of sx sw A as a double-float (about 44 bits; the groups are
//     split into a fixed number of parts added in a fixed order; the tile's scales come from a
//     shared-memory copy made at the start), sigma = |SiLU(g~) u~| in fp32, and the tile's
//     counts of sigma's bits 30..20 added to the layer's histogram.
//  -- barrier 1 -- (between arriving and waiting, the rows of the tile's most salient
//     channels are hinted into L2 for Stage 2)
//  4. Top-k, redundantly in every block: the layer's salience and histogram come in by bulk
//     copy; channels in bins above the bin b1 of the k-th largest key are taken, the
//     candidates of bin b1 are listed in channel order and ranked among themselves (equal
//     values to the lower channel), and every taken channel's place in the ascending mask is
//     counted; the block keeps its balanced slice [k p / P, k (p + 1) / P) (and writes that
//     slice of the mask out when asked).
//  5. Stage 2 over the slice: each selected channel's gate row, up row and down column are one
//     contiguous run, copied by one cp.async.bulk into a ring of shared-memory stages; NG
//     groups of warps consume alternate channels (gate/up dot products with fp32 x in
//     registers, a reduce-scatter across each warp and a group barrier, s = SiLU(g) u,
//     y += s W_down[:, j]). The block's partial output goes to global memory.
//  -- barrier 2 --
//  6. Block p adds the partial outputs of its columns over all blocks in block order, so y
//     is bit-reproducible on a given device.
// Other modes run a subset: the mask alone, the Stage-1 intermediates alone (test hook), or
// Stage 2 over every channel (dense) or over a given mask. Every wait (mbarrier phases, grid
// barriers) is bounded: one that runs out records PROX_ERR_TIMEOUT in the status word and
// the block carries on, so the launch always ends.
#include "prox_fused_impl.cuh"

namespace prox {

namespace fused_detail {

FusedFn fused_fn_bf16(const FusedShape& s) {
#define PROX_FUSED(run, cw, cpt) \
    if (s.RUN == run && s.CW == cw && s.CPTMAX == cpt) return fused_token_kernel<run, cw, cpt, false>;
    PROX_FUSED(4, 4, 2)
    PROX_FUSED(4, 8, 2)
    PROX_FUSED(4, 16, 2)
    PROX_FUSED(8, 4, 4)
    PROX_FUSED(8, 8, 4)
    PROX_FUSED(8, 16, 4)
    PROX_FUSED(16, 4, 4)
    PROX_FUSED(16, 8, 4)
    PROX_FUSED(16, 16, 4)
#undef PROX_FUSED
    return nullptr;
}

FusedFn fused_fn(const FusedShape& s, bool fp8) { return fp8 ? fused_fn_fp8(s) : fused_fn_bf16(s); }

}  // namespace fused_detail

using namespace fused_detail;

bool fused_supported(int d, int F, int sms) {
    FusedShape s, s8;
    if (!fused_shape(d, F, sms, s, static_cast<size_t>(6) * d) || !fused_fn(s, false) ||
        !fused_shape(d, F, sms, s8, static_cast<size_t>(3) * d + 16))
        return false;
    static int coop = -1;
    if (coop < 0) {
        int dev = 0, v = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&v, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess)
            return false;
        coop = v;
    }
    return coop != 0;
}

int launch_fused(const uint8_t* packed, const PackedLayout& L, int d, int F, const FusedCall& c,
                 uint8_t* ws, const WsLayout& W, int sms, cudaStream_t s) {
    FusedShape sh;
    if (!fused_shape(d, F, sms, sh, L.row_bytes)) return PROX_ERR_UNSUPPORTED;
    const FusedFn fn = fused_fn(sh, L.format == PROX_FORMAT_FP8);
    if (!fn) return PROX_ERR_UNSUPPORTED;
    if (sms > W.P) return PROX_ERR_WORKSPACE;   // the partial outputs need one row per block
    if (ensure_dynamic_smem(reinterpret_cast<const void*>(fn), sh.smem) != PROX_OK) return PROX_ERR_CUDA;
    FusedParams p{};
    p.codes = L.codes(packed);
    p.scales = L.scales(packed);
    p.rows = reinterpret_cast<const uint16_t*>(L.rows(packed));
    p.row_bytes = L.row_bytes;
    p.x = c.x;
    p.d = d;
    p.F = F;
    p.k = c.k;
    p.k_in = c.k_in;
    p.mode = c.mode;
    p.idx_in = c.idx_in;
    p.idx = c.idx;
    p.sigma = c.sigma;
    p.ypart = reinterpret_cast<float*>(ws + W.ypart);
    p.y = c.y;
    p.ctl = reinterpret_cast<FusedControl*>(ws + W.fctl);
    p.status = &reinterpret_cast<Control*>(ws + W.control)->status;
    p.spin = kDefaultSpinCycles;
    p.region_bytes = static_cast<int>(sh.region);
    p.nstage_log2 = sh.nstage_log2;
    p.NG = sh.NG;
    p.WPG = sh.WPG;
    p.CPT = sh.CPT;
    p.write_idx = c.write_idx ? 1 : 0;
    // the early hint pays while the likely-kept proxy rows fit L2 (126 MB) with room to spare
    p.prefetch_codes = static_cast<size_t>(c.k_in) * F <= (static_cast<size_t>(48) << 20) ? 1 : 0;
    p.scales_smem = sh.scales_smem ? 1 : 0;
    p.dbg_qx = c.dbg_qx;
    p.dbg_sx = c.dbg_sx;
    p.dbg_gate = c.dbg_gate;
    p.dbg_up = c.dbg_up;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(sms);
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = sh.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;   // every block resident at once
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t err = cudaLaunchKernelEx(&cfg, fn, p);
    if (err != cudaSuccess) return cuda_fail(err, "fused single-token launch");
    count_launch();
    return PROX_OK;
}

}  // namespace prox

// Internal interface between the C ABI (prox_api.cu) and the kernels: buffer layouts and
// launch functions. Not part of the public header.
#pragma once

#include "prox_common.cuh"

namespace prox {

constexpr size_t kAlign = PROX_ALIGN;
inline size_t align_up(size_t v, size_t a = kAlign) { return (v + a - 1) / a * a; }

// ------------------------------------------------------------------ packed layer layout
// One buffer holds codes, scales and rows at these offsets; a split layer keeps the proxy
// (codes and scales, proxy_bytes) in a buffer of its own and only the rows (from offset 0) in
// the packed buffer. Kernels get their operands through codes(), scales() and rows().
struct PackedLayout {
    size_t codes_off, scales_off, rows_off, row_bytes, proxy_bytes, total;
    int format;   // PROX_FORMAT_BF16: rows [F][3][d] bf16; PROX_FORMAT_FP8: [F][3 d + 16] bytes
    const uint8_t* proxy = nullptr;   // split layer: the proxy's own buffer

    const uint8_t* codes(const uint8_t* packed) const { return (proxy ? proxy : packed) + codes_off; }
    const uint32_t* scales(const uint8_t* packed) const {
        return reinterpret_cast<const uint32_t*>((proxy ? proxy : packed) + scales_off);
    }
    const uint8_t* rows(const uint8_t* packed) const { return packed + rows_off; }
};

inline PackedLayout packed_layout(int d, int F, int format = PROX_FORMAT_BF16) {
    PackedLayout L;
    L.format = format;
    L.codes_off = 0;
    L.scales_off = align_up(static_cast<size_t>(d) * F);
    L.proxy_bytes = align_up(L.scales_off + static_cast<size_t>(d / 128) * F * 4);
    L.rows_off = L.proxy_bytes;
    L.row_bytes = format == PROX_FORMAT_FP8 ? static_cast<size_t>(3) * d + 16 : static_cast<size_t>(6) * d;
    L.total = align_up(L.rows_off + static_cast<size_t>(F) * L.row_bytes);
    return L;
}

// The layout of a descriptor: `total` is what its packed buffer must hold.
inline PackedLayout packed_layout_of(const prox_packed* w) {
    PackedLayout L = packed_layout(w->d_model, w->d_ff, w->format);
    if (w->proxy) {
        L.proxy = static_cast<const uint8_t*>(w->proxy);
        L.rows_off = 0;
        L.total = align_up(static_cast<size_t>(w->d_ff) * L.row_bytes);
    }
    return L;
}

// ------------------------------------------------------------------ token tiles
// Tokens are processed in tiles whose Stage-2 activations and partial outputs live in
// registers; wider rows leave room for fewer tokens per tile.
inline int tile_tokens(int d) { return d <= 4096 ? 4 : (d <= 8192 ? 2 : 1); }
// Token width of the Stage-1 kernel for B tokens in tiles of TB: the whole batch if it fits
// one tile (1, 2 or 4), else the tile width.
inline int stage1_width(int B, int TB) {
    const int n = B < TB ? B : TB;
    return n <= 1 ? 1 : (n <= 2 ? 2 : 4);
}
inline int token_tiles(int B, int TB) { return (B + TB - 1) / TB; }

// Stage 1 work split. A warp reads one kept input row's codes for 32 * CPL channels with
// one load of CPL bytes per lane (CPL = 16 for one token, 8 for two, 4 for four: the
// per-token integer sums of a lane's channels stay in registers). A block of 8 warps owns
// one tile of 32 * CPL channels and a slice of consecutive groups of 128 inputs; the S <= 8
// slices of a tile form one thread-block cluster, which adds their partial sums through
// distributed shared memory. All blocks should be resident at once (two per SM).
constexpr int kStage1MaxSlices = 8;
struct Stage1Plan {
    int CPL, tiles, S, gps;   // channels per lane, channel tiles, group slices, groups per slice
};
inline Stage1Plan stage1_plan(int d, int F, int TB, int sms) {
    Stage1Plan pl;
    const int G = d / 128;
    pl.CPL = TB <= 1 ? 16 : (TB == 2 ? 8 : 4);
    pl.tiles = (F + 32 * pl.CPL - 1) / (32 * pl.CPL);
    int S = (2 * sms) / pl.tiles;   // tiles * S <= 2 * sms: one wave
    S = S < 1 ? 1 : (S > G ? G : S);
    if (S > kStage1MaxSlices) S = kStage1MaxSlices;
    pl.gps = (G + S - 1) / S;
    pl.S = (G + pl.gps - 1) / pl.gps;
    return pl;
}

// Stage-2 pipeline: one stage = the three rows of one channel (6 d bytes); the number of
// stages is a power of two so ring positions and phases are shifts and masks.
constexpr size_t kStage2SmemBudget = 200 * 1024;
constexpr int kStage2ListMax = 1024;   // channels one block may own (indices staged in smem)
inline int stage2_nstage_log2(int d) {
    const size_t per = static_cast<size_t>(6) * d;
    int lg = 1;
    while (lg < 4 && (per << (lg + 1)) <= kStage2SmemBudget) ++lg;
    return lg;   // 2 .. 16 stages
}
// blocks of the Stage-2 grid: one per SM, more if a block would own too many channels
inline int stage2_blocks(int F, int sms) {
    const int need = (F + kStage2ListMax - 1) / kStage2ListMax;
    return sms > need ? sms : need;
}

// Batch Stage 2 on the tensor cores: a batch of kTcMinBatch or more tokens (padded to BP = 8
// or 16 MMA columns per bf16 half) runs one tcgen05 kernel over the union of all their
// masks; a block owns at most kTcListMax channels of the union. A single token stays on the
// CUDA cores (a GEMV; its bulk-copy stream is the faster one).
constexpr int kTcMinBatch = 2;
constexpr int kTcMaxTokens = 16;
constexpr int kTcListMax = 384;
inline int tc_tokens(int B) { return B < kTcMinBatch ? 0 : (B <= 8 ? 8 : 16); }
inline int tc_blocks(int F, int sms) {
    const int need = (F + kTcListMax - 1) / kTcListMax;
    return sms > need ? sms : need;
}

// ------------------------------------------------------------------ fused single-token path
// One persistent launch of one block per SM runs the whole single-token path (input selection,
// Stage 1, top-k, Stage 2, the cross-block sum) with grid-wide barriers between the steps that
// exchange data across blocks. Block p owns a tile of at most kFusedTileMax channels in Stage 1.
constexpr int kFusedThreads = 512;
constexpr int kFusedMaxBlocks = 256;
constexpr int kFusedTileMax = 256;
struct GridBarrier {
    unsigned long long arrived;   // total block arrivals over every barrier so far (only grows)
};
// Lives in the cleared control region of a workspace: prox_workspace_init zeroes it and every
// fused launch leaves the histogram zeroed again for the next one.
struct FusedControl {
    GridBarrier bar;
    int pad[6];
    unsigned readers;   // blocks that read the histogram in a launch without a later barrier
    int pad2[3];
    int hist[2048];     // the layer's salience histogram over bits 30..20 (count per bin)
};

// ------------------------------------------------------------------ workspace layout
struct WsLayout {
    size_t control, fctl, xbuf, ybuf, grows, gqx, gcnt, gq, sx, ghist, qxh, sigma, idx, ulist,
        ubits, xhl, ypart, total;
    int TB, P, BPtc;
};

// Workspace of one call shape. Stage-1 inputs are kept per token tile and per group of 128
// inputs: grows [G][128] (the group's kept inputs, ascending, padded to a multiple of 4 with
// copies of the last), gcnt [G] (padded counts), gq [G + 1] (quad offsets: exclusive sums of
// gcnt / 4), gqx [TB][G][128] int8 codes, sx [TB][G] scales, ghist [TB][2048]; each of these
// is repeated for every tile of TB tokens. For a batch (2+ tokens), qxh [16][d] holds every
// token's activation codes as f16 (0 where dropped; rows past the batch 0) for the
// tensor-core Stage 1. ubits [F] holds the batch union's token bits
// (compacted with ulist on the CUDA-core path, one word per channel on the tensor-core path).
inline WsLayout ws_layout(int d, int F, int B, int sms) {
    WsLayout W;
    const int G = d / 128;
    W.TB = tile_tokens(d);
    W.P = stage2_blocks(F, sms);
    W.BPtc = tc_tokens(B);
    size_t o = 0;
    auto take = [&](size_t bytes) { const size_t at = o; o = align_up(o + bytes); return at; };
    W.control = take(sizeof(Control));
    W.fctl = take(sizeof(FusedControl));
    W.xbuf = take(static_cast<size_t>(B) * d * 4);
    W.ybuf = take(static_cast<size_t>(B) * d * 4);
    const size_t nt = static_cast<size_t>(token_tiles(B, W.TB));   // per-tile buffers below
    W.grows = take(nt * d * 4);
    W.gqx = take(nt * W.TB * d);
    W.gcnt = take(nt * G * 4);
    W.gq = take(nt * (G + 1) * 4);
    W.sx = take(nt * W.TB * G * 4);
    W.ghist = take(nt * W.TB * 2048 * 4);
    W.qxh = take(W.BPtc > 0 ? static_cast<size_t>(kTcMaxTokens) * d * 2 : 0);
    W.sigma = take(static_cast<size_t>(B) * F * 4);
    W.idx = take(static_cast<size_t>(B) * F * 4);
    W.ulist = take(static_cast<size_t>(F) * 4);
    W.ubits = take(static_cast<size_t>(F) * 4);
    W.xhl = take(static_cast<size_t>(2) * W.BPtc * d * 2);
    size_t part = static_cast<size_t>(W.P) * W.TB;
    if (W.BPtc > 0 && static_cast<size_t>(tc_blocks(F, sms)) * W.BPtc > part)
        part = static_cast<size_t>(tc_blocks(F, sms)) * W.BPtc;
    W.ypart = take(part * d * 4);
    W.total = o;
    return W;
}

// Bytes of the control region that prox_workspace_init clears (the control block and the
// fused path's barrier and histogram, which follow it).
inline size_t ws_control_bytes() { return align_up(sizeof(Control)) + align_up(sizeof(FusedControl)); }

// ------------------------------------------------------------------ launches
// Records a failed CUDA call (the error and what was being done) for prox_last_cuda_error;
// returns PROX_ERR_CUDA so callers can `return cuda_fail(...)`.
int cuda_fail(cudaError_t err, const char* what);
const char* last_cuda_error();
inline int cuda_ok(cudaError_t err, const char* what) {
    return err == cudaSuccess ? PROX_OK : cuda_fail(err, what);
}

// Counts one kernel launch enqueued by the library (for prox_launch_count). Every launch
// site calls it once per launch it issues, including launches recorded into a CUDA graph.
void count_launch();
uint64_t launch_count();

// Raises `fn`'s dynamic shared-memory limit on the current device to at least `bytes`. The
// limit is a per-function, per-device setting that the runtime checks against static plus
// dynamic shared memory, so every launch with dynamic shared memory goes through here; the
// largest value set so far is cached, so the runtime is called only when a launch needs more.
int ensure_dynamic_smem(const void* fn, size_t bytes);

// Launches `kernel` with programmatic dependent launch: its blocks may be scheduled while the
// previous kernel on the stream finishes, and each kernel calls grid_dep_wait() before it
// touches anything an earlier kernel writes.
template <typename... KArgs, typename... Args>
inline int launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                      cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t err = cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
    if (err != cudaSuccess) return cuda_fail(err, "kernel launch");
    count_launch();
    return PROX_OK;
}

int launch_pack(const uint16_t* w_gate, const uint16_t* w_up, const uint16_t* w_down, int d,
                int F, const PackedLayout& L, uint8_t* base, cudaStream_t s);

// Input selection + activation quantization (Stage 1 inputs) for all B tokens, one block
// per tile of W.TB tokens. Also clears the tiles' salience histograms (ws + W.ghist) that
// Stage 1 fills for the top-k, and zbits [F] (if not null) for the top-k's channel bitmap.
// dense_codes: also write every token's codes as f16 into qxh (for the tensor-core Stage 1).
int launch_input_quant(const float* x, int d, int F, int B, int k_in, uint8_t* ws,
                       const WsLayout& W, uint32_t* zbits, bool dense_codes, int8_t* dbg_qx,
                       float* dbg_sx, cudaStream_t s);

// Stage-1 proxy projections + salience for all B tokens (grid z: token tiles);
// sigma [B][F].
int launch_stage1(const uint8_t* packed, const PackedLayout& L, int d, int F, int B, uint8_t* ws,
                  const WsLayout& W, float* sigma, int32_t* dbg_gate, int32_t* dbg_up, int sms,
                  cudaStream_t s);

// Stage 1 of a batch (2..16 tokens) on the tensor cores: the same exact per-group integers
// from f16 MMAs over the dense activation codes qxh, the same double-float scaling; sigma [B][F]
// and the top-k histograms. Needs input_quant to have written qxh.
bool stage1_tc_supported(int d, int F, int B, int sms);
int launch_stage1_tc(const uint8_t* packed, const PackedLayout& L, int d, int F, int B,
                     uint8_t* ws, const WsLayout& W, float* sigma, int32_t* dbg_gate,
                     int32_t* dbg_up, int sms, cudaStream_t s);

// Per-token top-k of the salience [B][F] -> ascending channel indices (row stride k), one
// block per token. ghist, if not null, holds per token the 2048-bin histogram of the
// salience bits 30..20 (Stage 1 builds it). bits, if not null, receives bit b of every
// channel token b selected (atomic OR; the caller clears it first).
int launch_topk(const float* sigma, int F, int B, int k, int32_t* idx, const int* ghist,
                uint32_t* bits, int* status, cudaStream_t s);

// bits [F] |= (1 << b) for every channel of idx row b (rows of length k, B <= 32); the
// caller clears bits first.
int launch_mask_bits(const int32_t* idx, int B, int k, int F, uint32_t* bits, int* status,
                     cudaStream_t s);

// Union of nb index rows (row stride k) -> ascending list + per-entry token bits + count.
int launch_union(const int32_t* idx_tile, int nb, int k, int F, int32_t* ulist, uint32_t* ubits,
                 int* count, int* status, cudaStream_t s);

// Stage 2 over a channel list for one tile; list == nullptr means every channel.
int launch_stage2(const uint8_t* packed, const PackedLayout& L, int d, int F, const float* x_tile,
                  int nb, const int32_t* list, const uint32_t* lbits, const int* count_dev,
                  int count_host, float* y_tile, uint8_t* ws, const WsLayout& W, int sms,
                  cudaStream_t s);

// Sum of per-block partial outputs ypart [P][TB][d] over blocks, in block order, for the
// first nb rows of each block -> y [nb][d].
int launch_reduce_partials(const float* ypart, int P, int TB, int d, int nb, float* y,
                           cudaStream_t s);

// Batch Stage 2 on the tensor cores over the channels whose word in bits [F] is nonzero
// (bit b: token b selected the channel; bits == nullptr: every channel for every token) for
// nb <= kTcMaxTokens tokens; needs a workspace laid out for a batch of at least kTcMinBatch
// tokens. Splits x into bf16 pairs, runs the MMA kernel, reduces.
bool stage2_tc_supported(int d, int F, int nb, int sms);
int launch_stage2_tc(const uint8_t* packed, const PackedLayout& L, int d, int F, const float* x,
                     int nb, const uint32_t* bits, float* y, uint8_t* ws, const WsLayout& W,
                     int sms, cudaStream_t s);

// Single-token Stage 2 that selects its channels itself from the salience and Stage 1's
// histogram (the top-k is folded into the Stage-2 kernel's front end).
bool stage2_select_supported(int d, int F);
// dbg_sel (nullable): every selected channel, the sure ones then the boundary winners.
int launch_stage2_select(const uint8_t* packed, const PackedLayout& L, int d, int F,
                         const float* x, const float* sigma, const int* ghist, int k, float* y,
                         int32_t* dbg_sel, uint8_t* ws, const WsLayout& W, int sms,
                         cudaStream_t s);

// The fused single-token path. mode is a set of FusedMode bits:
//   kFusedStage1  input selection, Stage-1 GEMV, salience (into sigma)
//   kFusedSelect  top-k of the salience into idx (ascending)
//   kFusedStage2  Stage 2 + cross-block sum into y, over the mask from kFusedSelect, or over
//                 every channel (kFusedDense), or over idx_in (kFusedGiven)
enum FusedMode : int {
    kFusedStage1 = 1,
    kFusedSelect = 2,
    kFusedStage2 = 4,
    kFusedDense = 8,
    kFusedGiven = 16,
};
struct FusedCall {
    const float* x = nullptr;
    int k = 0, k_in = 0, mode = 0;
    const int32_t* idx_in = nullptr;   // kFusedGiven: [k] ascending
    int32_t* idx = nullptr;            // kFusedSelect: [k] ascending mask
    bool write_idx = false;            // store the mask into idx (else only used in-kernel)
    float* sigma = nullptr;            // kFusedStage1: [F] written
    float* y = nullptr;                // kFusedStage2: [d] written
    int8_t* dbg_qx = nullptr;          // Stage-1 intermediates (test hook), each nullable
    float* dbg_sx = nullptr;
    int32_t* dbg_gate = nullptr;
    int32_t* dbg_up = nullptr;
};
bool fused_supported(int d, int F, int sms);
int launch_fused(const uint8_t* packed, const PackedLayout& L, int d, int F, const FusedCall& c,
                 uint8_t* ws, const WsLayout& W, int sms, cudaStream_t s);

int launch_rmsnorm(const float* y, float* x_out, int batch, int d, float eps, cudaStream_t s);

int launch_iota(int32_t* out, int n, int rows, cudaStream_t s);

int launch_wait_probe(int* status, long long spin_cycles, cudaStream_t s);

}  // namespace prox

// The C ABI declared in include/prox.h: argument validation, buffer carving and the order
// of launches. Every step of the computation runs in the kernels; this file only decides
// what to launch, on which stream, with which pointers.
#include <algorithm>
#include <cmath>
#include <cstdio>
#include <mutex>

#include "prox_kernels.cuh"

using namespace prox;

namespace {

constexpr int kMaxDModel = 16384;
constexpr int kMaxDff = 53248;   // the top-k block keeps one salience row in shared memory

bool shape_ok(int d, int F) {
    return d >= 128 && d <= kMaxDModel && d % 128 == 0 && F >= 32 && F <= kMaxDff && F % 32 == 0;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool sparsity_ok(double s) { return s >= 0.0 && s < 1.0; }

int k_rule(double s, int n) {
    const double v = std::floor((1.0 - s) * static_cast<double>(n) + 0.5);
    long long k = static_cast<long long>(v);
    if (k < 1) k = 1;
    if (k > n) k = n;
    return static_cast<int>(k);
}

int device_sms() {
    static std::mutex mu;
    static int cache[128] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return -1;
    std::lock_guard<std::mutex> lock(mu);
    if (cache[dev] == 0) {
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
        cache[dev] = sms;
    }
    return cache[dev];
}

// Checks a packed descriptor. Returns PROX_OK or an error code.
int check_packed(const prox_packed* w) {
    if (!w || !w->base) return PROX_ERR_INVALID_ARG;
    if (w->group != PROX_GROUP || !shape_ok(w->d_model, w->d_ff)) return PROX_ERR_INVALID_ARG;
    if (w->format != PROX_FORMAT_BF16 && w->format != PROX_FORMAT_FP8) return PROX_ERR_INVALID_ARG;
    if (!aligned(w->base, kAlign)) return PROX_ERR_WORKSPACE;
    if (w->proxy) {
        if (!aligned(w->proxy, kAlign)) return PROX_ERR_WORKSPACE;
        cudaPointerAttributes a{};
        if (cudaPointerGetAttributes(&a, w->proxy) != cudaSuccess || a.type != cudaMemoryTypeDevice) {
            cudaGetLastError();
            return PROX_ERR_INVALID_ARG;   // a split layer's proxy must be in device memory
        }
    }
    if (w->bytes < packed_layout_of(w).total) return PROX_ERR_WORKSPACE;
    return PROX_OK;
}

// Stage 2 over FP8 rows runs in the single-token fused kernel only (a batch token by token).
bool fp8_stage2_ok(const prox_packed* w, int sms) {
    return w->format != PROX_FORMAT_FP8 || fused_supported(w->d_model, w->d_ff, sms);
}
bool is_fp8(const prox_packed* w) { return w->format == PROX_FORMAT_FP8; }

int check_ws(void* ws, size_t ws_bytes, int d, int F, int B, int sms, WsLayout& W) {
    if (!ws) return PROX_ERR_INVALID_ARG;
    if (!aligned(ws, kAlign)) return PROX_ERR_WORKSPACE;
    W = ws_layout(d, F, B, sms);
    if (ws_bytes < W.total) return PROX_ERR_WORKSPACE;
    return PROX_OK;
}

#define PROX_TRY(expr)                 \
    do {                               \
        const int rc_ = (expr);        \
        if (rc_ != PROX_OK) return rc_; \
    } while (0)

// Stage 2 for one tile of tokens: a single token uses its mask directly, several tokens
// share the union of their masks (one read of each selected row per tile).
int run_stage2_tile(const prox_packed* w, const PackedLayout& L, const float* xt, int nb,
                    const int32_t* idx_tile, int k, bool dense, float* yt, uint8_t* ws,
                    const WsLayout& W, int sms, cudaStream_t s) {
    const int d = w->d_model, F = w->d_ff;
    const uint8_t* packed = static_cast<const uint8_t*>(w->base);
    if (dense)
        return launch_stage2(packed, L, d, F, xt, nb, nullptr, nullptr, nullptr, F, yt, ws, W,
                             sms, s);
    if (nb == 1)
        return launch_stage2(packed, L, d, F, xt, nb, idx_tile, nullptr, nullptr, k, yt, ws, W,
                             sms, s);
    Control* ctrl = reinterpret_cast<Control*>(ws + W.control);
    int32_t* ulist = reinterpret_cast<int32_t*>(ws + W.ulist);
    uint32_t* ubits = reinterpret_cast<uint32_t*>(ws + W.ubits);
    PROX_TRY(launch_union(idx_tile, nb, k, F, ulist, ubits, &ctrl->union_count, &ctrl->status, s));
    return launch_stage2(packed, L, d, F, xt, nb, ulist, ubits, &ctrl->union_count, 0, yt, ws, W,
                         sms, s);
}

// Stage 2 of a whole batch on the tensor cores: one pass over the union of every token's mask.
// bits: the batch's channel bitmap (nullptr: every channel); if idx is given instead, the
// bitmap is built from it first.
int run_stage2_tc(const prox_packed* w, const PackedLayout& L, const float* x, int B,
                  const int32_t* idx, int k, const uint32_t* bits, float* y, uint8_t* ws,
                  const WsLayout& W, int sms, cudaStream_t s) {
    const int d = w->d_model, F = w->d_ff;
    const uint8_t* packed = static_cast<const uint8_t*>(w->base);
    if (idx) {
        uint32_t* ubits = reinterpret_cast<uint32_t*>(ws + W.ubits);
        Control* ctrl = reinterpret_cast<Control*>(ws + W.control);
        PROX_TRY(cuda_ok(cudaMemsetAsync(ubits, 0, static_cast<size_t>(F) * 4, s),
                         "clearing the channel bitmap"));
        PROX_TRY(launch_mask_bits(idx, B, k, F, ubits, &ctrl->status, s));
        bits = ubits;
    }
    return launch_stage2_tc(packed, L, d, F, x, B, bits, y, ws, W, sms, s);
}

bool use_tc(const prox_packed* w, int B, const WsLayout& W, int sms) {
    return W.BPtc >= B && stage2_tc_supported(w->d_model, w->d_ff, B, sms);
}

struct Debug {
    int8_t* qx = nullptr;
    float* sx = nullptr;
    int32_t* acc_gate = nullptr;
    int32_t* acc_up = nullptr;
    float* salience = nullptr;
};

// Test hook of the single-token path whose Stage 2 selects its channels itself.
int32_t* g_fused_sel = nullptr;

// The whole path. y == nullptr stops after the mask. Stage 1 and the top-k run once for
// all B tokens (in tiles of W.TB tokens inside each kernel); Stage 2 runs per tile on the
// CUDA cores, or once for the batch on the tensor cores.
int run_path(const prox_packed* w, const float* x, int B, double sparsity, double in_sparsity,
             float* y, int32_t* idx_out, uint8_t* ws, const WsLayout& W, int sms, cudaStream_t s,
             const Debug* dbg) {
    const int d = w->d_model, F = w->d_ff;
    const PackedLayout L = packed_layout_of(w);
    const uint8_t* packed = static_cast<const uint8_t*>(w->base);
    const int k = k_rule(sparsity, F);
    const int k_in = k_rule(in_sparsity, d);
    const bool all_channels = (k == F) && !dbg;
    int32_t* idx = idx_out ? idx_out : reinterpret_cast<int32_t*>(ws + W.idx);
    float* sigma = (dbg && dbg->salience) ? dbg->salience : reinterpret_cast<float*>(ws + W.sigma);
    int* status = &reinterpret_cast<Control*>(ws + W.control)->status;
    uint32_t* ubits = reinterpret_cast<uint32_t*>(ws + W.ubits);
    const bool tc = y && !dbg && use_tc(w, B, W, sms);
    if (y && !fp8_stage2_ok(w, sms)) return PROX_ERR_UNSUPPORTED;
    if (B > 1 && ((B == 2 && !all_channels) || (y && is_fp8(w))) && !dbg && !g_fused_sel &&
        fused_supported(d, F, sms)) {
        // two tokens: two single-token launches measured faster than the batch kernels (on
        // 4096 x 14336, 106 us against 122 us; from three tokens on the batch kernels win; at
        // sparsity 0 the tensor-core dense FFN wins and the result stays that of prox_dense_ffn).
        // FP8 rows: Stage 2 exists in the single-token kernel only, so a batch goes token by token
        for (int b = 0; b < B; ++b)
            PROX_TRY(run_path(w, x + static_cast<size_t>(b) * d, 1, sparsity, in_sparsity,
                              y ? y + static_cast<size_t>(b) * d : nullptr,
                              idx_out ? idx_out + static_cast<size_t>(b) * k : nullptr, ws, W, sms, s,
                              nullptr));
        return PROX_OK;
    }
    if (B == 1 && !g_fused_sel && fused_supported(d, F, sms)) {
        // one token: the whole path in one persistent launch
        FusedCall c;
        c.x = x;
        c.k = k;
        c.k_in = k_in;
        c.sigma = sigma;
        if (all_channels) {
            if (idx_out) PROX_TRY(launch_iota(idx, F, B, s));
            if (!y) return PROX_OK;
            c.mode = kFusedStage2 | kFusedDense;
        } else if (dbg) {
            c.mode = kFusedStage1;
            c.dbg_qx = dbg->qx;
            c.dbg_sx = dbg->sx;
            c.dbg_gate = dbg->acc_gate;
            c.dbg_up = dbg->acc_up;
        } else {
            c.mode = kFusedStage1 | kFusedSelect | (y ? kFusedStage2 : 0);
            c.idx = idx;
            c.write_idx = idx_out != nullptr;
        }
        c.y = y;
        return launch_fused(packed, L, d, F, c, ws, W, sms, s);
    }
    if (all_channels) {
        // sparsity 0: every channel is kept, the ranking cannot change the result
        if (idx_out) PROX_TRY(launch_iota(idx, F, B, s));
        if (!y) return PROX_OK;
        if (tc) return run_stage2_tc(w, L, x, B, nullptr, F, nullptr, y, ws, W, sms, s);
        for (int t0 = 0; t0 < B; t0 += W.TB) {
            const int nb = B - t0 < W.TB ? B - t0 : W.TB;
            PROX_TRY(run_stage2_tile(w, L, x + static_cast<size_t>(t0) * d, nb, nullptr, F, true,
                                     y + static_cast<size_t>(t0) * d, ws, W, sms, s));
        }
        return PROX_OK;
    }
    // a batch larger than one token tile runs its proxy GEMV on the tensor cores (over the
    // dense activation codes); within one tile the CUDA-core kernel reads only the tile's
    // union of kept inputs, which measured faster
    const bool s1tc = B > W.TB && W.BPtc > 0 && stage1_tc_supported(d, F, B, sms);
    PROX_TRY(launch_input_quant(x, d, F, B, k_in, ws, W, tc ? ubits : nullptr, s1tc,
                                dbg ? dbg->qx : nullptr, dbg ? dbg->sx : nullptr, s));
    if (s1tc)
        PROX_TRY(launch_stage1_tc(packed, L, d, F, B, ws, W, sigma, dbg ? dbg->acc_gate : nullptr,
                                  dbg ? dbg->acc_up : nullptr, sms, s));
    else
        PROX_TRY(launch_stage1(packed, L, d, F, B, ws, W, sigma, dbg ? dbg->acc_gate : nullptr,
                               dbg ? dbg->acc_up : nullptr, sms, s));
    if (dbg) return PROX_OK;
    const int* ghist = reinterpret_cast<const int*>(ws + W.ghist);
    if (g_fused_sel && y && !idx_out && B == 1 && stage2_select_supported(d, F)) {
        // one token, mask not wanted: Stage 2 selects its channels itself
        return launch_stage2_select(packed, L, d, F, x, sigma, ghist, k, y, g_fused_sel, ws, W,
                                    sms, s);
    }
    PROX_TRY(launch_topk(sigma, F, B, k, idx, ghist, tc ? ubits : nullptr, status, s));
    if (!y) return PROX_OK;
    if (tc) return run_stage2_tc(w, L, x, B, nullptr, k, ubits, y, ws, W, sms, s);
    for (int t0 = 0; t0 < B; t0 += W.TB) {
        const int nb = B - t0 < W.TB ? B - t0 : W.TB;
        PROX_TRY(run_stage2_tile(w, L, x + static_cast<size_t>(t0) * d, nb,
                                 idx + static_cast<size_t>(t0) * k, k, false,
                                 y + static_cast<size_t>(t0) * d, ws, W, sms, s));
    }
    return PROX_OK;
}

// Tokens of one tile: calls above PROX_MAX_BATCH tokens run tile by tile, every tile exactly
// as a call of its own (each token keeps its own inputs and mask, so tiling changes nothing
// but the number of passes over the weights).
inline int tile_batch(int batch) { return batch < PROX_MAX_BATCH ? batch : PROX_MAX_BATCH; }

template <class Fn>
int for_token_tiles(int batch, Fn&& fn) {
    for (int t0 = 0; t0 < batch; t0 += PROX_MAX_BATCH) {
        const int nb = batch - t0 < PROX_MAX_BATCH ? batch - t0 : PROX_MAX_BATCH;
        PROX_TRY(fn(t0, nb));
    }
    return PROX_OK;
}

bool tokens_ok(int batch) { return batch >= 1 && batch <= PROX_MAX_TOKENS; }

}  // namespace

extern "C" {

size_t prox_packed_bytes(int d_model, int d_ff, int group) {
    if (group != PROX_GROUP || !shape_ok(d_model, d_ff)) return 0;
    return packed_layout(d_model, d_ff).total;
}

size_t prox_workspace_bytes(int d_model, int d_ff, int batch) {
    if (!shape_ok(d_model, d_ff) || !tokens_ok(batch)) return 0;
    const int sms = device_sms();
    if (sms <= 0) return 0;
    return ws_layout(d_model, d_ff, tile_batch(batch), sms).total;
}

int prox_workspace_init(void* ws, size_t ws_bytes, void* stream) {
    if (!ws) return PROX_ERR_INVALID_ARG;
    if (!aligned(ws, kAlign)) return PROX_ERR_WORKSPACE;
    const size_t need = ws_control_bytes();
    if (ws_bytes < align_up(sizeof(Control))) return PROX_ERR_WORKSPACE;
    const size_t n = ws_bytes < need ? ws_bytes : need;
    return cuda_ok(cudaMemsetAsync(ws, 0, n, static_cast<cudaStream_t>(stream)), "clearing the workspace");
}

int prox_cost_model_bytes(int d_model, int d_ff, prox_cost_model* out) {
    if (!out || !shape_ok(d_model, d_ff)) return PROX_ERR_INVALID_ARG;
    const double d = d_model, F = d_ff, G = d_model / 128;
    out->in_cost = F;
    out->fixed_cost = 4.0 * G * F;
    out->ch_cost = 6.0 * d;
    out->dense_cost = 6.0 * d * F;
    return PROX_OK;
}

int prox_cost_model_fit(const double* k_in, const double* k, const double* t, int n, double dense_t,
                        double min_cost, prox_cost_model* out) {
    if (!k_in || !k || !t || !out || n < 3 || !(dense_t > 0.0) || !(min_cost >= 0.0) ||
        !std::isfinite(dense_t))
        return PROX_ERR_INVALID_ARG;
    // normal equations of the fit t ~ a k_in + b + c k, unknowns (a, b, c)
    double M[3][3] = {{0, 0, 0}, {0, 0, 0}, {0, 0, 0}}, r[3] = {0, 0, 0};
    for (int i = 0; i < n; ++i) {
        if (!std::isfinite(k_in[i]) || !std::isfinite(k[i]) || !std::isfinite(t[i]) ||
            k_in[i] < 0.0 || k[i] < 0.0 || t[i] < 0.0)
            return PROX_ERR_INVALID_ARG;
        const double v[3] = {k_in[i], 1.0, k[i]};
        for (int a = 0; a < 3; ++a) {
            r[a] += v[a] * t[i];
            for (int b = 0; b < 3; ++b) M[a][b] += v[a] * v[b];
        }
    }
    // Gaussian elimination with partial pivoting
    double A[3][4];
    for (int a = 0; a < 3; ++a) {
        for (int b = 0; b < 3; ++b) A[a][b] = M[a][b];
        A[a][3] = r[a];
    }
    double scale = 0.0;
    for (int a = 0; a < 3; ++a)
        for (int b = 0; b < 3; ++b) scale = std::max(scale, std::fabs(A[a][b]));
    for (int col = 0; col < 3; ++col) {
        int best = col;
        for (int row = col + 1; row < 3; ++row)
            if (std::fabs(A[row][col]) > std::fabs(A[best][col])) best = row;
        if (!(std::fabs(A[best][col]) > 1e-12 * scale)) return PROX_ERR_INVALID_ARG;
        if (best != col) {
            for (int b = 0; b < 4; ++b) std::swap(A[col][b], A[best][b]);
        }
        for (int row = 0; row < 3; ++row) {
            if (row == col) continue;
            const double f = A[row][col] / A[col][col];
            for (int b = col; b < 4; ++b) A[row][b] -= f * A[col][b];
        }
    }
    const double a = A[0][3] / A[0][0], b = A[1][3] / A[1][1], c = A[2][3] / A[2][2];
    out->in_cost = std::max(a, min_cost);
    out->fixed_cost = std::max(b, 0.0);
    out->ch_cost = std::max(c, min_cost);
    out->dense_cost = dense_t;
    return PROX_OK;
}

int prox_choose_sparsity(const prox_cost_model* cost, int d_model, int d_ff, double target,
                         double anchor, double min_input_kept, double* input_sparsity,
                         double* sparsity, double* effective) {
    if (!cost || d_model < 1 || d_ff < 1) return PROX_ERR_INVALID_ARG;
    if (!(cost->in_cost > 0.0) || !(cost->ch_cost > 0.0) || !(cost->dense_cost > 0.0) ||
        !(cost->fixed_cost >= 0.0))
        return PROX_ERR_INVALID_ARG;
    if (!(target >= 0.0 && target < 1.0) || !sparsity_ok(anchor) ||
        !(min_input_kept > 0.0 && min_input_kept <= 1.0))
        return PROX_ERR_INVALID_ARG;
    const int d = d_model, F = d_ff;
    const double budget = (1.0 - target) * cost->dense_cost;
    long long k_in_min = static_cast<long long>(std::ceil(min_input_kept * d));
    if (k_in_min < 1) k_in_min = 1;
    if (k_in_min > d) k_in_min = d;
    const long long k_anchor = k_rule(anchor, F);
    double v = std::floor((budget - cost->fixed_cost - cost->ch_cost * static_cast<double>(k_anchor)) /
                          cost->in_cost);
    long long k_in, k;
    if (v >= d) {
        k_in = d;
        const double kk = std::floor((budget - cost->fixed_cost - cost->in_cost * static_cast<double>(d)) /
                                     cost->ch_cost);
        k = kk >= F ? F : static_cast<long long>(kk);
    } else if (v >= static_cast<double>(k_in_min)) {
        k_in = static_cast<long long>(v);
        k = k_anchor;
    } else {
        k_in = k_in_min;
        const double kk = std::floor((budget - cost->fixed_cost - cost->in_cost * static_cast<double>(k_in)) /
                                     cost->ch_cost);
        if (kk < 1.0) return PROX_ERR_UNSUPPORTED;
        k = static_cast<long long>(kk);
    }
    const double c = (cost->in_cost * static_cast<double>(k_in) + cost->fixed_cost +
                      cost->ch_cost * static_cast<double>(k)) / cost->dense_cost;
    if (input_sparsity) *input_sparsity = 1.0 - static_cast<double>(k_in) / d;
    if (sparsity) *sparsity = 1.0 - static_cast<double>(k) / F;
    if (effective) *effective = 1.0 - c;
    return PROX_OK;
}

int prox_k_for(double sparsity, int n) {
    if (!sparsity_ok(sparsity) || n < 1) return -1;
    return k_rule(sparsity, n);
}

namespace {
int pack_format(const uint16_t* w_gate, const uint16_t* w_up, const uint16_t* w_down,
                int d_model, int d_ff, int group, void* packed_dev, size_t packed_bytes,
                void* stream, prox_packed* out, int format) {
    if (!w_gate || !w_up || !w_down || !packed_dev || !out) return PROX_ERR_INVALID_ARG;
    if (group != PROX_GROUP || !shape_ok(d_model, d_ff)) return PROX_ERR_INVALID_ARG;
    if (!aligned(w_gate, 16) || !aligned(w_up, 16) || !aligned(w_down, 16)) return PROX_ERR_INVALID_ARG;
    if (!aligned(packed_dev, kAlign)) return PROX_ERR_WORKSPACE;
    const PackedLayout L = packed_layout(d_model, d_ff, format);
    if (packed_bytes < L.total) return PROX_ERR_WORKSPACE;
    PROX_TRY(launch_pack(w_gate, w_up, w_down, d_model, d_ff, L, static_cast<uint8_t*>(packed_dev),
                         static_cast<cudaStream_t>(stream)));
    out->d_model = d_model;
    out->d_ff = d_ff;
    out->group = group;
    out->format = format;
    out->base = packed_dev;
    out->bytes = packed_bytes;
    out->proxy = nullptr;
    return PROX_OK;
}
}  // namespace

int prox_pack_weights(const uint16_t* w_gate, const uint16_t* w_up, const uint16_t* w_down,
                      int d_model, int d_ff, int group, void* packed_dev, size_t packed_bytes,
                      void* stream, prox_packed* out) {
    return pack_format(w_gate, w_up, w_down, d_model, d_ff, group, packed_dev, packed_bytes, stream,
                       out, PROX_FORMAT_BF16);
}

int prox_pack_weights_fp8(const uint16_t* w_gate, const uint16_t* w_up, const uint16_t* w_down,
                          int d_model, int d_ff, int group, void* packed_dev, size_t packed_bytes,
                          void* stream, prox_packed* out) {
    return pack_format(w_gate, w_up, w_down, d_model, d_ff, group, packed_dev, packed_bytes, stream,
                       out, PROX_FORMAT_FP8);
}

size_t prox_packed_bytes_fp8(int d_model, int d_ff, int group) {
    if (group != PROX_GROUP || !shape_ok(d_model, d_ff)) return 0;
    return packed_layout(d_model, d_ff, PROX_FORMAT_FP8).total;
}

int prox_build_mask(const prox_packed* w, const float* x, int batch, double sparsity,
                    double input_sparsity, int32_t* idx_out, void* ws, size_t ws_bytes,
                    void* stream) {
    PROX_TRY(check_packed(w));
    if (!x || !idx_out || !tokens_ok(batch)) return PROX_ERR_INVALID_ARG;
    if (!sparsity_ok(sparsity) || !sparsity_ok(input_sparsity)) return PROX_ERR_INVALID_ARG;
    if (!aligned(x, 16)) return PROX_ERR_INVALID_ARG;
    const int sms = device_sms();
    if (sms <= 0) return PROX_ERR_CUDA;
    WsLayout W;
    PROX_TRY(check_ws(ws, ws_bytes, w->d_model, w->d_ff, tile_batch(batch), sms, W));
    const int d = w->d_model, F = w->d_ff, k = k_rule(sparsity, F);
    return for_token_tiles(batch, [&](int t0, int nb) {
        return run_path(w, x + static_cast<size_t>(t0) * d, nb, sparsity, input_sparsity, nullptr,
                        idx_out + static_cast<size_t>(t0) * k, static_cast<uint8_t*>(ws),
                        ws_layout(d, F, nb, sms), sms, static_cast<cudaStream_t>(stream), nullptr);
    });
}

namespace {

// Stage 2 of one tile of at most PROX_MAX_BATCH tokens over a given mask.
int sparse_ffn_tile(const prox_packed* w, const float* x, int batch, const int32_t* idx, int k,
                    float* y, void* ws, const WsLayout& W, int sms, void* stream) {
    const PackedLayout L = packed_layout_of(w);
    const int d = w->d_model;
    if (batch == 1 && fused_supported(d, w->d_ff, sms)) {
        FusedCall c;
        c.x = x;
        c.k = k;
        c.idx_in = idx;
        c.y = y;
        c.mode = kFusedStage2 | kFusedGiven;
        return launch_fused(static_cast<const uint8_t*>(w->base), L, d, w->d_ff, c,
                            static_cast<uint8_t*>(ws), W, sms, static_cast<cudaStream_t>(stream));
    }
    if (use_tc(w, batch, W, sms))
        return run_stage2_tc(w, L, x, batch, idx, k, nullptr, y, static_cast<uint8_t*>(ws), W,
                             sms, static_cast<cudaStream_t>(stream));
    for (int t0 = 0; t0 < batch; t0 += W.TB) {
        const int nb = batch - t0 < W.TB ? batch - t0 : W.TB;
        PROX_TRY(run_stage2_tile(w, L, x + static_cast<size_t>(t0) * d, nb,
                                 idx + static_cast<size_t>(t0) * k, k, false,
                                 y + static_cast<size_t>(t0) * d, static_cast<uint8_t*>(ws), W, sms,
                                 static_cast<cudaStream_t>(stream)));
    }
    return PROX_OK;
}

// Stage 2 over every channel for one tile of at most PROX_MAX_BATCH tokens.
int dense_ffn_tile(const prox_packed* w, const float* x, int batch, float* y, void* ws,
                   const WsLayout& W, int sms, void* stream) {
    const PackedLayout L = packed_layout_of(w);
    const int d = w->d_model;
    if (batch == 1 && fused_supported(d, w->d_ff, sms)) {
        FusedCall c;
        c.x = x;
        c.k = w->d_ff;
        c.y = y;
        c.mode = kFusedStage2 | kFusedDense;
        return launch_fused(static_cast<const uint8_t*>(w->base), L, d, w->d_ff, c,
                            static_cast<uint8_t*>(ws), W, sms, static_cast<cudaStream_t>(stream));
    }
    if (use_tc(w, batch, W, sms))
        return run_stage2_tc(w, L, x, batch, nullptr, w->d_ff, nullptr, y,
                             static_cast<uint8_t*>(ws), W, sms, static_cast<cudaStream_t>(stream));
    for (int t0 = 0; t0 < batch; t0 += W.TB) {
        const int nb = batch - t0 < W.TB ? batch - t0 : W.TB;
        PROX_TRY(run_stage2_tile(w, L, x + static_cast<size_t>(t0) * d, nb, nullptr, w->d_ff, true,
                                 y + static_cast<size_t>(t0) * d, static_cast<uint8_t*>(ws), W, sms,
                                 static_cast<cudaStream_t>(stream)));
    }
    return PROX_OK;
}

}  // namespace

int prox_sparse_ffn(const prox_packed* w, const float* x, int batch, const int32_t* idx, int k,
                    float* y, void* ws, size_t ws_bytes, void* stream) {
    PROX_TRY(check_packed(w));
    if (!x || !idx || !y || !tokens_ok(batch)) return PROX_ERR_INVALID_ARG;
    if (k < 1 || k > w->d_ff) return PROX_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(y, 16)) return PROX_ERR_INVALID_ARG;
    const int sms = device_sms();
    if (sms <= 0) return PROX_ERR_CUDA;
    WsLayout W;
    PROX_TRY(check_ws(ws, ws_bytes, w->d_model, w->d_ff, tile_batch(batch), sms, W));
    if (!fp8_stage2_ok(w, sms)) return PROX_ERR_UNSUPPORTED;
    const int d = w->d_model, F = w->d_ff;
    if (is_fp8(w)) {   // token by token through the single-token kernel
        for (int b = 0; b < batch; ++b)
            PROX_TRY(sparse_ffn_tile(w, x + static_cast<size_t>(b) * d, 1,
                                     idx + static_cast<size_t>(b) * k, k, y + static_cast<size_t>(b) * d,
                                     ws, W, sms, stream));
        return PROX_OK;
    }
    return for_token_tiles(batch, [&](int t0, int nb) {
        return sparse_ffn_tile(w, x + static_cast<size_t>(t0) * d, nb,
                               idx + static_cast<size_t>(t0) * k, k, y + static_cast<size_t>(t0) * d,
                               ws, ws_layout(d, F, nb, sms), sms, stream);
    });
}

int prox_ffn_forward(const prox_packed* w, const float* x, int batch, double sparsity,
                     double input_sparsity, float* y, int32_t* idx_out, void* ws, size_t ws_bytes,
                     void* stream) {
    PROX_TRY(check_packed(w));
    if (!x || !y || !tokens_ok(batch)) return PROX_ERR_INVALID_ARG;
    if (!sparsity_ok(sparsity) || !sparsity_ok(input_sparsity)) return PROX_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(y, 16)) return PROX_ERR_INVALID_ARG;
    const int sms = device_sms();
    if (sms <= 0) return PROX_ERR_CUDA;
    WsLayout W;
    PROX_TRY(check_ws(ws, ws_bytes, w->d_model, w->d_ff, tile_batch(batch), sms, W));
    const int d = w->d_model, F = w->d_ff, k = k_rule(sparsity, F);
    return for_token_tiles(batch, [&](int t0, int nb) {
        return run_path(w, x + static_cast<size_t>(t0) * d, nb, sparsity, input_sparsity,
                        y + static_cast<size_t>(t0) * d,
                        idx_out ? idx_out + static_cast<size_t>(t0) * k : nullptr,
                        static_cast<uint8_t*>(ws), ws_layout(d, F, nb, sms), sms,
                        static_cast<cudaStream_t>(stream), nullptr);
    });
}

int prox_ffn_forward_host(const prox_packed* w, const float* x_host, int batch, double sparsity,
                          double input_sparsity, float* y_host, void* ws, size_t ws_bytes,
                          void* stream) {
    PROX_TRY(check_packed(w));
    if (!x_host || !y_host || !tokens_ok(batch)) return PROX_ERR_INVALID_ARG;
    if (!sparsity_ok(sparsity) || !sparsity_ok(input_sparsity)) return PROX_ERR_INVALID_ARG;
    const int sms = device_sms();
    if (sms <= 0) return PROX_ERR_CUDA;
    WsLayout W;
    PROX_TRY(check_ws(ws, ws_bytes, w->d_model, w->d_ff, tile_batch(batch), sms, W));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* wsb = static_cast<uint8_t*>(ws);
    const int d = w->d_model, F = w->d_ff;
    PROX_TRY(for_token_tiles(batch, [&](int t0, int nb) {
        // the tile's x and y go through the workspace's own buffers
        const WsLayout Wt = ws_layout(d, F, nb, sms);
        float* xd = reinterpret_cast<float*>(wsb + Wt.xbuf);
        float* yd = reinterpret_cast<float*>(wsb + Wt.ybuf);
        const size_t off = static_cast<size_t>(t0) * d;
        const size_t bytes = static_cast<size_t>(nb) * d * sizeof(float);
        PROX_TRY(cuda_ok(cudaMemcpyAsync(xd, x_host + off, bytes, cudaMemcpyHostToDevice, s),
                         "copying x to the device"));
        PROX_TRY(run_path(w, xd, nb, sparsity, input_sparsity, yd, nullptr, wsb, Wt, sms, s, nullptr));
        return cuda_ok(cudaMemcpyAsync(y_host + off, yd, bytes, cudaMemcpyDeviceToHost, s),
                       "copying y to the host");
    }));
    return cuda_ok(cudaStreamSynchronize(s), "waiting for the stream");
}

int prox_dense_ffn(const prox_packed* w, const float* x, int batch, float* y, void* ws,
                   size_t ws_bytes, void* stream) {
    PROX_TRY(check_packed(w));
    if (!x || !y || !tokens_ok(batch)) return PROX_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(y, 16)) return PROX_ERR_INVALID_ARG;
    const int sms = device_sms();
    if (sms <= 0) return PROX_ERR_CUDA;
    WsLayout W;
    PROX_TRY(check_ws(ws, ws_bytes, w->d_model, w->d_ff, tile_batch(batch), sms, W));
    if (!fp8_stage2_ok(w, sms)) return PROX_ERR_UNSUPPORTED;
    const int d = w->d_model, F = w->d_ff;
    if (is_fp8(w)) {   // token by token through the single-token kernel
        for (int b = 0; b < batch; ++b)
            PROX_TRY(dense_ffn_tile(w, x + static_cast<size_t>(b) * d, 1, y + static_cast<size_t>(b) * d,
                                    ws, W, sms, stream));
        return PROX_OK;
    }
    return for_token_tiles(batch, [&](int t0, int nb) {
        return dense_ffn_tile(w, x + static_cast<size_t>(t0) * d, nb, y + static_cast<size_t>(t0) * d,
                              ws, ws_layout(d, F, nb, sms), sms, stream);
    });
}

int prox_rmsnorm(const float* y, float* x_out, int batch, int d_model, float eps, void* stream) {
    if (!y || !x_out || batch < 1 || d_model < 1 || !(eps >= 0.f)) return PROX_ERR_INVALID_ARG;
    return launch_rmsnorm(y, x_out, batch, d_model, eps, static_cast<cudaStream_t>(stream));
}

int prox_get_status(void* ws, void* stream) {
    if (!ws) return PROX_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int host = 0;
    Control* ctrl = static_cast<Control*>(ws);
    PROX_TRY(cuda_ok(cudaStreamSynchronize(s), "waiting for the stream"));
    PROX_TRY(cuda_ok(cudaMemcpyAsync(&host, &ctrl->status, sizeof(int), cudaMemcpyDeviceToHost, s),
                     "reading the status word"));
    PROX_TRY(cuda_ok(cudaMemsetAsync(&ctrl->status, 0, sizeof(int), s), "clearing the status word"));
    PROX_TRY(cuda_ok(cudaStreamSynchronize(s), "waiting for the stream"));
    return host;
}

const char* prox_last_cuda_error(void) { return last_cuda_error(); }

uint64_t prox_launch_count(void) { return launch_count(); }

const char* prox_error_string(int code) {
    switch (code) {
        case PROX_OK: return "ok";
        case PROX_ERR_INVALID_ARG: return "invalid argument";
        case PROX_ERR_WORKSPACE: return "workspace or packed buffer too small or misaligned";
        case PROX_ERR_CUDA: return "CUDA runtime error";
        case PROX_ERR_TIMEOUT: return "device wait timed out";
        case PROX_ERR_BOUNDS: return "device index out of range";
        case PROX_ERR_UNSUPPORTED: return "unsupported";
        default: return "unknown error";
    }
}

int prox_debug_stage1(const prox_packed* w, const float* x, int batch, double input_sparsity,
                      int8_t* qx_out, float* sx_out, int32_t* acc_gate, int32_t* acc_up,
                      float* salience, void* ws, size_t ws_bytes, void* stream) {
    PROX_TRY(check_packed(w));
    if (!x || batch < 1 || batch > PROX_MAX_BATCH || !sparsity_ok(input_sparsity))
        return PROX_ERR_INVALID_ARG;
    const int sms = device_sms();
    if (sms <= 0) return PROX_ERR_CUDA;
    WsLayout W;
    PROX_TRY(check_ws(ws, ws_bytes, w->d_model, w->d_ff, batch, sms, W));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t acc_bytes = static_cast<size_t>(batch) * (w->d_model / 128) * w->d_ff * 4;
    if (acc_gate) PROX_TRY(cuda_ok(cudaMemsetAsync(acc_gate, 0, acc_bytes, s), "clearing acc_gate"));
    if (acc_up) PROX_TRY(cuda_ok(cudaMemsetAsync(acc_up, 0, acc_bytes, s), "clearing acc_up"));
    Debug dbg;
    dbg.qx = qx_out;
    dbg.sx = sx_out;
    dbg.acc_gate = acc_gate;
    dbg.acc_up = acc_up;
    dbg.salience = salience;
    return run_path(w, x, batch, 0.5, input_sparsity, nullptr, nullptr, static_cast<uint8_t*>(ws), W,
                    sms, s, &dbg);
}

int prox_debug_fused_forward(const prox_packed* w, const float* x, double sparsity,
                             double input_sparsity, float* y, int32_t* sel_out, void* ws,
                             size_t ws_bytes, void* stream) {
    PROX_TRY(check_packed(w));
    if (!x || !y || !sel_out) return PROX_ERR_INVALID_ARG;
    if (!sparsity_ok(sparsity) || !sparsity_ok(input_sparsity)) return PROX_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(y, 16)) return PROX_ERR_INVALID_ARG;
    if (k_rule(sparsity, w->d_ff) == w->d_ff || !stage2_select_supported(w->d_model, w->d_ff) ||
        w->format != PROX_FORMAT_BF16)
        return PROX_ERR_UNSUPPORTED;
    const int sms = device_sms();
    if (sms <= 0) return PROX_ERR_CUDA;
    WsLayout W;
    PROX_TRY(check_ws(ws, ws_bytes, w->d_model, w->d_ff, 1, sms, W));
    static std::mutex mu;   // the hook pointer is process-wide
    std::lock_guard<std::mutex> lock(mu);
    g_fused_sel = sel_out;
    const int rc = run_path(w, x, 1, sparsity, input_sparsity, y, nullptr, static_cast<uint8_t*>(ws),
                            W, sms, static_cast<cudaStream_t>(stream), nullptr);
    g_fused_sel = nullptr;
    return rc;
}

int prox_debug_union(const int32_t* idx, int batch, int k, int d_ff, int32_t* union_out,
                     uint32_t* bits_out, int32_t* count_out, void* ws, size_t ws_bytes,
                     void* stream) {
    if (!idx || !union_out || !bits_out || !count_out || !ws) return PROX_ERR_INVALID_ARG;
    if (batch < 1 || batch > 32 || k < 1 || d_ff < 1 || d_ff > kMaxDff || k > d_ff)
        return PROX_ERR_INVALID_ARG;
    if (ws_bytes < align_up(sizeof(Control))) return PROX_ERR_WORKSPACE;
    Control* ctrl = static_cast<Control*>(ws);
    return launch_union(idx, batch, k, d_ff, union_out, bits_out, count_out, &ctrl->status,
                        static_cast<cudaStream_t>(stream));
}

int prox_debug_wait_timeout(void* ws, size_t ws_bytes, long long spin_cycles, void* stream) {
    if (!ws || spin_cycles < 0) return PROX_ERR_INVALID_ARG;
    if (ws_bytes < align_up(sizeof(Control))) return PROX_ERR_WORKSPACE;
    Control* ctrl = static_cast<Control*>(ws);
    return launch_wait_probe(&ctrl->status, spin_cycles, static_cast<cudaStream_t>(stream));
}

}  // extern "C"

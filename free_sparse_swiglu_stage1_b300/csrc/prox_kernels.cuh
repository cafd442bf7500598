// Internal interface between the C ABI (prox_api.cu) and the kernels: buffer layouts and
// launch functions. Not part of the public header.
#pragma once

#include "prox_common.cuh"

namespace prox {

constexpr size_t kAlign = PROX_ALIGN;
inline size_t align_up(size_t v, size_t a = kAlign) { return (v + a - 1) / a * a; }

// ------------------------------------------------------------------ packed layer layout
struct PackedLayout {
    size_t codes_off, scales_off, rows_off, total;
};

inline PackedLayout packed_layout(int d, int F) {
    PackedLayout L;
    L.codes_off = 0;
    L.scales_off = align_up(static_cast<size_t>(d) * F);
    L.rows_off = align_up(L.scales_off + static_cast<size_t>(d / 128) * F * 4);
    L.total = align_up(L.rows_off + static_cast<size_t>(F) * 3 * d * 2);
    return L;
}

// ------------------------------------------------------------------ token tiles
// Tokens are processed in tiles whose Stage-2 activations and partial outputs live in
// registers; wider rows leave room for fewer tokens per tile.
inline int tile_tokens(int d) { return d <= 4096 ? 4 : (d <= 8192 ? 2 : 1); }

// Stage-1 split of the kept rows (blocks of 128 channels x S row slices), bounded so the
// partial buffer stays small: nblk * S <= 8 * SMs.
inline int stage1_splits(int nblk, int nrows_est, int sms) {
    int S = (4 * sms + nblk / 2) / nblk;
    S = S < 1 ? 1 : S;
    const int smax = (8 * sms) / nblk;
    if (S > smax) S = smax < 1 ? 1 : smax;
    const int by_rows = nrows_est / 64;   // keep >= 8 rows per warp
    if (S > by_rows) S = by_rows < 1 ? 1 : by_rows;
    return S;
}
inline int stage1_splits_max(int nblk, int sms) {
    const int smax = (8 * sms) / nblk;
    return smax < 1 ? 1 : smax;
}

// Stage-2 pipeline: one stage = the three rows of one channel (6 d bytes).
constexpr size_t kStage2SmemBudget = 200 * 1024;
inline int stage2_nstage(int d) {
    int n = static_cast<int>(kStage2SmemBudget / (static_cast<size_t>(6) * d));
    return n > 16 ? 16 : (n < 2 ? 2 : n);
}
inline int stage2_batch(int nstage) { return nstage >= 8 ? 4 : (nstage >= 4 ? 2 : 1); }
// 16-byte column chunks per consumer thread: blocks stay at <= 512 consumers
inline int stage2_cpt(int d) { return d <= 2048 ? 1 : (d <= 8192 ? 2 : 4); }
inline int stage2_consumers(int d) {
    const int chunks = d / 8;
    const int cpt = stage2_cpt(d);
    int nt = (chunks / cpt + 31) / 32 * 32;
    return nt < 32 ? 32 : nt;
}

// ------------------------------------------------------------------ workspace layout
struct WsLayout {
    size_t control, s1_cnt, xbuf, ybuf, rows, qxt, sx, gstart, s1part, sigma, idx, ulist, ubits,
        ypart, total;
    int TB, S_max, P, nblk;
};

inline WsLayout ws_layout(int d, int F, int B, int sms) {
    WsLayout W;
    const int G = d / 128;
    W.TB = tile_tokens(d);
    W.nblk = (F + 127) / 128;
    W.S_max = stage1_splits_max(W.nblk, sms);
    W.P = sms;
    size_t o = 0;
    auto take = [&](size_t bytes) { const size_t at = o; o = align_up(o + bytes); return at; };
    W.control = take(sizeof(Control));
    W.s1_cnt = take(static_cast<size_t>(W.nblk) * 4);
    W.xbuf = take(static_cast<size_t>(B) * d * 4);
    W.ybuf = take(static_cast<size_t>(B) * d * 4);
    W.rows = take(static_cast<size_t>(d) * 4);
    W.qxt = take(static_cast<size_t>(d) * 4);
    W.sx = take(static_cast<size_t>(W.TB) * G * 4);
    W.gstart = take(static_cast<size_t>(G + 2) * 4);
    W.s1part = take(static_cast<size_t>(W.S_max) * W.TB * F * 16);
    W.sigma = take(static_cast<size_t>(B) * F * 4);
    W.idx = take(static_cast<size_t>(B) * F * 4);
    W.ulist = take(static_cast<size_t>(F) * 4);
    W.ubits = take(static_cast<size_t>(F) * 4);
    W.ypart = take(static_cast<size_t>(W.P) * W.TB * d * 4);
    W.total = o;
    return W;
}

// Bytes of the control region that prox_workspace_init clears (control block + counters).
inline size_t ws_control_bytes(int nblk) { return align_up(sizeof(Control)) + align_up(nblk * 4); }

// ------------------------------------------------------------------ launches
int launch_pack(const uint16_t* w_gate, const uint16_t* w_up, const uint16_t* w_down, int d,
                int F, const PackedLayout& L, uint8_t* base, cudaStream_t s);

// Input selection + activation quantization for one tile of nb tokens (Stage 1 inputs).
int launch_input_quant(const float* x, int d, int nb, int k_in, uint8_t* ws, const WsLayout& W,
                       int8_t* dbg_qx, float* dbg_sx, cudaStream_t s);

// Stage-1 proxy projections + salience for one tile.
int launch_stage1(const uint8_t* packed, const PackedLayout& L, int d, int F, int nb, int k_in,
                  uint8_t* ws, const WsLayout& W, float* sigma_tile, int32_t* dbg_gate,
                  int32_t* dbg_up, int sms, cudaStream_t s);

// Per-token top-k of the salience -> ascending channel indices (row stride k).
int launch_topk(const float* sigma_tile, int F, int nb, int k, int32_t* idx_tile,
                cudaStream_t s);

// Union of nb index rows (row stride k) -> ascending list + per-entry token bits + count.
int launch_union(const int32_t* idx_tile, int nb, int k, int F, int32_t* ulist, uint32_t* ubits,
                 int* count, int* status, cudaStream_t s);

// Stage 2 over a channel list for one tile; list == nullptr means every channel.
int launch_stage2(const uint8_t* packed, const PackedLayout& L, int d, int F, const float* x_tile,
                  int nb, const int32_t* list, const uint32_t* lbits, const int* count_dev,
                  int count_host, float* y_tile, uint8_t* ws, const WsLayout& W, int sms,
                  cudaStream_t s);

int launch_rmsnorm(const float* y, float* x_out, int batch, int d, float eps, cudaStream_t s);

int launch_iota(int32_t* out, int n, int rows, cudaStream_t s);

int launch_wait_probe(int* status, long long spin_cycles, cudaStream_t s);

}  // namespace prox

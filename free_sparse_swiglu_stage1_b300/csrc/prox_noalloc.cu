// prox_sparse_ffn_noalloc: the Stage-2 sparse FFN of prox_sparse_ffn for callers that cannot
// hand the library a workspace -- code that runs where device allocation is not allowed or
// not affordable, such as a serving runtime that has reserved all device memory for its own
// pool, or a latency-critical loop that cannot take cudaMalloc's implicit synchronization.
//
// The per-block partial sums, the batch union and the status word live in one file-scope
// device array of fixed size instead of a caller workspace. Every GPU that loads the library
// holds this array until the process exits. The host never dereferences the array's name:
// the first call on each device, with that device current, asks the runtime for the
// array's device address (cudaGetSymbolAddress) and caches it; later calls reuse it.
// Nothing here allocates: no cudaMalloc, no cudaFree, no allocating library routine.
#include <mutex>

#include "prox_kernels.cuh"

using namespace prox;

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[PROX_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 128;

// Device address of the scratch array on the current device, looked up once per device.
int scratch_address(uint8_t** out) {
    static std::mutex mu;
    static void* addr[kMaxDevices] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PROX_ERR_CUDA;
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return PROX_ERR_CUDA;
        addr[dev] = p;
    }
    *out = static_cast<uint8_t*>(addr[dev]);
    return PROX_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int prox_sparse_ffn_noalloc(const prox_packed* w, const float* x, int batch,
                                       const int32_t* idx, int k, float* y, int* status_out,
                                       void* stream) {
    // the same argument rules as prox_sparse_ffn
    if (!w || !w->base || !x || !idx || !y) return PROX_ERR_INVALID_ARG;
    const int d = w->d_model, F = w->d_ff;
    if (w->group != PROX_GROUP || d < 128 || d % 128 != 0 || F < 32 || F % 32 != 0)
        return PROX_ERR_INVALID_ARG;
    if (w->format != PROX_FORMAT_BF16) return PROX_ERR_UNSUPPORTED;   // bf16 rows only
    if (batch < 1 || batch > PROX_MAX_BATCH || k < 1 || k > F) return PROX_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(y)) return PROX_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(w->base) % kAlign) != 0) return PROX_ERR_WORKSPACE;
    if (w->proxy && (reinterpret_cast<uintptr_t>(w->proxy) % kAlign) != 0) return PROX_ERR_WORKSPACE;
    const PackedLayout L = packed_layout_of(w);   // Stage 2 reads the rows only
    if (w->bytes < L.total) return PROX_ERR_WORKSPACE;

    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        return PROX_ERR_CUDA;

    // the scratch this call needs: control block, batch union, per-block partial outputs
    WsLayout W{};
    W.TB = tile_tokens(d);
    const int TB = batch < W.TB ? (batch <= 1 ? 1 : (batch <= 2 ? 2 : 4)) : W.TB;
    W.TB = TB;
    W.P = stage2_blocks(F, sms);
    size_t o = 0;
    auto take = [&](size_t bytes) { const size_t at = o; o = align_up(o + bytes); return at; };
    W.control = take(sizeof(Control));
    W.ulist = take(static_cast<size_t>(F) * 4);
    W.ubits = take(static_cast<size_t>(F) * 4);
    W.ypart = take(static_cast<size_t>(W.P) * TB * d * 4);
    W.total = o;
    if (W.total > PROX_NOALLOC_SCRATCH_BYTES) return PROX_ERR_WORKSPACE;

    uint8_t* ws = nullptr;
    if (scratch_address(&ws) != PROX_OK) return PROX_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the array keeps the previous call's contents: the status word and the union count
    // must start at zero
    if (cudaMemsetAsync(ws + W.control, 0, sizeof(Control), s) != cudaSuccess) return PROX_ERR_CUDA;

    Control* ctrl = reinterpret_cast<Control*>(ws + W.control);
    const uint8_t* packed = static_cast<const uint8_t*>(w->base);
    for (int t0 = 0; t0 < batch; t0 += TB) {
        const int nb = batch - t0 < TB ? batch - t0 : TB;
        const float* xt = x + static_cast<size_t>(t0) * d;
        const int32_t* it = idx + static_cast<size_t>(t0) * k;
        float* yt = y + static_cast<size_t>(t0) * d;
        int rc;
        if (nb == 1) {
            rc = launch_stage2(packed, L, d, F, xt, 1, it, nullptr, nullptr, k, yt, ws, W, sms, s);
        } else {
            int32_t* ulist = reinterpret_cast<int32_t*>(ws + W.ulist);
            uint32_t* ubits = reinterpret_cast<uint32_t*>(ws + W.ubits);
            rc = launch_union(it, nb, k, F, ulist, ubits, &ctrl->union_count, &ctrl->status, s);
            if (rc == PROX_OK)
                rc = launch_stage2(packed, L, d, F, xt, nb, ulist, ubits, &ctrl->union_count, 0,
                                   yt, ws, W, sms, s);
        }
        if (rc != PROX_OK) return rc;
    }
    if (status_out) {
        int host = 0;
        if (cudaMemcpyAsync(&host, &ctrl->status, sizeof(int), cudaMemcpyDeviceToHost, s) !=
                cudaSuccess ||
            cudaStreamSynchronize(s) != cudaSuccess)
            return PROX_ERR_CUDA;
        *status_out = host;
    }
    return PROX_OK;
}

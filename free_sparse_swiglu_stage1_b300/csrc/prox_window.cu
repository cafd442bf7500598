// Proxy-memory reduction by a sliding window over a layer stack (technical summary,
// "Significance and Claims": storing the INT4 proxies costs about 12% extra memory, and
// sliding-window schemes are named as the way to cut it; the pages describe no scheme).
//
// Reading used here: a decode step visits the layers in order 0, 1, ..., L - 1, and the next
// step starts again at 0. Only S proxy slots live in device memory; every layer's proxy
// (codes and scales, the part of the packed layer Stage 1 reads) lives in pinned host memory.
// When layer l is acquired, the window is the S layers l, l + 1, ..., l + S - 1 (cyclically):
// each of them is resident in a slot or being copied into one. Releasing layer l frees its slot
// for the next layer that enters the window, l + S. Copies run on the window's own stream and
// overlap the compute of the layers before them; events order every copy after the compute
// that last read its slot, and every compute after the copy it reads. Device memory for
// proxies drops from L to S layers' worth; Stage 2's rows stay resident.
//
// The slot policy is a plain host class (WindowPlan), shared by the CUDA-backed window and a
// test hook that runs it on the host alone.
#include <cstring>
#include <new>
#include <vector>

#include "prox_kernels.cuh"

namespace prox {
namespace {

struct Copy {
    int slot, layer;
};

// Which layer each slot holds (or is receiving) and which slots are in use by a compute.
class WindowPlan {
public:
    WindowPlan(int layers, int slots) : L_(layers), S_(slots), held_(slots, -1), busy_(slots, 0) {}

    int slot_of(int layer) const {
        for (int s = 0; s < S_; ++s)
            if (held_[s] == layer) return s;
        return -1;
    }
    bool busy(int slot) const { return busy_[slot] != 0; }

    // Acquire `layer`: returns its slot (-1 if every slot is in use) and appends the copies to
    // issue, in order: first the layer itself if it is not resident, then the layers after it
    // in the window that fit into free slots.
    int acquire(int layer, std::vector<Copy>& copies) {
        int s = slot_of(layer);
        if (s < 0) {
            s = victim(layer);
            if (s < 0) return -1;
            held_[s] = layer;
            copies.push_back({s, layer});
        }
        busy_[s] = 1;
        prefetch(layer, 1, copies);
        return s;
    }

    // Release `layer` (acquired before): its slot may be refilled, with the layers of the
    // window that starts at the next layer.
    int release(int layer, std::vector<Copy>& copies) {
        const int s = slot_of(layer);
        if (s < 0 || !busy_[s]) return -1;
        busy_[s] = 0;
        prefetch((layer + 1) % L_, 0, copies);
        return s;
    }

private:
    bool in_window(int start, int layer) const {
        if (S_ >= L_) return true;
        const int ahead = ((layer - start) % L_ + L_) % L_;
        return ahead < S_;
    }
    // A slot for `layer`: an empty one, else an idle one holding a layer outside the window
    // that starts at `start` (the lowest index, so the choice is deterministic).
    int victim_for(int start) const {
        for (int s = 0; s < S_; ++s)
            if (held_[s] < 0) return s;
        for (int s = 0; s < S_; ++s)
            if (!busy_[s] && !in_window(start, held_[s])) return s;
        return -1;
    }
    // A slot for the layer being acquired: as above, else any idle slot (a caller that
    // leaves the decode order may evict a layer the window would have kept).
    int victim(int layer) const {
        const int s = victim_for(layer);
        if (s >= 0) return s;
        for (int t = 0; t < S_; ++t)
            if (!busy_[t]) return t;
        return -1;
    }
    void prefetch(int start, int first, std::vector<Copy>& copies) {
        const int n = S_ < L_ ? S_ : L_;
        for (int j = first; j < n; ++j) {
            const int m = (start + j) % L_;
            if (slot_of(m) >= 0) continue;
            const int s = victim_for(start);
            if (s < 0) return;
            held_[s] = m;
            copies.push_back({s, m});
        }
    }

    int L_, S_;
    std::vector<int> held_;
    std::vector<char> busy_;
};

}  // namespace
}  // namespace prox

using prox::Copy;
using prox::WindowPlan;

struct prox_window {
    WindowPlan plan;
    int layers, slots;
    size_t proxy_bytes;
    std::vector<const void*> host;
    uint8_t* slot_mem;
    cudaStream_t copy = nullptr;
    std::vector<cudaEvent_t> ready, freed;
    std::vector<char> freed_set;   // the slot's last reader recorded `freed`
    uint64_t n_copies = 0, n_bytes = 0;

    prox_window(int L, int S) : plan(L, S), layers(L), slots(S) {}
};

namespace {

int issue(prox_window* w, const std::vector<Copy>& copies) {
    for (const Copy& c : copies) {
        if (w->freed_set[c.slot] &&
            cudaStreamWaitEvent(w->copy, w->freed[c.slot], 0) != cudaSuccess)
            return PROX_ERR_CUDA;
        if (cudaMemcpyAsync(w->slot_mem + static_cast<size_t>(c.slot) * w->proxy_bytes,
                            w->host[c.layer], w->proxy_bytes, cudaMemcpyHostToDevice,
                            w->copy) != cudaSuccess ||
            cudaEventRecord(w->ready[c.slot], w->copy) != cudaSuccess)
            return PROX_ERR_CUDA;
        ++w->n_copies;
        w->n_bytes += w->proxy_bytes;
    }
    return PROX_OK;
}

void destroy(prox_window* w) {
    if (!w) return;
    if (w->copy) cudaStreamSynchronize(w->copy);
    for (cudaEvent_t e : w->ready)
        if (e) cudaEventDestroy(e);
    for (cudaEvent_t e : w->freed)
        if (e) cudaEventDestroy(e);
    if (w->copy) cudaStreamDestroy(w->copy);
    delete w;
}

}  // namespace

extern "C" {

size_t prox_proxy_bytes(int d_model, int d_ff, int group) {
    if (group != PROX_GROUP || d_model < 128 || d_model % 128 || d_model > 16384 || d_ff < 32 ||
        d_ff % 32 || d_ff > 53248)
        return 0;
    return prox::packed_layout(d_model, d_ff).proxy_bytes;
}

size_t prox_rows_bytes(int d_model, int d_ff, int group, int format) {
    if (prox_proxy_bytes(d_model, d_ff, group) == 0) return 0;
    if (format != PROX_FORMAT_BF16 && format != PROX_FORMAT_FP8) return 0;
    const prox::PackedLayout L = prox::packed_layout(d_model, d_ff, format);
    return prox::align_up(static_cast<size_t>(d_ff) * L.row_bytes);
}

int prox_split_packed(const prox_packed* full, void* rows_dev, size_t rows_bytes, void* proxy_out,
                      size_t proxy_bytes, void* stream, prox_packed* out) {
    if (!full || !full->base || full->proxy || !rows_dev || !proxy_out || !out)
        return PROX_ERR_INVALID_ARG;
    const int d = full->d_model, F = full->d_ff;
    const size_t pb = prox_proxy_bytes(d, F, full->group);
    const size_t rb = prox_rows_bytes(d, F, full->group, full->format);
    if (pb == 0 || rb == 0) return PROX_ERR_INVALID_ARG;
    const prox::PackedLayout L = prox::packed_layout(d, F, full->format);
    if (full->bytes < L.total || rows_bytes < rb || proxy_bytes < pb) return PROX_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(rows_dev) % PROX_ALIGN) ||
        (reinterpret_cast<uintptr_t>(proxy_out) % PROX_ALIGN))
        return PROX_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const uint8_t* src = static_cast<const uint8_t*>(full->base);
    if (cudaMemcpyAsync(proxy_out, src, pb, cudaMemcpyDefault, s) != cudaSuccess ||
        cudaMemcpyAsync(rows_dev, src + L.rows_off, static_cast<size_t>(F) * L.row_bytes,
                        cudaMemcpyDefault, s) != cudaSuccess)
        return PROX_ERR_CUDA;
    *out = *full;
    out->base = rows_dev;
    out->bytes = rows_bytes;
    out->proxy = proxy_out;
    return PROX_OK;
}

int prox_window_create(int n_layers, int n_slots, int d_model, int d_ff,
                       const void* const* host_proxies, void* slots_dev, size_t slots_bytes,
                       prox_window** out) {
    if (!out || !host_proxies || !slots_dev || n_layers < 1 || n_slots < 1)
        return PROX_ERR_INVALID_ARG;
    *out = nullptr;
    const size_t pb = prox_proxy_bytes(d_model, d_ff, PROX_GROUP);
    if (pb == 0) return PROX_ERR_INVALID_ARG;
    for (int l = 0; l < n_layers; ++l)
        if (!host_proxies[l]) return PROX_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(slots_dev) % PROX_ALIGN) ||
        slots_bytes < static_cast<size_t>(n_slots) * pb)
        return PROX_ERR_WORKSPACE;
    prox_window* w = new (std::nothrow) prox_window(n_layers, n_slots);
    if (!w) return PROX_ERR_INVALID_ARG;
    w->proxy_bytes = pb;
    w->host.assign(host_proxies, host_proxies + n_layers);
    w->slot_mem = static_cast<uint8_t*>(slots_dev);
    w->ready.assign(n_slots, nullptr);
    w->freed.assign(n_slots, nullptr);
    w->freed_set.assign(n_slots, 0);
    bool ok = cudaStreamCreateWithFlags(&w->copy, cudaStreamNonBlocking) == cudaSuccess;
    for (int s = 0; ok && s < n_slots; ++s)
        ok = cudaEventCreateWithFlags(&w->ready[s], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&w->freed[s], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
        destroy(w);
        return PROX_ERR_CUDA;
    }
    *out = w;
    return PROX_OK;
}

int prox_window_acquire(prox_window* w, int layer, prox_packed* desc, void* stream) {
    if (!w || !desc || layer < 0 || layer >= w->layers) return PROX_ERR_INVALID_ARG;
    if (prox_proxy_bytes(desc->d_model, desc->d_ff, desc->group) != w->proxy_bytes)
        return PROX_ERR_INVALID_ARG;
    std::vector<Copy> copies;
    const int s = w->plan.acquire(layer, copies);
    if (s < 0) return PROX_ERR_UNSUPPORTED;   // every slot is held by an acquired layer
    const int rc = issue(w, copies);
    if (rc != PROX_OK) return rc;
    if (cudaStreamWaitEvent(static_cast<cudaStream_t>(stream), w->ready[s], 0) != cudaSuccess)
        return PROX_ERR_CUDA;
    desc->proxy = w->slot_mem + static_cast<size_t>(s) * w->proxy_bytes;
    return PROX_OK;
}

int prox_window_release(prox_window* w, int layer, void* stream) {
    if (!w || layer < 0 || layer >= w->layers) return PROX_ERR_INVALID_ARG;
    const int s = w->plan.slot_of(layer);
    if (s < 0 || !w->plan.busy(s)) return PROX_ERR_INVALID_ARG;
    // the slot's reader is everything enqueued on `stream` so far
    if (cudaEventRecord(w->freed[s], static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return PROX_ERR_CUDA;
    w->freed_set[s] = 1;
    std::vector<Copy> copies;
    w->plan.release(layer, copies);
    return issue(w, copies);
}

int prox_window_stats(const prox_window* w, uint64_t* copies, uint64_t* bytes) {
    if (!w) return PROX_ERR_INVALID_ARG;
    if (copies) *copies = w->n_copies;
    if (bytes) *bytes = w->n_bytes;
    return PROX_OK;
}

int prox_window_destroy(prox_window* w) {
    if (!w) return PROX_ERR_INVALID_ARG;
    destroy(w);
    return PROX_OK;
}

int prox_debug_window_plan(int n_layers, int n_slots, const int* ops, int n_ops, int* slot_out,
                           int* copy_log, int copy_cap, int* n_copies) {
    if (n_layers < 1 || n_slots < 1 || !ops || n_ops < 0 || !slot_out || !n_copies ||
        (copy_cap > 0 && !copy_log))
        return PROX_ERR_INVALID_ARG;
    WindowPlan plan(n_layers, n_slots);
    int nc = 0;
    for (int i = 0; i < n_ops; ++i) {
        std::vector<Copy> copies;
        const int op = ops[i];
        const int layer = op >= 0 ? op : -1 - op;
        if (layer >= n_layers) return PROX_ERR_INVALID_ARG;
        slot_out[i] = op >= 0 ? plan.acquire(layer, copies) : plan.release(layer, copies);
        for (const Copy& c : copies) {
            if (nc < copy_cap) {
                copy_log[3 * nc] = i;
                copy_log[3 * nc + 1] = c.slot;
                copy_log[3 * nc + 2] = c.layer;
            }
            ++nc;
        }
    }
    *n_copies = nc;
    return PROX_OK;
}

}  // extern "C"

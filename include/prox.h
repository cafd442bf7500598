/*
 * prox.h -- C ABI of the B300 (sm_103a) Prox sparse SwiGLU FFN decode path.
 *
 * The method: "Prox: Training-Free FFN Activation Sparsity via Approximate
 * Intermediate-Channel Salience in LLMs". Stage 1 applies input sparsity to the FFN input
 * x and runs INT4 proxies of W_gate and W_up to rank the intermediate channels by the
 * magnitude of s~ = u~ (.) h~, giving one shared channel mask. Stage 2 computes only the
 * masked channels exactly from the bf16 weights and runs the down projection over the same
 * channels (technical summary, "Methodology: The Prox Framework"; the authors' abstract).
 *
 * Conventions for every call below.
 *  - Ownership: every pointer is caller-owned memory; "device" pointers are CUDA device
 *    memory of the current device. The library allocates nothing and frees nothing.
 *  - Asynchrony: calls enqueue kernels on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) and return at once. Only prox_get_status and prox_ffn_forward_host wait.
 *  - Validation happens on the host before any launch. On a returned error nothing was
 *    launched and no output was written.
 *  - Errors: PROX_OK (0) or a negative PROX_ERR_* code. Device-side faults the kernels
 *    detect themselves (a bounded wait that ran out, an index out of range) are recorded in
 *    a status word inside the workspace and reported by prox_get_status.
 *  - Layouts are row-major. bf16 is passed as uint16_t bit patterns.
 *  - Shapes: d_model a multiple of 128 in [128, 16384]; d_ff a multiple of 32 in
 *    [32, 53248]; batch in [1, PROX_MAX_TOKENS] (prox_debug_* and prox_sparse_ffn_noalloc:
 *    [1, PROX_MAX_BATCH]). Inputs must be finite.
 *  - Large batches: the pages leave large-batch serving open (technical summary,
 *    "Significance and Claims", limitations). A call with more than PROX_MAX_BATCH tokens
 *    runs as consecutive tiles of PROX_MAX_BATCH tokens (the last one ragged), each tile
 *    exactly as a call of its own; every token still gets its own input set and mask, so the
 *    result is the same as tile-sized calls. The workspace of such a call is that of one
 *    full tile (prox_workspace_bytes returns the same size for any batch >= PROX_MAX_BATCH).
 *  - Sparsities are fractions in [0, 1). The kept counts are
 *        k    = clamp(floor((1 - sparsity) * d_ff + 0.5), 1, d_ff)
 *        k_in = clamp(floor((1 - input_sparsity) * d_model + 0.5), 1, d_model)
 *    computed in IEEE double (see prox_k_for). The pages ask for at least 30% of the inputs
 *    to be kept (technical summary, "Sparsity Allocation", Stage 1 constraint); this is
 *    documented, not enforced.
 *  - A workspace must be initialised once with prox_workspace_init before its first use;
 *    calls that overlap in time (different streams) need different workspaces.
 */
#ifndef PROX_H_
#define PROX_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PROX_OK               0
#define PROX_ERR_INVALID_ARG (-1)  /* null pointer, bad shape, sparsity outside [0,1)      */
#define PROX_ERR_WORKSPACE   (-2)  /* workspace or packed buffer too small or misaligned   */
#define PROX_ERR_CUDA        (-3)  /* a CUDA runtime call or launch failed                 */
#define PROX_ERR_TIMEOUT     (-4)  /* device status: a bounded wait ran out                */
#define PROX_ERR_BOUNDS      (-5)  /* device status: an index was out of range             */
#define PROX_ERR_UNSUPPORTED (-6)  /* valid request the library does not implement        */

#define PROX_GROUP      128        /* proxy quantization group along d_model               */
#define PROX_FORMAT_BF16  0        /* packed Stage-2 rows: the layer's bf16 weights        */
#define PROX_FORMAT_FP8   1        /* packed Stage-2 rows: FP8 E4M3 with fp32 row scales   */
#define PROX_MAX_BATCH  16         /* tokens per tile (one pass of the batch kernels)      */
#define PROX_MAX_TOKENS 1024       /* tokens per call; larger calls run tile by tile       */
#define PROX_ALIGN      256        /* required alignment of packed and workspace buffers   */

/* Descriptor of one packed layer. A plain view of caller-owned device memory that
 * prox_pack_weights (or prox_pack_weights_fp8) fills; copy it freely. Field meaning:
 *   d_model, d_ff, group  the layer shape and the proxy group (128);
 *   format                PROX_FORMAT_BF16 or PROX_FORMAT_FP8 (how the Stage-2 rows are kept);
 *   base, bytes           the packed device buffer (PROX_ALIGN-aligned) and its size.
 * Packed layout inside base (offsets are multiples of PROX_ALIGN, in this order):
 *   codes  [d_model][d_ff] uint8: byte (i, j) holds the INT4 proxy codes of input i for
 *          channel j, W_gate in the low nibble and W_up in the high nibble, each stored
 *          as q + 8 with q in [-7, 7] (input-major, so a kept input is one row);
 *   scales [d_model/128][d_ff] uint32: the fp16 group scales, W_gate's in the low half and
 *          W_up's in the high half;
 *   rows   [d_ff][3][d_model] bf16: for channel j the rows W_gate[j,:], W_up[j,:] and
 *          W_down[:,j] one after another (channel-major, one contiguous run per channel).
 *          With PROX_FORMAT_FP8 instead [d_ff][3 d_model + 16] bytes: per channel the same
 *          three rows as FP8 E4M3 codes (one byte each), then the three rows' fp32 scales
 *          and one fp32 zero; a weight is code * scale.
 *   proxy  NULL for the layout above. Otherwise a split layer (prox_split_packed): the
 *          proxy -- codes, then scales at the same offsets as above, prox_proxy_bytes
 *          bytes -- lives at `proxy` (device memory, PROX_ALIGN-aligned) and base holds only
 *          the rows, from offset 0 (prox_rows_bytes bytes). Compute calls check that proxy
 *          is device memory and return PROX_ERR_INVALID_ARG if it is not. */
typedef struct prox_packed {
    int32_t d_model;
    int32_t d_ff;
    int32_t group;
    int32_t format;
    void*   base;
    size_t  bytes;
    void*   proxy;
} prox_packed;

/* Cost model of one layer for prox_choose_sparsity: per token, the sparse path costs
 *   in_cost * k_in + fixed_cost + ch_cost * k
 * (k_in kept inputs, k selected channels) and the dense FFN dense_cost, in any one unit
 * (bytes of HBM traffic, or measured microseconds). */
typedef struct prox_cost_model {
    double in_cost;      /* per kept input (Stage 1 reads one proxy row)                    */
    double fixed_cost;   /* independent of the sparsities (proxy scales, selections)        */
    double ch_cost;      /* per selected channel (Stage 2 reads three bf16 rows)            */
    double dense_cost;   /* the dense SwiGLU FFN of the same layer                          */
} prox_cost_model;

/* The HBM-byte cost model of a layer shape: in_cost = d_ff (one byte of INT4 gate+up codes
 * per channel), fixed_cost = 4 * (d_model / 128) * d_ff (fp16 scales of both proxies),
 * ch_cost = 6 * d_model, dense_cost = 6 * d_model * d_ff. PROX_ERR_INVALID_ARG for a bad
 * shape or a NULL out. */
int prox_cost_model_bytes(int d_model, int d_ff, prox_cost_model* out);

/* A cost model fitted to measured times: the least-squares fit of
 *   t = in_cost * k_in + fixed_cost + ch_cost * k
 * over n >= 3 measurements (k_in[i], k[i], t[i]) of the sparse path on one layer shape, with
 * dense_cost = dense_t (the dense FFN's measured time, same unit). Host-only. Coefficients
 * that come out below min_cost (noise on a term the path barely depends on) are raised to it,
 * so the model stays valid for prox_choose_sparsity. PROX_ERR_INVALID_ARG for NULL
 * pointers, n < 3, non-finite or negative inputs, dense_t <= 0, or measurements whose
 * (k_in, k) points do not determine the three coefficients. */
int prox_cost_model_fit(const double* k_in, const double* k, const double* t, int n, double dense_t,
                        double min_cost, prox_cost_model* out);

/* Sparsity allocation (technical summary, "Sparsity Allocation": the Stage 2 sparsity is
 * anchored around 70%, Stage 1 keeps at least 30% of the inputs, and a cost model chooses the
 * two sparsities for a target effective sparsity, counting the proxy's overhead). The pages
 * give no formula; this call implements the following reading.
 *   Effective sparsity = 1 - C, with C = (in_cost k_in + fixed_cost + ch_cost k) / dense_cost
 *   the sparse path's cost relative to the dense FFN. For `target` in [0, 1), the budget is
 *   C <= 1 - target. Rule: keep k = prox_k_for(anchor, d_ff) channels and the most inputs
 *   the budget allows; if that is every input, keep every input and the most channels that
 *   fit; if it is fewer than ceil(min_input_kept * d_model), keep that many inputs and the
 *   most channels that fit.
 *   Outputs (any may be NULL): input_sparsity = 1 - k_in / d_model and sparsity =
 *   1 - k / d_ff (prox_k_for maps them back to k_in and k), effective = 1 - C.
 * Host-only: launches nothing. PROX_ERR_INVALID_ARG for bad arguments (costs must be
 * positive, 0 <= anchor < 1, 0 < min_input_kept <= 1), PROX_ERR_UNSUPPORTED if no allocation
 * fits the budget. */
int prox_choose_sparsity(const prox_cost_model* cost, int d_model, int d_ff, double target,
                         double anchor, double min_input_kept, double* input_sparsity,
                         double* sparsity, double* effective);

/* Bytes prox_pack_weights needs for one layer; 0 if the shape is invalid. */
size_t prox_packed_bytes(int d_model, int d_ff, int group);

/* Bytes prox_pack_weights_fp8 needs for one layer; 0 if the shape is invalid. */
size_t prox_packed_bytes_fp8(int d_model, int d_ff, int group);

/* Workspace bytes a call on this layer shape and batch needs on the CURRENT device (it
 * depends on the device's SM count); 0 if the shape is invalid. One workspace serves every
 * call on shapes no larger than the ones it was sized for. A batch above PROX_MAX_BATCH
 * needs the workspace of PROX_MAX_BATCH tokens. */
size_t prox_workspace_bytes(int d_model, int d_ff, int batch);

/* Clears the workspace's status word and its self-resetting counters. Call once after
 * allocating a workspace, and again after prox_get_status reported a device error. */
int prox_workspace_init(void* ws, size_t ws_bytes, void* stream);

/* The kept-count rule above: clamp(floor((1 - sparsity) * n + 0.5), 1, n); -1 if the
 * sparsity is outside [0, 1) or n < 1. */
int prox_k_for(double sparsity, int n);

/* Builds the Stage-1 proxies and the Stage-2 channel-major rows of one layer
 * (technical summary, Stage 1 "Input Sparsity & Quantization": INT4 proxy weights for the
 * up and gate projections; Stage 2 "Exact Projections": the original bf16 weights).
 *   w_gate [d_ff][d_model], w_up [d_ff][d_model], w_down [d_model][d_ff]: device bf16 in
 *          nn.Linear layout; read only, not needed after the call's kernels finish.
 *   group  must be 128.
 *   packed_dev / packed_bytes: device buffer of at least prox_packed_bytes() bytes,
 *          PROX_ALIGN-aligned; written by the kernels.
 *   out    host descriptor, filled on success.
 * Proxy rule per channel j and group g of 128 inputs: a = max |w|,
 * sw = fp16(fp32(a) / 7), q = clamp(rint(fp32(w) / fp32(sw)), -7, 7), q = 0 if sw == 0. */
int prox_pack_weights(const uint16_t* w_gate, const uint16_t* w_up, const uint16_t* w_down,
                      int d_model, int d_ff, int group,
                      void* packed_dev, size_t packed_bytes, void* stream, prox_packed* out);

/* prox_pack_weights with the Stage-2 rows kept as FP8 E4M3 instead of bf16 (technical
 * summary, "Experimental Results", Compatibility: Prox is orthogonal to weight quantization
 * such as FP8). The INT4 proxies are built from the same bf16 weights as in
 * prox_pack_weights, so Stage 1 and the mask do not change; Stage 2 multiplies with the
 * FP8 weights and reads half the bytes. Rule per row r (W_gate[j,:], W_up[j,:], W_down[:,j]):
 * s = fp32(max |w|) / 448, code = e4m3(fp32(w) / s) rounded to nearest even and saturated
 * at 448 (both divisions in IEEE binary32), code = 0 if s == 0. Arguments as for
 * prox_pack_weights (packed_bytes >= prox_packed_bytes_fp8); out->format = PROX_FORMAT_FP8.
 * Calls that run Stage 2 on such a layer (prox_sparse_ffn, prox_ffn_forward,
 * prox_ffn_forward_host, prox_dense_ffn) run a batch token by token through the single-token
 * kernel; prox_build_mask and prox_debug_stage1 are unchanged (Stage 1 reads the proxies). */
int prox_pack_weights_fp8(const uint16_t* w_gate, const uint16_t* w_up, const uint16_t* w_down,
                          int d_model, int d_ff, int group,
                          void* packed_dev, size_t packed_bytes, void* stream, prox_packed* out);

/* Stage 1 alone: input sparsity, INT4 proxy projections, salience |SiLU(g~) * u~| and the
 * top-k channel mask (technical summary, Stage 1 "Proxy Activation" and "Mask
 * Generation"; abstract: the mask comes from the magnitude ranking of the entries).
 *   x       [batch][d_model] fp32, device.
 *   idx_out [batch][k] int32, device: per token the k selected channels in ascending order;
 *           equal salience goes to the lower channel index.
 *   ws      device workspace of at least prox_workspace_bytes(d_model, d_ff, batch). */
int prox_build_mask(const prox_packed* w, const float* x, int batch,
                    double sparsity, double input_sparsity,
                    int32_t* idx_out, void* ws, size_t ws_bytes, void* stream);

/* Stage 2 alone, for a given mask (technical summary, Stage 2 "Exact Projections" and
 * "Final Output"): for each token b, y_b = sum over j in idx[b] of
 * SiLU(W_gate[j,:] . x_b) * (W_up[j,:] . x_b) * W_down[:, j], with bf16 weights and fp32
 * accumulation. One token runs on the CUDA cores with fp32 activations; a batch of 2 to 16
 * runs once over the union of its masks on the tensor cores, with x and SiLU(g) * u each
 * entered as a pair of bf16 values hi + lo (about 17 significant bits). The cross-block sum
 * runs in a fixed order, so the result is bit-reproducible on a given device.
 *   x   [batch][d_model] fp32 device;  idx [batch][k] int32 device, each row strictly
 *   ascending in [0, d_ff);  y [batch][d_model] fp32 device (written). 1 <= k <= d_ff. */
int prox_sparse_ffn(const prox_packed* w, const float* x, int batch, const int32_t* idx,
                    int k, float* y, void* ws, size_t ws_bytes, void* stream);

/* The whole path: Stage 1 mask, then Stage 2 over it (technical summary, "Methodology: The
 * Prox Framework": Stage 1 "Lightweight Proxy Construction" builds the shared mask m_s, Stage
 * 2 "Exact Sparse Computation" computes the masked channels exactly; the authors' abstract:
 * all three projections run sparse under the one mask). At sparsity 0 every channel is kept
 * and Stage 1 is skipped (the result is the dense FFN). One token runs the whole path in one
 * launch; two tokens run as two such launches; 3 to 16 tokens run the batch kernels (Stage 2
 * on the tensor cores over the union of the masks), larger batches 16-token tiles of those.
 *   y       [batch][d_model] fp32 device (written).
 *   idx_out [batch][k] int32 device, or NULL when the mask is not wanted. */
int prox_ffn_forward(const prox_packed* w, const float* x, int batch,
                     double sparsity, double input_sparsity,
                     float* y, int32_t* idx_out, void* ws, size_t ws_bytes, void* stream);

/* prox_ffn_forward with HOST input and output: copies x_host (batch x d_model fp32) to the
 * workspace, runs the path, copies y back to y_host, and waits for the stream. Pinned host
 * buffers make the copies asynchronous with respect to other streams. */
int prox_ffn_forward_host(const prox_packed* w, const float* x_host, int batch,
                          double sparsity, double input_sparsity,
                          float* y_host, void* ws, size_t ws_bytes, void* stream);

/* Bytes of the library's own device scratch used by prox_sparse_ffn_noalloc. */
#define PROX_NOALLOC_SCRATCH_BYTES (8u << 20)

/* prox_sparse_ffn without a workspace, for callers that cannot allocate device memory for
 * one: for example a serving runtime that has already reserved all device memory for its
 * own pool, or a latency-critical loop that cannot afford the implicit synchronization of
 * cudaMalloc. The pages have no counterpart to this call; it only changes where the
 * scratch lives, not what is computed. Arguments are those of prox_sparse_ffn. It runs the
 * CUDA-core Stage-2 kernels (fp32 activations): one token on its own, a batch in token tiles
 * over each tile's union. The result agrees with prox_sparse_ffn (whose single-token Stage 2
 * is the fused kernel's) within the Stage-2 tolerance, not bit for bit.
 *   Scratch: a fixed array of PROX_NOALLOC_SCRATCH_BYTES (8 MiB) inside the library, held
 *   by every GPU that loads the library until the process exits. A call needs
 *   256 + 8*d_ff + SMs * tile * d_model * 4 bytes (rounded to 256-byte pieces), where tile
 *   is the batch's token tile (1 for one token, 2 for two, up to 4 when d_model <= 4096);
 *   with 148 SMs and d_ff up to 53248 that allows: at d_model <= 2048 any batch; at
 *   d_model 4096 a batch of at most 2 tokens (a 3-token or larger batch takes 4-token tiles,
 *   about 9.7 MB); at d_model 8192 a single token. Larger requests return
 *   PROX_ERR_WORKSPACE before anything is launched.
 *   Set-up: the first call on each device looks up the array's device address (with that
 *   device current) and caches it; make that first call before any stream capture.
 *   Sharing: every call on a device uses the same array, and the array keeps the last
 *   call's contents (each call clears what must start at zero). Calls whose work overlaps
 *   on the GPU -- on different streams, or from different threads -- race on it and must
 *   be serialized by the caller.
 *   status_out: if not NULL, the call waits for `stream` and stores the device status
 *   (PROX_OK, PROX_ERR_BOUNDS, PROX_ERR_TIMEOUT) there; if NULL the call stays asynchronous.
 * The call allocates nothing (no cudaMalloc, cudaFree or allocating library routine). */
int prox_sparse_ffn_noalloc(const prox_packed* w, const float* x, int batch, const int32_t* idx,
                            int k, float* y, int* status_out, void* stream);

/* Dense SwiGLU FFN over every channel with the same kernel and weights (the baseline a
 * sparse call is compared with; technical summary, "Problem Statement"). */
int prox_dense_ffn(const prox_packed* w, const float* x, int batch, float* y,
                   void* ws, size_t ws_bytes, void* stream);

/* Unit-gain RMSNorm between stacked layers: x_out = y / sqrt(mean(y^2) + eps), per row.
 * y and x_out are [batch][d_model] fp32 device and may alias. */
int prox_rmsnorm(const float* y, float* x_out, int batch, int d_model, float eps,
                 void* stream);

/* Waits for `stream`, then returns and clears the workspace's device status word:
 * PROX_OK, PROX_ERR_TIMEOUT or PROX_ERR_BOUNDS (or PROX_ERR_CUDA if the wait failed). */
int prox_get_status(void* ws, void* stream);

/* Text for an error code (static storage). */
const char* prox_error_string(int code);

/* The last CUDA failure behind a PROX_ERR_CUDA returned on the calling thread: what the
 * library was doing and the runtime's error name and text ("none" if there was none).
 * Thread-local storage, valid until the thread's next failing call. */
const char* prox_last_cuda_error(void);

/* Number of kernel launches the library has enqueued in this process so far, on any thread
 * and device. A launch recorded into a CUDA graph under stream capture counts once, when it is
 * recorded (graph replays do not call the library). Memory copies and memsets are not kernel
 * launches of the library and are not counted. */
uint64_t prox_launch_count(void);

/* ---- Proxy-memory reduction: a sliding window of device-resident proxies over a layer stack.
 * The pages name sliding-window schemes as the way to cut the ~12% memory the INT4 proxies
 * add (technical summary, "Significance and Claims") and describe none. Reading used here:
 * a decode step visits layers 0, 1, ..., L-1 in order (then 0 again for the next token).
 * Every layer's proxy (the codes and scales Stage 1 reads) lives in pinned host memory and
 * only S slots of proxies live in device memory. Acquiring layer l guarantees that l and the
 * next S-1 layers (cyclically) are resident or being copied; releasing l lets the layer
 * l+S take its slot. Copies run on the window's own stream, ordered by events after the
 * compute that last read a slot and before the compute that reads it. Device memory for
 * proxies drops from L * prox_proxy_bytes to S * prox_proxy_bytes; the price is the
 * host-to-device traffic of one proxy per layer visit whenever S < L. */

/* Bytes of one layer's proxy (codes and scales) and of its Stage-2 rows alone; 0 for an
 * invalid shape or format. */
size_t prox_proxy_bytes(int d_model, int d_ff, int group);
size_t prox_rows_bytes(int d_model, int d_ff, int group, int format);

/* Splits a packed layer (proxy == NULL) into its rows and its proxy: copies the rows to
 * rows_dev (device, PROX_ALIGN-aligned, >= prox_rows_bytes) and the proxy to proxy_out (device
 * or pinned host memory, PROX_ALIGN-aligned, >= prox_proxy_bytes), both enqueued on `stream`.
 * `out` becomes the split descriptor {base = rows_dev, proxy = proxy_out}; it is usable by
 * compute calls while proxy points at device memory holding this layer's proxy (the window
 * sets it on every acquire). The full buffer may be freed once the copies have finished. */
int prox_split_packed(const prox_packed* full, void* rows_dev, size_t rows_bytes,
                      void* proxy_out, size_t proxy_bytes, void* stream, prox_packed* out);

typedef struct prox_window prox_window;   /* opaque; one per layer stack */

/* Creates a window of n_slots device slots over n_layers layers of one shape (group 128).
 *   host_proxies [n_layers]: each layer's proxy as written by prox_split_packed, in pinned
 *       host memory (pageable memory works but the copies then do not overlap compute);
 *   slots_dev: device memory, PROX_ALIGN-aligned, >= n_slots * prox_proxy_bytes bytes.
 * All three stay caller-owned and must outlive the window. The window creates one CUDA
 * stream and 2 * n_slots events on the current device (freed by prox_window_destroy); it
 * allocates no device memory. Not thread-safe: one window is driven from one host thread. */
int prox_window_create(int n_layers, int n_slots, int d_model, int d_ff,
                       const void* const* host_proxies, void* slots_dev, size_t slots_bytes,
                       prox_window** out);

/* Makes layer `layer`'s proxy available to work enqueued on `stream` after this call, and
 * points desc->proxy (a split descriptor of that layer) at its slot. Issues the copies the
 * window needs (this layer if it is not resident, then the following layers into free
 * slots). PROX_ERR_UNSUPPORTED if every slot is held by an acquired, unreleased layer. */
int prox_window_acquire(prox_window* w, int layer, prox_packed* desc, void* stream);

/* Ends layer `layer`'s use of its slot: work enqueued on `stream` so far is its last reader.
 * The slot is then refilled (after that work) with the next layer that enters the window.
 * PROX_ERR_INVALID_ARG if the layer is not acquired. */
int prox_window_release(prox_window* w, int layer, void* stream);

/* Host-to-device copies the window has issued, and their bytes. */
int prox_window_stats(const prox_window* w, uint64_t* copies, uint64_t* bytes);

/* Waits for the window's copies, then frees its stream and events. */
int prox_window_destroy(prox_window* w);

/* Test hook: runs the window's slot policy on the host alone (no CUDA call). ops[i] >= 0
 * acquires layer ops[i], ops[i] < 0 releases layer -1 - ops[i]. slot_out[i]: the slot the
 * op used (-1: acquire found every slot in use, or release of a layer not acquired).
 * copy_log [copy_cap][3]: (op index, slot, layer) of every copy in issue order; n_copies:
 * how many copies were issued (may exceed copy_cap; only copy_cap are logged). */
int prox_debug_window_plan(int n_layers, int n_slots, const int* ops, int n_ops, int* slot_out,
                           int* copy_log, int copy_cap, int* n_copies);

/* Test hook: the same input-selection and Stage-1 kernels as prox_build_mask, also storing
 * the exact integer intermediates (technical summary, Stage 1 "Proxy Activation").
 *   qx_out   [batch][d_model] int8: the activation codes (0 on rejected inputs);
 *   sx_out   [batch][d_model/128] fp32: the activation group scales;
 *   acc_gate, acc_up [batch][d_model/128][d_ff] int32: A[g][j] = sum over kept i in group g
 *            of qx_i * q[j][i] (zeroed by the call, then accumulated);
 *   salience [batch][d_ff] fp32: |SiLU(g~) * u~|.
 * Any of the outputs may be NULL. */
int prox_debug_stage1(const prox_packed* w, const float* x, int batch, double input_sparsity,
                      int8_t* qx_out, float* sx_out, int32_t* acc_gate, int32_t* acc_up,
                      float* salience, void* ws, size_t ws_bytes, void* stream);

/* Test hook for a single-token variant whose Stage-2 kernel selects its channels itself
 * (the top-k folded into Stage 2's front; prox_ffn_forward keeps the separate top-k, which
 * measured faster): runs that variant on x [1][d_model]
 * and also writes every selected channel to sel_out [k] int32 (device): first the channels
 * above the histogram bin of the k-th salience, in ascending order, then the winners inside
 * that bin, in ascending order. PROX_ERR_UNSUPPORTED if the shape or sparsity does not take
 * that path (sparsity 0 is the dense FFN). */
int prox_debug_fused_forward(const prox_packed* w, const float* x, double sparsity,
                             double input_sparsity, float* y, int32_t* sel_out, void* ws,
                             size_t ws_bytes, void* stream);

/* Test hook for the union kernel (the CUDA-core batch path of prox_sparse_ffn_noalloc):
 * the ascending union of the rows of idx [batch][k]
 * (device int32) and, per union entry, a bit mask of the tokens that selected it.
 *   union_out [d_ff] int32, bits_out [d_ff] uint32, count_out [1] int32: device. */
int prox_debug_union(const int32_t* idx, int batch, int k, int d_ff,
                     int32_t* union_out, uint32_t* bits_out, int32_t* count_out,
                     void* ws, size_t ws_bytes, void* stream);

/* Test hook for the bounded waits: launches one block that waits on a barrier nothing ever
 * completes, giving up after about `spin_cycles` SM clock cycles. It then records
 * PROX_ERR_TIMEOUT in the workspace's status word and returns; no GPU fault is involved. */
int prox_debug_wait_timeout(void* ws, size_t ws_bytes, long long spin_cycles, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PROX_H_ */

/*
 * qlora.h -- C ABI of the NF4 + double-quantized LoRA linear layer on B300
 * (sm_103a).
 *
 * What the calls compute (sources are web pages on QLoRA, cited by title and
 * section):
 *  - The frozen base weight W [N out, K in] is stored as 4-bit NormalFloat
 *    codes: 16 levels taken from the quantiles of a standard normal, each bin
 *    holding an equal share of the distribution, with an exact zero
 *    (inquiringlines.com "Can we finetune huge language models on a single
 *    GPU?", mechanism paragraph; ashishsrivastav.com "QLoRA: Fine-Tuning a 70B
 *    on One GPU", section "NF4 Quantization: Beyond Standard INT4"). Each weight
 *    maps to the closest level of its block, once, before training (same
 *    section).
 *  - The per-block scaling constants are themselves quantized to INT8 ("double
 *    quantization"; same page, section "Double Quantization: Squeezing the
 *    Constants"; inquiringlines.com, same paragraph: about 0.37 bit per
 *    parameter saved).
 *  - Dequantization to the bf16 compute type happens on the fly inside the
 *    forward and backward passes (ashishsrivastav.com, same section;
 *    serverroom.net "Fine-tuning an LLM on a GPU: memory requirements for LoRA
 *    and QLoRA", section "What LoRA and QLoRA change in memory": compute dtype
 *    bf16).
 *  - Gradients flow through the frozen 4-bit weights into low-rank adapters A
 *    [r, K] and B [N, r]; only the adapters get gradients
 *    (inquiringlines.com, same paragraph; xingyuzhitong.com "Fine-Tuning Memory
 *    Requirements: Full Training vs LoRA vs QLoRA", sections "LoRA: freeze the
 *    base, train small adapters" and "QLoRA: quantize the frozen base to 4
 *    bits"). Adapter dropout is 0 and there is no bias (serverroom.net, adapter
 *    setup listing).
 *
 * Fixed format (readings where the pages are silent):
 *  - blocks of 64 consecutive weights in row-major order (cols % 64 == 0), so
 *    a block never crosses a row;
 *  - codes: byte i holds element 2i in its high nibble, element 2i+1 in its
 *    low nibble;
 *  - absmax_q: one int8 per block, symmetric, in [-127, 127];
 *  - absmax_scale: one fp32 per group of 256 consecutive blocks (the last
 *    group may be partial);
 *  - absmax_mean: one fp32 for the whole tensor, subtracted before the int8
 *    step;
 *  - reconstructed absmax a' = fp32(q) * scale + mean (two rounded fp32
 *    operations, no fused multiply-add); dequantized weight
 *    w' = bf16_rne(fp32(L[code] * a')).
 *  - LoRA: Y = X W'^T + s (X A^T) B^T with s = alpha / r passed as `scale`.
 *
 * Conventions for every call:
 *  - All tensors are row-major and contiguous; bf16 tensors are passed as
 *    void pointers to 2-byte elements.
 *  - Pointers are DEVICE pointers unless a comment says otherwise. The caller
 *    owns every buffer; the library never allocates, frees or synchronizes,
 *    and enqueues all work on `stream` (a cudaStream_t; NULL = legacy default
 *    stream).
 *  - Every argument is validated on the host before anything is launched. On
 *    an error, nothing is launched, outputs are untouched, the status is
 *    returned and qlora_last_error() describes it.
 *  - A launch failure returns QLORA_ERR_CUDA. Faults inside kernels surface at
 *    the caller's next synchronization. Pipelined kernels bound every wait;
 *    a wait that runs out sets a device error word, which
 *    qlora_check_device_status() reports as QLORA_ERR_TIMEOUT.
 *  - The calls keep no state between calls and may run concurrently on
 *    different streams when their buffers do not overlap. No kernel waits
 *    for a thread block that may not be resident: work shared between thread
 *    blocks outside a cluster is finished by whichever contributor arrives
 *    last, so concurrent calls progress however the GPU divides its SMs.
 *  - Alignment: every device pointer must be 16-byte aligned.
 */
#ifndef QLORA_B300_H
#define QLORA_B300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *qlora_stream_t; /* same type as cudaStream_t */

typedef enum {
    QLORA_OK = 0,
    QLORA_ERR_NULL = 1,        /* a required pointer is NULL */
    QLORA_ERR_SHAPE = 2,       /* a size is out of range (e.g. cols % 64 != 0, M < 0) */
    QLORA_ERR_ALIGN = 3,       /* a device pointer is not 16-byte aligned */
    QLORA_ERR_WORKSPACE = 4,   /* workspace smaller than the size query returns */
    QLORA_ERR_RANK = 5,        /* LoRA rank outside [1, 128] */
    QLORA_ERR_CUDA = 6,        /* a CUDA runtime call or launch failed */
    QLORA_ERR_TIMEOUT = 7,     /* a bounded wait inside a kernel ran out */
    QLORA_ERR_UNSUPPORTED = 8  /* device is not sm_103 / needed driver entry point missing */
} qlora_status;

/* A quantized weight: all pointers are device pointers owned by the caller. */
typedef struct {
    int64_t rows;           /* N: output features */
    int64_t cols;           /* K: input features, cols % 64 == 0 */
    uint8_t *codes;         /* rows*cols/2 bytes, layout above */
    int8_t *absmax_q;       /* nb = rows*cols/64 int8 codes */
    float *absmax_scale;    /* ng = ceil(nb/256) fp32 scales */
    float *absmax_mean;     /* 1 fp32 */
} qlora_nf4_weight;

/* Storage variants of the 4-bit weight (the same kernels decode all four):
 *  - table: QLORA_TABLE_NF4, the NormalFloat levels above, or
 *    QLORA_TABLE_INT4, the INT4 baseline the NF4 levels are compared against
 *    (ashishsrivastav.com, section "NF4 Quantization: Beyond Standard INT4":
 *    16 evenly spaced levels). Reading: symmetric absmax INT4, level i is
 *    (i - 7) / 7 rounded to fp32 (code 7 the exact zero, codes 0 and 14 are
 *    -1 and +1, code 15 is never chosen), nearest level with ties to the lower
 *    code as for NF4;
 *  - double_quant: 1 keeps the absmax double-quantized (absmax_q,
 *    absmax_scale, absmax_mean, as qlora_nf4_weight); 0 keeps it as one fp32
 *    per block in `absmax` (4.5 bits per weight: xingyuzhitong.com, section
 *    "QLoRA: quantize the frozen base to 4 bits"), a' = absmax as stored.
 * Arrays not used by the variant may be NULL. All pointers are device
 * pointers owned by the caller, 16-byte aligned. */
#define QLORA_TABLE_NF4 0
#define QLORA_TABLE_INT4 1
typedef struct {
    int64_t rows;           /* N */
    int64_t cols;           /* K, cols % 64 == 0 */
    int32_t table;          /* QLORA_TABLE_NF4 or QLORA_TABLE_INT4 */
    int32_t double_quant;   /* 1: absmax_q/absmax_scale/absmax_mean; 0: absmax */
    uint8_t *codes;         /* rows*cols/2 bytes */
    int8_t *absmax_q;       /* double_quant: nb int8 codes */
    float *absmax_scale;    /* double_quant: ceil(nb/256) fp32 */
    float *absmax_mean;     /* double_quant: 1 fp32 */
    float *absmax;          /* !double_quant: nb fp32 */
} qlora_q4_weight;

/* ---- sizes (host-only, no GPU needed) --------------------------------- */

/* Bytes of packed codes: rows*cols/2. Returns 0 for invalid sizes. */
size_t qlora_nf4_codes_bytes(int64_t rows, int64_t cols);
/* Number of blocks (int8 absmax codes): rows*cols/64. */
size_t qlora_nf4_absmax_count(int64_t rows, int64_t cols);
/* Number of fp32 second-level scales: ceil(blocks / 256). */
size_t qlora_nf4_scale_count(int64_t rows, int64_t cols);
/* Total bytes of one quantized weight (codes + int8 codes + scales + mean),
 * each array padded to 16 bytes as the library requires. */
size_t qlora_nf4_storage_bytes(int64_t rows, int64_t cols);
/* Workspace bytes qlora_nf4_quantize needs. */
size_t qlora_nf4_quantize_workspace(int64_t rows, int64_t cols);

/* Host copy of the 16 fp32 NF4 levels the kernels use (ascending; code 7 is
 * the exact zero). */
void qlora_nf4_table(float levels[16]);

/* Host copy of the 16 fp32 levels of a table (QLORA_TABLE_NF4 or
 * QLORA_TABLE_INT4); all zero for an unknown table. */
void qlora_q4_table(int table, float levels[16]);

/* ---- codec ------------------------------------------------------------- */

/* Quantizes a bf16 weight W [rows, cols] (device) into `out`, whose rows/cols
 * must be set and whose arrays must be allocated (sizes above). Encodes each
 * block of 64 with its exact absmax (nearest level, ties to the lower code),
 * then double-quantizes the absmax: mean = fp32(S / nb) with S the pairwise
 * (balanced binary tree, zero-padded to a power of two, leaves in block
 * order) fp64 sum of the absmax values; per group g of 256 blocks,
 * c = fp32(a - mean), scale_g = fp32(max|c| / 127), q = clamp(rint(fp32(c /
 * scale_g)), -127, 127) (q = 0 when scale_g == 0). Inputs must be finite.
 * `ws` is a device workspace of at least qlora_nf4_quantize_workspace bytes.
 * Sources: ashishsrivastav.com, sections "NF4 Quantization" and "Double
 * Quantization"; inquiringlines.com, mechanism paragraph. */
qlora_status qlora_nf4_quantize(const void *W, qlora_nf4_weight *out, void *ws, size_t ws_bytes,
                                qlora_stream_t stream);

/* Quantizes like qlora_nf4_quantize, bit for bit, but takes no workspace and
 * allocates nothing. The pages have no counterpart: this is an interface
 * variant for callers that cannot allocate device memory, for example a
 * plugin inside a host application or framework that owns every device
 * buffer through its own pool and hands the plugin only its inputs and
 * outputs, or code that must not trigger cudaMalloc's implicit device
 * synchronization (or its failure under fragmentation) mid-run.
 *  - Scratch comes from one array of QLORA_NF4_NOALLOC_SCRATCH_BYTES compiled
 *    into the library; every GPU that loads the library holds it until the
 *    process exits. A weight whose quantize workspace
 *    (qlora_nf4_quantize_workspace) exceeds that size is rejected with
 *    QLORA_ERR_WORKSPACE and nothing is launched (16 MiB covers about
 *    2.6e8 weights, e.g. 28672 x 8192).
 *  - The first call in each CUDA context (on each device, with that device
 *    current) looks up the array's device address once and caches it for
 *    that context; make that first call before any stream capture.
 *  - All calls share the one array, which keeps the last call's contents;
 *    nothing in it needs to start at zero. Calls that can overlap on the GPU
 *    (different streams without ordering between them) race on it: order
 *    them.
 *  - The caller still passes W and allocates `out`'s arrays as for
 *    qlora_nf4_quantize. */
#define QLORA_NF4_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)
qlora_status qlora_nf4_quantize_noalloc(const void *W, qlora_nf4_weight *out, qlora_stream_t stream);

/* Writes the dequantized bf16 weight W' [rows, cols] (device) to `out`:
 * w' = bf16_rne(fp32(L[code] * a')) with a' = fp32(q)*scale + mean.
 * Source: ashishsrivastav.com, section "Double Quantization" (dequantize on
 * the fly to the compute type). */
qlora_status qlora_nf4_dequantize(const qlora_nf4_weight *w, void *out, qlora_stream_t stream);

/* ---- deployment: merge the adapter, quantize again ---------------------- */

/* Workspace bytes of qlora_lora_merge_requantize for a [rows, cols] weight
 * (the merged bf16 weight plus the quantizer's workspace). */
size_t qlora_lora_merge_workspace(int64_t rows, int64_t cols);

/* Folds the adapter into the base weight and quantizes the result:
 *   merged[n, k] = bf16_rne( w'[n, k] + scale * t[n, k] ),
 *   t[n, k] = sum over j = 0 .. r-1 of B[n, j] * A[j, k],
 * every step a separately rounded fp32 operation in that order (t starts at
 * 0; no fused multiply-add), w' the dequantized base weight; then `out` gets
 * the NF4 + double-quantized form of `merged`, exactly as qlora_nf4_quantize
 * would produce it. A [r, K] and B [N, r] are bf16 (1 <= r <= 128); `out`
 * has the same shape as `w` and may be `w` itself (in-place requantization:
 * the merge reads `w` before the quantizer writes `out`). `ws` is a device
 * workspace of qlora_lora_merge_workspace bytes; the merged bf16 weight is
 * its first rows * cols * 2 bytes after the call.
 * Source: xingyuzhitong.com "Fine-Tuning Memory Requirements", section
 * "Choosing a method" (adapters merged into the base weights for
 * deployment). */
qlora_status qlora_lora_merge_requantize(const qlora_nf4_weight *w, const void *A, const void *B, int r,
                                         float scale, qlora_nf4_weight *out, void *ws, size_t ws_bytes,
                                         qlora_stream_t stream);

/* The storage variants (qlora_q4_weight): quantize, dequantize, forward and
 * backward exactly as the qlora_nf4_* / qlora_linear_* calls, which are these
 * calls with table = QLORA_TABLE_NF4 and double_quant = 1. Without double
 * quantization the quantizer writes the exact block absmax to `absmax` and
 * needs no workspace (ws may be NULL, ws_bytes 0); with it, the workspace is
 * qlora_nf4_quantize_workspace bytes. The linear workspaces are the same as
 * for qlora_linear_fwd / qlora_linear_bwd. */
qlora_status qlora_q4_quantize(const void *W, qlora_q4_weight *out, void *ws, size_t ws_bytes, qlora_stream_t stream);
qlora_status qlora_q4_dequantize(const qlora_q4_weight *w, void *out, qlora_stream_t stream);
size_t qlora_q4_linear_fwd_workspace(int64_t M, const qlora_q4_weight *w, int r);
size_t qlora_q4_linear_bwd_workspace(int64_t M, const qlora_q4_weight *w, int r);
qlora_status qlora_q4_linear_fwd(const void *X, int64_t M, const qlora_q4_weight *w, const void *A, const void *B,
                                 int r, float scale, void *Y, void *U_save, void *ws, size_t ws_bytes,
                                 qlora_stream_t stream);
qlora_status qlora_q4_linear_bwd(const void *dY, const void *X, const void *U_saved, int64_t M,
                                 const qlora_q4_weight *w, const void *A, const void *B, int r, float scale, void *dX,
                                 float *dA, float *dB, void *ws, size_t ws_bytes, qlora_stream_t stream);

/* ---- linear layer with LoRA ------------------------------------------- */

/* Workspace bytes for qlora_linear_fwd / qlora_linear_bwd at these sizes. */
size_t qlora_linear_fwd_workspace(int64_t M, const qlora_nf4_weight *w, int r);
size_t qlora_linear_bwd_workspace(int64_t M, const qlora_nf4_weight *w, int r);

/* Forward:  Y = X W'^T + scale * (X A^T) B^T.
 *   X      bf16 [M, K]        input activations (K = w->cols)
 *   w      quantized W [N, K] (N = w->rows)
 *   A      bf16 [r, K]        LoRA down-projection
 *   B      bf16 [N, r]        LoRA up-projection
 *   scale  LoRA scale s (alpha / r)
 *   Y      bf16 [M, N]        output (overwritten)
 *   U_save bf16 [M, r] or NULL: receives U = X A^T (rounded to bf16) for the
 *          backward pass
 *   ws     device workspace of qlora_linear_fwd_workspace bytes
 * M may be 0 (nothing is launched). 1 <= r <= 128.
 * Accumulation is fp32 over bf16 operands; the LoRA term enters as extra
 * contraction steps over (s*U rounded to bf16) and B. */
qlora_status qlora_linear_fwd(const void *X, int64_t M, const qlora_nf4_weight *w, const void *A,
                              const void *B, int r, float scale, void *Y, void *U_save, void *ws,
                              size_t ws_bytes, qlora_stream_t stream);

/* Backward (no gradient for the frozen W):
 *   V  = dY B                                    [M, r]
 *   dX = dY W' + scale * V A                     bf16 [M, K]  (overwritten)
 *   dB = scale * dY^T U                          fp32 [N, r]  (overwritten)
 *   dA = scale * V^T X                           fp32 [r, K]  (overwritten)
 *   dY bf16 [M, N]; X bf16 [M, K]; U_saved bf16 [M, r] from the forward, or
 *   NULL to recompute U = X A^T. dA and dB are complete sums over the M rows
 *   given (a data-parallel caller all-reduces them across replicas). */
qlora_status qlora_linear_bwd(const void *dY, const void *X, const void *U_saved, int64_t M,
                              const qlora_nf4_weight *w, const void *A, const void *B, int r,
                              float scale, void *dX, float *dA, float *dB, void *ws,
                              size_t ws_bytes, qlora_stream_t stream);

/* ---- projection groups: several layers that share their input ---------- */

/* A group is 1..QLORA_MAX_GROUP LoRA linear layers that read the same X
 * [M, K] with their own weights: the attention's q, k and v projections, or
 * the MLP's gate and up projections (xingyuzhitong.com "Fine-Tuning Memory
 * Requirements", section "LoRA: freeze the base, train small adapters", and
 * serverroom.net, section "Setting up Unsloth on the server": adapters on
 * q/k/v/o/gate/up/down). One grouped call computes, for every projection g,
 *   Y_g = X W_g'^T + scale * (X A_g^T) B_g^T
 * and the backward the adapter gradients of every projection and
 *   dX = sum_g ( dY_g W_g' + scale * (dY_g B_g) A_g )     bf16 [M, K]
 * (the gradient of the shared input). The arithmetic per projection is the
 * single-layer calls' (the same results up to fp32 summation order); the
 * group runs as one fused GEMM launch over all projections' output columns
 * (forward) or over all their rows (dX), one LoRA down-projection over the
 * stacked A_g, and reads X once per pass instead of once per projection.
 * With few tokens (M <= 16, K a multiple of 256) the forward is one
 * weight-streaming launch over all projections' rows; smaller backwards run
 * projection by projection.
 * Requirements: every weight has the same cols K; one rank r for all,
 * r % 8 == 0 and 8 <= r <= 128; one scale. All pointers are device
 * pointers, 16-byte aligned, owned by the caller. A QLORA_ERR_* status is
 * returned before anything is launched when a requirement fails. */
#define QLORA_MAX_GROUP 4
typedef struct {
    const qlora_nf4_weight *w; /* W_g [N_g, K] */
    const void *A;             /* bf16 [r, K] */
    const void *B;             /* bf16 [N_g, r] */
    void *Y;                   /* forward: bf16 [M, N_g] output (overwritten) */
    const void *dY;            /* backward: bf16 [M, N_g] */
    float *dA;                 /* backward: fp32 [r, K] output (overwritten) */
    float *dB;                 /* backward: fp32 [N_g, r] output (overwritten) */
} qlora_proj;

/* Workspace bytes of qlora_group_fwd / qlora_group_bwd for these sizes
 * (0 for invalid arguments). */
size_t qlora_group_fwd_workspace(int64_t M, const qlora_proj *proj, int n, int r);
size_t qlora_group_bwd_workspace(int64_t M, const qlora_proj *proj, int n, int r);

/* Forward of n projections (fields w, A, B, Y of each are used).
 * U_save: bf16 [M, n * r] or NULL; receives U_g = X A_g^T (bf16) in columns
 * [g * r, (g + 1) * r), the layout qlora_group_bwd reads. */
qlora_status qlora_group_fwd(const void *X, int64_t M, const qlora_proj *proj, int n, int r, float scale,
                             void *U_save, void *ws, size_t ws_bytes, qlora_stream_t stream);

/* Backward of n projections (fields w, A, B, dY, dA, dB of each are used):
 * dA_g, dB_g as qlora_linear_bwd computes them for projection g, and dX
 * above. U_saved: the forward's U_save [M, n * r], or NULL to recompute. */
qlora_status qlora_group_bwd(const void *X, const void *U_saved, int64_t M, const qlora_proj *proj, int n, int r,
                             float scale, void *dX, void *ws, size_t ws_bytes, qlora_stream_t stream);

/* ---- optimizer step for the adapters ----------------------------------- */

/* One AdamW step on n fp32 parameters (the flattened adapter A or B master
 * weights), with decoupled weight decay, in this order:
 *   p = p * (1 - lr * weight_decay)
 *   m = beta1 * m + (1 - beta1) * g ;  v = beta2 * v + (1 - beta2) * g^2
 *   p = p - (lr / (1 - beta1^step)) * m / (sqrt(v) / sqrt(1 - beta2^step) + eps)
 * computed in fp32 (the bias corrections in fp64 on the host). `grad` is the
 * fp32 gradient qlora_linear_bwd wrote (dA or dB); `param_bf16`, if not NULL,
 * receives bf16_rne(p), the adapter the next qlora_linear_fwd reads.
 * "Paged" optimizer state: param, m and v may be device memory, managed
 * memory (the driver pages it between host and device) or pinned host
 * memory (read and written over the interconnect); pointers the device
 * cannot reach (pageable host memory) are rejected with
 * QLORA_ERR_UNSUPPORTED before anything is launched. step >= 1 counts the
 * steps taken so far including this one. param, grad, m and v must be
 * 16-byte aligned, param_bf16 8-byte aligned.
 * Sources: inquiringlines.com note, mechanism paragraph (paged optimizers);
 * ashishsrivastav.com, section "Paged Optimizers: Managing Fragmentation";
 * addaly.com lesson "Fitting a fine-tune in 16 GB" (paged AdamW). The rule
 * itself is the standard decoupled-decay AdamW the pages name but do not
 * write out. */
qlora_status qlora_adamw_step(float *param, uint16_t *param_bf16, const float *grad, float *m, float *v, int64_t n,
                              float lr, float beta1, float beta2, float eps, float weight_decay, int64_t step,
                              qlora_stream_t stream);

/* ---- diagnostics ------------------------------------------------------- */

/* Message for the last error on the calling thread ("" if none). */
const char *qlora_last_error(void);

/* Synchronizes `stream`, then reads and clears the device error word set by
 * bounded waits that ran out. Returns QLORA_OK, QLORA_ERR_TIMEOUT (message
 * names the kernel and wait) or QLORA_ERR_CUDA. */
qlora_status qlora_check_device_status(qlora_stream_t stream);

/* Test hook: sets the time limit, in microseconds, of the bounded pipeline
 * waits in the kernels (0 or less restores the default of 2 s). A limit of 1
 * makes a wait that is not satisfied within about 1 us (plus the hardware's
 * own suspend interval, up to about 80 us) run out. The kernels' waits for
 * their own copies and tensor-core work before they exit are not affected.
 * Host-side setting, applies to later launches on all streams. */
void qlora_set_wait_limit(int64_t microseconds);

/* Profiling of the library's own kernels, for benchmarks. Between
 * qlora_profile_start() and qlora_profile_stop(), every kernel launch is
 * counted by kind and bracketed by a pair of CUDA events recorded on its
 * launch stream (the library creates and destroys these events; nothing else
 * changes). qlora_profile_stop() waits for the recorded events and fills, per
 * kind, the summed device time in ms and the number of launches; it returns
 * the total number of launches, or -1 on a CUDA error. Not thread-safe: one
 * profiling session at a time. */
enum {
    QLORA_KERNEL_QUANTIZE = 0,   /* encode + tree sum + double quantization */
    QLORA_KERNEL_DEQUANT = 1,    /* standalone dequantize */
    QLORA_KERNEL_LORA_PRE = 2,   /* U = X A^T, V = dY B, B^T */
    QLORA_KERNEL_FWD_GEMM = 3,   /* fused dequant + tcgen05 forward GEMM */
    QLORA_KERNEL_FWD_SIMT = 4,   /* small-M / CUDA-core forward */
    QLORA_KERNEL_DX_GEMM = 5,    /* fused dequant + tcgen05 dX GEMM */
    QLORA_KERNEL_DX_SIMT = 6,    /* small-M / CUDA-core dX */
    QLORA_KERNEL_GRADS = 7,      /* dA, dB reductions */
    QLORA_KERNEL_OPTIM = 8,      /* AdamW step of the adapters */
    QLORA_KERNEL_KINDS = 9
};
void qlora_profile_start(void);
int qlora_profile_stop(double ms_per_kind[QLORA_KERNEL_KINDS], int launches_per_kind[QLORA_KERNEL_KINDS]);

/* Library version string. */
const char *qlora_version(void);

/* Diagnostic, host only (no device access): the work schedule the fused
 * tensor-core GEMM would run for an output of M rows and Nd columns with
 * nk_main main 64-deep k-steps and lora_steps LoRA k-steps (forward: Nd = N,
 * nk_main = K / 64; dX: Nd = K, nk_main = ceil(N / 64); lora_steps =
 * ceil(r / 64)) on a device holding `pairs_resident` (1..74) CTA pairs at
 * once. Writes to out[0..3] the tile height in rows (512 or 256), the number
 * of tiles run data-parallel, the pairs launched and the number of tiles T;
 * then one record of 9 values per segment, pair by pair in the order each pair
 * runs them: pair, tile, first output row, first output column, first k-step,
 * k-steps, role (0 whole tile, 1 head: the tile's first k-steps, 2 tail: a
 * later part of the tile), the tile's head pair h and its number of
 * contributors n (pairs h .. h + n - 1; h = pair and n = 1 for a whole tile).
 * Of a shared tile's contributors, whichever arrives last adds the others'
 * fp32 partials and writes the output. Returns the number of records, -1
 * when `cap` (values available in out) is too small, -2 for invalid
 * arguments.
 * Tiles are 256 output columns wide; a tile's k-steps are the main steps then
 * the LoRA steps. */
int64_t qlora_debug_gemm_segments(int64_t M, int64_t Nd, int64_t nk_main, int lora_steps, int pairs_resident,
                                  int64_t *out, int64_t cap);

/* Diagnostic, host only (no device access): the split the few-token forward
 * (M <= 16, K a multiple of 256) uses for M tokens and an N x K weight. Tasks
 * of 32 rows x 256 k are numbered row tile by row tile (tile t holds tasks t P
 * .. t P + P - 1, P = K / 256) and split evenly over W warps (16 per CTA for
 * M <= 8, 12 for M > 8, at most 148 CTAs). Writes out[0..3] = T tasks,
 * W warps, P, row tiles; then each warp's first task and one past its last
 * (2 W values); then each row tile's first and last contributing warp (2 x
 * tiles values). A tile whose two warps are equal is finished by that warp;
 * otherwise the last of its warps to arrive finishes it. Returns the number of
 * values written, -1 when `cap` is too small, -2 for invalid arguments. */
int64_t qlora_debug_few_split(int64_t M, int64_t N, int64_t K, int64_t *out, int64_t cap);

#ifdef __cplusplus
}
#endif
#endif /* QLORA_B300_H */

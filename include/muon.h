/*
 * muon.h -- C ABI of a batched Muon optimizer step for one GB300 (sm_103a).
 *
 * One call of muon_step() runs, for every matrix of a ragged batch and on one
 * CUDA stream:
 *
 *   1. M <- beta*M + G                       one fp32 momentum state per
 *      parameter ("Training a 1T-Params MoE on EU public infrastructure",
 *      tanhow.com, optimizer-state paragraph); or beta*M + (1 - beta)*G with
 *      the `dampening` variant;
 *   2. X = M (rows <= cols) or M^T (rows > cols), so that A = X X^T is the
 *      smaller Gram matrix;  X <- X / (||X||_F + eps);
 *   3. `ns_iters` Newton-Schulz iterations (5 per step: "ZAYA1 MoE training on
 *      MI300X", hotelren.com/news/3048137, section 4.3), each
 *        A  = X X^T          upper-triangle tiles only, mirrored
 *        A2 = A A^T = A A    the same symmetric kernel reused
 *        X <- a X + b A X + c A2 X
 *      ("AMD GPU深度学习优化与ZAYA1大模型实践", jsqmd.com/news/1098463,
 *      section 4.2 内存高效Muon优化器), computed as X <- a X + (b A + c A2) X;
 *   4. W <- W - lr * scale_coeff * sqrt(max(rows, cols)) * O, O = X oriented
 *      back to rows x cols (hotelren.com, section 4.3: lr scale
 *      0.2 x sqrt(max(a, b))).
 *
 * Matrices are independent: a matrix's results do not depend on the other
 * matrices of the batch or on their order (whole-matrix ownership as in the
 * FlexShard paragraph of tanhow.com).
 *
 * Memory.  W, G, M, O_out and the workspace are device memory owned by the
 * caller; the library never allocates or frees device memory.  A handle owns
 * host-side state only (configuration, error text, profiling events).
 *
 * Streams.  muon_step() is asynchronous on `stream` (a cudaStream_t passed as
 * void*, NULL = the legacy default stream) and never synchronises the host.
 * W, G, M and the workspace must stay alive until the stream has passed the
 * step.  A handle is not thread-safe; use one handle per host thread.
 *
 * Errors.  Every descriptor is validated before anything is launched; on an
 * error nothing is launched and W, M are untouched.  Non-finite values in G or
 * M are not errors: they propagate to that matrix's W and M only.
 */
#ifndef MUON_GB300_H
#define MUON_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct muon_handle_s* muon_handle;

typedef enum {
    MUON_OK = 0,
    MUON_ERR_INVALID_ARG = 1,   /* a NULL pointer, a bad size, stride or alignment, aliasing */
    MUON_ERR_UNSUPPORTED = 2,   /* device is not sm_103, handle has no device, unknown mode */
    MUON_ERR_WORKSPACE = 3,     /* workspace NULL, misaligned (256 B) or smaller than required */
    MUON_ERR_CUDA = 4,          /* a CUDA runtime call failed; text in muon_last_error_message */
    MUON_ERR_TIMEOUT = 5        /* a kernel gave up a bounded wait (reported by muon_check_status) */
} muon_status;

typedef enum { MUON_F32 = 0, MUON_BF16 = 1 } muon_dtype;

typedef enum {
    /* bf16 tensor-core operands, fp32 accumulation; X kept as the bf16 pair
       hi = bf16(x), lo = bf16(x - hi); A and (bA + cA^2) stored bf16 with
       their diagonals in fp32 */
    MUON_MODE_BF16 = 0,
    /* fp32 operands on the CUDA cores throughout: the validation mode */
    MUON_MODE_FP32_VALIDATE = 1
} muon_mode;

typedef struct {
    float beta;         /* momentum factor, default 0.95 */
    float a, b, c;      /* Newton-Schulz coefficients, default 3.4445, -4.7750, 2.0315 */
    float eps;          /* added to ||X||_F, default 1e-7 */
    float scale_coeff;  /* update scale coefficient, default 0.2 */
    int32_t ns_iters;   /* Newton-Schulz iterations, 0..64, default 5 */
    int32_t nesterov;   /* 0: NS input is the new momentum; 1: G + beta * (new momentum) */
    int32_t mode;       /* muon_mode, default MUON_MODE_BF16 */
    int32_t dampening;  /* 0 (default): M <- beta*M + G; 1: M <- beta*M + (1 - beta)*G, the
                           moving-average form, and the Nesterov input (1 - beta)*G + beta*M.
                           The pages fix neither form; the second is a variant. */
} muon_config;

/* One whole weight matrix, rows x cols, every buffer row-major with its own
 * leading dimension (elements).  Pointers are device pointers, 16-byte
 * aligned; ld * element size must be a multiple of 16 bytes; ld >= cols.
 * W, G, M and O_out must not overlap.  rows == 0 or cols == 0 is a valid
 * empty matrix that is skipped (its pointers may be NULL). */
typedef struct {
    int64_t rows, cols;
    void* W;              /* in/out weights, dtype w_dtype */
    int32_t w_dtype;      /* muon_dtype */
    int32_t reserved0;
    int64_t ldw;
    const float* G;       /* in: fp32 gradient */
    int64_t ldg;
    float* M;             /* in/out: fp32 momentum */
    int64_t ldm;
    float lr;             /* learning rate of this matrix */
    int32_t reserved1;
    float* O_out;         /* optional out: fp32 O (rows x cols), or NULL */
    int64_t ldo;
} muon_matrix_desc;

/* Per-phase device time, summed over the steps recorded since profiling was
 * enabled or last read.  Phases: 0 momentum+norm, 1 Gram X X^T, 2 Gram A A
 * with the b/c combine, 3 GEMM with the a X epilogue, 4 apply. */
#define MUON_NUM_PHASES 5
typedef struct {
    double ms[MUON_NUM_PHASES];
    int64_t launches[MUON_NUM_PHASES];
    int64_t steps;
} muon_phase_stats;

/* Fills the defaults listed above. */
void muon_config_default(muon_config* cfg);

/* Creates a handle for CUDA device `device` (must be sm_103 or newer), or a
 * host-only planning handle when device == -1 (muon_workspace_size and
 * argument validation work; muon_step returns MUON_ERR_UNSUPPORTED after
 * validating).  cfg NULL means defaults.  Allocates no device memory. */
muon_status muon_create(const muon_config* cfg, int device, muon_handle* out);

/* Bytes of workspace muon_step() needs for this batch (validates the
 * descriptors; n == 0 gives 0). */
muon_status muon_workspace_size(muon_handle h, const muon_matrix_desc* descs, int n, size_t* bytes);

/* One Muon step over `n` matrices.  `ws` is device memory of at least
 * muon_workspace_size() bytes, 256-byte aligned, that overlaps none of the
 * descriptors' buffers (MUON_ERR_INVALID_ARG otherwise), used only by this
 * call while it runs on `stream` (its contents need not be preserved between
 * calls).  n == 0 launches nothing and returns MUON_OK.
 *
 * The handle keeps the plans of its most recent batches (up to 32): a call
 * whose descriptor array is byte-for-byte one seen before, with the same
 * workspace pointer, skips validation and planning and launches the kernels
 * with the parameter blocks and TMA tensor maps built then (they depend on
 * nothing else: the configuration is fixed per handle). */
muon_status muon_step(muon_handle h, const muon_matrix_desc* descs, int n,
                      void* ws, size_t ws_bytes, void* stream);

/* Synchronises `stream`, then reads and clears the kernels' status word in
 * `ws`: MUON_ERR_TIMEOUT if a kernel of an earlier step gave up a bounded
 * wait, else MUON_OK (or MUON_ERR_CUDA if the stream reports an error).
 * ws == NULL reads and clears the status word of muon_step_noalloc's fixed
 * array on the handle's device; the workspace of the handle's most recent
 * muon_step_host call holds one status word per staging slot, and all of them
 * are read and cleared.  A step whose wait timed out leaves W unchanged when
 * the time-out happened before its last kernel started. */
muon_status muon_check_status(muon_handle h, void* ws, void* stream);

muon_status muon_destroy(muon_handle h);

const char* muon_status_string(muon_status s);

/* Text of the last error seen by this handle ("" if none). */
const char* muon_last_error_message(muon_handle h);

/* Enables (1) or disables (0) per-phase CUDA-event timing on the launching
 * stream.  Events are recorded around the phases of each step; at most 1024
 * steps are kept until read. */
muon_status muon_set_profiling(muon_handle h, int enable);

/* Waits for the recorded events and returns the per-phase sums; resets them. */
muon_status muon_read_profile(muon_handle h, muon_phase_stats* out);

/* Number of kernel launches this handle has issued since it was created. */
int64_t muon_launch_count(muon_handle h);

/* Number of step plans this handle has built (validation, tile lists, tensor
 * maps); a batch repeated with the same descriptors and workspace reuses its
 * plan and does not add to it. */
int64_t muon_plan_builds(muon_handle h);

/* Number of steps this handle has run as a CUDA-graph replay.  A cached
 * plan's first step launches its kernels one by one; from its second step on
 * the handle replays them as a graph it captured once (one launch call instead
 * of about 17), unless profiling is enabled or the caller's stream is being
 * captured, when the kernels are launched one by one. */
int64_t muon_graph_launches(muon_handle h);

/* ---- Steps on buffers in host memory ------------------------------------
 *
 * The optimizer state may live in host memory when HBM is short: the pages
 * keep activations in Grace memory and move them over NVLink-C2C ("Training a
 * 1T-Params MoE on EU public infrastructure", tanhow.com, activation-offload
 * paragraph).  muon_step_host runs the step on descriptors whose W, G, M or
 * O_out (as selected by `host_buffers`) are host pointers: it copies chunks
 * of whole matrices into device staging slots, runs muon_step on each chunk
 * and copies W, M and O_out back, with the copies of one chunk overlapping
 * the step of another (a copy-in, a step and a copy-out stream owned by the
 * handle, ordered by events; one cudaMemcpy2DAsync per buffer).  Buffers not
 * selected are device pointers, used in place.  The results equal
 * muon_step's on the same values bit for bit. */
#define MUON_HOST_W 1
#define MUON_HOST_G 2
#define MUON_HOST_M 4
#define MUON_HOST_O 8

typedef struct {
    int32_t host_buffers;     /* MUON_HOST_* bits: which buffers are host pointers */
    int32_t chunk_matrices;   /* matrices per chunk (>= 1) */
    int32_t slots;            /* device staging slots in the ring (>= 2) */
    int32_t reserved;         /* 0 */
} muon_host_pipeline;

/* Bytes of device workspace muon_step_host needs for this batch and pipeline:
 * `slots` staging slots, each holding one chunk's host-resident buffers and
 * the workspace of its muon_step. */
muon_status muon_host_workspace_size(muon_handle h, const muon_matrix_desc* descs, int n,
                                     const muon_host_pipeline* pl, size_t* bytes);

/* One Muon step over `n` matrices whose selected buffers are in host memory.
 * Host buffers should be page-locked (cudaHostAlloc / cudaHostRegister) for
 * the copies to be asynchronous; they, and the device workspace `ws` (at
 * least muon_host_workspace_size() bytes, 256-byte aligned), must stay alive
 * and untouched until `stream` has passed the step: the call only enqueues
 * work.  The handle's copy and step streams wait for the work already on
 * `stream`, and `stream` waits for their last copy.  Errors as muon_step; a
 * descriptor error launches and copies nothing; a launch error part-way
 * returns MUON_ERR_CUDA with copies of earlier chunks possibly still in flight
 * on the handle's streams (synchronise the device before reusing the host
 * buffers).  muon_check_status(h, ws, stream) reads the status words of every
 * chunk's step. */
muon_status muon_step_host(muon_handle h, const muon_matrix_desc* descs, int n,
                           const muon_host_pipeline* pl, void* ws, size_t ws_bytes, void* stream);

/* Size of the fixed device workspace that muon_step_noalloc uses. */
#define MUON_STATIC_WORKSPACE_BYTES (64u * 1024u * 1024u)

/* muon_step without a caller-provided workspace, for callers that may not
 * allocate device memory (a runtime that reserves all memory at start-up and
 * forbids later cudaMalloc, or a plugin confined to a host framework's
 * tensors).  The pages describe no such entry point; it exists only for
 * those callers.
 *
 * The scratch space is one fixed __device__ array of
 * MUON_STATIC_WORKSPACE_BYTES, held by every GPU that loads this library
 * until the process exits.  The call allocates nothing: no cudaMalloc,
 * cudaFree or allocating library routine.  The first call on a device looks
 * up the array's device address (cudaGetSymbolAddress) with that device
 * current; make that first call before any stream capture.
 *
 * A batch whose muon_workspace_size() exceeds the array returns
 * MUON_ERR_WORKSPACE with an explanation in muon_last_error_message and
 * launches nothing.  All calls on a device share the array, which keeps the
 * last call's contents (nothing in it needs to start at zero); calls that
 * overlap on the GPU race on it and must be serialised by the caller.
 * Otherwise identical to muon_step().  The kernels' status word sits at the
 * start of the fixed array: muon_check_status(h, NULL, stream) reads and
 * clears it. */
muon_status muon_step_noalloc(muon_handle h, const muon_matrix_desc* descs, int n, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MUON_GB300_H */

/*
 * efla.h -- C ABI of the GB300 (sm_103a) library for the Exact Flow Linear
 * Attention (EFLA) token mixer.
 *
 * The method (gist.science summary of arXiv 2512.12602, "Exact Flow Linear
 * Attention: Exact Solution from Continuous-Time Dynamics", page es,
 * section "Metodologia"):
 *   item 1  ODE under zero-order hold:  dS/dt = -k_t k_t^T S + k_t v_t^T
 *   item 2  rank-1 closed form:         exp(-beta A) = I - ((1 - e^{-beta lambda})/lambda) A,
 *                                       lambda = ||k||^2
 *   item 3  exact update:               S_t = (I - alpha_t k_t k_t^T) S_{t-1} + alpha_t k_t v_t^T,
 *                                       alpha_t = (1 - e^{-beta_t lambda_t}) / lambda_t,
 *           evaluated chunkwise with the WY/UT representation the same item names.
 * Read-out (not on the pages; the delta-rule convention): o_t = S_t^T q_t, with
 * S_t the state after token t's update.
 *
 * General conventions of every entry point below:
 *  - Every array pointer is a DEVICE pointer owned by the caller; the library
 *    never allocates, frees or retains memory, and never synchronises except
 *    in efla_get_status().
 *  - Tensors are dense, contiguous and row-major:
 *        q, k      [B, H, L, dk]      v, o      [B, H, L, dv]
 *        beta      [B, H, L]  fp32    S0, S_final, dS_final, dS0  [B, H, dk, dv]  fp32
 *    (S is dk x dv, the shape of k v^T; row index = key dimension.)
 *  - Element types: q, k, v (and dO) are `dtype`; o (and dq, dk, dv) are
 *    `out_dtype`; beta, states and dbeta are always fp32.  All arithmetic is
 *    fp32 (accumulation, state, alpha).
 *  - Every pointer must be 16-byte aligned.
 *  - Supported sizes: dk, dv multiples of 16 in [16, 128]; chunk in {16, 32, 64};
 *    L >= 0 (L % chunk != 0 is allowed: the tail is handled exactly); B, H >= 0.
 *    Empty inputs (B*H == 0 or L == 0) launch nothing except the S0 -> S_final copy.
 *  - q is NOT scaled inside (the caller applies any 1/sqrt(dk)); k is NOT
 *    normalised (lambda is the raw ||k||^2); beta may be any finite value.
 *  - Non-finite inputs propagate to outputs; no input value traps the GPU.
 *  - Validation failures return before any launch; a launch failure returns
 *    EFLA_ERR_CUDA.  Work is enqueued asynchronously on `stream`; kernel-side
 *    failures are reported by efla_get_status().
 *  - efla_last_error() returns a human-readable message for the last non-OK
 *    status returned on the calling thread.
 */
#ifndef EFLA_H
#define EFLA_H

#include <stddef.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    EFLA_OK = 0,
    EFLA_ERR_INVALID_ARG = 1,   /* null pointer, negative size, forbidden aliasing */
    EFLA_ERR_UNSUPPORTED = 2,   /* size or dtype outside the supported set */
    EFLA_ERR_ALIGNMENT = 3,     /* a pointer is not 16-byte aligned */
    EFLA_ERR_WORKSPACE = 4,     /* workspace pointer null or smaller than required */
    EFLA_ERR_CUDA = 5,          /* a CUDA runtime call or launch failed */
    EFLA_ERR_TIMEOUT = 6,       /* a bounded device-side wait gave up (see efla_get_status) */
    EFLA_ERR_BOUNDS = 7         /* debug builds only: a tensor-core kernel's global write fell
                                   outside its buffer and was skipped (see efla_get_status) */
} efla_status;

typedef enum { EFLA_F32 = 0, EFLA_BF16 = 1 } efla_dtype;

/* EFLA_EXACT: alpha_t = (1 - e^{-beta_t lambda_t})/lambda_t (page es, Metodologia item 3).
 * EFLA_EULER: alpha_t = beta_t, the delta rule that the pages identify as the explicit
 *             Euler step of the same ODE (page es, "Contribuciones Clave", first item). */
typedef enum { EFLA_EXACT = 0, EFLA_EULER = 1 } efla_mode;

/* Which kernels run efla_fwd.
 * EFLA_PATH_TENSOR: tcgen05 tensor-core kernels (bf16 q/k/v, dk = dv = 128, chunk 64);
 *   every MMA operand is staged in fp16 with fp32 accumulation.  A sequence that staging
 *   cannot represent -- its largest key norm ||k|| outside [2^-10, 64], its largest query
 *   norm below 2^-11 or with ||q|| or ||k|| ||q|| at 2^15 or more, its largest |v| or |S0|
 *   element below 2^-10 (all-zero tensors excepted), or a non-finite final state (an fp16
 *   overflow of the state, W, U' or Ta reaches it as inf or NaN) -- is recomputed within
 *   the same call, token by token in fp32, so the results hold for any finite input; such
 *   a sequence costs about a microsecond per token instead of a few nanoseconds.  A few
 *   long sequences
 *   (B*H <= 32, L a multiple of 64 with at least 256 chunks) run segment-parallel: each
 *   sequence splits into 4..64 segments whose affine state maps S_end = P S_start + Q
 *   are chained in fp32 before the outputs are computed (more workspace; same results
 *   up to rounding).
 * EFLA_PATH_SIMT: fp32 CUDA-core kernels, any supported shape and dtype (full fp32 range).
 * EFLA_PATH_AUTO: TENSOR when the shape allows it, else SIMT.
 * efla_bwd: AUTO runs its products on the tensor pipe (mma.sync, tf32 operands, fp32
 *   accumulation) for bf16 inputs with dk = 128, chunk 64 and dv in {64, 128}, and on
 *   the fp32 CUDA cores otherwise; SIMT keeps every shape on the fp32 CUDA cores;
 *   TENSOR (the tcgen05 forward kernels) is rejected.
 * efla_step always runs on CUDA cores (TENSOR is rejected there). */
typedef enum { EFLA_PATH_AUTO = 0, EFLA_PATH_SIMT = 1, EFLA_PATH_TENSOR = 2 } efla_path;

typedef struct {
    int B, H, L, dk, dv, chunk;
    efla_dtype dtype;       /* q, k, v, dO */
    efla_dtype out_dtype;   /* o, dq, dk, dv */
    efla_mode mode;
    efla_path path;
} efla_shape;

/* Bytes of device workspace efla_fwd / efla_bwd need for this shape (0 on an invalid
 * shape).  The workspace is scratch for one call: its contents on entry are ignored. */
size_t efla_fwd_workspace_size(const efla_shape* shape);
size_t efla_bwd_workspace_size(const efla_shape* shape);

/* Chunked forward pass (page es, Metodologia item 3: update rule, alpha, WY/UT chunking).
 *   in : q, k [B,H,L,dk] dtype; v [B,H,L,dv] dtype; beta [B,H,L] fp32;
 *        S0 [B,H,dk,dv] fp32 or NULL (zero initial state)
 *   out: o [B,H,L,dv] out_dtype; S_final [B,H,dk,dv] fp32 or NULL (not written)
 * S_final may alias S0 exactly (resume in place); o must not overlap any input.
 * workspace: device scratch of at least efla_fwd_workspace_size(shape) bytes. */
efla_status efla_fwd(const efla_shape* shape,
                     const void* q, const void* k, const void* v, const float* beta,
                     const float* S0, void* o, float* S_final,
                     void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Backward pass of efla_fwd: gradients of  sum(o * dO) + sum(S_final * dS_final)
 * (reverse-mode differentiation of the update rule and alpha of page es, Metodologia
 * item 3; the pages state no backward pass).
 *   in : q, k, v, beta, S0 (NULL = zeros) as in efla_fwd; dO [B,H,L,dv] dtype;
 *        dS_final [B,H,dk,dv] fp32 or NULL (zeros)
 *   out: dq, dk [B,H,L,dk] out_dtype; dv [B,H,L,dv] out_dtype; dbeta [B,H,L] fp32;
 *        dS0 [B,H,dk,dv] fp32 or NULL (not written)
 * Outputs must not overlap inputs or each other. */
efla_status efla_bwd(const efla_shape* shape,
                     const void* q, const void* k, const void* v, const float* beta,
                     const float* S0, const void* dO, const float* dS_final,
                     void* dq, void* dk, void* dv, float* dbeta, float* dS0,
                     void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* ---- Training with a recorded forward (stored chunk states instead of recomputing them).
 * efla_bwd recomputes every chunk's entering state S_c with a sequential scan over the
 * chunks (the update rule of page es, Metodologia item 3, in its chunked form).  A caller
 * that keeps the forward's states until the backward skips that scan: efla_fwd_save
 * writes, beside o and S_final, a record of (fp32, in this order, each block 256-byte
 * aligned; NC = ceil(L / chunk))
 *     S_c   [B,H,NC,dk,dv]     the state entering chunk c (S_0 = S0, or zero)
 *     U'_c  [B,H,NC,chunk,dv]  the chunk's corrected values U' = U - W S_c
 *           (= alpha_t (v_t - S_{t-1}^T k_t) for each token t; rows past L are zero)
 *     T_c   [B,H,NC,chunk,chunk]  (I + strict_lower(diag(alpha) K K^T))^{-1} of the chunk
 *     alpha [B,H,NC,chunk]     alpha_t (zero past L)
 * and efla_bwd_saved computes the gradients of efla_bwd from it, without the state scan
 * and, on the tensor-core shapes, without re-preparing the chunks.  The record costs
 * efla_fwd_states_size() bytes of device memory held from forward to backward. */
size_t efla_fwd_states_size(const efla_shape* shape);

/* efla_fwd plus the record above in `states` (at least efla_fwd_states_size bytes,
 * 16-byte aligned, overlapping nothing else; NULL: plain efla_fwd).  Same results,
 * workspace and errors as efla_fwd. */
efla_status efla_fwd_save(const efla_shape* shape,
                          const void* q, const void* k, const void* v, const float* beta,
                          const float* S0, void* o, float* S_final, float* states, size_t states_bytes,
                          void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Bytes of device workspace efla_bwd_saved needs (less than efla_bwd's: no state scan). */
size_t efla_bwd_saved_workspace_size(const efla_shape* shape);

/* efla_bwd from a record written by efla_fwd_save with the same shape and inputs: the
 * gradients of  sum(o * dO) + sum(S_final * dS_final)  with respect to q, k, v, beta and
 * S0 (whose value the record holds), without the state scan.  Arguments and errors as
 * efla_bwd; `states` is read only. */
efla_status efla_bwd_saved(const efla_shape* shape,
                           const void* q, const void* k, const void* v, const float* beta,
                           const float* states, size_t states_bytes, const void* dO, const float* dS_final,
                           void* dq, void* dk, void* dv, float* dbeta, float* dS0,
                           void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Which backward a training step of this shape should use, given `free_bytes` of device
 * memory for the backward's scratch and anything kept from the forward: 1 = record the
 * states (efla_fwd_save + efla_bwd_saved; the record plus that backward's workspace), 0 =
 * recompute them (efla_fwd + efla_bwd; efla_bwd's workspace), -1 = neither fits (or the
 * shape is invalid).  Of the forms that fit, the faster is chosen:
 *  - on the tensor-core shapes that run in one pass (bf16, dk = dv = 128, chunk 64, not
 *    segment-parallel), efla_bwd: it records the states with the tcgen05 forward while its
 *    reverse scan runs beside it, which beats recording them in the training forward;
 *  - on every other shape, the recorded form: it skips a sequential state scan. */
int efla_bwd_plan(const efla_shape* shape, size_t free_bytes);

/* One recurrent decode step for B*H sequences (page es, Metodologia item 3, one token):
 *   S <- (I - alpha k k^T) S + alpha k v^T  in place;  o = S^T q  (after the update).
 *   in : q, k [B,H,dk] dtype; v [B,H,dv] dtype; beta [B,H] fp32
 *   in/out: S [B,H,dk,dv] fp32 (updated in place)
 *   out: o [B,H,dv] out_dtype (must not overlap S or the inputs)
 * shape->L must be 1; shape->chunk is ignored.  Needs no workspace. */
efla_status efla_step(const efla_shape* shape,
                      const void* q, const void* k, const void* v, const float* beta,
                      float* S, void* o, cudaStream_t stream);

/* ---- The token mixer's input projections (page es, "Resultados Experimentales" item 1:
 * the EFLA layers of the 340M and 1.3B language models; the pages name the models, not
 * their layer equations -- the read taken here is the usual linear-attention layer's):
 *     q = (x Wq^T) / sqrt(dk),  k = x Wk^T,  v = x Wv^T,  beta = sigmoid(x Wb^T)
 * per token x (d_model = D wide) and head h.  One tcgen05 GEMM with bf16 operands and fp32
 * accumulation; q, k, v are written in the [B, H, L, dk] layout efla_fwd takes.
 *   in : x [B, L, D] bf16; w [3 H dk + H, D] bf16 = the rows of Wq (H dk), Wk (H dk),
 *        Wv (H dk) and Wb (H), each row one output feature (a linear layer's weight)
 *   out: q, k, v [B, H, L, dk] bf16; beta [B, H, L] fp32
 * Supported: dk = 128, L a multiple of 128, D a multiple of 64 (>= 64), H even in
 * [2, 32]; else EFLA_ERR_UNSUPPORTED.  16-byte alignment; outputs must not overlap the
 * inputs or each other.  Needs no workspace. */
typedef struct { int B, L, D, H, dk; } efla_mixer_shape;
efla_status efla_mixer_proj(const efla_mixer_shape* shape, const void* x, const void* w,
                            void* q, void* k, void* v, float* beta, cudaStream_t stream);

/* Size of the device scratch array the library itself owns for efla_fwd_noalloc:
 * 40 MiB, held on every GPU that loads the library until the process exits. */
#define EFLA_NOALLOC_SCRATCH_BYTES (40u << 20)

/* efla_fwd for callers that cannot allocate device memory.  The paper has no
 * counterpart to this entry point: it serves callers such as plugins whose host
 * application owns the device allocator and forbids other allocations, and
 * real-time or embedded loops that may not allocate once running.  Arguments,
 * layouts, results and errors are those of efla_fwd, without the workspace: the
 * scratch comes from the library's own EFLA_NOALLOC_SCRATCH_BYTES device array.
 *  - A shape whose efla_fwd_workspace_size() exceeds EFLA_NOALLOC_SCRATCH_BYTES is
 *    rejected with EFLA_ERR_UNSUPPORTED (efla_last_error() names both sizes).
 *  - It calls no cudaMalloc, cudaFree or allocating library routine.
 *  - The first call on a device looks up the array's device address on that device
 *    (cudaGetSymbolAddress); make that first call before any stream capture.  The address
 *    is kept for the life of the process and belongs to the device's primary context (the
 *    one the CUDA runtime uses): after cudaDeviceReset, or with another context current
 *    on that device, it no longer points at the array, so do neither in a process that
 *    uses this entry point.
 *  - All calls share the array, which keeps the last call's contents (nothing in it
 *    needs clearing between calls).  Calls that overlap on the GPU race on it: the
 *    caller must serialise them (one stream at a time per device). */
efla_status efla_fwd_noalloc(const efla_shape* shape,
                             const void* q, const void* k, const void* v, const float* beta,
                             const float* S0, void* o, float* S_final, cudaStream_t stream);

/* Synchronises `stream`, then reports any asynchronous launch/kernel error
 * (EFLA_ERR_CUDA) or a device-side status word set by a bounded wait (EFLA_ERR_TIMEOUT),
 * and clears that word.  A library built with -DEFLA_DEBUG (libefla_gb300_debug.so) also
 * checks, tile by tile, that every global write of the tensor-core kernels lies inside its
 * buffer; a write that does not is skipped and reported here as EFLA_ERR_BOUNDS (before a
 * timeout, if both happened).  The status word is one per device (the current one), shared by
 * every stream and thread that uses the library on it: a timeout in work queued on one
 * stream is reported to, and cleared by, whichever call of efla_get_status on that device
 * comes first.  Callers that keep several streams busy at once should treat a timeout as
 * affecting all of them. */
efla_status efla_get_status(cudaStream_t stream);

/* Static string for a status code; never NULL. */
const char* efla_status_string(efla_status status);

/* Message for the last non-OK status returned on the calling thread ("" if none). */
const char* efla_last_error(void);

/* Diagnostic (no counterpart on the pages): one tcgen05 tile product through the
 * same shared-memory layouts, descriptors and tensor-memory path the tensor-core
 * forward uses:  D[128 x N] = C + A[128 x K] B[N x K]^T, with C, D fp32 row-major,
 * N in {64, 128, 192, 256}, K in {64, 128}; all device pointers.  A is fp16 row-major [128][K]
 * (staged K-major) or, with flags bit 0, its transpose [K][128] (staged MN-major), or,
 * with flags bit 2, [128][K] placed in tensor memory as the MMA's A operand;
 * B is [N][K] or, with flags bit 1, [K][N]. */
efla_status efla_tc_selftest(int N, int K, int flags, const void* A, const void* B, const float* C,
                             float* D, cudaStream_t stream);

/* Diagnostic (no counterpart on the pages) of the bounded device-side waits every
 * tensor-core kernel uses: one thread waits on something that never happens -- kind 0
 * an mbarrier missing one of its two arrivals, kind 1 a global flag nothing sets --
 * gives up after `limit` polls (1 .. 2^20) and records the timeout in the device status
 * word, exactly as the kernels do.  The next efla_get_status(stream) then returns
 * EFLA_ERR_TIMEOUT and clears the word; the context stays usable.  Invalid kind or
 * limit: EFLA_ERR_INVALID_ARG before any launch. */
efla_status efla_wait_selftest(int kind, int limit, cudaStream_t stream);

/* Kernel-level timing for measurement tools (no counterpart on the pages).
 * efla_profile_begin() switches timing on for the calling thread: every later
 * efla_fwd / efla_bwd / efla_step call on that thread records a CUDA event on its
 * stream before its first kernel and after each kernel it launches (the library
 * creates these events; nothing else is allocated).  efla_profile_end() synchronises
 * those events, switches timing off, and fills up to `cap` entries with each
 * distinct kernel's name (static strings), total milliseconds and launch count;
 * it returns the number of distinct kernels (or -1 on a CUDA error). */
efla_status efla_profile_begin(void);
int efla_profile_end(int cap, const char** names, float* total_ms, int* launches);

#ifdef __cplusplus
}
#endif

#endif /* EFLA_H */

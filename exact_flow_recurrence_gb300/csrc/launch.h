// launch.h -- internal (C++) interface between the C ABI layer and the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>

namespace efla {

// Bit of the device status words set by a debug build's bounds check (a skipped write);
// efla_get_status reports it as EFLA_ERR_BOUNDS.  Bit 0 is a bounded wait that expired.
constexpr unsigned kStatusBounds = 4u;

// Validated problem geometry.  C = chunk, NC = ceil(L / C).
struct Dims {
    int B, H, L, dk, dv, C, NC;
    int in_bf16;   // q, k, v, dO are bf16 (else fp32)
    int out_bf16;  // o, dq, dk, dv are bf16 (else fp32)
    int euler;     // alpha := beta
    int tensor;    // forward runs on the tcgen05 kernels
    long long BH() const { return (long long)B * H; }
};

inline size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// ------------------------------------------------------------------ forward
// Workspace of the SIMT chunked forward (all fp32):
//   alpha [BH][NC*C]        W, U, Up [BH][NC][C][dk|dv|dv]      Sc [BH][NC][dk][dv]
// Up = U - W Sc (the chunk's corrected values), Sc = state entering the chunk.
struct FwdWs {
    float* alpha;
    float* W;
    float* U;
    float* Up;
    float* Sc;
    float* T;     // null, or where the preparation also writes T [BH][NC][C][C] (a record)
};
size_t fwd_ws_bytes(const Dims& d);
FwdWs fwd_ws_carve(const Dims& d, void* base);

cudaError_t launch_fwd_simt(const Dims& d, const void* q, const void* k, const void* v,
                            const float* beta, const float* S0, void* o, float* S_final,
                            const FwdWs& ws, cudaStream_t st);

// Tensor-core forward (fwd_tc.cu): bf16 inputs, dk = dv = 128, chunk 64.
// Workspace: the Ta and P^T images, [BH][NC][64*64] fp16 each, then [BH][NC] int flags and
// [BH][NC][2] fp32 per-chunk norm maxima; in the segment-parallel form three
// [BH*nseg][128][128] fp32 state arrays, the final states and per-sequence words follow.
bool fwd_tc_supported(const Dims& d);
// Segments per sequence of the segment-parallel form (1: the plain form), a function of
// the shape alone: few sequences (B*H <= 32) of at least 256 whole chunks.
int fwd_tc_segments(const Dims& d);
size_t fwd_tc_ws_bytes(const Dims& d);
// rec_S / rec_Up / rec_T / rec_alpha (all null, or all set): the chunk-state record,
// S_c [BH][NC][128][128], U' [BH][NC][64][128], T [BH][NC][64][64], alpha [BH][NC][64] fp32.
// With a record, o may be null (not written).
// With rec_fp32 (one word per sequence; one-pass shapes only, else cudaErrorInvalidValue)
// the record's S_c and U' are written as fp16 images (see fwd_tc.cu) and rec_fp32 marks the
// sequences whose record is fp32 instead (recomputed in fp32).
// prepared: the chunk images (and norms, T, alpha) are already in `ws` (launch_tc_prep), so
// only the sequence CTAs run, with no flags; one-pass shapes only.
cudaError_t launch_fwd_tc(const Dims& d, const void* q, const void* k, const void* v,
                          const float* beta, const float* S0, void* o, float* S_final, void* ws,
                          cudaStream_t st, float* rec_S = nullptr, float* rec_Up = nullptr,
                          float* rec_T = nullptr, float* rec_alpha = nullptr, int* rec_fp32 = nullptr,
                          bool prepared = false);
// The chunk preparation alone, on every SM: the Ta and P^T images and the chunk norms at the
// start of `ws` (the layout both the forward's and the reverse scan's workspaces begin
// with), and T and alpha into rec_T, rec_alpha when given.
cudaError_t launch_tc_prep(const Dims& d, const void* q, const void* k, const float* beta, void* ws, float* rec_T,
                           float* rec_alpha, cudaStream_t st);
cudaError_t launch_tc_selftest(int N, int K, int flags, const void* A, const void* B,
                               const float* C, float* D, cudaStream_t st);
cudaError_t launch_wait_selftest(int kind, uint32_t limit, cudaStream_t st);
// Reads and clears the tensor-core kernels' device status word (synchronous).
cudaError_t tc_status_read_clear(unsigned int* status);

// ----------------------------------------------------------------- backward
// Workspace of the chunked backward: the forward workspace plus (fp32)
//   T, P [BH][NC][C][C]   dUp [BH][NC][C][dv]   dSc [BH][NC][dk][dv]
// T = (I + strict_lower(diag(alpha) K K^T))^{-1}, P = tril(Q K^T) (diagonal included),
// dSc = gradient w.r.t. the state leaving the chunk, dUp = gradient w.r.t. Up.
struct BwdWs {
    FwdWs f;
    float* T;
    float* P;
    float* dUp;
    float* dSc;
    void* tc;    // the tcgen05 reverse scan's images, flags, norms and marks (or null)
};
size_t bwd_ws_bytes(const Dims& d);
BwdWs bwd_ws_carve(const Dims& d, void* base);
// The chunk-state record (efla_fwd_save), each part 256-byte aligned, fp32:
//   S_c [BH][NC][dk][dv], U' [BH][NC][C][dv]  (the Sc and Up arrays of the forward workspace),
//   T [BH][NC][C][C], alpha [BH][NC][C]       (the chunk preparation's T and alpha)
size_t states_bytes(const Dims& d);
float* states_Up(const Dims& d, float* states);
float* states_T(const Dims& d, float* states);
float* states_alpha(const Dims& d, float* states);
// Backward workspace without Sc and Up, which come from a record instead.
size_t bwd_saved_ws_bytes(const Dims& d);
BwdWs bwd_saved_ws_carve(const Dims& d, void* base, const float* states);

// Tensor-pipe kernels of the backward (bwd_mma.cu): bf16 inputs, dk = 128, chunk 64,
// dv in {64, 128}, and d.tensor set (the caller's path allows them).  launch_prep_mma writes alpha, W, U, T and P; launch_scan_mma writes Up
// and Sc; launch_rscan_mma writes dUp, dSc (and dS0); launch_grad_mma reads alpha, T, Sc,
// dSc, Up and dUp.  With a work list (device words: list, and list_n its length) the
// preparation covers only the listed sequences and the gradients only the listed chunks, on
// a small grid, so an empty list costs one short launch.
bool grad_mma_supported(const Dims& d);
cudaError_t launch_prep_mma(const Dims& d, const void* q, const void* k, const void* v,
                            const float* beta, const BwdWs& ws, cudaStream_t st, const int* list = nullptr,
                            const int* list_n = nullptr);
cudaError_t launch_scan_mma(const Dims& d, const void* k, const float* S0, const BwdWs& ws,
                            cudaStream_t st);
// mask: null, or [BH] words; then only the sequences whose word is set are computed.
cudaError_t launch_rscan_mma(const Dims& d, const void* q, const void* k, const void* dO,
                             const float* dS_final, float* dS0, const BwdWs& ws, cudaStream_t st,
                             const int* mask = nullptr);

// The reverse scan on tcgen05 (bwd_tc.cu): bf16 inputs, dk = dv = 128, chunk 64.  Writes
// dS0, and per chunk dSc and dUp as fp16 images in the operand layout of launch_grad_tc
// (dSc [n-block 2][d 128][64 n], dUp [n-block 2][j 64][64 n], 128-byte swizzled rows;
// 32 and 16 KB per chunk), into its workspace.  seq_bad [BH] marks the sequences out of
// its fp16 staging's range (also listed in bad_list, bad_n of them): those are recomputed
// with that mask by launch_rscan_mma into the fp32 dSc, dUp arrays, and their images are not
// used.
struct RsTcOut {
    int* seq_bad;
    int* bad_n;
    int* bad_list;
    unsigned char* gimg;
    unsigned char* uimg;
};
bool rscan_tc_supported(const Dims& d);
size_t rscan_tc_ws_bytes(const Dims& d);
RsTcOut rscan_tc_outputs(const Dims& d, void* ws);
cudaError_t launch_rscan_tc(const Dims& d, const void* q, const void* k, const void* dO, const float* beta,
                            const float* dS_final, float* dS0, void* ws, cudaStream_t st, bool prepared = false);
cudaError_t bt_status_read_clear(unsigned int* status);
cudaError_t launch_grad_mma(const Dims& d, const void* q, const void* k, const void* v,
                            const void* dO, const float* beta, const BwdWs& ws, void* dq, void* dk,
                            void* dv, float* dbeta, cudaStream_t st, const int* list = nullptr,
                            const int* list_n = nullptr);

// The per-chunk gradients on tcgen05 (grad_tc.cu): bf16 inputs, dk = dv = 128, chunk 64.
// dSc and dUp come from the reverse scan's images (rs), or from the fp32 arrays for the
// sequences rs.seq_bad marks; Sc and Up are fp32, or (fwd_fp32 non-null) the forward's fp16
// images for the sequences whose word there is clear.  Lists the chunks out of its fp16 staging's range in its
// workspace (grad_tc_list: count, then chunk indices), for launch_grad_mma; launch_widen
// first gives those chunks fp32 dSc, dUp copies of their images.
bool grad_tc_supported(const Dims& d);
size_t grad_tc_ws_bytes(const Dims& d);
struct GtList {
    int* n;
    int* chunks;
    int* fwd_fp32;   // [BH] record-format words of a forward recording fp16 images (launch_fwd_tc)
};
GtList grad_tc_list(const Dims& d, void* ws);
cudaError_t launch_grad_tc(const Dims& d, const void* q, const void* k, const void* v, const void* dO,
                           const float* beta, const float* alpha, const float* T, const float* Sc, const float* dSc,
                           const float* Up, const float* dUp, const RsTcOut& rs, const int* fwd_fp32, void* dq,
                           void* dk, void* dv, float* dbeta, const GtList& redo, cudaStream_t st);
cudaError_t launch_widen(const Dims& d, const RsTcOut& rs, const GtList& redo, const int* fwd_fp32, float* Sc,
                         float* Up, float* dSc, float* dUp, cudaStream_t st);
cudaError_t gt_status_read_clear(unsigned int* status);

// Whether efla_bwd on this shape records the chunk states with the tcgen05 forward (beside
// its reverse scan) instead of a separate preparation and state scan: bf16, dk = dv = 128,
// chunk 64, one-pass (not segment-parallel) shapes on the tensor path.
bool bwd_runs_recording_forward(const Dims& d);
// have_states: ws.f.Sc and ws.f.Up already hold the chunk states (a record): no state scan.
cudaError_t launch_bwd_simt(const Dims& d, const void* q, const void* k, const void* v,
                            const float* beta, const float* S0, const void* dO,
                            const float* dS_final, void* dq, void* dk, void* dv, float* dbeta,
                            float* dS0, const BwdWs& ws, cudaStream_t st, bool have_states = false);

// ------------------------------------------------------------ mixer projections
// mixer_proj.cu: x [B L][D] bf16 times [Wq; Wk; Wv; Wb]^T ([3 H 128 + H][D] bf16) ->
// q (scaled by 1/sqrt(128)), k, v [B][H][L][128] bf16, beta = sigmoid [B][H][L] fp32.
// Needs L % 128 == 0, D % 64 == 0, H even and <= 32.
cudaError_t launch_mixer_proj(int B, int L, int D, int H, const void* x, const void* w, void* q, void* k, void* v,
                              float* beta, cudaStream_t st);
// Reads and clears the projection kernel's device status word (synchronous).
cudaError_t proj_status_read_clear(unsigned int* status);

// ------------------------------------------------------------------- decode
cudaError_t launch_step(const Dims& d, const void* q, const void* k, const void* v,
                        const float* beta, float* S, void* o, cudaStream_t st);
// Reads and clears the decode step's device status word (synchronous).
cudaError_t sd_status_read_clear(unsigned int* status);

// -------------------------------------------------------------- profiling
// Records a CUDA event on `st` labelled `name` when the calling thread has kernel
// timing switched on (efla_profile_begin); a no-op otherwise.  An entry point
// calls prof_mark(nullptr, st) before its first launch and prof_mark("kernel", st)
// after each launch; the time between consecutive marks is charged to the kernel.
void prof_mark(const char* name, cudaStream_t st);

// Sets the message efla_last_error() returns on the calling thread.
void set_last_error(const char* fmt, ...);

// ------------------------------------------------------------------ helpers
// S_final <- S0 (or zeros when S0 == nullptr) for empty sequences.
cudaError_t launch_state_copy(long long n, const float* S0, float* S_final, cudaStream_t st);

}  // namespace efla

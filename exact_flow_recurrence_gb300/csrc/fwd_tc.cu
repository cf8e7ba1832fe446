// fwd_tc.cu -- tensor-core (tcgen05) chunked forward of EFLA for dk = dv = 128,
// chunk 64, bf16 inputs.
//
// Same chunk algebra as the SIMT path (page es, Metodologia item 3, WY/UT form):
//   T = (I + strict_lower(diag(alpha) K K^T))^{-1},  Ta = T diag(alpha)
//   W = Ta K,  U = Ta V,  Up = U - W S,  O = Q S + tril(Q K^T) Up,  S' = S + K^T Up
// evaluated in transposed form so that every MMA has M = 128 (d_k or d_v rows):
//   W^T = K^T Ta^T        U^T = V^T Ta^T                      (M = 128, N = 64, K = 64)
//   [ (W S)^T | (Q S)^T ] = S^T [ W^T | Q^T ]                 (M = 128, N = 128, K = 128)
//   Up^T = U^T - (W S)^T
//   O^T = (Q S)^T + Up^T P^T,   S^T += Up^T K                 (M = 128, K = 64)
//   tril(Q K^T) from [Q; K] K^T                               (M = 128, N = 64, K = 128)
//
// Precision: every MMA operand is staged in fp16 (11-bit significand), with fp32
// accumulation in tensor memory.  bf16 operands are measurably too coarse for a
// 1e-2 max|err|/rms bound on the outputs (the U' and P operands dominate the
// error); fp16 keeps the bf16 tensor rate and represents bf16 inputs exactly
// in its normal range.  Intermediate magnitudes must stay below 65504.
//
// Two kernels:
//   k_tmat   -- chunk-parallel: Gram matrix G = K K^T of two chunks per CTA on
//               tcgen05, alpha, T by fp32 forward substitution, Ta written as an
//               fp16 image already in the 128-byte-swizzled K-major layout.
//   k_fwd_tc -- one CTA per sequence, sequential over chunks: S^T lives in tensor
//               memory (fp32) for the whole sequence; per chunk the raw K, Q, V
//               rows and the Ta image arrive by bulk async copy (prefetched one
//               chunk ahead) and are converted to fp16 operand tiles.
// Every wait on an mbarrier is bounded; on expiry the kernel records
// EFLA_ERR_TIMEOUT in a device status word, drains its own outstanding copies
// and MMAs (again bounded), frees its tensor memory and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "launch.h"
#include "tc_common.cuh"
#include "tc_ptx.cuh"

namespace efla {

using namespace tc;

// device status word: bit 0 = a bounded wait expired; kStatusBounds (debug builds) = a write
// was skipped
__device__ unsigned int g_tc_status = 0;


__device__ __forceinline__ void record_timeout() { atomicOr(&g_tc_status, 1u); }

// Token-by-token fp32 evaluation of one sequence (page es, Metodologia item 3, the
// update rule in its recurrent form):
//   lambda = ||k||^2,  alpha = alpha_of(beta, lambda),  r = v - S^T k,
//   o = S^T q + alpha (k.q) r  (= S'^T q, the state after the update),  S' = S + alpha k r^T.
// Used for sequences the fp16 staging cannot represent (see above).  512 threads
// (tid < 512) take part: thread (g = tid / 128, j = tid % 128) holds S[32g .. 32g+31][j]
// in registers; each token costs two barriers of those 512 threads (named barrier
// `bar`).  Inputs are the sequence's own rows: q, k [L][128], v [L][128] bf16, beta [L];
// S0 [128][128] fp32 or null; o [L][128] (bf16 or fp32) or null (not written); S_final
// [128][128] or null (may be S0).  `smf` needs kRecSmemFloats floats of shared memory.  With rec_S / rec_Up (the
// sequence's part of the chunk-state record, chunks of 64 tokens) it also writes the state
// entering every chunk and each token's corrected value alpha_t r_t (zero past L).
constexpr int kRecThreads = 512;
constexpr int kRecBuf = 3 * 128 + 4;                       // k, q, v, beta of one token
constexpr int kRecSmemFloats = 2 * kRecBuf + 4 * 128 * 2 + 4;

__device__ __noinline__ void seq_recurrent_fp32(const __nv_bfloat16* q, const __nv_bfloat16* k,
                                                const __nv_bfloat16* v, const float* beta, const float* S0,
                                                void* o, int out_bf16, float* S_final, int L, int euler,
                                                float* smf, int tid, int bar, float* rec_S, float* rec_Up) {
    const int g = tid >> 7, j = tid & 127;
    float* tok = smf;                          // [2][kRecBuf]
    float2* part = reinterpret_cast<float2*>(smf + 2 * kRecBuf);   // [4][128]: (S^T k, S^T q) partials
    float* scal = smf + 2 * kRecBuf + 4 * 128 * 2;                 // lambda, k.q
    float s[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) s[i] = S0 ? S0[(size_t)(32 * g + i) * 128 + j] : 0.f;
    // this thread's share of a token's inputs: tid < 384 one element of k | q | v, tid 384 beta
    auto fetch = [&](int t) -> float {
        if (t >= L || tid > 384) return 0.f;
        if (tid == 384) return beta[t];
        const __nv_bfloat16* src = tid < 128 ? k : (tid < 256 ? q : v);
        return __bfloat162float(src[(size_t)t * 128 + (tid & 127)]);
    };
    float cur = fetch(0), nxt = fetch(1);
    for (int t = 0; t < L; ++t) {
        float* tb = tok + (t & 1) * kRecBuf;
        if (rec_S && (t & 63) == 0) {
#pragma unroll
            for (int i = 0; i < 32; ++i) rec_S[(size_t)(t >> 6) * 16384 + (size_t)(32 * g + i) * 128 + j] = s[i];
        }
        if (tid <= 384) tb[tid] = cur;
        cur = nxt;
        nxt = fetch(t + 2);
        asm volatile("bar.sync %0, %1;" ::"r"(bar), "r"(kRecThreads) : "memory");
        float pk = 0.f, pq = 0.f;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            pk = fmaf(s[i], tb[32 * g + i], pk);
            pq = fmaf(s[i], tb[128 + 32 * g + i], pq);
        }
        part[g * 128 + j] = make_float2(pk, pq);
        if (tid < 32) {
            float lam = 0.f, kq = 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float kk = tb[tid + 32 * i];
                lam = fmaf(kk, kk, lam);
                kq = fmaf(kk, tb[128 + tid + 32 * i], kq);
            }
            lam = warp_sum(lam);
            kq = warp_sum(kq);
            if (tid == 0) {
                scal[0] = lam;
                scal[1] = kq;
            }
        }
        asm volatile("bar.sync %0, %1;" ::"r"(bar), "r"(kRecThreads) : "memory");
        float sk = 0.f, sq = 0.f;
#pragma unroll
        for (int gg = 0; gg < 4; ++gg) {
            const float2 p = part[gg * 128 + j];
            sk += p.x;
            sq += p.y;
        }
        const float al = alpha_of(tb[384], scal[0], euler);
        const float r = tb[256 + j] - sk;
        if (g == 0 && o) {
            const float ot = fmaf(al * scal[1], r, sq);
            if (out_bf16) ((__nv_bfloat16*)o)[(size_t)t * 128 + j] = __float2bfloat16_rn(ot);
            else ((float*)o)[(size_t)t * 128 + j] = ot;
        }
        const float ar = al * r;
        if (rec_Up && g == 0) rec_Up[(size_t)t * 128 + j] = ar;
#pragma unroll
        for (int i = 0; i < 32; ++i) s[i] = fmaf(tb[32 * g + i], ar, s[i]);
    }
    if (rec_Up && g == 0)
        for (int t = L; t < ((L + 63) & ~63); ++t) rec_Up[(size_t)t * 128 + j] = 0.f;
    if (S_final) {
        asm volatile("bar.sync %0, %1;" ::"r"(bar), "r"(kRecThreads) : "memory");   // S0 may be S_final
#pragma unroll
        for (int i = 0; i < 32; ++i) S_final[(size_t)(32 * g + i) * 128 + j] = s[i];
    }
}

// =============================================================== self-test
// D[128 x N] = C + A[128 x K] B[N x K]^T.  A is given row-major as [128][K] (staged
// K-major) or, with flags bit 0, as A^T [K][128] (staged MN-major), or, with flags
// bit 2, row-major [128][K] placed in tensor memory (packed fp16 pairs); B is
// [N][K] or, with bit 1, B^T [K][N].  Exercises both descriptor layouts, the
// tensor-memory A operand, the instruction descriptor, commit, and TMEM loads/stores
// used by the kernels below.
__device__ __forceinline__ void stage_tile(unsigned char* dst, const __half* src, int rows, int cols,
                                           int nthr) {
    // src row-major [rows][cols]; dst: cols/64 blocks of rows x 128 B, SW128
    for (int u = threadIdx.x; u < rows * (cols / 8); u += nthr) {
        const int r = u / (cols / 8), ch = u % (cols / 8);
        const uint4 v = *reinterpret_cast<const uint4*>(src + (size_t)r * cols + ch * 8);
        *reinterpret_cast<uint4*>(dst + (ch / 8) * (rows * 128) + sw128(r, (ch % 8) * 8)) = v;
    }
}

__global__ void __launch_bounds__(128, 1) k_tc_selftest(int N, int K, int flags, const __half* A,
                                                        const __half* B, const float* C, float* D) {
    extern __shared__ __align__(1024) unsigned char sm_raw[];
    unsigned char* sm = (unsigned char*)(((uintptr_t)sm_raw + 1023) & ~(uintptr_t)1023);
    unsigned char* As = sm;                         // 128*K*2 bytes
    unsigned char* Bs = sm + 128 * K * 2;           // N*K*2 bytes
    uint64_t* bar = (uint64_t*)(Bs + N * K * 2);
    uint32_t* slot = (uint32_t*)(bar + 1);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool a_mn = flags & 1, b_mn = flags & 2, a_tm = flags & 4;

    if (a_mn) stage_tile(As, A, K, 128, 128);       // 2 blocks of K rows (M 0-63 | 64-127)
    else if (!a_tm) stage_tile(As, A, 128, K, 128); // K/64 blocks of 128 rows
    if (b_mn) stage_tile(Bs, B, K, N, 128);
    else stage_tile(Bs, B, N, K, 128);
    if (tid == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(slot, 512);
        tmem_relinquish();
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = *slot;
    if (a_tm) {   // A row (this thread's lane) -> columns 256.. as packed fp16 pairs
        const uint32_t* arow = reinterpret_cast<const uint32_t*>(A + (size_t)(warp * 32 + lane) * K);
        for (int c0 = 0; c0 < K / 2; c0 += 16) {
            uint32_t v[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = arow[c0 + i];   // (A[r][2c], A[r][2c+1]) low, high
            tmem_st16u(taddr(tb, warp * 32, 256 + c0), v);
        }
    }
    // D <- C through tcgen05.st
    for (int c0 = 0; c0 < N; c0 += 16) {
        float v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = C[(size_t)(warp * 32 + lane) * N + c0 + i];
        tmem_st16(taddr(tb, warp * 32, c0), v);
    }
    tmem_st_wait();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
        tc_fence_after();
        const uint32_t idesc = idesc_f16(128, N, a_mn, b_mn);
        for (int s = 0; s < K / 16; ++s) {
            const uint64_t bd = b_mn ? sdesc_sw128(smem_u32(Bs + s * 2048), K * 128)
                                     : sdesc_sw128(smem_u32(Bs + (s / 4) * (N * 128) + (s % 4) * 32));
            if (a_tm) {
                mma_f16_ts(tb, tb + 256 + 8 * s, bd, idesc, 1u);
            } else {
                const uint64_t ad = a_mn ? sdesc_sw128(smem_u32(As + s * 2048), K * 128)
                                         : sdesc_sw128(smem_u32(As + (s / 4) * 16384 + (s % 4) * 32));
                mma_f16_ss(tb, ad, bd, idesc, 1u);
            }
        }
        mma_commit(bar);
    }
    const bool ok = __syncthreads_and(mbar_wait(bar, 0, kWaitLimit));
    if (!ok) {
        if (tid == 0) record_timeout();
        mbar_wait(bar, 0, kWaitLimit);
    }
    tc_fence_after();
    if (ok) {
        for (int c0 = 0; c0 < N; c0 += 16) {
            float v[16];
            tmem_ld16(taddr(tb, warp * 32, c0), v);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i) D[(size_t)(warp * 32 + lane) * N + c0 + i] = v[i];
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tb, 512);
}

cudaError_t launch_tc_selftest(int N, int K, int flags, const void* A, const void* B,
                               const float* C, float* D, cudaStream_t st) {
    const size_t sm = 1024 + (size_t)128 * K * 2 + (size_t)N * K * 2 + 64;
    cudaError_t e = cudaFuncSetAttribute(k_tc_selftest, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)sm);
    if (e != cudaSuccess) return e;
    k_tc_selftest<<<1, 128, sm, st>>>(N, K, flags, (const __half*)A, (const __half*)B, C, D);
    prof_mark("efla_tc_selftest", st);
    return cudaGetLastError();
}

// ================================================================= k_tmat
// The chunk preparation (tmat_chunk, tc_common.cuh) as a kernel of its own: one chunk
// per CTA, 128 threads, four CTAs per SM so that the phases of different chunks overlap.
__global__ void __launch_bounds__(kTmThreads, 4)
    k_tmat(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q, TmatArgs a) {
    extern __shared__ __align__(1024) unsigned char sm_raw[];
    unsigned char* sm = (unsigned char*)(((uintptr_t)sm_raw + 1023) & ~(uintptr_t)1023);
    uint64_t* bar = (uint64_t*)(sm + kTmBar);
    uint32_t* slot = (uint32_t*)(bar + 2);
    const int tid = threadIdx.x;
    if (tid == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        fence_mbar_init();
    }
    if (tid < 32) {
        tmem_alloc(slot, 128);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = *slot;
    // the chunk of the CTA one wave of resident CTAs later (4 per SM): its rows go to L2 now
    uint32_t nsm;
    asm("mov.u32 %0, %%nsmid;" : "=r"(nsm));
    const long long lin = (long long)blockIdx.y * gridDim.x + blockIdx.x, nxt = lin + 4ll * nsm;
    const bool pf = nxt < (long long)gridDim.x * gridDim.y;
    tmat_chunk(&tm_k, &tm_q, a, sm, bar, 0, tb, 1, tid, blockIdx.x, blockIdx.y, nullptr, &g_tc_status,
               pf ? nxt % gridDim.x : -1, pf ? (int)(nxt / gridDim.x) : 0);
    tc_fence_before();
    __syncthreads();
    if (tid < 32) tmem_dealloc(tb, 128);
}

// =============================================================== k_fwd_tc
// One CTA per sequence, warp-specialized and pipelined one chunk deep.  A tcgen05.mma
// of M = 128, K = 16 occupies the tensor pipe for about the same time for any N up to
// ~176, so the chunk step is arranged to issue few, wide instructions:
//   MMA3(c)  [(W S)^T | (Q S)^T] = S^T [W; Q]^T                  8 x N=128
//   MMA5(c)  [O^T | S^T] += Up^T [P^T | K]                       4 x N=192
//   W(c+1)   W^T = K^T Ta^T                                      4 x N=64
//   U(c+1)   U^T = V^T Ta^T                                      4 x N=64
// issued in the order MMA3(c), W(c+1), MMA5(c), U(c+1): each of the next chunk's
// products fills one of the tensor pipe's waits for the epilogue warps (Up after
// MMA3, the S^T copy after MMA5).  P^T and Ta come from k_tmat.
//   M  (warp 0)      : one thread issues the MMAs
//   E1 (warps 1-8)   : Up^T = U^T - (W S)^T (packed fp16, in tensor memory); the W rows
//                      of chunk c+1 (from W^T in tensor memory) while MMA5(c) runs; then
//                      the fp16 copy of S^T for MMA3(c+1) and O -> global
//   E2 (warps 9-11, 13-15, 17-18: none shares the MMA issuer's scheduler, whose few
//                      shared-memory and barrier accesses queue behind this group's
//                      traffic otherwise)
//                    : once MMA5(c) has freed slot c mod 3, converts chunk c+3 (raw K,
//                      Q, V rows loaded into registers one chunk earlier) into fp16 operand
//                      tiles there; issues the loads of chunk c+4, and one thread an L2
//                      prefetch of chunk c+6's rows (so that those loads find them in L2).
//                      Off the chunk-to-chunk path: it works two chunks ahead.
//   B  (warp 19)     : one thread bulk-copies each chunk's Ta and P^T images as soon as
//                      its slot is free (issuing a bulk copy can hold a thread for a long
//                      time, so no thread on the chunk-to-chunk path does it)
// Hand-offs are mbarriers (every wait bounded):
//   ops_full[s]  E2 (256) + B (1 + image bytes) -> M   slot s holds Q, K, P^T of its chunk
//                                                       and its V/Ta buffer V and Ta
//   ops_empty[s] MMA5 commit -> E2, B                   slot s free again
//   vt_free[v]   U commit -> E2, B                      V/Ta buffer v free again
//   m_w          W commit -> E1
//   m3, m5       MMA3 / MMA5 commits -> E1
//   rdy3         E1 (256: W rows of c written, S^T copy of c-1 written, O of c-1 read)
//                -> M: MMA3(c) may start
//   rdy5         E1 (256: Up^T of c) -> M: MMA5(c) may start
// The issuing thread polls as few barriers as possible: under the operand traffic of
// the other warps every shared-memory access it makes costs hundreds of cycles.
struct FwdTcArgs {
    const __nv_bfloat16* q;
    const __nv_bfloat16* k;
    const __nv_bfloat16* v;   // unused by k_fwd_tc<true> (all values zero)
    const uint16_t* Ta;
    const uint16_t* Pt;
    const float* S0;
    void* o;
    float* S_final;
    int* flags;     // [BH][NC] image-ready flags (fused launch) or null (k_tmat ran before)
    TmatArgs prep;  // preparation work of the fused launch's other CTAs
    int* seq_bad;   // segment-parallel form: one word per original sequence, set when a
                    // segment's staging went out of range (recomputed afterwards); null:
                    // each CTA recomputes its own sequence in fp32 when that happens
    float* rec_S;   // chunk-state record (k_fwd_tc<*, 1>): S_c [BH][NC][128][128] fp32
    float* rec_Up;  //   and U' [BH][NC][64][128] fp32 (tail rows zero)
    int* rec_fp32;  // k_fwd_tc<*, 2>: [BH], set for a sequence recomputed in fp32 (its record
                    //   is fp32 as above; every other sequence's is the fp16 images)
    int L, NC, out_bf16, BH, nseg;
};

// The record's fp16 image form (k_fwd_tc<*, 2>, for the backward's own workspace): each
// chunk's S_c and U' as the 128-byte-swizzled fp16 tiles the gradient kernel stages, in the
// first 32 KB (S_c: [n-block 2][d 128][64 n]) and 16 KB (U': [n-block 2][j 64][64 n]) of
// that chunk's fp32 slots.  Element (row r, column n) of an image with `rows` rows per
// n-block, as a byte offset:
__device__ __forceinline__ uint32_t img_off(int r, int n, int rows) {
    return (uint32_t)(n >> 6) * (uint32_t)(rows * 128) + sw128(r, n & 63);
}

// Shared-memory map (byte offsets from a 1024-aligned base).  Every operand tile is
// fp16 SW128 in rows of 128 bytes; a "d-block" holds elements 64b..64b+63 of d.
// Three chunk slots (chunk c in slot c mod 3, so that the inputs of chunk c+2 can be
// written while chunks c and c+1 are in use), each:
//   +0      P^T  [64 rows j][64 i]                    MN-major B block of MMA5 (image from k_tmat)
//   +8192   d-block 0: W rows (i), Q rows (i), K rows (j), 64 rows each
//   +32768  d-block 1: the same
// so that [W; Q] (rows 0..127 of a d-block) is the K-major B of MMA3, K rows read as
// rows = token the MN-major A (K^T) of W, and P^T, K d-block 0, K d-block 1 sit 24576
// bytes apart: one MN-major B of N = 192.  Two V/Ta buffers (chunk c in buffer c mod 2,
// read by W(c) and U(c) only), each:
//   +0      V    2 n-blocks x [64 rows j]             MN-major A (V^T) of U
//   +16384  Ta   [64 rows i][64 j]                    K-major B (Ta^T) of W and U (image from k_tmat)
// The state and Up never pass through shared memory: S^T accumulates in tensor
// memory and its fp16 copy and Up^T (packed fp16 pairs) are tensor-memory A operands.
constexpr uint32_t kSlotBytes = 57344;
constexpr uint32_t kSlotPt = 0;
constexpr uint32_t kSlotBlk = 8192;       // + d-block * kBlkStride
constexpr uint32_t kBlkStride = 24576;
constexpr uint32_t kBlkW = 0, kBlkQ = 8192, kBlkK = 16384;
constexpr uint32_t kOffVT = 3 * kSlotBytes;     // V/Ta buffers
constexpr uint32_t kVTBytes = 24576;
constexpr uint32_t kVTV = 0;              // + n-block * 8192
constexpr uint32_t kVTTa = 16384;
constexpr uint32_t kOffBar = kOffVT + 2 * kVTBytes;   // mbarriers, TMEM slot, flags
constexpr size_t kFwdTcSmem = 1024 + kOffBar + 256;
static_assert(kFwdTcSmem <= 232448, "shared memory per CTA");

// TMEM columns (lane = row).  fp32 accumulators unless noted.
constexpr uint32_t kColX = 0;     // (W S)^T [n][i]; after the Up epilogue, cols [0,16) and
                                  //   [32,48) hold Up^T as packed fp16 (tokens 0..31 | 32..63)
constexpr uint32_t kColO = 64;    // (Q S)^T -> O^T [n][i]                         64 cols
constexpr uint32_t kColS = 128;   // S^T     [n][d]                              128 cols
constexpr uint32_t kColU = 256;   // U^T     [n][i], two buffers              2 x 64 cols;
                                  //   once chunk c's U is consumed, buffer c&1 holds the
                                  //   fp16 copy of S^T (packed, 64 cols) read by MMA3(c+1)
constexpr uint32_t kColW = 384;   // W^T     [d][i]                              64 cols

constexpr uint32_t kColUp = 448;  // k_fwd_tc<*, 2>: Up^T packed fp16 here (64 free columns), so that
                                  //   it outlives MMA3(c+1) for the record's image
// tensor-memory column of k-step s (16 tokens) of the packed Up^T operand, and the first
// column group `grp`'s 32 tokens pack into
template <int kRec>
__device__ __forceinline__ uint32_t up_col(int s) {
    return kRec == 2 ? kColUp + 8 * s : kColX + 8 * s + (s >= 2 ? 16 : 0);
}
template <int kRec>
__device__ __forceinline__ uint32_t up_pack_col(int grp) {
    return kRec == 2 ? kColUp + 16 * grp : kColX + 32 * grp;
}

constexpr int kFwdThreads = 20 * 32;   // warps 12 and 16 stay idle
constexpr int kMinPrepCtas = 16;        // fused launch only with at least this many preparation CTAs


// Clears the image-ready flags of a fused launch.  The fused kernel is its programmatic
// dependent: its CTAs are scheduled as soon as these have started, set up their barriers and
// tensor memory, and wait (griddepcontrol.wait) for this grid's completion before touching
// global memory.
__global__ void k_zero_flags(int* flags, int n) {
    griddep_launch_dependents();
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) flags[i] = 0;
}

// kZeroV: every value is zero (v is not read).  kRec: also write the chunk-state record,
// in fp32 (1) or as fp16 images (2; a sequence recomputed in fp32 keeps the fp32 form).
template <bool kZeroV, int kRec = 0>
__global__ void __launch_bounds__(kFwdThreads, 1)
    k_fwd_tc(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q, FwdTcArgs a) {
    extern __shared__ __align__(1024) unsigned char sm_raw[];
    unsigned char* sm = (unsigned char*)(((uintptr_t)sm_raw + 1023) & ~(uintptr_t)1023);
    if (blockIdx.x >= a.BH) {
        // ======================= preparation CTA (fused launch) =======================
        // Four groups of 128 threads (warps 4g..4g+3) each run k_tmat's work on one chunk
        // at a time, taking the chunks in chunk-major order (all sequences' chunk 0
        // first), so that the sequence CTAs find their images early; warps 16..19 idle.
        const int tid = threadIdx.x, warp = tid >> 5, g = warp >> 2;
        uint32_t* pslot = (uint32_t*)(sm + 4 * kTmGroupBytes);
        unsigned char* gsm = sm + g * kTmGroupBytes;
        uint64_t* gbar = (uint64_t*)(gsm + kTmBar);
        if (warp < 16 && (tid & 127) == 0) {
            mbar_init(&gbar[0], 1);
            mbar_init(&gbar[1], 1);
            fence_mbar_init();
        }
        if (warp == 0) {
            tmem_alloc(pslot, 512);
            tmem_relinquish();
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        griddep_wait();   // (fused launch: the flags are clear from here on)
        const uint32_t tbase = *pslot;
        if (warp < 16) {
            const int nworkers = (gridDim.x - a.BH) * 4, total = a.BH * a.NC;
            uint32_t ph = 0;
            // At the launch every group and every sequence CTA loads at once.  The groups whose
            // first chunk is not in the first chunk row, which the sequences wait on before their
            // first product, start about a microsecond later so that row's tiles arrive sooner
            // (a plain clock spin: it waits on nobody).  Measured on the 340M-layer forward: -1%
            // at 2000 cycles, mixed at 4000, +2% at 8000.
            if ((blockIdx.x - a.BH) * 4 + g >= a.BH) {
                const long long t0c = clock64();
                while (clock64() - t0c < 2000) {}
            }
            for (int w = (blockIdx.x - a.BH) * 4 + g; w < total; w += nworkers, ph ^= 1u) {
                const int c = w / a.BH, bhw = w - c * a.BH;
                const int wn = w + nworkers, cn = wn / a.BH;   // this group's next chunk
                if (!tmat_chunk(&tm_k, &tm_q, a.prep, gsm, gbar, ph, tbase + 128 * g, 1 + g, tid & 127, bhw,
                                c, a.flags + (size_t)bhw * a.NC + c, &g_tc_status, wn < total ? wn - cn * a.BH : -1,
                                cn))
                    break;
            }
        }
        tc_fence_before();
        __syncthreads();
        if (warp == 0) tmem_dealloc(tbase, 512);
        return;
    }
    uint64_t* bars = (uint64_t*)(sm + kOffBar);
    uint64_t* ops_full = bars + 0;      // [3]
    uint64_t* ops_empty = bars + 3;     // [3]
    uint64_t* m_w = bars + 6;
    uint64_t* m3 = bars + 7;
    uint64_t* m5 = bars + 8;
    uint64_t* rdy3 = bars + 9;
    uint64_t* rdy5 = bars + 10;
    uint64_t* vt_free = bars + 11;      // [2]
    uint64_t* st_free = bars + 13;      // [3] k_fwd_tc<*, 2>: slot s's record images read out
    uint32_t* slot = (uint32_t*)(bars + 16);
    volatile int* s_abort = (volatile int*)(slot + 1);
    // staging checks: [0] bit 0 = a non-finite final state, bit 1 = recompute this
    // sequence; [1], [2] largest ||k||^2, ||q||^2; [3] largest |v| or |S0| element
    // (fp32 bit patterns, >= 0)
    unsigned* s_stat = slot + 2;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int q4 = warp & 3;            // TMEM lane quadrant of this warp
    const int row = q4 * 32 + lane;     // TMEM lane = matrix row this thread reads
    const long long bh = blockIdx.x;
    const int L = a.L, NC = a.NC;
    const size_t seq_tok = (size_t)bh * L;

    if (tid == 0) {
        for (int i = 0; i < 3; ++i) {
            mbar_init(&ops_full[i], 257);
            mbar_init(&ops_empty[i], 1);
        }
        mbar_init(&vt_free[0], 1);
        mbar_init(&vt_free[1], 1);
        for (int i = 0; i < 3; ++i) mbar_init(&st_free[i], 1);
        mbar_init(m_w, 1);
        mbar_init(m3, 1);
        mbar_init(m5, 1);
        mbar_init(rdy3, 256);
        mbar_init(rdy5, 256);
        *s_abort = 0;
        s_stat[0] = s_stat[1] = s_stat[2] = s_stat[3] = 0u;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    griddep_wait();   // (fused launch: the flags are clear from here on; otherwise a no-op)
    const uint32_t tb = *slot;

    // bounded wait; on expiry every role stops at its next wait that does not succeed
    // at once (the flag is read only off the fast path)
    auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
        if (mbar_try_wait(bar, parity)) return true;
        if (*s_abort) return false;
        if (mbar_wait(bar, parity, kWaitLimit)) return true;
        *s_abort = 1;
        return false;
    };

    if (warp >= 1 && warp <= 8) {
        // ============================ E1: Up^T, O, S^T ============================
        // Thread (TMEM lane n = row, column half grp).  Each thread only writes tensor-
        // memory cells of its own lane inside the column range it has just read itself.
        const int grp = (warp - 1) >> 2;
        auto pack16 = [](const float* v, uint32_t (&w)[16]) {
#pragma unroll
            for (int i = 0; i < 16; ++i) w[i] = pack_f16x2(v[2 * i], v[2 * i + 1]);
        };
        // ---- W rows of chunk c from W^T in tensor memory (lane d, column i), tokens of
        // half grp: 16x256b loads hand each thread fp16-packable pairs of the 8x8 tiles
        // (d rows, i columns) that stmatrix.trans stores as rows i of 8 consecutive d --
        // 16-byte operand chunks.  Made visible to the tensor core; the caller's next
        // rdy3 arrival publishes them.
        const int mj = lane >> 3, rho = lane & 7;   // stmatrix tile and row this lane addresses
        float s0max = 0.f;     // largest |S0| element this thread loaded
        float nfacc = 0.f;     // NaN once a non-finite final-state element passed this thread
        auto ep2a_work = [&](int c) -> bool {
            if (!wait(m_w, c & 1)) return false;
            tc_fence_after();
            const uint32_t wbase = smem_u32(sm + (c % 3) * kSlotBytes + kSlotBlk + kBlkW);
#pragma unroll
            for (int lh = 0; lh < 32; lh += 16) {
                uint32_t r[2][8];   // both 16-column blocks of this half in flight at once
#pragma unroll
                for (int h = 0; h < 2; ++h) tmem_ld_16x256b_x2(taddr(tb, q4 * 32 + lh, kColW + grp * 32 + 16 * h), r[h]);
                tmem_ld_wait();
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    // tiles: columns cb..cb+7 lanes +0..7 | +8..15, columns cb+8.. the same
                    const int cb = grp * 32 + 16 * h;
                    const uint32_t m0 = pack_f16x2(__uint_as_float(r[h][0]), __uint_as_float(r[h][1]));
                    const uint32_t m1 = pack_f16x2(__uint_as_float(r[h][2]), __uint_as_float(r[h][3]));
                    const uint32_t m2 = pack_f16x2(__uint_as_float(r[h][4]), __uint_as_float(r[h][5]));
                    const uint32_t m3t = pack_f16x2(__uint_as_float(r[h][6]), __uint_as_float(r[h][7]));
                    const int i = cb + 8 * (mj >> 1) + rho;
                    const int d0 = q4 * 32 + lh + (mj & 1) * 8;
                    stmatrix_x4_trans(wbase + (d0 >> 6) * kBlkStride + sw128(i, d0 & 63), m0, m1, m2, m3t);
                }
            }
            fence_async_smem();
            return true;
        };
        {   // initial state S^T[n][d] (fp32) and its fp16 copy in U buffer 1 (read by MMA3(0))
            const int db = grp * 64;
            float v[64];
#pragma unroll
            for (int i = 0; i < 64; ++i) {
                // (values all zero: the segment-parallel P pass, which always starts from I)
                v[i] = kZeroV ? (db + i == row ? 1.f : 0.f)
                              : (a.S0 ? a.S0[((size_t)bh * 128 + db + i) * 128 + row] : 0.f);
                s0max = fmaxf(s0max, fabsf(v[i]));
            }
            if (kRec && dbg_in(a.rec_S + (size_t)bh * NC * 16384, 65536, a.rec_S, (size_t)a.BH * NC * 65536,
                               &g_tc_status)) {
                if constexpr (kRec == 2) {
                    unsigned char* img = (unsigned char*)(a.rec_S + (size_t)bh * NC * 16384);
#pragma unroll
                    for (int i = 0; i < 64; ++i)
                        *reinterpret_cast<__half*>(img + img_off(db + i, row, 128)) = __float2half_rn(v[i]);
                } else {
#pragma unroll
                    for (int i = 0; i < 64; ++i) a.rec_S[(size_t)bh * NC * 16384 + (db + i) * 128 + row] = v[i];
                }
            }
#pragma unroll
            for (int c0 = 0; c0 < 64; c0 += 16)
                tmem_st16(taddr(tb, q4 * 32, kColS + db + c0), *reinterpret_cast<float(*)[16]>(v + c0));
            uint32_t w[16];
            pack16(v, w);
            tmem_st16u(taddr(tb, q4 * 32, kColU + 64 + grp * 32), w);
            pack16(v + 32, w);
            tmem_st16u(taddr(tb, q4 * 32, kColU + 64 + grp * 32 + 16), w);
            tmem_st_wait();
        }
        if (ep2a_work(0)) {
            tc_fence_before();
            mbar_arrive(rdy3);
        }
        for (int c = 0; c < NC; ++c) {
            const uint32_t par = c & 1;
            const int nv = min(64, L - c * 64);
            const size_t tok0 = seq_tok + (size_t)c * 64;
            const uint32_t ucol = kColU + (c & 1) * 64;
            // ---- ep4: Up^T[n][i] = U^T - (W S)^T for tokens i in [32 grp, 32 grp + 32),
            //      packed fp16 into X columns [32 grp, 32 grp + 16)
            if (!wait(m3, par)) break;
            tc_fence_after();
            float u[32];   // this thread's U' values (recorded after the hand-off below)
            {
                const int cbeg = grp * 32;
                float d[32];
                tmem_ld16(taddr(tb, q4 * 32, ucol + cbeg), *reinterpret_cast<float(*)[16]>(u));
                tmem_ld16(taddr(tb, q4 * 32, ucol + cbeg + 16), *reinterpret_cast<float(*)[16]>(u + 16));
                tmem_ld16(taddr(tb, q4 * 32, kColX + cbeg), *reinterpret_cast<float(*)[16]>(d));
                tmem_ld16(taddr(tb, q4 * 32, kColX + cbeg + 16), *reinterpret_cast<float(*)[16]>(d + 16));
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 32; ++i) u[i] -= d[i];
                uint32_t w[16];
                pack16(u, w);
                tmem_st16u(taddr(tb, q4 * 32, up_pack_col<kRec>(grp)), w);
                tmem_st_wait();
            }
            tc_fence_before();
            mbar_arrive(rdy5);
            if (kRec == 2 && tid == 32 && c > 0) {   // chunk c-1's images have left slot (c-1) mod 3
                bulk_wait_read();
                mbar_arrive(&st_free[(c - 1) % 3]);
            }
            if (kRec == 1 && dbg_in(a.rec_Up + ((size_t)bh * NC + c) * 8192, 32768, a.rec_Up,
                                    (size_t)a.BH * NC * 32768, &g_tc_status)) {   // off the chain: MMA5(c) is released
                if constexpr (kRec == 1) {   // (kRec == 2: the image leaves with S_{c+1}'s, below)
                    float* up = a.rec_Up + ((size_t)bh * NC + c) * 8192 + (size_t)(grp * 32) * 128 + row;
#pragma unroll
                    for (int i = 0; i < 32; ++i) __stcs(up + i * 128, u[i]);
                }
            }
            // ---- W rows of chunk c+1 while MMA5(c) runs (W(c+1) precedes it on the tensor pipe)
            if (c + 1 < NC && !ep2a_work(c + 1)) break;
            // ---- ep6: S^T -> fp16 copy in U buffer c&1 (this thread's half of it); O -> global
            if (!wait(m5, par)) break;
            tc_fence_after();
            {
                const int cbeg = grp * 32;
                {
                    float sv[64];
#pragma unroll
                    for (int c0 = 0; c0 < 64; c0 += 16)
                        tmem_ld16(taddr(tb, q4 * 32, kColS + grp * 64 + c0), *reinterpret_cast<float(*)[16]>(sv + c0));
                    tmem_ld_wait();
                    uint32_t w[16];
                    pack16(sv, w);
                    tmem_st16u(taddr(tb, q4 * 32, ucol + grp * 32), w);
                    pack16(sv + 32, w);
                    tmem_st16u(taddr(tb, q4 * 32, ucol + grp * 32 + 16), w);
                }
                float v[32];
                tmem_ld16(taddr(tb, q4 * 32, kColO + cbeg), *reinterpret_cast<float(*)[16]>(v));
                tmem_ld16(taddr(tb, q4 * 32, kColO + cbeg + 16), *reinterpret_cast<float(*)[16]>(v + 16));
                tmem_ld_wait();
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(rdy3);
                const size_t oes = a.out_bf16 ? 2 : 4;
                if (!a.o) {
                    // the outputs are not wanted (a recording run for the backward, or the
                    // P and Q passes of the segment-parallel form)
                } else if (!dbg_in((char*)a.o + tok0 * 128 * oes, (size_t)nv * 128 * oes, a.o,
                                   (size_t)a.BH * L * 128 * oes, &g_tc_status)) {
                    // a debug build found this chunk's rows outside o: skipped
                } else if (a.out_bf16) {
                    __nv_bfloat16* op = (__nv_bfloat16*)a.o;
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (cbeg + i < nv) op[(tok0 + cbeg + i) * 128 + row] = __float2bfloat16_rn(v[i]);
                } else {
                    float* op = (float*)a.o;
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (cbeg + i < nv) op[(tok0 + cbeg + i) * 128 + row] = v[i];
                }
                if (kRec == 1 && c + 1 < NC &&
                    dbg_in(a.rec_S + ((size_t)bh * NC + c + 1) * 16384, 65536, a.rec_S, (size_t)a.BH * NC * 65536,
                           &g_tc_status)) {
                    // the state entering chunk c + 1, off the chain: S^T in tensor memory
                    // changes only in MMA5(c + 1), which waits for this thread's next arrival
                    // on rdy5 (after these reads)
                    float* rs = a.rec_S + ((size_t)bh * NC + c + 1) * 16384 + (size_t)(grp * 64) * 128 + row;
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        float sv[32];
                        tmem_ld16(taddr(tb, q4 * 32, kColS + grp * 64 + 32 * hh), *reinterpret_cast<float(*)[16]>(sv));
                        tmem_ld16(taddr(tb, q4 * 32, kColS + grp * 64 + 32 * hh + 16),
                                  *reinterpret_cast<float(*)[16]>(sv + 16));
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) __stcs(rs + (32 * hh + i) * 128, sv[i]);
                    }
                }
                if constexpr (kRec == 2) {
                    // The record as fp16 images: the state entering chunk c+1 (the fp16 copy
                    // just made, read by MMA3(c+1) and overwritten by U(c+2), after this
                    // thread's next rdy5 arrival) and chunk c's U' (packed at kColUp, rewritten
                    // by this thread's next Up epilogue), built with stmatrix.trans from 16x256b
                    // fragments (as the reverse scan builds its images) in the d-blocks of slot
                    // c mod 3, free since MMA5(c); one bulk copy each.  The slot goes back to
                    // E2 once the copies have read it (st_free, after the next Up epilogue).
                    const uint32_t base = smem_u32(sm + (c % 3) * kSlotBytes + kSlotBlk);
                    const int off = 4 * (rho >> 1) + (rho & 1) + 2 * (mj & 1);
#pragma unroll
                    for (int lh = 0; lh < 32; lh += 16) {
                        const int n0 = q4 * 32 + lh + 8 * (mj >> 1);
                        const uint32_t nb = (uint32_t)(n0 >> 6);
                        if (c + 1 < NC) {
                            uint32_t r[16];
                            tmem_ld_16x256b_x4(taddr(tb, q4 * 32 + lh, ucol + grp * 32), r);
                            tmem_ld_wait();
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                stmatrix_x4_trans(base + nb * 16384u + sw128(grp * 64 + 16 * k + off, n0 & 63), r[4 * k],
                                                  r[4 * k + 1], r[4 * k + 2], r[4 * k + 3]);
                        }
                        uint32_t r2[8];
                        tmem_ld_16x256b_x2(taddr(tb, q4 * 32 + lh, kColUp + grp * 16), r2);
                        tmem_ld_wait();
#pragma unroll
                        for (int k = 0; k < 2; ++k)
                            stmatrix_x4_trans(base + 32768u + nb * 8192u + sw128(grp * 32 + 16 * k + off, n0 & 63),
                                              r2[4 * k], r2[4 * k + 1], r2[4 * k + 2], r2[4 * k + 3]);
                    }
                    fence_async_smem();
                    group_sync(7, 256);
                    if (tid == 32) {
                        const size_t ch = (size_t)bh * NC + c;
                        const uint32_t sb = (uint32_t)(c % 3) * kSlotBytes + kSlotBlk;
                        if (c + 1 < NC && dbg_in(a.rec_S + (ch + 1) * 16384, 32768, a.rec_S,
                                                 (size_t)a.BH * NC * 65536, &g_tc_status))
                            bulk_s2g(a.rec_S + (ch + 1) * 16384, sm + sb, 32768u);
                        if (dbg_in(a.rec_Up + ch * 8192, 16384, a.rec_Up, (size_t)a.BH * NC * 32768, &g_tc_status))
                            bulk_s2g(a.rec_Up + ch * 8192, sm + sb + 32768, 16384u);
                        bulk_commit();
                    }
                }
            }
        }
        // ---- final state S^T[n][d] -> S_final[d][n], checked for non-finite values on the
        // way; then the staging checks (with the input maxima of E2 and B, after their arrival
        // on named barrier 5) decide whether the sequence is recomputed in fp32.  When S_final
        // aliases S0 the store waits for that decision (a recomputation re-reads S0).
        const bool ran = !*s_abort;
        const int db = grp * 64;
        const bool in_place = a.S_final && a.S_final == a.S0 && !a.seq_bad;
        if (ran) {
            tc_fence_after();
            float v[64];
#pragma unroll
            for (int c0 = 0; c0 < 64; c0 += 16)
                tmem_ld16(taddr(tb, q4 * 32, kColS + db + c0), *reinterpret_cast<float(*)[16]>(v + c0));
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 64; ++i) nonfinite_acc(nfacc, v[i]);
            if (a.S_final && !in_place &&
                dbg_in(a.S_final + (size_t)bh * 16384, 65536, a.S_final, (size_t)a.BH * 65536, &g_tc_status)) {
#pragma unroll
                for (int i = 0; i < 64; ++i) a.S_final[((size_t)bh * 128 + db + i) * 128 + row] = v[i];
            }
        }
        if (__any_sync(0xffffffffu, nfacc != 0.f) && lane == 0) atomicOr(&s_stat[0], 1u);
        const unsigned wmax = __reduce_max_sync(0xffffffffu, __float_as_uint(s0max));
        if (lane == 0) atomicMax(&s_stat[3], wmax);
        group_sync(5, 544);
        const bool redo = ran && ((s_stat[0] & 1u) ||
                                  staging_out_of_range(__uint_as_float(s_stat[1]), __uint_as_float(s_stat[2]),
                                                       __uint_as_float(s_stat[3])));
        if (redo && tid == 32) {
            if (a.seq_bad) atomicOr(&a.seq_bad[blockIdx.x / a.nseg], 1);
            else s_stat[0] |= 2u;   // read after the teardown barrier
        }
        if (ran && in_place && !redo &&
            dbg_in(a.S_final + (size_t)bh * 16384, 65536, a.S_final, (size_t)a.BH * 65536, &g_tc_status)) {
            for (int c0 = 0; c0 < 64; c0 += 16) {
                float v[16];
                tmem_ld16(taddr(tb, q4 * 32, kColS + db + c0), v);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 16; ++i) a.S_final[((size_t)bh * 128 + db + c0 + i) * 128 + row] = v[i];
            }
        }
    } else if (warp >= 9 && warp <= 18 && (warp & 3) != 0) {
        // ============================ E2: operands ============================
        // ---- inputs.  Thread et owns 16-byte chunk ch = et & 15 (8 elements of d, or of
        // n for V) of rows rs + 16 mm (rs = et >> 4, mm = 0..3) of each of K, Q, V: a warp
        // reads two consecutive 256-byte rows per load.  Its swizzled chunk position
        // (ch & 7) ^ (row & 7) is the same for all four rows, so every store is a
        // per-thread base plus a compile-time offset.
        const int w9 = warp - 9, et = (w9 - (w9 >> 2)) * 32 + lane;   // 0..255
        const int cch = et & 15, rs = et >> 4;
        const uint32_t pos = (uint32_t)((((cch & 7) ^ (rs & 7)) << 4) + rs * 128);
        const uint32_t dblk = kSlotBlk + (cch >> 3) * kBlkStride + pos;
        const uint32_t dK = dblk + kBlkK, dQ = dblk + kBlkQ;
        const uint32_t dV = kVTV + (cch >> 3) * 8192u + pos;
        // Without an output (the segment passes that only carry the state, the recording runs)
        // Q feeds only the unread O^T columns: its rows are not read (the tile stays zero)
        const bool no_o = a.o == nullptr;
        uint4 raw[12];
        // global loads of rows of chunk c (zero past the end of the sequence): K and Q
        // (which = 0, 1) or V (which = 2).  Consumed only by store(), so their latency
        // overlaps the work on the chunks before it.
        auto load = [&](int c, int w0, int w1) {
            const int nv = min(64, L - c * 64);
            const size_t tok = seq_tok + (size_t)c * 64 + rs;
#pragma unroll
            for (int which = w0; which < w1; ++which) {
                const __nv_bfloat16* src = which == 0 ? a.k : (which == 1 ? a.q : a.v);
#pragma unroll
                for (int mm = 0; mm < 4; ++mm)
                    raw[which * 4 + mm] =
                        (rs + 16 * mm < nv && !(kZeroV && which == 2) && !(no_o && which == 1))
                            ? __ldcs(reinterpret_cast<const uint4*>(src + (tok + 16 * mm) * 128) + cch)
                            : make_uint4(0, 0, 0, 0);
            }
        };
        // fp16 operand tiles of chunk c into slot c mod 3 and V/Ta buffer c mod 2
        float vmax = 0.f;   // largest |v| element this thread converted
        auto store = [&](int c) {
            const int si = c % 3;
            const uint32_t sb = (uint32_t)si * kSlotBytes, vb = kOffVT + (uint32_t)(c & 1) * kVTBytes;
#pragma unroll
            for (int which = 0; which < 3; ++which)
#pragma unroll
                for (int mm = 0; mm < 4; ++mm) {
                    const uint32_t dst = (which == 0 ? sb + dK : (which == 1 ? sb + dQ : vb + dV)) + mm * 2048;
                    *reinterpret_cast<uint4*>(sm + dst) =
                        which == 2 ? bf16x8_to_f16x8_max(raw[which * 4 + mm], vmax) : bf16x8_to_f16x8(raw[which * 4 + mm]);
                }
            fence_async_smem();
            mbar_arrive(&ops_full[si]);   // all E2 threads, after their own stores
        };
        load(0, 0, 3);
        store(0);
        for (int c = 1; c < 3 && c < NC; ++c) {
            load(c, 0, 3);
            // V/Ta buffer c mod 2 is free once U(c-2) is done
            if (c >= 2 && !wait(&vt_free[c & 1], ((c - 2) >> 1) & 1)) break;
            store(c);
        }
        if (NC > 3) load(3, 0, 3);
        for (int c = 0; c + 3 < NC; ++c) {
            {
                // slot (c+3) mod 3 is free once MMA5(c) is done (with image records: once
                // chunk c's images staged there are read out), V/Ta buffer (c+3) mod 2 once
                // U(c+1) is (issued right after MMA5(c))
                if (!wait(kRec == 2 ? &st_free[c % 3] : &ops_empty[c % 3], (c / 3) & 1)) break;
                if (!wait(&vt_free[(c + 1) & 1], ((c + 1) >> 1) & 1)) break;
                store(c + 3);
                if (c + 4 < NC) load(c + 4, 0, 3);
                if (et == 0 && c + 6 < NC) {   // rows two chunks beyond those toward L2: the register loads hit it
                    const size_t r0 = (seq_tok + (size_t)(c + 6) * 64) * 128;
                    const uint32_t bytes = (uint32_t)min(64, L - (c + 6) * 64) * 256u;
                    bulk_prefetch_l2(a.k + r0, bytes);
                    if (!no_o) bulk_prefetch_l2(a.q + r0, bytes);
                    if (!kZeroV) bulk_prefetch_l2(a.v + r0, bytes);
                }
            }
        }
        // |v| maximum for the staging checks; then E1 (waiting on named barrier 5) may read it
        {
            const unsigned wm = __reduce_max_sync(0xffffffffu, __float_as_uint(vmax));
            if (lane == 0) atomicMax(&s_stat[3], wm);
        }
        asm volatile("bar.arrive 5, 544;" ::: "memory");
    } else if (warp == 19) {
        // ============================ B: image copies ============================
        // (also gathers the chunks' largest key and query norms for the staging checks)
        if (lane == 0) {
            for (int c = 0; c < NC; ++c) {
                const int si = c % 3;
                // slot c mod 3 is free once MMA5(c-3) is done, V/Ta buffer c mod 2 once U(c-2) is
                if (c >= 3 && !wait(&ops_empty[si], ((c - 3) / 3) & 1)) break;
                if (c >= 2 && !wait(&vt_free[c & 1], ((c - 2) >> 1) & 1)) break;
                if (a.flags) {   // fused launch: wait (bounded) until chunk c's images are published
                    const int* f = a.flags + (size_t)bh * NC + c;
                    uint32_t n = 0;
                    while (ld_acquire_gpu(f) == 0 && ++n < kFlagPollLimit && !*s_abort) __nanosleep(64);
                    if (n >= kFlagPollLimit || *s_abort) {
                        *s_abort = 1;
                        break;
                    }
                    fence_proxy_async_global();
                }
                // (without an output, P^T only feeds the unread O^T columns of MMA5: not copied)
                mbar_arrive_expect_tx(&ops_full[si], a.o ? 16384u : 8192u);
                bulk_g2s(sm + kOffVT + (c & 1) * kVTBytes + kVTTa, a.Ta + ((size_t)bh * NC + c) * 4096, 8192u,
                         &ops_full[si]);
                if (a.o)
                    bulk_g2s(sm + si * kSlotBytes + kSlotPt, a.Pt + ((size_t)bh * NC + c) * 4096, 8192u,
                             &ops_full[si]);
            }
        }
        // the chunks' largest key and query norms, read once every flag has been acquired
        // (the warp barrier orders lane 0's acquires before the other lanes' reads)
        __syncwarp();
        if (!*s_abort) {
            float mk2 = 0.f, mq2 = 0.f;
            for (int c = lane; c < NC; c += 32) {
                const float2 nq = *reinterpret_cast<const float2*>(a.prep.cnorm + ((size_t)bh * NC + c) * 2);
                mk2 = fmaxf(mk2, nq.x);
                mq2 = fmaxf(mq2, nq.y);
            }
            const unsigned k2 = __reduce_max_sync(0xffffffffu, __float_as_uint(mk2));
            const unsigned q2 = __reduce_max_sync(0xffffffffu, __float_as_uint(mq2));
            if (lane == 0) {
                s_stat[1] = k2;
                s_stat[2] = q2;
            }
        }
        asm volatile("bar.arrive 5, 544;" ::: "memory");
    } else if (warp == 0 && lane == 0) {
        // ============================ M: MMA issue ============================
        const uint32_t id_kk128 = idesc_f16(128, 128);
        const uint32_t id_mk64 = idesc_f16(128, 64, true, false);
        const uint32_t id_km192 = idesc_f16(128, 192, false, true);
        auto slot_at = [&](int c) { return smem_u32(sm + (c % 3) * kSlotBytes); };
        auto vt_at = [&](int c) { return smem_u32(sm + kOffVT + (c & 1) * kVTBytes); };
        auto mma_w = [&](int c) {     // W^T = K^T Ta^T
            const uint32_t s0 = slot_at(c), ta = vt_at(c) + kVTTa;
            for (int s = 0; s < 4; ++s)
                mma_f16_ss(tb + kColW, sdesc_sw128(s0 + kSlotBlk + kBlkK + s * 2048, kBlkStride),
                           sdesc_sw128(ta + s * 32), id_mk64, s > 0);
            mma_commit(m_w);
        };
        auto mma_u = [&](int c) {     // U^T = V^T Ta^T; the V/Ta buffer is free after it
            const uint32_t vt = vt_at(c), ta = vt + kVTTa;
            for (int s = 0; s < 4; ++s)
                mma_f16_ss(tb + kColU + (c & 1) * 64, sdesc_sw128(vt + kVTV + s * 2048, 8192),
                           sdesc_sw128(ta + s * 32), id_mk64, s > 0);
            mma_commit(&vt_free[c & 1]);
        };
        if (wait(&ops_full[0], 0)) {
            tc_fence_after();
            mma_w(0);
            mma_u(0);
        }
        for (int c = 0; c < NC; ++c) {
            const uint32_t s0 = slot_at(c);
            // MMA3(c): [(W S)^T | (Q S)^T] = S^T [W; Q]^T; S^T (fp16) from tensor memory
            if (!wait(rdy3, c & 1)) break;
            tc_fence_after();
            const uint32_t scol = kColU + ((c + 1) & 1) * 64;
            for (int s = 0; s < 8; ++s)
                mma_f16_ts(tb + kColX, tb + scol + 8 * s,
                           sdesc_sw128(s0 + kSlotBlk + (s / 4) * kBlkStride + kBlkW + (s % 4) * 32),
                           id_kk128, s > 0);
            mma_commit(m3);
            // W(c+1) fills the tensor pipe while E1 computes Up
            if (c + 1 < NC) {
                if (!wait(&ops_full[(c + 1) % 3], ((c + 1) / 3) & 1)) break;
                tc_fence_after();
                mma_w(c + 1);
            }
            // MMA5(c): [O^T | S^T] += Up^T [P^T | K]; Up^T (fp16) from tensor memory
            if (!wait(rdy5, c & 1)) break;
            tc_fence_after();
            for (int s = 0; s < 4; ++s)
                mma_f16_ts(tb + kColO, tb + up_col<kRec>(s), sdesc_sw128(s0 + kSlotPt + s * 2048, kBlkStride),
                           id_km192, 1u);
            mma_commit(m5);
            mma_commit(&ops_empty[c % 3]);
            // U(c+1) fills it while E1 copies S^T and reads O
            if (c + 1 < NC) mma_u(c + 1);
        }
    }

    // ---- teardown: every thread arrives here (record image copies complete first)
    if (kRec == 2 && tid == 32) bulk_wait_all();
    __syncthreads();
    if (*s_abort) {
        if (tid == 0) record_timeout();
        // drain: a commit after all issued MMAs, awaited with a bound, then the copies
        if (warp == 0 && lane == 0) {
            mma_commit(m5);
        }
        __syncthreads();
        mbar_wait(m5, 0, kWaitLimit);   // either parity completing ends the drain
        mbar_wait(m5, 1, kWaitLimit);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tb, 512);
    // ---- a sequence the fp16 staging could not represent: recompute it token by token in
    // fp32 (o and S_final overwritten; S_final was not written, so an aliased S0 is intact)
    const size_t ob = a.out_bf16 ? 2 : 4;
    if ((s_stat[0] & 2u) && tid < kRecThreads &&
        (!a.o || dbg_in((char*)a.o + seq_tok * 128 * ob, (size_t)L * 128 * ob, a.o, (size_t)a.BH * L * 128 * ob,
                        &g_tc_status)) &&
        (!a.S_final || dbg_in(a.S_final + (size_t)bh * 16384, 65536, a.S_final, (size_t)a.BH * 65536, &g_tc_status)) &&
        (!kRec || (dbg_in(a.rec_S + (size_t)bh * NC * 16384, (size_t)NC * 65536, a.rec_S, (size_t)a.BH * NC * 65536,
                          &g_tc_status) &&
                   dbg_in(a.rec_Up + (size_t)bh * NC * 8192, (size_t)NC * 32768, a.rec_Up,
                          (size_t)a.BH * NC * 32768, &g_tc_status)))) {
        seq_recurrent_fp32(a.q + seq_tok * 128, a.k + seq_tok * 128, a.v + seq_tok * 128, a.prep.beta + seq_tok,
                           a.S0 ? a.S0 + (size_t)bh * 16384 : nullptr, a.o ? (char*)a.o + seq_tok * 128 * ob : nullptr,
                           a.out_bf16,
                           a.S_final ? a.S_final + (size_t)bh * 16384 : nullptr, L, a.prep.euler,
                           reinterpret_cast<float*>(sm), tid, 6,
                           kRec ? a.rec_S + (size_t)bh * NC * 16384 : nullptr,
                           kRec ? a.rec_Up + (size_t)bh * NC * 8192 : nullptr);
        if (kRec == 2 && tid == 0) a.rec_fp32[bh] = 1;   // this sequence's record is fp32
    }
}

cudaError_t launch_tmat(const Dims& d, const CUtensorMap* tm_k, const CUtensorMap* tm_q, const TmatArgs& ta,
                        cudaStream_t st) {
    cudaError_t e = cudaFuncSetAttribute(k_tmat, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTmatSmem);
    if (e != cudaSuccess) return e;
    k_tmat<<<dim3((unsigned)d.BH(), (unsigned)d.NC), kTmThreads, kTmatSmem, st>>>(*tm_k, *tm_q, ta);
    prof_mark("efla_tc_tmat", st);
    return cudaGetLastError();
}

// ================================================================ launch
// Ta images then P^T images, [BH][NC][64*64] fp16 each, then the image-ready flags [BH][NC]
static size_t images_bytes(const Dims& d) { return align256((size_t)d.BH() * d.NC * 4096 * 2 * 2); }

// ------------------------------------------------------- segment-parallel forward
// A few long sequences leave most SMs idle while each sequence CTA walks its chunks one
// after another.  Over a segment of its chunks the state map is affine,
// S_end = P S_start + Q (P the product of the tokens' I - alpha k k^T, Q the end state
// reached from zero), so a sequence of nseg segments runs as nseg independent sequences:
//   1. the preparation images of every chunk (they depend on k, q, beta only), once;
//   2. every segment with v = 0 (k_fwd_tc<true>) from S0 = I  -> P   (d_k = d_v, so I is
//      a valid state);
//   3. every segment from S0 = 0             -> Q;
//   4. k_seg_combine, sequential over a sequence's segments in fp32:
//      S_start(0) = S0, S_start(s + 1) = P_s S_start(s) + Q_s; the last is S_final;
//   5. every segment from S_start(s), writing o.
// P comes from its own pass (not as the difference of a pass from I and one from 0), so
// its rounding error is relative to P itself.
// Only pass 5 writes o.  Segments are whole chunks, so
// [B, H, L, d] is read as [B, H nseg, L / nseg, d] with no copy.
constexpr int kSegCtas = 128;   // sequence CTAs the segments aim to fill

int fwd_tc_segments(const Dims& d) {
    if (!fwd_tc_supported(d) || d.L % 64 || d.NC < 256 || d.BH() > kSegCtas / 4) return 1;
    int n = 1;
    while (d.BH() * n * 2 <= kSegCtas && d.NC % (n * 2) == 0 && d.NC / (n * 2) >= 16) n *= 2;
    return n >= 4 ? n : 1;
}

static Dims seg_dims(const Dims& d, int nseg) {
    Dims s = d;
    s.H = d.H * nseg;
    s.L = d.L / nseg;
    s.NC = d.NC / nseg;
    return s;
}

static size_t seg_states_bytes(const Dims& d, int nseg) { return align256((size_t)d.BH() * nseg * 128 * 128 * 4); }

// Chunk-level arrays after the images: the image-ready flags [BH][NC] int and the chunks'
// largest key and query norms [BH][NC][2] fp32.
static size_t chunk_arrays_bytes(const Dims& d) {
    return align256((size_t)d.BH() * d.NC * sizeof(int)) + align256((size_t)d.BH() * d.NC * 2 * sizeof(float));
}
static float* cnorm_of(const Dims& d, void* ws) {
    return (float*)((char*)ws + images_bytes(d) + align256((size_t)d.BH() * d.NC * sizeof(int)));
}

// Segment-parallel workspace after those: three [BH nseg][128][128] fp32 arrays (I then
// S_start; P; Q), the final states [BH][128][128] fp32, and one out-of-range word per
// sequence.
size_t fwd_tc_ws_bytes(const Dims& d) {
    size_t n = images_bytes(d) + chunk_arrays_bytes(d);
    const int nseg = fwd_tc_segments(d);
    if (nseg > 1)
        n += 3 * seg_states_bytes(d, nseg) + seg_states_bytes(d, 1) + align256((size_t)d.BH() * sizeof(int));
    return n;
}

// Last step of the segment-parallel form, one CTA per sequence: a sequence whose staging
// went out of range in any pass is recomputed in fp32 from S0 (still intact: the chained
// final states went to the workspace); every other one copies its final state out.
struct SegFinishArgs {
    const __nv_bfloat16* q;
    const __nv_bfloat16* k;
    const __nv_bfloat16* v;
    const float* beta;
    const float* S0;
    const float* S_end;
    const int* seq_bad;
    void* o;
    float* S_final;
    float* rec_S;    // chunk-state record or null
    float* rec_Up;
    int L, NC, out_bf16, euler;
};

__global__ void __launch_bounds__(kRecThreads, 1) k_seg_finish(SegFinishArgs f) {
    __shared__ float smf[kRecSmemFloats];
    const long long bh = blockIdx.x;
    const size_t tok = (size_t)bh * f.L;
    if (f.seq_bad[bh]) {
        const size_t ob = f.out_bf16 ? 2 : 4;
        seq_recurrent_fp32(f.q + tok * 128, f.k + tok * 128, f.v + tok * 128, f.beta + tok,
                           f.S0 ? f.S0 + bh * 16384 : nullptr, (char*)f.o + tok * 128 * ob, f.out_bf16,
                           f.S_final ? f.S_final + bh * 16384 : nullptr, f.L, f.euler, smf, threadIdx.x, 1,
                           f.rec_S ? f.rec_S + bh * f.NC * 16384 : nullptr,
                           f.rec_S ? f.rec_Up + bh * f.NC * 8192 : nullptr);
        return;
    }
    if (f.S_final) {
        const float4* src = reinterpret_cast<const float4*>(f.S_end + bh * 16384);
        float4* dst = reinterpret_cast<float4*>(f.S_final + bh * 16384);
        for (int i = threadIdx.x; i < 4096; i += kRecThreads) dst[i] = src[i];
    }
}

// One CTA per (sequence, 16 state columns).  P_s is loaded whole into shared memory for
// each segment; the slice S[:, n0 .. n0 + 15] is advanced through the segments.
constexpr int kCbCols = 16;
constexpr int kCbLdp = 132;   // 16-byte rows (cp.async granules); row reads at most 2-way bank conflicts
constexpr size_t kCbSmem = (size_t)(2 * 128 * kCbLdp + 128 * kCbCols) * sizeof(float);

__device__ __forceinline__ void cpa16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cpa_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cpa_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// S_start(0) = S0, S_start(s + 1) = P_s S_start(s) + Q_s over a sequence's segments, in
// fp32, one CTA per sequence and 16-column slice of the state (the columns are
// independent).  P_{s+1} is copied into the second of two shared buffers (cp.async) while
// the product with P_s runs.
__global__ void __launch_bounds__(256) k_seg_combine(const float* __restrict__ P, const float* __restrict__ Q,
                                                     const float* S0, float* __restrict__ Sstart,
                                                     float* S_final, int nseg) {
    extern __shared__ __align__(16) float smc[];
    float* Ss = smc + 2 * 128 * kCbLdp;           // [128][16] state slice, after two [128][kCbLdp] P buffers
    auto pbuf = [&](int i) { return smc + i * 128 * kCbLdp; };
    const long long bh = blockIdx.x;
    const int n0 = blockIdx.y * kCbCols, tid = threadIdx.x;
    const int x = tid >> 1, c0 = (tid & 1) * 8;   // this thread: row x, columns c0 .. c0 + 7
    auto load_P = [&](int s, float* dst) {        // 128 rows x 32 granules of 16 bytes
        const float* Pg = P + ((size_t)bh * nseg + s) * 16384;
        for (int e = tid; e < 128 * 32; e += 256) {
            const int r = e >> 5, g = e & 31;
            cpa16(dst + r * kCbLdp + 4 * g, Pg + r * 128 + 4 * g);
        }
        cpa_commit();
    };
    load_P(0, pbuf(0));
    for (int e = tid; e < 128 * kCbCols; e += 256) {
        const int r = e >> 4, cc = e & 15;
        Ss[e] = S0 ? S0[((size_t)bh * 128 + r) * 128 + n0 + cc] : 0.f;
    }
    for (int s = 0; s < nseg; ++s) {
        const size_t seg = (size_t)bh * nseg + s;
        const float* Qg = Q + seg * 16384;
        const float* Pm = pbuf(s & 1);
        if (s + 1 < nseg) load_P(s + 1, pbuf((s + 1) & 1));   // its buffer was last read in step s - 1
        else cpa_commit();                                    // (an empty group keeps the count)
        float acc[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) acc[j] = Qg[(size_t)x * 128 + n0 + c0 + j];
        cpa_wait<1>();     // this thread's part of P_s has landed
        __syncthreads();   // all of P_s and Ss are visible
        for (int e = tid; e < 128 * kCbCols; e += 256) {
            const int r = e >> 4, cc = e & 15;
            Sstart[seg * 16384 + (size_t)r * 128 + n0 + cc] = Ss[e];
        }
        for (int y = 0; y < 128; ++y) {
            const float p = Pm[x * kCbLdp + y];
            const float4 s0 = *reinterpret_cast<const float4*>(Ss + y * kCbCols + c0);
            const float4 s1 = *reinterpret_cast<const float4*>(Ss + y * kCbCols + c0 + 4);
            acc[0] = fmaf(p, s0.x, acc[0]); acc[1] = fmaf(p, s0.y, acc[1]);
            acc[2] = fmaf(p, s0.z, acc[2]); acc[3] = fmaf(p, s0.w, acc[3]);
            acc[4] = fmaf(p, s1.x, acc[4]); acc[5] = fmaf(p, s1.y, acc[5]);
            acc[6] = fmaf(p, s1.z, acc[6]); acc[7] = fmaf(p, s1.w, acc[7]);
        }
        __syncthreads();   // every thread has read Ss and P_s
#pragma unroll
        for (int j = 0; j < 8; ++j) Ss[x * kCbCols + c0 + j] = acc[j];
    }
    cpa_wait<0>();
    __syncthreads();
    if (S_final)
        for (int e = tid; e < 128 * kCbCols; e += 256) {
            const int r = e >> 4, cc = e & 15;
            S_final[((size_t)bh * 128 + r) * 128 + n0 + cc] = Ss[e];
        }
}

bool fwd_tc_supported(const Dims& d) {
    return d.in_bf16 && d.dk == 128 && d.dv == 128 && d.C == 64 && d.L > 0;
}

static cudaError_t launch_fwd_tc_segmented(const Dims& d, int nseg, const void* q, const void* k,
                                           const void* v, const float* beta, const float* S0, void* o,
                                           float* S_final, void* ws, cudaStream_t st, float* rec_S,
                                           float* rec_Up, float* rec_T, float* rec_alpha) {
    const Dims s = seg_dims(d, nseg);
    CUtensorMap tm_k, tm_q;
    cudaError_t e = bf16_rows_map(&tm_k, k, s);
    if (e == cudaSuccess) e = bf16_rows_map(&tm_q, q, s);
    if (e != cudaSuccess) return e;
    uint16_t* Ta = (uint16_t*)ws;
    uint16_t* Pt = Ta + (size_t)s.BH() * s.NC * 4096;
    char* p = (char*)ws + images_bytes(s) + chunk_arrays_bytes(s);
    float* Sst = (float*)p;                      // the segments' start states
    float* Pb = (float*)(p + seg_states_bytes(d, nseg));
    float* Qb = (float*)(p + 2 * seg_states_bytes(d, nseg));
    float* Se = (float*)(p + 3 * seg_states_bytes(d, nseg));
    int* bad = (int*)(p + 3 * seg_states_bytes(d, nseg) + seg_states_bytes(d, 1));
    const int BHs = (int)s.BH();
    TmatArgs ta{(const __nv_bfloat16*)k, (const __nv_bfloat16*)q, beta, Ta, Pt, cnorm_of(s, ws), rec_T, rec_alpha,
                s.L, s.NC, s.euler, s.BH() * s.NC};
    FwdTcArgs fa{(const __nv_bfloat16*)q, (const __nv_bfloat16*)k, (const __nv_bfloat16*)v, Ta, Pt,
                 Sst, o, Pb, nullptr, ta, bad, nullptr, nullptr, nullptr, s.L, s.NC, s.out_bf16, BHs, nseg};
    if ((e = cudaMemsetAsync(bad, 0, (size_t)d.BH() * sizeof(int), st)) != cudaSuccess) return e;
    if ((e = cudaFuncSetAttribute(k_tmat, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTmatSmem)) != cudaSuccess)
        return e;
    if ((e = cudaFuncSetAttribute(k_fwd_tc<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kFwdTcSmem)) != cudaSuccess)
        return e;
    if ((e = cudaFuncSetAttribute(k_fwd_tc<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kFwdTcSmem)) != cudaSuccess)
        return e;
    if (rec_S && (e = cudaFuncSetAttribute(k_fwd_tc<false, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)kFwdTcSmem)) != cudaSuccess)
        return e;
    if ((e = cudaFuncSetAttribute(k_seg_combine, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kCbSmem)) !=
        cudaSuccess)
        return e;
    k_tmat<<<dim3((unsigned)BHs, (unsigned)s.NC), kTmThreads, kTmatSmem, st>>>(tm_k, tm_q, ta);
    prof_mark("efla_tc_tmat", st);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    fa.o = nullptr;   // the P and Q passes write no o (the last pass writes it)
    fa.S0 = nullptr;  // (the P pass starts from I without reading a state)
    k_fwd_tc<true><<<(unsigned)BHs, kFwdThreads, kFwdTcSmem, st>>>(tm_k, tm_q, fa);   // P (v = 0)
    prof_mark("efla_tc_fwd", st);
    fa.S0 = nullptr;
    fa.S_final = Qb;
    k_fwd_tc<false><<<(unsigned)BHs, kFwdThreads, kFwdTcSmem, st>>>(tm_k, tm_q, fa);   // Q
    prof_mark("efla_tc_fwd", st);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    k_seg_combine<<<dim3((unsigned)d.BH(), 128 / kCbCols), 256, kCbSmem, st>>>(Pb, Qb, S0, Sst, Se, nseg);
    prof_mark("efla_seg_combine", st);
    fa.S0 = Sst;
    fa.S_final = nullptr;
    fa.o = o;
    if (rec_S) {   // o (and the chunk-state record: every chunk's entering state is known here)
        fa.rec_S = rec_S;
        fa.rec_Up = rec_Up;
        k_fwd_tc<false, 1><<<(unsigned)BHs, kFwdThreads, kFwdTcSmem, st>>>(tm_k, tm_q, fa);
    } else {
        k_fwd_tc<false><<<(unsigned)BHs, kFwdThreads, kFwdTcSmem, st>>>(tm_k, tm_q, fa);   // o
    }
    prof_mark("efla_tc_fwd", st);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    SegFinishArgs sf{(const __nv_bfloat16*)q, (const __nv_bfloat16*)k, (const __nv_bfloat16*)v, beta, S0, Se, bad,
                     o, S_final, rec_S, rec_Up, d.L, d.NC, d.out_bf16, d.euler};
    k_seg_finish<<<(unsigned)d.BH(), kRecThreads, 0, st>>>(sf);
    prof_mark("efla_seg_finish", st);
    return cudaGetLastError();
}

cudaError_t launch_tc_prep(const Dims& d, const void* q, const void* k, const float* beta, void* ws, float* rec_T,
                          float* rec_alpha, cudaStream_t st) {
    CUtensorMap tm_k, tm_q;
    cudaError_t e = bf16_rows_map(&tm_k, k, d);
    if (e == cudaSuccess) e = bf16_rows_map(&tm_q, q, d);
    if (e != cudaSuccess) return e;
    uint16_t* Ta = (uint16_t*)ws;
    uint16_t* Pt = Ta + (size_t)d.BH() * d.NC * 4096;
    TmatArgs ta{(const __nv_bfloat16*)k, (const __nv_bfloat16*)q, beta, Ta, Pt, cnorm_of(d, ws), rec_T, rec_alpha,
                d.L, d.NC, d.euler, d.BH() * d.NC};
    return launch_tmat(d, &tm_k, &tm_q, ta, st);
}

cudaError_t launch_fwd_tc(const Dims& d, const void* q, const void* k, const void* v,
                          const float* beta, const float* S0, void* o, float* S_final, void* ws,
                          cudaStream_t st, float* rec_S, float* rec_Up, float* rec_T, float* rec_alpha,
                          int* rec_fp32, bool prepared) {
    const int nseg = fwd_tc_segments(d);
    if (nseg > 1 && (rec_fp32 || prepared)) return cudaErrorInvalidValue;   // one-pass form only
    if (nseg > 1)
        return launch_fwd_tc_segmented(d, nseg, q, k, v, beta, S0, o, S_final, ws, st, rec_S, rec_Up, rec_T,
                                       rec_alpha);
    CUtensorMap tm_k, tm_q;
    cudaError_t e0 = bf16_rows_map(&tm_k, k, d);
    if (e0 == cudaSuccess) e0 = bf16_rows_map(&tm_q, q, d);
    if (e0 != cudaSuccess) return e0;
    uint16_t* Ta = (uint16_t*)ws;
    uint16_t* Pt = Ta + (size_t)d.BH() * d.NC * 4096;
    int* flags = (int*)((char*)ws + images_bytes(d));
    const int BH = (int)d.BH();
    TmatArgs ta{(const __nv_bfloat16*)k, (const __nv_bfloat16*)q, beta, Ta, Pt, cnorm_of(d, ws), rec_T, rec_alpha,
                d.L, d.NC, d.euler, d.BH() * d.NC};
    FwdTcArgs fa{(const __nv_bfloat16*)q, (const __nv_bfloat16*)k, (const __nv_bfloat16*)v, Ta, Pt,
                 S0, o, S_final, nullptr, ta, nullptr, rec_S, rec_Up, rec_fp32, d.L, d.NC, d.out_bf16, BH, 1};
    const void* kern = !rec_S ? (const void*)k_fwd_tc<false>
                              : rec_fp32 ? (const void*)k_fwd_tc<false, 2> : (const void*)k_fwd_tc<false, 1>;
    if (rec_fp32 && (e0 = cudaMemsetAsync(rec_fp32, 0, (size_t)BH * sizeof(int), st)) != cudaSuccess) return e0;
    cudaError_t e = cudaFuncSetAttribute(k_tmat, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTmatSmem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kFwdTcSmem);
    if (e != cudaSuccess) return e;
    // One cooperative launch when the sequences leave enough SMs for preparation CTAs
    // (co-residency of all CTAs is what makes waiting on their flags safe); else the
    // preparation kernel first, then the sequences.
    int dev = 0, nsm = 0, coop = 0, per_sm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev)) != cudaSuccess) return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kFwdThreads, kFwdTcSmem)) != cudaSuccess)
        return e;
    const int prep_ctas = nsm * per_sm - BH;
    if (!prepared && coop && prep_ctas >= kMinPrepCtas) {
        fa.flags = flags;
        const int nf = BH * d.NC;
        k_zero_flags<<<(unsigned)((nf + 255) / 256 < 64 ? (nf + 255) / 256 : 64), 256, 0, st>>>(flags, nf);
        prof_mark("efla_zero_flags", st);   // (with timing on, the event between them costs the overlap)
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        // cooperative (all CTAs co-resident: waiting on flags is safe) and a programmatic
        // dependent of the flag clearing (its set-up overlaps that kernel and the launch gap)
        void* args[] = {&tm_k, &tm_q, &fa};
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(BH + prep_ctas));
        cfg.blockDim = dim3(kFwdThreads);
        cfg.dynamicSmemBytes = kFwdTcSmem;
        cfg.stream = st;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 2;
        e = cudaLaunchKernelExC(&cfg, kern, args);
        prof_mark("efla_tc_fused", st);
        return e != cudaSuccess ? e : cudaGetLastError();
    }
    if (!prepared) {
        k_tmat<<<dim3((unsigned)BH, (unsigned)d.NC), kTmThreads, kTmatSmem, st>>>(tm_k, tm_q, ta);
        prof_mark("efla_tc_tmat", st);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    if (rec_S && rec_fp32)
        k_fwd_tc<false, 2><<<(unsigned)BH, kFwdThreads, kFwdTcSmem, st>>>(tm_k, tm_q, fa);
    else if (rec_S)
        k_fwd_tc<false, 1><<<(unsigned)BH, kFwdThreads, kFwdTcSmem, st>>>(tm_k, tm_q, fa);
    else
        k_fwd_tc<false><<<(unsigned)BH, kFwdThreads, kFwdTcSmem, st>>>(tm_k, tm_q, fa);
    if (!prepared) prof_mark("efla_tc_fwd", st);
    return cudaGetLastError();
}

// Diagnostic of the bounded waits: kind 0 waits on an mbarrier that never completes
// (one of its two arrivals), kind 1 polls a global flag that nothing sets; either gives
// up after `limit` polls and records the timeout in the status word, as the forward's
// own waits do.
__device__ int g_never_set = 0;

__global__ void k_wait_selftest(int kind, uint32_t limit) {
    __shared__ uint64_t bar;
    if (kind == 0) {
        mbar_init(&bar, 2);
        fence_mbar_init();
        mbar_arrive(&bar);
        if (!mbar_wait(&bar, 0, limit)) record_timeout();
    } else {
        uint32_t n = 0;
        while (ld_acquire_gpu(&g_never_set) == 0 && ++n < limit) __nanosleep(64);
        if (n >= limit) record_timeout();
    }
}

cudaError_t launch_wait_selftest(int kind, uint32_t limit, cudaStream_t st) {
    k_wait_selftest<<<1, 1, 0, st>>>(kind, limit);
    prof_mark("efla_wait_selftest", st);
    return cudaGetLastError();
}

cudaError_t tc_status_read_clear(unsigned int* status) {
    unsigned int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(status, g_tc_status, sizeof(unsigned int));
    if (e != cudaSuccess) return e;
    return *status ? cudaMemcpyToSymbol(g_tc_status, &zero, sizeof(unsigned int)) : cudaSuccess;
}

}  // namespace efla

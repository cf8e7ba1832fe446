// tc_common.cuh -- pieces shared by the tcgen05 forward (fwd_tc.cu) and the tcgen05
// reverse scan of the backward (bwd_tc.cu): wait limits, fp16 operand conversion, the
// range of the fp16 staging, named barriers, and the chunk preparation (tmat_chunk: the
// UT transform's Ta image, the P^T image and the chunk's largest key and query norms).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "launch.h"
#include "tc_ptx.cuh"

namespace efla {

using namespace tc;

constexpr uint32_t kWaitLimit = 1u << 24;
constexpr uint32_t kFlagPollLimit = 1u << 22;   // global-flag polls, 64 ns apart at least

// 8 bf16 (one uint4) -> 8 fp16 (one uint4)
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 raw) {
    const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&raw);
    uint4 out;
    __half2* h = reinterpret_cast<__half2*>(&out);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __float22half2_rn(__bfloat1622float2(b[i]));
    return out;
}

// The same conversion, raising m to the largest magnitude among the 8 values (a NaN
// leaves m unchanged; it reaches the outputs, where it is seen).
__device__ __forceinline__ uint4 bf16x8_to_f16x8_max(uint4 raw, float& m) {
    const __nv_bfloat162* b = reinterpret_cast<const __nv_bfloat162*>(&raw);
    uint4 out;
    __half2* h = reinterpret_cast<__half2*>(&out);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(b[i]);
        m = fmaxf(m, fmaxf(fabsf(f.x), fabsf(f.y)));
        h[i] = __float22half2_rn(f);
    }
    return out;
}

__device__ __forceinline__ uint32_t pack_f16x2(float a, float b) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

// acc stays +0 while every x is finite and becomes NaN after an infinite or NaN x
// (x * 0 is NaN exactly for those); one fused multiply-add per value.
__device__ __forceinline__ void nonfinite_acc(float& acc, float x) {
    asm("fma.rn.f32 %0, %1, 0f00000000, %0;" : "+f"(acc) : "f"(x));
}

// ----------------------------------------------------- range of the fp16 staging
// Every MMA operand of the recurrence is staged in fp16.  A value beyond fp16's range
// becomes infinite there; values far below its normal range lose precision instead.
// Measured with a simulation of this kernel's staging (fp32 accumulation) against the
// fp64 recurrence, max|err|/rms of o stays below 1e-2 while, over one sequence, the largest
// key norm ||k|| is within [2^-10, 64], the largest query norm ||q|| at least 2^-11 and the
// largest |v| or |S0| element at least 2^-10 (zero tensors are exact).  The P^T image
// (entries k.q) and the Q tiles stay finite while ||k|| ||q|| and ||q|| are below 2^15;
// an overflow anywhere else (the state, W, U', Ta) reaches the final state as inf or NaN.
// A sequence outside these bounds, or with a non-finite final state, is recomputed by
// seq_recurrent_fp32 below.  Norms come from the preparation's Gram diagonals (squared).
constexpr float kStageK2Max = 64.f * 64.f;
constexpr float kStageK2Min = 1.f / (1024.f * 1024.f);
constexpr float kStageQ2Min = 1.f / (2048.f * 2048.f);
constexpr float kStageKQ2Max = 32768.f * 32768.f;
constexpr float kStageVMin = 1.f / 1024.f;

__device__ __forceinline__ bool staging_out_of_range(float mk2, float mq2, float mv) {
    return mk2 > kStageK2Max || (mk2 > 0.f && mk2 < kStageK2Min) || (mq2 > 0.f && mq2 < kStageQ2Min) ||
           mq2 >= kStageKQ2Max || mk2 * mq2 >= kStageKQ2Max || (mv > 0.f && mv < kStageVMin);
}

// ================================================================= k_tmat
// Chunk-parallel preparation for the tensor-core forward: one chunk (64 tokens) per
// CTA, 128 threads, four CTAs per SM so that the phases of different chunks overlap.
//   1. K and Q rows of the chunk, bf16 as stored, by four TMA tensor copies straight
//      into SW128 tiles [K; Q] (128 rows; rows past the end of the sequence read as
//      zero).
//   2. One tcgen05 product [K; Q] [K; Q]^T (M = N = 128, bf16 operands: every product
//      of two bf16 values is exact in fp32): in lanes 0..63 (the K rows) columns 0..63
//      are G = K K^T and columns 64..127 are K Q^T.  lambda_j = ||k_j||^2 = G_jj; alpha.
//   3. A = strict_lower(diag(alpha) G) in fp32; the P^T image: (K Q^T)[j][i] for
//      i >= j, i.e. P = tril(Q K^T) transposed (fp16, SW128, rows j).
//   4. T = (I + A)^{-1}, blocked: the four 16x16 diagonal blocks by substitution, then
//      T21 = -T22 A21 T11 at the 32x32 and at the 64x64 level as split-tf32 mma.sync warp
//      tiles (about fp32 accuracy; k ranges bounded by the zero triangles).
//   5. Ta = T diag(alpha) as the fp16 SW128 image (rows i); both images leave by bulk copy.
struct TmatArgs {
    const __nv_bfloat16* k;
    const __nv_bfloat16* q;
    const float* beta;
    uint16_t* Ta;           // [BH][NC][64*64] fp16 images (SW128 K-major, rows i, cols j)
    uint16_t* Pt;           // [BH][NC][64*64] fp16 images (SW128, rows j, cols i)
    float* cnorm;           // [BH][NC][2]: largest ||k||^2 and ||q||^2 of the chunk's tokens
    float* rec_T;           // or null: T [BH][NC][64][64] fp32 and alpha [BH][NC][64] of the
    float* rec_alpha;       //   chunk-state record
    int L, NC, euler;
    long long nch;          // chunks of the launch (B H NC): the extent of the per-chunk arrays
};

constexpr int kTmThreads = 128;
constexpr int kLd = 68;                  // fp32 row stride of T (16-byte rows for float4 reads)
constexpr int kLdA = 68;                 // fp32 row stride of A (= 4 mod 32 banks: the tensor-pipe
                                         // fragment loads and the diagonal blocks' reads are conflict-free)
// shared memory (offsets from a 1024-aligned base)
constexpr uint32_t kTmTiles = 0;         // 2 d-blocks x [K rows | Q rows] x 128 B (bf16); dead after the MMA
constexpr uint32_t kTmA = 0;             // [64][kLdA] fp32 A                        17408 B
constexpr uint32_t kTmY = 17408;         // [32][40] fp32 product intermediate        5120 B
constexpr uint32_t kTmPt = 22528;        // P^T image                                 8192 B
constexpr uint32_t kTmTaImg = 0;         // Ta image, once A is dead                  8192 B
constexpr uint32_t kTmT = 32768;         // [64][kLd] fp32 T                         17408 B
constexpr uint32_t kTmAl = 50176;        // alpha[64]
constexpr uint32_t kTmBar = 50688;       // mbarriers, TMEM slot; +32: the chunk's largest ||k||^2, ||q||^2
constexpr size_t kTmatSmem = 1024 + kTmBar + 64;
constexpr uint32_t kTmGroupBytes = 51200;   // one group's area inside a larger CTA (1024-aligned)
static_assert(kTmBar + 64 <= kTmGroupBytes, "group area");

__device__ __forceinline__ uint4 pack8_f16(const float* v) {
    uint4 w;
    w.x = pack_f16x2(v[0], v[1]);
    w.y = pack_f16x2(v[2], v[3]);
    w.z = pack_f16x2(v[4], v[5]);
    w.w = pack_f16x2(v[6], v[7]);
    return w;
}

// Named barrier of `count` threads (a multiple of 32), and its AND-reduction form.
__device__ __forceinline__ void group_sync(int id, int count = 128) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ bool group_sync_and(int id, bool pred, int count = 128) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.b32 p, %1, 0;\n\t"
        "bar.red.and.pred q, %2, %3, p;\n\t"
        "selp.b32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

// One chunk (bh, c) of the preparation by a group of 128 threads: tid 0..127, its four
// warps aligned to the tensor-memory lane quadrants.  The group owns `sm` (kTmGroupBytes,
// 1024-aligned), the initialised mbarriers bar[0..1] (this chunk completes their phase
// `ph`), 128 tensor-memory columns at `tb` and named barrier `bid`.  With `flag`, the
// images are published by a release store of 1 there once they are in global memory.
// With pf_bh >= 0, the K and Q rows of chunk (pf_bh, pf_c) -- the one this group, or the
// CTA a wave later, prepares next -- are prefetched into L2 while this chunk's tiles load.
// Returns false after a wait timed out (recorded in *status, bit 0).
__device__ __forceinline__ bool tmat_chunk(const CUtensorMap* tm_k, const CUtensorMap* tm_q, const TmatArgs& a,
                                           unsigned char* sm, uint64_t* bar, uint32_t ph, uint32_t tb,
                                           int bid, int tid, long long bh, int c, int* flag,
                                           unsigned int* status, long long pf_bh = -1, int pf_c = 0) {
    const int warp = tid >> 5, lane = tid & 31;
    float* al = (float*)(sm + kTmAl);                // alpha [64]
    const int t0 = c * 64;
    const int nrow = min(64, a.L - t0);              // valid token rows in this chunk

    // ---- 1. [K; Q] tiles by TMA (x = 64 blk: a multiple of 8 bf16 elements)
    if (tid == 0) {
        mbar_arrive_expect_tx(&bar[0], 4u * 8192u);
        for (int blk = 0; blk < 2; ++blk) {
            tma_load_3d(sm + kTmTiles + blk * 16384, tm_k, 64 * blk, t0, (int)bh, &bar[0]);
            tma_load_3d(sm + kTmTiles + blk * 16384 + 8192, tm_q, 64 * blk, t0, (int)bh, &bar[0]);
        }
        if (pf_bh >= 0) {   // whole 256-byte rows of the sequence, inside it
            const size_t row0 = (size_t)pf_bh * a.L + (size_t)pf_c * 64;
            const uint32_t bytes = (uint32_t)min(64, a.L - pf_c * 64) * 256u;
            bulk_prefetch_l2(a.k + row0 * 128, bytes);
            bulk_prefetch_l2(a.q + row0 * 128, bytes);
        }
    }
    const float beta_j = tid < nrow ? a.beta[bh * a.L + t0 + tid] : 0.f;   // in flight with the tiles
    unsigned* nrm = (unsigned*)(sm + kTmBar + 32);   // largest ||k||^2, ||q||^2 (fp32 bits, >= 0)
    if (tid == 0) nrm[0] = nrm[1] = 0u;
    tc_fence_before();
    group_sync(bid);
    tc_fence_after();

    // ---- 2. [K; Q] [K; Q]^T
    if (tid == 0) {
        if (mbar_wait(&bar[0], ph, kWaitLimit)) {
            tc_fence_after();
            const uint32_t idesc = idesc_f16(128, 128, false, false, true);
            for (int s = 0; s < 8; ++s) {
                const uint64_t d = sdesc_sw128(smem_u32(sm + kTmTiles + (s / 4) * 16384 + (s % 4) * 32));
                mma_f16_ss(tb, d, d, idesc, s > 0 ? 1u : 0u);
            }
            mma_commit(&bar[1]);
        } else {
            atomicOr(status, 1u);
            mbar_wait(&bar[0], ph, kWaitLimit);   // let the copies land before the group moves on
        }
    }
    bool ok = group_sync_and(bid, mbar_wait(&bar[1], ph, kWaitLimit));
    if (!ok) {
        atomicOr(status, 1u);
        mbar_wait(&bar[1], ph, kWaitLimit);   // drain this group's MMA before its tensor memory is reused
    }
    tc_fence_after();
    if (ok && warp < 2) {
        // ---- 3. TMEM lane j = token j.  lambda_j = G_jj gives alpha_j, and row j of A is
        // A[j][i] = alpha_j G[j][i], i < j (one register scale, 16-byte rows).  (The P^T
        // image comes from the query lanes, below.)
        const int j = tid;
        float* A = (float*)(sm + kTmA);
        float v[64];   // one row of 64 columns per batch: the four loads share one wait
#pragma unroll
        for (int c16 = 0; c16 < 64; c16 += 16)
            tmem_ld16(taddr(tb, warp * 32, c16), *reinterpret_cast<float(*)[16]>(v + c16));
        tmem_ld_wait();
        float lam = 0.f;
#pragma unroll
        for (int i = 0; i < 64; ++i) lam = (i == j) ? v[i] : lam;
        {   // rows past the sequence are zero
            const unsigned m = __reduce_max_sync(0xffffffffu, __float_as_uint(lam));
            if (lane == 0) atomicMax(&nrm[0], m);
        }
        const float aj = j < nrow ? alpha_of(beta_j, lam, a.euler) : 0.f;
        al[j] = aj;   // scales column j of the Ta image
#pragma unroll
        for (int i = 0; i < 64; i += 4)   // 16-byte rows: 8 lanes per wavefront, none sharing a bank
            *reinterpret_cast<float4*>(A + j * kLdA + i) =
                make_float4(i < j ? aj * v[i] : 0.f, i + 1 < j ? aj * v[i + 1] : 0.f,
                            i + 2 < j ? aj * v[i + 2] : 0.f, i + 3 < j ? aj * v[i + 3] : 0.f);
    } else if (ok) {
        // TMEM lane 64 + i = query token i: column j < 64 of its row is P[i][j] = q_i . k_j,
        // column 64 + i is ||q_i||^2.  The P^T image (rows j, columns i, kept for i >= j) is
        // built from 16x256b fragments with stmatrix.trans: register k of lane t holds row
        // (t >> 2) + 8 ((k >> 1) & 1), column 2 (t & 3) + (k & 1) + 8 (k >> 2) of a 16 x 16 tile.
        {
            const uint32_t img = smem_u32(sm + kTmPt);
            const int mj = lane >> 3, rho = lane & 7;   // stmatrix tile and row this lane addresses
#pragma unroll
            for (int lh = 0; lh < 32; lh += 16) {
                const int ib = (warp - 2) * 32 + lh;   // query rows ib .. ib + 15
#pragma unroll
                for (int c0 = 0; c0 < 64; c0 += 16) {
                    uint32_t r[8];
                    tmem_ld_16x256b_x2(taddr(tb, warp * 32 + lh, c0), r);
                    tmem_ld_wait();
                    float f[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const int ii = ib + (lane >> 2) + 8 * ((k >> 1) & 1);
                        const int jj = c0 + 2 * (lane & 3) + (k & 1) + 8 * (k >> 2);
                        f[k] = ii >= jj ? __uint_as_float(r[k]) : 0.f;
                    }
                    stmatrix_x4_trans(img + sw128(c0 + 8 * (mj >> 1) + rho, ib + (mj & 1) * 8),
                                      pack_f16x2(f[0], f[1]), pack_f16x2(f[2], f[3]), pack_f16x2(f[4], f[5]),
                                      pack_f16x2(f[6], f[7]));
                }
            }
        }
        const int i = tid - 64;
        float v[64];
#pragma unroll
        for (int c16 = 0; c16 < 64; c16 += 16)
            tmem_ld16(taddr(tb, warp * 32, 64 + c16), *reinterpret_cast<float(*)[16]>(v + c16));
        tmem_ld_wait();
        float qq = 0.f;
#pragma unroll
        for (int cc = 0; cc < 64; ++cc) qq = (cc == i) ? v[cc] : qq;
        const unsigned m = __reduce_max_sync(0xffffffffu, __float_as_uint(qq));
        if (lane == 0) atomicMax(&nrm[1], m);
    }
    tc_fence_before();
    group_sync(bid);
    if (ok && tid == 0) {   // published with the images (the flag's release orders it)
        float* cn = a.cnorm + ((size_t)bh * a.NC + c) * 2;
        if (dbg_in(cn, 8, a.cnorm, (size_t)a.nch * 8, status)) {
            cn[0] = __uint_as_float(nrm[0]);
            cn[1] = __uint_as_float(nrm[1]);
        }
    }
    if (!ok) return false;

    // ---- 4. T = (I + A)^{-1}
    const float* A = (const float*)(sm + kTmA);
    float* T = (float*)(sm + kTmT);
    float* Y = (float*)(sm + kTmY);
    if (tid < 64) {   // 4a. diagonal block b = tid >> 4, column cc = tid & 15: forward substitution
        const int o = 16 * (tid >> 4), cc = tid & 15;
        float x[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) x[i] = (i == cc) ? 1.f : 0.f;
#pragma unroll
        for (int jj = 0; jj < 15; ++jj)
#pragma unroll
            for (int i = jj + 1; i < 16; ++i) x[i] = fmaf(-A[(o + i) * kLdA + o + jj], x[jj], x[i]);
#pragma unroll
        for (int i = 0; i < 16; ++i) T[(o + i) * kLd + o + cc] = x[i];
    }
    group_sync(bid);
    {   // 4b. 32x32 level on the tensor pipe: block be = warp >> 1 (rows/cols 32 be ..);
        // warp (w & 1) owns columns 8 (w & 1) .. +7 of Y = A21 T11 and then of T21 = -T22 Y
        // (split-tf32 as in 4c; T11[k][n] = 0 for k < n bounds the first k range)
        const int g = lane >> 2, t = lane & 3, be = warp >> 1, o = 32 * be, n0 = 8 * (warp & 1);
        float* Yb = Y + be * 16 * 24;   // row stride 24 (= 24 mod 32): conflict-free fragment loads
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        for (int k0 = n0; k0 < 16; k0 += 8) {
            uint32_t ah[4], alo[4], bh[2], blo[2];
            split_tf32(A[(o + 16 + g) * kLdA + o + k0 + t], ah[0], alo[0]);
            split_tf32(A[(o + 24 + g) * kLdA + o + k0 + t], ah[1], alo[1]);
            split_tf32(A[(o + 16 + g) * kLdA + o + k0 + t + 4], ah[2], alo[2]);
            split_tf32(A[(o + 24 + g) * kLdA + o + k0 + t + 4], ah[3], alo[3]);
            split_tf32(T[(o + k0 + t) * kLd + o + n0 + g], bh[0], blo[0]);
            split_tf32(T[(o + k0 + t + 4) * kLd + o + n0 + g], bh[1], blo[1]);
            mma_16x8x8_3xtf32(acc, ah, alo, bh, blo);
        }
        *reinterpret_cast<float2*>(Yb + g * 24 + n0 + 2 * t) = make_float2(acc[0], acc[1]);
        *reinterpret_cast<float2*>(Yb + (g + 8) * 24 + n0 + 2 * t) = make_float2(acc[2], acc[3]);
        acc[0] = acc[1] = acc[2] = acc[3] = 0.f;
        group_sync(bid);
        for (int k0 = 0; k0 < 16; k0 += 8) {   // T22[m][k] = 0 for k > m
            uint32_t ah[4], alo[4], bh[2], blo[2];
            split_tf32(T[(o + 16 + g) * kLd + o + 16 + k0 + t], ah[0], alo[0]);
            split_tf32(T[(o + 24 + g) * kLd + o + 16 + k0 + t], ah[1], alo[1]);
            split_tf32(T[(o + 16 + g) * kLd + o + 16 + k0 + t + 4], ah[2], alo[2]);
            split_tf32(T[(o + 24 + g) * kLd + o + 16 + k0 + t + 4], ah[3], alo[3]);
            split_tf32(Yb[(k0 + t) * 24 + n0 + g], bh[0], blo[0]);
            split_tf32(Yb[(k0 + t + 4) * 24 + n0 + g], bh[1], blo[1]);
            mma_16x8x8_3xtf32(acc, ah, alo, bh, blo);
        }
        *reinterpret_cast<float2*>(T + (o + 16 + g) * kLd + o + n0 + 2 * t) = make_float2(-acc[0], -acc[1]);
        *reinterpret_cast<float2*>(T + (o + 24 + g) * kLd + o + n0 + 2 * t) = make_float2(-acc[2], -acc[3]);
        group_sync(bid);
    }
    {   // 4c. 64x64 level on the tensor pipe: warp w owns the 16x16 tile (rows 16 (w & 1),
        // columns 16 (w >> 1)) of Y = A21 T11 and then of T21 = -T22 Y.  Split-tf32 products
        // (x = hi + lo, hi lo both tf32; hi hi + hi lo + lo hi, fp32 accumulation) keep about
        // fp32 accuracy; the zero triangles of T11 and T22 bound the k ranges.
        const int g = lane >> 2, t = lane & 3, m0 = 16 * (warp & 1), n0 = 16 * (warp >> 1);
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        for (int k0 = n0; k0 < 32; k0 += 8) {   // T11[k][n] = 0 for k < n
            uint32_t ah[4], alo[4];
            split_tf32(A[(32 + m0 + g) * kLdA + k0 + t], ah[0], alo[0]);
            split_tf32(A[(40 + m0 + g) * kLdA + k0 + t], ah[1], alo[1]);
            split_tf32(A[(32 + m0 + g) * kLdA + k0 + t + 4], ah[2], alo[2]);
            split_tf32(A[(40 + m0 + g) * kLdA + k0 + t + 4], ah[3], alo[3]);
#pragma unroll
            for (int ni = 0; ni < 2; ++ni) {
                uint32_t bh[2], blo[2];
                split_tf32(T[(k0 + t) * kLd + n0 + 8 * ni + g], bh[0], blo[0]);
                split_tf32(T[(k0 + t + 4) * kLd + n0 + 8 * ni + g], bh[1], blo[1]);
                mma_16x8x8_3xtf32(acc[ni], ah, alo, bh, blo);
            }
        }
#pragma unroll
        for (int ni = 0; ni < 2; ++ni) {
            const int cc = n0 + 8 * ni + 2 * t;
            *reinterpret_cast<float2*>(Y + (m0 + g) * 40 + cc) = make_float2(acc[ni][0], acc[ni][1]);
            *reinterpret_cast<float2*>(Y + (m0 + g + 8) * 40 + cc) = make_float2(acc[ni][2], acc[ni][3]);
            acc[ni][0] = acc[ni][1] = acc[ni][2] = acc[ni][3] = 0.f;
        }
        group_sync(bid);
        for (int k0 = 0; k0 < m0 + 16; k0 += 8) {   // T22[m][k] = 0 for k > m
            uint32_t ah[4], alo[4];
            split_tf32(T[(32 + m0 + g) * kLd + 32 + k0 + t], ah[0], alo[0]);
            split_tf32(T[(40 + m0 + g) * kLd + 32 + k0 + t], ah[1], alo[1]);
            split_tf32(T[(32 + m0 + g) * kLd + 32 + k0 + t + 4], ah[2], alo[2]);
            split_tf32(T[(40 + m0 + g) * kLd + 32 + k0 + t + 4], ah[3], alo[3]);
#pragma unroll
            for (int ni = 0; ni < 2; ++ni) {
                uint32_t bh[2], blo[2];
                split_tf32(Y[(k0 + t) * 40 + n0 + 8 * ni + g], bh[0], blo[0]);
                split_tf32(Y[(k0 + t + 4) * 40 + n0 + 8 * ni + g], bh[1], blo[1]);
                mma_16x8x8_3xtf32(acc[ni], ah, alo, bh, blo);
            }
        }
#pragma unroll
        for (int ni = 0; ni < 2; ++ni) {
            const int cc = n0 + 8 * ni + 2 * t;
            *reinterpret_cast<float2*>(T + (32 + m0 + g) * kLd + cc) = make_float2(-acc[ni][0], -acc[ni][1]);
            *reinterpret_cast<float2*>(T + (40 + m0 + g) * kLd + cc) = make_float2(-acc[ni][2], -acc[ni][3]);
        }
        group_sync(bid);
    }
    if (a.rec_T && dbg_in(a.rec_T + ((size_t)bh * a.NC + c) * 4096, 16384, a.rec_T, (size_t)a.nch * 16384, status) &&
        dbg_in(a.rec_alpha + ((size_t)bh * a.NC + c) * 64, 256, a.rec_alpha, (size_t)a.nch * 256, status)) {
        // the chunk-state record keeps T (fp32, zero above the diagonal) and alpha
        float* dst = a.rec_T + ((size_t)bh * a.NC + c) * 4096;
        for (int e = tid; e < 64 * 16; e += kTmThreads) {
            const int i = e >> 4, j4 = (e & 15) * 4;
            *reinterpret_cast<float4*>(dst + i * 64 + j4) =
                j4 < 16 * ((i >> 4) + 1) ? *reinterpret_cast<const float4*>(T + i * kLd + j4)
                                         : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        if (tid < 64) a.rec_alpha[((size_t)bh * a.NC + c) * 64 + tid] = al[tid];
    }
    // ---- 5. Ta[i][j] = T[i][j] alpha_j (zero above the diagonal): row i = tid >> 1,
    // columns 32 (tid & 1) .. +31, as the fp16 SW128 image (A is dead: its space is reused)
    {
        const int i = tid >> 1, h = tid & 1;
        unsigned char* img = sm + kTmTaImg;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            const int j0 = 32 * h + 8 * g;
            if (j0 >= 16 * ((i >> 4) + 1)) {   // above the diagonal blocks: zero (never written in T)
                *reinterpret_cast<uint4*>(img + sw128(i, j0)) = make_uint4(0u, 0u, 0u, 0u);
                continue;
            }
            const float4 ta = *reinterpret_cast<const float4*>(T + i * kLd + j0);
            const float4 tc4 = *reinterpret_cast<const float4*>(T + i * kLd + j0 + 4);
            const float4 a0 = *reinterpret_cast<const float4*>(al + j0);
            const float4 a1 = *reinterpret_cast<const float4*>(al + j0 + 4);
            const float v[8] = {ta.x * a0.x, ta.y * a0.y, ta.z * a0.z, ta.w * a0.w,
                                tc4.x * a1.x, tc4.y * a1.y, tc4.z * a1.z, tc4.w * a1.w};
            *reinterpret_cast<uint4*>(img + sw128(i, j0)) = pack8_f16(v);
        }
    }
    fence_async_smem();
    group_sync(bid);
    if (tid == 0) {
        const size_t io = ((size_t)bh * a.NC + c) * 4096;
        if (dbg_in(a.Ta + io, 8192, a.Ta, (size_t)a.nch * 8192, status)) bulk_s2g(a.Ta + io, sm + kTmTaImg, 8192u);
        if (dbg_in(a.Pt + io, 8192, a.Pt, (size_t)a.nch * 8192, status)) bulk_s2g(a.Pt + io, sm + kTmPt, 8192u);
        bulk_commit();
        if (flag) {   // publish: the images are in global memory before the flag is
            bulk_wait_all();
            fence_proxy_async_global();
            st_release_gpu(flag, 1);
        } else {
            bulk_wait_read();
        }
    }
    group_sync(bid);   // the group's shared memory is free again
    return true;
}

// Tensor map of a bf16 [BH][L][128] array, boxes of 64 rows x 64 columns with the
// 128-byte swizzle (the operand tile layout); rows past L read as zero.
inline cudaError_t bf16_rows_map(CUtensorMap* m, const void* base, const Dims& d) {
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    if (!encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                         cudaEnableDefault, &q);
        if (e != cudaSuccess) return e;
        if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
        encode = (PFN_cuTensorMapEncodeTiled_v12000)fn;
    }
    const cuuint64_t dims[3] = {128, (cuuint64_t)d.L, (cuuint64_t)d.BH()};
    const cuuint64_t strides[2] = {256, (cuuint64_t)d.L * 256};   // bytes, dimensions 1 and 2
    const cuuint32_t box[3] = {64, 64, 1};
    const cuuint32_t elem[3] = {1, 1, 1};
    const CUresult r = encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                              box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// The chunk preparation as a kernel of its own (fwd_tc.cu), over every chunk of d, for a
// consumer that runs after it (no image-ready flags).
cudaError_t launch_tmat(const Dims& d, const CUtensorMap* tm_k, const CUtensorMap* tm_q, const TmatArgs& ta,
                        cudaStream_t st);

}  // namespace efla

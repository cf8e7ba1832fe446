// common.cuh -- device helpers shared by the EFLA kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "launch.h"

namespace efla {

// ---------------------------------------------------------------- element io
// Debug builds (compiled with -DEFLA_DEBUG) check the global writes of the tensor-core
// kernels tile by tile: a write of `bytes` at p must lie inside [base, base + extent bytes).
// A write outside is skipped and kStatusBounds is set in `status` (the kernel file's device
// status word); efla_get_status then reports EFLA_ERR_BOUNDS.  Release builds compile the
// check to `true`.  (kStatusBounds: launch.h.)
__device__ __forceinline__ bool dbg_in(const void* p, size_t bytes, const void* base, size_t extent,
                                       unsigned* status) {
#ifdef EFLA_DEBUG
    const char* c = static_cast<const char*>(p);
    const char* b = static_cast<const char*>(base);
    if (c < b || c + bytes > b + extent) {
        atomicOr(status, kStatusBounds);
        return false;
    }
#else
    (void)p, (void)bytes, (void)base, (void)extent, (void)status;
#endif
    return true;
}

__device__ __forceinline__ float ld_elem(const float* p) { return __ldg(p); }
__device__ __forceinline__ float ld_elem(const __nv_bfloat16* p) { return __bfloat162float(*p); }

__device__ __forceinline__ void st_elem(float* p, float x) { *p = x; }
__device__ __forceinline__ void st_elem(__nv_bfloat16* p, float x) { *p = __float2bfloat16_rn(x); }

// ------------------------------------------------------------------- alpha
// alpha = (1 - e^{-beta lambda}) / lambda  (exact flow of the rank-1 ODE over one token),
// evaluated as beta * phi(x), x = beta*lambda, phi(x) = -expm1(-x)/x, phi(0) = 1, so that
// alpha -> beta as lambda -> 0.  Euler mode: alpha = beta.
__device__ __forceinline__ float alpha_of(float beta, float lambda, int euler) {
    if (euler) return beta;
    float x = beta * lambda;
    if (x == 0.0f) return beta;
    return beta * (-expm1f(-x) / x);
}

// d alpha / d beta = e^{-beta lambda}   (1 in Euler mode)
__device__ __forceinline__ float dalpha_dbeta_of(float beta, float lambda, int euler) {
    if (euler) return 1.0f;
    return expf(-beta * lambda);
}

// d alpha / d lambda = beta^2 phi'(x),  phi'(x) = (x e^{-x} + expm1(-x)) / x^2.
// Near x = 0 that quotient cancels, so |x| < 0.5 uses the Taylor series of phi'
// (phi(x) = sum_n (-x)^n/(n+1)!  =>  phi'(x) = sum_{n>=1} n (-1)^n x^{n-1} / (n+1)!).
__device__ __forceinline__ float dalpha_dlambda_of(float beta, float lambda, int euler) {
    if (euler) return 0.0f;
    float x = beta * lambda;
    float dphi;
    if (fabsf(x) < 0.5f) {
        // Horner form of -1/2 + x/3 - x^2/8 + x^3/30 - x^4/144 + x^5/840 - x^6/5760 + x^7/45360
        dphi = 1.0f / 45360.0f;
        dphi = fmaf(dphi, x, -1.0f / 5760.0f);
        dphi = fmaf(dphi, x, 1.0f / 840.0f);
        dphi = fmaf(dphi, x, -1.0f / 144.0f);
        dphi = fmaf(dphi, x, 1.0f / 30.0f);
        dphi = fmaf(dphi, x, -1.0f / 8.0f);
        dphi = fmaf(dphi, x, 1.0f / 3.0f);
        dphi = fmaf(dphi, x, -0.5f);
    } else {
        dphi = (x * expf(-x) + expm1f(-x)) / (x * x);
    }
    return beta * beta * dphi;
}

// ------------------------------------------------------------- reductions
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// ------------------------------------------------------- block-level matmul
// out(m, n) <- sum_{kk < K} a(m,kk) * b(kk,n)  for all m < M, n < N, every thread
// of the block (NT threads) participating.  a, b and the store are functors so
// that transposes and masks are explicit at the call site.  Each thread owns
// 4 rows x 1 column per pass (rows m, m+M/4, m+M/2, m+3M/4) so that one b load
// feeds four FMAs; requires M % 4 == 0.
template <int NT, typename FA, typename FB, typename FS>
__device__ __forceinline__ void block_mm(int M, int N, int K, FA a, FB b, FS store) {
    const int Mq = M >> 2;
    for (int idx = threadIdx.x; idx < Mq * N; idx += NT) {
        const int m = idx / N;
        const int n = idx - m * N;
        float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
        for (int kk = 0; kk < K; ++kk) {
            const float bb = b(kk, n);
            s0 = fmaf(a(m, kk), bb, s0);
            s1 = fmaf(a(m + Mq, kk), bb, s1);
            s2 = fmaf(a(m + 2 * Mq, kk), bb, s2);
            s3 = fmaf(a(m + 3 * Mq, kk), bb, s3);
        }
        store(m, n, s0);
        store(m + Mq, n, s1);
        store(m + 2 * Mq, n, s2);
        store(m + 3 * Mq, n, s3);
    }
}

// Same contraction with a per-output summation range [lo, hi) given by
// krange(m, n, lo, hi) (triangular products); one output per thread per pass.
template <int NT, typename FA, typename FB, typename FK, typename FS>
__device__ __forceinline__ void block_mm_ranged(int M, int N, FA a, FB b, FK krange, FS store) {
    for (int idx = threadIdx.x; idx < M * N; idx += NT) {
        const int m = idx / N;
        const int n = idx - m * N;
        int lo, hi;
        krange(m, n, lo, hi);
        float s = 0.f;
        for (int kk = lo; kk < hi; ++kk) s = fmaf(a(m, kk), b(kk, n), s);
        store(m, n, s);
    }
}

}  // namespace efla

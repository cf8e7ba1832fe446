// bwd_mma.cu -- per-chunk gradients of the chunked backward on the tensor pipe.
//
// Same mathematics as the per-chunk gradient kernels of bwd_simt.cu (reverse-mode
// differentiation of the chunk form of page es, Metodologia item 3; the pages give no
// backward pass), for bf16 inputs with d_k = 128, chunk 64 and d_v in {64, 128}:
//   D   = tril(dO Up^T)                       dQ = dO S^T + D K
//   dW  = -dUp S^T                            dT = dW (aK)^T + dUp (aV)^T   (strictly lower part)
//   dKa = T^T dW,  dVa = T^T dUp              dV = diag(alpha) dVa
//   X   = dT T^T,  dA = strict_lower(-T^T X), dG = diag(alpha) dA,  G = K K^T
//   dK  = D^T Q + Up G'^T + (dG + dG^T) K + diag(alpha) dKa + 2 diag(dlambda) K
//   dalpha_i = sum_{j<i} dA_ij G_ij + <dKa_i, k_i> + <dVa_i, v_i>
// Every product is a warp-tiled mma.sync m16n8k8 with tf32 operands (fp32 values rounded
// to nearest once, when they are staged in shared memory; bf16 inputs are exact in tf32)
// and fp32 accumulation.  Triangular operands bound each tile's k range, and tiles that
// lie wholly above the diagonal of a triangular result are skipped.  Row sums for dalpha
// go through fixed per-source slots, so the result does not depend on warp timing.
#include <stdint.h>

#include "common.cuh"
#include "launch.h"

namespace efla {
namespace {

constexpr int kGmThreads = 256;    // 8 warps
constexpr int kC = 64, kDk = 128, kBV = 64;
constexpr int kLd = 68;            // row stride of [*][64] tiles (68 = 4 mod 32 banks)
constexpr int kLdk = 132;          // row stride of [*][128] tiles
struct GmArgs {
    const void* q;
    const void* k;
    const void* v;
    const void* dO;
    const float* beta;
    const float* alpha;
    const float* T;
    const float* Sc;
    const float* dSc;
    const float* Up;
    const float* dUp;
    void* dq;
    void* dk;
    void* dv;
    float* dbeta;
    const int* list;     // null (every chunk, one per CTA), or the chunks to compute
    const int* list_n;   //   and their number (device words)
    int L, dv_, NC, euler, out_bf16;
};

__device__ __forceinline__ float tf32r(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return __uint_as_float(r);
}

__device__ __forceinline__ float4 tf32r4(float4 v) {
    return make_float4(tf32r(v.x), tf32r(v.y), tf32r(v.z), tf32r(v.w));
}

__device__ __forceinline__ void mma_tf32(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    asm("mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// acc[mi][ni] += sum over k in [k0, k1) of A(m, k) B(k, n) for the warp's tile: rows
// m0 + 16 mi + {g, g + 8}, columns n0 + 8 ni + {2t, 2t + 1} (g = lane / 4, t = lane % 4).
// A(m, k) = A[m am + k ak] and B(k, n) = B[k bk + n bn] hold tf32-rounded values; k0 and
// k1 are multiples of 8.
template <int MI, int NI>
__device__ __forceinline__ void tile_mma(float (&acc)[MI][NI][4], const float* A, int am, int ak,
                                         const float* B, int bk, int bn, int m0, int n0, int k0,
                                         int k1) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const float* Ab = A + (m0 + g) * am + t * ak;
    const float* Bb = B + t * bk + (n0 + g) * bn;
#pragma unroll 2
    for (int k = k0; k < k1; k += 8) {
        uint32_t a[MI][4], b[NI][2];
#pragma unroll
        for (int mi = 0; mi < MI; ++mi) {
            const float* p = Ab + 16 * mi * am + k * ak;
            a[mi][0] = __float_as_uint(p[0]);
            a[mi][1] = __float_as_uint(p[8 * am]);
            a[mi][2] = __float_as_uint(p[4 * ak]);
            a[mi][3] = __float_as_uint(p[8 * am + 4 * ak]);
        }
#pragma unroll
        for (int ni = 0; ni < NI; ++ni) {
            const float* p = Bb + k * bk + 8 * ni * bn;
            b[ni][0] = __float_as_uint(p[0]);
            b[ni][1] = __float_as_uint(p[4 * bk]);
        }
#pragma unroll
        for (int mi = 0; mi < MI; ++mi)
#pragma unroll
            for (int ni = 0; ni < NI; ++ni) mma_tf32(acc[mi][ni], a[mi], b[ni]);
    }
}

template <int MI, int NI>
__device__ __forceinline__ void zero(float (&acc)[MI][NI][4]) {
#pragma unroll
    for (int mi = 0; mi < MI; ++mi)
#pragma unroll
        for (int ni = 0; ni < NI; ++ni)
#pragma unroll
            for (int r = 0; r < 4; ++r) acc[mi][ni][r] = 0.f;
}

__device__ __forceinline__ void st_pair(void* p, size_t i, float x0, float x1, int bf16) {
    if (bf16)
        *reinterpret_cast<__nv_bfloat162*>((__nv_bfloat16*)p + i) = __floats2bfloat162_rn(x0, x1);
    else
        *reinterpret_cast<float2*>((float*)p + i) = make_float2(x0, x1);
}

// 8 bf16 (16 bytes) -> two float4 in shared memory, or zeros for a row past the sequence.
__device__ __forceinline__ void stage_bf16x8(float* dst, const __nv_bfloat16* src, bool ok) {
    float4 lo = make_float4(0.f, 0.f, 0.f, 0.f), hi = lo;
    if (ok) {
        const uint4 raw = *reinterpret_cast<const uint4*>(src);
        const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.x));
        const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.y));
        const float2 f2 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.z));
        const float2 f3 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw.w));
        lo = make_float4(f0.x, f0.y, f1.x, f1.y);
        hi = make_float4(f2.x, f2.y, f3.x, f3.y);
    }
    *reinterpret_cast<float4*>(dst) = lo;
    *reinterpret_cast<float4*>(dst + 4) = hi;
}

// ------------------------------------------------------------ chunk preparation
// Per chunk: lambda, alpha, P = tril(Q K^T) (diagonal included), A = strict_lower(diag(alpha)
// K K^T), T = (I + A)^{-1}, W = T diag(alpha) K, U = T diag(alpha) V.  The Gram products run
// on the tensor pipe with exact (bf16) operands; T is a blocked forward substitution (16 x 16
// diagonal blocks in fp32 on the CUDA cores, then one block row at a time,
// T_bj = -T_bb sum_{m<b} A_bm T_mj, as split-tf32 warp tiles); W and U are tf32 products.
constexpr int kPmThreads = 256;
constexpr int kLdY = 48;
constexpr int kPmK = 0;                          // K, later tf32(alpha K)   [64][kLdk]
constexpr int kPmV = kPmK + kC * kLdk;           // V, later tf32(alpha V)   [64][kLdk]
constexpr int kPmQ = kPmV + kC * kLdk;           // Q [64][kLdk]; then A (later tf32 T) and T
constexpr int kPmA = kPmQ;                       // [64][kLd]
constexpr int kPmT = kPmQ + kC * kLd;            // [64][kLd]
constexpr int kPmY = kPmQ + 2 * kC * kLd;        // block-row products [16][kLdY]
constexpr int kPmAl = kPmY + 16 * kLdY;          // alpha [64], lambda [64]
constexpr size_t kPmSmem = (size_t)(kPmAl + 2 * kC) * sizeof(float);
static_assert(2 * kC * kLd >= kC * kLdk, "A and T must cover Q's rows");

struct PmArgs {
    const void* q;
    const void* k;
    const void* v;
    const float* beta;
    float* alpha;
    float* W;
    float* U;
    float* T;
    float* P;
    const int* list;     // null (every chunk, one per CTA), or the sequences to prepare
    const int* list_n;   //   and their number (device words)
    int L, dv_, NC, euler;
};

// One 16x8 tile of d += A B in split tf32 (x = hi + lo, both tf32; hi hi + hi lo + lo hi with
// fp32 accumulation keeps about fp32 accuracy): A(m, k) = A[(m0 + m) lda + k],
// B(k, n) = B[k ldb + n0 + n], k in [k0, k1) (multiples of 8).
__device__ __forceinline__ void tile16x8_3xtf32(float (&d)[4], const float* A, int lda, int m0, const float* B,
                                                int ldb, int n0, int k0, int k1) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    for (int k = k0; k < k1; k += 8) {
        const float av[4] = {A[(m0 + g) * lda + k + t], A[(m0 + g + 8) * lda + k + t],
                             A[(m0 + g) * lda + k + t + 4], A[(m0 + g + 8) * lda + k + t + 4]};
        const float bv[2] = {B[(k + t) * ldb + n0 + g], B[(k + t + 4) * ldb + n0 + g]};
        uint32_t ah[4], alo[4], bh[2], blo[2];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            ah[e] = __float_as_uint(tf32r(av[e]));
            alo[e] = __float_as_uint(tf32r(av[e] - __uint_as_float(ah[e])));
        }
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            bh[e] = __float_as_uint(tf32r(bv[e]));
            blo[e] = __float_as_uint(tf32r(bv[e] - __uint_as_float(bh[e])));
        }
        mma_tf32(d, alo, bh);
        mma_tf32(d, ah, blo);
        mma_tf32(d, ah, bh);
    }
}

// One block row of the blocked inverse (rows 16 BI .. 16 BI + 15, columns below 16 BI), after
// the diagonal blocks and the block rows above it: warp w < 2 BI owns columns 8w .. 8w + 7 of
// Y = A[rows][0, 16 BI) T and then of -T_bb Y.  T[m][c] = 0 for m < c bounds the first k range;
// T_bb is lower triangular (its zeros above the diagonal add nothing).
template <int BI>
__device__ __forceinline__ void tinv_block_row(const float* As, float* Ts, float* Ys, int tid) {
    constexpr int w = 16 * BI;
    const int warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
    __syncthreads();
    if (warp < w / 8) {
        const int n0 = 8 * warp;
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        tile16x8_3xtf32(d, As, kLd, w, Ts, kLd, n0, n0, w);
        *reinterpret_cast<float2*>(Ys + g * kLdY + n0 + 2 * t) = make_float2(d[0], d[1]);
        *reinterpret_cast<float2*>(Ys + (g + 8) * kLdY + n0 + 2 * t) = make_float2(d[2], d[3]);
    }
    __syncthreads();
    if (warp < w / 8) {
        const int n0 = 8 * warp;
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        tile16x8_3xtf32(d, Ts + w, kLd, w, Ys, kLdY, n0, 0, 16);
        *reinterpret_cast<float2*>(Ts + (w + g) * kLd + n0 + 2 * t) = make_float2(-d[0], -d[1]);
        *reinterpret_cast<float2*>(Ts + (w + g + 8) * kLd + n0 + 2 * t) = make_float2(-d[2], -d[3]);
    }
}

// One chunk's preparation (the body of k_prep_mma).
__device__ __forceinline__ void prep_mma_chunk(const PmArgs& a, const long long bh, const int c) {
    extern __shared__ __align__(16) float sm[];
    const int dv = a.dv_;
    const int t0 = c * kC, nvalid = min(kC, a.L - t0);
    const long long tok0 = bh * a.L + t0;
    const size_t chunk = (size_t)bh * a.NC + c;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
    float* Ks = sm + kPmK;
    float* Vs = sm + kPmV;
    float* Qs = sm + kPmQ;
    float* As = sm + kPmA;
    float* Ts = sm + kPmT;
    float* Ys = sm + kPmY;
    float* al = sm + kPmAl;
    float* lam = al + kC;
    const int wm = 32 * (warp & 1), wn = 32 * (warp >> 1);
    const int qm = 16 * (warp & 3), qn = 32 * (warp >> 2);
    const bool lower_tile = qn <= qm + 14;

    {
        const __nv_bfloat16* Qg = (const __nv_bfloat16*)a.q + tok0 * kDk;
        const __nv_bfloat16* Kg = (const __nv_bfloat16*)a.k + tok0 * kDk;
        const __nv_bfloat16* Vg = (const __nv_bfloat16*)a.v + tok0 * dv;
        for (int idx = tid; idx < kC * kDk / 8; idx += kPmThreads) {
            const int i = idx >> 4, x8 = (idx & 15) * 8;
            stage_bf16x8(Ks + i * kLdk + x8, Kg + (size_t)i * kDk + x8, i < nvalid);
            stage_bf16x8(Qs + i * kLdk + x8, Qg + (size_t)i * kDk + x8, i < nvalid);
        }
        const int per = dv / 8;
        for (int idx = tid; idx < kC * per; idx += kPmThreads) {
            const int i = idx / per, x8 = (idx - i * per) * 8;
            stage_bf16x8(Vs + i * kLdk + x8, Vg + (size_t)i * dv + x8, i < nvalid);
        }
    }
    __syncthreads();
    for (int i = warp; i < kC; i += kPmThreads / 32) {
        float s = 0.f;
        for (int x = lane; x < kDk; x += 32) s = fmaf(Ks[i * kLdk + x], Ks[i * kLdk + x], s);
        s = warp_sum(s);
        if (lane == 0) {
            const float al_i = alpha_of(i < nvalid ? a.beta[tok0 + i] : 0.f, s, a.euler);
            lam[i] = s;
            al[i] = al_i;
            a.alpha[chunk * kC + i] = al_i;
        }
    }
    float pa[1][4][4], ga[1][4][4];
    zero(pa); zero(ga);
    if (lower_tile) {
        tile_mma<1, 4>(pa, Qs, kLdk, 1, Ks, 1, kLdk, qm, qn, 0, kDk);
        tile_mma<1, 4>(ga, Ks, kLdk, 1, Ks, 1, kLdk, qm, qn, 0, kDk);
    }
    {
        float* Pg = a.P + chunk * kC * kC;
#pragma unroll
        for (int ni = 0; ni < 4; ++ni) {
            const int r0 = qm + g, r1 = r0 + 8, cc = qn + 8 * ni + 2 * t;
            *reinterpret_cast<float2*>(Pg + r0 * kC + cc) =
                make_float2(cc <= r0 ? pa[0][ni][0] : 0.f, cc + 1 <= r0 ? pa[0][ni][1] : 0.f);
            *reinterpret_cast<float2*>(Pg + r1 * kC + cc) =
                make_float2(cc <= r1 ? pa[0][ni][2] : 0.f, cc + 1 <= r1 ? pa[0][ni][3] : 0.f);
        }
    }
    __syncthreads();   // Q read for the last time; alpha ready
    for (int idx = tid; idx < kC * kLd; idx += kPmThreads) Ts[idx] = 0.f;
#pragma unroll
    for (int ni = 0; ni < 4; ++ni) {
        const int r0 = qm + g, r1 = r0 + 8, cc = qn + 8 * ni + 2 * t;
        As[r0 * kLd + cc] = cc < r0 ? al[r0] * ga[0][ni][0] : 0.f;
        As[r0 * kLd + cc + 1] = cc + 1 < r0 ? al[r0] * ga[0][ni][1] : 0.f;
        As[r1 * kLd + cc] = cc < r1 ? al[r1] * ga[0][ni][2] : 0.f;
        As[r1 * kLd + cc + 1] = cc + 1 < r1 ? al[r1] * ga[0][ni][3] : 0.f;
    }
    __syncthreads();
    // diagonal blocks: lane (16 b + j) of warps 0-1 substitutes column j of block b
    if (warp < 2) {
        const int b = 2 * warp + (lane >> 4), j = lane & 15, o = 16 * b;
        float col[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float x = (i == j) ? 1.f : 0.f;
#pragma unroll
            for (int m = 0; m < i; ++m)
                if (m >= j) x = fmaf(-As[(o + i) * kLd + o + m], col[m], x);
            col[i] = x;
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) Ts[(o + i) * kLd + o + j] = col[i];
    }
    // block rows 1..3: Y = sum_{m < 16 b} A[16 b + r][m] T[m][c], then T[16 b + r][c] = -T_bb Y
    tinv_block_row<1>(As, Ts, Ys, tid);
    tinv_block_row<2>(As, Ts, Ys, tid);
    tinv_block_row<3>(As, Ts, Ys, tid);
    __syncthreads();
    // T out; tf32 operands: T over A, alpha K over K, alpha V over V
    {
        float* Tg = a.T + chunk * kC * kC;
        for (int idx = tid; idx < kC * kC / 4; idx += kPmThreads) {
            const int i = idx >> 4, j4 = (idx & 15) * 4;
            const float4 tv = *reinterpret_cast<const float4*>(Ts + i * kLd + j4);
            *reinterpret_cast<float4*>(Tg + i * kC + j4) = tv;
            *reinterpret_cast<float4*>(As + i * kLd + j4) = tf32r4(tv);
        }
        for (int idx = tid; idx < kC * kDk / 4; idx += kPmThreads) {
            const int i = idx >> 5, x4 = (idx & 31) * 4;
            float4 kv = *reinterpret_cast<const float4*>(Ks + i * kLdk + x4);
            const float s = al[i];
            kv = make_float4(s * kv.x, s * kv.y, s * kv.z, s * kv.w);
            *reinterpret_cast<float4*>(Ks + i * kLdk + x4) = tf32r4(kv);
        }
        const int per = dv / 4;
        for (int idx = tid; idx < kC * per; idx += kPmThreads) {
            const int i = idx / per, x4 = (idx - i * per) * 4;
            float4 vv = *reinterpret_cast<const float4*>(Vs + i * kLdk + x4);
            const float s = al[i];
            vv = make_float4(s * vv.x, s * vv.y, s * vv.z, s * vv.w);
            *reinterpret_cast<float4*>(Vs + i * kLdk + x4) = tf32r4(vv);
        }
    }
    __syncthreads();
    // W = T (alpha K), U = T (alpha V)   (T[i][j] = 0 for j > i)
    {
        float wa[2][4][4];
        zero(wa);
        tile_mma<2, 4>(wa, As, kLd, 1, Ks, kLdk, 1, wm, wn, 0, wm + 32);
        float* Wg = a.W + chunk * kC * kDk;
#pragma unroll
        for (int mi = 0; mi < 2; ++mi)
#pragma unroll
            for (int ni = 0; ni < 4; ++ni) {
                const int r0 = wm + 16 * mi + g, cc = wn + 8 * ni + 2 * t;
                *reinterpret_cast<float2*>(Wg + r0 * kDk + cc) = make_float2(wa[mi][ni][0], wa[mi][ni][1]);
                *reinterpret_cast<float2*>(Wg + (r0 + 8) * kDk + cc) =
                    make_float2(wa[mi][ni][2], wa[mi][ni][3]);
            }
    }
    {
        float* Ug = a.U + chunk * kC * dv;
        if (dv == kDk) {
            float ua[2][4][4];
            zero(ua);
            tile_mma<2, 4>(ua, As, kLd, 1, Vs, kLdk, 1, wm, wn, 0, wm + 32);
#pragma unroll
            for (int mi = 0; mi < 2; ++mi)
#pragma unroll
                for (int ni = 0; ni < 4; ++ni) {
                    const int r0 = wm + 16 * mi + g, cc = wn + 8 * ni + 2 * t;
                    *reinterpret_cast<float2*>(Ug + r0 * dv + cc) = make_float2(ua[mi][ni][0], ua[mi][ni][1]);
                    *reinterpret_cast<float2*>(Ug + (r0 + 8) * dv + cc) =
                        make_float2(ua[mi][ni][2], ua[mi][ni][3]);
                }
        } else {   // dv = 64
            float ua[1][4][4];
            zero(ua);
            tile_mma<1, 4>(ua, As, kLd, 1, Vs, kLdk, 1, qm, qn, 0, qm + 16);
#pragma unroll
            for (int ni = 0; ni < 4; ++ni) {
                const int r0 = qm + g, cc = qn + 8 * ni + 2 * t;
                *reinterpret_cast<float2*>(Ug + r0 * dv + cc) = make_float2(ua[0][ni][0], ua[0][ni][1]);
                *reinterpret_cast<float2*>(Ug + (r0 + 8) * dv + cc) = make_float2(ua[0][ni][2], ua[0][ni][3]);
            }
        }
    }
}

template <bool kList>
__global__ void __launch_bounds__(kPmThreads, 2) k_prep_mma(PmArgs a) {
    if constexpr (!kList) {   // every chunk, one per CTA
        prep_mma_chunk(a, blockIdx.x, blockIdx.y);
        return;
    }
    const int n = *a.list_n * a.NC;   // the listed sequences' chunks, grid-stride
    for (int w = blockIdx.x; w < n; w += gridDim.x) {
        prep_mma_chunk(a, a.list[w / a.NC], w % a.NC);
        __syncthreads();   // shared memory is reused by the next chunk
    }
}

// ------------------------------------------------------------------ the two scans
// Both scans are sequential over a sequence's chunks and parallel over sequences and
// 64-column value slices.  The state (or its gradient) slice [128][64] lives in fp32 mma
// accumulators for the whole sequence; a tf32 copy in shared memory feeds the products that
// read it.  Each chunk's operands arrive by cp.async into single buffers that are refilled as
// soon as the product reading them is done, so every load overlaps the other product.

__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool ok) {
    const uint32_t d = (uint32_t)__cvta_generic_to_shared(dst);
    const int n = ok ? 16 : 0;   // 0: fill with zeros, read nothing
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src), "r"(n) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Operand views: element (r, c) at p[r rs + c cs], returned as tf32 bits.
struct VF32 {      // already tf32-rounded fp32
    const float* p; int rs, cs;
    __device__ __forceinline__ uint32_t operator()(int r, int c) const { return __float_as_uint(p[r * rs + c * cs]); }
};
struct VF32R {     // fp32, rounded here
    const float* p; int rs, cs;
    __device__ __forceinline__ uint32_t operator()(int r, int c) const { return __float_as_uint(tf32r(p[r * rs + c * cs])); }
};
struct VF32RN {    // fp32, negated and rounded here
    const float* p; int rs, cs;
    __device__ __forceinline__ uint32_t operator()(int r, int c) const { return __float_as_uint(tf32r(-p[r * rs + c * cs])); }
};
struct VBF16 {     // bf16 (exact in tf32)
    const __nv_bfloat16* p; int rs, cs;
    __device__ __forceinline__ uint32_t operator()(int r, int c) const {
        return (uint32_t)__bfloat16_as_ushort(p[r * rs + c * cs]) << 16;
    }
};

// tile_mma over operand views (same tile and fragment conventions as tile_mma)
template <int MI, int NI, class VA, class VB>
__device__ __forceinline__ void tile_mma_v(float (&acc)[MI][NI][4], const VA& A, const VB& B, int m0, int n0,
                                           int k0, int k1) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll 2
    for (int k = k0; k < k1; k += 8) {
        uint32_t a[MI][4], b[NI][2];
#pragma unroll
        for (int mi = 0; mi < MI; ++mi) {
            const int r = m0 + 16 * mi + g;
            a[mi][0] = A(r, k + t);
            a[mi][1] = A(r + 8, k + t);
            a[mi][2] = A(r, k + t + 4);
            a[mi][3] = A(r + 8, k + t + 4);
        }
#pragma unroll
        for (int ni = 0; ni < NI; ++ni) {
            b[ni][0] = B(k + t, n0 + 8 * ni + g);
            b[ni][1] = B(k + t + 4, n0 + 8 * ni + g);
        }
#pragma unroll
        for (int mi = 0; mi < MI; ++mi)
#pragma unroll
            for (int ni = 0; ni < NI; ++ni) mma_tf32(acc[mi][ni], a[mi], b[ni]);
    }
}

constexpr int kScThreads = 256;
constexpr int kLdb = 136;   // bf16 row stride of [64][128] tiles (272 bytes)
constexpr int kLdo = 72;    // bf16 row stride of [64][64] tiles (144 bytes)

// Fragment <-> global [128][dv] state slice (columns v0 ..): rows m0 + 16 mi + {g, g+8}.
__device__ __forceinline__ void frag_load_state(float (&s)[2][4][4], const float* src, int dv, int m0, int n0) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int mi = 0; mi < 2; ++mi)
#pragma unroll
        for (int ni = 0; ni < 4; ++ni) {
            const int r = m0 + 16 * mi + g, cc = n0 + 8 * ni + 2 * t;
            float2 lo = make_float2(0.f, 0.f), hi = lo;
            if (src) {
                lo = *reinterpret_cast<const float2*>(src + (size_t)r * dv + cc);
                hi = *reinterpret_cast<const float2*>(src + (size_t)(r + 8) * dv + cc);
            }
            s[mi][ni][0] = lo.x; s[mi][ni][1] = lo.y; s[mi][ni][2] = hi.x; s[mi][ni][3] = hi.y;
        }
}
// Writes the slice to global memory (dst, row stride dv) and its tf32 copy to shared (ld kLd).
__device__ __forceinline__ void frag_store_state(const float (&s)[2][4][4], float* dst, int dv, float* sh,
                                                 int m0, int n0) {
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int mi = 0; mi < 2; ++mi)
#pragma unroll
        for (int ni = 0; ni < 4; ++ni) {
            const int r = m0 + 16 * mi + g, cc = n0 + 8 * ni + 2 * t;
            if (dst) {
                *reinterpret_cast<float2*>(dst + (size_t)r * dv + cc) = make_float2(s[mi][ni][0], s[mi][ni][1]);
                *reinterpret_cast<float2*>(dst + (size_t)(r + 8) * dv + cc) = make_float2(s[mi][ni][2], s[mi][ni][3]);
            }
            if (sh) {
                *reinterpret_cast<float2*>(sh + r * kLd + cc) = make_float2(tf32r(s[mi][ni][0]), tf32r(s[mi][ni][1]));
                *reinterpret_cast<float2*>(sh + (r + 8) * kLd + cc) =
                    make_float2(tf32r(s[mi][ni][2]), tf32r(s[mi][ni][3]));
            }
        }
}

// ---- state scan: Sc[c] = S;  Up = U - W S;  S += K^T Up
constexpr int kSsW = 0;                         // W  fp32 [64][kLdk]
constexpr int kSsU = kSsW + kC * kLdk;          // U  fp32 [64][kLd]
constexpr int kSsK = kSsU + kC * kLd;           // K  bf16 [64][kLdb]
constexpr int kSsS = kSsK + kC * kLdb / 2;      // tf32 S  [128][kLd]
constexpr int kSsUp = kSsS + kDk * kLd;         // tf32 Up [64][kLd]
constexpr size_t kSsSmem = (size_t)(kSsUp + kC * kLd) * sizeof(float);

struct SsArgs {
    const void* k;
    const float* W;
    const float* U;
    const float* S0;
    float* Up;
    float* Sc;
    float* S_final;
    int L, dv_, NC;
};

__global__ void __launch_bounds__(kScThreads, 1) k_scan_mma(SsArgs a) {
    extern __shared__ __align__(16) float sm[];
    const long long bh = blockIdx.x;
    const int v0 = blockIdx.y * kBV, dv = a.dv_;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
    float* Ws = sm + kSsW;
    float* Us = sm + kSsU;
    __nv_bfloat16* Kb = reinterpret_cast<__nv_bfloat16*>(sm + kSsK);
    float* Ss = sm + kSsS;
    float* Ups = sm + kSsUp;
    const int sm0 = 32 * (warp & 3), sn0 = 32 * (warp >> 2);   // state tile [128][64]
    const int qm = 16 * (warp & 3), qn = 32 * (warp >> 2);     // Up tile [64][64]

    auto load_WU = [&](int c) {
        const size_t chunk = (size_t)bh * a.NC + c;
        const float* Wg = a.W + chunk * kC * kDk;
        const float* Ug = a.U + chunk * kC * dv + v0;
        for (int e = tid; e < kC * kDk / 4; e += kScThreads) {
            const int i = e >> 5, x4 = (e & 31) * 4;
            cp_async16(Ws + i * kLdk + x4, Wg + i * kDk + x4, true);
        }
        for (int e = tid; e < kC * kBV / 4; e += kScThreads) {
            const int i = e >> 4, n4 = (e & 15) * 4;
            cp_async16(Us + i * kLd + n4, Ug + (size_t)i * dv + n4, true);
        }
        cp_async_commit();
    };
    auto load_K = [&](int c) {
        const int nvalid = min(kC, a.L - c * kC);
        const __nv_bfloat16* Kg = (const __nv_bfloat16*)a.k + (bh * a.L + (long long)c * kC) * kDk;
        for (int e = tid; e < kC * kDk / 8; e += kScThreads) {
            const int i = e >> 4, x8 = (e & 15) * 8;
            cp_async16(Kb + i * kLdb + x8, i < nvalid ? Kg + (size_t)i * kDk + x8 : Kg, i < nvalid);
        }
        cp_async_commit();
    };

    float S[2][4][4];
    frag_load_state(S, a.S0 ? a.S0 + (size_t)bh * kDk * dv + v0 : nullptr, dv, sm0, sn0);
    load_WU(0);
    for (int c = 0; c < a.NC; ++c) {
        const size_t chunk = (size_t)bh * a.NC + c;
        load_K(c);
        frag_store_state(S, a.Sc + chunk * kDk * dv + v0, dv, Ss, sm0, sn0);
        cp_async_wait<1>();   // W, U of chunk c
        __syncthreads();
        {   // Up = U - W S
            float up[1][4][4];
            zero(up);
            tile_mma_v<1, 4>(up, VF32R{Ws, kLdk, 1}, VF32{Ss, kLd, 1}, qm, qn, 0, kDk);
            float* Upg = a.Up + chunk * kC * dv + v0;
#pragma unroll
            for (int ni = 0; ni < 4; ++ni) {
                const int r0 = qm + g, r1 = r0 + 8, cc = qn + 8 * ni + 2 * t;
                const float u0 = Us[r0 * kLd + cc] - up[0][ni][0], u1 = Us[r0 * kLd + cc + 1] - up[0][ni][1];
                const float u2 = Us[r1 * kLd + cc] - up[0][ni][2], u3 = Us[r1 * kLd + cc + 1] - up[0][ni][3];
                *reinterpret_cast<float2*>(Upg + (size_t)r0 * dv + cc) = make_float2(u0, u1);
                *reinterpret_cast<float2*>(Upg + (size_t)r1 * dv + cc) = make_float2(u2, u3);
                *reinterpret_cast<float2*>(Ups + r0 * kLd + cc) = make_float2(tf32r(u0), tf32r(u1));
                *reinterpret_cast<float2*>(Ups + r1 * kLd + cc) = make_float2(tf32r(u2), tf32r(u3));
            }
        }
        cp_async_wait<0>();   // K of chunk c
        __syncthreads();      // Up visible; W, U buffers free
        if (c + 1 < a.NC) load_WU(c + 1);
        // S += K^T Up
        tile_mma_v<2, 4>(S, VBF16{Kb, 1, kLdb}, VF32{Ups, kLd, 1}, sm0, sn0, 0, kC);
        __syncthreads();      // K, Up and S copies free
    }
    if (a.S_final) frag_store_state(S, a.S_final + (size_t)bh * kDk * dv + v0, dv, nullptr, sm0, sn0);
}

// ---- reverse scan (G = gradient w.r.t. the state leaving chunk c):
//   dSc[c] = G;  dUp = P^T dO + K G;  G += Q^T dO - W^T dUp;  dS0 = G after chunk 0
constexpr int kRsP = 0;                          // P  fp32 [64 j][kLd]  (P[j][i], zero for i > j)
constexpr int kRsK = kRsP + kC * kLd;            // K  bf16 [64][kLdb]
constexpr int kRsQ = kRsK + kC * kLdb / 2;       // Q  bf16 [64][kLdb]
constexpr int kRsW = kRsQ + kC * kLdb / 2;       // W  fp32 [64][kLdk]
constexpr int kRsO = kRsW + kC * kLdk;           // dO bf16 [2][64][kLdo]
constexpr int kRsG = kRsO + kC * kLdo;           // tf32 G  [128][kLd]
constexpr int kRsU = kRsG + kDk * kLd;           // tf32 dUp [64][kLd]
constexpr size_t kRsSmem = (size_t)(kRsU + kC * kLd) * sizeof(float);

struct RsArgs {
    const void* q;
    const void* k;
    const void* dO;
    const float* W;
    const float* P;
    const float* dS_final;
    float* dUp;
    float* dSc;
    float* dS0;
    const int* mask;   // null, or [BH]: only sequences whose word is set are computed
    int L, dv_, NC;
};

__global__ void __launch_bounds__(kScThreads, 1) k_rscan_mma(RsArgs a) {
    if (a.mask && !a.mask[blockIdx.x]) return;
    extern __shared__ __align__(16) float sm[];
    const long long bh = blockIdx.x;
    const int v0 = blockIdx.y * kBV, dv = a.dv_;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
    float* Ps = sm + kRsP;
    __nv_bfloat16* Kb = reinterpret_cast<__nv_bfloat16*>(sm + kRsK);
    __nv_bfloat16* Qb = reinterpret_cast<__nv_bfloat16*>(sm + kRsQ);
    float* Ws = sm + kRsW;
    __nv_bfloat16* Ob = reinterpret_cast<__nv_bfloat16*>(sm + kRsO);   // two buffers
    float* Gs = sm + kRsG;
    float* dUs = sm + kRsU;
    const int sm0 = 32 * (warp & 3), sn0 = 32 * (warp >> 2);
    const int qm = 16 * (warp & 3), qn = 32 * (warp >> 2);

    auto load_PKO = [&](int c) {
        const size_t chunk = (size_t)bh * a.NC + c;
        const int nvalid = min(kC, a.L - c * kC);
        const long long tok0 = bh * a.L + (long long)c * kC;
        const float* Pg = a.P + chunk * kC * kC;
        for (int e = tid; e < kC * kC / 4; e += kScThreads) {
            const int j = e >> 4, i4 = (e & 15) * 4;
            cp_async16(Ps + j * kLd + i4, Pg + j * kC + i4, true);
        }
        const __nv_bfloat16* Kg = (const __nv_bfloat16*)a.k + tok0 * kDk;
        for (int e = tid; e < kC * kDk / 8; e += kScThreads) {
            const int i = e >> 4, x8 = (e & 15) * 8;
            cp_async16(Kb + i * kLdb + x8, i < nvalid ? Kg + (size_t)i * kDk + x8 : Kg, i < nvalid);
        }
        __nv_bfloat16* Od = Ob + (c & 1) * kC * kLdo;
        const __nv_bfloat16* Og = (const __nv_bfloat16*)a.dO + tok0 * dv + v0;
        for (int e = tid; e < kC * kBV / 8; e += kScThreads) {
            const int i = e >> 3, n8 = (e & 7) * 8;
            cp_async16(Od + i * kLdo + n8, i < nvalid ? Og + (size_t)i * dv + n8 : Og, i < nvalid);
        }
        cp_async_commit();
    };
    auto load_QW = [&](int c) {
        const size_t chunk = (size_t)bh * a.NC + c;
        const int nvalid = min(kC, a.L - c * kC);
        const __nv_bfloat16* Qg = (const __nv_bfloat16*)a.q + (bh * a.L + (long long)c * kC) * kDk;
        for (int e = tid; e < kC * kDk / 8; e += kScThreads) {
            const int i = e >> 4, x8 = (e & 15) * 8;
            cp_async16(Qb + i * kLdb + x8, i < nvalid ? Qg + (size_t)i * kDk + x8 : Qg, i < nvalid);
        }
        const float* Wg = a.W + chunk * kC * kDk;
        for (int e = tid; e < kC * kDk / 4; e += kScThreads) {
            const int i = e >> 5, x4 = (e & 31) * 4;
            cp_async16(Ws + i * kLdk + x4, Wg + i * kDk + x4, true);
        }
        cp_async_commit();
    };

    float G[2][4][4];
    frag_load_state(G, a.dS_final ? a.dS_final + (size_t)bh * kDk * dv + v0 : nullptr, dv, sm0, sn0);
    load_PKO(a.NC - 1);
    for (int c = a.NC - 1; c >= 0; --c) {
        const size_t chunk = (size_t)bh * a.NC + c;
        const __nv_bfloat16* Od = Ob + (c & 1) * kC * kLdo;
        load_QW(c);
        frag_store_state(G, a.dSc + chunk * kDk * dv + v0, dv, Gs, sm0, sn0);
        cp_async_wait<1>();   // P, K, dO of chunk c
        __syncthreads();
        {   // dUp = P^T dO + K G   (P[j][i] = 0 for j < i)
            float du[1][4][4];
            zero(du);
            tile_mma_v<1, 4>(du, VF32R{Ps, 1, kLd}, VBF16{Od, kLdo, 1}, qm, qn, qm, kC);
            tile_mma_v<1, 4>(du, VBF16{Kb, kLdb, 1}, VF32{Gs, kLd, 1}, qm, qn, 0, kDk);
            float* dUg = a.dUp + chunk * kC * dv + v0;
#pragma unroll
            for (int ni = 0; ni < 4; ++ni) {
                const int r0 = qm + g, r1 = r0 + 8, cc = qn + 8 * ni + 2 * t;
                *reinterpret_cast<float2*>(dUg + (size_t)r0 * dv + cc) = make_float2(du[0][ni][0], du[0][ni][1]);
                *reinterpret_cast<float2*>(dUg + (size_t)r1 * dv + cc) = make_float2(du[0][ni][2], du[0][ni][3]);
                *reinterpret_cast<float2*>(dUs + r0 * kLd + cc) = make_float2(tf32r(du[0][ni][0]), tf32r(du[0][ni][1]));
                *reinterpret_cast<float2*>(dUs + r1 * kLd + cc) = make_float2(tf32r(du[0][ni][2]), tf32r(du[0][ni][3]));
            }
        }
        cp_async_wait<0>();   // Q, W of chunk c
        __syncthreads();      // dUp visible; P and K buffers free
        if (c > 0) load_PKO(c - 1);
        // G += Q^T dO - W^T dUp
        tile_mma_v<2, 4>(G, VBF16{Qb, 1, kLdb}, VBF16{Od, kLdo, 1}, sm0, sn0, 0, kC);
        tile_mma_v<2, 4>(G, VF32RN{Ws, 1, kLdk}, VF32{dUs, kLd, 1}, sm0, sn0, 0, kC);
        __syncthreads();      // Q, W, dO(c) and the G / dUp copies free
    }
    if (a.dS0) frag_store_state(G, a.dS0 + (size_t)bh * kDk * dv + v0, dv, nullptr, sm0, sn0);
}

// ------------------------------------------------------------ per-chunk gradients
// Phase 1 walks the value dimension in 32-column slices, double-buffered: slice s + 1 is in
// flight (cp.async) while slice s is multiplied.  T, Q and K arrive with slice 0 and stay;
// bf16 operands stay bf16 in shared memory, and every thread rounds the fp32 chunks it
// copied to tf32 in place once they land (its own copies are visible to it after the
// wait), before the barrier that publishes them.  Phase 2 reuses the slice buffers.
constexpr int kSv = 32;                           // value columns per slice
constexpr int kLs = 36;                           // fp32 row stride of [*][32] slices
constexpr int kLso = 40;                          // bf16 row stride of [64][32] slices (80 bytes)
constexpr int kSlots = 14;                        // dalpha sources: 8 (value slices) + 4 + 2
constexpr int kGmT = 0;                           // T fp32 [64][kLd] (tf32 after slice 0 lands)
constexpr int kGmQ = kGmT + kC * kLd;             // Q bf16 [64][kLdb]
constexpr int kGmK = kGmQ + kC * kLdb / 2;        // K bf16 [64][kLdb]
constexpr int kGmPart = kGmK + kC * kLdb / 2;     // dalpha partial sums [16][64]
constexpr int kGmAl = kGmPart + 16 * kC;          // alpha, beta, lambda [64] each
constexpr int kGmR = kGmAl + 3 * kC;              // slice buffers | phase-2 tiles
// one slice: S, dS' fp32 [128][kLs]; Up, dUp fp32 [64][kLs]; dO, V bf16 [64][kLso]
constexpr int kSlS = 0, kSldS = kSlS + kDk * kLs, kSlUp = kSldS + kDk * kLs, kSldU = kSlUp + kC * kLs;
constexpr int kSlO = kSldU + kC * kLs, kSlV = kSlO + kC * kLso / 2, kSlice = kSlV + kC * kLso / 2;
constexpr int kPh2 = 3 * kC * kLd + kC * kLdk;    // D (then E), dT, X [64][kLd]; dW [64][kLdk]
constexpr int kGmRegion = 2 * kSlice > kPh2 ? 2 * kSlice : kPh2;
constexpr size_t kGmSmem = (size_t)(kGmR + kGmRegion) * sizeof(float);
static_assert(kGmR % 4 == 0 && kSlice % 4 == 0 && kSlO % 4 == 0 && kSlV % 4 == 0, "16-byte regions");

// One chunk's gradients (the body of k_grad_mma).
__device__ __forceinline__ void grad_mma_chunk(const GmArgs& a, const long long bh, const int c) {
    extern __shared__ __align__(16) float sm[];
    const int dv = a.dv_, ns = dv / kSv;
    const int t0 = c * kC, nvalid = min(kC, a.L - t0);
    const long long tok0 = bh * a.L + t0;
    const size_t chunk = (size_t)bh * a.NC + c;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
    const int obf = a.out_bf16;

    float* Ts = sm + kGmT;
    __nv_bfloat16* Qb = reinterpret_cast<__nv_bfloat16*>(sm + kGmQ);
    __nv_bfloat16* Kb = reinterpret_cast<__nv_bfloat16*>(sm + kGmK);
    float* part = sm + kGmPart;
    float* al = sm + kGmAl;
    float* bet = al + kC;
    float* lam = bet + kC;
    float* R = sm + kGmR;
    float* dWs = R;                    // phase 2 views
    float* Ds = dWs + kC * kLdk;       // D, later E = dG + dG^T
    float* dTs = Ds + kC * kLd;
    float* Xs = dTs + kC * kLd;

    const int wm = 32 * (warp & 1), wn = 32 * (warp >> 1);    // [64][128] tiles 32 x 32
    const int qm = 16 * (warp & 3), qn = 32 * (warp >> 2);    // [64][64] tiles 16 x 32
    const int vn = 16 * (warp >> 2);                          // [64][32] tiles 16 x 16 (rows qm)
    const bool lower_tile = qn <= qm + 14;

    const __nv_bfloat16* dOg = (const __nv_bfloat16*)a.dO + tok0 * dv;
    const __nv_bfloat16* Vg = (const __nv_bfloat16*)a.v + tok0 * dv;
    auto load_slice = [&](int s) {
        float* b = R + (s & 1) * kSlice;
        const int v0 = s * kSv;
        const float* Scg = a.Sc + chunk * kDk * dv + v0;
        const float* dScg = a.dSc + chunk * kDk * dv + v0;
        for (int e = tid; e < kDk * kSv / 4; e += kGmThreads) {
            const int x = e >> 3, n4 = (e & 7) * 4;
            cp_async16(b + kSlS + x * kLs + n4, Scg + (size_t)x * dv + n4, true);
            cp_async16(b + kSldS + x * kLs + n4, dScg + (size_t)x * dv + n4, true);
        }
        const float* Upg = a.Up + chunk * kC * dv + v0;
        const float* dUg = a.dUp + chunk * kC * dv + v0;
        for (int e = tid; e < kC * kSv / 4; e += kGmThreads) {
            const int i = e >> 3, n4 = (e & 7) * 4;
            cp_async16(b + kSlUp + i * kLs + n4, Upg + (size_t)i * dv + n4, true);
            cp_async16(b + kSldU + i * kLs + n4, dUg + (size_t)i * dv + n4, true);
        }
        __nv_bfloat16* Ob = reinterpret_cast<__nv_bfloat16*>(b + kSlO);
        __nv_bfloat16* Vb = reinterpret_cast<__nv_bfloat16*>(b + kSlV);
        for (int e = tid; e < kC * kSv / 8; e += kGmThreads) {
            const int i = e >> 2, n8 = (e & 3) * 8;
            const bool ok = i < nvalid;
            cp_async16(Ob + i * kLso + n8, ok ? dOg + (size_t)i * dv + v0 + n8 : dOg, ok);
            cp_async16(Vb + i * kLso + n8, ok ? Vg + (size_t)i * dv + v0 + n8 : Vg, ok);
        }
    };

    auto round_own = [&](float* p) {   // a 16-byte chunk this thread copied, to tf32
        float4* q4 = reinterpret_cast<float4*>(p);
        *q4 = tf32r4(*q4);
    };
    auto round_slice = [&](int s) {   // the fp32 chunks of slice s that this thread copied
        float* b = R + (s & 1) * kSlice;
        for (int e = tid; e < kDk * kSv / 4; e += kGmThreads) {
            const int x = e >> 3, n4 = (e & 7) * 4;
            round_own(b + kSlS + x * kLs + n4);
            round_own(b + kSldS + x * kLs + n4);
        }
        for (int e = tid; e < kC * kSv / 4; e += kGmThreads) {
            const int i = e >> 3, n4 = (e & 7) * 4;
            round_own(b + kSlUp + i * kLs + n4);
            round_own(b + kSldU + i * kLs + n4);
        }
    };

    {   // T, Q, K and slice 0 in one group
        const float* Tg = a.T + chunk * kC * kC;
        for (int e = tid; e < kC * kC / 4; e += kGmThreads) {
            const int i = e >> 4, j4 = (e & 15) * 4;
            cp_async16(Ts + i * kLd + j4, Tg + i * kC + j4, true);
        }
        const __nv_bfloat16* Qg = (const __nv_bfloat16*)a.q + tok0 * kDk;
        const __nv_bfloat16* Kg = (const __nv_bfloat16*)a.k + tok0 * kDk;
        for (int e = tid; e < kC * kDk / 8; e += kGmThreads) {
            const int i = e >> 4, x8 = (e & 15) * 8;
            const bool ok = i < nvalid;
            cp_async16(Qb + i * kLdb + x8, ok ? Qg + (size_t)i * kDk + x8 : Qg, ok);
            cp_async16(Kb + i * kLdb + x8, ok ? Kg + (size_t)i * kDk + x8 : Kg, ok);
        }
        load_slice(0);
        cp_async_commit();
        if (tid < kC) {
            al[tid] = a.alpha[chunk * kC + tid];
            bet[tid] = tid < nvalid ? a.beta[tok0 + tid] : 0.f;
        }
    }

    float dQa[2][4][4], dKa[2][4][4], dWa[2][4][4], Da[1][4][4], dTa[1][4][4];
    zero(dQa); zero(dKa); zero(dWa); zero(Da); zero(dTa);

    // ---- phase 1
    for (int s = 0; s < ns; ++s) {
        if (s + 1 < ns) {
            load_slice(s + 1);
            cp_async_commit();
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        if (s == 0)   // T (copied with the same indexing) to tf32
            for (int e = tid; e < kC * kC / 4; e += kGmThreads) round_own(Ts + (e >> 4) * kLd + (e & 15) * 4);
        round_slice(s);
        __syncthreads();
        const float* b = R + (s & 1) * kSlice;
        const VF32 Sv{b + kSlS, 1, kLs}, dSv{b + kSldS, 1, kLs};           // B(n, x) = S[x][n]
        const VF32 UpA{b + kSlUp, kLs, 1}, dUA{b + kSldU, kLs, 1};         // A(i, n)
        const VBF16 OA{reinterpret_cast<const __nv_bfloat16*>(b + kSlO), kLso, 1};
        // dQ += dO S^T,  dW += dUp S^T (negated below),  dK += Up dS'^T
        tile_mma_v<2, 4>(dQa, OA, Sv, wm, wn, 0, kSv);
        tile_mma_v<2, 4>(dWa, dUA, Sv, wm, wn, 0, kSv);
        tile_mma_v<2, 4>(dKa, UpA, dSv, wm, wn, 0, kSv);
        if (lower_tile) {   // D += dO Up^T,  dT += dUp V^T (alpha_j applied later)
            tile_mma_v<1, 4>(Da, OA, VF32{b + kSlUp, 1, kLs}, qm, qn, 0, kSv);
            tile_mma_v<1, 4>(dTa, dUA, VBF16{reinterpret_cast<const __nv_bfloat16*>(b + kSlV), 1, kLso},
                             qm, qn, 0, kSv);
        }
        {   // dVa = T^T dUp;  dV = alpha dVa;  dalpha += <dVa, v>
            float va[1][2][4];
            zero(va);
            tile_mma_v<1, 2>(va, VF32{Ts, 1, kLd}, VF32{b + kSldU, kLs, 1}, qm, vn, qm, kC);
            const __nv_bfloat16* Vb = reinterpret_cast<const __nv_bfloat16*>(b + kSlV);
            const int r0 = qm + g, r1 = r0 + 8, v0 = s * kSv;
            float p0 = 0.f, p1 = 0.f;
#pragma unroll
            for (int ni = 0; ni < 2; ++ni) {
                const int cc = vn + 8 * ni + 2 * t;
                if (r0 < nvalid)
                    st_pair(a.dv, (size_t)(tok0 + r0) * dv + v0 + cc, al[r0] * va[0][ni][0],
                            al[r0] * va[0][ni][1], obf);
                if (r1 < nvalid)
                    st_pair(a.dv, (size_t)(tok0 + r1) * dv + v0 + cc, al[r1] * va[0][ni][2],
                            al[r1] * va[0][ni][3], obf);
                p0 = fmaf(va[0][ni][0], __bfloat162float(Vb[r0 * kLso + cc]), p0);
                p0 = fmaf(va[0][ni][1], __bfloat162float(Vb[r0 * kLso + cc + 1]), p0);
                p1 = fmaf(va[0][ni][2], __bfloat162float(Vb[r1 * kLso + cc]), p1);
                p1 = fmaf(va[0][ni][3], __bfloat162float(Vb[r1 * kLso + cc + 1]), p1);
            }
            p0 += __shfl_xor_sync(0xffffffffu, p0, 1);
            p0 += __shfl_xor_sync(0xffffffffu, p0, 2);
            p1 += __shfl_xor_sync(0xffffffffu, p1, 1);
            p1 += __shfl_xor_sync(0xffffffffu, p1, 2);
            if (t == 0) {
                part[(2 * s + (warp >> 2)) * kC + r0] = p0;
                part[(2 * s + (warp >> 2)) * kC + r1] = p1;
            }
        }
        __syncthreads();   // slice s read: its buffer may be refilled
    }

    // ---- phase 2 (the slice buffers become dW, D, dT, X)
#pragma unroll
    for (int mi = 0; mi < 2; ++mi)
#pragma unroll
        for (int ni = 0; ni < 4; ++ni) {
            const int r0 = wm + 16 * mi + g, cc = wn + 8 * ni + 2 * t;
            *reinterpret_cast<float2*>(dWs + r0 * kLdk + cc) = make_float2(tf32r(-dWa[mi][ni][0]), tf32r(-dWa[mi][ni][1]));
            *reinterpret_cast<float2*>(dWs + (r0 + 8) * kLdk + cc) =
                make_float2(tf32r(-dWa[mi][ni][2]), tf32r(-dWa[mi][ni][3]));
        }
#pragma unroll
    for (int ni = 0; ni < 4; ++ni) {   // D = tril(dO Up^T), diagonal included
        const int r0 = qm + g, r1 = r0 + 8, cc = qn + 8 * ni + 2 * t;
        Ds[r0 * kLd + cc] = cc <= r0 ? tf32r(Da[0][ni][0]) : 0.f;
        Ds[r0 * kLd + cc + 1] = cc + 1 <= r0 ? tf32r(Da[0][ni][1]) : 0.f;
        Ds[r1 * kLd + cc] = cc <= r1 ? tf32r(Da[0][ni][2]) : 0.f;
        Ds[r1 * kLd + cc + 1] = cc + 1 <= r1 ? tf32r(Da[0][ni][3]) : 0.f;
    }
    for (int i = warp; i < kC; i += kGmThreads / 32) {   // lambda_i = ||k_i||^2
        float sq = 0.f;
        for (int x = lane; x < kDk; x += 32) {
            const float kx = __bfloat162float(Kb[i * kLdb + x]);
            sq = fmaf(kx, kx, sq);
        }
        sq = warp_sum(sq);
        if (lane == 0) lam[i] = sq;
    }
    __syncthreads();
    const VBF16 KB{Kb, kLdb, 1};    // B(j, x) = K[j][x]   (also A(i, x) = K[i][x])
    const VBF16 KT{Kb, 1, kLdb};    // B(x, j) = K[j][x]
    // dQ += D K (D[i][j] = 0 for j > i),  dK += D^T Q (D[j][i] = 0 for j < i)
    tile_mma_v<2, 4>(dQa, VF32{Ds, kLd, 1}, KB, wm, wn, 0, wm + 32);
    tile_mma_v<2, 4>(dKa, VF32{Ds, 1, kLd}, VBF16{Qb, kLdb, 1}, wm, wn, wm, kC);
    {   // dKa = T^T dW;  dK += alpha dKa;  dalpha += <dKa, k>
        float ka[2][4][4];
        zero(ka);
        tile_mma_v<2, 4>(ka, VF32{Ts, 1, kLd}, VF32{dWs, kLdk, 1}, wm, wn, wm, kC);
#pragma unroll
        for (int mi = 0; mi < 2; ++mi) {
            const int r0 = wm + 16 * mi + g, r1 = r0 + 8;
            const float a0 = al[r0], a1 = al[r1];
            float p0 = 0.f, p1 = 0.f;
#pragma unroll
            for (int ni = 0; ni < 4; ++ni) {
                const int cc = wn + 8 * ni + 2 * t;
                dKa[mi][ni][0] = fmaf(a0, ka[mi][ni][0], dKa[mi][ni][0]);
                dKa[mi][ni][1] = fmaf(a0, ka[mi][ni][1], dKa[mi][ni][1]);
                dKa[mi][ni][2] = fmaf(a1, ka[mi][ni][2], dKa[mi][ni][2]);
                dKa[mi][ni][3] = fmaf(a1, ka[mi][ni][3], dKa[mi][ni][3]);
                p0 = fmaf(ka[mi][ni][0], __bfloat162float(Kb[r0 * kLdb + cc]), p0);
                p0 = fmaf(ka[mi][ni][1], __bfloat162float(Kb[r0 * kLdb + cc + 1]), p0);
                p1 = fmaf(ka[mi][ni][2], __bfloat162float(Kb[r1 * kLdb + cc]), p1);
                p1 = fmaf(ka[mi][ni][3], __bfloat162float(Kb[r1 * kLdb + cc + 1]), p1);
            }
            p0 += __shfl_xor_sync(0xffffffffu, p0, 1);
            p0 += __shfl_xor_sync(0xffffffffu, p0, 2);
            p1 += __shfl_xor_sync(0xffffffffu, p1, 1);
            p1 += __shfl_xor_sync(0xffffffffu, p1, 2);
            if (t == 0) {
                part[(8 + (warp >> 1)) * kC + r0] = p0;
                part[(8 + (warp >> 1)) * kC + r1] = p1;
            }
        }
    }
    // dT = (dUp V^T + dW K^T) diag(alpha), strictly lower part kept
    if (lower_tile) tile_mma_v<1, 4>(dTa, VF32{dWs, kLdk, 1}, KT, qm, qn, 0, kDk);
#pragma unroll
    for (int ni = 0; ni < 4; ++ni) {
        const int r0 = qm + g, r1 = r0 + 8, cc = qn + 8 * ni + 2 * t;
        const float a0 = al[cc], a1 = al[cc + 1];
        dTs[r0 * kLd + cc] = cc < r0 ? tf32r(a0 * dTa[0][ni][0]) : 0.f;
        dTs[r0 * kLd + cc + 1] = cc + 1 < r0 ? tf32r(a1 * dTa[0][ni][1]) : 0.f;
        dTs[r1 * kLd + cc] = cc < r1 ? tf32r(a0 * dTa[0][ni][2]) : 0.f;
        dTs[r1 * kLd + cc + 1] = cc + 1 < r1 ? tf32r(a1 * dTa[0][ni][3]) : 0.f;
    }
    __syncthreads();
    {   // X = dT T^T, strictly lower part (dT[i][l] = 0 for l >= i, T[j][l] = 0 for l > j)
        float xa[1][4][4];
        zero(xa);
        if (lower_tile)
            tile_mma_v<1, 4>(xa, VF32{dTs, kLd, 1}, VF32{Ts, 1, kLd}, qm, qn, 0, min(qn + 32, qm + 16));
#pragma unroll
        for (int ni = 0; ni < 4; ++ni) {
            const int r0 = qm + g, r1 = r0 + 8, cc = qn + 8 * ni + 2 * t;
            Xs[r0 * kLd + cc] = cc < r0 ? tf32r(xa[0][ni][0]) : 0.f;
            Xs[r0 * kLd + cc + 1] = cc + 1 < r0 ? tf32r(xa[0][ni][1]) : 0.f;
            Xs[r1 * kLd + cc] = cc < r1 ? tf32r(xa[0][ni][2]) : 0.f;
            Xs[r1 * kLd + cc + 1] = cc + 1 < r1 ? tf32r(xa[0][ni][3]) : 0.f;
        }
    }
    __syncthreads();
    {   // dA = strict_lower(-T^T X), G = K K^T; dalpha += sum_{j<i} dA G; E = dG + dG^T over D
        float da[1][4][4], ga[1][4][4];
        zero(da); zero(ga);
        if (lower_tile) {
            tile_mma_v<1, 4>(da, VF32{Ts, 1, kLd}, VF32{Xs, kLd, 1}, qm, qn, qm, kC);
            tile_mma_v<1, 4>(ga, KB, KT, qm, qn, 0, kDk);
        }
        const int r0 = qm + g, r1 = r0 + 8;
        float p0 = 0.f, p1 = 0.f;
#pragma unroll
        for (int ni = 0; ni < 4; ++ni) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int r = e < 2 ? r0 : r1, cc = qn + 8 * ni + 2 * t + (e & 1);
                if (cc < r) {
                    const float dA = -da[0][ni][e];
                    if (e < 2) p0 = fmaf(dA, ga[0][ni][e], p0);
                    else p1 = fmaf(dA, ga[0][ni][e], p1);
                    const float dG = tf32r(al[r] * dA);
                    Ds[r * kLd + cc] = dG;
                    Ds[cc * kLd + r] = dG;
                } else if (cc == r) {
                    Ds[r * kLd + cc] = 0.f;
                }
            }
        }
        p0 += __shfl_xor_sync(0xffffffffu, p0, 1);
        p0 += __shfl_xor_sync(0xffffffffu, p0, 2);
        p1 += __shfl_xor_sync(0xffffffffu, p1, 1);
        p1 += __shfl_xor_sync(0xffffffffu, p1, 2);
        if (t == 0) {
            part[(12 + (warp >> 2)) * kC + r0] = p0;
            part[(12 + (warp >> 2)) * kC + r1] = p1;
        }
    }
    __syncthreads();
    tile_mma_v<2, 4>(dKa, VF32{Ds, kLd, 1}, KB, wm, wn, 0, kC);   // dK += E K
    // dalpha (fixed order over its sources), dK += 2 dlambda K, outputs
#pragma unroll
    for (int mi = 0; mi < 2; ++mi) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int r = wm + 16 * mi + g + 8 * h;
            float dal = 0.f;
            for (int q = 0; q < kSlots; ++q)
                if (q >= 8 || q < 2 * ns) dal += part[q * kC + r];
            const float dl2 = 2.f * dal * dalpha_dlambda_of(bet[r], lam[r], a.euler);
            if (r < nvalid) {
#pragma unroll
                for (int ni = 0; ni < 4; ++ni) {
                    const int cc = wn + 8 * ni + 2 * t;
                    const float k0 = __bfloat162float(Kb[r * kLdb + cc]), k1 = __bfloat162float(Kb[r * kLdb + cc + 1]);
                    st_pair(a.dq, (size_t)(tok0 + r) * kDk + cc, dQa[mi][ni][2 * h], dQa[mi][ni][2 * h + 1], obf);
                    st_pair(a.dk, (size_t)(tok0 + r) * kDk + cc, fmaf(dl2, k0, dKa[mi][ni][2 * h]),
                            fmaf(dl2, k1, dKa[mi][ni][2 * h + 1]), obf);
                }
            }
        }
    }
    if (tid < nvalid) {
        float dal = 0.f;
        for (int q = 0; q < kSlots; ++q)
            if (q >= 8 || q < 2 * ns) dal += part[q * kC + tid];
        a.dbeta[tok0 + tid] = dal * dalpha_dbeta_of(bet[tid], lam[tid], a.euler);
    }
}

template <bool kList>
__global__ void __launch_bounds__(kGmThreads, 1) k_grad_mma(GmArgs a) {
    if constexpr (!kList) {   // every chunk, one per CTA
        grad_mma_chunk(a, blockIdx.x, blockIdx.y);
        return;
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");   // (a programmatic dependent: the list is final)
    const int n = *a.list_n;   // the listed chunks, grid-stride
    for (int w = blockIdx.x; w < n; w += gridDim.x) {
        const int chunk = a.list[w];
        grad_mma_chunk(a, chunk / a.NC, chunk % a.NC);
        __syncthreads();   // shared memory is reused by the next chunk
    }
}

}  // namespace

bool grad_mma_supported(const Dims& d) {
    return d.tensor && d.in_bf16 && d.dk == kDk && d.C == kC && (d.dv == 64 || d.dv == 128);
}

cudaError_t launch_scan_mma(const Dims& d, const void* k, const float* S0, const BwdWs& ws,
                            cudaStream_t st) {
    SsArgs sa{k, ws.f.W, ws.f.U, S0, ws.f.Up, ws.f.Sc, nullptr, d.L, d.dv, d.NC};
    cudaError_t e = cudaFuncSetAttribute(k_scan_mma, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSsSmem);
    if (e != cudaSuccess) return e;
    k_scan_mma<<<dim3((unsigned)d.BH(), d.dv / kBV), kScThreads, kSsSmem, st>>>(sa);
    return cudaGetLastError();
}

cudaError_t launch_rscan_mma(const Dims& d, const void* q, const void* k, const void* dO,
                             const float* dS_final, float* dS0, const BwdWs& ws, cudaStream_t st,
                             const int* mask) {
    RsArgs ra{q, k, dO, ws.f.W, ws.P, dS_final, ws.dUp, ws.dSc, dS0, mask, d.L, d.dv, d.NC};
    cudaError_t e = cudaFuncSetAttribute(k_rscan_mma, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kRsSmem);
    if (e != cudaSuccess) return e;
    k_rscan_mma<<<dim3((unsigned)d.BH(), d.dv / kBV), kScThreads, kRsSmem, st>>>(ra);
    return cudaGetLastError();
}

// Grid of a list-driven launch: a few CTAs per SM, so an empty list costs one small launch.
static cudaError_t list_grid(unsigned* grid, long long work, int per_sm) {
    int dev = 0, nsm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const long long g = (long long)nsm * per_sm;
    *grid = (unsigned)(work < g ? (work > 0 ? work : 1) : g);
    return cudaSuccess;
}

cudaError_t launch_prep_mma(const Dims& d, const void* q, const void* k, const void* v,
                            const float* beta, const BwdWs& ws, cudaStream_t st, const int* list,
                            const int* list_n) {
    PmArgs pa{q, k, v, beta, ws.f.alpha, ws.f.W, ws.f.U, ws.T, ws.P, list, list_n, d.L, d.dv, d.NC, d.euler};
    cudaError_t e;
    if (list) {
        unsigned grid = 0;
        if ((e = list_grid(&grid, d.BH() * d.NC, 2)) != cudaSuccess) return e;
        if ((e = cudaFuncSetAttribute(k_prep_mma<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPmSmem)) !=
            cudaSuccess)
            return e;
        k_prep_mma<true><<<grid, kPmThreads, kPmSmem, st>>>(pa);
    } else {
        if ((e = cudaFuncSetAttribute(k_prep_mma<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)kPmSmem)) != cudaSuccess)
            return e;
        k_prep_mma<false><<<dim3((unsigned)d.BH(), d.NC), kPmThreads, kPmSmem, st>>>(pa);
    }
    return cudaGetLastError();
}

cudaError_t launch_grad_mma(const Dims& d, const void* q, const void* k, const void* v,
                            const void* dO, const float* beta, const BwdWs& ws, void* dq, void* dk,
                            void* dv, float* dbeta, cudaStream_t st, const int* list, const int* list_n) {
    GmArgs ga{q, k, v, dO, beta, ws.f.alpha, ws.T, ws.f.Sc, ws.dSc, ws.f.Up, ws.dUp,
              dq, dk, dv, dbeta, list, list_n, d.L, d.dv, d.NC, d.euler, d.out_bf16};
    cudaError_t e;
    if (list) {
        unsigned grid = 0;
        if ((e = list_grid(&grid, d.BH() * d.NC, 1)) != cudaSuccess) return e;
        if ((e = cudaFuncSetAttribute(k_grad_mma<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGmSmem)) !=
            cudaSuccess)
            return e;
        // a programmatic dependent of the launch before it (k_widen), like that one
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(kGmThreads);
        cfg.dynamicSmemBytes = kGmSmem;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if ((e = cudaLaunchKernelEx(&cfg, k_grad_mma<true>, ga)) != cudaSuccess) return e;
    } else {
        if ((e = cudaFuncSetAttribute(k_grad_mma<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)kGmSmem)) != cudaSuccess)
            return e;
        k_grad_mma<false><<<dim3((unsigned)d.BH(), d.NC), kGmThreads, kGmSmem, st>>>(ga);
    }
    return cudaGetLastError();
}

}  // namespace efla

// bwd_simt.cu -- chunkwise backward pass of EFLA on CUDA cores (fp32 arithmetic).
//
// Reverse-mode differentiation of the chunk form used by the forward pass
// (page es, Metodologia item 3: update rule and alpha; the pages state no
// backward pass, so everything here follows from calculus on that form):
//   forward per chunk:  A = strict_lower(diag(alpha) G), G = K K^T, T = (I + A)^{-1},
//                       W = T diag(alpha) K, U = T diag(alpha) V, Up = U - W S,
//                       S' = S + K^T Up,  O = Q S + P Up,  P = tril(Q K^T)
//   reverse scan (sequential over chunks, G' = dLoss/dS'):
//                       dUp = P^T dO + K G'
//                       dS  = G' + Q^T dO - W^T dUp
//   per-chunk gradients (parallel over chunks):
//                       D   = tril(dO Up^T)                (diagonal included)
//                       dQ  = dO S^T + D K
//                       dK  = D^T Q + Up G'^T + (dG + dG^T) K + diag(alpha) dKa + 2 diag(dlambda) K
//                       dW  = -dUp S^T,  dT = dW (aK)^T + dUp (aV)^T
//                       dKa = T^T dW,    dVa = T^T dUp,   dV = diag(alpha) dVa
//                       dA  = strict_lower(-T^T dT T^T),   dG = diag(alpha) dA
//                       dalpha_i = sum_{j<i} dA_ij G_ij + <dKa_i, k_i> + <dVa_i, v_i>
//                       dbeta = dalpha * dalpha/dbeta,  dlambda = dalpha * dalpha/dlambda
#include "common.cuh"
#include "launch.h"

namespace efla {

constexpr int kNTb = 256;

// The backward kernels stage every operand through shared memory, so the element
// type of q, k, v, dO (and of dq, dk, dv) is a runtime flag rather than a template
// parameter: one instantiation per kernel keeps the build short.
__device__ __forceinline__ float ld_in(const void* p, size_t i, int bf16) {
    return bf16 ? __bfloat162float(((const __nv_bfloat16*)p)[i]) : __ldg((const float*)p + i);
}
__device__ __forceinline__ void st_out(void* p, size_t i, float x, int bf16) {
    if (bf16) ((__nv_bfloat16*)p)[i] = __float2bfloat16_rn(x);
    else ((float*)p)[i] = x;
}

cudaError_t launch_prep_for_bwd(const Dims& d, const void* q, const void* k, const void* v,
                                const float* beta, const BwdWs& ws, cudaStream_t st);
cudaError_t launch_scan_for_bwd(const Dims& d, const void* k, const float* S0, const BwdWs& ws,
                                cudaStream_t st);

size_t bwd_ws_bytes(const Dims& d) {
    const size_t bh = (size_t)d.BH(), nc = (size_t)d.NC, C = d.C;
    return fwd_ws_bytes(d) + 2 * align256(bh * nc * C * C * 4) + align256(bh * nc * C * d.dv * 4) +
           align256(bh * nc * (size_t)d.dk * d.dv * 4) + rscan_tc_ws_bytes(d) + grad_tc_ws_bytes(d);
}

size_t states_bytes(const Dims& d) {
    const size_t bh = (size_t)d.BH(), nc = (size_t)d.NC;
    return align256(bh * nc * d.dk * d.dv * 4) + align256(bh * nc * d.C * d.dv * 4) +
           align256(bh * nc * d.C * d.C * 4) + align256(bh * nc * d.C * 4);
}

float* states_Up(const Dims& d, float* states) {
    return (float*)((char*)states + align256((size_t)d.BH() * d.NC * d.dk * d.dv * 4));
}

float* states_T(const Dims& d, float* states) {
    return (float*)((char*)states_Up(d, states) + align256((size_t)d.BH() * d.NC * d.C * d.dv * 4));
}

float* states_alpha(const Dims& d, float* states) {
    return (float*)((char*)states_T(d, states) + align256((size_t)d.BH() * d.NC * d.C * d.C * 4));
}

// alpha [BH][NC*C], W [BH][NC*C][dk], U [BH][NC*C][dv], then T, P, dUp, dSc as in bwd_ws_carve
size_t bwd_saved_ws_bytes(const Dims& d) {
    const size_t bh = (size_t)d.BH(), T = (size_t)d.NC * d.C, nc = (size_t)d.NC, C = d.C;
    return align256(bh * T * 4) + align256(bh * T * d.dk * 4) + align256(bh * T * d.dv * 4) +
           2 * align256(bh * nc * C * C * 4) + align256(bh * nc * C * d.dv * 4) +
           align256(bh * nc * (size_t)d.dk * d.dv * 4) + rscan_tc_ws_bytes(d) + grad_tc_ws_bytes(d);
}

BwdWs bwd_saved_ws_carve(const Dims& d, void* base, const float* states) {
    const size_t bh = (size_t)d.BH(), T = (size_t)d.NC * d.C, nc = (size_t)d.NC, C = d.C;
    BwdWs w;
    char* p = (char*)base;
    w.f.alpha = (float*)p; p += align256(bh * T * 4);
    w.f.W = (float*)p;     p += align256(bh * T * d.dk * 4);
    w.f.U = (float*)p;     p += align256(bh * T * d.dv * 4);
    w.f.Sc = const_cast<float*>(states);
    w.f.Up = states_Up(d, const_cast<float*>(states));
    w.f.T = nullptr;
    w.T = (float*)p;   p += align256(bh * nc * C * C * 4);
    w.P = (float*)p;   p += align256(bh * nc * C * C * 4);
    w.dUp = (float*)p; p += align256(bh * nc * C * d.dv * 4);
    w.dSc = (float*)p; p += align256(bh * nc * (size_t)d.dk * d.dv * 4);
    w.tc = rscan_tc_supported(d) ? (void*)p : nullptr;
    return w;
}

BwdWs bwd_ws_carve(const Dims& d, void* base) {
    const size_t bh = (size_t)d.BH(), nc = (size_t)d.NC, C = d.C;
    BwdWs w;
    w.f = fwd_ws_carve(d, base);
    char* p = (char*)base + fwd_ws_bytes(d);
    w.T = (float*)p;   p += align256(bh * nc * C * C * 4);
    w.P = (float*)p;   p += align256(bh * nc * C * C * 4);
    w.dUp = (float*)p; p += align256(bh * nc * C * d.dv * 4);
    w.dSc = (float*)p; p += align256(bh * nc * (size_t)d.dk * d.dv * 4);
    w.tc = rscan_tc_supported(d) ? (void*)p : nullptr;
    return w;
}

// ------------------------------------------------------------- reverse scan
struct RScanArgs {
    const void* q;
    const void* k;
    const void* dO;
    const float* W;
    const float* P;
    const float* dS_final;   // nullable
    float* dUp;
    float* dSc;              // gradient w.r.t. the state leaving each chunk
    float* dS0;              // nullable
    int L, dk, dv, C, NC, BV, in_bf16;
};

static size_t rscan_smem(const Dims& d, int BV) {
    const size_t C = d.C;
    return ((size_t)d.dk * BV + C * (C + 1) + 3 * C * (d.dk + 1) + 2 * C * (BV + 1)) * sizeof(float);
}

__global__ void __launch_bounds__(kNTb) k_rscan(RScanArgs a) {
    extern __shared__ float sm[];
    const long long bh = blockIdx.x;
    const int v0 = blockIdx.y * a.BV;
    const int C = a.C, dk = a.dk, dv = a.dv, BV = a.BV, L = a.L;
    const int ldk = dk + 1, ldc = C + 1, ldb = BV + 1;
    float* dSs = sm;                // [dk][BV]
    float* Ps = dSs + dk * BV;      // [C][ldc]
    float* Ks = Ps + C * ldc;       // [C][ldk]
    float* Qs = Ks + C * ldk;       // [C][ldk]
    float* Ws = Qs + C * ldk;       // [C][ldk]
    float* dOs = Ws + C * ldk;      // [C][ldb]
    float* dUs = dOs + C * ldb;     // [C][ldb]
    const int bf = a.in_bf16;

    for (int idx = threadIdx.x; idx < dk * BV; idx += kNTb) {
        const int r = idx / BV, n = idx - r * BV;
        dSs[idx] = a.dS_final ? a.dS_final[((size_t)bh * dk + r) * dv + v0 + n] : 0.f;
    }
    for (int c = a.NC - 1; c >= 0; --c) {
        const int t0 = c * C;
        const int nvalid = min(C, L - t0);
        const long long tok0 = bh * L + t0;
        const size_t chunk = (size_t)bh * a.NC + c;
        const float* Pg = a.P + chunk * C * C;
        const float* Wg = a.W + chunk * C * dk;
        for (int idx = threadIdx.x; idx < C * C; idx += kNTb) {
            const int i = idx / C, j = idx - i * C;
            Ps[i * ldc + j] = Pg[idx];
        }
        for (int idx = threadIdx.x; idx < C * dk; idx += kNTb) {
            const int i = idx / dk, x = idx - i * dk;
            const bool ok = i < nvalid;
            Ks[i * ldk + x] = ok ? ld_in(a.k, (tok0 + i) * dk + x, bf) : 0.f;
            Qs[i * ldk + x] = ok ? ld_in(a.q, (tok0 + i) * dk + x, bf) : 0.f;
            Ws[i * ldk + x] = Wg[idx];
        }
        for (int idx = threadIdx.x; idx < C * BV; idx += kNTb) {
            const int i = idx / BV, n = idx - i * BV;
            dOs[i * ldb + n] = i < nvalid ? ld_in(a.dO, (tok0 + i) * dv + v0 + n, bf) : 0.f;
        }
        __syncthreads();
        float* dScg = a.dSc + chunk * dk * dv;
        for (int idx = threadIdx.x; idx < dk * BV; idx += kNTb) {
            const int r = idx / BV, n = idx - r * BV;
            dScg[(size_t)r * dv + v0 + n] = dSs[idx];
        }
        // dUp = P^T dO + K dS'
        float* dUg = a.dUp + chunk * C * dv;
        for (int idx = threadIdx.x; idx < C * BV; idx += kNTb) {
            const int i = idx / BV, n = idx - i * BV;
            float s = 0.f;
            for (int j = i; j < C; ++j) s = fmaf(Ps[j * ldc + i], dOs[j * ldb + n], s);
            for (int x = 0; x < dk; ++x) s = fmaf(Ks[i * ldk + x], dSs[x * BV + n], s);
            dUs[i * ldb + n] = s;
            dUg[(size_t)i * dv + v0 + n] = s;
        }
        __syncthreads();
        // dS = dS' + Q^T dO - W^T dUp
        for (int idx = threadIdx.x; idx < dk * BV; idx += kNTb) {
            const int x = idx / BV, n = idx - x * BV;
            float s = 0.f;
            for (int i = 0; i < C; ++i) {
                s = fmaf(Qs[i * ldk + x], dOs[i * ldb + n], s);
                s = fmaf(-Ws[i * ldk + x], dUs[i * ldb + n], s);
            }
            dSs[idx] += s;
        }
        __syncthreads();
    }
    if (a.dS0) {
        for (int idx = threadIdx.x; idx < dk * BV; idx += kNTb) {
            const int r = idx / BV, n = idx - r * BV;
            a.dS0[((size_t)bh * dk + r) * dv + v0 + n] = dSs[idx];
        }
    }
}

// Reverse scan specialised for d_k = 128, C = 64 and a 64-column slice of d_v (the LM
// shapes): one CTA of 512 threads per (sequence, slice).  The state-gradient slice
// dS [128 x 64] stays in registers (a 4 x 4 tile per thread; mirrored in shared memory
// for the dUp product), and every product reads 128-bit vectors, so a thread issues
// one shared-memory load per eight FMAs instead of two per FMA.  Same arithmetic as
// k_rscan, in a different summation order.
constexpr int kRs2Threads = 512;
constexpr int kRs2Q = 132, kRs2K = 68, kRs2N = 68;   // padded row strides (floats)
constexpr size_t kRs2Smem =
    (64 * 64 + 2 * 64 * kRs2Q + 128 * kRs2K + 2 * 64 * kRs2N + 128 * kRs2N) * sizeof(float);

__global__ void __launch_bounds__(kRs2Threads, 1) k_rscan128(RScanArgs a) {
    extern __shared__ float sm[];
    float* Ps = sm;                     // [64 j][64 i]   (zero above the diagonal)
    float* Qs = Ps + 64 * 64;           // [64 i][kRs2Q]
    float* Ws = Qs + 64 * kRs2Q;        // [64 i][kRs2Q]
    float* Kt = Ws + 64 * kRs2Q;        // [128 x][kRs2K]  K transposed
    float* dOs = Kt + 128 * kRs2K;      // [64 i][kRs2N]
    float* dUs = dOs + 64 * kRs2N;      // [64 i][kRs2N]
    float* dSs = dUs + 64 * kRs2N;      // [128 x][kRs2N]
    const int tid = threadIdx.x;
    const long long bh = blockIdx.x;
    const int v0 = blockIdx.y * 64, dv = a.dv, L = a.L, bf = a.in_bf16;
    const int x0 = (tid >> 4) * 4, n0 = (tid & 15) * 4;   // dS tile
    const int i0 = (tid >> 4) * 2;                        // dUp tile (rows i0, i0+1; columns n0..)

    float dS[4][4];
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
        if (a.dS_final) z = *reinterpret_cast<const float4*>(a.dS_final + ((size_t)bh * 128 + x0 + r) * dv + v0 + n0);
        dS[r][0] = z.x; dS[r][1] = z.y; dS[r][2] = z.z; dS[r][3] = z.w;
        *reinterpret_cast<float4*>(dSs + (x0 + r) * kRs2N + n0) = z;
    }
    for (int c = a.NC - 1; c >= 0; --c) {
        const int t0 = c * 64, nvalid = min(64, L - t0);
        const long long tok0 = bh * L + t0;
        const size_t chunk = (size_t)bh * a.NC + c;
        __syncthreads();   // the previous chunk's readers of the staged tiles are done
        {   // P (fp32, [j][i]) and W (fp32, [i][x]) from the workspace
            const float4* Pg = reinterpret_cast<const float4*>(a.P + chunk * 4096);
            for (int e = tid; e < 1024; e += kRs2Threads) reinterpret_cast<float4*>(Ps)[e] = Pg[e];
            const float4* Wg = reinterpret_cast<const float4*>(a.W + chunk * 64 * 128);
            for (int e = tid; e < 2048; e += kRs2Threads) {
                const int i = e >> 5, x = (e & 31) * 4;
                *reinterpret_cast<float4*>(Ws + i * kRs2Q + x) = Wg[e];
            }
        }
        {   // Q rows, K rows transposed, dO slice (bf16 or fp32 inputs); rows past L are zero
            const int i = tid & 63, xg = tid >> 6;   // row i, 16 columns 16 xg .. +15
            const bool ok = i < nvalid;
            float qv[16], kv[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const size_t off = (size_t)(tok0 + i) * 128 + 16 * xg + e;
                qv[e] = ok ? ld_in(a.q, off, bf) : 0.f;
                kv[e] = ok ? ld_in(a.k, off, bf) : 0.f;
            }
#pragma unroll
            for (int e = 0; e < 16; e += 4)
                *reinterpret_cast<float4*>(Qs + i * kRs2Q + 16 * xg + e) = make_float4(qv[e], qv[e + 1], qv[e + 2], qv[e + 3]);
#pragma unroll
            for (int e = 0; e < 16; ++e) Kt[(16 * xg + e) * kRs2K + i] = kv[e];
            const int ng = xg;   // 8 columns 8 ng .. +7 of the dO slice
            float ov[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) ov[e] = ok ? ld_in(a.dO, (size_t)(tok0 + i) * dv + v0 + 8 * ng + e, bf) : 0.f;
            *reinterpret_cast<float4*>(dOs + i * kRs2N + 8 * ng) = make_float4(ov[0], ov[1], ov[2], ov[3]);
            *reinterpret_cast<float4*>(dOs + i * kRs2N + 8 * ng + 4) = make_float4(ov[4], ov[5], ov[6], ov[7]);
        }
        // gradient w.r.t. the state leaving this chunk
        float* dScg = a.dSc + chunk * 128 * dv;
#pragma unroll
        for (int r = 0; r < 4; ++r)
            *reinterpret_cast<float4*>(dScg + (size_t)(x0 + r) * dv + v0 + n0) =
                make_float4(dS[r][0], dS[r][1], dS[r][2], dS[r][3]);
        __syncthreads();
        {   // dUp = P^T dO + K dS  (rows i0, i0+1; columns n0..n0+3)
            float u[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll 8
            for (int j = 0; j < 64; ++j) {
                const float2 p = *reinterpret_cast<const float2*>(Ps + j * 64 + i0);
                const float4 d = *reinterpret_cast<const float4*>(dOs + j * kRs2N + n0);
                u[0][0] = fmaf(p.x, d.x, u[0][0]); u[0][1] = fmaf(p.x, d.y, u[0][1]);
                u[0][2] = fmaf(p.x, d.z, u[0][2]); u[0][3] = fmaf(p.x, d.w, u[0][3]);
                u[1][0] = fmaf(p.y, d.x, u[1][0]); u[1][1] = fmaf(p.y, d.y, u[1][1]);
                u[1][2] = fmaf(p.y, d.z, u[1][2]); u[1][3] = fmaf(p.y, d.w, u[1][3]);
            }
#pragma unroll 8
            for (int x = 0; x < 128; ++x) {
                const float2 k2 = *reinterpret_cast<const float2*>(Kt + x * kRs2K + i0);
                const float4 sv = *reinterpret_cast<const float4*>(dSs + x * kRs2N + n0);
                u[0][0] = fmaf(k2.x, sv.x, u[0][0]); u[0][1] = fmaf(k2.x, sv.y, u[0][1]);
                u[0][2] = fmaf(k2.x, sv.z, u[0][2]); u[0][3] = fmaf(k2.x, sv.w, u[0][3]);
                u[1][0] = fmaf(k2.y, sv.x, u[1][0]); u[1][1] = fmaf(k2.y, sv.y, u[1][1]);
                u[1][2] = fmaf(k2.y, sv.z, u[1][2]); u[1][3] = fmaf(k2.y, sv.w, u[1][3]);
            }
            float* dUg = a.dUp + chunk * 64 * dv;
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                const float4 w4 = make_float4(u[r][0], u[r][1], u[r][2], u[r][3]);
                *reinterpret_cast<float4*>(dUs + (i0 + r) * kRs2N + n0) = w4;
                *reinterpret_cast<float4*>(dUg + (size_t)(i0 + r) * dv + v0 + n0) = w4;
            }
        }
        __syncthreads();
        // dS += Q^T dO - W^T dUp  (rows x0..x0+3, columns n0..n0+3)
#pragma unroll 4
        for (int i = 0; i < 64; ++i) {
            const float4 q4 = *reinterpret_cast<const float4*>(Qs + i * kRs2Q + x0);
            const float4 w4 = *reinterpret_cast<const float4*>(Ws + i * kRs2Q + x0);
            const float4 d4 = *reinterpret_cast<const float4*>(dOs + i * kRs2N + n0);
            const float4 u4 = *reinterpret_cast<const float4*>(dUs + i * kRs2N + n0);
            const float qa[4] = {q4.x, q4.y, q4.z, q4.w}, wa[4] = {w4.x, w4.y, w4.z, w4.w};
            const float da[4] = {d4.x, d4.y, d4.z, d4.w}, ua[4] = {u4.x, u4.y, u4.z, u4.w};
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int n = 0; n < 4; ++n) dS[r][n] = fmaf(qa[r], da[n], fmaf(-wa[r], ua[n], dS[r][n]));
        }
#pragma unroll
        for (int r = 0; r < 4; ++r)
            *reinterpret_cast<float4*>(dSs + (x0 + r) * kRs2N + n0) = make_float4(dS[r][0], dS[r][1], dS[r][2], dS[r][3]);
    }
    if (a.dS0) {
#pragma unroll
        for (int r = 0; r < 4; ++r)
            *reinterpret_cast<float4*>(a.dS0 + ((size_t)bh * 128 + x0 + r) * dv + v0 + n0) =
                make_float4(dS[r][0], dS[r][1], dS[r][2], dS[r][3]);
    }
}

// ------------------------------------------------------- per-chunk gradients
struct GradArgs {
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
    int L, dk_, dv_, C, NC, BV, euler, in_bf16, out_bf16;
};

constexpr int kEPT = 32;   // register-resident [C][dk] elements per thread: 64*128/256

// k_grad128's shared memory: its value-major phase-1 views take 2 BV (d_k + 4) + 4 BV (C + 4)
// floats where k_grad's take 2 d_k (BV + 1) + 4 C (BV + 1).
static size_t grad128_smem(const Dims& d, int BV) {
    const size_t C = d.C, ldc = C + 1, ldk = d.dk + 1;
    const size_t slices = 2 * (size_t)BV * (d.dk + 4) + 4 * (size_t)BV * (C + 4);
    const size_t qk = 2 * C * ldk;
    const size_t ldr = (size_t)(d.dk > BV ? d.dk : BV) + 1;
    return (4 * C * ldc + (slices > qk ? slices : qk) + C * ldk + C * ldr + 4 * C) * sizeof(float);
}

static size_t grad_smem(const Dims& d, int BV) {
    const size_t C = d.C, ldc = C + 1, ldk = d.dk + 1, ldb = BV + 1;
    const size_t slices = 2 * (size_t)d.dk * ldb + 4 * C * ldb;
    const size_t qk = 2 * C * ldk;
    const size_t ldr = (size_t)(d.dk > BV ? d.dk : BV) + 1;   // product scratch row
    return (4 * C * ldc + (slices > qk ? slices : qk) + C * ldk + C * ldr + 4 * C) * sizeof(float);
}

__global__ void __launch_bounds__(kNTb, 1) k_grad(GradArgs a) {
    extern __shared__ float sm[];
    const long long bh = blockIdx.x;
    const int c = blockIdx.y;
    const int C = a.C, dk = a.dk_, dv = a.dv_, BV = a.BV, L = a.L;
    const int ldc = C + 1, ldk = dk + 1, ldb = BV + 1;
    const int t0 = c * C;
    const int nvalid = min(C, L - t0);
    const long long tok0 = bh * L + t0;
    const size_t chunk = (size_t)bh * a.NC + c;
    const int tid = threadIdx.x;

    float* Ts = sm;                 // [C][ldc]
    float* Ds = Ts + C * ldc;       // [C][ldc]  tril(dO Up^T), later dG
    float* dTs = Ds + C * ldc;      // [C][ldc]  dT, later dA
    float* Xs = dTs + C * ldc;      // [C][ldc]  dT T^T, later G
    float* R1 = Xs + C * ldc;       // union: phase-1 slices | phase-2 Q, K
    const size_t slices = 2 * (size_t)dk * ldb + 4 * (size_t)C * ldb;
    const size_t qk = 2 * (size_t)C * ldk;
    float* dWs = R1 + (slices > qk ? slices : qk);   // [C][ldk]
    const int ldr = (dk > BV ? dk : BV) + 1;
    float* PR = dWs + C * ldk;      // [C][ldr]  per-element products for fixed-order row sums
    float* al = PR + C * ldr;       // [C]
    float* dal = al + C;            // [C]
    float* lam = dal + C;           // [C]
    float* bet = lam + C;           // [C]
    // phase-1 views of R1
    float* Scs = R1;                // [dk][ldb]
    float* dScs = Scs + dk * ldb;   // [dk][ldb]
    float* dOs = dScs + dk * ldb;   // [C][ldb]
    float* Ups = dOs + C * ldb;     // [C][ldb]
    float* dUs = Ups + C * ldb;     // [C][ldb]
    float* Vs = dUs + C * ldb;      // [C][ldb]
    // phase-2 views of R1
    float* Qs = R1;                 // [C][ldk]
    float* Ks = Qs + C * ldk;       // [C][ldk]

    const int bf = a.in_bf16, obf = a.out_bf16;

    const float* Tg = a.T + chunk * C * C;
    for (int idx = tid; idx < C * C; idx += kNTb) {
        const int i = idx / C, j = idx - i * C;
        Ts[i * ldc + j] = Tg[idx];
        Ds[i * ldc + j] = 0.f;
        dTs[i * ldc + j] = 0.f;
    }
    for (int i = tid; i < C; i += kNTb) {
        al[i] = a.alpha[chunk * C + i];
        bet[i] = i < nvalid ? a.beta[tok0 + i] : 0.f;
        dal[i] = 0.f;
    }

    float rdQ[kEPT], rdK[kEPT], rdW[kEPT];
#pragma unroll
    for (int m = 0; m < kEPT; ++m) { rdQ[m] = 0.f; rdK[m] = 0.f; rdW[m] = 0.f; }

    const float* Scg = a.Sc + chunk * dk * dv;
    const float* dScg = a.dSc + chunk * dk * dv;
    const float* Upg = a.Up + chunk * C * dv;
    const float* dUg = a.dUp + chunk * C * dv;

    // ---- phase 1: products over the value dimension, one BV-column slice at a time
    for (int v0 = 0; v0 < dv; v0 += BV) {
        __syncthreads();
        for (int idx = tid; idx < dk * BV; idx += kNTb) {
            const int x = idx / BV, n = idx - x * BV;
            Scs[x * ldb + n] = Scg[(size_t)x * dv + v0 + n];
            dScs[x * ldb + n] = dScg[(size_t)x * dv + v0 + n];
        }
        for (int idx = tid; idx < C * BV; idx += kNTb) {
            const int i = idx / BV, n = idx - i * BV;
            const bool ok = i < nvalid;
            dOs[i * ldb + n] = ok ? ld_in(a.dO, (tok0 + i) * dv + v0 + n, bf) : 0.f;
            Vs[i * ldb + n] = ok ? ld_in(a.v, (tok0 + i) * dv + v0 + n, bf) : 0.f;
            Ups[i * ldb + n] = Upg[(size_t)i * dv + v0 + n];
            dUs[i * ldb + n] = dUg[(size_t)i * dv + v0 + n];
        }
        __syncthreads();
        // dQ += dO S^T,  dK += Up G'^T,  dW -= dUp S^T
#pragma unroll
        for (int m = 0; m < kEPT; ++m) {
            const int e = tid + m * kNTb;
            if (e < C * dk) {
                const int i = e / dk, x = e - i * dk;
                float sq = 0.f, sk = 0.f, sw = 0.f;
                for (int n = 0; n < BV; ++n) {
                    const float s = Scs[x * ldb + n];
                    sq = fmaf(dOs[i * ldb + n], s, sq);
                    sk = fmaf(Ups[i * ldb + n], dScs[x * ldb + n], sk);
                    sw = fmaf(dUs[i * ldb + n], s, sw);
                }
                rdQ[m] += sq;
                rdK[m] += sk;
                rdW[m] -= sw;
            }
        }
        // D += tril(dO Up^T);  dT += dUp (alpha V)^T
        for (int idx = tid; idx < C * C; idx += kNTb) {
            const int i = idx / C, j = idx - i * C;
            float sd = 0.f, st = 0.f;
            for (int n = 0; n < BV; ++n) {
                const float g = dUs[i * ldb + n];
                if (j <= i) sd = fmaf(dOs[i * ldb + n], Ups[j * ldb + n], sd);
                st = fmaf(g, Vs[j * ldb + n], st);
            }
            Ds[i * ldc + j] += sd;
            dTs[i * ldc + j] += al[j] * st;
        }
        // dVa = T^T dUp;  dV = alpha dVa;  dalpha += <dVa, v> (row sums in a fixed order)
        for (int idx = tid; idx < C * BV; idx += kNTb) {
            const int j = idx / BV, n = idx - j * BV;
            float s = 0.f;
            for (int i = j; i < C; ++i) s = fmaf(Ts[i * ldc + j], dUs[i * ldb + n], s);
            if (j < nvalid) st_out(a.dv, (tok0 + j) * dv + v0 + n, al[j] * s, obf);
            PR[j * ldr + n] = s * Vs[j * ldb + n];
        }
        __syncthreads();
        for (int j = tid; j < C; j += kNTb) {
            float s = 0.f;
            for (int n = 0; n < BV; ++n) s += PR[j * ldr + n];
            dal[j] += s;
        }
    }
    __syncthreads();

    // ---- phase 2: Q and K in R1, dW in smem
    for (int idx = tid; idx < C * dk; idx += kNTb) {
        const int i = idx / dk, x = idx - i * dk;
        const bool ok = i < nvalid;
        Qs[i * ldk + x] = ok ? ld_in(a.q, (tok0 + i) * dk + x, bf) : 0.f;
        Ks[i * ldk + x] = ok ? ld_in(a.k, (tok0 + i) * dk + x, bf) : 0.f;
    }
#pragma unroll
    for (int m = 0; m < kEPT; ++m) {
        const int e = tid + m * kNTb;
        if (e < C * dk) {
            const int i = e / dk, x = e - i * dk;
            dWs[i * ldk + x] = rdW[m];
        }
    }
    __syncthreads();
    // lambda_i = ||k_i||^2 (one warp per row)
    {
        const int warp = tid >> 5, lane = tid & 31;
        for (int i = warp; i < C; i += kNTb / 32) {
            float s = 0.f;
            for (int x = lane; x < dk; x += 32) s = fmaf(Ks[i * ldk + x], Ks[i * ldk + x], s);
            s = warp_sum(s);
            if (lane == 0) lam[i] = s;
        }
    }
    // dQ += D K;  dK += D^T Q;  dKa = T^T dW -> dK += alpha dKa, dalpha += <dKa, k>
#pragma unroll
    for (int m = 0; m < kEPT; ++m) {
        const int e = tid + m * kNTb;
        if (e < C * dk) {
            const int i = e / dk, x = e - i * dk;
            float sq = 0.f, sk = 0.f, ska = 0.f;
            for (int j = 0; j <= i; ++j) sq = fmaf(Ds[i * ldc + j], Ks[j * ldk + x], sq);
            for (int j = i; j < C; ++j) {
                sk = fmaf(Ds[j * ldc + i], Qs[j * ldk + x], sk);
                ska = fmaf(Ts[j * ldc + i], dWs[j * ldk + x], ska);
            }
            rdQ[m] += sq;
            rdK[m] += sk + al[i] * ska;
            PR[i * ldr + x] = ska * Ks[i * ldk + x];
        }
    }
    // dT += dW (alpha K)^T
    for (int idx = tid; idx < C * C; idx += kNTb) {
        const int i = idx / C, j = idx - i * C;
        float s = 0.f;
        for (int x = 0; x < dk; ++x) s = fmaf(dWs[i * ldk + x], Ks[j * ldk + x], s);
        dTs[i * ldc + j] += al[j] * s;
    }
    __syncthreads();
    // dalpha_i += <dKa_i, k_i>  (fixed-order row sums)
    for (int i = tid; i < C; i += kNTb) {
        float s = 0.f;
        for (int x = 0; x < dk; ++x) s += PR[i * ldr + x];
        dal[i] += s;
    }
    // X = dT T^T   (T[j][l] = 0 for l > j)
    for (int idx = tid; idx < C * C; idx += kNTb) {
        const int i = idx / C, j = idx - i * C;
        float s = 0.f;
        for (int l = 0; l <= j; ++l) s = fmaf(dTs[i * ldc + l], Ts[j * ldc + l], s);
        Xs[i * ldc + j] = s;
    }
    __syncthreads();
    // dA = strict_lower(-T^T X), written over dT
    for (int idx = tid; idx < C * C; idx += kNTb) {
        const int i = idx / C, j = idx - i * C;
        float s = 0.f;
        if (j < i)
            for (int l = i; l < C; ++l) s = fmaf(Ts[l * ldc + i], Xs[l * ldc + j], s);
        dTs[i * ldc + j] = -s;
    }
    __syncthreads();
    // G = K K^T (strictly lower part) over X;  dG = diag(alpha) dA over D
    for (int idx = tid; idx < C * C; idx += kNTb) {
        const int i = idx / C, j = idx - i * C;
        float g = 0.f;
        if (j < i)
            for (int x = 0; x < dk; ++x) g = fmaf(Ks[i * ldk + x], Ks[j * ldk + x], g);
        Xs[i * ldc + j] = g;
        Ds[i * ldc + j] = (j < i) ? al[i] * dTs[i * ldc + j] : 0.f;
    }
    __syncthreads();
    // dalpha_i += sum_{j<i} dA_ij G_ij
    {
        const int warp = tid >> 5, lane = tid & 31;
        for (int i = warp; i < C; i += kNTb / 32) {
            float s = 0.f;
            for (int j = lane; j < i; j += 32) s = fmaf(dTs[i * ldc + j], Xs[i * ldc + j], s);
            s = warp_sum(s);
            if (lane == 0) dal[i] += s;
        }
    }
    __syncthreads();
    // dK += (dG + dG^T) K + 2 dlambda K;  dbeta
#pragma unroll
    for (int m = 0; m < kEPT; ++m) {
        const int e = tid + m * kNTb;
        if (e < C * dk) {
            const int i = e / dk, x = e - i * dk;
            float s = 0.f;
            for (int j = 0; j < i; ++j) s = fmaf(Ds[i * ldc + j], Ks[j * ldk + x], s);
            for (int j = i + 1; j < C; ++j) s = fmaf(Ds[j * ldc + i], Ks[j * ldk + x], s);
            const float dl = dal[i] * dalpha_dlambda_of(bet[i], lam[i], a.euler);
            s = fmaf(2.f * dl, Ks[i * ldk + x], s);
            if (i < nvalid) {
                st_out(a.dq, (tok0 + i) * dk + x, rdQ[m], obf);
                st_out(a.dk, (tok0 + i) * dk + x, rdK[m] + s, obf);
            }
        }
    }
    for (int i = tid; i < nvalid; i += kNTb)
        a.dbeta[tok0 + i] = dal[i] * dalpha_dbeta_of(bet[i], lam[i], a.euler);
}

__global__ void __launch_bounds__(kNTb, 1) k_grad128(GradArgs a) {
    extern __shared__ float sm[];
    const long long bh = blockIdx.x;
    const int c = blockIdx.y;
    const int C = a.C, dk = a.dk_, dv = a.dv_, BV = a.BV, L = a.L;
    const int ldc = C + 1, ldk = dk + 1;
    const int t0 = c * C;
    const int nvalid = min(C, L - t0);
    const long long tok0 = bh * L + t0;
    const size_t chunk = (size_t)bh * a.NC + c;
    const int tid = threadIdx.x;
    const int xc = tid & 127, ih = 32 * (tid >> 7);   // this thread: column xc of rows ih .. ih+31

    float* Ts = sm;                 // [C][ldc]
    float* Ds = Ts + C * ldc;       // [C][ldc]  tril(dO Up^T), later dG
    float* dTs = Ds + C * ldc;      // [C][ldc]  dT, later dA
    float* Xs = dTs + C * ldc;      // [C][ldc]  dT T^T, later G
    float* R1 = Xs + C * ldc;       // union: phase-1 slices | phase-2 Q, K
    const size_t slices = 2 * (size_t)BV * (128 + 4) + 4 * (size_t)BV * (64 + 4);   // value-major views
    const size_t qk = 2 * (size_t)C * ldk;
    float* dWs = R1 + (slices > qk ? slices : qk);   // [C][ldk]
    const int ldr = (dk > BV ? dk : BV) + 1;
    float* PR = dWs + C * ldk;      // [C][ldr]  per-element products for fixed-order row sums
    float* al = PR + C * ldr;       // [C]
    float* dal = al + C;            // [C]
    float* lam = dal + C;           // [C]
    float* bet = lam + C;           // [C]
    // phase-1 views of R1, value-index major: [n][x] and [n][i] (rows of 16-byte multiples)
    constexpr int ldx = 128 + 4, ldi = 64 + 4;
    float* Scs = R1;                // [BV][ldx]  S^T
    float* dScs = Scs + BV * ldx;   // [BV][ldx]  dS'^T
    float* dOs = dScs + BV * ldx;   // [BV][ldi]  dO^T
    float* Ups = dOs + BV * ldi;    // [BV][ldi]  Up^T
    float* dUs = Ups + BV * ldi;    // [BV][ldi]  dUp^T
    float* Vs = dUs + BV * ldi;     // [BV][ldi]  V^T
    // phase-2 views of R1
    float* Qs = R1;                 // [C][ldk]
    float* Ks = Qs + C * ldk;       // [C][ldk]

    const int bf = a.in_bf16, obf = a.out_bf16;

    const float* Tg = a.T + chunk * C * C;
    for (int idx = tid; idx < C * C; idx += kNTb) {
        const int i = idx / C, j = idx - i * C;
        Ts[i * ldc + j] = Tg[idx];
        Ds[i * ldc + j] = 0.f;
        dTs[i * ldc + j] = 0.f;
    }
    for (int i = tid; i < C; i += kNTb) {
        al[i] = a.alpha[chunk * C + i];
        bet[i] = i < nvalid ? a.beta[tok0 + i] : 0.f;
        dal[i] = 0.f;
    }

    float rdQ[kEPT], rdK[kEPT], rdW[kEPT];
#pragma unroll
    for (int m = 0; m < kEPT; ++m) { rdQ[m] = 0.f; rdK[m] = 0.f; rdW[m] = 0.f; }

    const float* Scg = a.Sc + chunk * dk * dv;
    const float* dScg = a.dSc + chunk * dk * dv;
    const float* Upg = a.Up + chunk * C * dv;
    const float* dUg = a.dUp + chunk * C * dv;

    // ---- phase 1: products over the value dimension, one BV-column slice at a time
    for (int v0 = 0; v0 < dv; v0 += BV) {
        __syncthreads();
        for (int idx = tid; idx < dk * BV; idx += kNTb) {
            const int x = idx / BV, n = idx - x * BV;
            Scs[n * ldx + x] = Scg[(size_t)x * dv + v0 + n];
            dScs[n * ldx + x] = dScg[(size_t)x * dv + v0 + n];
        }
        for (int idx = tid; idx < C * BV; idx += kNTb) {
            const int i = idx / BV, n = idx - i * BV;
            const bool ok = i < nvalid;
            dOs[n * ldi + i] = ok ? ld_in(a.dO, (tok0 + i) * dv + v0 + n, bf) : 0.f;
            Vs[n * ldi + i] = ok ? ld_in(a.v, (tok0 + i) * dv + v0 + n, bf) : 0.f;
            Ups[n * ldi + i] = Upg[(size_t)i * dv + v0 + n];
            dUs[n * ldi + i] = dUg[(size_t)i * dv + v0 + n];
        }
        __syncthreads();
        // dQ += dO S^T,  dK += Up G'^T,  dW -= dUp S^T: per value index n, one S / dS' scalar
        // for this thread's column and the 32 rows' dO / Up / dUp as 128-bit (warp-wide
        // broadcast) loads
        for (int n = 0; n < BV; ++n) {
            const float sx = Scs[n * ldx + xc], dsx = dScs[n * ldx + xc];
#pragma unroll
            for (int m = 0; m < kEPT; m += 4) {
                const float4 o4 = *reinterpret_cast<const float4*>(dOs + n * ldi + ih + m);
                const float4 u4 = *reinterpret_cast<const float4*>(Ups + n * ldi + ih + m);
                const float4 g4 = *reinterpret_cast<const float4*>(dUs + n * ldi + ih + m);
                rdQ[m] = fmaf(o4.x, sx, rdQ[m]); rdQ[m + 1] = fmaf(o4.y, sx, rdQ[m + 1]);
                rdQ[m + 2] = fmaf(o4.z, sx, rdQ[m + 2]); rdQ[m + 3] = fmaf(o4.w, sx, rdQ[m + 3]);
                rdK[m] = fmaf(u4.x, dsx, rdK[m]); rdK[m + 1] = fmaf(u4.y, dsx, rdK[m + 1]);
                rdK[m + 2] = fmaf(u4.z, dsx, rdK[m + 2]); rdK[m + 3] = fmaf(u4.w, dsx, rdK[m + 3]);
                rdW[m] = fmaf(-g4.x, sx, rdW[m]); rdW[m + 1] = fmaf(-g4.y, sx, rdW[m + 1]);
                rdW[m + 2] = fmaf(-g4.z, sx, rdW[m + 2]); rdW[m + 3] = fmaf(-g4.w, sx, rdW[m + 3]);
            }
        }
        // D += tril(dO Up^T);  dT += dUp (alpha V)^T
        for (int idx = tid; idx < C * C; idx += kNTb) {
            const int i = idx / C, j = idx - i * C;
            float sd = 0.f, st = 0.f;
            for (int n = 0; n < BV; ++n) {
                const float g = dUs[n * ldi + i];
                if (j <= i) sd = fmaf(dOs[n * ldi + i], Ups[n * ldi + j], sd);
                st = fmaf(g, Vs[n * ldi + j], st);
            }
            Ds[i * ldc + j] += sd;
            dTs[i * ldc + j] += al[j] * st;
        }
        // dVa = T^T dUp;  dV = alpha dVa;  dalpha += <dVa, v> (row sums in a fixed order)
        for (int idx = tid; idx < C * BV; idx += kNTb) {
            const int n = idx / C, j = idx - n * C;
            float s = 0.f;
            for (int i = j; i < C; ++i) s = fmaf(Ts[i * ldc + j], dUs[n * ldi + i], s);
            if (j < nvalid) st_out(a.dv, (tok0 + j) * dv + v0 + n, al[j] * s, obf);
            PR[j * ldr + n] = s * Vs[n * ldi + j];
        }
        __syncthreads();
        for (int j = tid; j < C; j += kNTb) {
            float s = 0.f;
            for (int n = 0; n < BV; ++n) s += PR[j * ldr + n];
            dal[j] += s;
        }
    }
    __syncthreads();

    // ---- phase 2: Q and K in R1, dW in smem
    for (int idx = tid; idx < C * dk; idx += kNTb) {
        const int i = idx / dk, x = idx - i * dk;
        const bool ok = i < nvalid;
        Qs[i * ldk + x] = ok ? ld_in(a.q, (tok0 + i) * dk + x, bf) : 0.f;
        Ks[i * ldk + x] = ok ? ld_in(a.k, (tok0 + i) * dk + x, bf) : 0.f;
    }
#pragma unroll
    for (int m = 0; m < kEPT; ++m) {
        {
            const int i = ih + m, x = xc;
            dWs[i * ldk + x] = rdW[m];
        }
    }
    __syncthreads();
    // lambda_i = ||k_i||^2 (one warp per row)
    {
        const int warp = tid >> 5, lane = tid & 31;
        for (int i = warp; i < C; i += kNTb / 32) {
            float s = 0.f;
            for (int x = lane; x < dk; x += 32) s = fmaf(Ks[i * ldk + x], Ks[i * ldk + x], s);
            s = warp_sum(s);
            if (lane == 0) lam[i] = s;
        }
    }
    // dQ += D K;  dK += D^T Q;  dKa = T^T dW -> dK += alpha dKa, dalpha += <dKa, k>.
    // Loop over j outside: one K / Q / dW value of this thread's column per j, and rows
    // ih..ih+31 of D (D^T), T (T^T) for all 32 of its rows at once (D, T are zero outside
    // their triangles, so the full range is exact).
    {
        float ska[kEPT];
#pragma unroll
        for (int m = 0; m < kEPT; ++m) ska[m] = 0.f;
        for (int j = 0; j < C; ++j) {
            const float kx = Ks[j * ldk + xc], qx = Qs[j * ldk + xc], wx = dWs[j * ldk + xc];
#pragma unroll
            for (int m = 0; m < kEPT; ++m) {
                const int i = ih + m;
                rdQ[m] = fmaf(Ds[i * ldc + j], kx, rdQ[m]);     // D[i][j], j <= i
                rdK[m] = fmaf(Ds[j * ldc + i], qx, rdK[m]);     // D[j][i], j >= i
                ska[m] = fmaf(Ts[j * ldc + i], wx, ska[m]);     // T[j][i], j >= i
            }
        }
#pragma unroll
        for (int m = 0; m < kEPT; ++m) {
            const int i = ih + m;
            rdK[m] = fmaf(al[i], ska[m], rdK[m]);
            PR[i * ldr + xc] = ska[m] * Ks[i * ldk + xc];
        }
    }
    // dT += dW (alpha K)^T
    for (int idx = tid; idx < C * C; idx += kNTb) {
        const int i = idx / C, j = idx - i * C;
        float s = 0.f;
        for (int x = 0; x < dk; ++x) s = fmaf(dWs[i * ldk + x], Ks[j * ldk + x], s);
        dTs[i * ldc + j] += al[j] * s;
    }
    __syncthreads();
    // dalpha_i += <dKa_i, k_i>  (fixed-order row sums)
    for (int i = tid; i < C; i += kNTb) {
        float s = 0.f;
        for (int x = 0; x < dk; ++x) s += PR[i * ldr + x];
        dal[i] += s;
    }
    // X = dT T^T   (T[j][l] = 0 for l > j)
    for (int idx = tid; idx < C * C; idx += kNTb) {
        const int i = idx / C, j = idx - i * C;
        float s = 0.f;
        for (int l = 0; l <= j; ++l) s = fmaf(dTs[i * ldc + l], Ts[j * ldc + l], s);
        Xs[i * ldc + j] = s;
    }
    __syncthreads();
    // dA = strict_lower(-T^T X), written over dT
    for (int idx = tid; idx < C * C; idx += kNTb) {
        const int i = idx / C, j = idx - i * C;
        float s = 0.f;
        if (j < i)
            for (int l = i; l < C; ++l) s = fmaf(Ts[l * ldc + i], Xs[l * ldc + j], s);
        dTs[i * ldc + j] = -s;
    }
    __syncthreads();
    // G = K K^T (strictly lower part) over X;  dG = diag(alpha) dA over D
    for (int idx = tid; idx < C * C; idx += kNTb) {
        const int i = idx / C, j = idx - i * C;
        float g = 0.f;
        if (j < i)
            for (int x = 0; x < dk; ++x) g = fmaf(Ks[i * ldk + x], Ks[j * ldk + x], g);
        Xs[i * ldc + j] = g;
        Ds[i * ldc + j] = (j < i) ? al[i] * dTs[i * ldc + j] : 0.f;
    }
    __syncthreads();
    // dalpha_i += sum_{j<i} dA_ij G_ij
    {
        const int warp = tid >> 5, lane = tid & 31;
        for (int i = warp; i < C; i += kNTb / 32) {
            float s = 0.f;
            for (int j = lane; j < i; j += 32) s = fmaf(dTs[i * ldc + j], Xs[i * ldc + j], s);
            s = warp_sum(s);
            if (lane == 0) dal[i] += s;
        }
    }
    __syncthreads();
    // dK += (dG + dG^T) K + 2 dlambda K;  dbeta.  dG is strictly lower, so (dG + dG^T)[i][j]
    // = dG[i][j] + dG[j][i] over the full range; j outside, as above.
    float sg[kEPT];
#pragma unroll
    for (int m = 0; m < kEPT; ++m) sg[m] = 0.f;
    for (int j = 0; j < C; ++j) {
        const float kx = Ks[j * ldk + xc];
#pragma unroll
        for (int m = 0; m < kEPT; ++m) {
            const int i = ih + m;
            sg[m] = fmaf(Ds[i * ldc + j] + Ds[j * ldc + i], kx, sg[m]);
        }
    }
#pragma unroll
    for (int m = 0; m < kEPT; ++m) {
        {
            const int i = ih + m, x = xc;
            float s = sg[m];
            const float dl = dal[i] * dalpha_dlambda_of(bet[i], lam[i], a.euler);
            s = fmaf(2.f * dl, Ks[i * ldk + x], s);
            if (i < nvalid) {
                st_out(a.dq, (tok0 + i) * dk + x, rdQ[m], obf);
                st_out(a.dk, (tok0 + i) * dk + x, rdK[m] + s, obf);
            }
        }
    }
    for (int i = tid; i < nvalid; i += kNTb)
        a.dbeta[tok0 + i] = dal[i] * dalpha_dbeta_of(bet[i], lam[i], a.euler);
}


// ------------------------------------------------------------------- launch
bool bwd_runs_recording_forward(const Dims& d) {
    return grad_mma_supported(d) && rscan_tc_supported(d) && fwd_tc_supported(d) && fwd_tc_segments(d) == 1;
}

// A second stream of this thread on the current device, for work that may run beside the
// caller's stream: forked from it and joined back with events, so that the caller still
// sees one stream (and a graph captured on it gets two branches).  Created on first use,
// never while the caller's stream is capturing; kept for the life of the thread.  Null when
// unavailable: the caller then runs everything on its own stream.
namespace {
struct SideStream {
    cudaStream_t s = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};
thread_local SideStream t_side[16];

SideStream* side_stream(cudaStream_t st) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 16) return nullptr;
    SideStream& ss = t_side[dev];
    if (!ss.s) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(st, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) return nullptr;
        if (cudaStreamCreateWithFlags(&ss.s, cudaStreamNonBlocking) != cudaSuccess) {
            ss.s = nullptr;
            return nullptr;
        }
        if (cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming) != cudaSuccess ||
            cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming) != cudaSuccess) {
            cudaStreamDestroy(ss.s);
            ss.s = nullptr;
            return nullptr;
        }
    }
    return &ss;
}
}  // namespace

cudaError_t launch_bwd_simt(const Dims& d, const void* q, const void* k, const void* v,
                            const float* beta, const float* S0, const void* dO,
                            const float* dS_final, void* dq, void* dk, void* dv, float* dbeta,
                            float* dS0, const BwdWs& ws_in, cudaStream_t st, bool have_states) {
    BwdWs ws = ws_in;
    cudaError_t e;
    // From a record on the tensor-core shapes nothing needs the preparation kernel: the
    // gradients read the record's T and alpha, the tcgen05 reverse scan prepares its own
    // images, and the preparation runs only for the sequences that scan marks (below).
    const bool rec_tc = have_states && grad_mma_supported(d) && ws.tc;
    // Without a record, on those shapes, the tcgen05 forward records S_c, U', T and alpha
    // into this workspace (outputs not written) in place of the preparation and the state
    // scan; its images go where the reverse scan's will (not yet used).  Few long sequences
    // (the forward's segment-parallel form) keep the preparation and the scan.
    const bool fwd_rec = !have_states && ws.tc && bwd_runs_recording_forward(d);
    if (rec_tc) {
        ws.f.alpha = states_alpha(d, ws.f.Sc);
        ws.T = states_T(d, ws.f.Sc);
    } else if (fwd_rec) {
        // The chunk preparation once, on every SM (images, norms, and T and alpha for the
        // gradients); then the recording forward (S_c and U' as fp16 images, fp32 for a
        // sequence recomputed in fp32) and the tcgen05 reverse scan side by side: the scan
        // needs none of the forward's results, and each takes one SM per sequence.
        e = launch_tc_prep(d, q, k, beta, ws.tc, ws.T, ws.f.alpha, st);
        if (e != cudaSuccess) return e;
        SideStream* side = side_stream(st);
        cudaStream_t st2 = side ? side->s : st;
        if (side) {
            if ((e = cudaEventRecord(side->fork, st)) != cudaSuccess) return e;
            if ((e = cudaStreamWaitEvent(st2, side->fork, 0)) != cudaSuccess) return e;
        }
        e = launch_fwd_tc(d, q, k, v, beta, S0, nullptr, nullptr, ws.tc, st, ws.f.Sc, ws.f.Up, ws.T, ws.f.alpha,
                          grad_tc_list(d, (char*)ws.tc + rscan_tc_ws_bytes(d)).fwd_fp32, true);
        if (e != cudaSuccess) return e;
        e = launch_rscan_tc(d, q, k, dO, beta, dS_final, dS0, ws.tc, st2, true);
        if (e != cudaSuccess) return e;
        if (side) {
            if ((e = cudaEventRecord(side->join, st2)) != cudaSuccess) return e;
            if ((e = cudaStreamWaitEvent(st, side->join, 0)) != cudaSuccess) return e;
        }
        prof_mark("efla_tc_fwd_rec+state_grad_scan_tc", st);
    } else {
        e = launch_prep_for_bwd(d, q, k, v, beta, ws, st);
        if (e != cudaSuccess) return e;
    }
    if (!have_states && !fwd_rec) {
        e = launch_scan_for_bwd(d, k, S0, ws, st);
        if (e != cudaSuccess) return e;
    }
    int BV = 32;
    while (BV > 16 && d.dv % BV) BV >>= 1;
    if (BV > d.dv) BV = d.dv;
    RScanArgs ra{q, k, dO, ws.f.W, ws.P, dS_final, ws.dUp, ws.dSc, dS0,
                 d.L, d.dk, d.dv, d.C, d.NC, BV, d.in_bf16};
    size_t sm = 0;
    if (grad_mma_supported(d) && ws.tc) {
        // tcgen05 reverse scan; the tf32 one recomputes the sequences it marked out of range
        if (!fwd_rec) {   // (with the recording forward it has run already, beside it)
            e = launch_rscan_tc(d, q, k, dO, beta, dS_final, dS0, ws.tc, st);
            if (e != cudaSuccess) return e;
        }
        const RsTcOut rs = rscan_tc_outputs(d, ws.tc);
        int* bad = rs.seq_bad;
        if (rec_tc || fwd_rec) {   // W and P of the marked sequences (into the workspace)
            BwdWs wp = ws_in;
            e = launch_prep_mma(d, q, k, v, beta, wp, st, rs.bad_list, rs.bad_n);
            prof_mark("efla_chunk_prep", st);
            if (e != cudaSuccess) return e;
        }
        e = launch_rscan_mma(d, q, k, dO, dS_final, dS0, ws_in, st, bad);
        if (e != cudaSuccess) return e;
    } else if (grad_mma_supported(d)) {
        e = launch_rscan_mma(d, q, k, dO, dS_final, dS0, ws, st);
        if (e != cudaSuccess) return e;
    } else if (d.dk == 128 && d.C == 64 && d.dv % 64 == 0) {   // register-tiled reverse scan
        e = cudaFuncSetAttribute(k_rscan128, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kRs2Smem);
        if (e != cudaSuccess) return e;
        k_rscan128<<<dim3((unsigned)d.BH(), d.dv / 64), kRs2Threads, kRs2Smem, st>>>(ra);
    } else {
        sm = rscan_smem(d, BV);
        e = cudaFuncSetAttribute(k_rscan, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
        if (e != cudaSuccess) return e;
        k_rscan<<<dim3((unsigned)d.BH(), d.dv / BV), kNTb, sm, st>>>(ra);
    }
    prof_mark("efla_state_grad_scan", st);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (grad_tc_supported(d) && ws.tc) {
        // tcgen05 gradients; the tf32 kernel recomputes the chunks they marked
        const GtList redo = grad_tc_list(d, (char*)ws.tc + rscan_tc_ws_bytes(d));
        const RsTcOut rs = rscan_tc_outputs(d, ws.tc);
        const int* fwd_fp32 = fwd_rec ? redo.fwd_fp32 : nullptr;
        e = launch_grad_tc(d, q, k, v, dO, beta, ws.f.alpha, ws.T, ws.f.Sc, ws.dSc, ws.f.Up, ws.dUp, rs, fwd_fp32,
                           dq, dk, dv, dbeta, redo, st);
        if (e != cudaSuccess) return e;
        e = launch_widen(d, rs, redo, fwd_fp32, ws.f.Sc, ws.f.Up, ws.dSc, ws.dUp, st);
        if (e != cudaSuccess) return e;
        e = launch_grad_mma(d, q, k, v, dO, beta, ws, dq, dk, dv, dbeta, st, redo.chunks, redo.n);
        prof_mark("efla_chunk_grad", st);
        return e;
    }
    if (grad_mma_supported(d)) {
        e = launch_grad_mma(d, q, k, v, dO, beta, ws, dq, dk, dv, dbeta, st);
        prof_mark("efla_chunk_grad", st);
        return e;
    }
    GradArgs ga{q, k, v, dO, beta, ws.f.alpha, ws.T, ws.f.Sc, ws.dSc, ws.f.Up, ws.dUp,
                dq, dk, dv, dbeta, d.L, d.dk, d.dv, d.C, d.NC, BV, d.euler, d.in_bf16, d.out_bf16};
    const bool tiled = d.dk == 128 && d.C == 64 && BV == 32;
    sm = tiled ? grad128_smem(d, BV) : grad_smem(d, BV);
    e = cudaFuncSetAttribute(tiled ? k_grad128 : k_grad, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return e;
    if (tiled)
        k_grad128<<<dim3((unsigned)d.BH(), d.NC), kNTb, sm, st>>>(ga);
    else
        k_grad<<<dim3((unsigned)d.BH(), d.NC), kNTb, sm, st>>>(ga);
    prof_mark("efla_chunk_grad", st);
    return cudaGetLastError();
}

}  // namespace efla

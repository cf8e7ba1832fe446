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
           align256(bh * nc * (size_t)d.dk * d.dv * 4);
}

BwdWs bwd_ws_carve(const Dims& d, void* base) {
    const size_t bh = (size_t)d.BH(), nc = (size_t)d.NC, C = d.C;
    BwdWs w;
    w.f = fwd_ws_carve(d, base);
    char* p = (char*)base + fwd_ws_bytes(d);
    w.T = (float*)p;   p += align256(bh * nc * C * C * 4);
    w.P = (float*)p;   p += align256(bh * nc * C * C * 4);
    w.dUp = (float*)p; p += align256(bh * nc * C * d.dv * 4);
    w.dSc = (float*)p;
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

// ------------------------------------------------------------------- launch
cudaError_t launch_bwd_simt(const Dims& d, const void* q, const void* k, const void* v,
                            const float* beta, const float* S0, const void* dO,
                            const float* dS_final, void* dq, void* dk, void* dv, float* dbeta,
                            float* dS0, const BwdWs& ws, cudaStream_t st) {
    cudaError_t e = launch_prep_for_bwd(d, q, k, v, beta, ws, st);
    if (e != cudaSuccess) return e;
    e = launch_scan_for_bwd(d, k, S0, ws, st);
    if (e != cudaSuccess) return e;
    int BV = 32;
    while (BV > 16 && d.dv % BV) BV >>= 1;
    if (BV > d.dv) BV = d.dv;
    RScanArgs ra{q, k, dO, ws.f.W, ws.P, dS_final, ws.dUp, ws.dSc, dS0,
                 d.L, d.dk, d.dv, d.C, d.NC, BV, d.in_bf16};
    size_t sm = rscan_smem(d, BV);
    e = cudaFuncSetAttribute(k_rscan, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return e;
    k_rscan<<<dim3((unsigned)d.BH(), d.dv / BV), kNTb, sm, st>>>(ra);
    prof_mark("efla_state_grad_scan", st);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    GradArgs ga{q, k, v, dO, beta, ws.f.alpha, ws.T, ws.f.Sc, ws.dSc, ws.f.Up, ws.dUp,
                dq, dk, dv, dbeta, d.L, d.dk, d.dv, d.C, d.NC, BV, d.euler, d.in_bf16, d.out_bf16};
    sm = grad_smem(d, BV);
    e = cudaFuncSetAttribute(k_grad, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return e;
    k_grad<<<dim3((unsigned)d.BH(), d.NC), kNTb, sm, st>>>(ga);
    prof_mark("efla_chunk_grad", st);
    return cudaGetLastError();
}

}  // namespace efla

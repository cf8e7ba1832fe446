// fwd_simt.cu -- chunkwise WY/UT forward pass of EFLA on CUDA cores (fp32 arithmetic).
//
// Per chunk of C tokens with keys K [C,dk], values V [C,dv], queries Q [C,dk] and
// alpha [C] (page es, Metodologia item 3: update rule and alpha, evaluated with the
// WY/UT chunkwise scheme the same item names):
//   A   = strict_lower(diag(alpha) K K^T)
//   T   = (I + A)^{-1}                          (unit lower triangular)
//   W   = T diag(alpha) K,   U = T diag(alpha) V
//   Up  = U - W S_c                             (S_c: state entering the chunk)
//   S_{c+1} = S_c + K^T Up
//   O   = Q S_c + tril(Q K^T) Up                (tril keeps the diagonal: o_t reads S_t)
// This is the token recurrence S_t = S_{t-1} + alpha_t k_t (v_t - S_{t-1}^T k_t)^T
// unrolled over the chunk: row t of Up is alpha_t (v_t - S_{t-1}^T k_t).
//
// Three kernels: k_prep (chunk-parallel: alpha, T, W, U), k_scan (sequential over
// chunks, parallel over sequences x value-column slices: Up, S) and k_out
// (chunk-parallel: O).  Tokens past L inside the last chunk are zero rows
// (k = v = q = 0, beta = 0), which leave the state untouched.
#include "common.cuh"
#include "launch.h"

namespace efla {

constexpr int kNT = 256;

// ---------------------------------------------------------------- workspace
size_t fwd_ws_bytes(const Dims& d) {
    const size_t bh = (size_t)d.BH(), T = (size_t)d.NC * d.C;
    return align256(bh * T * 4) + align256(bh * T * d.dk * 4) + 2 * align256(bh * T * d.dv * 4) +
           align256(bh * d.NC * (size_t)d.dk * d.dv * 4);
}

FwdWs fwd_ws_carve(const Dims& d, void* base) {
    const size_t bh = (size_t)d.BH(), T = (size_t)d.NC * d.C;
    char* p = (char*)base;
    FwdWs w;
    w.alpha = (float*)p; p += align256(bh * T * 4);
    w.W = (float*)p;     p += align256(bh * T * d.dk * 4);
    w.U = (float*)p;     p += align256(bh * T * d.dv * 4);
    w.Up = (float*)p;    p += align256(bh * T * d.dv * 4);
    w.Sc = (float*)p;
    w.T = nullptr;
    return w;
}

// --------------------------------------------------------------- k_prep
struct PrepArgs {
    const void* q;       // only read when P != nullptr
    const void* k;
    const void* v;
    const float* beta;
    float* alpha;        // [BH][NC*C]
    float* W;            // [BH][NC][C][dk]
    float* U;            // [BH][NC][C][dv]
    float* T;            // [BH][NC][C][C] or nullptr
    float* P;            // [BH][NC][C][C] or nullptr (tril(Q K^T), diagonal included)
    int L, dk, dv, C, NC, euler;
};

static size_t prep_smem(const Dims& d, bool with_q) {
    const int C = d.C;
    size_t f = (size_t)C * (d.dk + 1) + (size_t)C * (d.dv + 1) + 2 * (size_t)C * (C + 1) + C;
    if (with_q) f += (size_t)C * (d.dk + 1);
    return f * sizeof(float);
}

template <typename Tin>
__global__ void __launch_bounds__(kNT) k_prep(PrepArgs a) {
    extern __shared__ float sm[];
    const long long bh = blockIdx.x;
    const int c = blockIdx.y;
    const int C = a.C, dk = a.dk, dv = a.dv, L = a.L;
    const int ldk = dk + 1, ldv = dv + 1, ldc = C + 1;
    float* Ks = sm;                 // [C][ldk]
    float* Vs = Ks + C * ldk;       // [C][ldv]
    float* As = Vs + C * ldv;       // [C][ldc]
    float* Ts = As + C * ldc;       // [C][ldc]
    float* al = Ts + C * ldc;       // [C]
    float* Qs = al + C;             // [C][ldk]  (only with P)
    const Tin* kp = (const Tin*)a.k;
    const Tin* vp = (const Tin*)a.v;
    const int t0 = c * C;
    const long long tok0 = bh * L + t0;
    const int nvalid = min(C, L - t0);

    for (int idx = threadIdx.x; idx < C * dk; idx += kNT) {
        const int i = idx / dk, x = idx - i * dk;
        Ks[i * ldk + x] = i < nvalid ? ld_elem(kp + (tok0 + i) * dk + x) : 0.f;
    }
    for (int idx = threadIdx.x; idx < C * dv; idx += kNT) {
        const int i = idx / dv, x = idx - i * dv;
        Vs[i * ldv + x] = i < nvalid ? ld_elem(vp + (tok0 + i) * dv + x) : 0.f;
    }
    if (a.P) {
        const Tin* qp = (const Tin*)a.q;
        for (int idx = threadIdx.x; idx < C * dk; idx += kNT) {
            const int i = idx / dk, x = idx - i * dk;
            Qs[i * ldk + x] = i < nvalid ? ld_elem(qp + (tok0 + i) * dk + x) : 0.f;
        }
    }
    __syncthreads();

    // lambda_t = ||k_t||^2 and alpha_t, one warp per token
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = warp; i < C; i += kNT / 32) {
        float s = 0.f;
        for (int x = lane; x < dk; x += 32) {
            const float kx = Ks[i * ldk + x];
            s = fmaf(kx, kx, s);
        }
        s = warp_sum(s);
        if (lane == 0) {
            const float b = i < nvalid ? a.beta[tok0 + i] : 0.f;
            al[i] = alpha_of(b, s, a.euler);
        }
    }
    __syncthreads();

    // A = strict_lower(diag(alpha) K K^T)
    block_mm_ranged<kNT>(
        C, C, [&](int i, int x) { return Ks[i * ldk + x]; },
        [&](int x, int j) { return Ks[j * ldk + x]; },
        [&](int i, int j, int& lo, int& hi) { lo = 0; hi = (j < i) ? dk : 0; },
        [&](int i, int j, float s) { As[i * ldc + j] = al[i] * s; });
    if (a.P) {
        // P = tril(Q K^T), diagonal included
        float* Pg = a.P + ((size_t)bh * a.NC + c) * C * C;
        block_mm_ranged<kNT>(
            C, C, [&](int i, int x) { return Qs[i * ldk + x]; },
            [&](int x, int j) { return Ks[j * ldk + x]; },
            [&](int i, int j, int& lo, int& hi) { lo = 0; hi = (j <= i) ? dk : 0; },
            [&](int i, int j, float s) { Pg[(size_t)i * C + j] = s; });
    }
    __syncthreads();

    // T = (I + A)^{-1} by forward substitution over rows:
    //   (I + A) T = I  =>  T[i][:] = e_i - sum_{j<i} A[i][j] T[j][:]   (T[j][col] = 0 for col > j)
    for (int i = 0; i < C; ++i) {
        for (int col = threadIdx.x; col < C; col += kNT) {
            float x = (col == i) ? 1.f : 0.f;
            for (int j = col; j < i; ++j) x = fmaf(-As[i * ldc + j], Ts[j * ldc + col], x);
            Ts[i * ldc + col] = x;
        }
        __syncthreads();
    }

    // K <- diag(alpha) K, V <- diag(alpha) V
    for (int idx = threadIdx.x; idx < C * dk; idx += kNT) {
        const int i = idx / dk, x = idx - i * dk;
        Ks[i * ldk + x] *= al[i];
    }
    for (int idx = threadIdx.x; idx < C * dv; idx += kNT) {
        const int i = idx / dv, x = idx - i * dv;
        Vs[i * ldv + x] *= al[i];
    }
    __syncthreads();

    const size_t chunk = (size_t)bh * a.NC + c;
    float* Wg = a.W + chunk * C * dk;
    float* Ug = a.U + chunk * C * dv;
    // W = T (alpha K), U = T (alpha V); T is lower triangular, so j <= i
    block_mm_ranged<kNT>(
        C, dk, [&](int i, int j) { return Ts[i * ldc + j]; },
        [&](int j, int x) { return Ks[j * ldk + x]; },
        [&](int i, int, int& lo, int& hi) { lo = 0; hi = i + 1; },
        [&](int i, int x, float s) { Wg[(size_t)i * dk + x] = s; });
    block_mm_ranged<kNT>(
        C, dv, [&](int i, int j) { return Ts[i * ldc + j]; },
        [&](int j, int x) { return Vs[j * ldv + x]; },
        [&](int i, int, int& lo, int& hi) { lo = 0; hi = i + 1; },
        [&](int i, int x, float s) { Ug[(size_t)i * dv + x] = s; });
    for (int i = threadIdx.x; i < C; i += kNT) a.alpha[chunk * C + i] = al[i];
    if (a.T) {
        float* Tg = a.T + chunk * C * C;
        for (int idx = threadIdx.x; idx < C * C; idx += kNT) {
            const int i = idx / C, j = idx - i * C;
            Tg[idx] = Ts[i * ldc + j];
        }
    }
}

// --------------------------------------------------------------- k_scan
struct ScanArgs {
    const void* k;
    const float* W;
    const float* U;
    const float* S0;     // nullable
    float* Up;
    float* Sc;
    float* S_final;      // nullable
    int L, dk, dv, C, NC, BV;
};

static size_t scan_smem(const Dims& d, int BV) {
    return ((size_t)d.dk * BV + 2 * (size_t)d.C * (d.dk + 1) + (size_t)d.C * (BV + 1)) *
           sizeof(float);
}

template <typename Tin>
__global__ void __launch_bounds__(kNT) k_scan(ScanArgs a) {
    extern __shared__ float sm[];
    const long long bh = blockIdx.x;
    const int v0 = blockIdx.y * a.BV;
    const int C = a.C, dk = a.dk, dv = a.dv, BV = a.BV, L = a.L;
    const int ldk = dk + 1, ldu = BV + 1;
    float* Ss = sm;                 // [dk][BV]  state slice, fp32
    float* Ws = Ss + dk * BV;       // [C][ldk]
    float* Ks = Ws + C * ldk;       // [C][ldk]
    float* Us = Ks + C * ldk;       // [C][ldu]  U, then Up
    const Tin* kp = (const Tin*)a.k;

    for (int idx = threadIdx.x; idx < dk * BV; idx += kNT) {
        const int r = idx / BV, n = idx - r * BV;
        Ss[idx] = a.S0 ? a.S0[((size_t)bh * dk + r) * dv + v0 + n] : 0.f;
    }
    for (int c = 0; c < a.NC; ++c) {
        const int t0 = c * C;
        const int nvalid = min(C, L - t0);
        const long long tok0 = bh * L + t0;
        const size_t chunk = (size_t)bh * a.NC + c;
        const float* Wg = a.W + chunk * C * dk;
        const float* Ug = a.U + chunk * C * dv;
        for (int idx = threadIdx.x; idx < C * dk; idx += kNT) {
            const int i = idx / dk, x = idx - i * dk;
            Ws[i * ldk + x] = Wg[idx];
            Ks[i * ldk + x] = i < nvalid ? ld_elem(kp + (tok0 + i) * dk + x) : 0.f;
        }
        for (int idx = threadIdx.x; idx < C * BV; idx += kNT) {
            const int i = idx / BV, n = idx - i * BV;
            Us[i * ldu + n] = Ug[(size_t)i * dv + v0 + n];
        }
        __syncthreads();   // also orders the previous chunk's S update before this read
        float* Scg = a.Sc + chunk * dk * dv;
        for (int idx = threadIdx.x; idx < dk * BV; idx += kNT) {
            const int r = idx / BV, n = idx - r * BV;
            Scg[(size_t)r * dv + v0 + n] = Ss[idx];
        }
        // Up = U - W S
        float* Upg = a.Up + chunk * C * dv;
        block_mm<kNT>(
            C, BV, dk, [&](int i, int x) { return Ws[i * ldk + x]; },
            [&](int x, int n) { return Ss[x * BV + n]; },
            [&](int i, int n, float s) {
                const float u = Us[i * ldu + n] - s;
                Us[i * ldu + n] = u;
                Upg[(size_t)i * dv + v0 + n] = u;
            });
        __syncthreads();
        // S += K^T Up
        block_mm<kNT>(
            dk, BV, C, [&](int x, int i) { return Ks[i * ldk + x]; },
            [&](int i, int n) { return Us[i * ldu + n]; },
            [&](int x, int n, float s) { Ss[x * BV + n] += s; });
        __syncthreads();
    }
    if (a.S_final) {
        for (int idx = threadIdx.x; idx < dk * BV; idx += kNT) {
            const int r = idx / BV, n = idx - r * BV;
            a.S_final[((size_t)bh * dk + r) * dv + v0 + n] = Ss[idx];
        }
    }
}

// ---------------------------------------------------------------- k_out
struct OutArgs {
    const void* q;
    const void* k;
    const float* Sc;
    const float* Up;
    void* o;
    int L, dk, dv, C, NC, BV;
};

static size_t out_smem(const Dims& d, int BV) {
    const size_t C = d.C;
    return (2 * C * (d.dk + 1) + C * (C + 1) + (size_t)d.dk * BV + C * BV) * sizeof(float);
}

template <typename Tin, typename Tout>
__global__ void __launch_bounds__(kNT) k_out(OutArgs a) {
    extern __shared__ float sm[];
    const long long bh = blockIdx.x;
    const int c = blockIdx.y;
    const int v0 = blockIdx.z * a.BV;
    const int C = a.C, dk = a.dk, dv = a.dv, BV = a.BV, L = a.L;
    const int ldk = dk + 1, ldc = C + 1;
    float* Qs = sm;                 // [C][ldk]
    float* Ks = Qs + C * ldk;       // [C][ldk]
    float* Ps = Ks + C * ldk;       // [C][ldc]
    float* Ss = Ps + C * ldc;       // [dk][BV]
    float* Us = Ss + dk * BV;       // [C][BV]
    const Tin* qp = (const Tin*)a.q;
    const Tin* kp = (const Tin*)a.k;
    const int t0 = c * C;
    const int nvalid = min(C, L - t0);
    const long long tok0 = bh * L + t0;
    const size_t chunk = (size_t)bh * a.NC + c;

    for (int idx = threadIdx.x; idx < C * dk; idx += kNT) {
        const int i = idx / dk, x = idx - i * dk;
        const bool ok = i < nvalid;
        Qs[i * ldk + x] = ok ? ld_elem(qp + (tok0 + i) * dk + x) : 0.f;
        Ks[i * ldk + x] = ok ? ld_elem(kp + (tok0 + i) * dk + x) : 0.f;
    }
    const float* Scg = a.Sc + chunk * dk * dv;
    for (int idx = threadIdx.x; idx < dk * BV; idx += kNT) {
        const int r = idx / BV, n = idx - r * BV;
        Ss[idx] = Scg[(size_t)r * dv + v0 + n];
    }
    const float* Upg = a.Up + chunk * C * dv;
    for (int idx = threadIdx.x; idx < C * BV; idx += kNT) {
        const int i = idx / BV, n = idx - i * BV;
        Us[idx] = Upg[(size_t)i * dv + v0 + n];
    }
    __syncthreads();
    // P = tril(Q K^T), diagonal included
    block_mm_ranged<kNT>(
        C, C, [&](int i, int x) { return Qs[i * ldk + x]; },
        [&](int x, int j) { return Ks[j * ldk + x]; },
        [&](int i, int j, int& lo, int& hi) { lo = 0; hi = (j <= i) ? dk : 0; },
        [&](int i, int j, float s) { Ps[i * ldc + j] = s; });
    __syncthreads();
    // O = Q S_c + P Up
    Tout* op = (Tout*)a.o;
    for (int idx = threadIdx.x; idx < C * BV; idx += kNT) {
        const int i = idx / BV, n = idx - i * BV;
        if (i >= nvalid) continue;
        float s = 0.f;
        for (int x = 0; x < dk; ++x) s = fmaf(Qs[i * ldk + x], Ss[x * BV + n], s);
        for (int j = 0; j <= i; ++j) s = fmaf(Ps[i * ldc + j], Us[j * BV + n], s);
        st_elem(op + (tok0 + i) * dv + v0 + n, s);
    }
}

// ------------------------------------------------------------------- launch
static int pick_bv(int dv, int want) {
    int bv = want;
    while (bv > 16 && dv % bv) bv >>= 1;
    return bv > dv ? dv : bv;
}

template <typename Tin>
static cudaError_t run_prep(const Dims& d, const void* q, const void* k, const void* v,
                            const float* beta, float* alpha, float* W, float* U, float* T,
                            float* P, cudaStream_t st) {
    PrepArgs a{q, k, v, beta, alpha, W, U, T, P, d.L, d.dk, d.dv, d.C, d.NC, d.euler};
    const size_t sm = prep_smem(d, P != nullptr);
    cudaError_t e = cudaFuncSetAttribute(k_prep<Tin>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)sm);
    if (e != cudaSuccess) return e;
    k_prep<Tin><<<dim3((unsigned)d.BH(), d.NC), kNT, sm, st>>>(a);
    prof_mark("efla_chunk_prep", st);
    return cudaGetLastError();
}

template <typename Tin>
static cudaError_t run_scan(const Dims& d, const void* k, const float* W, const float* U,
                            const float* S0, float* Up, float* Sc, float* S_final,
                            cudaStream_t st) {
    const int BV = pick_bv(d.dv, 32);
    ScanArgs a{k, W, U, S0, Up, Sc, S_final, d.L, d.dk, d.dv, d.C, d.NC, BV};
    const size_t sm = scan_smem(d, BV);
    cudaError_t e = cudaFuncSetAttribute(k_scan<Tin>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)sm);
    if (e != cudaSuccess) return e;
    k_scan<Tin><<<dim3((unsigned)d.BH(), d.dv / BV), kNT, sm, st>>>(a);
    prof_mark("efla_state_scan", st);
    return cudaGetLastError();
}

template <typename Tin, typename Tout>
static cudaError_t fwd_impl(const Dims& d, const void* q, const void* k, const void* v,
                            const float* beta, const float* S0, void* o, float* S_final,
                            const FwdWs& ws, cudaStream_t st) {
    cudaError_t e = run_prep<Tin>(d, nullptr, k, v, beta, ws.alpha, ws.W, ws.U, ws.T, nullptr, st);
    if (e != cudaSuccess) return e;
    e = run_scan<Tin>(d, k, ws.W, ws.U, S0, ws.Up, ws.Sc, S_final, st);
    if (e != cudaSuccess) return e;
    const int BV = pick_bv(d.dv, 32);
    OutArgs oa{q, k, ws.Sc, ws.Up, o, d.L, d.dk, d.dv, d.C, d.NC, BV};
    const size_t sm = out_smem(d, BV);
    e = cudaFuncSetAttribute(k_out<Tin, Tout>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
    if (e != cudaSuccess) return e;
    k_out<Tin, Tout><<<dim3((unsigned)d.BH(), d.NC, d.dv / BV), kNT, sm, st>>>(oa);
    prof_mark("efla_chunk_out", st);
    return cudaGetLastError();
}

cudaError_t launch_fwd_simt(const Dims& d, const void* q, const void* k, const void* v,
                            const float* beta, const float* S0, void* o, float* S_final,
                            const FwdWs& ws, cudaStream_t st) {
    if (d.in_bf16) {
        return d.out_bf16 ? fwd_impl<__nv_bfloat16, __nv_bfloat16>(d, q, k, v, beta, S0, o, S_final, ws, st)
                          : fwd_impl<__nv_bfloat16, float>(d, q, k, v, beta, S0, o, S_final, ws, st);
    }
    return d.out_bf16 ? fwd_impl<float, __nv_bfloat16>(d, q, k, v, beta, S0, o, S_final, ws, st)
                      : fwd_impl<float, float>(d, q, k, v, beta, S0, o, S_final, ws, st);
}

// Shared with the backward pass (bwd_simt.cu).
cudaError_t launch_prep_for_bwd(const Dims& d, const void* q, const void* k, const void* v,
                                const float* beta, const BwdWs& ws, cudaStream_t st) {
    if (grad_mma_supported(d)) {
        const cudaError_t e = launch_prep_mma(d, q, k, v, beta, ws, st);
        prof_mark("efla_chunk_prep", st);
        return e;
    }
    return d.in_bf16
               ? run_prep<__nv_bfloat16>(d, q, k, v, beta, ws.f.alpha, ws.f.W, ws.f.U, ws.T, ws.P, st)
               : run_prep<float>(d, q, k, v, beta, ws.f.alpha, ws.f.W, ws.f.U, ws.T, ws.P, st);
}

cudaError_t launch_scan_for_bwd(const Dims& d, const void* k, const float* S0, const BwdWs& ws,
                                cudaStream_t st) {
    if (grad_mma_supported(d)) {
        const cudaError_t e = launch_scan_mma(d, k, S0, ws, st);
        prof_mark("efla_state_scan", st);
        return e;
    }
    return d.in_bf16 ? run_scan<__nv_bfloat16>(d, k, ws.f.W, ws.f.U, S0, ws.f.Up, ws.f.Sc, nullptr, st)
                     : run_scan<float>(d, k, ws.f.W, ws.f.U, S0, ws.f.Up, ws.f.Sc, nullptr, st);
}

// ------------------------------------------------------------- state copy
__global__ void k_state_copy(long long n, const float* __restrict__ src, float* __restrict__ dst) {
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n;
         i += (long long)gridDim.x * blockDim.x)
        dst[i] = src ? src[i] : 0.f;
}

cudaError_t launch_state_copy(long long n, const float* S0, float* S_final, cudaStream_t st) {
    if (n <= 0) return cudaSuccess;
    long long blocks = (n + 255) / 256;
    if (blocks > 152 * 16) blocks = 152 * 16;
    k_state_copy<<<(unsigned)blocks, 256, 0, st>>>(n, S0, S_final);
    prof_mark("efla_state_copy", st);
    return cudaGetLastError();
}

}  // namespace efla

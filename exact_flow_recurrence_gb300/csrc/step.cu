// step.cu -- single-token recurrent decode step of EFLA (fp32 state, in place).
//
// For each sequence (page es, Metodologia item 3, applied to one token):
//   lambda = ||k||^2,  alpha = (1 - e^{-beta lambda}) / lambda
//   r      = v - S^T k                      (one read pass over S)
//   S     <- S + alpha k r^T                (= (I - alpha k k^T) S + alpha k v^T; one write pass)
//   o      = S_new^T q = S^T q + alpha (k . q) r
// The step is HBM-bound: 2 * dk * dv * 4 bytes of state traffic per sequence.
// A CTA of 256 threads owns DVC state columns of one sequence (all of them for
// dv < 128; half of them, two CTAs per sequence, for dv = 128): the columns of
// S^T k and S^T q are independent sums, so the only cost of the split is reading
// q and k twice.  Each thread keeps its share of the slice (rows g, g + RP, ...;
// four adjacent columns) in registers between the read and the write, so S
// crosses HBM exactly twice.  Loads and stores are 128-bit and each warp touches
// whole 256-byte row segments; three CTAs per SM keep one CTA's loads or stores
// in flight while another reduces.
#include "common.cuh"
#include "launch.h"

namespace efla {

struct StepArgs {
    const void* q;
    const void* k;
    const void* v;
    const float* beta;
    float* S;
    void* o;
    int dk, dv, euler;
};

template <typename Tin, typename Tout, int DV>   // DV: state columns of this CTA
__global__ void __launch_bounds__(256, DV <= 64 ? 3 : 2) k_step(StepArgs a) {
    constexpr int NT = 256;
    constexpr int C4 = DV / 4;          // float4 columns per state row
    constexpr int RP = NT / C4;         // state rows covered by one pass of the block
    constexpr int RT = (128 + RP - 1) / RP;   // rows per thread for dk <= 128
    __shared__ float qs[128], ks[128], vs[DV], rs[DV];
    __shared__ float red_k[RP][DV + 1], red_q[RP][DV + 1];
    __shared__ float s_alpha, s_kq;

    const long long h = blockIdx.x;
    const int dk = a.dk, dv = a.dv, col0 = blockIdx.y * DV;
    const int tid = threadIdx.x;
    const int c4 = tid % C4, g = tid / C4;
    // when 256 is not a multiple of DV/4 the last few threads own no rows
    const bool act = tid < RP * C4;
    float* Sh = a.S + h * (long long)dk * dv + col0;

    // issue the state loads first: they are the long-latency part
    float4 s[RT];
#pragma unroll
    for (int m = 0; m < RT; ++m) {
        const int r = g + m * RP;
        if (act && r < dk) s[m] = *reinterpret_cast<const float4*>(Sh + (size_t)r * dv + 4 * c4);
    }
    const Tin* qp = (const Tin*)a.q + h * dk;
    const Tin* kp = (const Tin*)a.k + h * dk;
    const Tin* vp = (const Tin*)a.v + h * dv + col0;
    for (int i = tid; i < dk; i += NT) {
        qs[i] = ld_elem(qp + i);
        ks[i] = ld_elem(kp + i);
    }
    for (int j = tid; j < DV; j += NT) vs[j] = ld_elem(vp + j);
    __syncthreads();

    if (tid < 32) {
        float l = 0.f, kq = 0.f;
        for (int i = tid; i < dk; i += 32) {
            l = fmaf(ks[i], ks[i], l);
            kq = fmaf(ks[i], qs[i], kq);
        }
        l = warp_sum(l);
        kq = warp_sum(kq);
        if (tid == 0) {
            s_alpha = alpha_of(a.beta[h], l, a.euler);
            s_kq = kq;
        }
    }
    // partial column sums of S^T k and S^T q over this thread's rows
    float pk0 = 0.f, pk1 = 0.f, pk2 = 0.f, pk3 = 0.f;
    float pq0 = 0.f, pq1 = 0.f, pq2 = 0.f, pq3 = 0.f;
#pragma unroll
    for (int m = 0; m < RT; ++m) {
        const int r = g + m * RP;
        if (act && r < dk) {
            const float kr = ks[r], qr = qs[r];
            pk0 = fmaf(s[m].x, kr, pk0); pk1 = fmaf(s[m].y, kr, pk1);
            pk2 = fmaf(s[m].z, kr, pk2); pk3 = fmaf(s[m].w, kr, pk3);
            pq0 = fmaf(s[m].x, qr, pq0); pq1 = fmaf(s[m].y, qr, pq1);
            pq2 = fmaf(s[m].z, qr, pq2); pq3 = fmaf(s[m].w, qr, pq3);
        }
    }
    if (act) {
        red_k[g][4 * c4 + 0] = pk0; red_k[g][4 * c4 + 1] = pk1;
        red_k[g][4 * c4 + 2] = pk2; red_k[g][4 * c4 + 3] = pk3;
        red_q[g][4 * c4 + 0] = pq0; red_q[g][4 * c4 + 1] = pq1;
        red_q[g][4 * c4 + 2] = pq2; red_q[g][4 * c4 + 3] = pq3;
    }
    __syncthreads();

    const float alpha = s_alpha;
    if (tid < DV) {
        float sk = 0.f, sq = 0.f;
#pragma unroll 8
        for (int gg = 0; gg < RP; ++gg) {
            sk += red_k[gg][tid];
            sq += red_q[gg][tid];
        }
        const float r = vs[tid] - sk;
        rs[tid] = r;
        st_elem((Tout*)a.o + h * dv + col0 + tid, fmaf(alpha * s_kq, r, sq));
    }
    __syncthreads();

    const float r0 = rs[4 * c4 + 0], r1 = rs[4 * c4 + 1], r2 = rs[4 * c4 + 2], r3 = rs[4 * c4 + 3];
#pragma unroll
    for (int m = 0; m < RT; ++m) {
        const int r = g + m * RP;
        if (act && r < dk) {
            const float ak = alpha * ks[r];
            float4 t = s[m];
            t.x = fmaf(ak, r0, t.x);
            t.y = fmaf(ak, r1, t.y);
            t.z = fmaf(ak, r2, t.z);
            t.w = fmaf(ak, r3, t.w);
            *reinterpret_cast<float4*>(Sh + (size_t)r * dv + 4 * c4) = t;
        }
    }
}

template <typename Tin, typename Tout>
static cudaError_t step_dispatch(const Dims& d, const StepArgs& a, cudaStream_t st) {
    const dim3 grid((unsigned)d.BH());
    if (d.dv == 128) {   // two 64-column CTAs per sequence
        k_step<Tin, Tout, 64><<<dim3((unsigned)d.BH(), 2), 256, 0, st>>>(a);
        prof_mark("efla_decode_step", st);
        return cudaGetLastError();
    }
    switch (d.dv) {
        case 16: k_step<Tin, Tout, 16><<<grid, 256, 0, st>>>(a); break;
        case 32: k_step<Tin, Tout, 32><<<grid, 256, 0, st>>>(a); break;
        case 48: k_step<Tin, Tout, 48><<<grid, 256, 0, st>>>(a); break;
        case 64: k_step<Tin, Tout, 64><<<grid, 256, 0, st>>>(a); break;
        case 80: k_step<Tin, Tout, 80><<<grid, 256, 0, st>>>(a); break;
        case 96: k_step<Tin, Tout, 96><<<grid, 256, 0, st>>>(a); break;
        case 112: k_step<Tin, Tout, 112><<<grid, 256, 0, st>>>(a); break;
        default: return cudaErrorInvalidValue;
    }
    prof_mark("efla_decode_step", st);
    return cudaGetLastError();
}

cudaError_t launch_step(const Dims& d, const void* q, const void* k, const void* v,
                        const float* beta, float* S, void* o, cudaStream_t st) {
    StepArgs a{q, k, v, beta, S, o, d.dk, d.dv, d.euler};
    if (d.in_bf16)
        return d.out_bf16 ? step_dispatch<__nv_bfloat16, __nv_bfloat16>(d, a, st)
                          : step_dispatch<__nv_bfloat16, float>(d, a, st);
    return d.out_bf16 ? step_dispatch<float, __nv_bfloat16>(d, a, st)
                      : step_dispatch<float, float>(d, a, st);
}

}  // namespace efla

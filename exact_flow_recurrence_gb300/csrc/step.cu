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
//
// For dk = dv = 128 (each sequence's state one contiguous 64 KB block) the state goes
// through shared memory instead (k_step_tma): one persistent CTA per SM takes every
// gridDim.x-th sequence; a producer thread bulk-copies a sequence's state and its q, k, v
// rows into one of three 64 KB stages while eight consumer warps update the stage before
// and store the new state straight from registers (whole 512-byte rows per warp), so a
// stage is refilled as soon as its consumers are done with it.  The copies in need no
// registers and keep two states per SM in flight from HBM.
#include "common.cuh"
#include "launch.h"
#include "tc_common.cuh"

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

namespace {

__device__ unsigned int g_sd_status = 0;   // bit 0: a bounded wait of k_step_tma expired; kStatusBounds (debug builds): a write was skipped

constexpr int kSdConsumers = 256;                      // eight warps update the states
constexpr int kSdThreads = kSdConsumers + 32;          // and one producer warp copies them
constexpr int kSdStages = 3;
constexpr uint32_t kSdState = 128u * 128u * 4u;        // one sequence's fp32 state
constexpr uint32_t kSdStage = kSdState + 3u * 512u;    // + its q, k, v rows (fp32 at most)
constexpr uint32_t kSdRed = kSdStages * kSdStage;      // column partial sums [8][128] x 2 (fp32)
constexpr uint32_t kSdR = kSdRed + 8192u;              // r [128]
constexpr uint32_t kSdMisc = kSdR + 512u;              // alpha, k.q
constexpr uint32_t kSdBar = kSdMisc + 16u;             // full[3], done[3]
constexpr size_t kSdSmem = 128 + kSdBar + 2 * kSdStages * 8;
static_assert(kSdStage % 128 == 0, "stages stay 128-byte aligned");
static_assert(kSdSmem <= 232448, "shared memory per CTA");

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }

}  // namespace

// dk = dv = 128.  Stage s holds the state S[h] [128][128] and the rows q[h], k[h], v[h];
// full[s] completes when they have landed, done[s] when the 256 consumer threads have
// read the stage for the last time (after the column sums: each keeps its rows of S[h] and
// their k values in registers for the update, and the new S[h] and o[h] go to global memory
// from registers).  Consumer thread (warp w, lane l) owns columns 4l .. 4l+3 of rows w, w + 8, ...,
// w + 120: a warp reads and writes whole 512-byte rows.
// Every mbarrier wait is bounded; on expiry the status word is set, the consumers leave
// together (the wait's outcome is combined at a named barrier), and the producer lets
// the copies it issued land before it returns.
template <typename Tin, typename Tout>
__global__ void __launch_bounds__(kSdThreads, 1) k_step_tma(StepArgs a, int BH) {
    extern __shared__ unsigned char sd_raw[];
    unsigned char* sm = (unsigned char*)(((uintptr_t)sd_raw + 127) & ~(uintptr_t)127);
    uint64_t* full = (uint64_t*)(sm + kSdBar);
    uint64_t* done = full + kSdStages;
    float* red_k = (float*)(sm + kSdRed);
    float* red_q = red_k + 8 * 128;
    float* rs = (float*)(sm + kSdR);
    float* misc = (float*)(sm + kSdMisc);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const long long G = gridDim.x;
    constexpr uint32_t vb = 128u * sizeof(Tin);   // bytes of one q, k or v row
    if (tid == 0) {
        for (int s = 0; s < kSdStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&done[s], kSdConsumers);
        }
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kSdConsumers / 32) {
        // ================================ producer ================================
        if (lane == 0) {
            auto issue = [&](int s, long long h) {
                unsigned char* st = sm + s * kSdStage;
                mbar_arrive_expect_tx(&full[s], kSdState + 3u * vb);
                bulk_g2s(st, a.S + h * 16384, kSdState, &full[s]);
                bulk_g2s(st + kSdState, (const Tin*)a.q + h * 128, vb, &full[s]);
                bulk_g2s(st + kSdState + vb, (const Tin*)a.k + h * 128, vb, &full[s]);
                bulk_g2s(st + kSdState + 2 * vb, (const Tin*)a.v + h * 128, vb, &full[s]);
            };
            int issued = 0;
            while (issued < kSdStages && blockIdx.x + issued * G < BH) {
                issue(issued, blockIdx.x + issued * G);
                ++issued;
            }
            int it = 0;
            for (; blockIdx.x + it * G < BH; ++it) {
                const long long h = blockIdx.x + it * G;
                const int s = it % kSdStages;
                if (!mbar_wait(&done[s], (uint32_t)(it / kSdStages) & 1u, kWaitLimit)) {
                    atomicOr(&g_sd_status, 1u);
                    break;
                }
                if (h + kSdStages * G < BH) {   // the stage's next sequence (the consumers wrote it back)
                    issue(s, h + kSdStages * G);
                    ++issued;
                }
            }
            // (a run abandoned at item `it`: the loads issued beyond it land before the exit)
            for (int j = it; j < issued; ++j)
                mbar_wait(&full[j % kSdStages], (uint32_t)(j / kSdStages) & 1u, kWaitLimit);
            bulk_wait_all();
        }
        return;
    }

    // ================================ consumers ================================
    const int g = warp, c4 = lane;
    for (int it = 0; blockIdx.x + it * G < BH; ++it) {
        const long long h = blockIdx.x + it * G;
        const int s = it % kSdStages;
        const float beta_h = tid == 0 ? a.beta[h] : 0.f;   // in flight with the wait
        if (!group_sync_and(1, mbar_wait(&full[s], (uint32_t)(it / kSdStages) & 1u, kWaitLimit), kSdConsumers)) {
            if (tid == 0) atomicOr(&g_sd_status, 1u);
            break;
        }
        float* St = (float*)(sm + s * kSdStage);
        const Tin* qv = (const Tin*)(sm + s * kSdStage + kSdState);
        const Tin* kv = qv + 128;
        const Tin* vv = kv + 128;
        if (warp == 0) {   // lambda = ||k||^2 -> alpha, and k.q
            float l = 0.f, kq = 0.f;
            for (int i = lane; i < 128; i += 32) {
                const float ki = to_f(kv[i]);
                l = fmaf(ki, ki, l);
                kq = fmaf(ki, to_f(qv[i]), kq);
            }
            l = warp_sum(l);
            kq = warp_sum(kq);
            if (lane == 0) {
                misc[0] = alpha_of(beta_h, l, a.euler);
                misc[1] = kq;
            }
        }
        // partial column sums of S^T k and S^T q over this thread's 16 rows, which stay in
        // registers (with their k values) for the update: the stage goes back to the producer
        // as soon as this thread has read it
        float pk0 = 0.f, pk1 = 0.f, pk2 = 0.f, pk3 = 0.f, pq0 = 0.f, pq1 = 0.f, pq2 = 0.f, pq3 = 0.f;
        float4 sv[16];
        float kr[16];
#pragma unroll
        for (int m = 0; m < 16; ++m) {
            const int r = g + 8 * m;
            sv[m] = *reinterpret_cast<const float4*>(St + r * 128 + 4 * c4);
            kr[m] = to_f(kv[r]);
            const float qr = to_f(qv[r]);
            pk0 = fmaf(sv[m].x, kr[m], pk0); pk1 = fmaf(sv[m].y, kr[m], pk1);
            pk2 = fmaf(sv[m].z, kr[m], pk2); pk3 = fmaf(sv[m].w, kr[m], pk3);
            pq0 = fmaf(sv[m].x, qr, pq0); pq1 = fmaf(sv[m].y, qr, pq1);
            pq2 = fmaf(sv[m].z, qr, pq2); pq3 = fmaf(sv[m].w, qr, pq3);
        }
        const float vt = tid < 128 ? to_f(vv[tid]) : 0.f;
        mbar_arrive(&done[s]);
        *reinterpret_cast<float4*>(red_k + g * 128 + 4 * c4) = make_float4(pk0, pk1, pk2, pk3);
        *reinterpret_cast<float4*>(red_q + g * 128 + 4 * c4) = make_float4(pq0, pq1, pq2, pq3);
        group_sync(1, kSdConsumers);
        const float alpha = misc[0];   // (read before the next barrier: warp 0 rewrites it for the next state)
        if (tid < 128) {   // column tid: r = v - S^T k, o = S^T q + alpha (k.q) r
            float sk = 0.f, sq = 0.f;
#pragma unroll
            for (int gg = 0; gg < 8; ++gg) {
                sk += red_k[gg * 128 + tid];
                sq += red_q[gg * 128 + tid];
            }
            const float r = vt - sk;
            rs[tid] = r;
            Tout* op = (Tout*)a.o + h * 128 + tid;
            if (dbg_in(op, sizeof(Tout), a.o, (size_t)BH * 128 * sizeof(Tout), &g_sd_status))
                st_elem(op, fmaf(alpha * misc[1], r, sq));
        }
        group_sync(1, kSdConsumers);
        // S += alpha k r^T on this thread's rows, from and to registers, stored to global memory
        const float4 rr = *reinterpret_cast<const float4*>(rs + 4 * c4);
        float* Sg = a.S + h * 16384;
        const bool wr = dbg_in(Sg, kSdState, a.S, (size_t)BH * kSdState, &g_sd_status);
#pragma unroll
        for (int m = 0; m < 16; ++m) {
            const int r = g + 8 * m;
            const float ak = alpha * kr[m];
            float4 t = sv[m];
            t.x = fmaf(ak, rr.x, t.x);
            t.y = fmaf(ak, rr.y, t.y);
            t.z = fmaf(ak, rr.z, t.z);
            t.w = fmaf(ak, rr.w, t.w);
            if (wr) __stcs(reinterpret_cast<float4*>(Sg + r * 128 + 4 * c4), t);
        }
    }
}

template <typename Tin, typename Tout>
static cudaError_t step_dispatch(const Dims& d, const StepArgs& a, cudaStream_t st) {
    const dim3 grid((unsigned)d.BH());
    const auto al16 = [](const void* p) { return ((uintptr_t)p & 15u) == 0; };
    if (d.dk == 128 && d.dv == 128 && al16(a.S) && al16(a.q) && al16(a.k) && al16(a.v)) {
        int dev = 0, nsm = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k_step_tma<Tin, Tout>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSdSmem);
        if (e != cudaSuccess) return e;
        const long long BH = d.BH();
        k_step_tma<Tin, Tout><<<(unsigned)(BH < nsm ? BH : nsm), kSdThreads, kSdSmem, st>>>(a, (int)BH);
        prof_mark("efla_decode_step", st);
        return cudaGetLastError();
    }
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

namespace efla {
cudaError_t sd_status_read_clear(unsigned int* status) {
    unsigned int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(status, g_sd_status, sizeof(unsigned int));
    if (e != cudaSuccess) return e;
    return *status ? cudaMemcpyToSymbol(g_sd_status, &zero, sizeof(unsigned int)) : cudaSuccess;
}
}  // namespace efla

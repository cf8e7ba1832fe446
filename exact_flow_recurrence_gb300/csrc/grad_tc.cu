// grad_tc.cu -- the backward's per-chunk gradients on the tcgen05 tensor cores (bf16
// inputs, dk = dv = 128, chunk 64).
//
// Same mathematics as k_grad_mma (bwd_mma.cu; reverse-mode differentiation of the chunk
// form of page es, Metodologia item 3 -- the pages give no backward pass).  Per chunk, with
// S = S_c, G = dSc (gradient of the state leaving the chunk), U = U', dU = dU':
//   D = tril(dO U^T)  dQ = dO S^T + D K        dW = -dU S^T
//   dT = (dW K^T + dU V^T) diag(alpha), strictly lower      X = dT T^T
//   dA = strict_lower(-T^T X)   dG = diag(alpha) dA   Ms = dG + dG^T
//   dKa = T^T dW   dVa = T^T dU   dV = diag(alpha) dVa
//   dK = D^T Q + U G^T + Ms K + diag(alpha) dKa + 2 diag(dlambda) K
//   dalpha_j = sum_{m<j} dA_jm (K K^T)_jm + <dKa_j, k_j> + <dVa_j, v_j>
// Every product is a tcgen05.mma with M = 128 (fp16 operands staged in 128-byte-swizzled
// shared memory, fp32 accumulators in tensor memory), arranged so that the d dimension
// (or two stacked 64-row operands) fills M:
//   R2 | R1  [-dW^T | dQ^T] = S [dU; dO]^T (one N = 128 product)    R3  dK^T = G U^T
//   R5  [dU; dO] [V; U]^T -> dU V^T (lanes 0..63) and D = dO U^T (lanes 64..127)
//   R10 dVa^T = dU^T T
//   R6  dQ^T += K^T D^T           R7  dK^T += Q^T D           R8  [dW; K] K^T -> dW K^T, K K^T
//   R9  dKa^T = dW^T T            R11 X = [dT; 0] T^T         R12 dA' = [T | 0]^T X
//   R13 dK^T += K^T Ms
// in six dependent groups separated by epilogues (tensor memory -> registers -> fp16
// tiles).  One persistent CTA per SM walks the chunks; the next chunk's inputs are
// prefetched into L2 (bulk prefetches) while the current one computes, and the dq, dk and
// dv rows of a chunk (contiguous in memory) leave through shared-memory tiles by bulk
// copies.
//
// Staging: the bf16 dO, V, K, Q rows arrive by TMA (64 x 64 boxes with the 128-byte swizzle,
// i.e. straight into the tile layout; rows past the sequence read as zero) and are converted
// to fp16 in place -- dO and V before the first group, K and Q (first read by the second)
// while it runs.  K and Q go out before the wait for the previous chunk's output copies,
// since no output tile lives in their tiles.  T, alpha and beta are loaded through registers.
// G and dU arrive as the reverse scan's fp16 images (bwd_tc.cu), S and U' as the recording
// forward's (fwd_tc.cu), already in the tile layout, by bulk copy; for a sequence one of them
// recomputed in fp32 they are staged from the fp32 arrays through registers instead.
//
// Range: a chunk whose staged inputs leave fp16's range (largest |element| of S, G, U, dU,
// dO or T at 2^15 or more, or a nonzero tile entirely below 2^-14; G and dU checked when
// staged from fp32) or whose gradients come out non-finite is marked; k_grad_mma (tf32)
// recomputes exactly the marked chunks after (k_widen first gives an image-fed chunk its
// exact fp32 dSc and dUp).
#include <type_traits>

#include "common.cuh"
#include "launch.h"
#include "tc_common.cuh"
#include "tc_ptx.cuh"

namespace efla {

namespace {

__device__ unsigned int g_gt_status = 0;   // bit 0: a bounded wait expired; kStatusBounds (debug builds): a write was skipped

constexpr int kGtThreads = 512;   // 16 warps: lane quadrant q = warp & 3, column quarter h = warp >> 2
// shared memory (byte offsets from a 1024-aligned base); fp16 SW128 tiles, rows of 64
constexpr uint32_t kGtOU = 0;           // [dU; dO]: rows 0..63 dU, 64..127 dO; n-blocks 16 KB apart
constexpr uint32_t kGtUV = 32768;       // [V; U]:   rows 0..63 V,  64..127 U
constexpr uint32_t kGtWK = 65536;       // [dW; K]:  rows 0..63 dW, 64..127 K;  d-blocks 16 KB apart
constexpr uint32_t kGtQ = 98304;        // Q rows [64], d-blocks 8 KB apart
constexpr uint32_t kGtT = 114688;       // T rows [64][64], then a zero block (8 KB)
constexpr uint32_t kGtR = 131072;       // 64 KB reused: S and G for the first group, then:
constexpr uint32_t kGtS = kGtR;         //   S rows d [128], n-blocks 16 KB apart
constexpr uint32_t kGtG = kGtR + 32768; //   G likewise
constexpr uint32_t kGtD = kGtR;         //   D rows i [64][64]
constexpr uint32_t kGtdT = kGtR + 8192; //   [dT; 0] rows [128][64]; after X, dG fp32 [64][64] (swizzled)
constexpr uint32_t kGtX = kGtR + 24576; //   X rows m [64][64]
constexpr uint32_t kGtM = kGtR + 32768; //   Ms rows i [64][64]
constexpr uint32_t kGtGs = kGtR + 40960;//   K K^T fp32 [64][kGsLd]
constexpr int kGsLd = 68;
constexpr uint32_t kGtAux = kGtR + 65536;   // alpha, beta, lambda; dalpha parts [3][4][64]; dl2; tile maxima
constexpr uint32_t kGtBar = kGtAux + 8192;
constexpr size_t kGtSmem = 1024 + kGtBar + 64;
static_assert(kGtGs + 64 * kGsLd * 4 <= kGtR + 65536, "reused region");
static_assert(kGtAux + 1032 * 4 <= kGtBar, "aux region");
static_assert(kGtSmem <= 232448, "shared memory per CTA");

// tensor-memory columns (fp32 accumulators, lane = row)
// cW and cQ adjacent: R1 and R2 are one product of N = 128 into them
constexpr uint32_t cW = 0, cQ = 64, cK = 128, cR5 = 192, cR8 = 320, cKa = 384, cVa = 448;
constexpr uint32_t cX = cR5, cA = cR5 + 64;   // reuse R5's columns once they are read

constexpr float kGtHi = 32768.f, kGtLo = 1.f / 16384.f;

struct GtArgs {
    const __nv_bfloat16* q;
    const __nv_bfloat16* k;
    const __nv_bfloat16* v;
    const __nv_bfloat16* dO;
    const float* beta;
    const float* alpha;   // [BH][NC][64]
    const float* T;       // [BH][NC][64][64]
    const float* Sc;      // [BH][NC][128][128]
    const float* dSc;
    const float* Up;      // [BH][NC][64][128]
    const float* dUp;
    void* dq;
    void* dk;
    void* dv;
    float* dbeta;
    int* redo_n;          // chunks for k_grad_mma to recompute: their number,
    int* redo;            //   and their indices
    const int* seq_bad;   // [BH]: sequences whose dSc, dUp are the fp32 arrays (else the images)
    const int* fwd_fp32;  // null: Sc, Up are fp32; else [BH]: set for the sequences whose Sc, Up
                          //   are fp32, the others hold the forward's fp16 images there
    const unsigned char* gimg;   // [BH][NC] dSc images (32 KB)
    const unsigned char* uimg;   // [BH][NC] dUp images (16 KB)
    int L, NC, nchunks, euler, out_bf16;
};

__device__ __forceinline__ void tile_max(float& m, const float4& a) {
    m = fmaxf(m, fmaxf(fmaxf(fabsf(a.x), fabsf(a.y)), fmaxf(fabsf(a.z), fabsf(a.w))));
}

// 8 fp32 -> one 16-byte fp16 chunk (raising the tile maximum)
__device__ __forceinline__ uint4 f32x8_to_f16(const float4& a, const float4& b, float& m) {
    tile_max(m, a);
    tile_max(m, b);
    uint4 w;
    w.x = pack_f16x2(a.x, a.y);
    w.y = pack_f16x2(a.z, a.w);
    w.z = pack_f16x2(b.x, b.y);
    w.w = pack_f16x2(b.z, b.w);
    return w;
}

// read-only 16-byte loads (inputs the kernel never writes)
__device__ __forceinline__ float4 ldg4(const float* p) { return __ldg(reinterpret_cast<const float4*>(p)); }
__device__ __forceinline__ uint4 ldg_u4(const __nv_bfloat16* p) { return __ldg(reinterpret_cast<const uint4*>(p)); }

// element i of an output tile in shared memory (rows of 128, bf16 or fp32)
__device__ __forceinline__ void st_tile(unsigned char* t, int i, float x, int bf16) {
    if (bf16) reinterpret_cast<__nv_bfloat16*>(t)[i] = __float2bfloat16_rn(x);
    else reinterpret_cast<float*>(t)[i] = x;
}

// Column sums over the warp of 16 values per lane (recursive halving): lanes l and l ^ 1
// return the sum over all 32 lanes of x[(l >> 1) & 15].  x is overwritten.
__device__ __forceinline__ float xpose_sum16(float (&x)[16], int lane) {
#pragma unroll
    for (int n = 8, b = 16; n >= 1; n >>= 1, b >>= 1) {
        const bool up = (lane & b) != 0;
#pragma unroll
        for (int i = 0; i < n; ++i) {
            const float send = up ? x[i] : x[i + n];
            const float keep = up ? x[i + n] : x[i];
            x[i] = keep + __shfl_xor_sync(0xffffffffu, send, b);
        }
    }
    return x[0] + __shfl_xor_sync(0xffffffffu, x[0], 1);
}

__global__ void __launch_bounds__(kGtThreads, 1)
    k_grad_tc(const __grid_constant__ CUtensorMap tm_do, const __grid_constant__ CUtensorMap tm_v,
              const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q, GtArgs a) {
    extern __shared__ __align__(1024) unsigned char sm_raw[];
    unsigned char* sm = (unsigned char*)(((uintptr_t)sm_raw + 1023) & ~(uintptr_t)1023);
    float* al = (float*)(sm + kGtAux);     // alpha [64]
    float* bet = al + 64;                  // beta [64]
    float* lam = al + 128;                 // lambda [64]
    float* partV = al + 192;               // [4][64] <dVa_j, v_j> per lane quadrant
    float* partK = al + 448;               // [4][64] <dKa_j, k_j> per lane quadrant
    float* partA = al + 704;               // [4][64] sum_m dA_jm G_jm per column quarter
    float* dl2 = al + 960;                 // [64] 2 dalpha dalpha/dlambda
    unsigned* gmax = (unsigned*)(al + 1024);   // [6] largest |S|, |G|, |U|, |dU|, |dO|, |T| (fp32 bits)
    float* Gs = (float*)(sm + kGtGs);
    float* dGs = (float*)(sm + kGtdT);
    uint64_t* bar = (uint64_t*)(sm + kGtBar);
    uint64_t* ldb = bar + 1;               // the image copies of a chunk
    uint32_t* slot = (uint32_t*)(bar + 2);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int q = warp & 3, h = warp >> 2;   // lane quadrant, column quarter
    // the list-driven fallbacks after this kernel may be scheduled as this grid's CTAs leave
    // (they wait for its completion before reading the lists it writes)
    griddep_launch_dependents();
    const int row = q * 32 + lane;           // tensor-memory lane this thread reads
    const int jc = 16 * h + ((lane >> 1) & 15);   // the column a transposed sum leaves in this lane

    if (tid == 0) {
        mbar_init(bar, 1);
        mbar_init(ldb, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(slot, 512);
        tmem_relinquish();
    }
    *reinterpret_cast<uint4*>(sm + kGtT + 8192 + 16 * tid) = make_uint4(0, 0, 0, 0);   // the zero block after T
    if (tid < 6) gmax[tid] = 0u;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = *slot;
    uint32_t ph = 0, lph = 0;
    bool ok = true;

    // all threads: wait for the MMA group just committed (bounded; one outcome for all)
    auto mma_done = [&]() -> bool {
        const bool w = mbar_wait(bar, ph, kWaitLimit);
        ph ^= 1u;
        const bool all = __syncthreads_and(w);
        tc_fence_after();
        return all;
    };
    // the issuing thread's view of shared memory written by the others, then a commit
    auto sync_for_mma = [&]() {
        fence_async_smem();
        tmem_st_wait();
        tc_fence_before();
        __syncthreads();
    };

    for (int chunk = blockIdx.x; chunk < a.nchunks && ok; chunk += gridDim.x) {
        const long long bh = chunk / a.NC;
        const int c = chunk - (int)(bh * a.NC);
        const int nv = min(64, a.L - c * 64);
        const size_t tok0 = (size_t)bh * a.L + (size_t)c * 64;
        float mx[6] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f};   // largest |x| staged: S, G, U, dU, dO, T
        const bool img = a.seq_bad[bh] == 0;             // G and dU from the images
        const bool simg = a.fwd_fp32 && a.fwd_fp32[bh] == 0;   // S and U from the forward's images
        // ---------------- stage the chunk's operands (fp16, swizzled).  Each thread owns the
        // 8-wide column group n8 of rows r0 + 32 i; its 16-byte loads (34, or 22 when G and
        // dU come as images) go out in two batches, the second issued before the first is
        // converted.
        auto stage = [&](auto tag, auto stag) {
            constexpr bool IMG = decltype(tag)::value, SIMG = decltype(stag)::value;
            {
                const int r0 = tid >> 4, n8 = (tid & 15) * 8;
                const uint32_t blk = (uint32_t)(n8 >> 6) * 16384u;
                const float* Sg = a.Sc + (size_t)chunk * 16384 + r0 * 128 + n8;
                const float* Gg = a.dSc + (size_t)chunk * 16384 + r0 * 128 + n8;
                const float* Ug = a.Up + (size_t)chunk * 8192 + r0 * 128 + n8;
                const float* dUg = a.dUp + (size_t)chunk * 8192 + r0 * 128 + n8;
                float4 bs[16], bu[8];
                // T row r0t, and alpha, beta of token tid (the bf16 rows dO, V, K, Q come by TMA)
                float4 t0, t1;
                float alv = 0.f, betv = 0.f;
                const int r0t = tid >> 3, j8 = (tid & 7) * 8;
                auto load_rows = [&]() {
                    const float* Tg = a.T + (size_t)chunk * 4096 + r0t * 64 + j8;
                    t0 = ldg4(Tg);
                    t1 = ldg4(Tg + 4);
                    if (tid < 64) {
                        alv = __ldg(a.alpha + (size_t)chunk * 64 + tid);
                        betv = tid < nv ? __ldg(a.beta + tok0 + tid) : 0.f;
                    }
                };
                // with every fp32 tile arriving as an image the registers are free: the loads
                // go out before the wait for the previous chunk's output copies, not after it
                if constexpr (IMG && SIMG) load_rows();
#pragma unroll
                for (int i = 0; i < 4; ++i) {   // S, G rows d = r0 + 32 i
                    if constexpr (!SIMG) {
                        bs[4 * i] = ldg4(Sg + i * 4096);
                        bs[4 * i + 1] = ldg4(Sg + i * 4096 + 4);
                    }
                    if constexpr (!IMG) {
                        bs[4 * i + 2] = ldg4(Gg + i * 4096);
                        bs[4 * i + 3] = ldg4(Gg + i * 4096 + 4);
                    }
                }
#pragma unroll
                for (int j = 0; j < 2; ++j) {   // U, dU rows i = r0 + 32 j
                    if constexpr (!SIMG) {
                        bu[4 * j] = ldg4(Ug + j * 4096);
                        bu[4 * j + 1] = ldg4(Ug + j * 4096 + 4);
                    }
                    if constexpr (!IMG) {
                        bu[4 * j + 2] = ldg4(dUg + j * 4096);
                        bu[4 * j + 3] = ldg4(dUg + j * 4096 + 4);
                    }
                }
                const unsigned char* si = (const unsigned char*)(a.Sc + (size_t)chunk * 16384);
                const unsigned char* ui = (const unsigned char*)(a.Up + (size_t)chunk * 8192);
                bool in = true, sin = true;   // (thread 0's view; debug builds check the image copies)
                if (tid == 0) {   // every copy of the chunk counts on ldb; K and Q rows go first (no
                    // output tile of the previous chunk lives in their tiles)
                    in = !IMG || (dbg_in(a.gimg + (size_t)chunk * 32768, 32768, a.gimg, (size_t)a.nchunks * 32768,
                                         &g_gt_status) &&
                                  dbg_in(a.uimg + (size_t)chunk * 16384, 16384, a.uimg, (size_t)a.nchunks * 16384,
                                         &g_gt_status));
                    sin = !SIMG || (dbg_in(si, 32768, a.Sc, (size_t)a.nchunks * 65536, &g_gt_status) &&
                                    dbg_in(ui, 16384, a.Up, (size_t)a.nchunks * 32768, &g_gt_status));
                    fence_async_smem();
                    mbar_arrive_expect_tx(ldb, 65536u + (IMG && in ? 49152u : 0u) + (SIMG && sin ? 49152u : 0u));
                    // bf16 rows straight into their tile rows (128-byte swizzle, 64 x 64 boxes; rows
                    // past the sequence read as zero), converted in place below
                    for (int b = 0; b < 2; ++b) {
                        tma_load_3d(sm + kGtWK + b * 16384 + 8192, &tm_k, 64 * b, c * 64, (int)bh, ldb);
                        tma_load_3d(sm + kGtQ + b * 8192, &tm_q, 64 * b, c * 64, (int)bh, ldb);
                    }
                }
                // the previous chunk's output tiles (OU, UV, R) must be read out by the bulk stores
                if (tid == 0) bulk_wait_read();
                __syncthreads();
                if (tid == 0) {   // the other rows and the images
                    fence_async_smem();
                    for (int b = 0; b < 2; ++b) {
                        tma_load_3d(sm + kGtOU + b * 16384 + 8192, &tm_do, 64 * b, c * 64, (int)bh, ldb);
                        tma_load_3d(sm + kGtUV + b * 16384, &tm_v, 64 * b, c * 64, (int)bh, ldb);
                    }
                    if (IMG && in) {   // G rows d; dU rows i (OU rows 0..63)
                        bulk_g2s(sm + kGtG, a.gimg + (size_t)chunk * 32768, 32768u, ldb);
                        bulk_g2s(sm + kGtOU, a.uimg + (size_t)chunk * 16384, 8192u, ldb);
                        bulk_g2s(sm + kGtOU + 16384, a.uimg + (size_t)chunk * 16384 + 8192, 8192u, ldb);
                    }
                    if (SIMG && sin) {   // S rows d; U rows i (UV rows 64..127)
                        bulk_g2s(sm + kGtS, si, 32768u, ldb);
                        bulk_g2s(sm + kGtUV + 8192, ui, 8192u, ldb);
                        bulk_g2s(sm + kGtUV + 16384 + 8192, ui + 8192, 8192u, ldb);
                    }
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t off = blk + sw128(r0 + 32 * i, n8 & 63);
                    if constexpr (!SIMG)
                        *reinterpret_cast<uint4*>(sm + kGtS + off) = f32x8_to_f16(bs[4 * i], bs[4 * i + 1], mx[0]);
                    if constexpr (!IMG)
                        *reinterpret_cast<uint4*>(sm + kGtG + off) = f32x8_to_f16(bs[4 * i + 2], bs[4 * i + 3], mx[1]);
                }
                if constexpr (!(IMG && SIMG)) load_rows();
#pragma unroll
                for (int j = 0; j < 2; ++j) {   // dU -> OU rows i, U -> UV rows 64 + i
                    const int r = r0 + 32 * j;
                    if constexpr (!IMG)
                        *reinterpret_cast<uint4*>(sm + kGtOU + blk + sw128(r, n8 & 63)) =
                            f32x8_to_f16(bu[4 * j + 2], bu[4 * j + 3], mx[3]);
                    if constexpr (!SIMG)
                        *reinterpret_cast<uint4*>(sm + kGtUV + blk + sw128(64 + r, n8 & 63)) =
                            f32x8_to_f16(bu[4 * j], bu[4 * j + 1], mx[2]);
                }
                *reinterpret_cast<uint4*>(sm + kGtT + sw128(r0t, j8)) = f32x8_to_f16(t0, t1, mx[5]);
                if (tid < 64) {
                    al[tid] = alv;
                    bet[tid] = betv;
                }
            }
        };
        if (img && simg) stage(std::true_type{}, std::true_type{});
        else if (img) stage(std::true_type{}, std::false_type{});
        else if (simg) stage(std::false_type{}, std::true_type{});
        else stage(std::false_type{}, std::false_type{});
#pragma unroll
        for (int t = 0; t < 6; ++t) {   // tile maxima but dO's (read after the barrier below)
            if (t == 4) continue;
            const unsigned m = __reduce_max_sync(0xffffffffu, __float_as_uint(mx[t]));
            if (lane == 0) atomicMax(&gmax[t], m);
        }
        if (tid == 0) {   // next chunk's inputs toward L2 while this one computes
            const int nxt = chunk + gridDim.x;
            if (nxt < a.nchunks) {
                const long long nbh = nxt / a.NC;
                const int nc = nxt - (int)(nbh * a.NC);
                const size_t ntok = (size_t)nbh * a.L + (size_t)nc * 64;
                const uint32_t rows = (uint32_t)min(64, a.L - nc * 64) * 256u;
                const bool nsimg = a.fwd_fp32 && a.fwd_fp32[nbh] == 0;
                bulk_prefetch_l2(a.Sc + (size_t)nxt * 16384, nsimg ? 32768 : 65536);
                bulk_prefetch_l2(a.Up + (size_t)nxt * 8192, nsimg ? 16384 : 32768);
                if (a.seq_bad[nbh] == 0) {
                    bulk_prefetch_l2(a.gimg + (size_t)nxt * 32768, 32768);
                    bulk_prefetch_l2(a.uimg + (size_t)nxt * 16384, 16384);
                } else {
                    bulk_prefetch_l2(a.dSc + (size_t)nxt * 16384, 65536);
                    bulk_prefetch_l2(a.dUp + (size_t)nxt * 8192, 32768);
                }
                bulk_prefetch_l2(a.T + (size_t)nxt * 4096, 16384);
                bulk_prefetch_l2(a.alpha + (size_t)nxt * 64, 256);
                if ((ntok & 3) == 0 && (rows & 1023u) == 0)   // 16-byte aligned, whole 16-byte pieces
                    bulk_prefetch_l2(a.beta + ntok, rows / 64u);
                bulk_prefetch_l2(a.dO + ntok * 128, rows);
                bulk_prefetch_l2(a.v + ntok * 128, rows);
                bulk_prefetch_l2(a.k + ntok * 128, rows);
                bulk_prefetch_l2(a.q + ntok * 128, rows);
            }
        }
        {   // the image and row copies (bounded wait; one outcome for all)
            const bool w = mbar_wait(ldb, lph, kWaitLimit);
            lph ^= 1u;
            if (!(ok = __syncthreads_and(w))) break;
        }
        // rows bf16 -> fp16 in place, 16-byte pieces (0..1023 dO, then V, K, Q; 512 per 8 KB row
        // block): dO and V here, K and Q (read from the second group on) while the first runs
        auto convert_rows = [&](int k0, int k1) {
#pragma unroll
            for (int k = k0; k < k1; ++k) {
                const int i = tid + 512 * k, m = i >> 10, e = i & 1023, b = e >> 9;
                const uint32_t off = (uint32_t)(e & 511) * 16u +
                                     (m == 0 ? kGtOU + b * 16384 + 8192 : m == 1 ? kGtUV + b * 16384
                                              : m == 2 ? kGtWK + b * 16384 + 8192 : kGtQ + b * 8192);
                uint4* pc = reinterpret_cast<uint4*>(sm + off);
                *pc = m == 0 ? bf16x8_to_f16x8_max(*pc, mx[4]) : bf16x8_to_f16x8(*pc);
            }
        };
        {
            convert_rows(0, 4);
            const unsigned m4 = __reduce_max_sync(0xffffffffu, __float_as_uint(mx[4]));
            if (lane == 0) atomicMax(&gmax[4], m4);
        }
        sync_for_mma();
        // a chunk whose staged tiles leave fp16's range goes to the tf32 kernel: any element
        // at 2^15 or more, or a nonzero tile entirely below 2^-14 (subnormal)
        bool bad = false;
#pragma unroll
        for (int t = 0; t < 6; ++t) {
            const float m = __uint_as_float(gmax[t]);
            bad = bad || m >= kGtHi || (m > 0.f && m < kGtLo);
        }
        if (tid == 0) {
            tc_fence_after();
            const uint32_t i64 = idesc_f16(128, 64), i128 = idesc_f16(128, 128), imm64 = idesc_f16(128, 64, true, true);
            const uint32_t S0 = smem_u32(sm + kGtS), G0 = smem_u32(sm + kGtG), OU = smem_u32(sm + kGtOU),
                           UV = smem_u32(sm + kGtUV), T0 = smem_u32(sm + kGtT);
            for (int s = 0; s < 8; ++s) {
                const uint32_t ko = (uint32_t)(s >> 2) * 16384u + (uint32_t)(s & 3) * 32u;
                mma_f16_ss(tb + cW, sdesc_sw128(S0 + ko), sdesc_sw128(OU + ko), i128, s > 0);          // R2 | R1
                mma_f16_ss(tb + cK, sdesc_sw128(G0 + ko), sdesc_sw128(UV + 8192 + ko), i64, s > 0);    // R3
                mma_f16_ss(tb + cR5, sdesc_sw128(OU + ko), sdesc_sw128(UV + ko), i128, s > 0);         // R5
            }
            for (int s = 0; s < 4; ++s)   // R10: dVa^T = dU^T T
                mma_f16_ss(tb + cVa, sdesc_sw128(OU + s * 2048, 16384), sdesc_sw128(T0 + s * 2048, 8192), imm64, s > 0);
            mma_commit(bar);
        }
        convert_rows(4, 8);   // K and Q (fenced for the tensor core before the second group)
        if (!(ok = mma_done())) break;
        if (tid < 6) gmax[tid] = 0u;   // every thread has read them (barrier in mma_done)
        // ---------------- epilogue 1: D tile, dW rows and the packed -dW^T; dTt's zero rows
        float wv[16];
        {
            // -dW^T[d][i] for i in quarter h (this thread's lane d)
            tmem_ld16(taddr(tb, q * 32, cW + 16 * h), wv);
            // D = tril(dO U^T): lanes 64..127 (row i = lane - 64), columns 64 + j
            if (q >= 2) {
                float dd[16];
                tmem_ld16(taddr(tb, q * 32, cR5 + 64 + 16 * h), dd);
                tmem_ld_wait();
                const int i = row - 64;
#pragma unroll
                for (int c8 = 0; c8 < 2; ++c8) {
                    float v8[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int j = 16 * h + 8 * c8 + e;
                        v8[e] = j <= i ? dd[8 * c8 + e] : 0.f;
                    }
                    *reinterpret_cast<uint4*>(sm + kGtD + sw128(i, 16 * h + 8 * c8)) = pack8_f16(v8);
                }
            }
            tmem_ld_wait();
            // dW rows [i][d] (fp16) from dW^T = -(R2): 8x8 tiles through stmatrix.trans
            const int mj = lane >> 3, rho = lane & 7;
            const uint32_t wbase = smem_u32(sm + kGtWK);
#pragma unroll
            for (int lh = 0; lh < 32; lh += 16) {
                uint32_t r[8];
                tmem_ld_16x256b_x2(taddr(tb, q * 32 + lh, cW + 16 * h), r);
                tmem_ld_wait();
                const uint32_t m0 = pack_f16x2(-__uint_as_float(r[0]), -__uint_as_float(r[1]));
                const uint32_t m1 = pack_f16x2(-__uint_as_float(r[2]), -__uint_as_float(r[3]));
                const uint32_t m2 = pack_f16x2(-__uint_as_float(r[4]), -__uint_as_float(r[5]));
                const uint32_t m3 = pack_f16x2(-__uint_as_float(r[6]), -__uint_as_float(r[7]));
                const int i = 16 * h + 8 * (mj >> 1) + rho;
                const int d0 = q * 32 + lh + (mj & 1) * 8;
                stmatrix_x4_trans(wbase + (uint32_t)(d0 >> 6) * 16384u + sw128(i, d0 & 63), m0, m1, m2, m3);
            }
            // rows 64..127 of [dT; 0]
            *reinterpret_cast<uint4*>(sm + kGtdT + 8192 + 16 * tid) = make_uint4(0, 0, 0, 0);
        }
        tc_fence_before();
        __syncthreads();   // every read of the -dW^T columns is done
        tc_fence_after();
        {   // dW^T packed fp16 over its own columns (A operand of R9; even i low)
            uint32_t w[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) w[e] = pack_f16x2(-wv[2 * e], -wv[2 * e + 1]);
            tmem_st8u(taddr(tb, q * 32, cW + 8 * h), w);
        }
        sync_for_mma();
        // ---------------- group 2: R6, R7, R8, R9
        if (tid == 0) {
            tc_fence_after();
            const uint32_t i64 = idesc_f16(128, 64), imk = idesc_f16(128, 64, true, false),
                           imm = idesc_f16(128, 64, true, true), ikm = idesc_f16(128, 64, false, true);
            const uint32_t WK = smem_u32(sm + kGtWK), D0 = smem_u32(sm + kGtD), Q0 = smem_u32(sm + kGtQ),
                           T0 = smem_u32(sm + kGtT);
            for (int s = 0; s < 4; ++s) {
                mma_f16_ss(tb + cQ, sdesc_sw128(WK + 8192 + s * 2048, 16384), sdesc_sw128(D0 + s * 32), imk, 1u);  // R6
                mma_f16_ss(tb + cK, sdesc_sw128(Q0 + s * 2048, 8192), sdesc_sw128(D0 + s * 2048, 8192), imm, 1u); // R7
                mma_f16_ts(tb + cKa, tb + cW + 8 * s, sdesc_sw128(T0 + s * 2048, 8192), ikm, s > 0);            // R9
            }
            for (int s = 0; s < 8; ++s) {   // R8: [dW; K] K^T
                const uint32_t ko = (uint32_t)(s >> 2) * 16384u + (uint32_t)(s & 3) * 32u;
                mma_f16_ss(tb + cR8, sdesc_sw128(WK + ko), sdesc_sw128(WK + 8192 + ko), i64, s > 0);
            }
            mma_commit(bar);
        }
        // meanwhile: dV = alpha dVa (R10 is complete) and <dVa_j, v_j> per lane quadrant
        float nf = 0.f;   // NaN once a non-finite gradient passes this thread
        {
            float va[16], pv[16];
            tmem_ld16(taddr(tb, q * 32, cVa + 16 * h), va);
            tmem_ld_wait();
            const int n = row;
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const int j = 16 * h + e;
                const float x = va[e];
                const __half vh = *reinterpret_cast<const __half*>(sm + kGtUV + (uint32_t)(n >> 6) * 16384u + sw128(j, n & 63));
                pv[e] = x * __half2float(vh);
                const float dv = al[j] * x;
                nonfinite_acc(nf, dv);
                st_tile(sm + kGtOU, j * 128 + n, dv, a.out_bf16);
            }
            const float p = xpose_sum16(pv, lane);
            if ((lane & 1) == 0) partV[q * 64 + jc] = p;
            fence_async_smem();
        }
        if (!(ok = mma_done())) break;
        if (tid == 0) {   // dV rows of this chunk: one contiguous block
            const uint32_t es = a.out_bf16 ? 2u : 4u;
            if (dbg_in((char*)a.dv + tok0 * 128 * es, (size_t)nv * 128 * es, a.dv,
                       (size_t)(a.nchunks / a.NC) * a.L * 128 * es, &g_gt_status))
                bulk_s2g((char*)a.dv + tok0 * 128 * es, sm + kGtOU, (uint32_t)nv * 128u * es);
            bulk_commit();
        }
        // ---------------- epilogue 2: dT tile; K K^T to shared memory; <dKa_j, k_j>
        if (q < 2) {   // lanes i = 0..63: dT_im = (dW K^T + dU V^T)_im alpha_m, m < i
            float x8[16], y8[16];
            tmem_ld16(taddr(tb, q * 32, cR8 + 16 * h), x8);
            tmem_ld16(taddr(tb, q * 32, cR5 + 16 * h), y8);
            tmem_ld_wait();
            const int i = row;
#pragma unroll
            for (int c8 = 0; c8 < 2; ++c8) {
                float v8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int m = 16 * h + 8 * c8 + e;
                    v8[e] = m < i ? (x8[8 * c8 + e] + y8[8 * c8 + e]) * al[m] : 0.f;
                }
                *reinterpret_cast<uint4*>(sm + kGtdT + sw128(i, 16 * h + 8 * c8)) = pack8_f16(v8);
            }
        } else {       // lanes 64 + j: row j of K K^T
            float g[16];
            tmem_ld16(taddr(tb, q * 32, cR8 + 16 * h), g);
            tmem_ld_wait();
            const int j = row - 64;
#pragma unroll
            for (int e = 0; e < 16; e += 4)
                *reinterpret_cast<float4*>(Gs + j * kGsLd + 16 * h + e) = make_float4(g[e], g[e + 1], g[e + 2], g[e + 3]);
        }
        {   // <dKa_j, k_j> per lane quadrant (lane = d)
            float ka[16];
            tmem_ld16(taddr(tb, q * 32, cKa + 16 * h), ka);
            tmem_ld_wait();
            const int d = row;
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const int j = 16 * h + e;
                const __half kh =
                    *reinterpret_cast<const __half*>(sm + kGtWK + (uint32_t)(d >> 6) * 16384u + sw128(64 + j, d & 63));
                ka[e] *= __half2float(kh);
            }
            const float p = xpose_sum16(ka, lane);
            if ((lane & 1) == 0) partK[q * 64 + jc] = p;
        }
        sync_for_mma();
        // ---------------- group 3: R11  X = [dT; 0] T^T
        if (tid == 0) {
            tc_fence_after();
            const uint32_t dT0 = smem_u32(sm + kGtdT), T0 = smem_u32(sm + kGtT);
            for (int s = 0; s < 4; ++s)
                mma_f16_ss(tb + cX, sdesc_sw128(dT0 + s * 32), sdesc_sw128(T0 + s * 32), idesc_f16(128, 64), s > 0);
            mma_commit(bar);
        }
        if (!(ok = mma_done())) break;
        if (q < 2) {   // X rows m (strictly lower) -> fp16 tile
            float x[16];
            tmem_ld16(taddr(tb, q * 32, cX + 16 * h), x);
            tmem_ld_wait();
            const int m = row;
#pragma unroll
            for (int c8 = 0; c8 < 2; ++c8) {
                float v8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int j = 16 * h + 8 * c8 + e;
                    v8[e] = j < m ? x[8 * c8 + e] : 0.f;
                }
                *reinterpret_cast<uint4*>(sm + kGtX + sw128(m, 16 * h + 8 * c8)) = pack8_f16(v8);
            }
        }
        sync_for_mma();
        // ---------------- group 4: R12  dA' = [T | 0]^T X
        if (tid == 0) {
            tc_fence_after();
            const uint32_t T0 = smem_u32(sm + kGtT), X0 = smem_u32(sm + kGtX);
            for (int s = 0; s < 4; ++s)
                mma_f16_ss(tb + cA, sdesc_sw128(T0 + s * 2048, 8192), sdesc_sw128(X0 + s * 2048, 8192),
                           idesc_f16(128, 64, true, true), s > 0);
            mma_commit(bar);
        }
        if (!(ok = mma_done())) break;
        // ---------------- epilogue 4: dA, its part of dalpha, dG = alpha dA, then Ms tile
        if (q < 2) {
            float x[16];
            tmem_ld16(taddr(tb, q * 32, cA + 16 * h), x);
            tmem_ld_wait();
            const int i = row;
            float pa = 0.f;
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const int j = 16 * h + e;
                const float dA = j < i ? -x[e] : 0.f;
                pa = fmaf(dA, Gs[i * kGsLd + j], pa);
                dGs[i * 64 + (j ^ (i & 31))] = al[i] * dA;   // swizzled: column reads stay conflict-free
            }
            partA[h * 64 + i] = pa;
        }
        __syncthreads();
        {   // Ms = dG + dG^T (shared memory only: every warp), row i = tid & 63, columns 8 c8 .. + 7
            const int i = tid & 63, c8 = tid >> 6;
            float v8[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const int j = 8 * c8 + e;
                v8[e] = dGs[i * 64 + (j ^ (i & 31))] + dGs[j * 64 + (i ^ (j & 31))];
            }
            *reinterpret_cast<uint4*>(sm + kGtM + sw128(i, 8 * c8)) = pack8_f16(v8);
        }
        sync_for_mma();
        // ---------------- group 5: R13  dK^T += K^T Ms
        if (tid == 0) {
            tc_fence_after();
            const uint32_t WK = smem_u32(sm + kGtWK), M0 = smem_u32(sm + kGtM);
            for (int s = 0; s < 4; ++s)
                mma_f16_ss(tb + cK, sdesc_sw128(WK + 8192 + s * 2048, 16384), sdesc_sw128(M0 + s * 2048, 8192),
                           idesc_f16(128, 64, true, true), 1u);
            mma_commit(bar);
        }
        if (tid < 64) {   // dalpha_j in a fixed order; dbeta; 2 dalpha dalpha/dlambda
            const int j = tid;
            const float dal = partV[j] + partV[64 + j] + partV[128 + j] + partV[192 + j] + partK[j] + partK[64 + j] +
                              partK[128 + j] + partK[192 + j] + partA[j] + partA[64 + j] + partA[128 + j] +
                              partA[192 + j];
            lam[j] = Gs[j * kGsLd + j];
            dl2[j] = 2.f * dal * dalpha_dlambda_of(bet[j], lam[j], a.euler);
            const float db = dal * dalpha_dbeta_of(bet[j], lam[j], a.euler);
            nonfinite_acc(nf, db);
            if (j < nv && dbg_in(a.dbeta + tok0 + j, 4, a.dbeta, (size_t)(a.nchunks / a.NC) * a.L * 4, &g_gt_status))
                a.dbeta[tok0 + j] = db;
        }
        if (!(ok = mma_done())) break;
        // ---------------- final epilogue: dq, dk (lane = d)
        {
            const int d = row;
            float gq[16], gk[16], ka[16];
            tmem_ld16(taddr(tb, q * 32, cQ + 16 * h), gq);
            tmem_ld16(taddr(tb, q * 32, cK + 16 * h), gk);
            tmem_ld16(taddr(tb, q * 32, cKa + 16 * h), ka);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const int j = 16 * h + e;
                const __half kh =
                    *reinterpret_cast<const __half*>(sm + kGtWK + (uint32_t)(d >> 6) * 16384u + sw128(64 + j, d & 63));
                const float dk = fmaf(dl2[j], __half2float(kh), fmaf(al[j], ka[e], gk[e]));
                nonfinite_acc(nf, gq[e]);
                nonfinite_acc(nf, dk);
                st_tile(sm + kGtUV, j * 128 + d, gq[e], a.out_bf16);
                st_tile(sm + kGtR, j * 128 + d, dk, a.out_bf16);
            }
            fence_async_smem();
        }
        // a chunk the fp16 staging could not represent goes to the tf32 kernel
        const bool redo = __syncthreads_or(bad || nf != 0.f);
        if (tid == 0) {   // dQ and dK rows of this chunk
            if (redo) {
                const int i = atomicAdd(a.redo_n, 1);
                if (dbg_in(a.redo + i, 4, a.redo, (size_t)a.nchunks * 4, &g_gt_status)) a.redo[i] = chunk;
            }
            const uint32_t es = a.out_bf16 ? 2u : 4u;
            const size_t ext = (size_t)(a.nchunks / a.NC) * a.L * 128 * es;
            if (dbg_in((char*)a.dq + tok0 * 128 * es, (size_t)nv * 128 * es, a.dq, ext, &g_gt_status))
                bulk_s2g((char*)a.dq + tok0 * 128 * es, sm + kGtUV, (uint32_t)nv * 128u * es);
            if (dbg_in((char*)a.dk + tok0 * 128 * es, (size_t)nv * 128 * es, a.dk, ext, &g_gt_status))
                bulk_s2g((char*)a.dk + tok0 * 128 * es, sm + kGtR, (uint32_t)nv * 128u * es);
            bulk_commit();
        }
        tc_fence_before();
    }
    if (!ok) {   // a wait gave up: record it, and give the MMAs and copies in flight a bounded drain
        if (tid == 0) atomicOr(&g_gt_status, 1u);
        mbar_wait(bar, ph, kWaitLimit);
        mbar_wait(ldb, lph, kWaitLimit);
    }
    if (tid == 0) bulk_wait_all();   // shared sources read and global writes done before exit
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tb, 512);
}

// Exact fp32 copies of the fp16 images of the chunks k_grad_mma recomputes (listed chunks):
// dSc [d][n], dUp [j][n] from the reverse scan's images (sequences it did not mark), and Sc,
// Up in place from the forward's images in the first half of their own fp32 slots
// (sequences with fwd_fp32 clear; the images are copied to shared memory first).
__global__ void __launch_bounds__(256) k_widen(const unsigned char* gimg, const unsigned char* uimg,
                                               const int* redo_n, const int* redo, const int* seq_bad,
                                               const int* fwd_fp32, float* Sc, float* Up, float* dSc, float* dUp,
                                               int NC) {
    extern __shared__ __align__(16) unsigned char wsm[];   // S image (32 KB) and U' image (16 KB)
    griddep_wait();                 // the gradient kernel's list is complete
    griddep_launch_dependents();    // (the tf32 recompute after this waits for it in turn)
    const int n = *redo_n;
    for (int w = blockIdx.x; w < n; w += gridDim.x) {
        const int chunk = redo[w];
        if (fwd_fp32 && !fwd_fp32[chunk / NC]) {   // uniform across the CTA
            const uint4* si = reinterpret_cast<const uint4*>(Sc + (size_t)chunk * 16384);
            const uint4* ui = reinterpret_cast<const uint4*>(Up + (size_t)chunk * 8192);
            for (int e = threadIdx.x; e < 2048; e += 256) reinterpret_cast<uint4*>(wsm)[e] = si[e];
            for (int e = threadIdx.x; e < 1024; e += 256) reinterpret_cast<uint4*>(wsm + 32768)[e] = ui[e];
            __syncthreads();
            for (int e = threadIdx.x; e < 16384; e += 256) {
                const int d = e >> 7, nn = e & 127;
                Sc[(size_t)chunk * 16384 + e] =
                    __half2float(*reinterpret_cast<const __half*>(wsm + (nn >> 6) * 16384 + sw128(d, nn & 63)));
            }
            for (int e = threadIdx.x; e < 8192; e += 256) {
                const int j = e >> 7, nn = e & 127;
                Up[(size_t)chunk * 8192 + e] =
                    __half2float(*reinterpret_cast<const __half*>(wsm + 32768 + (nn >> 6) * 8192 + sw128(j, nn & 63)));
            }
            __syncthreads();   // the buffer is reused by the next listed chunk
        }
        if (seq_bad[chunk / NC]) continue;
        const unsigned char* g = gimg + (size_t)chunk * 32768;
        for (int e = threadIdx.x; e < 16384; e += 256) {
            const int d = e >> 7, n = e & 127;
            const __half x = *reinterpret_cast<const __half*>(g + (n >> 6) * 16384 + sw128(d, n & 63));
            dSc[(size_t)chunk * 16384 + e] = __half2float(x);
        }
        const unsigned char* u = uimg + (size_t)chunk * 16384;
        for (int e = threadIdx.x; e < 8192; e += 256) {
            const int j = e >> 7, n = e & 127;
            const __half x = *reinterpret_cast<const __half*>(u + (n >> 6) * 8192 + sw128(j, n & 63));
            dUp[(size_t)chunk * 8192 + e] = __half2float(x);
        }
    }
}

}  // namespace

bool grad_tc_supported(const Dims& d) {
    return d.tensor && d.in_bf16 && d.dk == 128 && d.dv == 128 && d.C == 64 && d.L > 0;
}

// workspace: the count of chunks to recompute, their indices, and the forward's
// per-sequence record-format words (fwd_fp32)
size_t grad_tc_ws_bytes(const Dims& d) {
    return grad_tc_supported(d)
               ? 256 + align256((size_t)d.BH() * d.NC * sizeof(int)) + align256((size_t)d.BH() * sizeof(int))
               : 0;
}

GtList grad_tc_list(const Dims& d, void* ws) {
    GtList l;
    l.n = (int*)ws;
    l.chunks = (int*)((char*)ws + 256);
    l.fwd_fp32 = (int*)((char*)ws + 256 + align256((size_t)d.BH() * d.NC * sizeof(int)));
    return l;
}

cudaError_t launch_grad_tc(const Dims& d, const void* q, const void* k, const void* v, const void* dO,
                           const float* beta, const float* alpha, const float* T, const float* Sc, const float* dSc,
                           const float* Up, const float* dUp, const RsTcOut& rs, const int* fwd_fp32, void* dq,
                           void* dk, void* dv, float* dbeta, const GtList& redo, cudaStream_t st) {
    const long long nch = d.BH() * d.NC;
    GtArgs ga{(const __nv_bfloat16*)q, (const __nv_bfloat16*)k, (const __nv_bfloat16*)v, (const __nv_bfloat16*)dO,
              beta, alpha, T, Sc, dSc, Up, dUp, dq, dk, dv, dbeta, redo.n, redo.chunks, rs.seq_bad, fwd_fp32,
              rs.gimg, rs.uimg, d.L, d.NC, (int)nch, d.euler, d.out_bf16};
    cudaError_t e = cudaMemsetAsync(redo.n, 0, sizeof(int), st);
    if (e != cudaSuccess) return e;
    if ((e = cudaFuncSetAttribute(k_grad_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGtSmem)) !=
        cudaSuccess)
        return e;
    int dev = 0, nsm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    const int grid = (int)(nch < nsm ? nch : nsm);
    CUtensorMap tm_do, tm_v, tm_k, tm_q;
    if ((e = bf16_rows_map(&tm_do, dO, d)) != cudaSuccess || (e = bf16_rows_map(&tm_v, v, d)) != cudaSuccess ||
        (e = bf16_rows_map(&tm_k, k, d)) != cudaSuccess || (e = bf16_rows_map(&tm_q, q, d)) != cudaSuccess)
        return e;
    k_grad_tc<<<grid, kGtThreads, kGtSmem, st>>>(tm_do, tm_v, tm_k, tm_q, ga);
    prof_mark("efla_chunk_grad_tc", st);
    return cudaGetLastError();
}

cudaError_t launch_widen(const Dims& d, const RsTcOut& rs, const GtList& redo, const int* fwd_fp32, float* Sc,
                         float* Up, float* dSc, float* dUp, cudaStream_t st) {
    const long long nch = d.BH() * d.NC;
    int dev = 0, nsm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const long long grid = nch < nsm ? nch : nsm;
    // a programmatic dependent of the gradient kernel: scheduled during its tail, waiting
    // in the kernel for its completion (an empty list then costs little beyond that wait)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = 49152;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, k_widen, rs.gimg, rs.uimg, (const int*)redo.n, (const int*)redo.chunks,
                           (const int*)rs.seq_bad, fwd_fp32, Sc, Up, dSc, dUp, (int)d.NC);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t gt_status_read_clear(unsigned int* status) {
    unsigned int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(status, g_gt_status, sizeof(unsigned int));
    if (e != cudaSuccess) return e;
    return *status ? cudaMemcpyToSymbol(g_gt_status, &zero, sizeof(unsigned int)) : cudaSuccess;
}

}  // namespace efla

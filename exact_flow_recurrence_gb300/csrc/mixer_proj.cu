// mixer_proj.cu -- the token mixer's input projections on the tcgen05 tensor cores.
//
// The EFLA layer of the language models the pages report on (page es, "Resultados
// Experimentales" item 1: 340M and 1.3B models) maps each token's hidden vector x
// (d_model wide) to one query, key and value per head and one beta per head:
//     q = (x Wq^T) / sqrt(dk),   k = x Wk^T,   v = x Wv^T,   beta = sigmoid(x Wb^T)
// One GEMM does all four: X [M = B L, D] times W^T, W = [Wq; Wk; Wv; Wb] stacked as
// [N = 3 H dk + H, D] (rows = output features, like a linear layer's weight), bf16
// operands, fp32 accumulation in tensor memory.  The epilogue scales q, rounds q, k, v to
// bf16 and stores them straight into the head-major [B, H, L, dk] layout efla_fwd reads;
// beta goes out as fp32 [B, H, L].
//
// Persistent kernel, one CTA per SM, 192 threads:
//   warp 0  one thread issues the TMA loads of X and W tiles (128 x 64 and 256 x 64 bf16,
//           128-byte swizzle) into a 4-stage ring
//   warp 1  one thread issues the MMAs (M = 128, N = 256, K = 16; N = 32 for the tile of
//           beta columns) into one of two tensor-memory accumulators (256 columns each)
//   warps 2-5  epilogue: tensor memory -> registers -> bf16 box in shared memory (the
//           same swizzle) -> TMA tensor store; double-buffered 16 KB boxes
// so the epilogue of one tile overlaps the main loop of the next.  Every wait is bounded;
// on expiry the kernel records EFLA_ERR_TIMEOUT, drains its own copies and MMAs, frees its
// tensor memory and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include "launch.h"
#include "tc_ptx.cuh"

namespace efla {

using namespace tc;

namespace {

__device__ unsigned int g_pj_status = 0;   // bit 0: a bounded wait expired

constexpr uint32_t kPjWaitLimit = 1u << 24;
constexpr int kPjThreads = 192;
constexpr int kPjStages = 4;
constexpr uint32_t kPjA = 128 * 64 * 2;                 // X tile
constexpr uint32_t kPjStageBytes = kPjA + 256 * 64 * 2; // + W tile
constexpr uint32_t kPjStg = kPjStages * kPjStageBytes;  // two 16 KB output boxes
constexpr uint32_t kPjBar = kPjStg + 2 * 16384;
constexpr size_t kPjSmem = 1024 + kPjBar + 128;
static_assert(kPjSmem <= 232448, "shared memory per CTA");

struct ProjArgs {
    float* beta;     // [B][H][L] fp32
    int K;           // d_model
    int L, H;
    int mt;          // token tiles (M / 128)
    int nt_qkv;      // 256-column tiles over q, k, v (3 H 128 / 256)
    int nt;          // nt_qkv + 1 (the beta columns)
    float qscale;    // 1 / sqrt(dk)
};

__device__ __forceinline__ void pj_group_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Named barrier 1 of the 128 epilogue threads that also ANDs a predicate across them, so
// that every epilogue thread takes the same branch after a wait one of them made.
__device__ __forceinline__ bool pj_group_and(bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.b32 p, %1, 0;\n\t"
        "bar.red.and.pred q, 1, 128, p;\n\t"
        "selp.b32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

__global__ void __launch_bounds__(kPjThreads, 1)
    k_mixer_proj(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                 const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                 const __grid_constant__ CUtensorMap tmV, ProjArgs a) {
    extern __shared__ __align__(1024) unsigned char sm_raw[];
    unsigned char* sm = (unsigned char*)(((uintptr_t)sm_raw + 1023) & ~(uintptr_t)1023);
    uint64_t* full = (uint64_t*)(sm + kPjBar);   // [4] stage loaded
    uint64_t* empty = full + 4;                  // [4] stage consumed by the MMAs
    uint64_t* accf = full + 8;                   // [2] accumulator complete
    uint64_t* acce = full + 10;                  // [2] accumulator read out
    uint64_t* drain = full + 12;
    uint32_t* slot = (uint32_t*)(full + 13);
    volatile int* s_abort = (volatile int*)(slot + 1);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int i = 0; i < 4; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&accf[i], 1);
            mbar_init(&acce[i], 128);
        }
        mbar_init(drain, 1);
        *s_abort = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(slot, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = *slot;
    const int ntiles = a.mt * a.nt, KB = a.K / 64;

    auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
        if (mbar_try_wait(bar, parity)) return true;
        if (*s_abort) return false;
        if (mbar_wait(bar, parity, kPjWaitLimit)) return true;
        *s_abort = 1;
        return false;
    };

    if (warp == 0 && lane == 0) {
        // ============================ producer: TMA loads ============================
        uint32_t it = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x) {
            const int mt = t / a.nt, nt = t - mt * a.nt;
            for (int kb = 0; kb < KB; ++kb, ++it) {
                const int s = it % kPjStages;
                const uint32_t ph = (it / kPjStages) & 1;
                if (!wait(&empty[s], ph ^ 1)) {
                    ok = false;
                    break;
                }
                mbar_arrive_expect_tx(&full[s], kPjStageBytes);
                tma_load_2d(sm + s * kPjStageBytes, &tmX, kb * 64, mt * 128, &full[s]);
                tma_load_2d(sm + s * kPjStageBytes + kPjA, &tmW, kb * 64, nt * 256, &full[s]);
            }
        }
        if (*s_abort)   // let this thread's copies land before the CTA leaves
            for (uint32_t i = it > kPjStages ? it - kPjStages : 0; i < it; ++i)
                mbar_wait(&full[i % kPjStages], (i / kPjStages) & 1, kPjWaitLimit);
    } else if (warp == 1 && lane == 0) {
        // ============================ MMA issue ============================
        const uint32_t id_full = idesc_f16(128, 256, false, false, true);
        const uint32_t id_beta = idesc_f16(128, 32, false, false, true);
        uint32_t it = 0;
        int j = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < ntiles && ok; t += gridDim.x, ++j) {
            const int nt = t % a.nt, acc = j & 1;
            if (!wait(&acce[acc], ((j >> 1) & 1) ^ 1)) break;
            tc_fence_after();
            const uint32_t d = tb + acc * 256;
            const uint32_t idesc = nt < a.nt_qkv ? id_full : id_beta;
            for (int kb = 0; kb < KB; ++kb, ++it) {
                const int s = it % kPjStages;
                if (!wait(&full[s], (it / kPjStages) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t A = smem_u32(sm + s * kPjStageBytes), B = A + kPjA;
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma_f16_ss(d, sdesc_sw128(A + k * 32), sdesc_sw128(B + k * 32), idesc, (kb | k) != 0);
                mma_commit(&empty[s]);
            }
            if (ok) mma_commit(&accf[acc]);
        }
        if (*s_abort) {   // drain: a commit after every MMA this thread issued
            mma_commit(drain);
            mbar_wait(drain, 0, kPjWaitLimit);
        }
    } else if (warp >= 2) {
        // ============================ epilogue ============================
        const int q4 = warp & 3, row = q4 * 32 + lane, et = tid - 64;
        int j = 0, ngrp = 0;
        for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++j) {
            const int mt = t / a.nt, nt = t - mt * a.nt, acc = j & 1;
            // one thread waits; the named barrier hands its outcome to all 128 (a named
            // barrier that some of them left early would never complete)
            if (!pj_group_and(et == 0 ? wait(&accf[acc], (j >> 1) & 1) : true)) break;
            tc_fence_after();
            const int bt = (mt * 128) / a.L, l0 = (mt * 128) % a.L;   // a tile never crosses a sequence
            if (nt < a.nt_qkv) {
                const int col0 = nt * 256, which = col0 / (a.H * 128), h0 = (col0 % (a.H * 128)) / 128;
                const float sc = which == 0 ? a.qscale : 1.f;
                const CUtensorMap* tm = which == 0 ? &tmQ : (which == 1 ? &tmK : &tmV);
                for (int g = 0; g < 4; ++g, ++ngrp) {
                    unsigned char* stg = sm + kPjStg + (ngrp & 1) * 16384;
                    float v[64];
#pragma unroll
                    for (int c0 = 0; c0 < 64; c0 += 16)
                        tmem_ld16(taddr(tb, q4 * 32, acc * 256 + g * 64 + c0), *reinterpret_cast<float(*)[16]>(v + c0));
                    tmem_ld_wait();
                    pj_group_sync();   // this box's previous store has finished reading it
#pragma unroll
                    for (int c8 = 0; c8 < 8; ++c8) {
                        uint4 w;
                        w.x = pack_bf16x2(v[8 * c8 + 0] * sc, v[8 * c8 + 1] * sc);
                        w.y = pack_bf16x2(v[8 * c8 + 2] * sc, v[8 * c8 + 3] * sc);
                        w.z = pack_bf16x2(v[8 * c8 + 4] * sc, v[8 * c8 + 5] * sc);
                        w.w = pack_bf16x2(v[8 * c8 + 6] * sc, v[8 * c8 + 7] * sc);
                        *reinterpret_cast<uint4*>(stg + sw128(row, 8 * c8)) = w;
                    }
                    fence_async_smem();
                    pj_group_sync();
                    if (et == 0) {
                        tma_store_2d(tm, (g & 1) * 64, (bt * a.H + h0 + (g >> 1)) * a.L + l0, stg);
                        bulk_commit();
                        bulk_wait_read_1();   // the other box is free again
                    }
                }
            } else {
                // beta = sigmoid(logit), columns 0 .. H-1 of this tile
                float v[32];
                tmem_ld16(taddr(tb, q4 * 32, acc * 256), *reinterpret_cast<float(*)[16]>(v));
                tmem_ld16(taddr(tb, q4 * 32, acc * 256 + 16), *reinterpret_cast<float(*)[16]>(v + 16));
                tmem_ld_wait();
#pragma unroll
                for (int h = 0; h < 32; ++h)
                    if (h < a.H) a.beta[((size_t)bt * a.H + h) * a.L + l0 + row] = 1.f / (1.f + expf(-v[h]));
            }
            tc_fence_before();
            mbar_arrive(&acce[acc]);
        }
        if (et == 0) bulk_wait_all();
    }

    __syncthreads();
    if (*s_abort && tid == 0) atomicOr(&g_pj_status, 1u);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tb, 512);
}

cudaError_t encode_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t rows, uint32_t box_inner,
                      uint32_t box_rows) {
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    if (!encode) {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess) return e;
        if (q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
        encode = (PFN_cuTensorMapEncodeTiled_v12000)fn;
    }
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {inner * 2};
    const cuuint32_t box[2] = {box_inner, box_rows};
    const cuuint32_t elem[2] = {1, 1};
    const CUresult r = encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                              elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_mixer_proj(int B, int L, int D, int H, const void* x, const void* w, void* q, void* k, void* v,
                              float* beta, cudaStream_t st) {
    const long long M = (long long)B * L;
    const int Nqkv = 3 * H * 128, N = Nqkv + H;
    CUtensorMap tmX, tmW, tmQ, tmK, tmV;
    cudaError_t e = encode_2d(&tmX, x, (uint64_t)D, (uint64_t)M, 64, 128);
    if (e == cudaSuccess) e = encode_2d(&tmW, w, (uint64_t)D, (uint64_t)N, 64, 256);
    if (e == cudaSuccess) e = encode_2d(&tmQ, q, 128, (uint64_t)M * H, 64, 128);
    if (e == cudaSuccess) e = encode_2d(&tmK, k, 128, (uint64_t)M * H, 64, 128);
    if (e == cudaSuccess) e = encode_2d(&tmV, v, 128, (uint64_t)M * H, 64, 128);
    if (e != cudaSuccess) return e;
    ProjArgs a{beta, D, L, H, (int)(M / 128), Nqkv / 256, Nqkv / 256 + 1, 0.08838834764831845f};
    int dev = 0, nsm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaFuncSetAttribute(k_mixer_proj, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPjSmem)) !=
        cudaSuccess)
        return e;
    const long long ntiles = (long long)a.mt * a.nt;
    const int grid = (int)(ntiles < nsm ? ntiles : nsm);
    k_mixer_proj<<<grid, kPjThreads, kPjSmem, st>>>(tmX, tmW, tmQ, tmK, tmV, a);
    prof_mark("efla_mixer_proj", st);
    return cudaGetLastError();
}

cudaError_t proj_status_read_clear(unsigned int* status) {
    unsigned int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(status, g_pj_status, sizeof(unsigned int));
    if (e != cudaSuccess) return e;
    return *status ? cudaMemcpyToSymbol(g_pj_status, &zero, sizeof(unsigned int)) : cudaSuccess;
}

}  // namespace efla

// bwd_tc.cu -- the backward's reverse scan on the tcgen05 tensor cores (bf16 inputs,
// dk = dv = 128, chunk 64).
//
// Reverse-mode differentiation of the chunked update of page es, Metodologia item 3 (the
// pages give no backward pass).  G = dL/dS_{c+1} (the gradient of the state leaving chunk
// c) runs backwards over a sequence's chunks:
//     dSc[c] = G;   dU' = P^T dO + K G;   G <- G + Q^T dO - W^T dU'      (G = dS_final first)
// and dS0 = G after chunk 0; P = tril(Q K^T), W = Ta K.  Evaluated transposed, so that
// every MMA has M = 128 (value rows n of G^T):
//     dU'^T  = dO^T P + G^T K^T          (M = 128, N = 64: 4 + 8 k-steps)
//     G^T   += dO^T Q + (-dU'^T) W       (M = 128, N = 128: 4 + 4 k-steps)
// G^T accumulates in tensor memory (fp32) for the whole sequence; its fp16 copy and the
// packed -dU'^T are tensor-memory A operands, as the state and U' are in the forward
// (fwd_tc.cu), whose structure this kernel mirrors: the Ta and P^T images come from the
// same chunk preparation (tc_common.cuh), here in reverse chunk order.
//
// Outputs: dS0, and per chunk dSc = G and dU' as fp16 images -- exactly the fp16 operand
// tiles the gradient kernel (grad_tc.cu) stages from them, 128-byte swizzled: dSc rows d,
// dU' rows j, each split in two 64-column n-blocks.  The epilogue warps build them with
// stmatrix from the fp16 copies in tensor memory into the operand slot the previous chunk
// has just freed, and one bulk copy per image writes them out, off the chain.
//
// Precision and range: the operands are staged in fp16 with fp32 accumulation, like the
// forward's.  A sequence outside the staging's range (the forward's key and query norm
// bounds, a largest |dO| or |dS_final| element below 2^-10 unless all zero, or a non-finite
// dS0 -- an fp16 overflow of G, dU' or W reaches it) is marked, and the tf32 reverse scan
// (bwd_mma.cu) recomputes exactly those sequences afterwards.
#include "common.cuh"
#include "launch.h"
#include "tc_common.cuh"
#include "tc_ptx.cuh"

namespace efla {

namespace {

__device__ unsigned int g_bt_status = 0;   // bit 0: a bounded wait expired; kStatusBounds (debug builds): a write was skipped

// Shared-memory map, as the forward's: three chunk slots (chunk p in slot p mod 3) of
//   +0      P^T  [64 rows j][64 i]   K-major B of dO^T P (image)
//   +8192   d-block 0: W rows (j), Q rows (i), K rows (j), 64 rows each
//   +32768  d-block 1: the same
// and two dO/Ta buffers (chunk p in buffer p mod 2) of
//   +0      dO   2 n-blocks x [64 rows i]   MN-major A (dO^T) of both products
//   +16384  Ta   [64 rows i][64 j]          K-major B (Ta^T) of W (image)
constexpr uint32_t kSlotBytes = 57344, kSlotPt = 0, kSlotBlk = 8192, kBlkStride = 24576;
constexpr uint32_t kBlkW = 0, kBlkQ = 8192, kBlkK = 16384;
constexpr uint32_t kOffOT = 3 * kSlotBytes, kOTBytes = 24576, kOTO = 0, kOTTa = 16384;
constexpr uint32_t kOffBar = kOffOT + 2 * kOTBytes;
constexpr size_t kBtSmem = 1024 + kOffBar + 256;
static_assert(kBtSmem <= 232448, "shared memory per CTA");
static_assert(4 * kTmGroupBytes + 64 <= kOffBar, "preparation groups fit");

// tensor-memory columns (lane = value row n)
constexpr uint32_t kColA = 0;      // dU'^T [n][j] fp32
constexpr uint32_t kColG = 128;    // G^T [n][d] fp32
constexpr uint32_t kColGh = 256;   // G^T fp16 copy, packed (A operand): column 32 g + i = d pair 64 g + 2i
constexpr uint32_t kColUp = 320;   // -dU'^T packed fp16 (A operand): column 16 g + i = j pair 32 g + 2i
constexpr uint32_t kColW = 384;    // W^T [d][j] fp32
constexpr uint32_t kImgG = 32768, kImgU = 16384;   // image bytes per chunk

__device__ __forceinline__ uint32_t up_col(int s) { return kColUp + 8 * s; }

constexpr int kBtThreads = 20 * 32;
constexpr int kMinPrepCtas = 16;

struct RsTcArgs {
    const __nv_bfloat16* q;
    const __nv_bfloat16* k;
    const __nv_bfloat16* dO;
    const uint16_t* Ta;
    const uint16_t* Pt;
    const float* dS_final;   // [BH][128][128] or null (zero)
    unsigned char* gimg;     // [BH][NC] dSc images, 32 KB each
    unsigned char* uimg;     // [BH][NC] dU' images, 16 KB each
    float* dS0;              // [BH][128][128] or null
    int* flags;              // image-ready flags (fused launch) or null
    int* seq_bad;            // [BH] set for a sequence out of the staging's range
    int* bad_n;              // number of such sequences, listed in bad_list
    int* bad_list;
    TmatArgs prep;
    int L, NC, BH;
};

__global__ void __launch_bounds__(kBtThreads, 1)
    k_rscan_tc(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q, RsTcArgs a) {
    extern __shared__ __align__(1024) unsigned char sm_raw[];
    unsigned char* sm = (unsigned char*)(((uintptr_t)sm_raw + 1023) & ~(uintptr_t)1023);
    if (blockIdx.x >= a.BH) {
        // ======================= preparation CTA (fused launch) =======================
        // As in the forward, in reverse chunk-major order (every sequence's last chunk first).
        const int tid = threadIdx.x, warp = tid >> 5, g = warp >> 2;
        uint32_t* pslot = (uint32_t*)(sm + 4 * kTmGroupBytes);
        unsigned char* gsm = sm + g * kTmGroupBytes;
        uint64_t* gbar = (uint64_t*)(gsm + kTmBar);
        if (warp < 16 && (tid & 127) == 0) {
            mbar_init(&gbar[0], 1);
            mbar_init(&gbar[1], 1);
            fence_mbar_init();
        }
        if (warp == 0) {
            tmem_alloc(pslot, 512);
            tmem_relinquish();
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        const uint32_t tbase = *pslot;
        if (warp < 16) {
            const int nworkers = (gridDim.x - a.BH) * 4, total = a.BH * a.NC;
            uint32_t ph = 0;
            for (int w = (blockIdx.x - a.BH) * 4 + g; w < total; w += nworkers, ph ^= 1u) {
                const int pidx = w / a.BH, bhw = w - pidx * a.BH, c = a.NC - 1 - pidx;
                const int wn = w + nworkers, pn = wn / a.BH;   // this group's next chunk
                if (!tmat_chunk(&tm_k, &tm_q, a.prep, gsm, gbar, ph, tbase + 128 * g, 1 + g, tid & 127, bhw, c,
                                a.flags + (size_t)bhw * a.NC + c, &g_bt_status, wn < total ? wn - pn * a.BH : -1,
                                a.NC - 1 - pn))
                    break;
            }
        }
        tc_fence_before();
        __syncthreads();
        if (warp == 0) tmem_dealloc(tbase, 512);
        return;
    }
    uint64_t* bars = (uint64_t*)(sm + kOffBar);
    uint64_t* ops_full = bars + 0;      // [3] slot and dO/Ta buffer of chunk p loaded
    uint64_t* ops_empty = bars + 3;     // [3] slot free (after the second product of its chunk)
    uint64_t* ot_free = bars + 6;       // [2] dO/Ta buffer free
    uint64_t* m_w = bars + 8;           // W^T of chunk p complete
    uint64_t* m_a = bars + 9;           // dU'^T complete
    uint64_t* m_b = bars + 10;          // G^T update complete
    uint64_t* rdy_a = bars + 11;        // E1: G^T copy written -> first product
    uint64_t* rdy_b = bars + 12;        // E1: -dU'^T packed and the W rows written -> second product
    uint64_t* st_free = bars + 13;      // [3] slot's image staging read out (E2 may refill it)
    uint32_t* slot = (uint32_t*)(bars + 16);
    volatile int* s_abort = (volatile int*)(slot + 1);
    // [0] bit 0 = non-finite dS0; [1], [2] largest ||k||^2, ||q||^2; [3] largest |dO| or
    // |dS_final| element (fp32 bit patterns, >= 0)
    unsigned* s_stat = slot + 2;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int q4 = warp & 3, row = q4 * 32 + lane;
    const long long bh = blockIdx.x;
    const int L = a.L, NC = a.NC;
    const size_t seq_tok = (size_t)bh * L;

    if (tid == 0) {
        for (int i = 0; i < 3; ++i) {
            mbar_init(&ops_full[i], 257);
            mbar_init(&ops_empty[i], 1);
        }
        mbar_init(&ot_free[0], 1);
        mbar_init(&ot_free[1], 1);
        mbar_init(m_w, 1);
        mbar_init(m_a, 1);
        mbar_init(m_b, 1);
        mbar_init(rdy_a, 256);
        mbar_init(rdy_b, 256);
        for (int i = 0; i < 3; ++i) mbar_init(&st_free[i], 1);
        *s_abort = 0;
        s_stat[0] = s_stat[1] = s_stat[2] = s_stat[3] = 0u;
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

    auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
        if (mbar_try_wait(bar, parity)) return true;
        if (*s_abort) return false;
        if (mbar_wait(bar, parity, kWaitLimit)) return true;
        *s_abort = 1;
        return false;
    };

    if (warp >= 1 && warp <= 8) {
        // ============================ E1: dU', G copy, W rows ============================
        const int grp = (warp - 1) >> 2;
        const int mj = lane >> 3, rho = lane & 7;
        float gmax = 0.f;    // largest |dS_final| element this thread loaded
        float nfacc = 0.f;   // NaN once a non-finite dS0 element passed this thread
        auto pack16 = [](const float* v, uint32_t (&w)[16]) {
#pragma unroll
            for (int i = 0; i < 16; ++i) w[i] = pack_f16x2(v[2 * i], v[2 * i + 1]);
        };
        // W rows of the chunk processed p-th, from W^T in tensor memory (as in the forward)
        auto w_rows = [&](int p) -> bool {
            if (!wait(m_w, p & 1)) return false;
            tc_fence_after();
            const uint32_t wbase = smem_u32(sm + (p % 3) * kSlotBytes + kSlotBlk + kBlkW);
#pragma unroll
            for (int lh = 0; lh < 32; lh += 16) {
                uint32_t r[2][8];
#pragma unroll
                for (int h = 0; h < 2; ++h) tmem_ld_16x256b_x2(taddr(tb, q4 * 32 + lh, kColW + grp * 32 + 16 * h), r[h]);
                tmem_ld_wait();
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int cb = grp * 32 + 16 * h;
                    const uint32_t m0 = pack_f16x2(__uint_as_float(r[h][0]), __uint_as_float(r[h][1]));
                    const uint32_t m1 = pack_f16x2(__uint_as_float(r[h][2]), __uint_as_float(r[h][3]));
                    const uint32_t m2 = pack_f16x2(__uint_as_float(r[h][4]), __uint_as_float(r[h][5]));
                    const uint32_t m3t = pack_f16x2(__uint_as_float(r[h][6]), __uint_as_float(r[h][7]));
                    const int i = cb + 8 * (mj >> 1) + rho;
                    const int d0 = q4 * 32 + lh + (mj & 1) * 8;
                    stmatrix_x4_trans(wbase + (d0 >> 6) * kBlkStride + sw128(i, d0 & 63), m0, m1, m2, m3t);
                }
            }
            fence_async_smem();
            return true;
        };
        // The fp16 images of chunk p's dSc (the G copy MMA1(p) read) and dU' (the packed
        // -dU'^T, sign restored) into the d-blocks of slot (p + 2) mod 3, free since the
        // previous chunk's second product: 16x256b tensor-memory loads give each thread
        // two packed columns of 8-lane rows, i.e. 8x8 fp16 tiles whose transposed rows
        // (one d or j, 8 consecutive n) are the images' 16-byte units.  Packed column P of
        // a group's 16-column block k holds the pair 2P, 2P + 1, so tile columns c map to
        // 16k + 4(c / 2) + (c % 2) (+ 2 for the odd packed columns).
        auto images = [&](int p) {
            const uint32_t base = smem_u32(sm + ((p + 2) % 3) * kSlotBytes + kSlotBlk);
            const int off = 4 * (rho >> 1) + (rho & 1) + 2 * (mj & 1);
#pragma unroll
            for (int lh = 0; lh < 32; lh += 16) {
                const int n0 = q4 * 32 + lh + 8 * (mj >> 1);
                const uint32_t nb = (uint32_t)(n0 >> 6);
                uint32_t r[16];
                tmem_ld_16x256b_x4(taddr(tb, q4 * 32 + lh, kColGh + grp * 32), r);
                uint32_t u[8];
                tmem_ld_16x256b_x2(taddr(tb, q4 * 32 + lh, kColUp + grp * 16), u);
                tmem_ld_wait();
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    stmatrix_x4_trans(base + nb * 16384u + sw128(grp * 64 + 16 * k + off, n0 & 63), r[4 * k],
                                      r[4 * k + 1], r[4 * k + 2], r[4 * k + 3]);
#pragma unroll
                for (int k = 0; k < 2; ++k)
                    stmatrix_x4_trans(base + kImgG + nb * 8192u + sw128(grp * 32 + 16 * k + off, n0 & 63),
                                      u[4 * k] ^ 0x80008000u, u[4 * k + 1] ^ 0x80008000u, u[4 * k + 2] ^ 0x80008000u,
                                      u[4 * k + 3] ^ 0x80008000u);
            }
            fence_async_smem();
        };
        const int db = grp * 64;
        // G^T[n][d] = dS_final[d][n] (fp32) and its fp16 copy, dSc of the last chunk (in
        // halves of 32 columns: fewer live registers)
        for (int h = 0; h < 2; ++h) {
            const int d0 = db + 32 * h;
            float v[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                v[i] = a.dS_final ? a.dS_final[((size_t)bh * 128 + d0 + i) * 128 + row] : 0.f;
                gmax = fmaxf(gmax, fabsf(v[i]));
            }
            tmem_st16(taddr(tb, q4 * 32, kColG + d0), *reinterpret_cast<float(*)[16]>(v));
            tmem_st16(taddr(tb, q4 * 32, kColG + d0 + 16), *reinterpret_cast<float(*)[16]>(v + 16));
            uint32_t w[16];
            pack16(v, w);
            tmem_st16u(taddr(tb, q4 * 32, kColGh + grp * 32 + 16 * h), w);
        }
        tmem_st_wait();
        if (w_rows(0)) {
            tc_fence_before();
            mbar_arrive(rdy_a);
        }
        for (int p = 0; p < NC; ++p) {
            const int c = NC - 1 - p;
            const uint32_t par = p & 1;
            // ---- dU'^T[n][j] for tokens j of half grp: to global (fp32), -dU'^T packed
            if (!wait(m_a, par)) break;
            tc_fence_after();
            {
                const int cbeg = grp * 32;
                float u[32];
                tmem_ld16(taddr(tb, q4 * 32, kColA + cbeg), *reinterpret_cast<float(*)[16]>(u));
                tmem_ld16(taddr(tb, q4 * 32, kColA + cbeg + 16), *reinterpret_cast<float(*)[16]>(u + 16));
                tmem_ld_wait();
                uint32_t w[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) w[i] = pack_f16x2(-u[2 * i], -u[2 * i + 1]);
                tmem_st16u(taddr(tb, q4 * 32, kColUp + grp * 16), w);
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(rdy_b);
            }
            // ---- chunk c's dSc and dU' images, written out by one bulk copy each (off the chain)
            images(p);
            group_sync(6, 256);
            if (tid == 32) {
                const uint32_t sb = (uint32_t)((p + 2) % 3) * kSlotBytes + kSlotBlk;
                const size_t ch = (size_t)bh * NC + c, nch = (size_t)a.BH * NC;
                if (dbg_in(a.gimg + ch * kImgG, kImgG, a.gimg, nch * kImgG, &g_bt_status))
                    bulk_s2g(a.gimg + ch * kImgG, sm + sb, kImgG);
                if (dbg_in(a.uimg + ch * kImgU, kImgU, a.uimg, nch * kImgU, &g_bt_status))
                    bulk_s2g(a.uimg + ch * kImgU, sm + sb + kImgG, kImgU);
                bulk_commit();
            }
            // ---- G^T -> fp16 copy (next chunk's first product); G is dSc of chunk c - 1
            if (!wait(m_b, par)) break;
            tc_fence_after();
            float v[64];
#pragma unroll
            for (int c0 = 0; c0 < 64; c0 += 16)
                tmem_ld16(taddr(tb, q4 * 32, kColG + db + c0), *reinterpret_cast<float(*)[16]>(v + c0));
            tmem_ld_wait();
            if (p + 1 < NC) {
                uint32_t w[16];
                pack16(v, w);
                tmem_st16u(taddr(tb, q4 * 32, kColGh + grp * 32), w);
                pack16(v + 32, w);
                tmem_st16u(taddr(tb, q4 * 32, kColGh + grp * 32 + 16), w);
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(rdy_a);
            } else {   // G after chunk 0 = dS0
#pragma unroll
                for (int i = 0; i < 64; ++i) nonfinite_acc(nfacc, v[i]);
                if (a.dS0 && dbg_in(a.dS0 + (size_t)bh * 16384, 65536, a.dS0, (size_t)a.BH * 65536, &g_bt_status)) {
                    float* d0 = a.dS0 + (size_t)bh * 16384 + (size_t)db * 128 + row;
#pragma unroll
                    for (int i = 0; i < 64; ++i) d0[i * 128] = v[i];
                }
            }
            if (tid == 32) {   // this chunk's images have left shared memory: E2 may refill the slot
                bulk_wait_read();
                mbar_arrive(&st_free[(p + 2) % 3]);
            }
            // ---- W rows of the next chunk while its first product runs (they are read by its
            // second product, which waits for this thread's next rdy_b arrival)
            if (p + 1 < NC && !w_rows(p + 1)) break;
        }
        // ---- the staging checks (E2's |dO| maximum and B's norms arrive on barrier 5)
        const bool ran = !*s_abort;
        if (__any_sync(0xffffffffu, nfacc != 0.f) && lane == 0) atomicOr(&s_stat[0], 1u);
        const unsigned wmax = __reduce_max_sync(0xffffffffu, __float_as_uint(gmax));
        if (lane == 0) atomicMax(&s_stat[3], wmax);
        group_sync(5, 544);
        if (ran && tid == 32 &&
            ((s_stat[0] & 1u) || staging_out_of_range(__uint_as_float(s_stat[1]), __uint_as_float(s_stat[2]),
                                                      __uint_as_float(s_stat[3])))) {
            a.seq_bad[bh] = 1;
            a.bad_list[atomicAdd(a.bad_n, 1)] = (int)bh;
        }
    } else if (warp >= 9 && warp <= 18 && (warp & 3) != 0) {
        // ============================ E2: operands ============================
        // K, Q rows of the chunk into its slot and dO rows into its dO/Ta buffer, fp16,
        // as the forward converts K, Q and V.
        const int w9 = warp - 9, et = (w9 - (w9 >> 2)) * 32 + lane;
        const int cch = et & 15, rs = et >> 4;
        const uint32_t pos = (uint32_t)((((cch & 7) ^ (rs & 7)) << 4) + rs * 128);
        const uint32_t dblk = kSlotBlk + (cch >> 3) * kBlkStride + pos;
        const uint32_t dK = dblk + kBlkK, dQ = dblk + kBlkQ;
        const uint32_t dOo = kOTO + (cch >> 3) * 8192u + pos;
        uint4 raw[12];
        float omax = 0.f;   // largest |dO| element this thread converted
        auto load = [&](int p) {
            const int c = NC - 1 - p;
            const int nv = min(64, L - c * 64);
            const size_t tok = seq_tok + (size_t)c * 64 + rs;
#pragma unroll
            for (int which = 0; which < 3; ++which) {
                const __nv_bfloat16* src = which == 0 ? a.k : (which == 1 ? a.q : a.dO);
#pragma unroll
                for (int mm = 0; mm < 4; ++mm)
                    raw[which * 4 + mm] = rs + 16 * mm < nv
                                              ? __ldcs(reinterpret_cast<const uint4*>(src + (tok + 16 * mm) * 128) + cch)
                                              : make_uint4(0, 0, 0, 0);
            }
        };
        auto store = [&](int p) {
            const uint32_t sb = (uint32_t)(p % 3) * kSlotBytes, ob = kOffOT + (uint32_t)(p & 1) * kOTBytes;
#pragma unroll
            for (int which = 0; which < 3; ++which)
#pragma unroll
                for (int mm = 0; mm < 4; ++mm) {
                    const uint32_t dst = (which == 0 ? sb + dK : (which == 1 ? sb + dQ : ob + dOo)) + mm * 2048;
                    *reinterpret_cast<uint4*>(sm + dst) =
                        which == 2 ? bf16x8_to_f16x8_max(raw[which * 4 + mm], omax) : bf16x8_to_f16x8(raw[which * 4 + mm]);
                }
            fence_async_smem();
            mbar_arrive(&ops_full[p % 3]);
        };
        load(0);
        for (int p = 0; p < NC; ++p) {
            // slot p mod 3 is free once the images staged there after chunk p-2's first
            // product are read out (that implies chunk p-3's second product is done); the
            // dO/Ta buffer p mod 2 once chunk p-2's second product is
            if (p >= 2 && !wait(&st_free[p % 3], ((p - 2) / 3) & 1)) break;
            if (p >= 2 && !wait(&ot_free[p & 1], ((p - 2) >> 1) & 1)) break;
            store(p);
            if (p + 1 < NC) load(p + 1);
        }
        {
            const unsigned wm = __reduce_max_sync(0xffffffffu, __float_as_uint(omax));
            if (lane == 0) atomicMax(&s_stat[3], wm);
        }
        asm volatile("bar.arrive 5, 544;" ::: "memory");
    } else if (warp == 19) {
        // ============================ B: image copies ============================
        if (lane == 0) {
            for (int p = 0; p < NC; ++p) {
                const int c = NC - 1 - p, si = p % 3;
                if (p >= 3 && !wait(&ops_empty[si], ((p - 3) / 3) & 1)) break;
                if (p >= 2 && !wait(&ot_free[p & 1], ((p - 2) >> 1) & 1)) break;
                if (a.flags) {   // fused launch: wait (bounded) until the chunk's images are published
                    const int* f = a.flags + (size_t)bh * NC + c;
                    uint32_t n = 0;
                    while (ld_acquire_gpu(f) == 0 && ++n < kFlagPollLimit && !*s_abort) __nanosleep(64);
                    if (n >= kFlagPollLimit || *s_abort) {
                        *s_abort = 1;
                        break;
                    }
                    fence_proxy_async_global();
                }
                mbar_arrive_expect_tx(&ops_full[si], 16384u);
                bulk_g2s(sm + kOffOT + (p & 1) * kOTBytes + kOTTa, a.Ta + ((size_t)bh * NC + c) * 4096, 8192u,
                         &ops_full[si]);
                bulk_g2s(sm + si * kSlotBytes + kSlotPt, a.Pt + ((size_t)bh * NC + c) * 4096, 8192u, &ops_full[si]);
            }
        }
        __syncwarp();
        if (!*s_abort) {   // the chunks' largest key and query norms (every flag acquired)
            float mk2 = 0.f, mq2 = 0.f;
            for (int c = lane; c < NC; c += 32) {
                const float2 nq = *reinterpret_cast<const float2*>(a.prep.cnorm + ((size_t)bh * NC + c) * 2);
                mk2 = fmaxf(mk2, nq.x);
                mq2 = fmaxf(mq2, nq.y);
            }
            const unsigned k2 = __reduce_max_sync(0xffffffffu, __float_as_uint(mk2));
            const unsigned q2 = __reduce_max_sync(0xffffffffu, __float_as_uint(mq2));
            if (lane == 0) {
                s_stat[1] = k2;
                s_stat[2] = q2;
            }
        }
        asm volatile("bar.arrive 5, 544;" ::: "memory");
    } else if (warp == 0 && lane == 0) {
        // ============================ M: MMA issue ============================
        const uint32_t id_mk64 = idesc_f16(128, 64, true, false);    // A MN-major, B K-major, N = 64
        const uint32_t id_kk64 = idesc_f16(128, 64);                 // both K-major (A from TMEM), N = 64
        const uint32_t id_mm128 = idesc_f16(128, 128, true, true);   // A MN-major, B MN-major, N = 128
        const uint32_t id_km128 = idesc_f16(128, 128, false, true);  // A from TMEM, B MN-major, N = 128
        auto slot_at = [&](int p) { return smem_u32(sm + (p % 3) * kSlotBytes); };
        auto ot_at = [&](int p) { return smem_u32(sm + kOffOT + (p & 1) * kOTBytes); };
        auto mma_w = [&](int p) {   // W^T = K^T Ta^T
            const uint32_t s0 = slot_at(p), ta = ot_at(p) + kOTTa;
            for (int s = 0; s < 4; ++s)
                mma_f16_ss(tb + kColW, sdesc_sw128(s0 + kSlotBlk + kBlkK + s * 2048, kBlkStride),
                           sdesc_sw128(ta + s * 32), id_mk64, s > 0);
            mma_commit(m_w);
        };
        if (wait(&ops_full[0], 0)) {
            tc_fence_after();
            mma_w(0);
        }
        for (int p = 0; p < NC; ++p) {
            const uint32_t s0 = slot_at(p), ob = ot_at(p) + kOTO;
            // dU'^T = dO^T P + G^T K^T   (after E1 made the G copy and the W rows)
            if (!wait(rdy_a, p & 1)) break;
            tc_fence_after();
            for (int s = 0; s < 4; ++s)
                mma_f16_ss(tb + kColA, sdesc_sw128(ob + s * 2048, 8192), sdesc_sw128(s0 + kSlotPt + s * 32), id_mk64,
                           s > 0);
            for (int s = 0; s < 8; ++s)
                mma_f16_ts(tb + kColA, tb + kColGh + 8 * s,
                           sdesc_sw128(s0 + kSlotBlk + (s / 4) * kBlkStride + kBlkK + (s % 4) * 32), id_kk64, 1u);
            mma_commit(m_a);
            // this chunk's dO^T Q fills the tensor pipe while E1 works
            for (int s = 0; s < 4; ++s)
                mma_f16_ss(tb + kColG, sdesc_sw128(ob + s * 2048, 8192),
                           sdesc_sw128(s0 + kSlotBlk + kBlkQ + s * 2048, kBlkStride), id_mm128, 1u);
            // G^T += (-dU'^T) W
            if (!wait(rdy_b, p & 1)) break;
            tc_fence_after();
            for (int s = 0; s < 4; ++s)
                mma_f16_ts(tb + kColG, tb + up_col(s), sdesc_sw128(s0 + kSlotBlk + kBlkW + s * 2048, kBlkStride),
                           id_km128, 1u);
            mma_commit(m_b);
            mma_commit(&ops_empty[p % 3]);
            mma_commit(&ot_free[p & 1]);
            // the next chunk's W, while E1 copies G (its W rows are read out during MMA1(p+1),
            // and W(p+2) is issued only after E1's rdy_b(p+1), i.e. after that read)
            if (p + 1 < NC) {
                if (!wait(&ops_full[(p + 1) % 3], ((p + 1) / 3) & 1)) break;
                tc_fence_after();
                mma_w(p + 1);
            }
        }
    }

    // ---- teardown: every thread arrives here (the image copies complete first)
    if (tid == 32) bulk_wait_all();
    __syncthreads();
    if (*s_abort) {
        if (tid == 0) atomicOr(&g_bt_status, 1u);
        if (warp == 0 && lane == 0) mma_commit(m_b);   // after every issued MMA
        __syncthreads();
        mbar_wait(m_b, 0, kWaitLimit);   // either parity completing ends the drain
        mbar_wait(m_b, 1, kWaitLimit);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tb, 512);
}

}  // namespace

bool rscan_tc_supported(const Dims& d) {
    return d.tensor && d.in_bf16 && d.dk == 128 && d.dv == 128 && d.C == 64 && d.L > 0;
}

// workspace: Ta and P^T images | flags | chunk norms | marked sequences [BH] | their count |
// their list [BH] | dSc images | dU' images
size_t rscan_tc_ws_bytes(const Dims& d) {
    if (!rscan_tc_supported(d)) return 0;
    const size_t nch = (size_t)d.BH() * d.NC;
    return align256(nch * 4096 * 2 * 2) + align256(nch * 4) + align256(nch * 8) + 2 * align256((size_t)d.BH() * 4) +
           256 + align256(nch * kImgG) + align256(nch * kImgU);
}

RsTcOut rscan_tc_outputs(const Dims& d, void* ws) {
    const size_t nch = (size_t)d.BH() * d.NC;
    char* p = (char*)ws + align256(nch * 4096 * 2 * 2) + align256(nch * 4) + align256(nch * 8);
    RsTcOut o;
    o.seq_bad = (int*)p;
    p += align256((size_t)d.BH() * 4);
    o.bad_n = (int*)p;
    o.bad_list = (int*)(p + 256);
    o.gimg = (unsigned char*)(p + 256 + align256((size_t)d.BH() * 4));
    o.uimg = o.gimg + align256(nch * kImgG);
    return o;
}

cudaError_t launch_rscan_tc(const Dims& d, const void* q, const void* k, const void* dO, const float* beta,
                            const float* dS_final, float* dS0, void* ws, cudaStream_t st, bool prepared) {
    CUtensorMap tm_k, tm_q;
    cudaError_t e = bf16_rows_map(&tm_k, k, d);
    if (e == cudaSuccess) e = bf16_rows_map(&tm_q, q, d);
    if (e != cudaSuccess) return e;
    const size_t nch = (size_t)d.BH() * d.NC;
    uint16_t* Ta = (uint16_t*)ws;
    uint16_t* Pt = Ta + nch * 4096;
    char* p = (char*)ws + align256(nch * 4096 * 2 * 2);
    int* flags = (int*)p;
    float* cnorm = (float*)(p + align256(nch * 4));
    const RsTcOut out = rscan_tc_outputs(d, ws);
    int* bad = out.seq_bad;
    const int BH = (int)d.BH();
    TmatArgs ta{(const __nv_bfloat16*)k, (const __nv_bfloat16*)q, beta, Ta, Pt, cnorm, nullptr, nullptr, d.L, d.NC,
                d.euler, d.BH() * d.NC};
    RsTcArgs ra{(const __nv_bfloat16*)q, (const __nv_bfloat16*)k, (const __nv_bfloat16*)dO, Ta, Pt, dS_final,
                out.gimg, out.uimg, dS0, nullptr, bad, out.bad_n, out.bad_list, ta, d.L, d.NC, BH};
    if ((e = cudaMemsetAsync(bad, 0, (size_t)BH * sizeof(int), st)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(out.bad_n, 0, sizeof(int), st)) != cudaSuccess) return e;
    if ((e = cudaFuncSetAttribute(k_rscan_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kBtSmem)) !=
        cudaSuccess)
        return e;
    int dev = 0, nsm = 0, coop = 0, per_sm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev)) != cudaSuccess) return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_rscan_tc, kBtThreads, kBtSmem)) != cudaSuccess)
        return e;
    const int prep_ctas = nsm * per_sm - BH;
    if (!prepared && coop && prep_ctas >= kMinPrepCtas) {
        ra.flags = flags;
        if ((e = cudaMemsetAsync(flags, 0, nch * sizeof(int), st)) != cudaSuccess) return e;
        void* args[] = {&tm_k, &tm_q, &ra};
        e = cudaLaunchCooperativeKernel((const void*)k_rscan_tc, dim3((unsigned)(BH + prep_ctas)), dim3(kBtThreads),
                                        args, kBtSmem, st);
        prof_mark("efla_state_grad_scan_tc", st);
        return e != cudaSuccess ? e : cudaGetLastError();
    }
    if (!prepared && (e = launch_tmat(d, &tm_k, &tm_q, ta, st)) != cudaSuccess) return e;
    k_rscan_tc<<<(unsigned)BH, kBtThreads, kBtSmem, st>>>(tm_k, tm_q, ra);
    if (!prepared) prof_mark("efla_state_grad_scan_tc", st);
    return cudaGetLastError();
}

cudaError_t bt_status_read_clear(unsigned int* status) {
    unsigned int zero = 0;
    cudaError_t e = cudaMemcpyFromSymbol(status, g_bt_status, sizeof(unsigned int));
    if (e != cudaSuccess) return e;
    return *status ? cudaMemcpyToSymbol(g_bt_status, &zero, sizeof(unsigned int)) : cudaSuccess;
}

}  // namespace efla

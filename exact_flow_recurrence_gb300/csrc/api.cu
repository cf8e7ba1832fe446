// api.cu -- the extern "C" boundary declared in include/efla.h: argument
// validation, workspace sizing, dispatch to the kernels, status reporting.
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>

#include <nvtx3/nvToolsExt.h>

#include "../../include/efla.h"
#include "launch.h"

namespace {
// An NVTX range around an entry point's host-side work (argument checks, launches), for
// timeline tools; with no tool attached the calls do nothing.
struct NvtxRange {
    explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange&) = delete;
    NvtxRange& operator=(const NvtxRange&) = delete;
};
}  // namespace

namespace {

thread_local char g_msg[512] = "";

efla_status fail(efla_status s, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof g_msg, fmt, ap);
    va_end(ap);
    return s;
}

efla_status cuda_fail(cudaError_t e, const char* where) {
    return fail(EFLA_ERR_CUDA, "%s: %s (%s)", where, cudaGetErrorName(e), cudaGetErrorString(e));
}

bool dim_ok(int d) { return d >= 16 && d <= 128 && d % 16 == 0; }
bool dtype_ok(int t) { return t == EFLA_F32 || t == EFLA_BF16; }
size_t esize(efla_dtype t) { return t == EFLA_BF16 ? 2 : 4; }
bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

struct Span {
    const void* p;
    size_t n;
    const char* name;
};

bool overlap(const Span& a, const Span& b) {
    if (!a.p || !b.p || a.n == 0 || b.n == 0) return false;
    const uintptr_t a0 = (uintptr_t)a.p, b0 = (uintptr_t)b.p;
    return a0 < b0 + b.n && b0 < a0 + a.n;
}

// Common shape validation.  needs_chunk: fwd/bwd (chunk in {16,32,64}); step: L == 1.
efla_status check_shape(const efla_shape* s, bool step, efla::Dims* d) {
    if (!s) return fail(EFLA_ERR_INVALID_ARG, "shape is NULL");
    if (s->B < 0 || s->H < 0 || s->L < 0)
        return fail(EFLA_ERR_INVALID_ARG, "negative size (B=%d H=%d L=%d)", s->B, s->H, s->L);
    if (!dim_ok(s->dk) || !dim_ok(s->dv))
        return fail(EFLA_ERR_UNSUPPORTED, "dk=%d dv=%d: need multiples of 16 in [16,128]", s->dk, s->dv);
    if (!dtype_ok(s->dtype) || !dtype_ok(s->out_dtype))
        return fail(EFLA_ERR_UNSUPPORTED, "dtype=%d out_dtype=%d: need EFLA_F32 or EFLA_BF16",
                    (int)s->dtype, (int)s->out_dtype);
    if (s->mode != EFLA_EXACT && s->mode != EFLA_EULER)
        return fail(EFLA_ERR_UNSUPPORTED, "mode=%d: need EFLA_EXACT or EFLA_EULER", (int)s->mode);
    if (s->path != EFLA_PATH_AUTO && s->path != EFLA_PATH_SIMT && s->path != EFLA_PATH_TENSOR)
        return fail(EFLA_ERR_UNSUPPORTED, "path=%d: need EFLA_PATH_AUTO, _SIMT or _TENSOR", (int)s->path);
    const long long bh = (long long)s->B * s->H;
    if (bh > 0x7fffffffLL) return fail(EFLA_ERR_UNSUPPORTED, "B*H=%lld exceeds 2^31-1", bh);
    int C = 1;
    if (step) {
        if (s->L != 1) return fail(EFLA_ERR_INVALID_ARG, "efla_step needs L == 1 (got %d)", s->L);
    } else {
        C = s->chunk;
        if (C != 16 && C != 32 && C != 64)
            return fail(EFLA_ERR_UNSUPPORTED, "chunk=%d: need 16, 32 or 64", C);
    }
    const long long NC = ((long long)s->L + C - 1) / C;
    if (!step && NC > 65535)
        return fail(EFLA_ERR_UNSUPPORTED, "L=%d gives %lld chunks (> 65535)", s->L, NC);
    d->B = s->B; d->H = s->H; d->L = s->L; d->dk = s->dk; d->dv = s->dv;
    d->C = C; d->NC = (int)NC;
    d->in_bf16 = s->dtype == EFLA_BF16;
    d->out_bf16 = s->out_dtype == EFLA_BF16;
    d->euler = s->mode == EFLA_EULER;
    d->tensor = 0;
    return EFLA_OK;
}

// Forward path choice (after check_shape).
efla_status pick_fwd_path(const efla_shape* s, efla::Dims* d) {
    const bool ok = efla::fwd_tc_supported(*d);
    if (s->path == EFLA_PATH_TENSOR && !ok && d->L > 0)
        return fail(EFLA_ERR_UNSUPPORTED,
                    "EFLA_PATH_TENSOR needs bf16 inputs, dk = dv = 128 and chunk 64 "
                    "(got dtype=%d dk=%d dv=%d chunk=%d)", (int)s->dtype, s->dk, s->dv, s->chunk);
    d->tensor = ok && s->path != EFLA_PATH_SIMT;
    return EFLA_OK;
}

size_t fwd_ws_for(const efla::Dims& d) {
    return d.tensor ? efla::fwd_tc_ws_bytes(d) : efla::fwd_ws_bytes(d);
}

efla_status check_ptrs(const Span* req, int nreq, const Span* opt, int nopt) {
    for (int i = 0; i < nreq; ++i) {
        if (!req[i].p) return fail(EFLA_ERR_INVALID_ARG, "%s is NULL", req[i].name);
        if (!aligned16(req[i].p)) return fail(EFLA_ERR_ALIGNMENT, "%s is not 16-byte aligned", req[i].name);
    }
    for (int i = 0; i < nopt; ++i)
        if (opt[i].p && !aligned16(opt[i].p))
            return fail(EFLA_ERR_ALIGNMENT, "%s is not 16-byte aligned", opt[i].name);
    return EFLA_OK;
}

// every output must not overlap any input or another output
efla_status check_alias(const Span* outs, int nout, const Span* ins, int nin) {
    for (int i = 0; i < nout; ++i) {
        for (int j = 0; j < nin; ++j)
            if (overlap(outs[i], ins[j]))
                return fail(EFLA_ERR_INVALID_ARG, "%s overlaps input %s", outs[i].name, ins[j].name);
        for (int j = i + 1; j < nout; ++j)
            if (overlap(outs[i], outs[j]))
                return fail(EFLA_ERR_INVALID_ARG, "%s overlaps %s", outs[i].name, outs[j].name);
    }
    return EFLA_OK;
}

}  // namespace

void efla::set_last_error(const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_msg, sizeof g_msg, fmt, ap);
    va_end(ap);
}

extern "C" {

const char* efla_status_string(efla_status s) {
    switch (s) {
        case EFLA_OK: return "EFLA_OK";
        case EFLA_ERR_INVALID_ARG: return "EFLA_ERR_INVALID_ARG";
        case EFLA_ERR_UNSUPPORTED: return "EFLA_ERR_UNSUPPORTED";
        case EFLA_ERR_ALIGNMENT: return "EFLA_ERR_ALIGNMENT";
        case EFLA_ERR_WORKSPACE: return "EFLA_ERR_WORKSPACE";
        case EFLA_ERR_CUDA: return "EFLA_ERR_CUDA";
        case EFLA_ERR_TIMEOUT: return "EFLA_ERR_TIMEOUT";
        case EFLA_ERR_BOUNDS: return "EFLA_ERR_BOUNDS";
    }
    return "EFLA_ERR_UNKNOWN";
}

const char* efla_last_error(void) { return g_msg; }

size_t efla_fwd_workspace_size(const efla_shape* shape) {
    efla::Dims d;
    if (check_shape(shape, false, &d) != EFLA_OK) return 0;
    if (pick_fwd_path(shape, &d) != EFLA_OK) return 0;
    return fwd_ws_for(d);
}

size_t efla_bwd_workspace_size(const efla_shape* shape) {
    efla::Dims d;
    if (check_shape(shape, false, &d) != EFLA_OK) return 0;
    if (shape->path == EFLA_PATH_TENSOR) return 0;
    d.tensor = shape->path != EFLA_PATH_SIMT;
    return efla::bwd_ws_bytes(d);
}

}  // extern "C"

namespace {

// efla_fwd, and efla_fwd_save when `states` is not null.
efla_status fwd_common(const efla_shape* shape, const void* q, const void* k, const void* v,
                       const float* beta, const float* S0, void* o, float* S_final, float* states,
                       size_t states_bytes, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    g_msg[0] = 0;
    efla::Dims d;
    efla_status st = check_shape(shape, false, &d);
    if (st != EFLA_OK) return st;
    if ((st = pick_fwd_path(shape, &d)) != EFLA_OK) return st;
    if (d.BH() == 0) return EFLA_OK;
    const size_t rec_need = efla::states_bytes(d);
    if (states) {
        if (!aligned16(states)) return fail(EFLA_ERR_ALIGNMENT, "states is not 16-byte aligned");
        if (states_bytes < rec_need)
            return fail(EFLA_ERR_INVALID_ARG, "states %zu bytes < required %zu", states_bytes, rec_need);
    }
    const size_t ntok = (size_t)d.BH() * d.L;
    const size_t ein = esize(shape->dtype), eout = esize(shape->out_dtype);
    const size_t sbytes = (size_t)d.BH() * d.dk * d.dv * 4;
    const Span sq{q, ntok * d.dk * ein, "q"}, sk{k, ntok * d.dk * ein, "k"},
        sv{v, ntok * d.dv * ein, "v"}, sb{beta, ntok * 4, "beta"}, sS0{S0, sbytes, "S0"},
        so{o, ntok * d.dv * eout, "o"}, sSf{S_final, sbytes, "S_final"},
        sw{workspace, workspace_bytes, "workspace"};
    if (d.L > 0) {
        const Span req[] = {sq, sk, sv, sb, so};
        const Span opt[] = {sS0, sSf, sw};
        if ((st = check_ptrs(req, 5, opt, 3)) != EFLA_OK) return st;
    } else {
        const Span opt[] = {sS0, sSf};
        if ((st = check_ptrs(nullptr, 0, opt, 2)) != EFLA_OK) return st;
    }
    // S_final may alias S0 exactly; any other overlap is an error
    if (S_final && S0 && S_final != (float*)S0 && overlap(sSf, sS0))
        return fail(EFLA_ERR_INVALID_ARG, "S_final partially overlaps S0");
    {
        const Span outs[] = {so, sSf};
        const Span ins[] = {sq, sk, sv, sb};
        if ((st = check_alias(outs, 2, ins, 4)) != EFLA_OK) return st;
        if (overlap(so, sS0)) return fail(EFLA_ERR_INVALID_ARG, "o overlaps input S0");
        const Span all[] = {sq, sk, sv, sb, sS0, so, sSf};
        for (const Span& x : all)
            if (overlap(sw, x)) return fail(EFLA_ERR_INVALID_ARG, "workspace overlaps %s", x.name);
        const Span srec{states, rec_need, "states"};
        const Span all2[] = {sq, sk, sv, sb, sS0, so, sSf, sw};
        for (const Span& x : all2)
            if (overlap(srec, x)) return fail(EFLA_ERR_INVALID_ARG, "states overlaps %s", x.name);
    }
    if (d.L == 0) {
        if (!S_final || S_final == S0) return EFLA_OK;
        efla::prof_mark(nullptr, stream);
        cudaError_t e = efla::launch_state_copy((long long)d.BH() * d.dk * d.dv, S0, S_final, stream);
        return e == cudaSuccess ? EFLA_OK : cuda_fail(e, "efla_fwd(state copy)");
    }
    const size_t need = fwd_ws_for(d);
    if (!workspace || workspace_bytes < need)
        return fail(EFLA_ERR_WORKSPACE, "workspace %zu bytes < required %zu", workspace_bytes, need);
    efla::prof_mark(nullptr, stream);
    cudaError_t e;
    if (d.tensor) {
        e = efla::launch_fwd_tc(d, q, k, v, beta, S0, o, S_final, workspace, stream, states,
                                states ? efla::states_Up(d, states) : nullptr,
                                states ? efla::states_T(d, states) : nullptr,
                                states ? efla::states_alpha(d, states) : nullptr);
    } else {
        efla::FwdWs ws = efla::fwd_ws_carve(d, workspace);
        if (states) {   // the preparation and the scan write straight into the record
            ws.Sc = states;
            ws.Up = efla::states_Up(d, states);
            ws.T = efla::states_T(d, states);
            ws.alpha = efla::states_alpha(d, states);
        }
        e = efla::launch_fwd_simt(d, q, k, v, beta, S0, o, S_final, ws, stream);
    }
    return e == cudaSuccess ? EFLA_OK : cuda_fail(e, states ? "efla_fwd_save" : "efla_fwd");
}

// efla_bwd, and efla_bwd_saved when `states` is not null (S0 then comes from the record).
efla_status bwd_common(const efla_shape* shape, const void* q, const void* k, const void* v,
                       const float* beta, const float* S0, const float* states, size_t states_bytes,
                       const void* dO, const float* dS_final, void* dq, void* dk, void* dv, float* dbeta,
                       float* dS0, void* workspace, size_t workspace_bytes, cudaStream_t stream);

}  // namespace

extern "C" {

efla_status efla_fwd(const efla_shape* shape, const void* q, const void* k, const void* v,
                     const float* beta, const float* S0, void* o, float* S_final,
                     void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    NvtxRange nvtx_range("efla_fwd");
    return fwd_common(shape, q, k, v, beta, S0, o, S_final, nullptr, 0, workspace, workspace_bytes, stream);
}

efla_status efla_fwd_save(const efla_shape* shape, const void* q, const void* k, const void* v,
                          const float* beta, const float* S0, void* o, float* S_final, float* states,
                          size_t states_bytes, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    NvtxRange nvtx_range("efla_fwd_save");
    return fwd_common(shape, q, k, v, beta, S0, o, S_final, states, states_bytes, workspace, workspace_bytes,
                      stream);
}

size_t efla_fwd_states_size(const efla_shape* shape) {
    efla::Dims d;
    if (check_shape(shape, false, &d) != EFLA_OK) return 0;
    return efla::states_bytes(d);
}

size_t efla_bwd_saved_workspace_size(const efla_shape* shape) {
    efla::Dims d;
    if (check_shape(shape, false, &d) != EFLA_OK) return 0;
    if (shape->path == EFLA_PATH_TENSOR) return 0;
    d.tensor = shape->path != EFLA_PATH_SIMT;
    return efla::bwd_saved_ws_bytes(d);
}

int efla_bwd_plan(const efla_shape* shape, size_t free_bytes) {
    efla::Dims d;
    if (check_shape(shape, false, &d) != EFLA_OK || shape->path == EFLA_PATH_TENSOR) return -1;
    d.tensor = shape->path != EFLA_PATH_SIMT;
    const bool rec_fits = efla::states_bytes(d) + efla::bwd_saved_ws_bytes(d) <= free_bytes;
    const bool bwd_fits = efla::bwd_ws_bytes(d) <= free_bytes;
    if (efla::bwd_runs_recording_forward(d)) {   // efla_bwd is the faster form here
        if (bwd_fits) return 0;
        return rec_fits ? 1 : -1;
    }
    if (rec_fits) return 1;
    return bwd_fits ? 0 : -1;
}

efla_status efla_bwd_saved(const efla_shape* shape, const void* q, const void* k, const void* v,
                           const float* beta, const float* states, size_t states_bytes, const void* dO,
                           const float* dS_final, void* dq, void* dk, void* dv, float* dbeta, float* dS0,
                           void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    NvtxRange nvtx_range("efla_bwd_saved");
    if (!states) {
        g_msg[0] = 0;
        return fail(EFLA_ERR_INVALID_ARG, "efla_bwd_saved: states is NULL");
    }
    return bwd_common(shape, q, k, v, beta, nullptr, states, states_bytes, dO, dS_final, dq, dk, dv, dbeta,
                      dS0, workspace, workspace_bytes, stream);
}

efla_status efla_bwd(const efla_shape* shape, const void* q, const void* k, const void* v,
                     const float* beta, const float* S0, const void* dO, const float* dS_final,
                     void* dq, void* dk, void* dv, float* dbeta, float* dS0,
                     void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    NvtxRange nvtx_range("efla_bwd");
    return bwd_common(shape, q, k, v, beta, S0, nullptr, 0, dO, dS_final, dq, dk, dv, dbeta, dS0, workspace,
                      workspace_bytes, stream);
}

}  // extern "C"

namespace {

efla_status bwd_common(const efla_shape* shape, const void* q, const void* k, const void* v,
                       const float* beta, const float* S0, const float* states, size_t states_bytes,
                       const void* dO, const float* dS_final, void* dq, void* dk, void* dv, float* dbeta,
                       float* dS0, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    g_msg[0] = 0;
    efla::Dims d;
    efla_status st = check_shape(shape, false, &d);
    if (st != EFLA_OK) return st;
    if (shape->path == EFLA_PATH_TENSOR)
        return fail(EFLA_ERR_UNSUPPORTED,
                    "efla_bwd: path must be AUTO (tensor-pipe products where the shape allows) or SIMT");
    d.tensor = shape->path != EFLA_PATH_SIMT;   // allows the tensor-pipe kernels
    if (d.BH() == 0) return EFLA_OK;
    const size_t rec_need = efla::states_bytes(d);
    if (states) {
        if (!aligned16(states)) return fail(EFLA_ERR_ALIGNMENT, "states is not 16-byte aligned");
        if (states_bytes < rec_need)
            return fail(EFLA_ERR_INVALID_ARG, "states %zu bytes < required %zu", states_bytes, rec_need);
    }
    const size_t ntok = (size_t)d.BH() * d.L;
    const size_t ein = esize(shape->dtype), eout = esize(shape->out_dtype);
    const size_t sbytes = (size_t)d.BH() * d.dk * d.dv * 4;
    const Span sq{q, ntok * d.dk * ein, "q"}, sk{k, ntok * d.dk * ein, "k"},
        sv{v, ntok * d.dv * ein, "v"}, sb{beta, ntok * 4, "beta"}, sS0{S0, sbytes, "S0"},
        sdO{dO, ntok * d.dv * ein, "dO"}, sdSf{dS_final, sbytes, "dS_final"},
        sdq{dq, ntok * d.dk * eout, "dq"}, sdk{dk, ntok * d.dk * eout, "dk"},
        sdv{dv, ntok * d.dv * eout, "dv"}, sdb{dbeta, ntok * 4, "dbeta"},
        sdS0{dS0, sbytes, "dS0"}, sw{workspace, workspace_bytes, "workspace"};
    if (d.L > 0) {
        const Span req[] = {sq, sk, sv, sb, sdO, sdq, sdk, sdv, sdb};
        const Span opt[] = {sS0, sdSf, sdS0, sw};
        if ((st = check_ptrs(req, 9, opt, 4)) != EFLA_OK) return st;
    } else {
        const Span opt[] = {sdSf, sdS0};
        if ((st = check_ptrs(nullptr, 0, opt, 2)) != EFLA_OK) return st;
    }
    {
        const Span srec{states, rec_need, "states"};
        const Span outs[] = {sdq, sdk, sdv, sdb, sdS0};
        const Span ins[] = {sq, sk, sv, sb, sS0, sdO, sdSf, srec};
        if ((st = check_alias(outs, 5, ins, 8)) != EFLA_OK) return st;
        const Span all[] = {sq, sk, sv, sb, sS0, sdO, sdSf, sdq, sdk, sdv, sdb, sdS0, srec};
        for (const Span& x : all)
            if (overlap(sw, x)) return fail(EFLA_ERR_INVALID_ARG, "workspace overlaps %s", x.name);
    }
    const char* where = states ? "efla_bwd_saved" : "efla_bwd";
    if (d.L == 0) {
        // no tokens: dS0 = dS_final
        if (!dS0) return EFLA_OK;
        efla::prof_mark(nullptr, stream);
        cudaError_t e = efla::launch_state_copy((long long)d.BH() * d.dk * d.dv, dS_final, dS0, stream);
        return e == cudaSuccess ? EFLA_OK : cuda_fail(e, where);
    }
    const size_t need = states ? efla::bwd_saved_ws_bytes(d) : efla::bwd_ws_bytes(d);
    if (!workspace || workspace_bytes < need)
        return fail(EFLA_ERR_WORKSPACE, "workspace %zu bytes < required %zu", workspace_bytes, need);
    const efla::BwdWs ws = states ? efla::bwd_saved_ws_carve(d, workspace, states) : efla::bwd_ws_carve(d, workspace);
    efla::prof_mark(nullptr, stream);
    cudaError_t e = efla::launch_bwd_simt(d, q, k, v, beta, S0, dO, dS_final, dq, dk, dv, dbeta,
                                          dS0, ws, stream, states != nullptr);
    return e == cudaSuccess ? EFLA_OK : cuda_fail(e, where);
}

}  // namespace

extern "C" {

efla_status efla_step(const efla_shape* shape, const void* q, const void* k, const void* v,
                      const float* beta, float* S, void* o, cudaStream_t stream) {
    NvtxRange nvtx_range("efla_step");
    g_msg[0] = 0;
    efla::Dims d;
    efla_status st = check_shape(shape, true, &d);
    if (st != EFLA_OK) return st;
    if (shape->path == EFLA_PATH_TENSOR)
        return fail(EFLA_ERR_UNSUPPORTED, "efla_step runs on CUDA cores: path must be AUTO or SIMT");
    if (d.BH() == 0) return EFLA_OK;
    const size_t n = (size_t)d.BH();
    const size_t ein = esize(shape->dtype), eout = esize(shape->out_dtype);
    const Span sq{q, n * d.dk * ein, "q"}, sk{k, n * d.dk * ein, "k"}, sv{v, n * d.dv * ein, "v"},
        sb{beta, n * 4, "beta"}, sS{S, n * d.dk * d.dv * 4, "S"}, so{o, n * d.dv * eout, "o"};
    const Span req[] = {sq, sk, sv, sb, sS, so};
    if ((st = check_ptrs(req, 6, nullptr, 0)) != EFLA_OK) return st;
    const Span outs[] = {sS, so};
    const Span ins[] = {sq, sk, sv, sb};
    if ((st = check_alias(outs, 2, ins, 4)) != EFLA_OK) return st;
    efla::prof_mark(nullptr, stream);
    cudaError_t e = efla::launch_step(d, q, k, v, beta, S, o, stream);
    return e == cudaSuccess ? EFLA_OK : cuda_fail(e, "efla_step");
}

efla_status efla_mixer_proj(const efla_mixer_shape* s, const void* x, const void* w, void* q, void* k, void* v,
                            float* beta, cudaStream_t stream) {
    NvtxRange nvtx_range("efla_mixer_proj");
    g_msg[0] = 0;
    if (!s) return fail(EFLA_ERR_INVALID_ARG, "shape is NULL");
    if (s->B < 0 || s->L < 0 || s->D < 0 || s->H < 0)
        return fail(EFLA_ERR_INVALID_ARG, "negative size (B=%d L=%d D=%d H=%d)", s->B, s->L, s->D, s->H);
    if (s->dk != 128 || s->L % 128 || s->D % 64 || s->D < 64 || s->H < 2 || s->H > 32 || s->H % 2)
        return fail(EFLA_ERR_UNSUPPORTED,
                    "efla_mixer_proj needs dk = 128, L % 128 == 0, D % 64 == 0 (D >= 64), even H in [2, 32] "
                    "(got L=%d D=%d H=%d dk=%d)", s->L, s->D, s->H, s->dk);
    const long long M = (long long)s->B * s->L;
    if (M == 0) return EFLA_OK;
    if (M * s->H > 0x7fffffffLL || (long long)s->D * (3 * s->H * 128 + s->H) > 0x7fffffffLL)
        return fail(EFLA_ERR_UNSUPPORTED, "efla_mixer_proj: B L H = %lld rows exceed 2^31-1", M * s->H);
    const size_t nw = (size_t)(3 * s->H * 128 + s->H) * s->D, nqkv = (size_t)M * s->H * 128;
    const Span sx{x, (size_t)M * s->D * 2, "x"}, sw{w, nw * 2, "w"}, sq{q, nqkv * 2, "q"}, sk{k, nqkv * 2, "k"},
        sv{v, nqkv * 2, "v"}, sb{beta, (size_t)M * s->H * 4, "beta"};
    const Span req[] = {sx, sw, sq, sk, sv, sb};
    efla_status st = check_ptrs(req, 6, nullptr, 0);
    if (st != EFLA_OK) return st;
    const Span outs[] = {sq, sk, sv, sb};
    const Span ins[] = {sx, sw};
    if ((st = check_alias(outs, 4, ins, 2)) != EFLA_OK) return st;
    efla::prof_mark(nullptr, stream);
    cudaError_t e = efla::launch_mixer_proj(s->B, s->L, s->D, s->H, x, w, q, k, v, beta, stream);
    return e == cudaSuccess ? EFLA_OK : cuda_fail(e, "efla_mixer_proj");
}

efla_status efla_wait_selftest(int kind, int limit, cudaStream_t stream) {
    g_msg[0] = 0;
    if ((kind != 0 && kind != 1) || limit < 1 || limit > (1 << 20))
        return fail(EFLA_ERR_INVALID_ARG, "efla_wait_selftest: kind 0 or 1, limit 1..2^20 (got %d, %d)",
                    kind, limit);
    efla::prof_mark(nullptr, stream);
    cudaError_t e = efla::launch_wait_selftest(kind, (uint32_t)limit, stream);
    return e == cudaSuccess ? EFLA_OK : cuda_fail(e, "efla_wait_selftest");
}

efla_status efla_get_status(cudaStream_t stream) {
    NvtxRange nvtx_range("efla_get_status");
    g_msg[0] = 0;
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e, "efla_get_status(sync)");
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "efla_get_status");
    unsigned int word = 0, word2 = 0, word3 = 0, word4 = 0, word5 = 0;
    e = efla::tc_status_read_clear(&word);
    if (e == cudaSuccess) e = efla::proj_status_read_clear(&word2);
    if (e == cudaSuccess) e = efla::bt_status_read_clear(&word3);
    if (e == cudaSuccess) e = efla::gt_status_read_clear(&word4);
    if (e == cudaSuccess) e = efla::sd_status_read_clear(&word5);
    if (e != cudaSuccess) return cuda_fail(e, "efla_get_status(status word)");
    word |= word2 | word3 | word4 | word5;
    if (word & efla::kStatusBounds)
        return fail(EFLA_ERR_BOUNDS, "a debug-build bounds check skipped a global write (status 0x%x)", word);
    if (word) return fail(EFLA_ERR_TIMEOUT, "a bounded device-side wait expired (status 0x%x)", word);
    return EFLA_OK;
}

efla_status efla_tc_selftest(int N, int K, int flags, const void* A, const void* B, const float* C,
                             float* D, cudaStream_t stream) {
    g_msg[0] = 0;
    if ((N != 64 && N != 128 && N != 192 && N != 256) || (K != 64 && K != 128) || (flags & ~7) ||
        ((flags & 5) == 5))
        return fail(EFLA_ERR_UNSUPPORTED, "efla_tc_selftest: N in {64, 128, 192, 256}, K in {64, 128}, flags in 0..7 without bits 0 and 2 together (got %d, %d, %d)",
                    N, K, flags);
    const Span req[] = {{A, 1, "A"}, {B, 1, "B"}, {C, 1, "C"}, {D, 1, "D"}};
    efla_status st = check_ptrs(req, 4, nullptr, 0);
    if (st != EFLA_OK) return st;
    efla::prof_mark(nullptr, stream);
    cudaError_t e = efla::launch_tc_selftest(N, K, flags, A, B, C, D, stream);
    return e == cudaSuccess ? EFLA_OK : cuda_fail(e, "efla_tc_selftest");
}

}  // extern "C"

// ------------------------------------------------------------------ profiling
#include <string.h>
#include <vector>

namespace {
struct ProfRec {
    const char* name;   // nullptr: an entry point's start mark
    cudaEvent_t ev;
};
thread_local bool g_prof_on = false;
thread_local std::vector<ProfRec>* g_prof = nullptr;
}  // namespace

void efla::prof_mark(const char* name, cudaStream_t st) {
    if (!g_prof_on) return;
    cudaEvent_t ev;
    if (cudaEventCreate(&ev) != cudaSuccess) return;
    cudaEventRecord(ev, st);
    g_prof->push_back(ProfRec{name, ev});
}

extern "C" efla_status efla_profile_begin(void) {
    if (!g_prof) g_prof = new std::vector<ProfRec>();
    for (auto& r : *g_prof) cudaEventDestroy(r.ev);
    g_prof->clear();
    g_prof_on = true;
    return EFLA_OK;
}

extern "C" int efla_profile_end(int cap, const char** names, float* total_ms, int* launches) {
    g_prof_on = false;
    if (!g_prof) return 0;
    int n = 0;
    bool err = false;
    for (size_t i = 1; i < g_prof->size(); ++i) {
        const ProfRec& r = (*g_prof)[i];
        if (!r.name) continue;
        float ms = 0.f;
        if (cudaEventSynchronize(r.ev) != cudaSuccess ||
            cudaEventElapsedTime(&ms, (*g_prof)[i - 1].ev, r.ev) != cudaSuccess) {
            err = true;
            break;
        }
        int j = 0;
        while (j < n && strcmp(names[j], r.name) != 0) ++j;
        if (j == n) {
            if (n == cap) continue;
            names[n] = r.name;
            total_ms[n] = 0.f;
            launches[n] = 0;
            ++n;
        }
        total_ms[j] += ms;
        launches[j] += 1;
    }
    for (auto& r : *g_prof) cudaEventDestroy(r.ev);
    g_prof->clear();
    return err ? -1 : n;
}

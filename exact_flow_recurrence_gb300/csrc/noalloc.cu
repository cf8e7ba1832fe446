// noalloc.cu -- efla_fwd_noalloc: the chunked forward pass for callers that
// cannot allocate device memory.
//
// efla_fwd needs a caller-supplied device workspace.  Some callers have no way
// to provide one: a plugin running inside a host application that owns the
// device allocator and forbids other allocations, or a real-time or embedded
// loop whose rules allow no allocation once it is running.  This entry point
// runs the same kernels as efla_fwd, with their scratch taken from a device
// array that belongs to this library (g_noalloc_scratch below).  It calls no
// cudaMalloc, cudaFree or allocating library routine.
//
// The array is a file-scope __device__ variable: every GPU that loads this
// library holds EFLA_NOALLOC_SCRATCH_BYTES of it until the process exits.  In
// host code its name is only a host-side stand-in, so its device address is
// looked up with cudaGetSymbolAddress, once per device, with that device
// current, by the first call of efla_fwd_noalloc on that device.  Make that
// first call before any stream capture.
//
// Every call shares the one array and it keeps the last call's contents.  The
// forward kernels write every workspace element before reading it, so nothing
// has to be cleared between calls; but calls that overlap on the GPU (two
// streams, or two threads, at once on one device) race on the array and must
// be serialised by the caller.
#include <mutex>

#include "../../include/efla.h"
#include "launch.h"

static __device__ __align__(256) unsigned char g_noalloc_scratch[EFLA_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of g_noalloc_scratch on the current device (looked up once per device).
efla_status scratch_on_current_device(void** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        efla::set_last_error("efla_fwd_noalloc: cudaGetDevice failed: %s", cudaGetErrorString(e));
        return EFLA_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) {
        efla::set_last_error("efla_fwd_noalloc: device %d is beyond the %d devices supported", dev,
                             kMaxDevices);
        return EFLA_ERR_UNSUPPORTED;
    }
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) {
            efla::set_last_error("efla_fwd_noalloc: cudaGetSymbolAddress on device %d failed: %s",
                                 dev, cudaGetErrorString(e));
            return EFLA_ERR_CUDA;
        }
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return EFLA_OK;
}

}  // namespace

extern "C" efla_status efla_fwd_noalloc(const efla_shape* shape, const void* q, const void* k,
                                        const void* v, const float* beta, const float* S0,
                                        void* o, float* S_final, cudaStream_t stream) {
    const size_t need = efla_fwd_workspace_size(shape);
    if (need == 0)   // invalid shape (efla_fwd reports why) or a shape that needs no scratch
        return efla_fwd(shape, q, k, v, beta, S0, o, S_final, nullptr, 0, stream);
    if (need > (size_t)EFLA_NOALLOC_SCRATCH_BYTES) {
        efla::set_last_error(
            "efla_fwd_noalloc: B=%d H=%d L=%d dk=%d dv=%d chunk=%d needs %zu bytes of scratch, "
            "more than the library's built-in %zu bytes (EFLA_NOALLOC_SCRATCH_BYTES); "
            "use efla_fwd with a caller workspace",
            shape->B, shape->H, shape->L, shape->dk, shape->dv, shape->chunk, need,
            (size_t)EFLA_NOALLOC_SCRATCH_BYTES);
        return EFLA_ERR_UNSUPPORTED;
    }
    void* ws = nullptr;
    const efla_status st = scratch_on_current_device(&ws);
    if (st != EFLA_OK) return st;
    return efla_fwd(shape, q, k, v, beta, S0, o, S_final, ws, (size_t)EFLA_NOALLOC_SCRATCH_BYTES,
                    stream);
}

// noalloc.cu -- gdn_fwd_noalloc: the forward pass for callers that cannot
// allocate device memory.
//
// gdn_fwd needs a caller-owned workspace for the per-chunk results that the
// chunk-parallel kernel hands to the scan.  Some callers cannot provide one:
// code that runs inside a host framework owning all device memory (a plugin or
// an inference runtime with a fixed, fully committed memory pool, where a
// cudaMalloc would fail or is not permitted), and code on a latency-critical
// path where cudaMalloc/cudaFree would synchronise the whole device and stall
// work running beside it.  This entry point runs the same forward with its
// scratch in a fixed array that lives in the library's own device memory.
//
// The array is GDN_FWD_NOALLOC_SCRATCH_BYTES (32 MiB) on every device that loads
// the library, held until the process exits.  Problems whose forward scratch
// (gdn_fwd_workspace_bytes) is larger are rejected before anything is enqueued.
// The array used is the current device's: the current device must be the one
// that holds the tensors and runs the stream (checked against q).  The first
// call on a device looks up the array's device address with
// cudaGetSymbolAddress (with that device current); make that first call outside
// any stream capture.  Every call on a device shares the one array, so calls
// that overlap on the GPU (for example on two streams) race: order them on one
// stream.  The array keeps what the previous call left.  Two parts of the
// scratch are read before a call writes them: the tensor-core path's error word
// and the work counters of its persistent kernels, at the start of the scratch.
// gdn_fwd clears both with a cudaMemsetAsync on the call's stream at the start
// of every tensor-core forward (run_fwd_tc), and that clear is what makes the
// reuse safe; every other scratch element is written before it is read.

#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "gdn.h"
#include "gdn_internal.h"

static __device__ __align__(256) unsigned char g_fwd_scratch[GDN_FWD_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_fwd_scratch on the current device, looked up once per
// device.  In host code the array's name is only a host-side stand-in; the
// kernels must be given the address cudaGetSymbolAddress returns.
gdn_status scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    char msg[256];
    if (e != cudaSuccess) {
        snprintf(msg, sizeof(msg), "gdn_fwd_noalloc: cudaGetDevice: %s", cudaGetErrorString(e));
        gdn::set_last_error(msg);
        return GDN_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) {
        snprintf(msg, sizeof(msg), "gdn_fwd_noalloc: device %d is beyond the %d supported", dev,
                 kMaxDevices);
        gdn::set_last_error(msg);
        return GDN_ERR_UNSUPPORTED;
    }
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_fwd_scratch);
        if (e != cudaSuccess || ptr == nullptr) {
            snprintf(msg, sizeof(msg), "gdn_fwd_noalloc: cudaGetSymbolAddress: %s",
                     cudaGetErrorString(e));
            gdn::set_last_error(msg);
            return GDN_ERR_CUDA;
        }
        g_scratch_addr[dev] = ptr;
    }
    *out = g_scratch_addr[dev];
    return GDN_OK;
}

}  // namespace

extern "C" gdn_status gdn_fwd_noalloc(const gdn_problem* p, const void* q, const void* k,
                                      const void* v, const void* alpha, const void* beta,
                                      const float* initial_state, void* o, float* final_state,
                                      void* stream) {
    const size_t need = gdn_fwd_workspace_bytes(p);  // 0 for an invalid or empty problem
    if (need == 0)  // gdn_fwd reports an invalid problem; an empty one needs no scratch
        return gdn_fwd(p, q, k, v, alpha, beta, initial_state, o, final_state, nullptr, nullptr,
                       0, stream);
    if (need > (size_t)GDN_FWD_NOALLOC_SCRATCH_BYTES) {
        char msg[256];
        snprintf(msg, sizeof(msg),
                 "gdn_fwd_noalloc: this problem needs %zu bytes of scratch, more than the fixed "
                 "%zu-byte array; use gdn_fwd with a caller-owned workspace",
                 need, (size_t)GDN_FWD_NOALLOC_SCRATCH_BYTES);
        gdn::set_last_error(msg);
        return GDN_ERR_UNSUPPORTED;
    }
    // the array of the current device: q must live there
    int dev = -1;
    cudaPointerAttributes attr;
    bool known = false;
    if (q && cudaGetDevice(&dev) == cudaSuccess) {
        known = cudaPointerGetAttributes(&attr, q) == cudaSuccess;
        if (!known) cudaGetLastError();  // a failed query must not be reported by a later launch
    }
    if (known && attr.type == cudaMemoryTypeDevice && attr.device != dev) {
        char msg[256];
        snprintf(msg, sizeof(msg),
                 "gdn_fwd_noalloc: q is on device %d but device %d is current; make the tensors' device "
                 "current before the call",
                 attr.device, dev);
        gdn::set_last_error(msg);
        return GDN_ERR_INVALID_ARG;
    }
    void* scratch = nullptr;
    gdn_status st = scratch_address(&scratch);
    if (st != GDN_OK) return st;
    return gdn_fwd(p, q, k, v, alpha, beta, initial_state, o, final_state, nullptr, scratch,
                   (size_t)GDN_FWD_NOALLOC_SCRATCH_BYTES, stream);
}

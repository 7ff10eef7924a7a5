// xs_noalloc.cu -- xs_attn_a2a_noalloc: the balanced fused call for callers
// that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc: a plug-in running inside a framework
// that owns all device memory through its own pool, a latency-critical path
// where cudaMalloc's implicit device-wide synchronisation is not acceptable,
// or a process whose device memory is fully reserved up front. They still pass
// q, k, v and out, but cannot hand the library a workspace. This entry point
// uses a scratch area compiled into the library instead: a file-scope device
// array of kScratchBytes (48 MiB) that every GPU which loads the library holds
// until the process exits. It calls no cudaMalloc, cudaFree or other
// allocating routine.
//
// Rules that follow from the shared scratch:
//   * every call on a device uses the same array, which keeps the previous
//     call's contents; calls that may overlap on the GPU (different streams,
//     no ordering between them) race on it and must not be issued;
//   * nothing in the array has to start at zero: the partial rows are written
//     before they are read, and each arrival counter carries the 48-bit
//     generation of the launch that wrote it, so a count left by an earlier
//     call reads as zero. A call therefore writes the array only from its
//     kernel, after every argument check has passed;
//   * the first call on a device looks up the array's device address
//     (cudaGetSymbolAddress) with that device current, so that first call
//     should come before any stream capture;
//   * a call whose balanced schedule needs more than kScratchBytes is rejected
//     with XS_ERR_WORKSPACE before anything is enqueued.
#include <cstdio>
#include <mutex>

#include "../../include/xs.h"
#include "xs_internal.h"

namespace {

constexpr size_t kScratchBytes = (size_t)48 << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

struct ScratchState {
    bool ready = false;
    unsigned char *ptr = nullptr;  // device address of g_noalloc_scratch on this device
};
ScratchState g_state[kMaxDevices];
std::mutex g_mu;

xs_status scratch_for_current_device(ScratchState *out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return (xs_status)xs::report_error(XS_ERR_CUDA, "cudaGetDevice failed");
    if (dev < 0 || dev >= kMaxDevices) return (xs_status)xs::report_error(XS_ERR_UNSUPPORTED, "device ordinal out of range");
    std::lock_guard<std::mutex> lk(g_mu);
    ScratchState &s = g_state[dev];
    if (!s.ready) {
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess || ptr == nullptr)
            return (xs_status)xs::report_error(XS_ERR_CUDA, "cudaGetSymbolAddress of the built-in scratch failed");
        s.ptr = static_cast<unsigned char *>(ptr);
        s.ready = true;
    }
    *out = s;
    return XS_OK;
}

}  // namespace

extern "C" xs_status xs_attn_a2a_noalloc(const void *q, const void *k, const void *v, void *out, int B, int S,
                                         int H, int D, int P, float scale, void *stream) {
    if (!q || !k || !v || !out)
        return (xs_status)xs::report_error(XS_ERR_NULL, "q, k, v and out must be non-NULL");
    // shapes and device first (no launch yet); bytes is the balanced schedule's need
    size_t need = 0;
    xs_status st = xs_attn_workspace_size(B, S, H, D, P, &need);
    if (st != XS_OK) return st;
    if (need == 0) return xs_attn_a2a_ws(q, k, v, out, B, S, H, D, P, scale, nullptr, 0, stream);
    if (need > kScratchBytes) {
        char msg[160];
        snprintf(msg, sizeof msg, "these shapes need %zu bytes of scratch; the built-in scratch holds %zu bytes", need,
                 kScratchBytes);
        return (xs_status)xs::report_error(XS_ERR_WORKSPACE, msg);
    }
    if (((uintptr_t)q | (uintptr_t)k | (uintptr_t)v | (uintptr_t)out) & 15u)
        return (xs_status)xs::report_error(XS_ERR_ALIGN, "q, k, v and out must be 16-byte aligned");
    ScratchState s;
    if ((st = scratch_for_current_device(&s)) != XS_OK) return st;
    // xs_attn_a2a_ws checks every remaining argument before it enqueues anything
    return xs_attn_a2a_ws(q, k, v, out, B, S, H, D, P, scale, s.ptr, kScratchBytes, stream);
}

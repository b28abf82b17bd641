// draft_head_top_tokens_static: the get_top_tokens draft step for callers that
// cannot allocate device memory (a plugin hook that is handed only its input
// and output buffers, or a serving loop that forbids cudaMalloc because it can
// synchronise the device). Its scratch (the per-draft, per-CTA argmax slots
// and the device error word) lives in a fixed array of this library instead
// of a caller-provided workspace.
#include <atomic>
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/drafthead.h"
#include "dh_common.cuh"
#include "dh_internal.h"

namespace {

// Scratch laid out as a draft-step workspace: the error word, the epoch and
// the two banks of argmax slots for up to DH_MAX_M drafts (zero at load; each
// step zeroes the slots it read, and a step whose wait ran out leaves its bank
// to the next step to zero). Every GPU that loads the library holds it until
// the process exits. In host code this name is only a host-side stand-in for
// the array: the device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_static_scratch[sizeof(dh::Workspace)];

constexpr int kMaxDevices = 64;
// the array's device address per device; first callers on several host
// threads may each look it up and store the same value
std::atomic<void*> g_scratch_addr[kMaxDevices];

// Device address of the scratch array on the current device, looked up once
// per device (with that device current).
int static_scratch(void** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return dh::record_cuda_error(e);
    if (dev < 0 || dev >= kMaxDevices) return dh::record_cuda_error(cudaErrorInvalidDevice);
    void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (p == nullptr) {
        e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess) return dh::record_cuda_error(e);
        if (p == nullptr) return dh::record_cuda_error(cudaErrorInvalidSymbol);
        g_scratch_addr[dev].store(p, std::memory_order_release);
    }
    *out = p;
    return DH_OK;
}

}  // namespace

int dh::static_scratch_address(void** out) { return static_scratch(out); }

extern "C" int draft_head_static_read_device_error(int* err, void* stream) {
    if (err == nullptr) return DH_ERR_ARG;
    void* scratch = nullptr;
    int st = static_scratch(&scratch);
    if (st != DH_OK) return st;
    return draft_head_read_device_error(scratch, err, stream);
}

extern "C" int draft_head_top_tokens_static(const dh_head_t* hd, const void* h, int M, int32_t* ids,
                                            float* top_logit, void* stream) {
    int st = dh::check_step_args(hd, h, M);  // M <= 16: the scratch holds slots for 16 drafts
    if (st != DH_OK) return st;
    if (ids == nullptr) return DH_ERR_ARG;
    if ((reinterpret_cast<uintptr_t>(ids) & 3u) != 0 || (reinterpret_cast<uintptr_t>(top_logit) & 3u) != 0)
        return DH_ERR_ALIGN;

    void* scratch = nullptr;
    st = static_scratch(&scratch);
    if (st != DH_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    dh::GemvArgs a = dh::step_args(hd, h, M, scratch);
    a.ids = ids;
    a.top = top_logit;
    const cudaError_t e = dh::launch_gemv(a, s);
    return e == cudaSuccess ? DH_OK : dh::record_cuda_error(e);
}

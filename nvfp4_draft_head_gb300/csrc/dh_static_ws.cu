// draft_head_top_tokens_static: the get_top_tokens draft step for callers that
// cannot allocate device memory (a plugin hook that is handed only its input
// and output buffers, or a serving loop that forbids cudaMalloc because it can
// synchronise the device). Its scratch (the per-draft, per-CTA argmax slots
// and the device error word) lives in a fixed array of this library instead
// of a caller-provided workspace.
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/drafthead.h"
#include "dh_common.cuh"
#include "dh_internal.h"

namespace {

// Scratch laid out as a draft-step workspace: the error word and argmax slots
// for up to DH_MAX_M drafts (zero at load; each launch zeroes the slots it
// used again). Every GPU that loads the library holds it until the process
// exits. In host code this name is only a host-side stand-in for the array:
// the device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_static_scratch[sizeof(dh::Workspace)];

constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {nullptr};

// Device address of the scratch array on the current device, looked up once
// per device (with that device current).
int static_scratch(void** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return dh::record_cuda_error(e);
    if (dev < 0 || dev >= kMaxDevices) return dh::record_cuda_error(cudaErrorInvalidDevice);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess) return dh::record_cuda_error(e);
        if (p == nullptr) return dh::record_cuda_error(cudaErrorInvalidSymbol);
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return DH_OK;
}

}  // namespace

extern "C" int draft_head_top_tokens_static(const dh_head_t* hd, const void* h, int M, int32_t* ids,
                                            float* top_logit, void* stream) {
    if (hd == nullptr || h == nullptr || ids == nullptr) return DH_ERR_ARG;
    if (M < 1 || M > DH_MAX_M) return DH_ERR_SHAPE;  // the scratch holds slots for 16 drafts
    if (hd->q == nullptr) return DH_ERR_ARG;
    if (hd->fmt != DH_FMT_NVFP4 && hd->fmt != DH_FMT_FP8 && hd->fmt != DH_FMT_BF16 && hd->fmt != DH_FMT_NVFP4_PACKED &&
        hd->fmt != DH_FMT_FP8_W8A8)
        return DH_ERR_ARG;
    if (hd->V <= 0 || hd->N <= 0 || hd->n_kept < 1 || hd->n_kept > hd->N || hd->N % 64 != 0)
        return DH_ERR_SHAPE;
    if (!dh::gemv_supported(hd->fmt, hd->K)) return DH_ERR_SHAPE;
    if (hd->fmt == DH_FMT_NVFP4 && (hd->sf == nullptr || hd->scale == nullptr)) return DH_ERR_ARG;
    if ((hd->fmt == DH_FMT_FP8 || hd->fmt == DH_FMT_NVFP4_PACKED || hd->fmt == DH_FMT_FP8_W8A8) &&
        hd->scale == nullptr)
        return DH_ERR_ARG;
    if (hd->idx == nullptr && (hd->fmt != DH_FMT_BF16 || hd->n_kept != hd->N || hd->N > hd->V))
        return DH_ERR_ARG;
    const uintptr_t al16 = reinterpret_cast<uintptr_t>(hd->q) | reinterpret_cast<uintptr_t>(h) |
                           reinterpret_cast<uintptr_t>(hd->sf);
    if ((al16 & 15u) != 0 || (reinterpret_cast<uintptr_t>(ids) & 3u) != 0 ||
        (reinterpret_cast<uintptr_t>(top_logit) & 3u) != 0)
        return DH_ERR_ALIGN;

    void* scratch = nullptr;
    int st = static_scratch(&scratch);
    if (st != DH_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    dh::GemvArgs a{};
    a.fmt = hd->fmt;
    a.K = hd->K;
    a.V = hd->V;
    a.N = hd->N;
    a.n_kept = hd->n_kept;
    a.q = hd->q;
    a.sf = hd->sf;
    a.scale = hd->scale;
    a.idx = hd->idx;
    a.idx_ascending = (hd->idx == nullptr || (hd->flags & DH_HEAD_IDX_ASCENDING)) ? 1 : 0;
    a.h = static_cast<const uint16_t*>(h);
    a.M = M;
    a.ids = ids;
    a.top = top_logit;
    a.ws = static_cast<dh::Workspace*>(scratch);
    const cudaError_t e = dh::launch_gemv(a, s);
    return e == cudaSuccess ? DH_OK : dh::record_cuda_error(e);
}

// C-ABI front end of libdrafthead.so: argument checks on the host, then the
// kernel launches of dh_quantize.cu and dh_gemv*.cu. See include/drafthead.h.
#include <cstdint>
#include <cstring>
#include <cuda_runtime.h>

#include "../../include/drafthead.h"
#include "dh_common.cuh"
#include "dh_internal.h"

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// cudaError_t behind the calling thread's last DH_ERR_CUDA (0 if none yet).
thread_local int t_last_cuda_error = 0;

}  // namespace

int dh::record_cuda_error(cudaError_t e) {
    t_last_cuda_error = static_cast<int>(e);
    return DH_ERR_CUDA;
}

namespace {

int cuda_status(cudaError_t e) { return e == cudaSuccess ? DH_OK : dh::record_cuda_error(e); }

int check_ws(const void* ws, size_t ws_bytes, size_t need) {
    if (ws == nullptr) return DH_ERR_ARG;
    if (!aligned(ws, DH_WORKSPACE_ALIGN) || ws_bytes < need) return DH_ERR_WORKSPACE;
    return DH_OK;
}

// Staging area of draft_head_top_tokens_host, after the draft-step part of a
// workspace: M hidden rows (BF16, K each), then M ids and M top logits.
constexpr size_t kStageIds = 2 * DH_MAX_M * sizeof(int32_t);
static_assert(sizeof(dh::Workspace) % DH_WORKSPACE_ALIGN == 0, "the staging area starts aligned");
size_t round_up(size_t n, size_t a) { return (n + a - 1) / a * a; }
size_t stage_h_bytes(int K, int M) { return round_up(static_cast<size_t>(M) * static_cast<size_t>(K) * 2, DH_WORKSPACE_ALIGN); }
size_t stage_bytes(int K, int M) { return stage_h_bytes(K, M) + round_up(kStageIds, DH_WORKSPACE_ALIGN); }

// True if p is page-locked host memory the device reads and writes at the
// same address (unified addressing), e.g. from cudaHostAlloc / pin_memory().
bool device_mapped(const void* p) {
    cudaPointerAttributes at;
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
    }
    return at.type == cudaMemoryTypeHost && at.devicePointer == p;
}

int check_gather(const void* W, int V, int K, const int32_t* idx, int N) {
    if (W == nullptr || idx == nullptr) return DH_ERR_ARG;
    if (V <= 0 || K <= 0 || N <= 0) return DH_ERR_SHAPE;
    if (K % 16 != 0 || N % 64 != 0) return DH_ERR_SHAPE;
    if (static_cast<long long>(N) * K >= (1ll << 40)) return DH_ERR_SHAPE;
    if (!aligned(W, 16) || !aligned(idx, 4)) return DH_ERR_ALIGN;
    return DH_OK;
}

}  // namespace

// Checks and argument block shared by every draft-step entry point (including
// the static-scratch one in dh_static_ws.cu).
static int check_head(const dh_head_t* hd) {
    if (hd == nullptr || hd->q == nullptr) return DH_ERR_ARG;
    if (hd->fmt != DH_FMT_NVFP4 && hd->fmt != DH_FMT_FP8 && hd->fmt != DH_FMT_BF16 && hd->fmt != DH_FMT_NVFP4_PACKED &&
        hd->fmt != DH_FMT_FP8_W8A8)
        return DH_ERR_ARG;
    if (hd->V <= 0 || hd->N <= 0 || hd->n_kept < 1 || hd->n_kept > hd->N) return DH_ERR_SHAPE;
    if (hd->N % 64 != 0) return DH_ERR_SHAPE;
    if (!dh::gemv_supported(hd->fmt, hd->K)) return DH_ERR_SHAPE;
    if (hd->fmt == DH_FMT_NVFP4 && (hd->sf == nullptr || hd->scale == nullptr)) return DH_ERR_ARG;
    if ((hd->fmt == DH_FMT_FP8 || hd->fmt == DH_FMT_NVFP4_PACKED || hd->fmt == DH_FMT_FP8_W8A8) &&
        hd->scale == nullptr)
        return DH_ERR_ARG;
    if (hd->idx == nullptr) {
        if (hd->fmt != DH_FMT_BF16) return DH_ERR_ARG;
        if (hd->n_kept != hd->N || hd->N > hd->V) return DH_ERR_SHAPE;
    }
    if (!aligned(hd->q, 16) || (hd->sf && !aligned(hd->sf, 16))) return DH_ERR_ALIGN;
    if ((hd->scale && !aligned(hd->scale, 4)) || (hd->idx && !aligned(hd->idx, 4))) return DH_ERR_ALIGN;
    return DH_OK;
}

int dh::check_step_args(const dh_head_t* hd, const void* h, int M) {
    int st = check_head(hd);
    if (st != DH_OK) return st;
    if (h == nullptr) return DH_ERR_ARG;
    if (M < 1 || M > DH_MAX_M) return DH_ERR_SHAPE;
    if (!aligned(h, 16)) return DH_ERR_ALIGN;
    return DH_OK;
}

dh::GemvArgs dh::step_args(const dh_head_t* hd, const void* h, int M, void* ws) {
    dh::GemvArgs a;
    std::memset(&a, 0, sizeof a);
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
    a.ws = static_cast<dh::Workspace*>(ws);
    return a;
}

extern "C" {

int draft_head_abi_version(void) { return DH_ABI_VERSION; }

int draft_head_last_cuda_error(const char** name) {
    if (name != nullptr) *name = cudaGetErrorName(static_cast<cudaError_t>(t_last_cuda_error));
    return t_last_cuda_error;
}

const char* draft_head_status_string(int status) {
    switch (status) {
        case DH_OK: return "ok";
        case DH_ERR_ARG: return "invalid argument (NULL pointer, unknown format or count)";
        case DH_ERR_SHAPE: return "unsupported shape";
        case DH_ERR_ALIGN: return "pointer not aligned as documented";
        case DH_ERR_WORKSPACE: return "workspace too small or misaligned";
        case DH_ERR_CUDA: return "CUDA call or kernel launch failed";
        case DH_ERR_TIMEOUT: return "bounded device wait timed out";
        case DH_ERR_DEVICE: return "device error word set";
        default: return "unknown status";
    }
}

int draft_head_build_index(const uint8_t* keep_host, int V, int32_t* idx_host, int cap, int* n_kept,
                           int* N) {
    if (keep_host == nullptr || idx_host == nullptr || n_kept == nullptr || N == nullptr) return DH_ERR_ARG;
    if (V <= 0 || cap < 0) return DH_ERR_ARG;
    int n = 0;
    for (int v = 0; v < V; ++v) {
        if (!keep_host[v]) continue;
        if (n >= cap) return DH_ERR_SHAPE;
        idx_host[n++] = v;
    }
    if (n == 0) return DH_ERR_ARG;
    const int pad = (64 - n % 64) % 64;
    if (n + pad > cap) return DH_ERR_SHAPE;
    for (int i = 0; i < pad; ++i) idx_host[n + i] = idx_host[0];
    *n_kept = n;
    *N = n + pad;
    return DH_OK;
}

size_t draft_head_quantize_workspace_bytes(void) { return dh::kWorkspaceHeader; }

int nvfp4_quantize_rows(const void* W, int V, int K, const int32_t* idx, int N, uint8_t* q,
                        uint8_t* sf, float* g, void* ws, size_t ws_bytes, void* stream) {
    int st = check_gather(W, V, K, idx, N);
    if (st != DH_OK) return st;
    if (q == nullptr || sf == nullptr || g == nullptr) return DH_ERR_ARG;
    if (!aligned(q, 16) || !aligned(sf, 16) || !aligned(g, 4)) return DH_ERR_ALIGN;
    if ((st = check_ws(ws, ws_bytes, dh::kWorkspaceHeader)) != DH_OK) return st;
    return cuda_status(dh::launch_nvfp4_quantize(static_cast<const uint16_t*>(W), V, K, idx, N, q, sf,
                                                 g, static_cast<dh::Workspace*>(ws),
                                                 static_cast<cudaStream_t>(stream)));
}

int fp8_quantize_rows(const void* W, int V, int K, const int32_t* idx, int N, uint8_t* q,
                      float* scale, void* ws, size_t ws_bytes, void* stream) {
    int st = check_gather(W, V, K, idx, N);
    if (st != DH_OK) return st;
    if (q == nullptr || scale == nullptr) return DH_ERR_ARG;
    if (!aligned(q, 16) || !aligned(scale, 4)) return DH_ERR_ALIGN;
    if ((st = check_ws(ws, ws_bytes, dh::kWorkspaceHeader)) != DH_OK) return st;
    return cuda_status(dh::launch_fp8_quantize(static_cast<const uint16_t*>(W), V, K, idx, N, q, scale,
                                               static_cast<dh::Workspace*>(ws),
                                               static_cast<cudaStream_t>(stream)));
}

int fp8_quantize_activations(const void* h, int M, int K, uint8_t* qx, float* sx, void* stream) {
    if (h == nullptr || qx == nullptr || sx == nullptr) return DH_ERR_ARG;
    if (M < 1 || K <= 0 || K % 16 != 0) return DH_ERR_SHAPE;
    if (static_cast<long long>(M) * K >= (1ll << 40) || M > 65535) return DH_ERR_SHAPE;
    if (!aligned(h, 16) || !aligned(qx, 16) || !aligned(sx, 4)) return DH_ERR_ALIGN;
    return cuda_status(dh::launch_fp8_act_quantize(static_cast<const uint16_t*>(h), M, K, qx, sx,
                                                   static_cast<cudaStream_t>(stream)));
}

int nvfp4_pack_head(const uint8_t* q, const uint8_t* sf, int N, int K, uint8_t* packed, void* stream) {
    if (q == nullptr || sf == nullptr || packed == nullptr) return DH_ERR_ARG;
    if (N <= 0 || K <= 0 || N % 16 != 0 || K % 128 != 0) return DH_ERR_SHAPE;
    if (static_cast<long long>(N) * K >= (1ll << 40)) return DH_ERR_SHAPE;
    if (!aligned(q, 16) || !aligned(sf, 16) || !aligned(packed, 16)) return DH_ERR_ALIGN;
    return cuda_status(dh::launch_nvfp4_pack(q, sf, N, K, packed, static_cast<cudaStream_t>(stream)));
}

size_t draft_head_workspace_bytes(const dh_head_t* hd, int M_max) {
    size_t b = sizeof(dh::Workspace);
    if (hd != nullptr && hd->K > 0 && M_max >= 1) b += stage_bytes(hd->K, M_max < DH_MAX_M ? M_max : DH_MAX_M);
    return b;
}

int draft_head_workspace_init(void* ws, size_t ws_bytes, void* stream) {
    int st = check_ws(ws, ws_bytes, sizeof(dh::Workspace));
    if (st != DH_OK) return st;
    return cuda_status(cudaMemsetAsync(ws, 0, sizeof(dh::Workspace), static_cast<cudaStream_t>(stream)));
}

int draft_head_top_tokens(const dh_head_t* hd, const void* h, int M, int32_t* ids, float* top_logit,
                          void* ws, size_t ws_bytes, void* stream) {
    int st = dh::check_step_args(hd, h, M);
    if (st != DH_OK) return st;
    if (ids == nullptr) return DH_ERR_ARG;
    if (!aligned(ids, 4) || (top_logit && !aligned(top_logit, 4))) return DH_ERR_ALIGN;
    if ((st = check_ws(ws, ws_bytes, sizeof(dh::Workspace))) != DH_OK) return st;
    dh::GemvArgs a = dh::step_args(hd, h, M, ws);
    a.ids = ids;
    a.top = top_logit;
    return cuda_status(dh::launch_gemv(a, static_cast<cudaStream_t>(stream)));
}

int draft_head_top_keys(const dh_head_t* hd, const void* h, int M, int64_t* keys, void* ws, size_t ws_bytes,
                        void* stream) {
    int st = dh::check_step_args(hd, h, M);
    if (st != DH_OK) return st;
    if (keys == nullptr) return DH_ERR_ARG;
    if (hd->idx != nullptr && !(hd->flags & DH_HEAD_IDX_ASCENDING)) return DH_ERR_ARG;  // keys carry ids
    if (!aligned(keys, 8)) return DH_ERR_ALIGN;
    if ((st = check_ws(ws, ws_bytes, sizeof(dh::Workspace))) != DH_OK) return st;
    dh::GemvArgs a = dh::step_args(hd, h, M, ws);
    a.keys = reinterpret_cast<unsigned long long*>(keys);
    return cuda_status(dh::launch_gemv(a, static_cast<cudaStream_t>(stream)));
}

int draft_head_keys_to_ids(const int64_t* keys, int M, int32_t* ids, float* top_logit, void* stream) {
    if (keys == nullptr || ids == nullptr) return DH_ERR_ARG;
    if (M < 1 || M > DH_MAX_M) return DH_ERR_SHAPE;
    if (!aligned(keys, 8) || !aligned(ids, 4) || (top_logit && !aligned(top_logit, 4))) return DH_ERR_ALIGN;
    return cuda_status(dh::launch_keys_to_ids(reinterpret_cast<const unsigned long long*>(keys), M, ids, top_logit,
                                              static_cast<cudaStream_t>(stream)));
}

int draft_head_top_tokens_host(const dh_head_t* hd, const void* h_host, int M, int32_t* ids_host, float* top_host,
                               void* ws, size_t ws_bytes, void* stream) {
    int st = check_head(hd);
    if (st != DH_OK) return st;
    if (h_host == nullptr || ids_host == nullptr) return DH_ERR_ARG;
    if (M < 1 || M > DH_MAX_M) return DH_ERR_SHAPE;
    if ((st = check_ws(ws, ws_bytes, sizeof(dh::Workspace) + stage_bytes(hd->K, M))) != DH_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t* stage = static_cast<uint8_t*>(ws) + sizeof(dh::Workspace);
    const size_t hbytes = static_cast<size_t>(M) * hd->K * 2;
    // Page-locked buffers the device can address: a one-CTA kernel gathers h
    // into the staging area and the draft step writes the ids (and top
    // logits) straight into the host buffers; no copy-engine transfer sits
    // between the kernels, so they keep their programmatic-launch overlap.
    if (aligned(h_host, 16) && aligned(ids_host, 4) && (top_host == nullptr || aligned(top_host, 4)) &&
        device_mapped(h_host) && device_mapped(ids_host) && (top_host == nullptr || device_mapped(top_host))) {
        cudaError_t e = dh::launch_stage_rows(h_host, stage, hbytes, s);
        if (e != cudaSuccess) return cuda_status(e);
        dh::GemvArgs a = dh::step_args(hd, stage, M, ws);
        a.ids = ids_host;
        a.top = top_host;
        return cuda_status(dh::launch_gemv(a, s));
    }
    int32_t* ids = reinterpret_cast<int32_t*>(stage + stage_h_bytes(hd->K, M));
    float* top = reinterpret_cast<float*>(ids + DH_MAX_M);
    cudaError_t e = cudaMemcpyAsync(stage, h_host, hbytes, cudaMemcpyHostToDevice, s);
    if (e != cudaSuccess) return cuda_status(e);
    dh::GemvArgs a = dh::step_args(hd, stage, M, ws);
    a.ids = ids;
    a.top = top_host ? top : nullptr;
    if ((e = dh::launch_gemv(a, s)) != cudaSuccess) return cuda_status(e);
    e = cudaMemcpyAsync(ids_host, ids, M * sizeof(int32_t), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess && top_host) e = cudaMemcpyAsync(top_host, top, M * sizeof(float), cudaMemcpyDeviceToHost, s);
    return cuda_status(e);
}

int draft_head_compute_logits(const dh_head_t* hd, const void* h, int M, float* out, void* ws,
                              size_t ws_bytes, void* stream) {
    int st = dh::check_step_args(hd, h, M);
    if (st != DH_OK) return st;
    if (out == nullptr) return DH_ERR_ARG;
    if (!aligned(out, 16)) return DH_ERR_ALIGN;
    if ((st = check_ws(ws, ws_bytes, sizeof(dh::Workspace))) != DH_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    dh::GemvArgs a = dh::step_args(hd, h, M, ws);
    a.out = out;
    cudaError_t e = dh::launch_fill_neg_inf(out, static_cast<size_t>(M) * hd->V, s);
    if (e != cudaSuccess) return cuda_status(e);
    return cuda_status(dh::launch_gemv(a, s));
}

int nvfp4_linear(const dh_head_t* w, const void* x, int M, float* y, void* ws, size_t ws_bytes, void* stream) {
    if (w == nullptr || w->q == nullptr || w->scale == nullptr || x == nullptr || y == nullptr) return DH_ERR_ARG;
    if (w->fmt != DH_FMT_NVFP4_PACKED) return DH_ERR_ARG;
    if (w->N <= 0 || w->N % 64 != 0 || !dh::linear_supported(w->K)) return DH_ERR_SHAPE;
    if (M < 1 || M > DH_MAX_M) return DH_ERR_SHAPE;
    if (static_cast<long long>(M) * w->N >= (1ll << 31)) return DH_ERR_SHAPE;
    if (!aligned(w->q, 16) || !aligned(w->scale, 4) || !aligned(x, 16) || !aligned(y, 16)) return DH_ERR_ALIGN;
    int st = check_ws(ws, ws_bytes, sizeof(dh::Workspace));
    if (st != DH_OK) return st;
    dh::GemvArgs a;
    std::memset(&a, 0, sizeof a);
    a.fmt = w->fmt;
    a.K = w->K;
    a.V = w->N;       // row n of the weight writes column n of y
    a.N = w->N;
    a.n_kept = w->N;
    a.q = w->q;
    a.scale = w->scale;
    a.idx = nullptr;
    a.idx_ascending = 1;
    a.h = static_cast<const uint16_t*>(x);
    a.M = M;
    a.out = y;
    a.ws = static_cast<dh::Workspace*>(ws);
    return cuda_status(dh::launch_gemv(a, static_cast<cudaStream_t>(stream)));
}

int draft_head_wait_probe(void* ws, size_t ws_bytes, int kind, unsigned int rounds, void* stream) {
    if (kind != 0 && kind != 1) return DH_ERR_ARG;
    if (rounds < 1 || rounds > (1u << 22)) return DH_ERR_ARG;
    int st;
    if (ws == nullptr) {  // the static scratch of draft_head_top_tokens_static
        if ((st = dh::static_scratch_address(&ws)) != DH_OK) return st;
    } else if ((st = check_ws(ws, ws_bytes, dh::kWorkspaceHeader)) != DH_OK) {
        return st;
    }
    return cuda_status(dh::launch_wait_probe(static_cast<dh::Workspace*>(ws), kind, rounds,
                                             static_cast<cudaStream_t>(stream)));
}

int draft_head_read_device_error(void* ws, int* err, void* stream) {
    if (ws == nullptr || err == nullptr) return DH_ERR_ARG;
    if (!aligned(ws, DH_WORKSPACE_ALIGN)) return DH_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    dh::Workspace* w = static_cast<dh::Workspace*>(ws);
    unsigned int v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, &w->error, sizeof v, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(&w->error, 0, sizeof v, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_status(e);
    *err = static_cast<int>(v);
    return DH_OK;
}

}  // extern "C"

// Internal interface between the C-ABI front end and the kernel files.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace dh {

struct Workspace;

struct GemvArgs {
    int fmt;
    int K;
    int V;
    int N;
    int n_kept;
    const void* q;
    const uint8_t* sf;
    const float* scale;
    const int32_t* idx;
    int idx_ascending;   // idx[0..n_kept) strictly ascending (or idx == nullptr)
    const uint16_t* h;   // BF16 [M][K]
    int M;
    int32_t* ids;        // top-tokens mode
    float* top;          // optional
    unsigned long long* keys;  // shard-keys mode (instead of ids / top): int64 keys [M]
    float* out;          // logits mode: fp32 [M][V]
    Workspace* ws;
};

// True if the draft-step kernels are compiled for (fmt, K).
bool gemv_supported(int fmt, int K);

// True if nvfp4_linear supports input width K (packed NVFP4 layout).
bool linear_supported(int K);

// Enqueue the GEMV + argmax (out == nullptr) or GEMV + logits scatter
// (out != nullptr; the -inf fill must already be enqueued). Returns a
// cudaError_t of the launch.
cudaError_t launch_gemv(const GemvArgs& a, cudaStream_t s);

// Repack a canonical NVFP4 head (q [N][K/2], sf [N][K/16]) into the
// tile-major layout of DH_FMT_NVFP4_PACKED (N % 16 == 0, K % 128 == 0).
cudaError_t launch_nvfp4_pack(const uint8_t* q, const uint8_t* sf, int N, int K, uint8_t* out, cudaStream_t s);

// Decode M shard keys (signed-order int64, see draft_head_top_keys) into ids
// and optional top logits. One single-warp kernel.
cudaError_t launch_keys_to_ids(const unsigned long long* keys, int M, int32_t* ids, float* top, cudaStream_t s);

// Copy `bytes` (a multiple of 16, both pointers 16-byte aligned) from
// device-addressable host memory into a device buffer with one CTA: it reads
// before the grid-dependency wait and writes after it (the draft step that
// read the buffer last may still be running).
cudaError_t launch_stage_rows(const void* src_host, void* dst, size_t bytes, cudaStream_t s);

// Fill out[0..count) with -inf.
cudaError_t launch_fill_neg_inf(float* out, size_t count, cudaStream_t s);

// Quantisers: amax pass + encode pass (ws->amax_bits is cleared first).
cudaError_t launch_nvfp4_quantize(const uint16_t* W, int V, int K, const int32_t* idx, int N,
                                  uint8_t* q, uint8_t* sf, float* g, Workspace* ws,
                                  cudaStream_t s);
cudaError_t launch_fp8_quantize(const uint16_t* W, int V, int K, const int32_t* idx, int N,
                                uint8_t* q, float* scale, Workspace* ws, cudaStream_t s);

// Per-token dynamic E4M3 quantisation of BF16 rows h [M][K] (K % 16 == 0):
// qx [M][K] codes, sx [M] scales. One CTA per row.
cudaError_t launch_fp8_act_quantize(const uint16_t* h, int M, int K, uint8_t* qx, float* sx, cudaStream_t s);

// Bounded-wait self-test (kind 0: global-memory poll, 1: mbarrier wait).
cudaError_t launch_wait_probe(Workspace* ws, int kind, uint32_t rounds, cudaStream_t s);

// Host-side checks of a draft-step call (head descriptor, h, 1 <= M <= 16):
// DH_OK or the dh_status to return; and the kernel arguments of the call
// (ids, top and out left empty).
int check_step_args(const struct dh_head* hd, const void* h, int M);
GemvArgs step_args(const struct dh_head* hd, const void* h, int M, void* ws);

// Device address of the static scratch of draft_head_top_tokens_static on the
// current device (looked up on first use): DH_OK or a dh_status.
int static_scratch_address(void** out);

// Remember e as the calling thread's last CUDA error (draft_head_last_cuda_error)
// and return DH_ERR_CUDA.
int record_cuda_error(cudaError_t e);

// Number of SMs of the current device (cached per device).
int sm_count();


}  // namespace dh

// Head build: gather of the kept rows W[idx[n], :] fused with their
// quantisation ("q38_draft.py", load_draft_model: make_linear(W[idx]
// .contiguous(), "marlin"); the gathered head is never materialised).
//
// Pass 1 (gather_amax_kernel): max |w| over the gathered rows, one float
// atomicMax per CTA (non-negative floats order like their bit patterns).
// Pass 2 encodes:
//   NVFP4 ("Qwen3.8-Flash-Next-ABLITERATED - MTP drafter, NVFP4 experts + 98K
//   FP8 head", "How it was built"): g = max(amax, 1e-12) / (6 * 448); per
//   16-element block two lanes each hold 8 elements, the block amax is one
//   warp shuffle; s = E4M3_RNE_sat(bamax / (6 g)); codes = E2M1_RNE(clamp(
//   w / (dec(s) g), +-6)); a zero decoded scale gives signed zeros.
//   FP8 ("FP8 MTP draft stack for vLLM ...", _fp8_convert_draft_head):
//   scale = max(amax, 1e-12) / 448; q = E4M3_RNE(clamp(w / scale, +-448)).
// All divisions and products are IEEE round-to-nearest (explicit __fdiv_rn /
// __fmul_rn, no contraction), so the codes are bit-exact.
#include <cuda_fp8.h>

#include "dh_common.cuh"
#include "dh_internal.h"

namespace dh {

constexpr int kQThreads = 256;

__device__ __forceinline__ float ld_amax(const Workspace* ws) {
    float amax = __uint_as_float(*reinterpret_cast<const volatile unsigned int*>(&ws->amax_bits));
    return amax < 1e-12f ? 1e-12f : amax;
}

// W rows are read as 16-byte chunks of 8 BF16; chunk c covers row c / (K/8).
__global__ void __launch_bounds__(kQThreads)
gather_amax_kernel(const uint4* __restrict__ W, int V, int K, const int32_t* __restrict__ idx,
                   int N, Workspace* ws) {
    const int cpr = K / 8;  // chunks per row
    const size_t total = static_cast<size_t>(N) * cpr;
    float am = 0.0f;
    for (size_t c = blockIdx.x * static_cast<size_t>(kQThreads) + threadIdx.x; c < total;
         c += static_cast<size_t>(gridDim.x) * kQThreads) {
        const int n = static_cast<int>(c / cpr), kc = static_cast<int>(c % cpr);
        const int id = __ldg(idx + n);
        if (id < 0 || id >= V) {
            atomicOr(&ws->error, kDevErrIdx);
            continue;
        }
        const uint4 v = ld_stream_v4(W + static_cast<size_t>(id) * cpr + kc);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) am = fmaxf(am, fmaxf(fabsf(bf16_lo(w[i])), fabsf(bf16_hi(w[i]))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, o));
    __shared__ float s_red[kQThreads / 32];
    if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = am;
    __syncthreads();
    if (threadIdx.x == 0) {
        float r = s_red[0];
        for (int i = 1; i < kQThreads / 32; ++i) r = fmaxf(r, s_red[i]);
        if (r > 0.0f) atomicMax(&ws->amax_bits, __float_as_uint(r));
    }
}

// E2M1 code of x (finite, already divided by the block's scale), round to
// nearest with ties to the even code, saturating at 6; the sign bit follows
// the sign of x. Thresholds are the midpoints of the E2M1 magnitudes
// {0, .5, 1, 1.5, 2, 3, 4, 6}; ">" leaves a midpoint on the even code below
// it and ">=" moves it to the even code above.
__device__ __forceinline__ uint32_t e2m1_code(float x) {
    const float a = fabsf(x);
    uint32_t c = (a > 0.25f) + (a >= 0.75f) + (a > 1.25f) + (a >= 1.75f) + (a > 2.5f) +
                 (a >= 3.5f) + (a > 5.0f);
    return c | (signbit(x) ? 8u : 0u);
}

__device__ __forceinline__ uint32_t e4m3_byte(float t) {
    return static_cast<uint32_t>(__nv_cvt_float_to_fp8(t, __NV_SATFINITE, __NV_E4M3));
}

__device__ __forceinline__ float e4m3_value(uint32_t b) {
    const __half_raw hr = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(b), __NV_E4M3);
    return __half2float(__half(hr));
}

// Two adjacent lanes share one 16-element block: the even lane holds elements
// 0..7, the odd lane 8..15. Chunk indices of a pair are (2i, 2i+1) in the same
// loop iteration because the grid stride is even.
__global__ void __launch_bounds__(kQThreads)
nvfp4_encode_kernel(const uint4* __restrict__ W, int V, int K, const int32_t* __restrict__ idx,
                    int N, uint32_t* __restrict__ q, uint8_t* __restrict__ sf, float* g_out,
                    Workspace* ws) {
    const float g = __fdiv_rn(ld_amax(ws), 2688.0f);
    const float den = __fmul_rn(6.0f, g);
    if (blockIdx.x == 0 && threadIdx.x == 0) *g_out = g;
    const int cpr = K / 8;
    const size_t total = static_cast<size_t>(N) * cpr;
    const unsigned lane = threadIdx.x & 31;
    const unsigned pair = 3u << (lane & ~1u);
    for (size_t c = blockIdx.x * static_cast<size_t>(kQThreads) + threadIdx.x; c < total;
         c += static_cast<size_t>(gridDim.x) * kQThreads) {
        const int n = static_cast<int>(c / cpr), kc = static_cast<int>(c % cpr);
        const int id = __ldg(idx + n);
        if (id < 0 || id >= V) continue;  // the amax pass has flagged it
        const uint4 v = ld_stream_v4(W + static_cast<size_t>(id) * cpr + kc);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        float x[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            x[2 * i] = bf16_lo(w[i]);
            x[2 * i + 1] = bf16_hi(w[i]);
        }
        float bamax = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) bamax = fmaxf(bamax, fabsf(x[i]));
        bamax = fmaxf(bamax, __shfl_xor_sync(pair, bamax, 1));
        const uint32_t s = e4m3_byte(__fdiv_rn(bamax, den));
        const float d = __fmul_rn(e4m3_value(s), g);
        uint32_t packed = 0u;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            uint32_t code;
            if (d == 0.0f) {
                code = signbit(x[i]) ? 8u : 0u;
            } else {
                float xi = __fdiv_rn(x[i], d);
                xi = fminf(fmaxf(xi, -6.0f), 6.0f);
                code = e2m1_code(xi);
            }
            packed |= code << (4 * i);
        }
        q[c] = packed;  // 8 codes = 4 bytes; chunk c starts at byte 4c of q
        if ((c & 1) == 0) sf[c >> 1] = static_cast<uint8_t>(s);
    }
}

__global__ void __launch_bounds__(kQThreads)
fp8_encode_kernel(const uint4* __restrict__ W, int V, int K, const int32_t* __restrict__ idx,
                  int N, uint2* __restrict__ q, float* scale_out, Workspace* ws) {
    const float scale = __fdiv_rn(ld_amax(ws), 448.0f);
    if (blockIdx.x == 0 && threadIdx.x == 0) *scale_out = scale;
    const int cpr = K / 8;
    const size_t total = static_cast<size_t>(N) * cpr;
    for (size_t c = blockIdx.x * static_cast<size_t>(kQThreads) + threadIdx.x; c < total;
         c += static_cast<size_t>(gridDim.x) * kQThreads) {
        const int n = static_cast<int>(c / cpr), kc = static_cast<int>(c % cpr);
        const int id = __ldg(idx + n);
        if (id < 0 || id >= V) continue;
        const uint4 v = ld_stream_v4(W + static_cast<size_t>(id) * cpr + kc);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t b[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float lo = fminf(fmaxf(__fdiv_rn(bf16_lo(w[i]), scale), -448.0f), 448.0f);
            float hi = fminf(fmaxf(__fdiv_rn(bf16_hi(w[i]), scale), -448.0f), 448.0f);
            b[2 * i] = e4m3_byte(lo);
            b[2 * i + 1] = e4m3_byte(hi);
        }
        q[c] = make_uint2(b[0] | (b[1] << 8) | (b[2] << 16) | (b[3] << 24),
                          b[4] | (b[5] << 8) | (b[6] << 16) | (b[7] << 24));
    }
}

// Per-token dynamic E4M3 quantisation of the hidden states (the activation
// half of the W8A8 head, "FP8 MTP draft stack for vLLM ...",
// _Fp8DraftHeadMethod.apply): one CTA per row m; the row's max |h| by warp
// shuffles and shared memory, then sx[m] = max(amax, 1e-12) / 448 and
// qx[m, k] = E4M3_RNE(clamp(h[m, k] / sx[m], +-448)), eight codes per thread
// and chunk. The draft-step kernel of the W8A8 head computes the same codes
// with the same device functions.
__global__ void __launch_bounds__(kQThreads)
fp8_act_quantize_kernel(const uint4* __restrict__ h, int K, uint2* __restrict__ qx, float* __restrict__ sx) {
    const int cpr = K / 8;  // 16-byte chunks of 8 BF16 per row
    const uint4* row = h + static_cast<size_t>(blockIdx.x) * cpr;
    float am = 0.0f;
    for (int c = threadIdx.x; c < cpr; c += kQThreads) {
        const uint4 v = row[c];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) am = fmaxf(am, fmaxf(fabsf(bf16_lo(w[i])), fabsf(bf16_hi(w[i]))));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, o));
    __shared__ float s_red[kQThreads / 32];
    if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = am;
    __syncthreads();
    float amax = s_red[0];
#pragma unroll
    for (int i = 1; i < kQThreads / 32; ++i) amax = fmaxf(amax, s_red[i]);
    const float s = act_fp8_scale(amax);
    if (threadIdx.x == 0) sx[blockIdx.x] = s;
    uint2* out = qx + static_cast<size_t>(blockIdx.x) * cpr;
    for (int c = threadIdx.x; c < cpr; c += kQThreads) {
        const uint4 v = row[c];
        out[c] = make_uint2(act_fp8_pair(v.x, s) | (act_fp8_pair(v.y, s) << 16),
                            act_fp8_pair(v.z, s) | (act_fp8_pair(v.w, s) << 16));
    }
}

cudaError_t launch_fp8_act_quantize(const uint16_t* h, int M, int K, uint8_t* qx, float* sx, cudaStream_t s) {
    fp8_act_quantize_kernel<<<M, kQThreads, 0, s>>>(reinterpret_cast<const uint4*>(h), K,
                                                     reinterpret_cast<uint2*>(qx), sx);
    return cudaGetLastError();
}

static int quant_blocks(int N, int K) {
    const size_t chunks = static_cast<size_t>(N) * (K / 8);
    const size_t want = (chunks + kQThreads - 1) / kQThreads;
    const size_t cap = static_cast<size_t>(sm_count() > 0 ? sm_count() : 1) * 8;
    return static_cast<int>(want < cap ? (want > 0 ? want : 1) : cap);
}

cudaError_t launch_nvfp4_quantize(const uint16_t* W, int V, int K, const int32_t* idx, int N,
                                  uint8_t* q, uint8_t* sf, float* g, Workspace* ws,
                                  cudaStream_t s) {
    cudaError_t e = cudaMemsetAsync(&ws->amax_bits, 0, sizeof(unsigned int), s);
    if (e != cudaSuccess) return e;
    const int blocks = quant_blocks(N, K);
    const uint4* W4 = reinterpret_cast<const uint4*>(W);
    gather_amax_kernel<<<blocks, kQThreads, 0, s>>>(W4, V, K, idx, N, ws);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    nvfp4_encode_kernel<<<blocks, kQThreads, 0, s>>>(W4, V, K, idx, N,
                                                      reinterpret_cast<uint32_t*>(q), sf, g, ws);
    return cudaGetLastError();
}

cudaError_t launch_fp8_quantize(const uint16_t* W, int V, int K, const int32_t* idx, int N,
                                uint8_t* q, float* scale, Workspace* ws, cudaStream_t s) {
    cudaError_t e = cudaMemsetAsync(&ws->amax_bits, 0, sizeof(unsigned int), s);
    if (e != cudaSuccess) return e;
    const int blocks = quant_blocks(N, K);
    const uint4* W4 = reinterpret_cast<const uint4*>(W);
    gather_amax_kernel<<<blocks, kQThreads, 0, s>>>(W4, V, K, idx, N, ws);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    fp8_encode_kernel<<<blocks, kQThreads, 0, s>>>(W4, V, K, idx, N, reinterpret_cast<uint2*>(q),
                                                    scale, ws);
    return cudaGetLastError();
}

}  // namespace dh

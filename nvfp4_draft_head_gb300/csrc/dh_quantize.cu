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
//   w / (dec(s) g), +-6)); a zero decoded scale gives signed zeros. The
//   element codes come from the hardware conversion cvt.rn.satfinite.e2m1x2
//   (round to nearest even, saturating at +-6, which is the clamp; a negative
//   quotient that rounds to zero keeps its sign).
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

// Chunks each thread has in flight: its dh_idx loads, then the dependent row
// loads, are issued for kU grid-stride iterations before any arithmetic.
constexpr int kU = 4;

// Position (row n, chunk kc of the row) of a thread's current chunk c =
// n * cpr + kc, advanced by the grid stride without dividing: the stride is
// sq rows and sr chunks.
template <typename I>
struct ChunkPos {
    I n;
    int kc;
    __device__ __forceinline__ void advance(I sq, int sr, int cpr) {
        kc += sr;
        n += sq;
        if (kc >= cpr) {
            kc -= cpr;
            ++n;
        }
    }
};

// Gathered 16-byte chunks: for the kU chunks c0 + u * stride of this thread
// (p = the position of c0), the chunk's row id (or -1 past the last row / for
// an id outside [0, V), which is recorded) and its 8 BF16 values. I is the
// chunk index type (32-bit when the head has fewer than 2^31 chunks).
template <typename I>
__device__ __forceinline__ void gather_chunks(const uint4* __restrict__ W, int V, int cpr, const int32_t* __restrict__ idx,
                                              I N, ChunkPos<I> p, I sq, int sr, Workspace* ws, bool flag_bad,
                                              int (&id)[kU], int (&kc)[kU], uint4 (&v)[kU]) {
#pragma unroll
    for (int u = 0; u < kU; ++u) {
        id[u] = p.n < N ? __ldg(idx + p.n) : -1;
        kc[u] = p.kc;
        if (p.n < N && (id[u] < 0 || id[u] >= V)) {
            if (flag_bad) atomicOr(&ws->error, kDevErrIdx);
            id[u] = -1;
        }
        p.advance(sq, sr, cpr);
    }
#pragma unroll
    for (int u = 0; u < kU; ++u)
        v[u] = id[u] >= 0 ? ld_stream_v4(W + static_cast<size_t>(id[u]) * cpr + kc[u]) : make_uint4(0, 0, 0, 0);
}

// Start position and stride (in rows and chunks) of this thread's chunks.
template <typename I>
__device__ __forceinline__ void chunk_start(int cpr, ChunkPos<I>& p, I& sq, int& sr) {
    const I c0 = static_cast<I>(blockIdx.x) * kQThreads + threadIdx.x;
    const I stride = static_cast<I>(gridDim.x) * kQThreads;
    p.n = c0 / static_cast<I>(cpr);
    p.kc = static_cast<int>(c0 % static_cast<I>(cpr));
    sq = stride / static_cast<I>(cpr);
    sr = static_cast<int>(stride % static_cast<I>(cpr));
}

// W rows are read as 16-byte chunks of 8 BF16; chunk c covers row c / (K/8).
template <typename I>
__global__ void __launch_bounds__(kQThreads)
gather_amax_kernel(const uint4* __restrict__ W, int V, int K, const int32_t* __restrict__ idx,
                   int N, Workspace* ws) {
    const int cpr = K / 8;  // chunks per row
    ChunkPos<I> p;
    I sq;
    int sr;
    chunk_start<I>(cpr, p, sq, sr);
    float am = 0.0f;
    for (; p.n < static_cast<I>(N);) {
        int id[kU], kcs[kU];
        uint4 v[kU];
        gather_chunks<I>(W, V, cpr, idx, static_cast<I>(N), p, sq, sr, ws, true, id, kcs, v);
#pragma unroll
        for (int u = 0; u < kU; ++u) p.advance(sq, sr, cpr);
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) am = fmaxf(am, fmaxf(fabsf(bf16_lo(w[i])), fabsf(bf16_hi(w[i]))));
        }
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

// E2M1 codes of (lo, hi), lo in the low nibble: RNE, saturating at +-6.
__device__ __forceinline__ uint32_t e2m1x2_code(float lo, float hi) {
    uint32_t r;
    asm("{\n\t.reg .b8 b;\n\tcvt.rn.satfinite.e2m1x2.f32 b, %1, %2;\n\tcvt.u32.u8 %0, b;\n\t}"
        : "=r"(r) : "f"(hi), "f"(lo));
    return r;
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
// loop iteration because the grid stride is even (and both lanes of a pair
// see the same row, so they skip an invalid row together).
template <typename I>
__global__ void __launch_bounds__(kQThreads)
nvfp4_encode_kernel(const uint4* __restrict__ W, int V, int K, const int32_t* __restrict__ idx,
                    int N, uint32_t* __restrict__ q, uint8_t* __restrict__ sf, float* g_out,
                    Workspace* ws) {
    const float g = __fdiv_rn(ld_amax(ws), 2688.0f);
    const float den = __fmul_rn(6.0f, g);
    if (blockIdx.x == 0 && threadIdx.x == 0) *g_out = g;
    const int cpr = K / 8;
    const unsigned lane = threadIdx.x & 31;
    const unsigned pair = 3u << (lane & ~1u);
    ChunkPos<I> p;
    I sq;
    int sr;
    chunk_start<I>(cpr, p, sq, sr);
    for (; p.n < static_cast<I>(N);) {
      int ids[kU], kcs[kU];
      uint4 vs[kU];
      ChunkPos<I> pu = p;
      gather_chunks<I>(W, V, cpr, idx, static_cast<I>(N), p, sq, sr, ws, false, ids, kcs, vs);  // amax pass flagged bad ids
#pragma unroll
      for (int u = 0; u < kU; ++u) p.advance(sq, sr, cpr);
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const I c = pu.n * static_cast<I>(cpr) + static_cast<I>(kcs[u]);
        pu.advance(sq, sr, cpr);
        if (ids[u] < 0) continue;
        const uint4 v = vs[u];
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
        if (d == 0.0f) {
#pragma unroll
            for (int i = 0; i < 8; ++i) packed |= (signbit(x[i]) ? 8u : 0u) << (4 * i);
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i)
                packed |= e2m1x2_code(__fdiv_rn(x[2 * i], d), __fdiv_rn(x[2 * i + 1], d)) << (8 * i);
        }
        q[c] = packed;  // 8 codes = 4 bytes; chunk c starts at byte 4c of q
        if ((c & 1) == 0) sf[c >> 1] = static_cast<uint8_t>(s);
      }
    }
}

template <typename I>
__global__ void __launch_bounds__(kQThreads)
fp8_encode_kernel(const uint4* __restrict__ W, int V, int K, const int32_t* __restrict__ idx,
                  int N, uint2* __restrict__ q, float* scale_out, Workspace* ws) {
    const float scale = __fdiv_rn(ld_amax(ws), 448.0f);
    if (blockIdx.x == 0 && threadIdx.x == 0) *scale_out = scale;
    const int cpr = K / 8;
    ChunkPos<I> p;
    I sq;
    int sr;
    chunk_start<I>(cpr, p, sq, sr);
    for (; p.n < static_cast<I>(N);) {
      int ids[kU], kcs[kU];
      uint4 vs[kU];
      ChunkPos<I> pu = p;
      gather_chunks<I>(W, V, cpr, idx, static_cast<I>(N), p, sq, sr, ws, false, ids, kcs, vs);
#pragma unroll
      for (int u = 0; u < kU; ++u) p.advance(sq, sr, cpr);
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const I c = pu.n * static_cast<I>(cpr) + static_cast<I>(kcs[u]);
        pu.advance(sq, sr, cpr);
        if (ids[u] < 0) continue;
        const uint4 v = vs[u];
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

// 32-bit chunk indices suffice (with room for the unrolled strides).
static bool small_index(int N, int K) {
    return static_cast<unsigned long long>(N) * (K / 8) < (1ull << 31);
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
    if (small_index(N, K)) {
        gather_amax_kernel<uint32_t><<<blocks, kQThreads, 0, s>>>(W4, V, K, idx, N, ws);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        nvfp4_encode_kernel<uint32_t><<<blocks, kQThreads, 0, s>>>(W4, V, K, idx, N, reinterpret_cast<uint32_t*>(q),
                                                                    sf, g, ws);
    } else {
        gather_amax_kernel<uint64_t><<<blocks, kQThreads, 0, s>>>(W4, V, K, idx, N, ws);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        nvfp4_encode_kernel<uint64_t><<<blocks, kQThreads, 0, s>>>(W4, V, K, idx, N, reinterpret_cast<uint32_t*>(q),
                                                                    sf, g, ws);
    }
    return cudaGetLastError();
}

cudaError_t launch_fp8_quantize(const uint16_t* W, int V, int K, const int32_t* idx, int N,
                                uint8_t* q, float* scale, Workspace* ws, cudaStream_t s) {
    cudaError_t e = cudaMemsetAsync(&ws->amax_bits, 0, sizeof(unsigned int), s);
    if (e != cudaSuccess) return e;
    const int blocks = quant_blocks(N, K);
    const uint4* W4 = reinterpret_cast<const uint4*>(W);
    if (small_index(N, K)) {
        gather_amax_kernel<uint32_t><<<blocks, kQThreads, 0, s>>>(W4, V, K, idx, N, ws);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        fp8_encode_kernel<uint32_t><<<blocks, kQThreads, 0, s>>>(W4, V, K, idx, N, reinterpret_cast<uint2*>(q), scale,
                                                                  ws);
    } else {
        gather_amax_kernel<uint64_t><<<blocks, kQThreads, 0, s>>>(W4, V, K, idx, N, ws);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        fp8_encode_kernel<uint64_t><<<blocks, kQThreads, 0, s>>>(W4, V, K, idx, N, reinterpret_cast<uint2*>(q), scale,
                                                                  ws);
    }
    return cudaGetLastError();
}

}  // namespace dh

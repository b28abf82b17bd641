// Draft step: split-N GEMV of BF16 hidden states against the draft head,
// fused with the argmax over kept rows and the dh_idx map ("q38_draft.py",
// get_top_tokens: dh_idx[draft_head(h).argmax(-1)]), or with the logits
// scatter of compute_logits (the -inf fill runs first as its own kernel).
//
// Work mapping. A warp reads the head as a flat byte stream in "groups" of R
// consecutive rows whose code bytes are a multiple of 512: lane l reads the 16
// bytes at offset 512*j + 16*l of the group (j < L), so every load instruction
// of a warp is one contiguous 512-byte segment. The (row, k-range) a lane sees
// at slot j is the same in every group, so the lane keeps its slice of h in
// registers for the whole kernel and dequantises in registers. Per-row sums are
// reduced with warp shuffles; each warp keeps its best (logit, row) key, the
// CTA publishes one 64-bit key per draft with atomicMax, and the last CTA to
// finish (ticket counter) maps the winning row through dh_idx and resets the
// keys and the ticket, so the kernel can be replayed from a CUDA graph.
//
// Arithmetic: E2M1 / E4M3 codes convert exactly to f16; h is scaled by a power
// of two so that it converts to f16 exactly; each product is exact in fp32 and
// sums are fp32 (mixed-precision FMA). NVFP4 block sums are scaled by their
// E4M3 block scale once per 16 elements; the global scale and the power of two
// are applied once per row.
#include <cuda_fp16.h>
#include <cuda_bf16.h>

#pragma once
#include "dh_common.cuh"
#include "dh_internal.h"

namespace dh {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

constexpr int cgcd(int a, int b) { return b == 0 ? a : cgcd(b, a % b); }

template <int FMT, int K>
struct Geom {
    static constexpr int EPU = FMT == 1 ? 32 : (FMT == 2 ? 16 : 8);  // elements per 16-byte load
    static constexpr int RB = K * 16 / EPU;                          // code bytes per row
    static constexpr int R = 512 / cgcd(512, RB);                     // rows per group
    static constexpr int L = R * RB / 512;                            // loads per lane per group
    static constexpr int HREG = EPU / 2;                              // 32-bit h words per slot
    static constexpr int SFB = FMT == 1 ? K / 16 : 0;                 // scale bytes per row
    static constexpr int CH = L <= 5 ? L : (L % 5 == 0 ? 5 : (L % 4 == 0 ? 4 : 1));  // loads in flight
    static_assert(K % 32 == 0, "K must be a multiple of 32");
    static_assert(R * RB == 512 * L, "group geometry");
};

// Decode one 16-byte slot of codes into 32-bit operand words: f16x2 pairs for
// NVFP4 (16 words) and FP8 (8 words), the raw bf16x2 words for BF16 (4 words).
// Word i holds elements 2i and 2i+1 of the slot (low half = even element).
template <int FMT, int HREG>
__device__ __forceinline__ void decode_slot(const uint4 c, uint32_t (&cf)[HREG]) {
    const uint32_t w[4] = {c.x, c.y, c.z, c.w};
    if constexpr (FMT == 1) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint32_t f[4];
            e2m1x8_to_f16x2(w[i], f);
#pragma unroll
            for (int b = 0; b < 4; ++b) cf[4 * i + b] = f[b];
        }
    } else if constexpr (FMT == 2) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            cf[2 * i] = e4m3x2_to_f16x2(w[i] & 0xFFFFu);
            cf[2 * i + 1] = e4m3x2_to_f16x2(w[i] >> 16);
        }
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) cf[i] = w[i];
    }
}

// Dot product of a decoded slot with the matching h words. NVFP4: the two
// 16-element blocks are summed separately and scaled by their E4M3 scales
// (s2 = the two scales as f16x2); FP8 / BF16: one plain sum.
template <int FMT, int HREG>
__device__ __forceinline__ float dot_slot(const uint32_t (&cf)[HREG], const uint32_t* hw, uint32_t s2) {
    if constexpr (FMT == 1) {
        float p0 = 0.0f, p1 = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) p0 = fma2_f16_f32(cf[i], hw[i], p0);
#pragma unroll
        for (int i = 8; i < 16; ++i) p1 = fma2_f16_f32(cf[i], hw[i], p1);
        return fmaf(p1, f16hi(s2), p0 * f16lo(s2));
    } else if constexpr (FMT == 2) {
        float p = 0.0f;
#pragma unroll
        for (int i = 0; i < HREG; ++i) p = fma2_f16_f32(cf[i], hw[i], p);
        return p;
    } else {
        float p = 0.0f;
#pragma unroll
        for (int i = 0; i < HREG; ++i) p = fma2_bf16_f32(cf[i], hw[i], p);
        return p;
    }
}

// Pack two h values (already scaled) into the operand format of the format:
// f16x2 for the quantised heads, bf16x2 for the BF16 head.
template <int FMT>
__device__ __forceinline__ uint32_t pack_h(float a, float b) {
    if constexpr (FMT == 3) {
        __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&v);
    } else {
        __half2 v = __floats2half2_rn(a, b);
        return *reinterpret_cast<uint32_t*>(&v);
    }
}

__device__ __forceinline__ float block_max(float v, float* s_red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    __syncthreads();
    if (lane == 0) s_red[warp] = v;
    __syncthreads();
    float r = s_red[0];
    for (int w = 1; w < kWarps; ++w) r = fmaxf(r, s_red[w]);
    return r;
}

// Publish the CTA's argmax keys; the last CTA maps rows to ids and resets.
__device__ __forceinline__ void finish_argmax(const GemvArgs& a, const unsigned long long* cta_key) {
    __shared__ bool s_last;
    if (threadIdx.x < a.M) {
        if (cta_key[threadIdx.x] != 0ull) atomicMax(&a.ws->keys[threadIdx.x], cta_key[threadIdx.x]);
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned int t = atomicAdd(&a.ws->ticket, 1u);
        s_last = (t == gridDim.x - 1);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (threadIdx.x < a.M) {
        const int m = threadIdx.x;
        const unsigned long long k = atomicExch(&a.ws->keys[m], 0ull);
        const uint32_t row = 0xFFFFFFFFu - static_cast<uint32_t>(k & 0xFFFFFFFFull);
        int id = -1;
        if (k != 0ull && row < static_cast<uint32_t>(a.N)) id = a.idx ? a.idx[row] : static_cast<int>(row);
        if (id < 0 || id >= a.V) {
            atomicOr(&a.ws->error, kDevErrIdx);
            id = -1;
        }
        a.ids[m] = id;
        if (a.top) a.top[m] = ordered_value(static_cast<uint32_t>(k >> 32));
    }
    if (threadIdx.x == 0) atomicExch(&a.ws->ticket, 0u);
}

// Write one logit of compute_logits at out[m, idx[row]].
__device__ __forceinline__ void scatter_one(const GemvArgs& a, int m, int row, float v) {
    int id = a.idx ? a.idx[row] : row;
    if (id < 0 || id >= a.V) {
        atomicOr(&a.ws->error, kDevErrIdx);
        return;
    }
    a.out[static_cast<size_t>(m) * a.V + id] = v;
}

template <int FMT, int K, int MT, bool LOGITS>
__global__ void __launch_bounds__(kThreads) gemv_kernel(const GemvArgs a) {
    using G = Geom<FMT, K>;
    constexpr int R = G::R, L = G::L, RB = G::RB, HREG = G::HREG, EPU = G::EPU, CH = G::CH;
    constexpr int KW = K / 2;  // packed h words per draft row
    extern __shared__ __align__(16) uint32_t s_hw[];  // [MT][K/2] packed h words
    __shared__ float s_red[kWarps];
    __shared__ float s_mul[MT];
    __shared__ unsigned long long s_key[kWarps][MT];
    __shared__ unsigned long long s_cta[MT];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

    // Stage h: per draft, a power-of-two prescale (quantised heads) and the
    // packed operand words. Rows m >= M are zero.
    const uint32_t* h32 = reinterpret_cast<const uint32_t*>(a.h);
    for (int m = 0; m < MT; ++m) {
        float am = 0.0f;
        if (m < a.M)
            for (int i = tid; i < KW; i += kThreads) {
                const uint32_t w = __ldg(h32 + m * KW + i);
                am = fmaxf(am, fmaxf(fabsf(bf16_lo(w)), fabsf(bf16_hi(w))));
            }
        am = block_max(am, s_red);
        const int e = (FMT == 3) ? 0 : f16_prescale_exponent(am);
        const float sc = exp2i(e);
        for (int i = tid; i < KW; i += kThreads) {
            float x0 = 0.0f, x1 = 0.0f;
            if (m < a.M) {
                const uint32_t w = __ldg(h32 + m * KW + i);
                x0 = bf16_lo(w) * sc;
                x1 = bf16_hi(w) * sc;
            }
            s_hw[m * KW + i] = pack_h<FMT>(x0, x1);
        }
        if (tid == 0) s_mul[m] = (FMT == 3 ? 1.0f : __ldg(a.scale)) * exp2i(-e);
    }
    __syncthreads();

    // Per-lane slot geometry (identical in every group).
    int rowj[L], wofs[L];
#pragma unroll
    for (int j = 0; j < L; ++j) {
        const int o = 512 * j + 16 * lane;
        rowj[j] = o / RB;
        wofs[j] = ((o % RB) * EPU / 16) / 2;
    }
    uint32_t hr[MT == 1 ? L : 1][HREG];
    if constexpr (MT == 1) {
#pragma unroll
        for (int j = 0; j < L; ++j)
#pragma unroll
            for (int i = 0; i < HREG; ++i) hr[j][i] = s_hw[wofs[j] + i];
    }
    float mul[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) mul[m] = s_mul[m];

    unsigned long long best[MT];
#pragma unroll
    for (int m = 0; m < MT; ++m) best[m] = 0ull;

    const uint8_t* qb = static_cast<const uint8_t*>(a.q);
    const int n_groups = a.N / R;
    const int nwarps = gridDim.x * kWarps;
    for (int grp = blockIdx.x * kWarps + warp; grp < n_groups; grp += nwarps) {
        const uint8_t* qg = qb + static_cast<size_t>(grp) * (R * RB) + 16 * lane;
        const uint8_t* sg = nullptr;
        if constexpr (FMT == 1) sg = a.sf + static_cast<size_t>(grp) * (R * G::SFB) + 2 * lane;
        float acc[MT][R];
#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int r = 0; r < R; ++r) acc[m][r] = 0.0f;

#pragma unroll
        for (int j0 = 0; j0 < L; j0 += CH) {
            uint4 c[CH];
            uint32_t sv[CH];
#pragma unroll
            for (int jj = 0; jj < CH; ++jj) {
                c[jj] = ld_stream_v4(qg + 512 * (j0 + jj));
                sv[jj] = 0u;
                if constexpr (FMT == 1) sv[jj] = ld_stream_u16(sg + 64 * (j0 + jj));
            }
#pragma unroll
            for (int jj = 0; jj < CH; ++jj) {
                const int j = j0 + jj;
                uint32_t cf[HREG];
                decode_slot<FMT, HREG>(c[jj], cf);
                const uint32_t s2 = (FMT == 1) ? e4m3x2_to_f16x2(sv[jj]) : 0u;
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    float part;
                    if constexpr (MT == 1) {
                        part = dot_slot<FMT, HREG>(cf, hr[j], s2);
                    } else {
                        uint32_t hw[HREG];
                        const uint4* hp = reinterpret_cast<const uint4*>(s_hw + m * KW + wofs[j]);
#pragma unroll
                        for (int i = 0; i < HREG / 4; ++i) {
                            const uint4 v = hp[i];
                            hw[4 * i] = v.x; hw[4 * i + 1] = v.y; hw[4 * i + 2] = v.z; hw[4 * i + 3] = v.w;
                        }
                        part = dot_slot<FMT, HREG>(cf, hw, s2);
                    }
                    if constexpr (R == 1) {
                        acc[m][0] += part;
                    } else {
#pragma unroll
                        for (int r = 0; r < R; ++r) acc[m][r] += (rowj[j] == r) ? part : 0.0f;
                    }
                }
            }
        }

#pragma unroll
        for (int m = 0; m < MT; ++m)
#pragma unroll
            for (int r = 0; r < R; ++r) {
                float v = acc[m][r];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
                const int row = grp * R + r;
                if (m < a.M && row < a.n_kept) {
                    const float y = v * mul[m];
                    if constexpr (LOGITS) {
                        if (lane == r) scatter_one(a, m, row, y);
                    } else {
                        const unsigned long long k = argmax_key(ordered_key(y), static_cast<uint32_t>(row));
                        best[m] = k > best[m] ? k : best[m];
                    }
                }
            }
    }

    if constexpr (!LOGITS) {
        if (lane == 0) {
#pragma unroll
            for (int m = 0; m < MT; ++m) s_key[warp][m] = best[m];
        }
        __syncthreads();
        if (tid < MT) {
            unsigned long long k = 0ull;
            for (int w = 0; w < kWarps; ++w) k = s_key[w][tid] > k ? s_key[w][tid] : k;
            s_cta[tid] = k;
        }
        __syncthreads();
        finish_argmax(a, s_cta);
    }
}

// ------------------------------------------------------- pipelined, M = 1 ----
//
// Persistent variant for one draft. A producer warp streams "chunks" of NCW
// consecutive groups (their code bytes and E4M3 scale bytes, both contiguous
// in the head) into an S-stage shared-memory ring with 1-D bulk async copies
// (cp.async.bulk, completion counted on an mbarrier per stage), so that
// S * chunk bytes per SM are in flight regardless of registers. NCW consumer
// warps each take one group of a chunk: they copy their slots from shared
// memory to registers (the same conflict-free 512-byte rows as the direct
// path), release the stage, and dequantise / dot / reduce as in gemv_kernel.
// CTA c owns chunks c, c + grid, c + 2 grid, ... Every wait is bounded: on a
// timeout the CTA records kDevErrTimeout, stops, waits (bounded) for its
// copies in flight and still takes part in the argmax hand-off.
template <int FMT, int K, int NCW, int S, bool LOGITS>
__global__ void __launch_bounds__((NCW + 1) * 32, 1) gemv_pipe_kernel(const GemvArgs a) {
    using G = Geom<FMT, K>;
    constexpr int R = G::R, L = G::L, RB = G::RB, HREG = G::HREG, EPU = G::EPU;
    constexpr int C = NCW;                              // groups per chunk
    constexpr int GQ = R * RB;                          // code bytes per group (512 L)
    constexpr int GS = (FMT == 1) ? R * G::SFB : 0;     // scale bytes per group (64 L)
    constexpr int STAGE = C * (GQ + GS);
    constexpr int KW = K / 2;
    constexpr int NC = NCW * 32;                        // consumer threads
    static_assert(GQ % 16 == 0 && GS % 16 == 0, "bulk copies move multiples of 16 bytes");
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* ring = smem;
    uint32_t* s_hw = reinterpret_cast<uint32_t*>(smem + S * STAGE);
    __shared__ __align__(8) uint64_t full[S];
    __shared__ __align__(8) uint64_t empty[S];
    __shared__ float s_red[NCW];
    __shared__ unsigned long long s_key[NCW];
    __shared__ unsigned long long s_cta[1];
    __shared__ int s_abort;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n_groups = a.N / R;
    const int n_chunks = (n_groups + C - 1) / C;
    const int my_chunks = static_cast<int>(blockIdx.x) < n_chunks
                              ? (n_chunks - 1 - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1
                              : 0;
    volatile int* abort_flag = &s_abort;

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], NCW);
        }
        s_abort = 0;
        mbar_init_fence();
    }
    __syncthreads();

    unsigned long long best = 0ull;
    if (warp == NCW) {
        // ---------------- producer ----------------
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            const uint8_t* qb = static_cast<const uint8_t*>(a.q);
            int issued = 0;
            for (int i = 0; i < my_chunks; ++i) {
                const int s = i % S;
                if (i >= S && !mbar_wait(&empty[s], ((i / S) - 1) & 1)) {
                    atomicOr(&a.ws->error, kDevErrTimeout);
                    *abort_flag = 1;
                }
                if (*abort_flag) break;
                const int g0 = (static_cast<int>(blockIdx.x) + i * static_cast<int>(gridDim.x)) * C;
                const int ng = min(C, n_groups - g0);
                uint8_t* st = ring + s * STAGE;
                mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(ng * (GQ + GS)));
                bulk_g2s(st, qb + static_cast<size_t>(g0) * GQ, static_cast<uint32_t>(ng * GQ), &full[s], pol);
                if constexpr (FMT == 1)
                    bulk_g2s(st + C * GQ, a.sf + static_cast<size_t>(g0) * GS, static_cast<uint32_t>(ng * GS),
                             &full[s], pol);
                ++issued;
            }
            if (*abort_flag) {  // let the copies already issued land before the CTA exits
                for (int i = issued > S ? issued - S : 0; i < issued; ++i) (void)mbar_wait(&full[i % S], (i / S) & 1);
            }
        }
        __syncwarp();
    } else {
        // ---------------- consumers ----------------
        const uint32_t* h32 = reinterpret_cast<const uint32_t*>(a.h);
        float am = 0.0f;
        for (int i = tid; i < KW; i += NC) {
            const uint32_t w = __ldg(h32 + i);
            am = fmaxf(am, fmaxf(fabsf(bf16_lo(w)), fabsf(bf16_hi(w))));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, o));
        if (lane == 0) s_red[warp] = am;
        named_bar_sync(1, NC);
        am = s_red[0];
#pragma unroll
        for (int w = 1; w < NCW; ++w) am = fmaxf(am, s_red[w]);
        const int e = (FMT == 3) ? 0 : f16_prescale_exponent(am);
        const float sc = exp2i(e);
        for (int i = tid; i < KW; i += NC) {
            const uint32_t w = __ldg(h32 + i);
            s_hw[i] = pack_h<FMT>(bf16_lo(w) * sc, bf16_hi(w) * sc);
        }
        named_bar_sync(1, NC);
        int rowj[L];
        uint32_t hr[L][HREG];
#pragma unroll
        for (int j = 0; j < L; ++j) {
            const int o = 512 * j + 16 * lane;
            rowj[j] = o / RB;
            const int wofs = ((o % RB) * EPU / 16) / 2;
#pragma unroll
            for (int i = 0; i < HREG; ++i) hr[j][i] = s_hw[wofs + i];
        }
        const float mul = (FMT == 3 ? 1.0f : __ldg(a.scale)) * exp2i(-e);

        for (int i = 0; i < my_chunks; ++i) {
            const int s = i % S;
            if (!mbar_wait(&full[s], (i / S) & 1)) {
                atomicOr(&a.ws->error, kDevErrTimeout);
                *abort_flag = 1;
            }
            if (*abort_flag) break;
            const int grp = (static_cast<int>(blockIdx.x) + i * static_cast<int>(gridDim.x)) * C + warp;
            const uint8_t* st = ring + s * STAGE;
            uint4 c[L];
            uint32_t sv[L];
            const bool have = grp < n_groups;
            if (have) {
#pragma unroll
                for (int j = 0; j < L; ++j) {
                    c[j] = *reinterpret_cast<const uint4*>(st + warp * GQ + 512 * j + 16 * lane);
                    sv[j] = 0u;
                    if constexpr (FMT == 1)
                        sv[j] = *reinterpret_cast<const uint16_t*>(st + C * GQ + warp * GS + 64 * j + 2 * lane);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            if (!have) continue;
            float acc[R];
#pragma unroll
            for (int r = 0; r < R; ++r) acc[r] = 0.0f;
#pragma unroll
            for (int j = 0; j < L; ++j) {
                uint32_t cf[HREG];
                decode_slot<FMT, HREG>(c[j], cf);
                const uint32_t s2 = (FMT == 1) ? e4m3x2_to_f16x2(sv[j]) : 0u;
                const float part = dot_slot<FMT, HREG>(cf, hr[j], s2);
                if constexpr (R == 1) {
                    acc[0] += part;
                } else {
#pragma unroll
                    for (int r = 0; r < R; ++r) acc[r] += (rowj[j] == r) ? part : 0.0f;
                }
            }
#pragma unroll
            for (int r = 0; r < R; ++r) {
                float v = acc[r];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
                const int row = grp * R + r;
                if (row < a.n_kept) {
                    const float y = v * mul;
                    if constexpr (LOGITS) {
                        if (lane == r) scatter_one(a, 0, row, y);
                    } else {
                        const unsigned long long k = argmax_key(ordered_key(y), static_cast<uint32_t>(row));
                        best = k > best ? k : best;
                    }
                }
            }
        }
    }
    __syncthreads();
    if constexpr (!LOGITS) {
        if (warp < NCW && lane == 0) s_key[warp] = best;
        __syncthreads();
        if (tid == 0) {
            unsigned long long k = 0ull;
            for (int w = 0; w < NCW; ++w) k = s_key[w] > k ? s_key[w] : k;
            s_cta[0] = k;
        }
        __syncthreads();
        finish_argmax(a, s_cta);
    }
}

// ---------------------------------------------------------------- launch ----

template <int FMT, int K, int MT, bool LOGITS>
inline cudaError_t launch_one(const GemvArgs& a, cudaStream_t s) {
    using G = Geom<FMT, K>;
    auto kern = gemv_kernel<FMT, K, MT, LOGITS>;
    const size_t smem = static_cast<size_t>(MT) * K * 2;
    static int occ = 0;  // resident CTAs per SM (same for every GB300)
    if (occ == 0) {
        cudaError_t e;
        if (smem > 48 * 1024) {
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
            if (e != cudaSuccess) return e;
        }
        int o = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, kern, kThreads, smem);
        if (e != cudaSuccess) return e;
        occ = o > 0 ? o : 1;
    }
    const int sms = sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    const int n_groups = a.N / G::R;
    int blocks = sms * occ;
    const int need = (n_groups + kWarps - 1) / kWarps;
    if (blocks > need) blocks = need;
    if (blocks < 1) blocks = 1;
    kern<<<blocks, kThreads, smem, s>>>(a);
    return cudaGetLastError();
}

// Stages of the M = 1 ring: as many as fit in about 160 KB, between 2 and 6.
template <int FMT, int K, int NCW>
constexpr int pipe_stages() {
    using G = Geom<FMT, K>;
    constexpr int stage = NCW * (G::R * G::RB + (FMT == 1 ? G::R * G::SFB : 0));
    constexpr int s = (160 * 1024) / stage;
    return s < 2 ? 2 : (s > 6 ? 6 : s);
}

template <int FMT, int K, bool LOGITS>
inline cudaError_t launch_pipe(const GemvArgs& a, cudaStream_t s) {
    using G = Geom<FMT, K>;
    constexpr int NCW = 8;
    constexpr int S = pipe_stages<FMT, K, NCW>();
    constexpr int STAGE = NCW * (G::R * G::RB + (FMT == 1 ? G::R * G::SFB : 0));
    auto kern = gemv_pipe_kernel<FMT, K, NCW, S, LOGITS>;
    const size_t smem = static_cast<size_t>(S) * STAGE + static_cast<size_t>(K) * 2;
    static int configured[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        configured[dev] = 1;
    }
    const int sms = sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    const int n_chunks = (a.N / G::R + NCW - 1) / NCW;
    const int blocks = n_chunks < sms ? n_chunks : sms;
    kern<<<blocks, (NCW + 1) * 32, smem, s>>>(a);
    return cudaGetLastError();
}

template <int FMT, int K, bool LOGITS>
inline cudaError_t launch_m(const GemvArgs& a, cudaStream_t s) {
    if (a.M <= 1) return launch_pipe<FMT, K, LOGITS>(a, s);
    if (a.M <= 2) return launch_one<FMT, K, 2, LOGITS>(a, s);
    if (a.M <= 4) return launch_one<FMT, K, 4, LOGITS>(a, s);
    if (a.M <= 8) return launch_one<FMT, K, 8, LOGITS>(a, s);
    return launch_one<FMT, K, 16, LOGITS>(a, s);
}

template <int FMT, int K>
inline cudaError_t launch_k(const GemvArgs& a, cudaStream_t s) {
    return a.out ? launch_m<FMT, K, true>(a, s) : launch_m<FMT, K, false>(a, s);
}

}  // namespace dh

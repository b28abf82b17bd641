// NVFP4 draft step fed by TMA: the same tensor-core GEMV as gemv_mma_kernel
// (block-diagonal B for one draft, block-scaled A for several), but the head
// tiles reach shared memory through the Tensor Memory Accelerator instead of
// per-thread loads, so the bytes in flight per SM are set by the number of
// pipeline stages, not by registers.
//
// A producer warp walks this CTA's tiles (16 head rows x all K): for each it
// arms the stage's mbarrier with the tile's byte count and issues one 2-D
// tensor copy per 128-wide k-window (a box of 16 rows x 64 code bytes, stored
// densely, so that the 8 threads of a shared-memory phase - two rows x four
// 16-byte pieces - hit 8 different bank groups) and one 1-D bulk copy of the
// tile's 16 x K/16 scale bytes. NW consumer warps (warp w owns windows w, w +
// NW, ...) wait for the stage, copy their pieces to registers, release the
// stage, and run the MMAs. Every wait is bounded: on a timeout the CTA sets
// kDevErrTimeout, stops waiting, and the producer waits (bounded) for the
// copies it issued before the CTA exits.
#pragma once

#include "dh_gemv_mma.cuh"

namespace dh {
namespace mma {

struct __align__(64) TmapParam {
    unsigned char bytes[128];
};

template <int K>
struct TmaCfg {
    static constexpr int NWIN = K / 128;
    static constexpr int BOX = 16 * 64;                       // bytes of one window box
    static constexpr int SFB = K / 16;                        // scale bytes per row
    static constexpr int STAGE = NWIN * BOX + 16 * SFB;       // bytes of one tile
    static constexpr int S = cmax(2, cmin(6, (176 * 1024) / STAGE));
    static constexpr size_t SMEM = static_cast<size_t>(S) * STAGE + 1024;  // + alignment slack
    static_assert(STAGE % 128 == 0, "stages stay 128-byte aligned");
};

template <int K, int MT, bool LOGITS>
__global__ void __launch_bounds__((Cfg<1, K, MT>::NW + 1) * 32, 1)
    gemv_tma_kernel(const GemvArgs a, const __grid_constant__ TmapParam tmap) {
    using C = Cfg<1, K, MT>;
    using T = TmaCfg<K>;
    constexpr int NW = C::NW, WPW = C::WPW, NT = C::NT, KW = K / 2, S = T::S;
    constexpr int NC = NW * 32;  // consumer threads
    constexpr int NRED = 16 * MT;
    constexpr int PS = (2 * 3 * NW * 16 * MT * 4 <= 16 * 1024) ? 3 : 1;  // tiles per reduction
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full[S];
    __shared__ __align__(8) uint64_t empty[S];
    __shared__ float s_part[2][PS][NW][16][MT];
    __shared__ unsigned long long s_best[PS * NRED];
    __shared__ float s_red[NW][MT];
    __shared__ float s_mul[MT];
    __shared__ int s_exp[MT];
    __shared__ unsigned long long s_cta[MT];
    __shared__ int s_abort;
    uint8_t* ring = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int n_tiles = a.N / 16;
    const int my_tiles = static_cast<int>(blockIdx.x) < n_tiles
                             ? (n_tiles - 1 - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1
                             : 0;
    volatile int* abort_flag = &s_abort;

    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], NW);
        }
        s_abort = 0;
        mbar_init_fence();
    }
    __syncthreads();

    if (warp == NW) {
        // ------------------------------------------------------ producer ----
        if (lane == 0) {
            tma_prefetch_desc(&tmap);
            const uint64_t pol = policy_evict_first();
            int issued = 0;
            for (int i = 0; i < my_tiles; ++i) {
                const int s = i % S;
                if (i >= S && !mbar_wait(&empty[s], ((i / S) - 1) & 1)) {
                    atomicOr(&a.ws->error, kDevErrTimeout);
                    *abort_flag = 1;
                }
                if (*abort_flag) break;
                const int tile = static_cast<int>(blockIdx.x) + i * static_cast<int>(gridDim.x);
                uint8_t* st = ring + static_cast<size_t>(s) * T::STAGE;
                mbar_arrive_expect_tx(&full[s], T::STAGE);
#pragma unroll 4
                for (int w = 0; w < T::NWIN; ++w) tma_load_2d(st + w * T::BOX, &tmap, 64 * w, 16 * tile, &full[s], pol);
                bulk_g2s(st + T::NWIN * T::BOX, a.sf + static_cast<size_t>(tile) * 16 * T::SFB, 16 * T::SFB, &full[s],
                         pol);
                ++issued;
            }
            if (*abort_flag) {  // let the copies already issued land before the CTA exits
                for (int i = issued > S ? issued - S : 0; i < issued; ++i) (void)mbar_wait(&full[i % S], (i / S) & 1);
            }
        }
        __syncwarp();
    } else {
        // ----------------------------------------------------- consumers ----
        const uint32_t* h32 = reinterpret_cast<const uint32_t*>(a.h);
        {
            float am[MT];
#pragma unroll
            for (int m = 0; m < MT; ++m) am[m] = 0.0f;
            for (int i = tid; i < KW; i += NC) {
#pragma unroll
                for (int m = 0; m < MT; ++m)
                    if (m < a.M) {
                        const uint32_t w = __ldg(h32 + m * KW + i);
                        am[m] = fmaxf(am[m], fmaxf(fabsf(bf16_lo(w)), fabsf(bf16_hi(w))));
                    }
            }
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                float v = am[m];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
                if (lane == 0) s_red[warp][m] = v;
            }
            for (int i = tid; i < PS * NRED; i += NC) s_best[i] = 0ull;
            named_bar_sync(1, NC);
            if (tid < MT) {
                float v = 0.0f;
                for (int w = 0; w < NW; ++w) v = fmaxf(v, s_red[w][tid]);
                const int e = f16_prescale_exponent(v);
                s_exp[tid] = e;
                s_mul[tid] = __ldg(a.scale) * exp2i(-e);
            }
            named_bar_sync(1, NC);
        }
        uint32_t hb[WPW][NT][16];
#pragma unroll
        for (int ww = 0; ww < WPW; ++ww)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int d = C::BLOCKDIAG ? 0 : g + 8 * nt;
                const int k0 = 128 * (warp + ww * NW) + 32 * t;
                const float sc = d < a.M ? exp2i(s_exp[d < MT ? d : 0]) : 0.0f;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    uint32_t w = 0u;
                    if (d < a.M) w = __ldg(h32 + d * KW + k0 / 2 + j);
                    __half2 v = __floats2half2_rn(bf16_lo(w) * sc, bf16_hi(w) * sc);
                    uint32_t u = *reinterpret_cast<uint32_t*>(&v);
                    if constexpr (C::BLOCKDIAG) u = ((j < 8) ? (t == g) : (t + 4 == g)) ? u : 0u;
                    hb[ww][nt][j] = u;
                }
            }
        const int blk0 = (2 * t < 4) ? 4 * t : 4 * t - 7;
        const int blk1 = blk0 + 2;

        for (int i = 0; i < my_tiles; ++i) {
            const int s = i % S;
            if (!*abort_flag && !mbar_wait(&full[s], (i / S) & 1)) {
                atomicOr(&a.ws->error, kDevErrTimeout);
                *abort_flag = 1;
            }
            const uint8_t* st = ring + static_cast<size_t>(s) * T::STAGE;
            uint4 cg[WPW], ch[WPW];
            uint2 sgv[WPW], shv[WPW];
#pragma unroll
            for (int ww = 0; ww < WPW; ++ww) {
                const int w = warp + ww * NW;
                cg[ww] = *reinterpret_cast<const uint4*>(st + w * T::BOX + g * 64 + 16 * t);
                ch[ww] = *reinterpret_cast<const uint4*>(st + w * T::BOX + (g + 8) * 64 + 16 * t);
                sgv[ww] = *reinterpret_cast<const uint2*>(st + T::NWIN * T::BOX + g * T::SFB + 8 * w);
                shv[ww] = *reinterpret_cast<const uint2*>(st + T::NWIN * T::BOX + (g + 8) * T::SFB + 8 * w);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);

            const int par = (i / PS) & 1, ps = i % PS;
            if constexpr (C::BLOCKDIAG) {
                float y0 = 0.0f, y1 = 0.0f;
#pragma unroll
                for (int ww = 0; ww < WPW; ++ww) {
                    float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        uint32_t fg0[4], fg1[4], fh0[4], fh1[4];
                        e2m1x8_to_f16x2(half ? cg[ww].y : cg[ww].x, fg0);
                        e2m1x8_to_f16x2(half ? cg[ww].w : cg[ww].z, fg1);
                        e2m1x8_to_f16x2(half ? ch[ww].y : ch[ww].x, fh0);
                        e2m1x8_to_f16x2(half ? ch[ww].w : ch[ww].z, fh1);
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const int ii = 4 * half + j;
                            mma_f16(d, fg0[j], fh0[j], fg1[j], fh1[j], hb[ww][0][ii], hb[ww][0][8 + ii]);
                        }
                    }
                    const uint32_t sel = static_cast<uint32_t>(blk0) | (static_cast<uint32_t>(blk1) << 4);
                    uint32_t s01g, s01h;
                    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(s01g) : "r"(sgv[ww].x), "r"(sgv[ww].y), "r"(sel));
                    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(s01h) : "r"(shv[ww].x), "r"(shv[ww].y), "r"(sel));
                    const uint32_t fg = e4m3x2_to_f16x2(s01g), fh = e4m3x2_to_f16x2(s01h);
                    y0 = fmaf(d[0], f16lo(fg), y0);
                    y0 = fmaf(d[1], f16hi(fg), y0);
                    y1 = fmaf(d[2], f16lo(fh), y1);
                    y1 = fmaf(d[3], f16hi(fh), y1);
                }
                y0 += __shfl_xor_sync(0xFFFFFFFFu, y0, 1);
                y0 += __shfl_xor_sync(0xFFFFFFFFu, y0, 2);
                y1 += __shfl_xor_sync(0xFFFFFFFFu, y1, 1);
                y1 += __shfl_xor_sync(0xFFFFFFFFu, y1, 2);
                if (t == 0) {
                    s_part[par][ps][warp][g][0] = y0;
                    s_part[par][ps][warp][g + 8][0] = y1;
                }
            } else {
                float d[NT][4];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int c = 0; c < 4; ++c) d[nt][c] = 0.0f;
#pragma unroll
                for (int ww = 0; ww < WPW; ++ww) {
                    const uint32_t sel = static_cast<uint32_t>(2 * t) | (static_cast<uint32_t>(2 * t + 1) << 4);
                    uint32_t s2g, s2h, sg0, sg1, sh0, sh1;
                    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(s2g) : "r"(sgv[ww].x), "r"(sgv[ww].y), "r"(sel));
                    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(s2h) : "r"(shv[ww].x), "r"(shv[ww].y), "r"(sel));
                    const uint32_t fgs = e4m3x2_to_f16x2(s2g), fhs = e4m3x2_to_f16x2(s2h);
                    asm("prmt.b32 %0, %1, 0, 0x1010;" : "=r"(sg0) : "r"(fgs));
                    asm("prmt.b32 %0, %1, 0, 0x3232;" : "=r"(sg1) : "r"(fgs));
                    asm("prmt.b32 %0, %1, 0, 0x1010;" : "=r"(sh0) : "r"(fhs));
                    asm("prmt.b32 %0, %1, 0, 0x3232;" : "=r"(sh1) : "r"(fhs));
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        uint32_t fg[4], fh[4];
                        const uint32_t wg = q4 == 0 ? cg[ww].x : (q4 == 1 ? cg[ww].y : (q4 == 2 ? cg[ww].z : cg[ww].w));
                        const uint32_t wh = q4 == 0 ? ch[ww].x : (q4 == 1 ? ch[ww].y : (q4 == 2 ? ch[ww].z : ch[ww].w));
                        e2m1x8_to_f16x2(wg, fg);
                        e2m1x8_to_f16x2(wh, fh);
                        const uint32_t sg = q4 < 2 ? sg0 : sg1, sh = q4 < 2 ? sh0 : sh1;
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            fg[j] = hmul2(fg[j], sg);
                            fh[j] = hmul2(fh[j], sh);
                        }
#pragma unroll
                        for (int jj = 0; jj < 2; ++jj) {
                            const int ii = 2 * q4 + jj;
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt)
                                mma_f16(d[nt], fg[2 * jj], fh[2 * jj], fg[2 * jj + 1], fh[2 * jj + 1],
                                        hb[ww][nt][2 * ii], hb[ww][nt][2 * ii + 1]);
                        }
                    }
                }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const int m0 = 8 * nt + 2 * t;
                    if (m0 < MT) {
                        s_part[par][ps][warp][g][m0] = d[nt][0];
                        s_part[par][ps][warp][g + 8][m0] = d[nt][2];
                    }
                    if (m0 + 1 < MT) {
                        s_part[par][ps][warp][g][m0 + 1] = d[nt][1];
                        s_part[par][ps][warp][g + 8][m0 + 1] = d[nt][3];
                    }
                }
            }
            if (ps == PS - 1 || i == my_tiles - 1) {
                named_bar_sync(1, NC);
                const int i0 = i - ps;
                for (int r = tid; r < PS * NRED; r += NC) {
                    const int pr = r / NRED, rem = r % NRED;
                    const int row_t = rem / MT, m = rem % MT;
                    if (pr > ps) continue;
                    float v = 0.0f;
#pragma unroll 4
                    for (int w = 0; w < NW; ++w) v += s_part[par][pr][w][row_t][m];
                    const int row = (static_cast<int>(blockIdx.x) + (i0 + pr) * static_cast<int>(gridDim.x)) * 16 + row_t;
                    if (m < a.M && row < a.n_kept) {
                        const float y = v * s_mul[m];
                        if constexpr (LOGITS) {
                            scatter_one(a, m, row, y);
                        } else {
                            const unsigned long long k = argmax_key(ordered_key(y), static_cast<uint32_t>(row));
                            if (k > s_best[r]) s_best[r] = k;
                        }
                    }
                }
            }
        }
    }
    __syncthreads();
    if constexpr (!LOGITS) {
        if (tid < MT) {
            unsigned long long k = 0ull;
            for (int r = tid; r < PS * NRED; r += MT) {
                const unsigned long long v = s_best[r];
                k = v > k ? v : k;
            }
            s_cta[tid] = k;
        }
        __syncthreads();
        finish_argmax(a, s_cta);
    }
}

template <int K, int MT, bool LOGITS>
inline cudaError_t launch_tma(const GemvArgs& a, cudaStream_t s) {
    using C = Cfg<1, K, MT>;
    using T = TmaCfg<K>;
    auto kern = gemv_tma_kernel<K, MT, LOGITS>;
    static int configured[64] = {0};
    static int occ[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(T::SMEM));
        if (e != cudaSuccess) return e;
        int o = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, kern, (C::NW + 1) * 32, T::SMEM);
        if (e != cudaSuccess) return e;
        occ[dev] = o > 0 ? o : 1;
        configured[dev] = 1;
    }
    TmapParam map;
    e = make_byte_tmap(map.bytes, a.q, static_cast<uint64_t>(K / 2), static_cast<uint64_t>(a.N), 64, 16);
    if (e != cudaSuccess) return e;
    const int sms = sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    const int n_tiles = a.N / 16;
    int blocks = sms * occ[dev];
    if (blocks > n_tiles) blocks = n_tiles;
    kern<<<blocks, (C::NW + 1) * 32, T::SMEM, s>>>(a, map);
    return cudaGetLastError();
}

template <int K, bool LOGITS>
inline cudaError_t launch_tma_m(const GemvArgs& a, cudaStream_t s) {
    if (a.M <= 1) return launch_tma<K, 1, LOGITS>(a, s);
    if (a.M <= 2) return launch_tma<K, 2, LOGITS>(a, s);
    if (a.M <= 4) return launch_tma<K, 4, LOGITS>(a, s);
    if (a.M <= 8) return launch_tma<K, 8, LOGITS>(a, s);
    return launch_tma<K, 16, LOGITS>(a, s);
}

template <int K>
inline cudaError_t launch_tma_k(const GemvArgs& a, cudaStream_t s) {
    return a.out ? launch_tma_m<K, true>(a, s) : launch_tma_m<K, false>(a, s);
}

}  // namespace mma
}  // namespace dh

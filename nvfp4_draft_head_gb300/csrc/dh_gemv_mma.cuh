// Draft step on the tensor cores: GEMV of BF16 hidden states against the draft
// head ("q38_draft.py", get_top_tokens / compute_logits: draft_head(h)), fused
// with the argmax over kept rows and the dh_idx map, or with the logits scatter.
//
// Why MMA for a GEMV. The head is streamed once per step, so the path is
// bound by HBM; but at ~7 TB/s the SMs must decode ~1.2e13 E2M1 weights per
// second, and a CUDA-core FMA per weight (plus its conversion to f32) leaves
// the kernel issue-bound. Here the only per-weight ALU work is the hardware
// E2M1 -> f16 conversion (two weights per instruction); the multiply-adds run
// in mma.sync m16n8k16 (f16 x f16 -> f32, products exact, f32 accumulation).
//
// Work split. A tile is 16 head rows x the whole K. One CTA of NW warps owns a
// tile at a time (tiles blockIdx.x, blockIdx.x + grid, ...); warp w owns the
// 128-wide k-windows w, w + NW, ... of every tile, so its slice of h stays in
// registers for the whole kernel. Thread (g = lane/4, t = lane%4) loads, for
// head rows g and g+8 of the tile, the 32 consecutive k of each of its windows
// starting at 32 t (one 16-byte load per row for NVFP4). Loads of the next
// P-1 tiles are in flight while a tile is computed. Per-warp partial logits go
// to shared memory (double-buffered by tile parity); after one __syncthreads
// per tile, 16 x MT reducer threads sum the NW partials, keep the best
// (logit, row) key of their (row, draft), or write the logit into out[m, idx].
//
// NVFP4 with one draft (the headline case) uses a block-diagonal B: the 8
// columns of the MMA are the 8 E4M3 blocks of a window instead of 8 drafts.
// Slot pair p of the 16 k-slots carries elements (2i, 2i+1) of block pi(p) in
// MMA i (i < 8), and B[slot][col] is h there when col == p and 0 otherwise, so
// after the 8 MMAs of a window D[row][col] is the un-scaled sum of block pi(col)
// of that row. Each thread then applies the two E4M3 scales of its two D
// columns with 4 FFMAs per window instead of one per weight.
// pi(p) = 2p for p < 4, 2(p-4)+1 for p >= 4 makes thread t's blocks 2t, 2t+1,
// i.e. its 32 consecutive codes.
// With several drafts (and for FP8 / BF16) the 8 columns are drafts: the NVFP4
// codes are multiplied by their block scale in f16 first (exact: at most 6
// significant bits, magnitude at most 2688), and D accumulates over all k.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "dh_common.cuh"
#include "dh_gemv_impl.cuh"
#include "dh_internal.h"

namespace dh {
namespace mma {

constexpr int cmin(int a, int b) { return a < b ? a : b; }
constexpr int cmax(int a, int b) { return a > b ? a : b; }

template <int FMT, int K, int MT>
struct Cfg {
    static constexpr int NWIN = K / 128;                     // 128-wide k-windows per row
    static constexpr int NW = NWIN <= 20 ? NWIN : 20;        // warps per CTA
    static constexpr int WPW = NWIN / NW;                    // windows per warp
    static constexpr int NT = MT <= 8 ? 1 : 2;               // n8 tiles of drafts
    static constexpr bool BLOCKDIAG = (FMT == 1 && MT == 1);
    static constexpr int BPE2 = FMT == 1 ? 1 : (FMT == 2 ? 2 : 4);  // bytes per 2 elements
    static constexpr int RB = K * BPE2 / 2;                   // code bytes per head row
    static constexpr int WB = 128 * BPE2 / 2;                 // code bytes per row and window
    static constexpr int CPR = WB / 4 / 16;                   // 16-byte loads per row, window, thread
    static constexpr int SFB = FMT == 1 ? K / 16 : 0;         // scale bytes per head row
    static constexpr int TILE_REGS = WPW * (8 * CPR + (FMT == 1 ? 4 : 0));
    static constexpr int P = cmax(1, cmin(3, 48 / TILE_REGS));  // tiles of loads in flight
    static constexpr int THREADS = NW * 32;
    static_assert(NWIN % NW == 0, "windows must split evenly over warps");
    static_assert(K % 128 == 0, "K must be a multiple of 128");
};

__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// Bytes of the loads of one tile for one thread: per window, CPR 16-byte
// pieces of row g and of row g+8, and (NVFP4) the window's 8 scale bytes of
// both rows.
template <int FMT, int K, int MT>
struct TileBuf {
    using C = Cfg<FMT, K, MT>;
    uint4 c[C::WPW][2][C::CPR];
    uint2 s[C::WPW][2];
};

template <int FMT, int K, int MT>
__device__ __forceinline__ void load_tile(TileBuf<FMT, K, MT>& b, const uint8_t* q, const uint8_t* sf, int tile,
                                          int warp, int g, int t) {
    using C = Cfg<FMT, K, MT>;
#pragma unroll
    for (int ww = 0; ww < C::WPW; ++ww) {
        const int w = warp + ww * C::NW;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const size_t row = static_cast<size_t>(tile) * 16 + g + 8 * h;
            const uint8_t* p = q + row * C::RB + w * C::WB + t * (C::WB / 4);
#pragma unroll
            for (int c = 0; c < C::CPR; ++c) b.c[ww][h][c] = ld_stream_v4(p + 16 * c);
            if constexpr (FMT == 1) {
                const uint8_t* ps = sf + row * C::SFB + 8 * w;
                uint2 v;
                asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(ps));
                b.s[ww][h] = v;
            }
        }
    }
}

// Byte i (0..15) of a 16-byte piece.
__device__ __forceinline__ uint32_t byte_of(const uint4& v, int i) {
    const uint32_t w = i < 4 ? v.x : (i < 8 ? v.y : (i < 12 ? v.z : v.w));
    return (w >> (8 * (i & 3))) & 0xFFu;
}

__device__ __forceinline__ uint32_t e2m1x2_to_f16x2(uint32_t byte) {
    uint32_t r;
    asm("{\n\t.reg .b8 b;\n\tcvt.u8.u32 b, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, b;\n\t}" : "=r"(r) : "r"(byte));
    return r;
}

// Word i (0..15) of a 64-byte run held as four 16-byte pieces.
template <int CPR>
__device__ __forceinline__ uint32_t word_of(const uint4 (&v)[CPR], int i) {
    const uint4& p = v[i >> 2];
    const int j = i & 3;
    return j == 0 ? p.x : (j == 1 ? p.y : (j == 2 ? p.z : p.w));
}

template <int FMT, int K, int MT, bool LOGITS>
__global__ void __launch_bounds__(Cfg<FMT, K, MT>::THREADS, 1) gemv_mma_kernel(const GemvArgs a) {
    using C = Cfg<FMT, K, MT>;
    constexpr int NW = C::NW, WPW = C::WPW, NT = C::NT, P = C::P, KW = K / 2;
    constexpr int NTH = C::THREADS;
    constexpr int NRED = 16 * MT;  // (row, draft) reducer slots of a tile
    // tiles whose partials are reduced after one __syncthreads
    constexpr int PS = (P > 1 && 2 * P * NW * 16 * MT * 4 <= 32 * 1024) ? P : 1;
    __shared__ float s_part[2][PS][NW][16][MT];
    __shared__ unsigned long long s_best[PS * NRED];
    __shared__ float s_red[NW][MT];
    __shared__ float s_mul[MT];
    __shared__ int s_exp[MT];
    __shared__ unsigned long long s_cta[MT];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int n_tiles = a.N / 16;
    const int my_tiles = static_cast<int>(blockIdx.x) < n_tiles
                             ? (n_tiles - 1 - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1
                             : 0;
    const uint8_t* q = static_cast<const uint8_t*>(a.q);

    // Issue the first P tiles' loads before anything else.
    TileBuf<FMT, K, MT> buf[P];
#pragma unroll
    for (int p = 0; p < P; ++p)
        if (p < my_tiles) load_tile<FMT, K, MT>(buf[p], q, a.sf, blockIdx.x + p * gridDim.x, warp, g, t);

    // Per-draft power-of-two prescale of h so that it converts to f16 exactly
    // (BF16 heads use h as it is).
    const uint32_t* h32 = reinterpret_cast<const uint32_t*>(a.h);
    {
        float am[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) am[m] = 0.0f;
        for (int i = tid; i < KW; i += NTH) {
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
        for (int i = tid; i < PS * NRED; i += NTH) s_best[i] = 0ull;
        __syncthreads();
        if (tid < MT) {
            float v = 0.0f;
            for (int w = 0; w < NW; ++w) v = fmaxf(v, s_red[w][tid]);
            const int e = (FMT == 3) ? 0 : f16_prescale_exponent(v);
            s_exp[tid] = e;
            s_mul[tid] = (FMT == 3 ? 1.0f : __ldg(a.scale)) * exp2i(-e);
        }
        __syncthreads();
    }

    // This thread's h words (B fragments), per window and n8 tile: word j holds
    // h[d][k0 + 2j], h[d][k0 + 2j + 1] with k0 = 128 w + 32 t and d = g + 8 nt
    // (d = 0 in the block-diagonal case, where the columns are blocks).
    uint32_t hb[WPW][NT][16];
#pragma unroll
    for (int ww = 0; ww < WPW; ++ww)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            // the draft of B column g (one draft only in the block-diagonal case)
            const int d = C::BLOCKDIAG ? 0 : g + 8 * nt;
            const int k0 = 128 * (warp + ww * NW) + 32 * t;
            const float sc = d < a.M ? exp2i(s_exp[d < MT ? d : 0]) : 0.0f;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                uint32_t w = 0u;
                if (d < a.M) w = __ldg(h32 + d * KW + k0 / 2 + j);
                if constexpr (FMT == 3) {
                    hb[ww][nt][j] = w;
                } else {
                    __half2 v = __floats2half2_rn(bf16_lo(w) * sc, bf16_hi(w) * sc);
                    hb[ww][nt][j] = *reinterpret_cast<uint32_t*>(&v);
                }
            }
        }
    if constexpr (C::BLOCKDIAG) {
        // b0 of MMA i is nonzero only for t == g (pair p = t), b1 only for
        // t + 4 == g (pair p = t + 4); keep word i of each half or zero.
#pragma unroll
        for (int ww = 0; ww < WPW; ++ww)
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const bool keep = (j < 8) ? (t == g) : (t + 4 == g);
                hb[ww][0][j] = keep ? hb[ww][0][j] : 0u;
            }
    }

    // Blocks of this thread's D columns 2t, 2t+1 under pi (block-diagonal case).
    const int blk0 = (2 * t < 4) ? 4 * t : 4 * t - 7;
    const int blk1 = blk0 + 2;

    const float* smul = s_mul;
    for (int it = 0; it < my_tiles; it += P) {
#pragma unroll
        for (int p = 0; p < P; ++p) {
            const int ti = it + p;
            if (ti >= my_tiles) break;
            TileBuf<FMT, K, MT>& b = buf[p];
            const int par = (PS == 1 ? ti : it / P) & 1;
            const int ps = PS == 1 ? 0 : p;
            if constexpr (C::BLOCKDIAG) {
                float y0 = 0.0f, y1 = 0.0f;  // partial logits of rows g, g+8
#pragma unroll
                for (int ww = 0; ww < WPW; ++ww) {
                    float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                    // MMA i takes byte i (block 2t) and byte 8+i (block 2t+1) of each row:
                    // words (0, 2) feed i < 4, words (1, 3) feed i >= 4.
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        uint32_t fg0[4], fg1[4], fh0[4], fh1[4];
                        const uint4& cg = b.c[ww][0][0];
                        const uint4& ch = b.c[ww][1][0];
                        e2m1x8_to_f16x2(half ? cg.y : cg.x, fg0);
                        e2m1x8_to_f16x2(half ? cg.w : cg.z, fg1);
                        e2m1x8_to_f16x2(half ? ch.y : ch.x, fh0);
                        e2m1x8_to_f16x2(half ? ch.w : ch.z, fh1);
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            const int i = 4 * half + j;
                            mma_f16(d, fg0[j], fh0[j], fg1[j], fh1[j], hb[ww][0][i], hb[ww][0][8 + i]);
                        }
                    }
                    // scales of blocks blk0, blk1 of rows g, g+8 (bytes of the window's 8)
                    const uint32_t sel = static_cast<uint32_t>(blk0) | (static_cast<uint32_t>(blk1) << 4);
                    uint32_t s01g, s01h;
                    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(s01g) : "r"(b.s[ww][0].x), "r"(b.s[ww][0].y), "r"(sel));
                    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(s01h) : "r"(b.s[ww][1].x), "r"(b.s[ww][1].y), "r"(sel));
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
                    uint32_t sg0 = 0u, sg1 = 0u, sh0 = 0u, sh1 = 0u;  // (s, s) f16x2 per row and block
                    if constexpr (FMT == 1) {
                        // blocks 2t, 2t+1 of the window: bytes 2t, 2t+1 of its 8 scale bytes
                        const uint32_t sel = static_cast<uint32_t>(2 * t) | (static_cast<uint32_t>(2 * t + 1) << 4);
                        uint32_t s2g, s2h;
                        asm("prmt.b32 %0, %1, %2, %3;" : "=r"(s2g) : "r"(b.s[ww][0].x), "r"(b.s[ww][0].y), "r"(sel));
                        asm("prmt.b32 %0, %1, %2, %3;" : "=r"(s2h) : "r"(b.s[ww][1].x), "r"(b.s[ww][1].y), "r"(sel));
                        const uint32_t fg = e4m3x2_to_f16x2(s2g), fh = e4m3x2_to_f16x2(s2h);
                        asm("prmt.b32 %0, %1, 0, 0x1010;" : "=r"(sg0) : "r"(fg));
                        asm("prmt.b32 %0, %1, 0, 0x3232;" : "=r"(sg1) : "r"(fg));
                        asm("prmt.b32 %0, %1, 0, 0x1010;" : "=r"(sh0) : "r"(fh));
                        asm("prmt.b32 %0, %1, 0, 0x3232;" : "=r"(sh1) : "r"(fh));
                    }
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        // MMAs i = 2 q4, 2 q4 + 1: NVFP4 codes 4i..4i+3 are bytes 2i, 2i+1,
                        // i.e. word q4 of the row's 16 bytes; blocks: q4 < 2 -> 2t, else 2t+1
                        uint32_t fg[4], fh[4];
                        if constexpr (FMT == 1) {
                            const uint4& cg = b.c[ww][0][0];
                            const uint4& ch = b.c[ww][1][0];
                            const uint32_t wg = q4 == 0 ? cg.x : (q4 == 1 ? cg.y : (q4 == 2 ? cg.z : cg.w));
                            const uint32_t wh = q4 == 0 ? ch.x : (q4 == 1 ? ch.y : (q4 == 2 ? ch.z : ch.w));
                            e2m1x8_to_f16x2(wg, fg);
                            e2m1x8_to_f16x2(wh, fh);
                            const uint32_t sg = q4 < 2 ? sg0 : sg1, sh = q4 < 2 ? sh0 : sh1;
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                fg[j] = hmul2(fg[j], sg);
                                fh[j] = hmul2(fh[j], sh);
                            }
                        }
#pragma unroll
                        for (int jj = 0; jj < 2; ++jj) {
                            const int i = 2 * q4 + jj;
                            uint32_t a0, a1, a2, a3;
                            if constexpr (FMT == 1) {
                                a0 = fg[2 * jj];
                                a1 = fh[2 * jj];
                                a2 = fg[2 * jj + 1];
                                a3 = fh[2 * jj + 1];
                            } else if constexpr (FMT == 2) {
                                const uint32_t wg = word_of<C::CPR>(b.c[ww][0], i), wh = word_of<C::CPR>(b.c[ww][1], i);
                                a0 = e4m3x2_to_f16x2(wg & 0xFFFFu);
                                a1 = e4m3x2_to_f16x2(wh & 0xFFFFu);
                                a2 = e4m3x2_to_f16x2(wg >> 16);
                                a3 = e4m3x2_to_f16x2(wh >> 16);
                            } else {
                                a0 = word_of<C::CPR>(b.c[ww][0], 2 * i);
                                a1 = word_of<C::CPR>(b.c[ww][1], 2 * i);
                                a2 = word_of<C::CPR>(b.c[ww][0], 2 * i + 1);
                                a3 = word_of<C::CPR>(b.c[ww][1], 2 * i + 1);
                            }
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt) {
                                if constexpr (FMT == 3)
                                    mma_bf16(d[nt], a0, a1, a2, a3, hb[ww][nt][2 * i], hb[ww][nt][2 * i + 1]);
                                else
                                    mma_f16(d[nt], a0, a1, a2, a3, hb[ww][nt][2 * i], hb[ww][nt][2 * i + 1]);
                            }
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
            // loads of the tile P steps ahead go into the buffer just consumed
            const int tn = ti + P;
            if (tn < my_tiles) load_tile<FMT, K, MT>(buf[p], q, a.sf, blockIdx.x + tn * gridDim.x, warp, g, t);
            if (PS == 1 || p == P - 1 || ti == my_tiles - 1) {
                __syncthreads();
                for (int r = tid; r < PS * NRED; r += NTH) {
                    const int pr = r / NRED, rem = r % NRED;
                    const int row_t = rem / MT, m = rem % MT;
                    const int tr = PS == 1 ? ti : it + pr;
                    if (tr > ti) continue;
                    float v = 0.0f;
#pragma unroll 4
                    for (int w = 0; w < NW; ++w) v += s_part[par][pr][w][row_t][m];
                    const int row = (blockIdx.x + tr * gridDim.x) * 16 + row_t;
                    if (m < a.M && row < a.n_kept) {
                        const float y = v * smul[m];
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
    if constexpr (!LOGITS) {
        __syncthreads();
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

template <int FMT, int K, int MT, bool LOGITS>
inline cudaError_t launch_mma(const GemvArgs& a, cudaStream_t s) {
    using C = Cfg<FMT, K, MT>;
    auto kern = gemv_mma_kernel<FMT, K, MT, LOGITS>;
    const int sms = sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    static int occ = 0;
    if (occ == 0) {
        int o = 0;
        const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, kern, C::THREADS, 0);
        if (e != cudaSuccess) return e;
        occ = o > 0 ? o : 1;
    }
    const int n_tiles = a.N / 16;
    int blocks = sms * occ;
    if (blocks > n_tiles) blocks = n_tiles;
    kern<<<blocks, C::THREADS, 0, s>>>(a);
    return cudaGetLastError();
}

template <int FMT, int K, bool LOGITS>
inline cudaError_t launch_mma_m(const GemvArgs& a, cudaStream_t s) {
    if (a.M <= 1) return launch_mma<FMT, K, 1, LOGITS>(a, s);
    if (a.M <= 2) return launch_mma<FMT, K, 2, LOGITS>(a, s);
    if (a.M <= 4) return launch_mma<FMT, K, 4, LOGITS>(a, s);
    if (a.M <= 8) return launch_mma<FMT, K, 8, LOGITS>(a, s);
    return launch_mma<FMT, K, 16, LOGITS>(a, s);
}

template <int FMT, int K>
inline cudaError_t launch_mma_k(const GemvArgs& a, cudaStream_t s) {
    return a.out ? launch_mma_m<FMT, K, true>(a, s) : launch_mma_m<FMT, K, false>(a, s);
}

}  // namespace mma
}  // namespace dh

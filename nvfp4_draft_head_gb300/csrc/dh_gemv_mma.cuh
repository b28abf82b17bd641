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
// registers for the whole kernel (in shared memory at 4 and 8 drafts). Thread
// (g = lane/4, t = lane%4) takes, for head rows g and g+8 of the tile, the 32
// consecutive k of each of its windows starting at 32 t (16 bytes per row for
// NVFP4). The packed NVFP4 head at up to four drafts streams through a
// shared-memory ring of whole tiles that one producer thread fills with 1-D
// bulk copies, its first tiles before the grid-dependency wait; every other
// kernel keeps the loads of the next P-1 tiles in flight in registers. Per-warp partial logits go
// to a ring of RS shared-memory slots guarded by mbarriers; reducer warps sum
// the NW partials of each (row, draft) in a fixed order (two drafts per
// float2 read at 16 drafts), keep the best (logit, id or row) key of each, or
// write the logit into out[m, idx].
//
// NVFP4 with one draft (the headline case) uses a block-diagonal B: the 8
// columns of the MMA are the 8 E4M3 blocks of a window instead of 8 drafts.
// Slot pair p of the 16 k-slots carries elements (2i, 2i+1) of block pi(p) in
// MMA i (i < 8), and B[slot][col] is h there when col == pi(p) and 0
// otherwise, so after the 8 MMAs of a window D[row][col] is the un-scaled sum
// of block col of that row. Each thread then applies the two E4M3 scales of
// its two D columns 2t, 2t+1 with 4 FFMAs per window instead of one per weight.
// pi(p) = 2p for p < 4, 2(p-4)+1 for p >= 4 makes thread t's A slots hold
// blocks 2t, 2t+1, i.e. its 32 consecutive codes, and its D columns the same
// two blocks, whose scales it loads as one word in the packed layout.
// With several drafts (and for FP8 / BF16) the 8 columns are drafts: the NVFP4
// codes are multiplied by their block scale in f16 first (exact: at most 6
// significant bits, magnitude at most 2688), and D accumulates over all k.
//
// W8A8 FP8 head ("FP8 MTP draft stack for vLLM ...", _Fp8DraftHeadMethod.apply:
// per-token dynamic E4M3 activations, scaled FP8 matmul). The compute warps
// quantise h themselves: each finds the max |h| of its windows per draft, the
// CTA's compute warps combine them in shared memory, and each warp encodes
// every live draft's 128 values of its window together (4 per lane), then
// hands each lane the 32 codes of its own k range (its B fragments). The multiply-adds
// are mma.sync m16n8k32 e4m3 x e4m3 -> f32 on the raw codes (products of two
// E4M3 values are exact in f32); a draft's partials are scaled by its
// activation scale, the reducer's sum by the head's scale.
#pragma once

#include <atomic>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "dh_common.cuh"
#include "dh_epilogue.cuh"
#include "dh_internal.h"

namespace dh {
namespace mma {

// Registers per thread for tile loads in flight plus the h fragments.
constexpr int kLoadRegBudget = 64;
constexpr int kMaxComputeWarps = 20;

constexpr int cmin(int a, int b) { return a < b ? a : b; }

// Largest divisor of n that is at most cap.
constexpr int largest_divisor_at_most(int n, int cap) {
    for (int d = cap < n ? cap : n; d > 1; --d)
        if (n % d == 0) return d;
    return 1;
}
constexpr int cmax(int a, int b) { return a > b ? a : b; }

constexpr int cclamp(int v, int lo, int hi) { return v < lo ? lo : (v > hi ? hi : v); }
// Tiles per CTA whose dh_idx entries the reducer stages in shared memory
// (a 64,064-row head on 152 SMs gives 27, a 98,304-row head 41); further
// tiles read dh_idx from global memory.
constexpr int kIdCap = 48;

// Kernel variants of the packed NVFP4 head (DH_FMT_NVFP4_PACKED): the
// shared-memory ring (template format 4) and register loads (format 6); the
// launcher picks one per call (packed_use_ring).
constexpr int kFmtPackedRing = 4;
constexpr int kFmtPackedLdg = 6;

// LG: the compute_logits variant (some choices depend on its extra register use)
template <int FMT, int K, int MT, bool LG = false>
struct Cfg {
    static constexpr int NWIN = K / 128;                     // 128-wide k-windows per row
    static constexpr bool PACKED = (FMT == kFmtPackedRing || FMT == kFmtPackedLdg);  // tile-major NVFP4 layout
    static constexpr bool NV = (FMT == 1 || PACKED);          // NVFP4 (canonical or packed layout)
    static constexpr bool BLOCKDIAG = (NV && MT == 1);
    static constexpr bool W8A8 = (FMT == 5);                  // FP8 head, FP8 activations
    // Packed layout, K = 2560, one or two drafts: two CTAs per SM, each of 10
    // compute warps that own two windows apiece. When one CTA of a launch
    // retires, a CTA of the next launch takes its place and starts streaming
    // while the other finishes, and each warp's per-tile hand-off and shuffles
    // cover two windows. Measured (one draft, 1,000 graph steps): 18.0 -> 17.0
    // µs top tokens, 19.8 -> 18.4 compute_logits; four drafts with one reducer
    // warp (two drafts per unit) and each window read from the ring just
    // before its math: 20.5 -> 19.7 top tokens, 22.1 -> 21.4 compute_logits
    // (with shared-memory h fragments, which its registers need); eight
    // drafts, compute_logits only: 23.3 -> 22.4 (top tokens 21.6 -> 22.9).
    static constexpr bool TWO_CTA = FMT == kFmtPackedRing && MT <= 8 && NWIN == 20;
    // Register-load kernels with more windows than compute warps (K = 4,096
    // and 5,120; the packed head at 16 drafts, and at 8 for K = 5,120, whose
    // two-window warps spill there; fewer drafts take the ring): the
    // K range is split over the two CTAs of a cluster, each with one window
    // per warp; the second CTA's reducer sends its sums into the first CTA's
    // shared memory (distributed shared memory), which writes the results.
    // Each SM reads half of h, whose replicated reads (all of h by every CTA,
    // 160 KB at K = 5,120 and 16 drafts) bounded these kernels, and no warp
    // holds two windows' h fragments (which spilled at 80 registers).
    static constexpr int KS =
        (FMT != kFmtPackedRing && NWIN > kMaxComputeWarps &&
         (FMT != kFmtPackedLdg || MT >= 16 || (MT >= 8 && NWIN > 2 * 16))) ? 2 : 1;
    static constexpr int NWC = NWIN / KS;                    // windows of one CTA
    static constexpr int XS = 4;                             // exchange slots of a pair
    static constexpr int NW = largest_divisor_at_most(NWC, TWO_CTA ? 10 : kMaxComputeWarps);  // compute warps
    static constexpr int WPW = NWC / NW;                     // windows per warp
    static constexpr int MINB = TWO_CTA ? 2 : 1;             // CTAs per SM the registers must allow
    static constexpr int NT = MT <= 8 ? 1 : 2;               // n8 tiles of drafts
    // suspend-time hint on pipeline waits: register-load kernels at one and
    // two drafts (measured faster there); the ring kernels wait without it
    // (one draft 16.98 -> 16.90 µs)
    static constexpr bool HINT = MT <= 2 && FMT != kFmtPackedRing;
    // tiles per CTA at least: 2 for the packed NVFP4 head at K <= 512, whose short
    // tiles leave the step latency-bound (fewer CTAs to hand the argmax over);
    // measured slower for K >= 2560 linears and no better for the FP8 head
    static constexpr int MIN_TILES = (PACKED && K <= 512) ? 2 : 1;

    static constexpr int BPE2 = NV ? 1 : ((FMT == 2 || W8A8) ? 2 : 4);  // bytes per 2 elements
    static constexpr int RB = K * BPE2 / 2;                   // code bytes per head row
    static constexpr int WB = 128 * BPE2 / 2;                 // code bytes per row and window
    static constexpr int CPR = WB / 4 / 16;                   // 16-byte loads per row, window, thread
    static constexpr int SFB = NV ? K / 16 : 0;               // scale bytes per head row
    static constexpr int WBLK = 16 * WB + 16 * 8;             // packed: bytes of one (tile, window) block
    // registers of one tile's loads: the codes, plus (NVFP4) the scale bytes:
    // one word in the packed layout, two rows' 8 bytes in the canonical one
    static constexpr int TILE_REGS = WPW * (8 * CPR + (PACKED ? 1 : (NV ? 4 : 0)));
    // NVFP4 at 4 and 8 drafts: the B fragments (h) come from shared memory (one
    // 8-byte load per MMA) instead of 16 registers: 22.1 -> 21.9 and 24.6 -> 23.7
    // µs per step. Slower at 2 drafts (+0.5 µs) and at 16 (+2.3 µs with two
    // tiles in flight; spills with three). Packed layout only: the canonical
    // layout's scale ring owns the dynamic shared memory.
    static constexpr bool SMB = !BLOCKDIAG && ((PACKED && WPW == 1 && (MT == 4 || MT == 8)) ||
                                               ((FMT == 3 || FMT == 5) && MT >= 16) ||
                                               (FMT == kFmtPackedRing && WPW == 2 &&
                                                ((MT == 4 && (NWIN > 32 || LG)) || (MT == 8 && LG))));
    // Register-load kernels: tiles of loads in flight in registers, as many as
    // fit next to the h fragments (16 registers per window and n8 tile) in the
    // 80 registers that 21+ warps per SM allow, up to a cap: three with one n8
    // tile, two at 16 drafts and for the FP8 heads (98,304 rows, one draft:
    // W8A16, where three spilled, 41.65 -> 40.66 µs top tokens and 44.14 ->
    // 42.64 compute_logits; W8A8 39.90 -> 39.18 and 42.64 -> 41.76); the
    // packed NVFP4 head (9 registers a tile) two at one draft (20.00 -> 19.94
    // µs against three), four at two and eight drafts (21.43 -> 20.99, 22.19 ->
    // 21.55; four at four drafts was slower), two at 16 (three spilled).
    static constexpr int PCAP = PACKED ? (MT == 1 ? 2 : (MT == 2 ? 4 : (MT >= 16 ? ((KS == 2 && NWIN > 32) ? 1 : 2) : 3)))
                                       : (MT >= 16 ? (W8A8 ? 2 : 1) : ((FMT == 2 || FMT == 5) ? 2 : 3));
    // Packed layout: the head streams through a ring of whole tiles in shared
    // memory, filled by one producer thread with 1-D bulk copies (the tiles of
    // this layout are contiguous). Its first RPRE tiles are issued before the
    // grid-dependency wait, so a launch reads its head while the preceding
    // kernel in the stream finishes; compute warps then read their windows of
    // each tile from shared memory, one tile ahead of the math with one window
    // per warp (P = 2). Issuing more tiles before the wait delays the
    // preceding launch's hand-off and this launch's first tiles behind the
    // burst (one draft, one CTA per SM: eight 18.0, four 17.3 µs; two CTAs per
    // SM: four 17.7, one 17.0).
    static constexpr bool RING = FMT == kFmtPackedRing;
    static constexpr int TB = NWIN * WBLK;                    // packed: bytes of one tile
    static constexpr int RPRE = TWO_CTA ? 1 : 4;
    static constexpr int P = RING ? ((WPW == 1 && MT <= 8) ? 2 : 1)
                                  : ((SMB && PACKED) ? (MT == 8 ? 4 : 3)
                                         : cmax(1, cmin(PCAP, (kLoadRegBudget - (SMB ? 0 : WPW * NT * 16)) / TILE_REGS)));
    // Canonical NVFP4 layout: a loader warp streams each tile's scale bytes
    // into a shared-memory ring with 1-D bulk copies.
    static constexpr bool SCALES = (FMT == 1);
    static constexpr bool LOADER = SCALES;
    // reducer unit: one row and DV drafts (one float2 read per partial at 16 drafts)
    static constexpr int DV = (MT >= 16 || (TWO_CTA && MT >= 4)) ? 2 : 1;
    // One draft: the partial sums are stored row-major ([slot][row][warp]), so
    // a reducer lane reads its row's partials with 16-byte loads and sums them
    // as a tree (one draft 21.3 -> 19.7 µs against the warp-major layout with
    // a sequential sum, where the single reducer warp fell behind).
    static constexpr bool RED_T = BLOCKDIAG;
    static constexpr int NRW = TWO_CTA ? 1 : (MT >= 16 ? (16 * MT / DV) / 32 : (MT >= 8 ? 4 : (MT >= 4 ? 2 : 1)));  // reducer warps
    static constexpr int THREADS = (NW + NRW + ((LOADER || RING) ? 1 : 0)) * 32;  // + reducers (+ loader / producer)
    static constexpr int SLOT = 16 * SFB;                              // bytes of one ring slot
    static constexpr int SS = 6;
    // partial-sum slots: register-load kernels eight for the packed one-draft
    // kernel (one draft 19.87 -> 19.73 µs against four), else four while they
    // fit in 40 KB, else two; the ring kernels as many as their budget holds
    // (2 to 16), in dynamic shared memory
    static constexpr int PART_SLOT = NW * 16 * MT * 4;                 // bytes of one partial-sum slot
    static constexpr int PART_BUDGET = TWO_CTA ? 10 * 1024 : 40 * 1024;
    static constexpr int RS = RING ? cclamp(PART_BUDGET / PART_SLOT, 2, 16)
                                   : ((PACKED && MT == 1) ? 8 : ((4 * NW * 16 * MT * 4 <= 40 * 1024) ? 4 : 2));
    static constexpr int PART_DYN = RING ? RS * PART_SLOT : 0;
    static constexpr int SMB_BYTES = SMB ? NW * WPW * NT * 8 * 32 * 8 : 0;
    // packed layout: dynamic shared memory of a CTA (one or two per SM) and
    // the tiles of its ring, as many as fit next to the partials and the h
    // fragments, 2 to 8. Two CTAs per SM: three tiles at one draft, four at
    // two and four drafts where the h fragments stay in registers (two drafts
    // 18.64 -> 18.52 µs, four 19.71 -> 19.55; one draft 16.76 -> 16.90 with four)
    static constexpr int RING_BUDGET = TWO_CTA ? (MT == 1 ? 96 : 104) * 1024 : 200 * 1024;
    static constexpr int RT = RING ? cclamp((RING_BUDGET - PART_DYN - SMB_BYTES) / TB, 2, 8) : 0;
    static constexpr int NSB = RING ? RT : SS;                         // tile / scale ring barriers
    // K split: the exchange area after the scale ring or the h fragments:
    // the sums' slots, the first CTA's own sums and ids of the tile in hand,
    // the slots' full and empty barriers, and (W8A8) the partner's max |h|
    // per draft with its barrier
    static constexpr int XOFF = LOADER ? SS * SLOT : SMB_BYTES;
    static constexpr int XB_BYTES = KS == 2 ? (XS + 2) * 16 * MT * 4 + 2 * XS * 8 + 16 * 4 + 8 : 0;
    static constexpr size_t DYN_SMEM = RING ? static_cast<size_t>(RT) * TB + PART_DYN + SMB_BYTES
                                            : static_cast<size_t>(XOFF + XB_BYTES);
    static_assert(!(KS == 2 && RING), "the K split is for the register-load kernels");
    static_assert(NWIN % KS == 0 && NWC % NW == 0, "windows must split evenly over CTAs and warps");
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

// D += A B with E4M3 A (16 x 32, row) and B (32 x 8, col), f32 accumulation.
__device__ __forceinline__ void mma_e4m3(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Code bytes of one tile held by one thread: per window, CPR 16-byte pieces of
// row g and of row g+8, and for NVFP4 the scale bytes: in the packed layout the
// word with the scales of blocks 2t, 2t+1 of rows g and g+8 (loaded with the
// codes), in the canonical one the window's 8 scale bytes of both rows (taken
// from the shared-memory scale ring).
template <int FMT, int K, int MT>
struct TileBuf {
    using C = Cfg<FMT, K, MT>;
    uint4 c[C::WPW][2][C::CPR];
    uint2 s[C::WPW][2];
    uint32_t sp[C::WPW];
};

// Shared-memory reads that stay where they stand in program order (not
// hoisted above the preceding math), so that a window's operands occupy
// registers only while it is processed.
__device__ __forceinline__ uint4 lds_v4_ordered(const void* p) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(smem_u32(p)) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t lds_u32_ordered(const void* p) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)) : "memory");
    return v;
}

template <int FMT, int K, int MT>
__device__ __forceinline__ void load_tile(TileBuf<FMT, K, MT>& b, const uint8_t* q, int tile, int wbase, int g,
                                          int t) {
    using C = Cfg<FMT, K, MT>;
#pragma unroll
    for (int ww = 0; ww < C::WPW; ++ww) {
        const int w = wbase + ww * C::NW;  // window
        if constexpr (C::PACKED) {
            // block (tile, w): 16 rows x 64 code bytes, then 4 scale bytes per lane
            const uint8_t* blk = q + (static_cast<size_t>(tile) * C::NWIN + w) * C::WBLK;
#pragma unroll
            for (int h = 0; h < 2; ++h) b.c[ww][h][0] = ld_stream_v4(blk + (g + 8 * h) * 64 + 16 * t);
            asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];"
                         : "=r"(b.sp[ww]) : "l"(blk + 16 * 64 + 4 * (4 * g + t)));
        } else {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const size_t row = static_cast<size_t>(tile) * 16 + g + 8 * h;
                const uint8_t* p = q + row * C::RB + w * C::WB + t * (C::WB / 4);
#pragma unroll
                for (int c = 0; c < C::CPR; ++c) b.c[ww][h][c] = ld_stream_v4(p + 16 * c);
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
__global__ void __launch_bounds__(Cfg<FMT, K, MT, LOGITS>::THREADS, Cfg<FMT, K, MT, LOGITS>::MINB)
    gemv_mma_kernel(const GemvArgs a) {
    using C = Cfg<FMT, K, MT, LOGITS>;
    constexpr int NW = C::NW, WPW = C::WPW, NT = C::NT, P = C::P, KW = K / 2, RS = C::RS;
    constexpr int NRED = 16 * MT;  // (row, draft) results of a tile
    constexpr int RTm = C::RT > 0 ? C::RT : 1;
    __shared__ __align__(16) float s_part_st[C::RING ? 1 : RS][NW][16][MT];
    __shared__ __align__(8) uint64_t full_p[RS];
    __shared__ __align__(8) uint64_t empty_p[RS];
    __shared__ __align__(8) uint64_t full_s[C::NSB];   // tile ring (packed) / scale ring (canonical)
    __shared__ __align__(8) uint64_t empty_s[C::NSB];
    // dynamic shared memory: packed layout [RT tiles][RS partial-sum slots][h
    // fragments]; canonical NVFP4 [SS][16 rows][K/16] scale bytes; otherwise
    // the h fragments (4 and 8 drafts)
    extern __shared__ __align__(128) uint8_t s_dyn[];
    float* const s_part = C::RING ? reinterpret_cast<float*>(s_dyn + static_cast<size_t>(C::RT) * C::TB)
                                  : &s_part_st[0][0][0][0];
    // partial sum of (ring slot, compute warp, tile row, draft)
    auto part = [&](int slot, int w, int row, int m) -> float* {
        if constexpr (C::RED_T) return s_part + (slot * 16 + row) * NW + w;
        return s_part + ((slot * NW + w) * 16 + row) * MT + m;
    };
    __shared__ unsigned long long s_best[NRED];
    __shared__ unsigned long long s_cta[MT];
    __shared__ int s_abort;
    __shared__ uint2 s_epoch;  // top-tokens mode: the workspace's epoch (slot bank) and dirty word
    __shared__ float s_amx[C::W8A8 ? NW : 1][16];  // W8A8: per compute warp and draft, max |h|
    // dh_idx of this CTA's first kIdCap tiles: [i][0..15] the rows' ids, [i][16]
    // the id of the row after the tile (copied when that row exists)
    __shared__ __align__(16) int s_ids[kIdCap * 20];
    // K split over a pair (dynamic shared memory): the second CTA's per-tile
    // sums [slot][row][draft] in the first CTA, which waits on xfull[slot];
    // the second waits on xempty[slot] until the first has read a slot
    float* const s_xb = reinterpret_cast<float*>(s_dyn + C::XOFF);
    uint64_t* const xfull = reinterpret_cast<uint64_t*>(s_dyn + C::XOFF + (C::XS + 2) * NRED * 4);
    uint64_t* const xempty = xfull + C::XS;
    float* const amx_rx = reinterpret_cast<float*>(xempty + C::XS);  // W8A8: the partner's max |h| per draft
    uint64_t* const amx_bar = reinterpret_cast<uint64_t*>(amx_rx + 16);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int n_tiles = a.N / 16;
    // tiles go to CTAs, or with the K split to pairs (clusters of two)
    const int crank = C::KS == 2 ? static_cast<int>(cluster_ctarank()) : 0;
    const int b0 = C::KS == 2 ? static_cast<int>(cluster_id_x()) : static_cast<int>(blockIdx.x);
    const int my_tiles = b0 < n_tiles
                             ? (n_tiles - 1 - b0) / static_cast<int>(C::KS == 2 ? cluster_count_x() : gridDim.x) + 1
                             : 0;
    // (the unit count is read where used, not held in a register)
    auto tile_of = [&](int i) { return b0 + i * static_cast<int>(C::KS == 2 ? cluster_count_x() : gridDim.x); };
    const int wbase = crank * C::NWC + warp;  // a compute warp's first window
    const bool xsend = C::KS == 2 && crank == 1;  // sends its sums instead of writing results
    const uint8_t* q = static_cast<const uint8_t*>(a.q);
    volatile int* abort_flag = &s_abort;
    // Wait for a pipeline barrier phase. The first test does not block and
    // does not read the shared abort flag; only a wait that has to block
    // checks it (a CTA whose waits already ran out stops waiting) and records
    // a timeout.
    auto pipe_wait = [&](uint64_t* bar, uint32_t parity) -> bool {
        if (mbar_test(bar, parity)) return true;
        if (*abort_flag) return false;
        if (mbar_wait<C::HINT>(bar, parity)) return true;
        atomicOr(&a.ws->error, kDevErrTimeout);
        *abort_flag = 1;
        return false;
    };

    // Issue the first P tiles' loads before anything else (compute warps; the
    // packed layout's producer issues its ring instead, below).
    TileBuf<FMT, K, MT> buf[P];
    if (!C::RING && warp < NW) {
#pragma unroll
        for (int p = 0; p < P; ++p)
            if (p < my_tiles) load_tile<FMT, K, MT>(buf[p], q, tile_of(p), wbase, g, t);
    }

    if (tid == 0) {
        for (int r = 0; r < RS; ++r) {
            mbar_init(&full_p[r], NW);
            mbar_init(&empty_p[r], C::NRW);
        }
        for (int r = 0; r < C::NSB; ++r) {
            mbar_init(&full_s[r], 1);
            mbar_init(&empty_s[r], NW);
        }
        if constexpr (C::KS == 2) {
            for (int r = 0; r < C::XS; ++r) {
                mbar_init(&xfull[r], 32 * C::NRW);
                mbar_init(&xempty[r], 32 * C::NRW);
            }
            mbar_init(amx_bar, 16);
        }
        s_abort = 0;
        mbar_init_fence();
    }
    __syncthreads();  // barriers initialised
    // K split: the partner's barriers are initialised before either CTA reaches
    // into the other's shared memory; every thread arrives here and waits
    // before its first access to the partner (reducer) or at the end
    if constexpr (C::KS == 2) cluster_arrive();
    // The loader's copies of ring slot i % SS (tile i of this CTA).
    const uint64_t pol = policy_evict_first();
    auto issue = [&](int i) {
        const int slot = i % C::SS;
        const size_t tile = static_cast<size_t>(tile_of(i));
        mbar_arrive_expect_tx(&full_s[slot], C::SLOT);
        bulk_g2s(s_dyn + slot * C::SLOT, a.sf + tile * C::SLOT, C::SLOT, &full_s[slot], pol);
    };
    // The producer's copy of tile i of this CTA into ring slot i % RT.
    auto issue_tile = [&](int i) {
        const int slot = i % RTm;
        mbar_arrive_expect_tx(&full_s[slot], C::TB);
        bulk_g2s(s_dyn + static_cast<size_t>(slot) * C::TB, q + static_cast<size_t>(tile_of(i)) * C::TB, C::TB,
                 &full_s[slot], pol);
    };
    int issued = 0;
    if (C::LOADER && warp == NW + C::NRW && lane == 0) {
        for (; issued < C::SS && issued < my_tiles; ++issued) issue(issued);
    }
    // The packed layout's producer issues its first tiles now: the head does
    // not depend on the preceding kernel, so these copies overlap its tail.
    if (C::RING && warp == NW + C::NRW && lane == 0) {
        for (; issued < cmin(C::RT, C::RPRE) && issued < my_tiles; ++issued) issue_tile(issued);
    }
    // The reducer warps start copying dh_idx for their tiles now: it belongs to
    // the head, so the copies overlap the preceding kernel's tail instead of
    // sitting on the reducer's path once the partials arrive.
    const int n_pre = (!xsend && (LOGITS || a.idx_ascending) && a.idx != nullptr &&
                       (reinterpret_cast<uintptr_t>(a.idx) & 15u) == 0)
                          ? (my_tiles < kIdCap ? my_tiles : kIdCap)
                          : 0;
    if (warp >= NW && warp < NW + C::NRW) {
        for (int c = (warp - NW) * 32 + lane; c < n_pre * 5; c += 32 * C::NRW) {
            const int i = c / 5, ch = c - 5 * i;  // 16-byte chunk ch of tile i: ids 16 tile + 4 ch ..
            const size_t e = static_cast<size_t>(tile_of(i)) * 16 + 4 * ch;
            if (e + 4 <= static_cast<size_t>(a.N)) cp_async16(&s_ids[20 * i + 4 * ch], a.idx + e);
        }
    }
    // Programmatic dependent launch: everything above only touched the head,
    // which the preceding kernel in the stream does not write; h, the
    // workspace and the outputs are used only after its completion.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    const uint32_t* h32 = reinterpret_cast<const uint32_t*>(a.h);

    if (C::RING && warp == NW + C::NRW) {
        // ------------------------------------------------------ producer ----
        // Refills a ring slot as soon as every compute warp has read it.
        if constexpr (C::RING) {
            if (lane == 0) {
                for (int i = issued; i < my_tiles; ++i) {
                    const int slot = i % RTm;
                    if (!pipe_wait(&empty_s[slot], ((i / RTm) - 1) & 1)) break;
                    issue_tile(i);
                    issued = i + 1;
                }
                if (*abort_flag) {  // let the copies already issued land before the CTA exits
                    for (int i = issued > RTm ? issued - RTm : 0; i < issued; ++i)
                        (void)mbar_wait<C::HINT>(&full_s[i % RTm], (i / RTm) & 1);
                }
            }
            __syncwarp();
        }
    } else if (warp == NW + C::NRW) {
        // -------------------------------------------------- scale loader ----
        // The 16 x K/16 scale bytes of a tile are contiguous (their per-row
        // 8-byte pieces would otherwise cost one L2 request per row and window).
        if constexpr (C::LOADER) {
            if (lane == 0) {
                for (int i = issued; i < my_tiles; ++i) {
                    const int slot = i % C::SS;
                    if (!mbar_wait<C::HINT>(&empty_s[slot], ((i / C::SS) - 1) & 1)) {
                        atomicOr(&a.ws->error, kDevErrTimeout);
                        *abort_flag = 1;
                    }
                    if (*abort_flag) break;
                    issue(i);
                    issued = i + 1;
                }
                if (*abort_flag) {  // let the copies already issued land before the CTA exits
                    for (int i = issued > C::SS ? issued - C::SS : 0; i < issued; ++i)
                        (void)mbar_wait<C::HINT>(&full_s[i % C::SS], (i / C::SS) & 1);
                }
            }
            __syncwarp();
        }
    } else if (warp >= NW) {
        // ------------------------------------------------------- reducer ----
        // Sums the NW partials of each tile in a fixed order and keeps the
        // best key per (row, draft), or writes the logits; never blocks the
        // compute warps except when it falls RS tiles behind.
        const int rl = (warp - NW) * 32 + lane;  // this reducer thread's first unit
        if (!LOGITS && rl == 0) s_epoch = load_epoch_dirty(a.ws);  // for the argmax hand-off
        cp_async_wait_all();  // this thread's dh_idx copies, then everyone's
        if constexpr (C::NRW > 1) named_bar_sync(1, 32 * C::NRW);
        else __syncwarp();
        for (int r = rl; r < NRED; r += 32 * C::NRW) s_best[r] = 0ull;
        const float gmul = (FMT == 3) ? 1.0f : __ldg(a.scale);
        constexpr int DV = C::DV;
        constexpr int UPR = MT / DV;                                    // units per row
        constexpr int NU = 16 * UPR;                                     // units per tile
        constexpr int SLOTS = (NU + 32 * C::NRW - 1) / (32 * C::NRW);  // units per reducer thread
        static_assert(C::KS == 1 || NU <= 32 * C::NRW, "K split: at most one unit per reducer thread");
        // K split: the logit of (tile row row_t, draft m0 + d), written or kept
        // as a key (the unsplit kernels do the same inline)
        auto emit = [&](int r0, int row_t, int m0, const float (&v)[DV], int id) {
            const int row = r0 + row_t;
            if (row >= a.n_kept) return;
#pragma unroll
            for (int d = 0; d < DV; ++d) {
                const int m = m0 + d;
                if (m >= a.M) break;
                if constexpr (LOGITS) {
                    // an id outside [0, V) is reported, not written
                    if (id >= 0 && id < a.V) a.out[static_cast<size_t>(m) * a.V + id] = v[d] * gmul;
                    else atomicOr(&a.ws->error, kDevErrIdx);
                } else {
                    // tie-break on the lower id (ascending dh_idx) or the lower row
                    const unsigned long long key = argmax_key(ordered_key(v[d] * gmul), static_cast<uint32_t>(id));
                    const int r = row_t * MT + m;
                    if (key > s_best[r]) s_best[r] = key;
                }
            }
        };
        // K split: wait for a barrier the partner arrives on (a CTA whose
        // waits already ran out stops waiting)
        auto xwait = [&](uint64_t* bar, uint32_t parity) {
            if (*abort_flag) return;
            if (!mbar_wait_cluster(bar, parity)) {
                atomicOr(&a.ws->error, kDevErrTimeout);
                *abort_flag = 1;
            }
        };
        // K split, first CTA: tile j's own sums wait (in this thread's place
        // of the exchange area's own-sum row) until the next tile's partials
        // are in; then the partner's sums of tile j (in flight meanwhile) are
        // added and the results written. Every reducer thread waits and
        // arrives; those with a unit (rl < NU) also read and write.
        float* const s_own = s_xb + C::XS * NRED;  // [unit][d], then the units' ids
        int* const s_ownid = reinterpret_cast<int*>(s_own + NRED);
        auto finish_prev = [&](int j) {
            const int xj = j % C::XS;
            xwait(&xfull[xj], (j / C::XS) & 1);
            if (rl < NU) {
                float v[DV];
#pragma unroll
                for (int d = 0; d < DV; ++d) v[d] = s_own[rl * DV + d] + s_xb[xj * NRED + rl * DV + d];
                emit(tile_of(j) * 16, rl / UPR, (rl % UPR) * DV, v, s_ownid[rl]);
            }
            if (j + C::XS < my_tiles) mbar_arrive_remote(cluster_map(&xempty[xj], 1));
        };
        if constexpr (C::KS == 2) cluster_wait();
        for (int i = 0; i < my_tiles; ++i) {
            const int slot = i % RS;
            const int tile = tile_of(i);
            // dh_idx of this tile's rows, fetched before waiting for the partials
            int ids_[SLOTS];
#pragma unroll
            for (int k = 0; k < SLOTS; ++k) {
                const int u = rl + k * 32 * C::NRW;
                const int row = tile * 16 + u / UPR;
                ids_[k] = (!xsend && (LOGITS || a.idx_ascending) && u < NU && row < a.n_kept)
                              ? (i < n_pre ? s_ids[20 * i + u / UPR] : (a.idx ? __ldg(a.idx + row) : row))
                              : row;
            }
            pipe_wait(&full_p[slot], (i / RS) & 1);
            const int xi = i % C::XS;
            if constexpr (C::KS == 2) {
                if (xsend) {
                    if (i >= C::XS) xwait(&xempty[xi], ((i / C::XS) - 1) & 1);  // the exchange slot is free
                } else if (i > 0) {
                    finish_prev(i - 1);
                }
            }
            const int r0 = tile * 16;
#pragma unroll
            for (int k = 0; k < SLOTS; ++k) {
                const int u = rl + k * 32 * C::NRW;
                if (u >= NU) break;
                const int row_t = u / UPR, m0 = (u % UPR) * DV;
                // fixed summation order over the warps, the same for every draft
                float v[DV];
#pragma unroll
                for (int d = 0; d < DV; ++d) v[d] = 0.0f;
                if constexpr (C::RED_T && NW % 4 == 0) {
                    // the row's NW partials are contiguous: four running sums, then a tree
                    const float4* pr = reinterpret_cast<const float4*>(part(slot, 0, row_t, 0));
                    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                    for (int w4 = 0; w4 < NW / 4; ++w4) {
                        const float4 q4 = pr[w4];
                        acc[0] += q4.x;
                        acc[1] += q4.y;
                        acc[2] += q4.z;
                        acc[3] += q4.w;
                    }
                    v[0] = (acc[0] + acc[1]) + (acc[2] + acc[3]);
                } else if constexpr (C::RED_T && NW % 2 == 0) {
                    // two running sums of float2 reads, then their sum
                    const float2* pr = reinterpret_cast<const float2*>(part(slot, 0, row_t, 0));
                    float acc[2] = {0.0f, 0.0f};
#pragma unroll
                    for (int w2 = 0; w2 < NW / 2; ++w2) {
                        const float2 q2 = pr[w2];
                        acc[0] += q2.x;
                        acc[1] += q2.y;
                    }
                    v[0] = acc[0] + acc[1];
                } else
#pragma unroll 4
                for (int w = 0; w < NW; ++w) {
                    if constexpr (DV == 4) {
                        const float4 q4 = *reinterpret_cast<const float4*>(part(slot, w, row_t, m0));
                        v[0] += q4.x;
                        v[1] += q4.y;
                        v[2] += q4.z;
                        v[3] += q4.w;
                    } else if constexpr (DV == 2) {
                        const float2 q2 = *reinterpret_cast<const float2*>(part(slot, w, row_t, m0));
                        v[0] += q2.x;
                        v[1] += q2.y;
                    } else {
                        v[0] += *part(slot, w, row_t, m0);
                    }
                }
                if constexpr (C::KS == 2) {
                    // this CTA's half of the K range: sent to the partner, or
                    // held until the partner's half of this tile is added
                    if (xsend) {
                        const uint32_t ra = cluster_map(&s_xb[xi * NRED + u * DV], 0);
                        if constexpr (DV == 2) st_cluster_f32x2(ra, v[0], v[1]);
                        else st_cluster_f32(ra, v[0]);
                    } else {
#pragma unroll
                        for (int d = 0; d < DV; ++d) s_own[u * DV + d] = v[d];
                        s_ownid[u] = ids_[k];
                    }
                } else {
                    const int row = r0 + row_t;
                    if (row >= a.n_kept) continue;
#pragma unroll
                    for (int d = 0; d < DV; ++d) {
                        const int m = m0 + d;
                        if (m >= a.M) break;
                        if constexpr (LOGITS) {
                            // an id outside [0, V) is reported, not written
                            const int id = ids_[k];
                            if (id >= 0 && id < a.V) a.out[static_cast<size_t>(m) * a.V + id] = v[d] * gmul;
                            else atomicOr(&a.ws->error, kDevErrIdx);
                        } else {
                            // tie-break on the lower id (ascending dh_idx) or the lower row
                            const unsigned long long key =
                                argmax_key(ordered_key(v[d] * gmul), static_cast<uint32_t>(ids_[k]));
                            const int r = row_t * MT + m;
                            if (key > s_best[r]) s_best[r] = key;
                        }
                    }
                }
            }
            if constexpr (C::KS == 2) {
                if (xsend) mbar_arrive_remote(cluster_map(&xfull[xi], 0));
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty_p[slot]);
        }
        if constexpr (C::KS == 2) {
            if (!xsend && my_tiles > 0) finish_prev(my_tiles - 1);
        }
        // K split: this thread's stores into the partner's shared memory and
        // arrivals on its barriers are complete before it passes the final
        // cluster barrier (the partner then exits)
        // (the first CTA reaches into the second only for the slots it frees
        // while more than XS tiles remain)
        if constexpr (C::KS == 2) {
            if (xsend || my_tiles > C::XS) cluster_fence();
        }
    } else {
        // -------------------------------------------------- compute warps ----
        // This thread's h words (B fragments), per window and n8 tile: word j
        // holds h[d][k0 + 2j], h[d][k0 + 2j + 1] with k0 = 128 w + 32 t and
        // d = g + 8 nt (d = 0 in the block-diagonal case, where the columns are
        // blocks). For the f16 MMAs, h is scaled by 2^e with e chosen per warp
        // and draft from the largest |h| over this warp's windows, so that every
        // BF16 value converts to f16 exactly; the warp's partial logits are
        // scaled back by 2^-e before they leave it.
        uint32_t hb[WPW][NT][16];
        float unscale[NT][2];  // 2^-e (W8A8: the activation scale) of the drafts of this thread's D columns
        if constexpr (C::W8A8) {
            // Per-token E4M3 codes of h: row max over the CTA's compute warps, then
            // word j of hb[ww][nt] = the codes of k0 + 4j .. k0 + 4j + 3.
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int d = g + 8 * nt;
                const bool live = d < a.M;
                float am = 0.0f;
#pragma unroll
                for (int ww = 0; ww < WPW; ++ww) {
                    const int k0 = 128 * (wbase + ww * NW) + 32 * t;
                    // the max |h| of this thread's 32 values (16-byte loads; the codes
                    // are made from a second read below): W8A8 4 drafts 42.3 -> 41.2 µs,
                    // 16 drafts 53.4 -> 50.6 µs against 4-byte loads
#pragma unroll
                    for (int j4 = 0; j4 < 4; ++j4) {
                        const uint4 v = live ? __ldg(reinterpret_cast<const uint4*>(h32 + d * KW + k0 / 2) + j4)
                                             : make_uint4(0u, 0u, 0u, 0u);
                        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                        for (int j = 0; j < 4; ++j) am = fmaxf(am, fmaxf(fabsf(bf16_lo(w4[j])), fabsf(bf16_hi(w4[j]))));
                    }
                }
                am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, 1));
                am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, 2));
                if (t == 0) s_amx[warp][d] = am;
            }
            named_bar_sync(2, NW * 32);  // compute warps only
            if constexpr (C::KS == 2) {
                // the per-token scale takes the max over the whole K range: each
                // CTA of the pair sends its max per draft to the other
                cluster_wait();  // the partner's barriers are initialised
                if (warp == 0 && lane < 16) {
                    float am = 0.0f;
                    for (int w2 = 0; w2 < NW; ++w2) am = fmaxf(am, s_amx[w2][lane]);
                    st_cluster_f32(cluster_map(&amx_rx[lane], crank ^ 1), am);
                    mbar_arrive_remote(cluster_map(amx_bar, crank ^ 1));
                    cluster_fence();
                }
                if (!*abort_flag && !mbar_wait_cluster(amx_bar, 0)) {
                    atomicOr(&a.ws->error, kDevErrTimeout);
                    *abort_flag = 1;
                }
            }
            float sx_own[NT];  // scale of this lane's draft g + 8 nt
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int d = g + 8 * nt;
                float am = 0.0f;
                for (int w2 = 0; w2 < NW; ++w2) am = fmaxf(am, s_amx[w2][d]);
                if constexpr (C::KS == 2) am = fmaxf(am, amx_rx[d]);
                sx_own[nt] = act_fp8_scale(am);
                unscale[nt][0] = __shfl_sync(0xFFFFFFFFu, sx_own[nt], 4 * (2 * t));
                unscale[nt][1] = __shfl_sync(0xFFFFFFFFu, sx_own[nt], 4 * (2 * t + 1));
#pragma unroll
                for (int ww = 0; ww < WPW; ++ww)
#pragma unroll
                    for (int j = 0; j < 8; ++j) hb[ww][nt][j] = 0u;
            }
            // The warp encodes each live draft together: lane l takes the 4 codes
            // of k = 128 w + 4 l .. 4 l + 3 (4 IEEE divisions instead of 32 per
            // lane and draft), then lane (g, t) collects words 8 t .. 8 t + 7 of
            // its own draft g + 8 nt.
#pragma unroll
            for (int d = 0; d < MT; ++d) {
                if (d >= a.M) break;
                const float sx = __shfl_sync(0xFFFFFFFFu, sx_own[d / 8], 4 * (d % 8));
#pragma unroll
                for (int ww = 0; ww < WPW; ++ww) {
                    const int kw = (128 * (wbase + ww * NW) + 4 * lane) / 2;  // u32 index of the lane's 4 values
                    const uint2 v2 = __ldg(reinterpret_cast<const uint2*>(h32 + d * KW + kw));
                    const uint32_t w0 = v2.x, w1 = v2.y;
                    const uint32_t word = act_fp8_pair(w0, sx) | (act_fp8_pair(w1, sx) << 16);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const uint32_t v = __shfl_sync(0xFFFFFFFFu, word, 8 * t + j);
                        if (g == d % 8) hb[ww][d / 8][j] = v;
                    }
                }
            }
        }
        uint2* s_hb = reinterpret_cast<uint2*>(s_dyn + (C::RING ? static_cast<size_t>(C::RT) * C::TB + C::PART_DYN : 0)) +
                      (C::SMB ? warp * WPW * NT * 8 * 32 : 0);  // [ww][nt][i][lane]
        if constexpr (C::W8A8 && C::SMB) {
            // the drafts' E4M3 codes (words 0..7 of hb) to shared memory
#pragma unroll
            for (int ww = 0; ww < WPW; ++ww)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        s_hb[((ww * NT + nt) * 8 + i) * 32 + lane] = make_uint2(hb[ww][nt][2 * i], hb[ww][nt][2 * i + 1]);
        }
#pragma unroll
        for (int nt = 0; nt < (C::W8A8 ? 0 : NT); ++nt) {
            const int d = C::BLOCKDIAG ? 0 : g + 8 * nt;
            const bool live = d < a.M;
            float am = 0.0f;
#pragma unroll
            for (int ww = 0; ww < WPW; ++ww) {
                const int k0 = 128 * (wbase + ww * NW) + 32 * t;
                if constexpr (!(MT == 1 && LOGITS)) {
                // 64 bytes of h per thread and window as four 16-byte loads (16 drafts:
                // 32.2 -> 28.5 µs per step, 4 drafts -0.3 µs; the one-draft
                // compute_logits kernel measured 0.7 µs slower with them and keeps
                // 4-byte loads)
#pragma unroll
                for (int j4 = 0; j4 < 4; ++j4) {
                    const uint4 v = live ? __ldg(reinterpret_cast<const uint4*>(h32 + d * KW + k0 / 2) + j4)
                                         : make_uint4(0u, 0u, 0u, 0u);
                    hb[ww][nt][4 * j4] = v.x;
                    hb[ww][nt][4 * j4 + 1] = v.y;
                    hb[ww][nt][4 * j4 + 2] = v.z;
                    hb[ww][nt][4 * j4 + 3] = v.w;
                }
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const uint32_t w = hb[ww][nt][j];
                    am = fmaxf(am, fmaxf(fabsf(bf16_lo(w)), fabsf(bf16_hi(w))));
                }
                } else {
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const uint32_t w = live ? __ldg(h32 + d * KW + k0 / 2 + j) : 0u;
                    hb[ww][nt][j] = w;
                    am = fmaxf(am, fmaxf(fabsf(bf16_lo(w)), fabsf(bf16_hi(w))));
                }
                }
            }
            // the 4 threads of a group (same g, so same draft) cover the window
            am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, 1));
            am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, 2));
            if constexpr (C::BLOCKDIAG) {
#pragma unroll
                for (int o = 4; o < 32; o <<= 1) am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, o));
            }
            const int e = (FMT == 3) ? 0 : f16_prescale_exponent(am);
            const float sc = exp2i(e);
            const float inv = exp2i(-e);
            if constexpr (FMT != 3) {
#pragma unroll
                for (int ww = 0; ww < WPW; ++ww)
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const uint32_t w = hb[ww][nt][j];
                        __half2 v = __floats2half2_rn(bf16_lo(w) * sc, bf16_hi(w) * sc);
                        hb[ww][nt][j] = *reinterpret_cast<uint32_t*>(&v);
                    }
            }
            if constexpr (C::SMB) {
                // to shared memory as soon as they are made
#pragma unroll
                for (int ww = 0; ww < WPW; ++ww)
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        s_hb[((ww * NT + nt) * 8 + i) * 32 + lane] = make_uint2(hb[ww][nt][2 * i], hb[ww][nt][2 * i + 1]);
            }
            if constexpr (C::BLOCKDIAG) {
                unscale[nt][0] = inv;
                unscale[nt][1] = inv;
#pragma unroll
                for (int ww = 0; ww < WPW; ++ww)
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        // slot pair p (block pi(p)) feeds D column pi(p): b0 of MMA i
                        // (pair t, block 2t) is nonzero only in column g == 2t, b1 (pair
                        // t + 4, block 2t + 1) only in column g == 2t + 1
                        const bool keep = (j < 8) ? (g == 2 * t) : (g == 2 * t + 1);
                        hb[ww][nt][j] = keep ? hb[ww][nt][j] : 0u;
                    }
            } else {
                // D columns 2t, 2t+1 hold drafts 8 nt + 2t (+1), whose scale lives
                // in the lanes of group g = 2t (+1)
                unscale[nt][0] = __shfl_sync(0xFFFFFFFFu, inv, 4 * (2 * t));
                unscale[nt][1] = __shfl_sync(0xFFFFFFFFu, inv, 4 * (2 * t + 1));
            }
        }
        if constexpr (C::SMB) __syncwarp();
        // Tile i's codes and scales into registers: from the ring (packed
        // layout: wait until the tile has landed, read this warp's windows,
        // free the slot) or with global loads.
        auto fetch = [&](TileBuf<FMT, K, MT>& b, int i) {
            if constexpr (C::RING) {
                const int rs = i % RTm;
                pipe_wait(&full_s[rs], (i / RTm) & 1);
                const uint8_t* tl = s_dyn + static_cast<size_t>(rs) * C::TB;
#pragma unroll
                for (int ww = 0; ww < WPW; ++ww) {
                    const uint8_t* blk = tl + (wbase + ww * NW) * C::WBLK;
                    b.c[ww][0][0] = *reinterpret_cast<const uint4*>(blk + g * 64 + 16 * t);
                    b.c[ww][1][0] = *reinterpret_cast<const uint4*>(blk + (g + 8) * 64 + 16 * t);
                    b.sp[ww] = *reinterpret_cast<const uint32_t*>(blk + 16 * 64 + 4 * lane);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty_s[rs]);
            } else {
                load_tile<FMT, K, MT>(b, q, tile_of(i), wbase, g, t);
            }
        };
        // Ring kernels with two windows per warp and n8 tiles of drafts: each
        // window's codes and scales are read from the ring just before its
        // math, not a tile ahead (one window's registers held instead of two:
        // the two-window h fragments leave no room at 80 registers)
        constexpr bool JIT = C::RING && WPW > 1 && !C::BLOCKDIAG;
        if constexpr (C::RING && !JIT) {
#pragma unroll
            for (int p = 0; p < P; ++p)
                if (p < my_tiles) fetch(buf[p], p);
        }
        // Hand tile ti's partial sums to the reducer (wait for the slot to be
        // free first).
        auto handoff = [&](int ti, const float (&out)[NT][4]) {
            const int slot = ti % RS;
            if (ti >= RS) pipe_wait(&empty_p[slot], ((ti / RS) - 1) & 1);
            if constexpr (C::BLOCKDIAG) {
                if (t == 0) {
                    *part(slot, warp, g, 0) = out[0][0] * unscale[0][0];
                    *part(slot, warp, g + 8, 0) = out[0][1] * unscale[0][0];
                }
            } else {
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const int m0 = 8 * nt + 2 * t;
                    if (m0 < MT) {
                        *part(slot, warp, g, m0) = out[nt][0] * unscale[nt][0];
                        *part(slot, warp, g + 8, m0) = out[nt][2] * unscale[nt][0];
                    }
                    if (m0 + 1 < MT) {
                        *part(slot, warp, g, m0 + 1) = out[nt][1] * unscale[nt][1];
                        *part(slot, warp, g + 8, m0 + 1) = out[nt][3] * unscale[nt][1];
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&full_p[slot]);
        };
        // Per tile: math, the loads (ring reads) P tiles ahead, hand-off.
        for (int it = 0; it < my_tiles; it += P) {
#pragma unroll
            for (int p = 0; p < P; ++p) {
                const int ti = it + p;
                if (ti >= my_tiles) break;
                TileBuf<FMT, K, MT>& b = buf[p];
                float out[NT][4];  // block-diagonal: out[0][0..1] = rows g, g+8
                const int rs = ti % RTm;  // ring slot of this tile
                if constexpr (JIT) pipe_wait(&full_s[rs], (ti / RTm) & 1);

                if constexpr (C::SCALES) {
                    const int ss = ti % C::SS;
                    pipe_wait(&full_s[ss], (ti / C::SS) & 1);
                    const uint8_t* st = s_dyn + ss * C::SLOT;
#pragma unroll
                    for (int ww = 0; ww < WPW; ++ww) {
                        const int w = wbase + ww * NW;
                        b.s[ww][0] = *reinterpret_cast<const uint2*>(st + g * C::SFB + 8 * w);
                        b.s[ww][1] = *reinterpret_cast<const uint2*>(st + (g + 8) * C::SFB + 8 * w);
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty_s[ss]);
                }
                if constexpr (C::BLOCKDIAG) {
                    float y0 = 0.0f, y1 = 0.0f;
#pragma unroll
                    for (int ww = 0; ww < WPW; ++ww) {
                        // two accumulators (one per half), summed at the end
                        float dc[2][4] = {{0.0f, 0.0f, 0.0f, 0.0f}, {0.0f, 0.0f, 0.0f, 0.0f}};
                        // MMA i takes byte i (block 2t) and byte 8+i (block 2t+1) of each
                        // row: words (0, 2) feed i < 4, words (1, 3) feed i >= 4.
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
                                mma_f16(dc[half], fg0[j], fh0[j], fg1[j], fh1[j], hb[ww][0][i],
                                        hb[ww][0][8 + i]);
                            }
                        }
                        float d[4];
#pragma unroll
                        for (int c = 0; c < 4; ++c) d[c] = dc[0][c] + dc[1][c];

                        // scales of blocks 2t, 2t+1 (this thread's D columns) of rows g, g+8
                        uint32_t s01g, s01h;
                        if constexpr (C::PACKED) {
                            s01g = b.sp[ww];
                            s01h = b.sp[ww] >> 16;
                        } else {
                            const uint32_t sel = static_cast<uint32_t>(2 * t) | (static_cast<uint32_t>(2 * t + 1) << 4);
                            asm("prmt.b32 %0, %1, %2, %3;" : "=r"(s01g) : "r"(b.s[ww][0].x), "r"(b.s[ww][0].y), "r"(sel));
                            asm("prmt.b32 %0, %1, %2, %3;" : "=r"(s01h) : "r"(b.s[ww][1].x), "r"(b.s[ww][1].y), "r"(sel));
                        }
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
                    out[0][0] = y0;
                    out[0][1] = y1;
                } else {
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                        for (int c = 0; c < 4; ++c) out[nt][c] = 0.0f;
                    if constexpr (C::W8A8) {
                        // MMA i: A words 2i (k 8i..8i+3 of the thread's 32) and 2i+1
                        // (k 8i+4..8i+7) of rows g, g+8; B the same k of the drafts' codes
#pragma unroll
                        for (int ww = 0; ww < WPW; ++ww)
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                const uint32_t a0 = word_of<C::CPR>(b.c[ww][0], 2 * i);
                                const uint32_t a1 = word_of<C::CPR>(b.c[ww][1], 2 * i);
                                const uint32_t a2 = word_of<C::CPR>(b.c[ww][0], 2 * i + 1);
                                const uint32_t a3 = word_of<C::CPR>(b.c[ww][1], 2 * i + 1);
#pragma unroll
                                for (int nt = 0; nt < NT; ++nt) {
                                    if constexpr (C::SMB) {
                                        const uint2 bb = s_hb[((ww * NT + nt) * 8 + i) * 32 + lane];
                                        mma_e4m3(out[nt], a0, a1, a2, a3, bb.x, bb.y);
                                    } else {
                                        mma_e4m3(out[nt], a0, a1, a2, a3, hb[ww][nt][2 * i], hb[ww][nt][2 * i + 1]);
                                    }
                                }
                            }
                    }
#pragma unroll
                    for (int ww = 0; ww < (C::W8A8 ? 0 : WPW); ++ww) {
                        if constexpr (JIT) {
                            const uint8_t* blk = s_dyn + static_cast<size_t>(rs) * C::TB + (wbase + ww * NW) * C::WBLK;
                            b.c[ww][0][0] = lds_v4_ordered(blk + g * 64 + 16 * t);
                            b.c[ww][1][0] = lds_v4_ordered(blk + (g + 8) * 64 + 16 * t);
                            b.sp[ww] = lds_u32_ordered(blk + 16 * 64 + 4 * lane);
                        }
                        uint32_t sg0 = 0u, sg1 = 0u, sh0 = 0u, sh1 = 0u;  // (s, s) f16x2 per row and block
                        if constexpr (C::NV) {
                            // blocks 2t, 2t+1 of the window: bytes 2t, 2t+1 of its 8 scale bytes
                            uint32_t s2g, s2h;
                            if constexpr (C::PACKED) {
                                s2g = b.sp[ww];
                                s2h = b.sp[ww] >> 16;
                            } else {
                                const uint32_t sel = static_cast<uint32_t>(2 * t) | (static_cast<uint32_t>(2 * t + 1) << 4);
                                asm("prmt.b32 %0, %1, %2, %3;" : "=r"(s2g) : "r"(b.s[ww][0].x), "r"(b.s[ww][0].y), "r"(sel));
                                asm("prmt.b32 %0, %1, %2, %3;" : "=r"(s2h) : "r"(b.s[ww][1].x), "r"(b.s[ww][1].y), "r"(sel));
                            }
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
                            if constexpr (C::NV) {
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
                                uint32_t a0 = 0u, a1 = 0u, a2 = 0u, a3 = 0u;
                                if constexpr (C::NV) {
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
                                } else if constexpr (FMT == 3) {
                                    a0 = word_of<C::CPR>(b.c[ww][0], 2 * i);
                                    a1 = word_of<C::CPR>(b.c[ww][1], 2 * i);
                                    a2 = word_of<C::CPR>(b.c[ww][0], 2 * i + 1);
                                    a3 = word_of<C::CPR>(b.c[ww][1], 2 * i + 1);
                                }
#pragma unroll
                                for (int nt = 0; nt < NT; ++nt) {
                                    if constexpr (FMT == 3) {
                                        if constexpr (C::SMB) {
                                            const uint2 bb = s_hb[((ww * NT + nt) * 8 + i) * 32 + lane];
                                            mma_bf16(out[nt], a0, a1, a2, a3, bb.x, bb.y);
                                        } else {
                                            mma_bf16(out[nt], a0, a1, a2, a3, hb[ww][nt][2 * i], hb[ww][nt][2 * i + 1]);
                                        }
                                    } else
                                        if constexpr (C::SMB) {
                                            const uint2 bb = s_hb[((ww * NT + nt) * 8 + i) * 32 + lane];
                                            mma_f16(out[nt], a0, a1, a2, a3, bb.x, bb.y);
                                        } else {
                                            mma_f16(out[nt], a0, a1, a2, a3, hb[ww][nt][2 * i], hb[ww][nt][2 * i + 1]);
                                        }
                                }
                            }
                        }
                    }
                }
                if constexpr (JIT) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty_s[rs]);  // this warp is done with the slot
                } else {
                    // loads of the tile P steps ahead go into the buffer just consumed
                    const int tn = ti + P;
                    if (tn < my_tiles) fetch(buf[p], tn);
                }
                handoff(ti, out);
            }
        }
    }
    // with the K split, neither CTA of a pair exits while the other may still
    // reach into its shared memory
    if constexpr (C::KS == 2) {
        __syncwarp();
        // compute warps: the wait of the arrival at the start (W8A8: made in the prologue)
        if (!C::W8A8 && warp < NW) cluster_wait();
        cluster_sync_all();
    } else {
        __syncthreads();
    }
    if constexpr (!LOGITS) {
        if (tid < MT) {
            unsigned long long k = 0ull;
            for (int row_t = 0; row_t < 16; ++row_t) {
                const unsigned long long v = s_best[row_t * MT + tid];
                k = v > k ? v : k;
            }
            s_cta[tid] = k;
        }
        __syncthreads();
        finish_argmax(a, s_cta, s_epoch.x, s_epoch.y);
    }
}

template <int FMT, int K, int MT, bool LOGITS>
inline cudaError_t launch_mma(const GemvArgs& a, cudaStream_t s) {
    using C = Cfg<FMT, K, MT, LOGITS>;
    auto kern = gemv_mma_kernel<FMT, K, MT, LOGITS>;
    const int sms = sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    const size_t smem = C::DYN_SMEM;
    // CTAs per SM, looked up once per device (first callers on several host
    // threads may each look it up; they store the same value)
    static std::atomic<int> occ[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(C::KS);
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = C::KS;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = C::KS == 2 ? 2 : 1;
    // resident CTAs: per SM x SMs, or with the K split 2 x the pairs that fit
    int resident = occ[dev].load(std::memory_order_relaxed);
    if (resident == 0) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e != cudaSuccess) return e;
        int o = 0;
        if constexpr (C::KS == 2) {
            e = cudaOccupancyMaxActiveClusters(&o, kern, &cfg);
            if (e != cudaSuccess) return e;
            if (o <= 0) return cudaErrorInvalidConfiguration;
            resident = C::KS * o;
        } else {
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, kern, C::THREADS, smem);
            if (e != cudaSuccess) return e;
            resident = sms * (o > 0 ? o : 1);
        }
        occ[dev].store(resident, std::memory_order_relaxed);
    }
    const int n_tiles = a.N / 16;
    int units = resident / C::KS;  // CTAs, or pairs
    if (units > n_tiles) units = n_tiles;
    if (units > (n_tiles + C::MIN_TILES - 1) / C::MIN_TILES) units = (n_tiles + C::MIN_TILES - 1) / C::MIN_TILES;
    if (units * C::KS > kMaxGrid) units = kMaxGrid / C::KS;  // one argmax slot per CTA
    cfg.gridDim = dim3(units * C::KS);
    e = cudaLaunchKernelEx(&cfg, kern, a);
    if (e != cudaSuccess) return e;
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

// Register-load kernels for 5 to 16 drafts only, at the widths where the ring
// kernels take every launch of up to 4 drafts (packed_use_ring).
template <int FMT, int K, bool LOGITS>
inline cudaError_t launch_mma_m_wide(const GemvArgs& a, cudaStream_t s) {
    if (a.M <= 4) return cudaErrorInvalidValue;
    if (a.M <= 8) return launch_mma<FMT, K, 8, LOGITS>(a, s);
    return launch_mma<FMT, K, 16, LOGITS>(a, s);
}

template <int FMT, int K>
inline cudaError_t launch_mma_k(const GemvArgs& a, cudaStream_t s) {
    return a.out ? launch_mma_m<FMT, K, true>(a, s) : launch_mma_m<FMT, K, false>(a, s);
}

// The ring kernels of the packed head, up to four drafts.
template <int K>
inline cudaError_t launch_ring_k(const GemvArgs& a, cudaStream_t s) {
    if (a.out) {
        if (a.M <= 1) return launch_mma<kFmtPackedRing, K, 1, true>(a, s);
        if (a.M <= 2) return launch_mma<kFmtPackedRing, K, 2, true>(a, s);
        if constexpr (K == 2560) {
            if (a.M > 4) return launch_mma<kFmtPackedRing, K, 8, true>(a, s);  // compute_logits only
        }
        return launch_mma<kFmtPackedRing, K, 4, true>(a, s);
    }
    if (a.M <= 1) return launch_mma<kFmtPackedRing, K, 1, false>(a, s);
    if (a.M <= 2) return launch_mma<kFmtPackedRing, K, 2, false>(a, s);
    return launch_mma<kFmtPackedRing, K, 4, false>(a, s);
}

// Packed head: the ring kernel for up to four drafts (eight for compute_logits
// at K = 2560), K >= 2560, on heads of at least eight tiles per SM or K >= 4096
// (one draft, 64,064 x 2560: 19.8 -> 16.9 µs; 4 drafts 21.4 -> 20.4); register
// loads otherwise (top tokens at 8 drafts and 16 drafts, where the ring
// measured 1.2 and 2.5 µs slower; the 4,032 x 256 head; the 1,024 - 4,608-row
// linears at K <= 2560).
inline bool packed_use_ring(const GemvArgs& a) {
    return (a.M <= 4 || (a.M <= 8 && a.K == 2560 && a.out != nullptr)) && a.K >= 2560 &&
           (a.N / 16 >= 8 * sm_count() || a.K >= 4096);
}

}  // namespace mma
}  // namespace dh

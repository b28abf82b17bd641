// Device helpers shared by the draft-head kernels (CUDA side only).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

namespace dh {

// CTAs a draft-step launch may use (the launcher caps its grid here).
constexpr int kMaxGrid = 1024;

// Layout of a workspace (callers allocate it). The quantisers use only the
// 256-byte header; a draft step also uses the epoch, the dirty word and the
// argmax slots. Draft steps alternate between two banks of slots (bank = epoch
// & 1). The collecting CTA zeroes every slot it read and advances the epoch; a
// slot written after its collector gave up waiting lands in a bank that the
// next step does not use, and that step zeroes it (see the dirty word) before
// the bank comes round again.
struct Workspace {
    unsigned int error;      // DH_DEVERR_* bits
    unsigned int amax_bits;  // quantisers: running max |w| as float bits
    unsigned int epoch;      // draft steps collected on this workspace
    unsigned int dirty;      // 0, or 1 | bank << 1 | drafts << 2 | CTAs << 8 of a step whose wait ran out
    unsigned int pad_[60];
    // per bank, draft and CTA: the CTA's best (ordered logit << 32 | ~id or
    // ~row) key, or 1 when it holds no kept row; 0 while not yet published
    unsigned long long slots[2][16][kMaxGrid];
};
constexpr size_t kWorkspaceHeader = 256;
static_assert(offsetof(Workspace, slots) == kWorkspaceHeader, "workspace header is 256 bytes");
static_assert(offsetof(Workspace, epoch) % 8 == 0 && offsetof(Workspace, dirty) == offsetof(Workspace, epoch) + 4,
              "epoch and dirty are read together");

constexpr unsigned int kDevErrIdx = 1u;

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Order-preserving map of a float to uint32: a < b  <=>  ord(a) < ord(b).
// -0 is folded onto +0 and every NaN onto the largest key, so that, like
// torch.argmax, a NaN wins and equal values tie.
__device__ __forceinline__ uint32_t ordered_key(float v) {
    uint32_t u = __float_as_uint(v);
    if (v != v) return 0xFFFFFFFFu;
    if (v == 0.0f) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float ordered_value(uint32_t k) {
    if (k == 0xFFFFFFFFu) return __uint_as_float(0x7FC00000u);
    uint32_t u = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
    return __uint_as_float(u);
}

// 64-bit argmax key: larger logit first, then the lower row.
__device__ __forceinline__ unsigned long long argmax_key(uint32_t ord, uint32_t row) {
    return (static_cast<unsigned long long>(ord) << 32) | (0xFFFFFFFFu - row);
}

// Streaming 16-byte load that does not allocate in L1 (the head is read once).
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}

__device__ __forceinline__ uint32_t ld_stream_u16(const void* p) {
    unsigned short r;
    asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(r) : "l"(p));
    return r;
}

// Four E2M1 pairs (one 32-bit word, 8 codes) to four f16x2: byte i -> out[i],
// low nibble -> low half. Exact: every E2M1 value is an f16.
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t w, uint32_t (&o)[4]) {
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "mov.b32 {b0, b1, b2, b3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
        : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3]) : "r"(w));
}

// f16x2 product (exact for an E2M1 code times an E4M3 scale).
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// Two E4M3 bytes (low 16 bits of w) to f16x2, low byte -> low half. Exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t w) {
    uint32_t r;
    asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}"
        : "=r"(r) : "r"(w));
    return r;
}

__device__ __forceinline__ float f16lo(uint32_t x) { return __half2float(__ushort_as_half((unsigned short)(x & 0xFFFFu))); }
__device__ __forceinline__ float f16hi(uint32_t x) { return __half2float(__ushort_as_half((unsigned short)(x >> 16))); }

// acc += a.lo * b.lo + a.hi * b.hi with f16 operands and an fp32 accumulator
// (each product is exact in fp32; two roundings of the running sum).
__device__ __forceinline__ float fma2_f16_f32(uint32_t a, uint32_t b, float acc) {
    asm("{\n\t.reg .f16 a0, a1, b0, b1;\n\t"
        "mov.b32 {a0, a1}, %1;\n\tmov.b32 {b0, b1}, %2;\n\t"
        "fma.rn.f32.f16 %0, a0, b0, %0;\n\tfma.rn.f32.f16 %0, a1, b1, %0;\n\t}"
        : "+f"(acc) : "r"(a), "r"(b));
    return acc;
}

// Same with BF16 operands.
__device__ __forceinline__ float fma2_bf16_f32(uint32_t a, uint32_t b, float acc) {
    asm("{\n\t.reg .b16 a0, a1, b0, b1;\n\t"
        "mov.b32 {a0, a1}, %1;\n\tmov.b32 {b0, b1}, %2;\n\t"
        "fma.rn.f32.bf16 %0, a0, b0, %0;\n\tfma.rn.f32.bf16 %0, a1, b1, %0;\n\t}"
        : "+f"(acc) : "r"(a), "r"(b));
    return acc;
}

// Per-token dynamic FP8 quantisation of hidden states, the activation half of
// the W8A8 head ("FP8 MTP draft stack for vLLM ...", _Fp8DraftHeadMethod.apply:
// scaled_fp8_quant(x, use_per_token_if_dynamic=True)). A row's scale is its
// max |h| clamped below at 1e-12, divided by 448 (IEEE division).
__device__ __forceinline__ float act_fp8_scale(float amax) {
    return __fdiv_rn(amax < 1e-12f ? 1e-12f : amax, 448.0f);
}

// E4M3 codes of the two BF16 values of w (low half -> low byte):
// E4M3_RNE(clamp(h / s, +-448)), the division IEEE round-to-nearest.
__device__ __forceinline__ uint32_t act_fp8_pair(uint32_t w, float s) {
    const float lo = fminf(fmaxf(__fdiv_rn(bf16_lo(w), s), -448.0f), 448.0f);
    const float hi = fminf(fmaxf(__fdiv_rn(bf16_hi(w), s), -448.0f), 448.0f);
    return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3));
}

// Power of two 2^e with e clamped to the normal float range.
__device__ __forceinline__ float exp2i(int e) {
    e = e < -126 ? -126 : (e > 127 ? 127 : e);
    return __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
}

// Exponent e such that amax * 2^e lies in [2^14, 2^15): the largest |h| then
// sits just under the f16 maximum and every BF16 value at most 2^24 times
// smaller converts to f16 exactly (BF16 has 8 significant bits, f16 11).
__device__ __forceinline__ int f16_prescale_exponent(float amax) {
    if (!(amax > 0.0f)) return 0;
    // floor(log2 amax) for a normal amax; a subnormal amax reads as -127 and
    // the resulting large exponent is clamped by exp2i.
    const int E = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFF) - 127;
    return 14 - E;
}

}  // namespace dh

// ------------------------------------------------------------------------
// Shared-memory pipeline primitives: mbarriers and 1-D bulk async copies
// (cp.async.bulk, the non-tensor TMA path). Every wait is bounded.
// ------------------------------------------------------------------------
namespace dh {

constexpr unsigned int kDevErrTimeout = 2u;   // a bounded pipeline wait gave up
constexpr uint32_t kWaitLimit = 1u << 22;     // try_wait rounds before giving up
constexpr uint32_t kSuspendNs = 1000;         // suspend-time hint of a try_wait round (ns)

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make barrier initialisation visible to the other threads and the async proxy.
__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;\n\tfence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 :: "r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(smem_u32(bar)) : "memory");
}

// Wait for the phase with the given parity to complete; false after `limit`
// rounds. HINT: each try_wait round suspends for at most kSuspendNs, so that
// `limit` rounds take a known time (kWaitLimit rounds ~ 4 s); without it a
// round lasts a system-dependent time. (Measured: the hinted form is faster in
// the one- and two-draft kernels, the plain form at 4 drafts and more.)
template <bool HINT = true>
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t limit = kWaitLimit) {
    const uint32_t a = smem_u32(bar);
    for (uint32_t i = 0; i < limit; ++i) {
        uint32_t done;
        if constexpr (HINT) {
            asm volatile("{\n\t.reg .pred p;\n\t"
                         "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
                         "selp.u32 %0, 1, 0, p;\n\t}"
                         : "=r"(done) : "r"(a), "r"(parity), "n"(kSuspendNs) : "memory");
        } else {
            asm volatile("{\n\t.reg .pred p;\n\t"
                         "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                         "selp.u32 %0, 1, 0, p;\n\t}"
                         : "=r"(done) : "r"(a), "r"(parity) : "memory");
        }
        if (done) return true;
    }
    return false;
}

// Non-blocking test of the phase with the given parity: true if it completed.
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(done) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return done != 0;
}

// Poll a 64-bit word in global memory (relaxed, device scope) until it is
// non-zero; returns it, or 0 after `limit` polls.
__device__ __forceinline__ unsigned long long poll_nonzero(const unsigned long long* p, uint32_t limit = kWaitLimit) {
    unsigned long long v = 0ull;
    for (uint32_t n = 0; n < limit; ++n) {
        asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
        if (v != 0ull) break;
    }
    return v;
}

// Bulk copy global -> this CTA's shared memory, completing `bytes` on `bar`.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
                 " [%0], [%1], %2, [%3], %4;"
                 :: "r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
                 : "memory");
}

// 16-byte asynchronous copy global -> shared (both 16-byte aligned), tracked
// per thread: cp_async_wait_all() returns once this thread's copies landed.
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(smem_u32(dst)), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.wait_all;" ::: "memory");
}

// L2 policy for data read once per step (the head): evict first.
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ------------------------------------------------------------------------
// Thread-block clusters of two CTAs: distributed shared memory between the
// CTAs of a pair (the partner's address of a shared variable, stores to it,
// arrivals on its mbarriers) and the cluster-wide barrier.
// ------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_id_x() {
    uint32_t r;
    asm("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}

__device__ __forceinline__ uint32_t cluster_count_x() {
    uint32_t r;
    asm("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}

// The shared::cluster address of `p` (a variable of this CTA) in CTA `rank`.
__device__ __forceinline__ uint32_t cluster_map(const void* p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}

__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float x) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" :: "r"(addr), "f"(x) : "memory");
}

__device__ __forceinline__ void st_cluster_f32x2(uint32_t addr, float x, float y) {
    asm volatile("st.shared::cluster.v2.f32 [%0], {%1, %2};" :: "r"(addr), "f"(x), "f"(y) : "memory");
}

// Arrive on an mbarrier of another CTA of the cluster (address from
// cluster_map), releasing this thread's earlier writes at cluster scope.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t bar) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" :: "r"(bar) : "memory");
}

// Bounded wait on a local mbarrier that another CTA of the cluster arrives on
// (acquire at cluster scope: its writes released by the arrivals are visible).
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, uint32_t limit = kWaitLimit) {
    const uint32_t a = smem_u32(bar);
    for (uint32_t i = 0; i < limit; ++i) {
        uint32_t done;
        asm volatile("{\n\t.reg .pred p;\n\t"
                     "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
                     "selp.u32 %0, 1, 0, p;\n\t}"
                     : "=r"(done) : "r"(a), "r"(parity), "n"(kSuspendNs) : "memory");
        if (done) return true;
    }
    return false;
}

// Every thread of every CTA of the cluster: a hardware barrier (no spin loop
// of ours). The arrival is relaxed: it does not wait for this thread's loads
// and stores in flight (a released arrival would hold the CTA until its tile
// loads or its result stores have landed); a thread whose remote accesses
// must be complete before the others pass calls cluster_fence() first.
__device__ __forceinline__ void cluster_arrive() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait() {
    asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

__device__ __forceinline__ void cluster_sync_all() {
    cluster_arrive();
    cluster_wait();
}

// This thread's earlier memory accesses, remote ones included, are performed
// at cluster scope before its later ones.
__device__ __forceinline__ void cluster_fence() {
    asm volatile("fence.acq_rel.cluster;" ::: "memory");
}

// Named barrier among `threads` threads (id 1..15; id 0 is __syncthreads).
__device__ __forceinline__ void named_bar_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(threads) : "memory");
}

}  // namespace dh

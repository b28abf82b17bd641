// Draft-step dispatch: format and hidden size -> kernel instantiation (one
// translation unit per head format, see dh_gemv_mma.cuh), plus the -inf fill
// of compute_logits.
#include "dh_common.cuh"
#include "dh_internal.h"

namespace dh {

cudaError_t launch_gemv_nvfp4(const GemvArgs& a, cudaStream_t s);
cudaError_t launch_gemv_fp8(const GemvArgs& a, cudaStream_t s);
cudaError_t launch_gemv_bf16(const GemvArgs& a, cudaStream_t s);
cudaError_t launch_gemv_nvfp4_packed(const GemvArgs& a, cudaStream_t s);
cudaError_t launch_gemv_fp8_w8a8(const GemvArgs& a, cudaStream_t s);
bool linear_extra_k(int K);
cudaError_t launch_linear_nvfp4_packed_extra(const GemvArgs& a, cudaStream_t s);

__global__ void fill_neg_inf_kernel(float4* out4, size_t n4, float* tail, int ntail) {
    // The GEMV launched next (programmatic stream serialisation) may start streaming
    // the head now; it waits for this grid to complete before it touches `out`
    // (compute_logits 16 drafts 30.6 -> 29.2 µs, one draft 22.0 -> 21.8 µs).
    asm volatile("griddepcontrol.launch_dependents;");
    // This grid is itself launched early (while the preceding kernel in the
    // stream, e.g. the previous step's GEMV, finishes); `out` is written only
    // once that kernel has completed and its writes are visible.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const float ninf = __uint_as_float(0xFF800000u);
    const float4 v = make_float4(ninf, ninf, ninf, ninf);
    for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n4;
         i += static_cast<size_t>(gridDim.x) * blockDim.x)
        out4[i] = v;
    if (blockIdx.x == 0 && threadIdx.x < ntail) tail[threadIdx.x] = ninf;
}


// Shard keys -> ids ("q38_draft.py", install: the local-argmax reduction ends
// with the winning id). The key's sign bit was flipped so that signed order
// equals the unsigned order of (ordered logit << 32 | ~id).
__global__ void keys_to_ids_kernel(const unsigned long long* keys, int M, int32_t* ids, float* top) {
    const int m = threadIdx.x;
    if (m >= M) return;
    const unsigned long long k = keys[m] ^ 0x8000000000000000ull;
    ids[m] = k == 0ull ? -1 : static_cast<int32_t>(0xFFFFFFFFu - static_cast<uint32_t>(k & 0xFFFFFFFFull));
    if (top) top[m] = k == 0ull ? __uint_as_float(0x7FC00000u) : ordered_value(static_cast<uint32_t>(k >> 32));
}

cudaError_t launch_keys_to_ids(const unsigned long long* keys, int M, int32_t* ids, float* top, cudaStream_t s) {
    keys_to_ids_kernel<<<1, 32, 0, s>>>(keys, M, ids, top);
    return cudaGetLastError();
}

// Hidden rows from page-locked host memory into the workspace staging area,
// 16 bytes per thread (a draft step's rows: M x K x 2 <= 16 x 5120 x 2 bytes).
// The loads are issued before the grid-dependency wait (the host wrote the
// rows before the call), the stores after it. The draft step launched next
// may start at once (it reads the staging area only after this grid has
// completed): end to end 18.86 -> 18.27 µs a step against a release after
// the stores.
__global__ void __launch_bounds__(1024) stage_rows_kernel(const uint4* src, uint4* dst, int n16) {
    constexpr int kPer = 10;  // 16-byte pieces per thread: 1024 x 10 x 16 = 160 KB
    asm volatile("griddepcontrol.launch_dependents;");
    uint4 v[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        const int i = threadIdx.x + j * blockDim.x;
        if (i < n16) v[j] = src[i];
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
        const int i = threadIdx.x + j * blockDim.x;
        if (i < n16) dst[i] = v[j];
    }
}

cudaError_t launch_stage_rows(const void* src_host, void* dst, size_t bytes, cudaStream_t s) {
    const int n16 = static_cast<int>(bytes / 16);
    if (bytes % 16 != 0 || n16 > 1024 * 10) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(n16 < 1024 ? ((n16 + 31) / 32) * 32 : 1024);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, stage_rows_kernel, static_cast<const uint4*>(src_host),
                                       static_cast<uint4*>(dst), n16);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// Self-test of the bounded waits: wait for an event that never happens (kind
// 0: a workspace word nothing writes, polled like the argmax hand-off's slots;
// kind 1: an mbarrier nothing arrives on, waited on like the pipeline's), give
// up after `rounds` and record DH_DEVERR_TIMEOUT, as the draft step does.
__global__ void wait_probe_kernel(Workspace* ws, int kind, uint32_t rounds) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    bool ok;
    if (kind == 0) {
        const unsigned long long* never = reinterpret_cast<const unsigned long long*>(&ws->pad_[0]);
        ok = poll_nonzero(never, rounds) != 0ull;
    } else {
        mbar_init(&bar, 1);
        mbar_init_fence();
        ok = mbar_wait(&bar, 0, rounds);
    }
    if (!ok) atomicOr(&ws->error, kDevErrTimeout);
}

cudaError_t launch_wait_probe(Workspace* ws, int kind, uint32_t rounds, cudaStream_t s) {
    wait_probe_kernel<<<1, 32, 0, s>>>(ws, kind, rounds);
    return cudaGetLastError();
}

int sm_count() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
    if (dev < 64 && cached[dev] > 0) return cached[dev];
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev < 64) cached[dev] = n;
    return n;
}

#define DH_GEMV_KS(X) X(256) X(2560) X(5120)

bool gemv_supported(int fmt, int K) {
    if (fmt < 1 || fmt > 5) return false;
#define DH_CASE(k) if (K == k) return true;
    DH_GEMV_KS(DH_CASE)
#undef DH_CASE
    return false;
}

bool linear_supported(int K) { return gemv_supported(4, K) || linear_extra_k(K); }

cudaError_t launch_gemv(const GemvArgs& a, cudaStream_t s) {
    if (a.fmt == 4 && a.out != nullptr && linear_extra_k(a.K)) return launch_linear_nvfp4_packed_extra(a, s);
    if (!gemv_supported(a.fmt, a.K)) return cudaErrorInvalidValue;
    if (a.fmt == 1) return launch_gemv_nvfp4(a, s);
    if (a.fmt == 2) return launch_gemv_fp8(a, s);
    if (a.fmt == 4) return launch_gemv_nvfp4_packed(a, s);
    if (a.fmt == 5) return launch_gemv_fp8_w8a8(a, s);
    return launch_gemv_bf16(a, s);
}

cudaError_t launch_fill_neg_inf(float* out, size_t count, cudaStream_t s) {
    const size_t n4 = count / 4;
    const int ntail = static_cast<int>(count - n4 * 4);
    const int sms = sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    // At most one block of four warps per SM: small enough to sit beside the
    // preceding GEMV's CTAs and the next GEMV's, which start streaming the head
    // while this grid waits. Launched with programmatic stream serialisation
    // (compute_logits one draft 18.33 -> 17.06 µs, two 19.64 -> 17.75, four
    // 21.33 -> 20.05, eight 22.40 -> 21.52, sixteen 28.43 -> 27.68; FP8 head
    // 42.55 -> 40.71; four blocks of 256 threads per SM: 16 drafts 29.48).
    size_t want = (n4 + 127) / 128;
    int blocks = static_cast<int>(want < static_cast<size_t>(sms) ? want : static_cast<size_t>(sms));
    if (blocks < 1) blocks = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks);
    cfg.blockDim = dim3(128);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, fill_neg_inf_kernel, reinterpret_cast<float4*>(out), n4, out + n4 * 4, ntail);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace dh

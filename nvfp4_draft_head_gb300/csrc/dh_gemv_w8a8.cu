// Draft-step kernels for the W8A8 FP8 head: the FP8 head's E4M3 codes times
// per-token E4M3 activations quantised inside the kernel (instantiations of
// dh_gemv_mma.cuh).
#include "dh_gemv_mma.cuh"

namespace dh {

cudaError_t launch_gemv_fp8_w8a8(const GemvArgs& a, cudaStream_t s) {
    switch (a.K) {
        case 256: return mma::launch_mma_k<5, 256>(a, s);
        case 2560: return mma::launch_mma_k<5, 2560>(a, s);
        case 5120: return mma::launch_mma_k<5, 5120>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace dh

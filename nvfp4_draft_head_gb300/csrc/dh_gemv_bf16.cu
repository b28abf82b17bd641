// Draft-step kernels for the BF16 head (instantiations of dh_gemv_mma.cuh).
#include "dh_gemv_mma.cuh"

namespace dh {

cudaError_t launch_gemv_bf16(const GemvArgs& a, cudaStream_t s) {
    switch (a.K) {
        case 256: return mma::launch_mma_k<3, 256>(a, s);
        case 2560: return mma::launch_mma_k<3, 2560>(a, s);
        case 5120: return mma::launch_mma_k<3, 5120>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace dh

// Draft-step kernels for the NVFP4 head in the packed tile-major layout
// (instantiations of dh_gemv_mma.cuh): the ring kernels here, the
// register-load kernels in dh_gemv_nvfp4p_ldg.cu.
#include "dh_gemv_mma.cuh"

namespace dh {

cudaError_t launch_gemv_nvfp4_packed_ldg(const GemvArgs& a, cudaStream_t s);

cudaError_t launch_gemv_nvfp4_packed(const GemvArgs& a, cudaStream_t s) {
    if (!mma::packed_use_ring(a)) return launch_gemv_nvfp4_packed_ldg(a, s);
    switch (a.K) {
        case 2560: return mma::launch_ring_k<2560>(a, s);
        case 5120: return mma::launch_ring_k<5120>(a, s);
        default: return launch_gemv_nvfp4_packed_ldg(a, s);
    }
}

}  // namespace dh

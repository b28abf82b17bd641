// Draft-step kernels for the NVFP4 head in the packed tile-major layout that
// keep their tile loads in registers (instantiations of dh_gemv_mma.cuh; the
// launcher in dh_gemv_nvfp4p.cu picks them or the ring kernels).
#include "dh_gemv_mma.cuh"

namespace dh {

cudaError_t launch_gemv_nvfp4_packed_ldg(const GemvArgs& a, cudaStream_t s) {
    switch (a.K) {
        case 256: return mma::launch_mma_k<mma::kFmtPackedLdg, 256>(a, s);
        case 2560: return mma::launch_mma_k<mma::kFmtPackedLdg, 2560>(a, s);
        // 1 to 4 drafts at K = 5,120 always take the ring kernels
        case 5120:
            return a.out ? mma::launch_mma_m_wide<mma::kFmtPackedLdg, 5120, true>(a, s)
                         : mma::launch_mma_m_wide<mma::kFmtPackedLdg, 5120, false>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace dh

// NVFP4 W4A16 linear layers of the MTP block ("q38_draft.py", MTP_QUANT_KEYS:
// fc_embedding, fc_hidden, qkv_proj, o_proj, shared_expert, quantised with the
// same NVFP4 recipe under the N % 64 / K % 16 rule): y = x W^T with fp32
// accumulation, run by the draft-step kernel in logits mode with no dh_idx
// (row n writes column n). Instantiations for the packed layout at the input
// widths the draft-step files do not cover.
#include "dh_gemv_mma.cuh"

namespace dh {

bool linear_extra_k(int K) { return K == 512 || K == 1024 || K == 2048 || K == 4096; }

cudaError_t launch_linear_nvfp4_packed_extra(const GemvArgs& a, cudaStream_t s) {
    if (a.out == nullptr) return cudaErrorInvalidValue;
    switch (a.K) {
        case 512: return mma::launch_mma_m<mma::kFmtPackedLdg, 512, true>(a, s);
        case 1024: return mma::launch_mma_m<mma::kFmtPackedLdg, 1024, true>(a, s);
        case 2048: return mma::launch_mma_m<mma::kFmtPackedLdg, 2048, true>(a, s);
        case 4096:
            if (mma::packed_use_ring(a)) {
                if (a.M <= 1) return mma::launch_mma<mma::kFmtPackedRing, 4096, 1, true>(a, s);
                if (a.M <= 2) return mma::launch_mma<mma::kFmtPackedRing, 4096, 2, true>(a, s);
                return mma::launch_mma<mma::kFmtPackedRing, 4096, 4, true>(a, s);
            }
            return mma::launch_mma_m_wide<mma::kFmtPackedLdg, 4096, true>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace dh

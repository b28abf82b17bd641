// Epilogues shared by the draft-step kernels: the grid-wide argmax hand-off
// ("q38_draft.py", get_top_tokens: dh_idx[draft_head(h).argmax(-1)]) and the
// logits scatter of compute_logits.
#pragma once

#include "dh_common.cuh"
#include "dh_internal.h"

namespace dh {

// Grid-wide argmax hand-off. Every CTA stores its best key per draft in its
// own workspace slot (1 when it holds no kept row). CTA 0 polls all slots
// until each is non-zero, zeroes them for the next launch, keeps the maximum
// and turns it into an id (the key carries the id itself when dh_idx is
// ascending, else the row). The key is its own "published" flag, so the
// hand-off costs one store and one poll round trip, with no fence, ticket or
// read-back after it.
__device__ __forceinline__ void finish_argmax(const GemvArgs& a, const unsigned long long* cta_key) {
    if (threadIdx.x < a.M) {
        const unsigned long long k = cta_key[threadIdx.x] != 0ull ? cta_key[threadIdx.x] : 1ull;
        asm volatile("st.relaxed.gpu.global.u64 [%0], %1;"
                     :: "l"(&a.ws->slots[threadIdx.x][blockIdx.x]), "l"(k) : "memory");
    }
    if (blockIdx.x != 0) return;
    __shared__ unsigned long long s_red[16];
    __shared__ int s_late;
    if (threadIdx.x < 16) s_red[threadIdx.x] = 0ull;
    if (threadIdx.x == 0) s_late = 0;
    __syncthreads();
    const int G = static_cast<int>(gridDim.x);
    for (int j = threadIdx.x; j < G * a.M; j += blockDim.x) {
        const int m = j / G, b = j - m * G;
        unsigned long long* p = &a.ws->slots[m][b];
        const unsigned long long v = poll_nonzero(p);
        if (v == 0ull) s_late = 1;
        asm volatile("st.relaxed.gpu.global.u64 [%0], 0;" :: "l"(p) : "memory");
        if (v > 1ull) atomicMax(&s_red[m], v);
    }
    __syncthreads();
    if (threadIdx.x == 0 && s_late) atomicOr(&a.ws->error, kDevErrTimeout);
    if (threadIdx.x < a.M) {
        const int m = threadIdx.x;
        const unsigned long long k = s_red[m];
        // low word: 0xFFFFFFFF - id with ascending ids, else 0xFFFFFFFF - row
        const uint32_t low = 0xFFFFFFFFu - static_cast<uint32_t>(k & 0xFFFFFFFFull);
        int id = -1;
        if (k != 0ull) {
            if (a.idx_ascending) id = static_cast<int>(low);
            else if (low < static_cast<uint32_t>(a.N)) id = a.idx[low];
        }
        if (id < 0 || id >= a.V) {
            atomicOr(&a.ws->error, kDevErrIdx);
            id = -1;
        }
        a.ids[m] = id;
        if (a.top) a.top[m] = ordered_value(static_cast<uint32_t>(k >> 32));
    }
}

}  // namespace dh

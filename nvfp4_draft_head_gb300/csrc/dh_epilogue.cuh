// Epilogues shared by the draft-step kernels: the grid-wide argmax hand-off
// ("q38_draft.py", get_top_tokens: dh_idx[draft_head(h).argmax(-1)]) and the
// logits scatter of compute_logits.
#pragma once

#include "dh_common.cuh"
#include "dh_internal.h"

namespace dh {

// Publish the CTA's argmax keys; the last CTA maps rows to ids and resets.
// The keys go out as relaxed reductions; the ticket increment has acq_rel
// semantics at GPU scope, which orders this CTA's reductions (made visible
// CTA-wide by the barrier before it) ahead of the increment and lets the last
// CTA see every other CTA's keys, without a separate fence round trip.
__device__ __forceinline__ void finish_argmax(const GemvArgs& a, const unsigned long long* cta_key) {
    __shared__ bool s_last;
    if (threadIdx.x < a.M) {
        if (cta_key[threadIdx.x] != 0ull)
            asm volatile("red.relaxed.gpu.global.max.u64 [%0], %1;"
                         :: "l"(&a.ws->keys[threadIdx.x]), "l"(cta_key[threadIdx.x]) : "memory");
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned int t;
        asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(t) : "l"(&a.ws->ticket) : "memory");
        s_last = (t == gridDim.x - 1);
    }
    __syncthreads();
    if (!s_last) return;
    if (threadIdx.x < a.M) {
        const int m = threadIdx.x;
        unsigned long long k;
        asm volatile("atom.relaxed.gpu.global.exch.b64 %0, [%1], 0;" : "=l"(k) : "l"(&a.ws->keys[m]) : "memory");
        const uint32_t row = 0xFFFFFFFFu - static_cast<uint32_t>(k & 0xFFFFFFFFull);
        int id = -1;
        if (k != 0ull && row < static_cast<uint32_t>(a.N)) id = a.idx ? a.idx[row] : static_cast<int>(row);
        if (id < 0 || id >= a.V) {
            atomicOr(&a.ws->error, kDevErrIdx);
            id = -1;
        }
        a.ids[m] = id;
        if (a.top) a.top[m] = ordered_value(static_cast<uint32_t>(k >> 32));
    }
    if (threadIdx.x == 0) a.ws->ticket = 0u;
}

// Write one logit of compute_logits at out[m, idx[row]].
__device__ __forceinline__ void scatter_one(const GemvArgs& a, int m, int row, float v) {
    int id = a.idx ? a.idx[row] : row;
    if (id < 0 || id >= a.V) {
        atomicOr(&a.ws->error, kDevErrIdx);
        return;
    }
    a.out[static_cast<size_t>(m) * a.V + id] = v;
}

}  // namespace dh

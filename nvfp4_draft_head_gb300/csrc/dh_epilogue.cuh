// Epilogues shared by the draft-step kernels: the grid-wide argmax hand-off
// ("q38_draft.py", get_top_tokens: dh_idx[draft_head(h).argmax(-1)]) and the
// logits scatter of compute_logits.
#pragma once

#include "dh_common.cuh"
#include "dh_internal.h"

namespace dh {

// Publish the CTA's argmax keys; the last CTA turns the winning key into an id
// (the key carries the id itself when dh_idx is ascending, else the row) and
// resets the workspace.
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
    if (threadIdx.x == 0) a.ws->ticket = 0u;
}

}  // namespace dh

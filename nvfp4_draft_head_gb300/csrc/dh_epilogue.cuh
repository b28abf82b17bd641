// Epilogue of the draft-step kernels in top-tokens mode: the grid-wide argmax
// ("q38_draft.py", get_top_tokens: dh_idx[draft_head(h).argmax(-1)]), or, for
// one shard of a vocabulary-sharded head, the keys that the local-argmax
// exchange combines ("q38_draft.py", install: use_local_argmax_reduction).
#pragma once

#include "dh_common.cuh"
#include "dh_internal.h"

namespace dh {

// Epoch and dirty word of the workspace (adjacent), read by every CTA after
// the grid-dependency wait (the preceding step has completed, so its updates
// are visible), early, so that the hand-off at the end does not wait for them.
__device__ __forceinline__ uint2 load_epoch_dirty(const Workspace* ws) {
    uint2 v;
    asm volatile("ld.relaxed.gpu.global.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(&ws->epoch) : "memory");
    return v;
}

// Grid-wide argmax hand-off. Every CTA stores its best key per draft in its
// own slot of bank (epoch & 1) (1 when it holds no kept row). CTA 0 polls the
// bank's slots until each is non-zero (bounded), zeroes them, keeps the
// maximum per draft and turns it into an id, or a shard key. The key is its
// own "published" flag: one store and one poll round trip, no fence or ticket.
//
// If a poll runs out, CTA 0 records the timeout and marks the bank dirty: the
// late CTA's store still lands there, before this launch completes. The next
// step collects from the other bank and zeroes the dirty one, so a late key
// never reaches a later step.
// The workspace's epoch and dirty word were read at the kernel's start.
__device__ __forceinline__ void finish_argmax(const GemvArgs& a, const unsigned long long* cta_key,
                                              unsigned int epoch, unsigned int dirty) {
    const unsigned int bank = epoch & 1u;
    if (threadIdx.x < a.M) {
        const unsigned long long k = cta_key[threadIdx.x] != 0ull ? cta_key[threadIdx.x] : 1ull;
        asm volatile("st.relaxed.gpu.global.u64 [%0], %1;"
                     :: "l"(&a.ws->slots[bank][threadIdx.x][blockIdx.x]), "l"(k) : "memory");
    }
    if (blockIdx.x != 0) return;
    __shared__ unsigned long long s_red[16];
    __shared__ int s_late;
    if (threadIdx.x < 16) s_red[threadIdx.x] = 0ull;
    if (threadIdx.x == 0) s_late = 0;
    __syncthreads();
    const int G = static_cast<int>(gridDim.x);
    const int total = G * a.M;
    // A thread reads up to four slots before it waits on any, so that with
    // more slots than threads (several drafts) the keys that are already
    // there cost one round trip, not one per slot.
    for (int j0 = threadIdx.x; j0 < total; j0 += 4 * static_cast<int>(blockDim.x)) {
        unsigned long long v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int j = j0 + u * static_cast<int>(blockDim.x);
            v[u] = 0ull;
            if (j < total) {
                const int m = j / G, b = j - m * G;
                asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v[u]) : "l"(&a.ws->slots[bank][m][b]) : "memory");
            }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int j = j0 + u * static_cast<int>(blockDim.x);
            if (j >= total) break;
            const int m = j / G, b = j - m * G;
            unsigned long long* p = &a.ws->slots[bank][m][b];
            if (v[u] == 0ull) v[u] = poll_nonzero(p);
            if (v[u] == 0ull) s_late = 1;
            asm volatile("st.relaxed.gpu.global.u64 [%0], 0;" :: "l"(p) : "memory");
            if (v[u] > 1ull) atomicMax(&s_red[m], v[u]);
        }
    }
    // a dirty bank left by an earlier step (never this step's bank): zero the
    // slots that step used
    if (dirty & 1u) {
        const unsigned int db = (dirty >> 1) & 1u, dm = (dirty >> 2) & 31u, dg = dirty >> 8;
        for (unsigned int j = threadIdx.x; j < dm * dg; j += blockDim.x)
            asm volatile("st.relaxed.gpu.global.u64 [%0], 0;" :: "l"(&a.ws->slots[db][j / dg][j % dg]) : "memory");
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned int d = 0u;
        if (s_late) {
            atomicOr(&a.ws->error, kDevErrTimeout);
            d = 1u | (bank << 1) | (static_cast<unsigned int>(a.M) << 2) | (static_cast<unsigned int>(G) << 8);
        }
        if (s_late || (dirty & 1u)) a.ws->dirty = d;
        a.ws->epoch = epoch + 1u;
    }
    if (threadIdx.x < a.M) {
        const int m = threadIdx.x;
        const unsigned long long k = s_red[m];
        if (a.keys) {
            // shard key: signed order equals the unsigned order of k (an int64
            // MAX all-reduce combines shards); a shard without a kept row gives
            // INT64_MIN, the identity of that maximum
            a.keys[m] = k ^ 0x8000000000000000ull;
            return;
        }
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

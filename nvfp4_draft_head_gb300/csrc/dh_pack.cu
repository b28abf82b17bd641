// Repack of an NVFP4 head from the canonical layout (codes [N][K/2], scales
// [N][K/16]) into the tile-major layout the draft-step kernels stream: for
// each tile of 16 rows and each 128-wide k-window, a 1,152-byte block holding
// the 16 rows' 64 code bytes of that window, row by row, and then their 128
// scale bytes in the order the GEMV's lanes use them: lane 4 g + t (g < 8,
// t < 4) finds at bytes 4 (4 g + t) .. + 3 the scales of blocks 2t, 2t+1 of
// row g, then of row g + 8 (the blocks of its 32 codes). Every warp load of
// the GEMV then covers 512 (codes) or 128 (scales) contiguous bytes, and a
// lane's four scale bytes are one 32-bit load. A pure permutation of bytes;
// run once after quantisation.
#include <cstdint>

#include "dh_common.cuh"
#include "dh_internal.h"

namespace dh {

constexpr int kBlk = 16 * 64 + 16 * 8;  // bytes of one (tile, window) block
constexpr int kChunks = kBlk / 16;      // 64 code chunks + 8 scale chunks

__global__ void nvfp4_pack_kernel(const uint8_t* __restrict__ q, const uint8_t* __restrict__ sf, int N, int K,
                                  uint8_t* __restrict__ out) {
    const int nwin = K / 128;
    const size_t total = static_cast<size_t>(N / 16) * nwin * kChunks;
    for (size_t c = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; c < total;
         c += static_cast<size_t>(gridDim.x) * blockDim.x) {
        const size_t blk = c / kChunks;
        const int j = static_cast<int>(c % kChunks);
        const int tile = static_cast<int>(blk / nwin), w = static_cast<int>(blk % nwin);
        uint4 v;
        if (j < 64) {  // row j/4 of the tile, 16-byte piece j%4 of the window's 64 code bytes
            const size_t row = static_cast<size_t>(tile) * 16 + j / 4;
            v = *reinterpret_cast<const uint4*>(q + row * (K / 2) + w * 64 + (j % 4) * 16);
        } else {       // lanes 4 g .. 4 g + 3, g = j - 64: scale bytes of rows g and g + 8
            const int g = j - 64;
            const size_t row = static_cast<size_t>(tile) * 16 + g;
            const uint2 a = *reinterpret_cast<const uint2*>(sf + row * (K / 16) + 8 * w);
            const uint2 b = *reinterpret_cast<const uint2*>(sf + (row + 8) * (K / 16) + 8 * w);
            // lane t: bytes 2t, 2t+1 of row g, then the same of row g + 8
            v = make_uint4(__byte_perm(a.x, b.x, 0x5410), __byte_perm(a.x, b.x, 0x7632),
                           __byte_perm(a.y, b.y, 0x5410), __byte_perm(a.y, b.y, 0x7632));
        }
        *reinterpret_cast<uint4*>(out + blk * kBlk + j * 16) = v;
    }
}

cudaError_t launch_nvfp4_pack(const uint8_t* q, const uint8_t* sf, int N, int K, uint8_t* out, cudaStream_t s) {
    const size_t total = static_cast<size_t>(N / 16) * (K / 128) * kChunks;
    const int sms = sm_count();
    if (sms <= 0) return cudaErrorInvalidDevice;
    size_t want = (total + 255) / 256;
    const size_t cap = static_cast<size_t>(sms) * 8;
    const int blocks = static_cast<int>(want < cap ? (want > 0 ? want : 1) : cap);
    nvfp4_pack_kernel<<<blocks, 256, 0, s>>>(q, sf, N, K, out);
    return cudaGetLastError();
}

}  // namespace dh

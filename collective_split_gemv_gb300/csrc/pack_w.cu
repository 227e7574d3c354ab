// Packs each slot's row-major W_r into the layout the persistent fused kernel
// streams with one contiguous bulk copy per 128 x 64 block (see the layout
// note beside PackWArgs in internal.h).
//
// The fused kernel's shared-memory stage for a block is the same either way:
// a TMA tensor load with 128-byte swizzle of the row-major block, or a plain
// copy of the packed block, which holds those bytes already in that order.
// Reading W as long contiguous runs instead of 128 rows of 128 bytes is what
// the layout buys (the bytes read per call are the same).  Packing is done
// once, when the weights are loaded: weights are read by every decode step.
#include <cuda_runtime.h>

#include "internal.h"

namespace symm {

namespace {

constexpr int kPackThreads = 256;
constexpr int kChunksPerBlock = (int)(kPackBlockBytes / 16);   // 1024

__global__ void __launch_bounds__(kPackThreads) pack_w_kernel(const PackWArgs a) {
    const int r = a.r0 + (int)blockIdx.y;
    const int J = (a.Kr + kPackCols - 1) / kPackCols;
    const int T = (a.N + kPackRows - 1) / kPackRows;
    const long long b = blockIdx.x;   // block of this slot; b == T * J is the zero block
    const int t = J > 0 ? (int)(b / J) : T;
    const int j = J > 0 ? (int)(b - (long long)t * J) : 0;
    const uint8_t *W = a.W + (long long)r * a.stride;
    uint4 *dst = reinterpret_cast<uint4 *>(a.Wp + (long long)r * a.stride + b * (long long)kPackBlockBytes);
    for (int p = threadIdx.x; p < kChunksPerBlock; p += kPackThreads) {
        const int i = p >> 3;                 // row of the block
        const int c = (p & 7) ^ (i & 7);      // chunk of that row stored at position p
        const int n = t * kPackRows + i;
        const int k = j * kPackCols + c * 8;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (t < T && n < a.N && k < a.Kr)     // Kr % 8 == 0: a chunk is all in or all out
            v = *reinterpret_cast<const uint4 *>(W + ((long long)n * a.Kr + k) * 2);
        dst[p] = v;
    }
}

}  // namespace

cudaError_t launch_pack_w(const PackWArgs &a, cudaStream_t s) {
    const size_t blocks = packed_w_blocks(a.N, a.Kr);
    if (blocks > 0x7fffffffu || a.R < 1 || a.R > 65535) return cudaErrorInvalidValue;
    // Plain stream order: the weights may have been written by the kernel just
    // before, and packing is not on the per-call path.
    pack_w_kernel<<<dim3((unsigned)blocks, (unsigned)a.R), kPackThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace symm

// 2-D tile reduce to one or several roots over R symmetric slots.
//
// For tile i (rows x cols elements of a row-major tensor with leading
// dimension ld_in, starting at in[i] in every slot):
//     out_root(i)[a][c] = bf16_rne( sum_{r=0}^{R-1} in_i,r[a][c] )
// summed in fp32 in rank order; only the root's output tile is written
// (PyTorch Symmetric Memory docs, op reference `tile_reduce` and
// `multi_root_tile_reduce`; the symmetric-memory talk's tile-communication
// segment: a tile is non-contiguous, so each thread is pointed at the start
// and end of every contiguous row itself).
//
// Layout of the work: blockIdx.y is the tile, blockIdx.x strides over its
// items.  An item is one 16-byte vector (8 columns of one row) when every
// row start of the input and output tiles is 16-byte aligned, else one
// element.  Each item reads its R values back to back and is stored once.
// HBM-bound: R * rows * cols * 2 bytes read, rows * cols * 2 written per tile.
#include <cuda_bf16.h>

#include <algorithm>

#include "internal.h"
#include "protocol.cuh"

namespace symm {

namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ void set8(float (&acc)[8], const uint4 &v) {
    acc[0] = bf16lo(v.x); acc[1] = bf16hi(v.x);
    acc[2] = bf16lo(v.y); acc[3] = bf16hi(v.y);
    acc[4] = bf16lo(v.z); acc[5] = bf16hi(v.z);
    acc[6] = bf16lo(v.w); acc[7] = bf16hi(v.w);
}

__device__ __forceinline__ void add8(float (&acc)[8], const uint4 &v) {
    acc[0] += bf16lo(v.x); acc[1] += bf16hi(v.x);
    acc[2] += bf16lo(v.y); acc[3] += bf16hi(v.y);
    acc[4] += bf16lo(v.z); acc[5] += bf16hi(v.z);
    acc[6] += bf16lo(v.w); acc[7] += bf16hi(v.w);
}

template <int RT, bool kVec>
__global__ void __launch_bounds__(kThreads) tile_reduce_kernel(const TileReduceArgs a) {
    chain_entry();
    const int R = RT > 0 ? RT : a.R;
    const int t = blockIdx.y;
    const uint8_t *in = a.in[t];
    uint8_t *out = a.out + (long long)a.root[t] * a.stride;
    const int per_row = kVec ? a.cols / 8 : a.cols;
    const long long items = (long long)a.rows * per_row;
    const long long step = (long long)gridDim.x * kThreads;
    for (long long v = (long long)blockIdx.x * kThreads + threadIdx.x; v < items; v += step) {
        const long long row = v / per_row;
        const long long col = (v - row * per_row) * (kVec ? 8 : 1);
        const uint8_t *src = in + (row * a.ld_in + col) * 2;
        uint8_t *dst = out + (row * a.ld_out + col) * 2;
        if (kVec) {
            float acc[8];
            if (RT > 0) {
                uint4 x[RT > 0 ? RT : 1];
#pragma unroll
                for (int q = 0; q < (RT > 0 ? RT : 1); ++q) x[q] = ld_v4(src + (long long)q * a.stride);
                set8(acc, x[0]);
#pragma unroll
                for (int q = 1; q < (RT > 0 ? RT : 1); ++q) add8(acc, x[q]);
            } else {
                set8(acc, ld_v4(src));
                for (int q = 1; q < R; ++q) add8(acc, ld_v4(src + (long long)q * a.stride));
            }
            uint4 o;
            __nv_bfloat162 p;
            p = __floats2bfloat162_rn(acc[0], acc[1]); o.x = *reinterpret_cast<uint32_t *>(&p);
            p = __floats2bfloat162_rn(acc[2], acc[3]); o.y = *reinterpret_cast<uint32_t *>(&p);
            p = __floats2bfloat162_rn(acc[4], acc[5]); o.z = *reinterpret_cast<uint32_t *>(&p);
            p = __floats2bfloat162_rn(acc[6], acc[7]); o.w = *reinterpret_cast<uint32_t *>(&p);
            st_v4(dst, o);
        } else {
            float acc = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(src));
            for (int q = 1; q < R; ++q)
                acc += __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(src + (long long)q * a.stride));
            *reinterpret_cast<__nv_bfloat16 *>(dst) = __float2bfloat16_rn(acc);
        }
    }
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

template <class Kern>
cudaError_t launch_tile(Kern kern, const TileReduceArgs &a, dim3 grid, cudaStream_t s) {
    return launch_kernel(kern, grid, dim3(kThreads), 0, s, a.chained != 0, a);
}

}  // namespace

cudaError_t launch_tile_reduce(const TileReduceArgs &a, cudaStream_t s) {
    bool vec = a.cols % 8 == 0 && a.ld_in % 8 == 0 && a.ld_out % 8 == 0 && aligned16(a.out);
    for (int i = 0; i < a.ntiles; ++i) vec = vec && aligned16(a.in[i]);
    int sms = 152, dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long items = (long long)a.rows * (vec ? a.cols / 8 : a.cols);
    long long bx = (items + kThreads - 1) / kThreads;
    // up to 16 CTAs per SM over all tiles together (eight resident at a time;
    // the hardware starts a fresh CTA wherever one retires), grid-stride beyond
    const long long cap = std::max<long long>(1, (long long)sms * 16 / a.ntiles);
    if (bx > cap) bx = cap;
    if (bx < 1) bx = 1;
    const dim3 grid((unsigned)bx, (unsigned)a.ntiles);
    if (vec) {
        switch (a.R) {
            case 2: return launch_tile(tile_reduce_kernel<2, true>, a, grid, s);
            case 4: return launch_tile(tile_reduce_kernel<4, true>, a, grid, s);
            case 8: return launch_tile(tile_reduce_kernel<8, true>, a, grid, s);
            default: return launch_tile(tile_reduce_kernel<0, true>, a, grid, s);
        }
    }
    return launch_tile(tile_reduce_kernel<0, false>, a, grid, s);
}

}  // namespace symm

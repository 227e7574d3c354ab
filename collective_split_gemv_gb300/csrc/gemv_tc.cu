// Fused row-parallel GEMV + one-shot all-reduce on the 5th-generation tensor
// cores (tcgen05) with TMA-fed shared memory, for batches wide enough that the
// CUDA-core path would be limited by instruction issue and shared-memory
// bandwidth rather than by HBM.
//
// One CTA per (row tile t of 128 rows, rank r, K-split s); blockIdx =
// (t * R + r) * S + s so the contributors of a tile run together (the
// communication-aware workgroup ordering of the fused GEMV + AllReduce in
// "Overlapping Collective Communication with Dependent Computation ...",
// Abstract).
//
//   D[128 x 16] (fp32, TMEM) += W_r tile [128 x 64] (bf16, smem, K-major)
//                               x x_r^T   [64 x 16]  (bf16, smem, K-major)
//
// per 64-wide K block, four tcgen05.mma.kind::f16 of K = 16 each.  x_r's rows
// b >= B and W_r's rows n >= N or columns k >= K/R are zero-filled by the TMA
// unit (out-of-bounds fill), so ragged shapes need no special code.
//
// Warp roles (192 threads):
//   warp 0     one lane issues TMA loads of W and x blocks into a ring of
//              kStages stages (mbarrier full/empty pairs);
//   warp 1     owns the TMEM allocation; one lane issues the MMAs and commits
//              each stage back to the producer, then the accumulator;
//   warps 2-5  epilogue: tcgen05.ld of their 32 TMEM lanes (rows) x 16
//              columns (batch), fp32 partial to the rank's scratch slot.
// All threads then run the publish / last-arriver protocol (protocol.cuh).
//
// Every mbarrier wait is bounded (%globaltimer); a wait that gives up latches
// a timeout in the status word, the CTA waits (bounded) for the copies it has
// in flight, frees its TMEM and returns without publishing.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "protocol.cuh"
#include "sm100.cuh"

namespace symm {

namespace {

constexpr int kM = kTcRows;                 // MMA M: rows of W per tile
constexpr int kN = 16;                      // MMA N: batch columns (padded)
constexpr int kBK = kTcBlockK;              // K elements per stage: one 128-byte swizzle row
constexpr int kStages = 6;
constexpr int kABytes = kM * kBK * 2;       // 16 KiB
constexpr int kBBytes = kN * kBK * 2;       // 2 KiB
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 32;          // smallest allocation; 16 are used
constexpr uint32_t kIdesc = mma_idesc_bf16_f32(kM, kN);

static_assert(kStageBytes % 1024 == 0, "stages must keep 1024-byte alignment for 128B swizzle");

__global__ void __launch_bounds__(kThreads, 1)
    gemv_ar_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                      const GemvArgs a, int kb_total, int kb_per_split) {
    chain_entry();
    // Thread 0 publishes; its read of the launch epoch overlaps the streaming.
    const uint32_t epoch = threadIdx.x == 0 ? read_launch_epoch(a) : 0u;
    extern __shared__ uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t full_bar[kStages];
    __shared__ __align__(8) uint64_t empty_bar[kStages];
    __shared__ __align__(8) uint64_t accum_bar;
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_sh;

    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);

    const int S = a.splits;
    const int bid = a.reverse_order ? (int)(gridDim.x - 1 - blockIdx.x) : (int)blockIdx.x;
    const int s = bid % S;
    const int tr = bid / S;
    const int r = tr % a.R;
    const int t = tr / a.R;
    const int kb0 = s * kb_per_split;
    const int nkb = max(0, min(kb0 + kb_per_split, kb_total) - kb0);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) {
            mbar_init(&full_bar[i], 1);
            mbar_init(&empty_bar[i], 1);
        }
        mbar_init(&accum_bar, 1);
        abort_sh = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) tmem_alloc(&tmem_base_sh, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;

    if (warp == 0) {
        if (lane == 0 && nkb > 0) {
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmW)) : "memory");
            asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmX)) : "memory");
            int issued = 0;
            for (int i = 0; i < nkb; ++i) {
                const int st = i % kStages;
                const uint32_t ph = (uint32_t)(i / kStages) & 1u;
                if (!mbar_wait(&empty_bar[st], ph ^ 1u, &abort_sh)) {
                    latch_status(a.status, kProtoTimeout, r, t, read_launch_epoch(a));
                    abort_sh = 1;
                    break;
                }
                mbar_arrive_expect_tx(&full_bar[st], (uint32_t)kStageBytes);
                const int k = (kb0 + i) * kBK;
                uint8_t *dst = smem + (size_t)st * kStageBytes;
                tma_load_3d(dst, &tmW, &full_bar[st], k, t * kM, r);
                tma_load_3d(dst + kABytes, &tmX, &full_bar[st], k, 0, r);
                issued = i + 1;
            }
            if (abort_sh) {
                // Wait (bounded) for the copies this thread still has in flight.
                volatile int never = 0;
                for (int j = max(0, issued - kStages); j < issued; ++j)
                    mbar_wait(&full_bar[j % kStages], (uint32_t)(j / kStages) & 1u, &never);
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && nkb > 0) {
            for (int i = 0; i < nkb; ++i) {
                const int st = i % kStages;
                const uint32_t ph = (uint32_t)(i / kStages) & 1u;
                if (!mbar_wait(&full_bar[st], ph, &abort_sh)) {
                    latch_status(a.status, kProtoTimeout, r, t, read_launch_epoch(a));
                    abort_sh = 1;
                    break;
                }
                tc_fence_after();
                const uint32_t a_addr = smem_u32(smem + (size_t)st * kStageBytes);
                const uint32_t b_addr = a_addr + kABytes;
#pragma unroll
                for (int kk = 0; kk < kBK / 16; ++kk)
                    tc_mma(tmem, smem_desc_sw128(a_addr + kk * 32), smem_desc_sw128(b_addr + kk * 32), kIdesc,
                           (i > 0 || kk > 0) ? 1u : 0u);
                tc_commit(&empty_bar[st]);
            }
            tc_commit(&accum_bar);
        }
    } else {
        // Epilogue: warp w reads TMEM lanes 32 * (w % 4) .. + 31 (rows of the tile).
        const int q = warp & 3;
        const int row = q * 32 + lane;
        const int n = t * kM + row;
        float v[16];
        bool ok = true;
        if (nkb > 0) {
            ok = mbar_wait_sleepy(&accum_bar, 0, &abort_sh);
            if (!ok) {
                latch_status(a.status, kProtoTimeout, r, t, read_launch_epoch(a));
                abort_sh = 1;
            }
            __syncwarp();
            ok = __all_sync(0xffffffffu, ok) != 0;
            if (ok) {
                tc_fence_after();
                tmem_ld_16(tmem + ((uint32_t)(q * 32) << 16), v);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = 0.f;
        }
        if (ok && n < a.N) {
            float *P = reinterpret_cast<float *>(a.scratch + (long long)r * a.stride +
                                                 (long long)s * a.partial_stride);
#pragma unroll
            for (int b = 0; b < kN; ++b)
                if (b < a.B) P[(size_t)b * a.N + n] = v[b];
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    if (abort_sh) return;
    publish_and_reduce(a, epoch, t, r, s);
}

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// A 3-D view [R][rows][Kr] of bf16 with the slot stride as the rank stride.
int encode_3d(CUtensorMap *m, const void *base, int Kr, int rows, int R, long long stride, int box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return -1;
    const cuuint64_t dims[3] = {(cuuint64_t)Kr, (cuuint64_t)rows, (cuuint64_t)R};
    const cuuint64_t strides[2] = {(cuuint64_t)Kr * 2, (cuuint64_t)stride};
    const cuuint32_t box[3] = {(cuuint32_t)kBK, (cuuint32_t)box_rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult rc = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return rc == CUDA_SUCCESS ? 0 : (int)rc;
}

}  // namespace

size_t tc_smem_bytes() { return (size_t)kStages * kStageBytes + 1024; }

int tc_encode_maps(const GemvArgs &a, void *maps) {
    CUtensorMap *m = static_cast<CUtensorMap *>(maps);
    int rc = encode_3d(&m[0], a.W, a.Kr, a.N, a.R, a.stride, kM);
    if (rc != 0) return rc;
    return encode_3d(&m[1], a.x, a.Kr, a.B, a.R, a.stride, kN);
}

cudaError_t launch_gemv_tc(const GemvArgs &a, const void *maps, cudaStream_t s) {
    const CUtensorMap *m = static_cast<const CUtensorMap *>(maps);
    const size_t smem = tc_smem_bytes();
    // The shared-memory attribute is per device: set it once for each device
    // a launch happens on (devices past 63 set it every time).
    static unsigned long long attr_devices = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) dev = 64;
    const unsigned long long bit = dev < 64 ? 1ull << dev : 0ull;
    if (bit == 0 || !(attr_devices & bit)) {
        cudaError_t e = cudaFuncSetAttribute(gemv_ar_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
        attr_devices |= bit;
    }
    const int kb_total = (a.Kr + kBK - 1) / kBK;
    const int kb_per_split = (kb_total + a.splits - 1) / a.splits;
    const unsigned grid = (unsigned)a.num_tiles * (unsigned)a.R * (unsigned)a.splits;
    return launch_kernel(gemv_ar_tc_kernel, dim3(grid), dim3(kThreads), smem, s, a.chained != 0, m[0], m[1], a,
                         kb_total, kb_per_split);
}

}  // namespace symm

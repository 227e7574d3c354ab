// Strided copies between one contiguous buffer and the R symmetric slots,
// done by the SMs: the engine behind symm_copy_to_slots / from_slots when
// the contiguous side is device memory or pinned host memory the GPU can
// address (on this platform every pinned allocation is mapped, and the
// GPU reads and writes it over the CPU-GPU link).
//
// Why a kernel and not a copy engine: a kernel is a link in a chain of
// programmatic dependent launches.  Staging a step's inputs with it lets the
// fused call that follows start (and load its weights) while the inputs
// arrive, and reading the result back with it keeps the whole step a chain
// of kernels; a copy-engine copy between two kernels would break the chain.
// Block r of the contiguous buffer (bytes per rank) corresponds to the
// symmetric pointer's instance in slot r.
#include <cuda_runtime.h>

#include "internal.h"
#include "protocol.cuh"

namespace symm {

namespace {

constexpr int kThreads = 256;

// v indexes 16-byte vectors (kVec) or bytes over nranks blocks of `bytes`.
template <bool kVec>
__global__ void __launch_bounds__(kThreads) copy_slots_kernel(const CopySlotsArgs a) {
    chain_entry();
    const size_t per = kVec ? a.bytes / 16 : a.bytes;
    const size_t total = per * (size_t)a.nranks;
    const size_t step = (size_t)gridDim.x * kThreads;
    for (size_t v = (size_t)blockIdx.x * kThreads + threadIdx.x; v < total; v += step) {
        const size_t r = v / per;
        const size_t off = (v - r * per) * (kVec ? 16 : 1);
        const uint8_t *src = a.src + (long long)r * a.src_stride + off;
        uint8_t *dst = a.dst + (long long)r * a.dst_stride + off;
        if (kVec)
            st_v4(dst, ld_v4(src));
        else
            *dst = *src;
    }
}

}  // namespace

cudaError_t launch_copy_slots(const CopySlotsArgs &a, cudaStream_t s) {
    const bool vec = a.bytes % 16 == 0 && a.src_stride % 16 == 0 && a.dst_stride % 16 == 0 &&
                     (reinterpret_cast<uintptr_t>(a.src) & 15u) == 0 && (reinterpret_cast<uintptr_t>(a.dst) & 15u) == 0;
    const size_t items = (vec ? a.bytes / 16 : a.bytes) * (size_t)a.nranks;
    int sms = 152, dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    size_t blocks = (items + kThreads - 1) / kThreads;
    const size_t cap = (size_t)sms * 16;   // twice the resident CTAs, grid-stride beyond
    if (blocks > cap) blocks = cap;
    if (blocks == 0) blocks = 1;
    auto kern = vec ? copy_slots_kernel<true> : copy_slots_kernel<false>;
    return launch_kernel(kern, dim3((unsigned)blocks), dim3(kThreads), 0, s, a.chained != 0, a);
}

}  // namespace symm

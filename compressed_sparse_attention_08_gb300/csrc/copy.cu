// Copies between device memory and pinned host memory done by the SMs, for moving a decode
// step's small inputs and outputs inside the step's stream. On a Grace-Blackwell GPU the SMs
// load and store pinned host memory directly over the chip-to-chip link; as a node of a
// captured graph, a copy-engine transfer of a step's 370 KB of inputs cost ~12 us, this
// kernel ~1 us.
#include "common.cuh"
#include "internal.h"

namespace dsv4 {
namespace {

constexpr int kCopyThreads = 256;

// 16-byte pieces, grid-stride. Waits for the kernel before it (programmatic dependent launch),
// whose output may be the source. The source is read with plain loads (it may be host memory
// written before the launch).
__global__ void __launch_bounds__(kCopyThreads) copy_kernel(uint4* dst, const uint4* src, size_t n16) {
    pdl_wait();
    const size_t stride = static_cast<size_t>(gridDim.x) * kCopyThreads;
    for (size_t i = static_cast<size_t>(blockIdx.x) * kCopyThreads + threadIdx.x; i < n16; i += stride)
        dst[i] = src[i];
}

}  // namespace

int launch_copy(void* dst, const void* src, size_t bytes, cudaStream_t stream) {
    const size_t n16 = bytes / 16;
    if (n16 == 0) return DSV4_OK;
    const int sms = sm_count() > 0 ? sm_count() : 148;
    const size_t want = (n16 + kCopyThreads - 1) / kCopyThreads;
    const unsigned ctas = static_cast<unsigned>(want < static_cast<size_t>(2 * sms) ? want : static_cast<size_t>(2 * sms));
    count_launch();
    return launch_k(copy_kernel, dim3(ctas), dim3(kCopyThreads), 0, stream, true, static_cast<uint4*>(dst),
                    static_cast<const uint4*>(src), n16) == cudaSuccess
               ? DSV4_OK
               : DSV4_ERR_LAUNCH;
}

}  // namespace dsv4

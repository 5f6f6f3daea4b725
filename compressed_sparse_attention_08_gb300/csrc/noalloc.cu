// Top-k on caller-given scores without any caller-supplied or allocated scratch memory.
//
// Some callers cannot allocate device memory at the point where they need the selection:
// code running inside an allocator callback or an allocator-free serving loop, a host
// runtime that forbids cudaMalloc after start-up, or a plug-in handed only its input and
// output buffers. dsv4_topk_noalloc serves them: its scratch space (error word, per-row
// histograms of the long-row path) is one file-scope device array. The
// driver reserves the array on a GPU when this library's device code is loaded there, which
// with lazy module loading happens at the first call of this entry point on that GPU (the
// symbol lookup below); it stays reserved until the process exits. Callers should therefore
// make a first call at start-up, before any stream capture. It runs exactly the same kernels
// as dsv4_topk.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace dsv4 {
namespace {

constexpr size_t kStaticScratchBytes = 16u << 20;   // 16 MiB on every GPU using the library
constexpr int kMaxDevices = 64;

// The shared scratch. In host code this name stands for the array but is not its device
// address: the address comes from cudaGetSymbolAddress, once per device.
static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

// Device address of g_static_scratch for each device, looked up once per device (one
// once_flag per device, so concurrent first calls from several host threads are safe); null
// when the lookup failed.
std::once_flag g_scratch_once[kMaxDevices];
uint8_t* g_scratch_addr[kMaxDevices] = {nullptr};

uint8_t* scratch_for_current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::call_once(g_scratch_once[dev], [dev] {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_static_scratch) == cudaSuccess && ptr != nullptr)
            g_scratch_addr[dev] = static_cast<uint8_t*>(ptr);
        else
            cudaGetLastError();
    });
    return g_scratch_addr[dev];
}

}  // namespace
}  // namespace dsv4

using namespace dsv4;

extern "C" int dsv4_topk_noalloc(const dsv4_topk_args* a, dsv4_stream_t stream) {
    if (!a || !a->scores || !a->n_vis || !a->idx_out) return DSV4_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(a->scores) | reinterpret_cast<uintptr_t>(a->n_vis) |
         reinterpret_cast<uintptr_t>(a->idx_out)) & 15u)
        return DSV4_ERR_INVALID_ARG;
    if (a->rows < 0 || a->max_comp < 1 || a->top_k < 1 || a->top_k > a->max_comp)
        return DSV4_ERR_INVALID_ARG;
    // the scratch this call needs must fit in the fixed array
    if (dsv4_topk_workspace_size(a) > kStaticScratchBytes) return DSV4_ERR_INVALID_ARG;
    int major = 0, minor = 0, dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        major != 10 || minor != 3)
        return DSV4_ERR_UNSUPPORTED;
    uint8_t* scratch = scratch_for_current_device();
    if (!scratch) return DSV4_ERR_LAUNCH;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // the array keeps the previous call's contents: clear the error word (the long-row
    // histograms are cleared by the launcher below)
    if (cudaMemsetAsync(scratch, 0, kWsHeader, st) != cudaSuccess) return DSV4_ERR_LAUNCH;
    TopkRows t;
    t.scores = a->scores;
    t.n_vis = a->n_vis;
    t.n_comp = nullptr;
    t.q_pos = nullptr;
    t.n_q = 1;
    t.ratio = 1;
    t.idx_out = a->idx_out;
    t.rows = a->rows;
    t.max_comp = a->max_comp;
    t.top_k = a->top_k;
    t.hist_zeroed = false;
    t.hist_built = false;
    t.pdl = true;
    return launch_topk(t, scratch + kWsHeader, reinterpret_cast<uint32_t*>(scratch), st);
}

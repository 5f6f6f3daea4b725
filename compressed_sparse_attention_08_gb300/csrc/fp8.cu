// FP8 E4M3 row quantization for the FP8 indexer keys and queries.
//
// Source: "nvfp4-megamoe-kernel: compare master..pure-nvfp4", single_shot_inference.py
// (indexer): "Indexer keys are stored as FP8_E4M3 in the KV cache". One fp32 scale per row,
// amax / 448 (448 is E4M3's largest finite value), computed in fp32 with IEEE division, and
// each code is the round-to-nearest-even, saturating E4M3 conversion of x / scale.
#include <cuda_fp8.h>

#include "common.cuh"
#include "internal.h"

namespace dsv4 {
namespace {

constexpr int kWarps = 8;

// One warp per row; each lane holds dim / 32 consecutive values.
template <int PER>
__global__ void __launch_bounds__(kWarps * 32)
quantize_rows_kernel(const __nv_bfloat16* __restrict__ x, int rows, uint8_t* __restrict__ q,
                     float* __restrict__ scale) {
    const int lane = threadIdx.x & 31;
    const long long row = static_cast<long long>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
    if (row >= rows) return;
    const __nv_bfloat16* xr = x + row * (32 * PER) + lane * PER;
    float v[PER];
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < PER; ++i) {
        v[i] = __bfloat162float(xr[i]);
        amax = fmaxf(amax, fabsf(v[i]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float sc = amax > 0.f ? amax / 448.0f : 1.0f;
    if (lane == 0) scale[row] = sc;
    uint8_t* qr = q + row * (32 * PER) + lane * PER;
#pragma unroll
    for (int i = 0; i < PER; ++i)
        qr[i] = static_cast<uint8_t>(__nv_cvt_float_to_fp8(v[i] / sc, __NV_SATFINITE, __NV_E4M3));
}

}  // namespace

int launch_quantize_rows_fp8(const void* x, int rows, int dim, void* q, float* scale, cudaStream_t stream) {
    if (rows == 0) return DSV4_OK;
    const dim3 grid(static_cast<unsigned>((rows + kWarps - 1) / kWarps));
    const auto* xb = static_cast<const __nv_bfloat16*>(x);
    auto* qb = static_cast<uint8_t*>(q);
    count_launch();
    cudaError_t e;
    switch (dim / 32) {
        case 1: e = launch_k(quantize_rows_kernel<1>, grid, dim3(kWarps * 32), 0, stream, false, xb, rows, qb, scale); break;
        case 2: e = launch_k(quantize_rows_kernel<2>, grid, dim3(kWarps * 32), 0, stream, false, xb, rows, qb, scale); break;
        case 4: e = launch_k(quantize_rows_kernel<4>, grid, dim3(kWarps * 32), 0, stream, false, xb, rows, qb, scale); break;
        case 8: e = launch_k(quantize_rows_kernel<8>, grid, dim3(kWarps * 32), 0, stream, false, xb, rows, qb, scale); break;
        case 16: e = launch_k(quantize_rows_kernel<16>, grid, dim3(kWarps * 32), 0, stream, false, xb, rows, qb, scale); break;
        case 32: e = launch_k(quantize_rows_kernel<32>, grid, dim3(kWarps * 32), 0, stream, false, xb, rows, qb, scale); break;
        default: return DSV4_ERR_INVALID_ARG;    // dims between the powers of two
    }
    return e == cudaSuccess ? DSV4_OK : DSV4_ERR_LAUNCH;
}

}  // namespace dsv4

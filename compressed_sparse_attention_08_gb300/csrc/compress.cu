// Block compressor + RMSNorm + partial RoPE (one CTA per compressed entry).
//
// Sources: "nvfp4-megamoe-kernel: compare v0.1-e2e-working...v-c1-c2-c3-20260602",
// compressor_reduce.cu (hca_compress_reduce_kernel, apply_kv_norm_kernel) with the fix of
// "nvfp4-megamoe-kernel: compare master..pure-nvfp4", commit "Fix two correctness bugs"
// item 1 (the positional bias enters the logits Z + B only), and PERFORMANCE_AUDIT.md "P5"
// (interleaved-pair RoPE of the last rope_dim channels).
//
// Design: the reduce is tiny (ratio x dim values per entry) and latency-bound, so the
// three steps are fused in one kernel: each thread owns channels c = tid + 128 i, runs the
// max pass and the exp/sum pass over the block's tokens in fp32 (reads hit L1), the CTA
// reduces sum(x^2) with warp shuffles, and the rope pairs are rotated from shared memory
// with angles formed in fp64 (positions reach 2^20, where an fp32 angle would be off by
// hundredths of a radian). One bf16 rounding at the output, written straight into the
// caller's cache rows.
#include "common.cuh"
#include "internal.h"

namespace dsv4 {
namespace {

constexpr int kThreads = 128;
constexpr int kMaxChan = 8;          // dim <= 1024

__global__ void __launch_bounds__(kThreads)
compress_kernel(const __nv_bfloat16* __restrict__ C, const __nv_bfloat16* __restrict__ Z,
                const float* __restrict__ bias, const float* __restrict__ gamma,
                const int64_t* __restrict__ pos0, __nv_bfloat16* __restrict__ out,
                const int32_t* __restrict__ out_row0, int tokens, int dim, int ratio,
                int rope_dim, int out_rows, float eps, double theta) {
    const int b = blockIdx.x;          // block (entry) within the sequence
    const int s = blockIdx.y;          // sequence
    const int tid = threadIdx.x;
    const int n_blocks = tokens / ratio;
    if (b >= n_blocks) return;

    __shared__ float y[1024];
    __shared__ float warp_sum[kThreads / 32];

    const size_t tok0 = static_cast<size_t>(s) * tokens + static_cast<size_t>(b) * ratio;
    float x[kMaxChan];
    float sq = 0.f;
#pragma unroll
    for (int i = 0; i < kMaxChan; ++i) {
        const int c = tid + i * kThreads;
        x[i] = 0.f;
        if (c >= dim) continue;
        float m = -INFINITY;
        for (int t = 0; t < ratio; ++t) {
            const float a = __bfloat162float(Z[(tok0 + t) * dim + c]) + bias[static_cast<size_t>(t) * dim + c];
            m = fmaxf(m, a);
        }
        float den = 0.f, num = 0.f;
        for (int t = 0; t < ratio; ++t) {
            const float a = __bfloat162float(Z[(tok0 + t) * dim + c]) + bias[static_cast<size_t>(t) * dim + c];
            const float e = expf(a - m);
            den += e;
            num = fmaf(e, __bfloat162float(C[(tok0 + t) * dim + c]), num);   // no bias on C
        }
        x[i] = num / den;
        sq = fmaf(x[i], x[i], sq);
    }
    // RMSNorm: mean of x^2 over all dim channels
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
    if ((tid & 31) == 0) warp_sum[tid >> 5] = sq;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kThreads / 32; ++w) tot += warp_sum[w];
    const float inv = 1.0f / sqrtf(tot / static_cast<float>(dim) + eps);
#pragma unroll
    for (int i = 0; i < kMaxChan; ++i) {
        const int c = tid + i * kThreads;
        if (c < dim) y[c] = x[i] * inv * gamma[c];
    }
    __syncthreads();
    // RoPE: pair j rotates channels (d0, d0 + 1), d0 = dim - rope_dim + 2j
    const int64_t pos = pos0[s] + static_cast<int64_t>(b) * ratio;
    for (int j = tid; j < rope_dim / 2; j += kThreads) {
        const int d0 = dim - rope_dim + 2 * j;
        const double ang = static_cast<double>(pos) * pow(theta, -2.0 * j / rope_dim);
        double sd, cd;
        sincos(ang, &sd, &cd);
        const float cs = static_cast<float>(cd), sn = static_cast<float>(sd);
        const float e = y[d0], o = y[d0 + 1];
        y[d0] = e * cs - o * sn;
        y[d0 + 1] = e * sn + o * cs;
    }
    __syncthreads();
    const int row = (out_row0 ? out_row0[s] : 0) + b;
    if (row < 0 || row >= out_rows) return;   // host checks make this unreachable
    __nv_bfloat16* dst = out + (static_cast<size_t>(s) * out_rows + row) * dim;
    for (int c = tid; c < dim; c += kThreads) dst[c] = __float2bfloat16_rn(y[c]);
}

}  // namespace

int launch_compress(const dsv4_compress_args& a, cudaStream_t stream) {
    const int n_blocks = a.tokens / a.ratio;
    if (a.batch == 0 || n_blocks == 0) return DSV4_OK;
    dim3 grid(n_blocks, a.batch);
    compress_kernel<<<grid, kThreads, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(a.C), static_cast<const __nv_bfloat16*>(a.Z), a.bias,
        a.gamma, a.pos0, static_cast<__nv_bfloat16*>(a.out), a.out_row0, a.tokens, a.dim,
        a.ratio, a.rope_dim, a.out_rows, a.eps, a.rope_theta);
    count_launch();
    return cudaGetLastError() == cudaSuccess ? DSV4_OK : DSV4_ERR_LAUNCH;
}

}  // namespace dsv4

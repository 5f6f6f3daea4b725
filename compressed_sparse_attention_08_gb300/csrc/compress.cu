// Block compressor + RMSNorm + partial RoPE (one CTA per compressed entry).
//
// Sources: "nvfp4-megamoe-kernel: compare v0.1-e2e-working...v-c1-c2-c3-20260602",
// compressor_reduce.cu (hca_compress_reduce_kernel, apply_kv_norm_kernel) with the fix of
// "nvfp4-megamoe-kernel: compare master..pure-nvfp4", commit "Fix two correctness bugs"
// item 1 (the positional bias enters the logits Z + B only), and PERFORMANCE_AUDIT.md "P5"
// (interleaved-pair RoPE of the last rope_dim channels).
//
// Two-stream (CSA) form, "nvfp4-megamoe-kernel: compare v0.1-e2e-working...v-c1-c2-c3-20260602",
// compressor_reduce.cu "CSA compressor reduce kernel": the projections carry 2*dim channels,
// entry i pools block i-1 from stream a (channels [0, dim)) and block i from stream b
// (channels [dim, 2 dim)) under one softmax per channel; the bias has 2*dim columns, on the
// logits only. Entry 0 reads its stream-a block from the previous-block buffer, if given.
//
// Design: the reduce is tiny (ratio x dim values per entry) and latency-bound, so the
// three steps are fused in one kernel, and one launch serves up to two compressions (the
// main KV and the indexer keys of a decode step). Each thread owns channels
// c = tid + 128 i and runs an online softmax (running max, rescaled sums) over the block's
// tokens in fp32, 8 tokens at a time with all loads of a chunk issued before any is used;
// the CTA reduces sum(x^2) with warp shuffles, and the rope pairs are rotated from shared
// memory.
// RoPE angles: positions reach 2^20, where an fp32 angle pos * f would be off by hundredths
// of a radian, so the angle is formed in fp64 from a host-computed table of the
// frequencies f_j = theta^(-2j/rope_dim), reduced to [-pi, pi] with a two-constant
// Cody-Waite reduction using fused multiply-adds (W. J. Cody and W. Waite, "Software Manual
// for the Elementary Functions", 1980; the FMA form as in J.-M. Muller, "Elementary
// Functions", ch. 11), and only then passed to the fp32 sincos. One bf16 rounding at the
// output, written straight into the caller's cache rows.
#include <cmath>

#include "common.cuh"
#include "internal.h"

namespace dsv4 {
namespace {

constexpr int kThreads = 128;
constexpr int kMaxChan = 8;          // dim <= 1024
constexpr int kMaxPairs = 64;        // rope_dim <= 128

struct CompressJob {
    const __nv_bfloat16* C;
    const __nv_bfloat16* Z;
    const __nv_bfloat16* prev_C;     // two-stream form: the block before C's first block, or null
    const __nv_bfloat16* prev_Z;
    int overlap;                     // 0: plain blocks; 1: two-stream (CSA) form, 2*dim channels
    const float* bias;
    const float* gamma;
    const int64_t* pos0;
    __nv_bfloat16* out;
    const int32_t* out_row0;
    int batch, tokens, dim, ratio, rope_dim, out_rows, n_blocks;
    float eps;
    double two_pi_hi, two_pi_lo, inv_two_pi;
    double freq[kMaxPairs];
};

// zero_p/zero_n16: a workspace region (16-byte words) this launch clears for the kernels after
// it (the fused decode step), so the step needs no separate memset; they read it only after
// waiting for this grid.
__global__ void __launch_bounds__(kThreads, 1)
compress_kernel(const __grid_constant__ CompressJob j0, const __grid_constant__ CompressJob j1,
                uint4* zero_p, unsigned zero_n16) {
    pdl_trigger();
    {
        const unsigned nthr = gridDim.x * gridDim.y * gridDim.z * kThreads;
        const unsigned gt = ((blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x) * kThreads + threadIdx.x;
        for (unsigned i = gt; i < zero_n16; i += nthr) zero_p[i] = make_uint4(0, 0, 0, 0);
    }
    // every field of the selected job once, into registers (a runtime choice between two
    // parameter structs would otherwise turn each use into a slow generic load)
    const bool second = blockIdx.z != 0;
    const __nv_bfloat16* __restrict__ Cp = second ? j1.C : j0.C;
    const __nv_bfloat16* __restrict__ Zp = second ? j1.Z : j0.Z;
    const __nv_bfloat16* __restrict__ prevCp = second ? j1.prev_C : j0.prev_C;
    const __nv_bfloat16* __restrict__ prevZp = second ? j1.prev_Z : j0.prev_Z;
    const int overlap = second ? j1.overlap : j0.overlap;
    const float* __restrict__ biasp = second ? j1.bias : j0.bias;
    const float* __restrict__ gammap = second ? j1.gamma : j0.gamma;
    const int64_t* pos0p = second ? j1.pos0 : j0.pos0;
    __nv_bfloat16* outp = second ? j1.out : j0.out;
    const int32_t* row0p = second ? j1.out_row0 : j0.out_row0;
    const int batch = second ? j1.batch : j0.batch;
    const int tokens = second ? j1.tokens : j0.tokens;
    const int dim = second ? j1.dim : j0.dim;
    const int ratio = second ? j1.ratio : j0.ratio;
    const int rope_dim = second ? j1.rope_dim : j0.rope_dim;
    const int out_rows = second ? j1.out_rows : j0.out_rows;
    const int n_blocks = second ? j1.n_blocks : j0.n_blocks;
    const float eps = second ? j1.eps : j0.eps;
    const double two_pi_hi = j0.two_pi_hi, two_pi_lo = j0.two_pi_lo, inv_two_pi = j0.inv_two_pi;
    const int b = blockIdx.x;          // block (entry) within the sequence
    const int s = blockIdx.y;          // sequence
    const int tid = threadIdx.x;
    if (b >= n_blocks || s >= batch) return;

    __shared__ float y[1024];
    __shared__ float warp_sum[kThreads / 32];
    __shared__ double freq[kMaxPairs];
    if (tid < kMaxPairs) freq[tid] = second ? j1.freq[tid] : j0.freq[tid];
    // loads that do not depend on the reduction, issued early
    const int64_t pos_s = pos0p[s];
    const int row_base = row0p ? row0p[s] : 0;

    const size_t tok0 = static_cast<size_t>(s) * tokens + static_cast<size_t>(b) * ratio;
    // channels per token row: dim, or 2*dim in the two-stream form (stream a | stream b)
    const size_t w = overlap ? 2 * static_cast<size_t>(dim) : static_cast<size_t>(dim);
    // stream a of this entry: the previous block's tokens (in C, or the previous-block buffer
    // for entry 0), or none for the sequence's first block
    const __nv_bfloat16* aC = nullptr;
    const __nv_bfloat16* aZ = nullptr;
    if (overlap) {
        if (b > 0) {
            aC = Cp + (tok0 - ratio) * w;
            aZ = Zp + (tok0 - ratio) * w;
        } else if (prevCp) {
            aC = prevCp + static_cast<size_t>(s) * ratio * w;
            aZ = prevZp + static_cast<size_t>(s) * ratio * w;
        }
    }
    // this entry's own tokens: all channels (plain) or stream b (channels dim..2*dim-1)
    const size_t own_off = overlap ? static_cast<size_t>(dim) : 0;
    const __nv_bfloat16* oC = Cp + tok0 * w + own_off;
    const __nv_bfloat16* oZ = Zp + tok0 * w + own_off;
    float x[kMaxChan];
    float sq = 0.f;
#pragma unroll
    for (int i = 0; i < kMaxChan; ++i) {
        const int c = tid + i * kThreads;
        x[i] = 0.f;
        if (c >= dim) continue;
        float m = -INFINITY, den = 0.f, num = 0.f;
        // online softmax over one segment of `ratio` tokens (row stride w), 8 tokens at a time
        auto segment = [&](const __nv_bfloat16* Cs, const __nv_bfloat16* Zs, const float* bs) {
            for (int t0 = 0; t0 < ratio; t0 += 8) {
                float a[8], cv[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int t = t0 + u;
                    if (t < ratio) {
                        a[u] = __bfloat162float(Zs[static_cast<size_t>(t) * w + c]) + bs[static_cast<size_t>(t) * w + c];
                        cv[u] = __bfloat162float(Cs[static_cast<size_t>(t) * w + c]);
                    } else {
                        a[u] = -INFINITY;
                        cv[u] = 0.f;
                    }
                }
                float mc = a[0];
#pragma unroll
                for (int u = 1; u < 8; ++u) mc = fmaxf(mc, a[u]);
                const float mn = fmaxf(m, mc);
                const float sc = m == -INFINITY ? 0.f : expf(m - mn);
                den *= sc;
                num *= sc;
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const float e = a[u] == -INFINITY ? 0.f : expf(a[u] - mn);
                    den += e;
                    num = fmaf(e, cv[u], num);   // no bias on C
                }
                m = mn;
            }
        };
        if (aC) segment(aC, aZ, biasp);                 // stream a: bias columns [0, dim)
        segment(oC, oZ, biasp + own_off);               // own block: bias columns [dim, 2 dim) in the two-stream form
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
        if (c < dim) y[c] = x[i] * inv * gammap[c];
    }
    __syncthreads();
    // RoPE: pair p rotates channels (d0, d0 + 1), d0 = dim - rope_dim + 2p, by pos * f_p
    const double pos = static_cast<double>(pos_s + static_cast<int64_t>(b) * ratio);
    for (int p = tid; p < rope_dim / 2; p += kThreads) {
        const int d0 = dim - rope_dim + 2 * p;
        const double ang = pos * freq[p];
        const double kq = rint(ang * inv_two_pi);
        double r = fma(-kq, two_pi_hi, ang);
        r = fma(-kq, two_pi_lo, r);
        float sn, cs;
        sincosf(static_cast<float>(r), &sn, &cs);
        const float e = y[d0], o = y[d0 + 1];
        y[d0] = e * cs - o * sn;
        y[d0 + 1] = e * sn + o * cs;
    }
    __syncthreads();
    const int row = row_base + b;
    if (row < 0 || row >= out_rows) return;     // rows outside the destination are not written
    __nv_bfloat16* dst = outp + (static_cast<size_t>(s) * out_rows + row) * dim;
    for (int c = tid; c < dim; c += kThreads) dst[c] = __float2bfloat16_rn(y[c]);
}

CompressJob make_job(const dsv4_compress_args& a) {
    CompressJob j;
    j.C = static_cast<const __nv_bfloat16*>(a.C);
    j.Z = static_cast<const __nv_bfloat16*>(a.Z);
    j.prev_C = static_cast<const __nv_bfloat16*>(a.prev_C);
    j.prev_Z = static_cast<const __nv_bfloat16*>(a.prev_Z);
    j.overlap = a.overlap;
    j.bias = a.bias;
    j.gamma = a.gamma;
    j.pos0 = a.pos0;
    j.out = static_cast<__nv_bfloat16*>(a.out);
    j.out_row0 = a.out_row0;
    j.batch = a.batch;
    j.tokens = a.tokens;
    j.dim = a.dim;
    j.ratio = a.ratio;
    j.rope_dim = a.rope_dim;
    j.out_rows = a.out_rows;
    j.n_blocks = a.tokens / a.ratio;
    j.eps = a.eps;
    // 2*pi as an unevaluated sum hi + lo of two doubles; lo = 2*pi - hi to double precision
    // (2*pi = 6.28318530717958647692528676655900576839...).
    j.two_pi_hi = 6.283185307179586;
    j.two_pi_lo = 2.4492935982947064e-16;
    j.inv_two_pi = 1.0 / j.two_pi_hi;
    for (int p = 0; p < kMaxPairs; ++p)
        j.freq[p] = p < a.rope_dim / 2 ? std::pow(a.rope_theta, -2.0 * p / a.rope_dim) : 0.0;
    return j;
}

}  // namespace

int launch_compress2(const dsv4_compress_args* a, const dsv4_compress_args* b, cudaStream_t stream,
                     void* zero, size_t zero_bytes) {
    const unsigned n16 = static_cast<unsigned>((zero_bytes + 15) / 16);
    auto memset_only = [&]() {
        return n16 == 0 || cudaMemsetAsync(zero, 0, size_t(n16) * 16, stream) == cudaSuccess ? DSV4_OK
                                                                                            : DSV4_ERR_LAUNCH;
    };
    if (!a && !b) return memset_only();
    if (!a) { a = b; b = nullptr; }
    const CompressJob j0 = make_job(*a);
    const CompressJob j1 = b ? make_job(*b) : j0;
    const int nb = j0.n_blocks > j1.n_blocks ? j0.n_blocks : j1.n_blocks;
    const int bs = j0.batch > j1.batch ? j0.batch : j1.batch;
    if (nb == 0 || bs == 0) return memset_only();
    dim3 grid(nb, bs, b ? 2 : 1);
    count_launch();
    return launch_k(compress_kernel, grid, dim3(kThreads), 0, stream, false, j0, j1,
                    static_cast<uint4*>(zero), n16) == cudaSuccess
               ? DSV4_OK : DSV4_ERR_LAUNCH;
}

int launch_compress(const dsv4_compress_args& a, cudaStream_t stream) {
    return launch_compress2(&a, nullptr, stream, nullptr, 0);
}

}  // namespace dsv4

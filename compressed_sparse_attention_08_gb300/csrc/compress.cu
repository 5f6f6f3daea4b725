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

#include <cuda_fp8.h>

#include "common.cuh"
#include "internal.h"

namespace dsv4 {
namespace {

// 256 threads at no more than 128 registers each (launch bounds of two CTAs per SM): a
// compressor CTA fits beside a scoring CTA, which the fused step starts while it runs
constexpr int kThreads = 256;
constexpr int kMaxChan = 4;          // channels per thread: dim <= 1024
// tokens per load round (every channel's loads in flight together): 4 for short blocks under
// the register bound above, 8 for long blocks (ratio >= 16, where nothing runs beside)
constexpr int kChunkShort = 4, kChunkLong = 8, kLongRatio = 16;
// long blocks with 8-channel vector loads: threads and tokens per load round
constexpr int kWideThreads = 512, kWideRound = 4;
constexpr int kMaxPairs = 64;        // rope_dim <= 128

struct CompressJob {
    const __nv_bfloat16* C;
    const __nv_bfloat16* Z;
    const __nv_bfloat16* prev_C;     // two-stream form: the block before C's first block, or null
    const __nv_bfloat16* prev_Z;
    int overlap;                     // 0: plain blocks; 1: two-stream (CSA) form, 2*dim channels
    float* out_scale;                // FP8 output: [batch, out_rows] entry scales, out holds E4M3
    int out_fp8;                     // 0 bf16; 1 FP8 entries; 2 mixed (FP8 + bf16 RoPE part)
    __nv_bfloat16* out_rope;         // mixed: [batch, out_rows, rope_dim]
    const float* bias;
    const float* gamma;
    const int64_t* pos0;
    __nv_bfloat16* out;
    const int32_t* out_row0;
    int batch, tokens, dim, ratio, rope_dim, out_rows, n_blocks;
    float eps;
    double freq[kMaxPairs];
};

// One compressed entry: the pooled tokens are `ratio` rows of the own block (channels
// own_off .. own_off + dim - 1 of rows oC/oZ, bias columns own_off..) and, in the two-stream
// form, `ratio` rows of the previous block's stream a (channels 0..dim-1 of aC/aZ, bias
// columns 0..), consecutive tokens `w` elements apart.
struct EntryIn {
    const __nv_bfloat16* aC;     // stream a (null: none)
    const __nv_bfloat16* aZ;
    const __nv_bfloat16* oC;     // own block, row 0, channel 0 of the row
    const __nv_bfloat16* oZ;
    size_t w, own_off;
    const float* bias;           // [ratio, w]
    const float* gamma;          // [dim]
    int dim, ratio, rope_dim;
    float eps;
    double pos;                  // RoPE position of the entry
    __nv_bfloat16* dst;          // the entry's output row, or null (computed, not stored)
    uint8_t* dst8;               // FP8 output: the entry's E4M3 row (dst is then null), or null
    float* dst_scale;            // FP8 output: the entry's scale
    int q_dim;                   // FP8 output: channels [0, q_dim) quantized (dim, or
                                 // dim - rope_dim for the mixed KV storage)
    __nv_bfloat16* dst_rope;     // mixed KV storage: channels [q_dim, dim) as bf16, or null
};

template <int NT>
__device__ void entry_finish(const EntryIn& in, const double* freq, float* y, float* warp_sum);

// The whole CTA (kThreads) computes one entry: per-channel online softmax of Z + bias over the
// pooled tokens and the weighted sum of C in fp32, RMSNorm over the dim channels, RoPE of the
// last rope_dim channels with the angle formed in fp64 and Cody-Waite reduced, one bf16
// rounding. freq: the rope frequencies in shared memory (already visible to the CTA).
template <int kChunk>
__device__ void entry_math(const EntryIn& in, const double* freq, float* y, float* warp_sum) {
    const int tid = threadIdx.x;
    const int dim = in.dim, ratio = in.ratio;
    const size_t w = in.w;
    // per channel (c = tid + i * kThreads): online softmax of Z + bias over the pooled tokens
    // and the weighted sum of C, kChunk tokens at a time; each round issues the loads of all
    // of the thread's channels before any is used (the rounds are dependent memory trips)
    float m[kMaxChan], den[kMaxChan], num[kMaxChan];
#pragma unroll
    for (int i = 0; i < kMaxChan; ++i) { m[i] = -INFINITY; den[i] = 0.f; num[i] = 0.f; }
    auto segment = [&](const __nv_bfloat16* Cs, const __nv_bfloat16* Zs, const float* bs) {
        for (int t0 = 0; t0 < ratio; t0 += kChunk) {
            // every load of the round (the thread's channels x kChunk tokens) is issued before
            // the first use: a use right behind its load would stall the in-order issue of the
            // loads after it
            __nv_bfloat16 zr[kMaxChan][kChunk], cr[kMaxChan][kChunk];
            float br[kMaxChan][kChunk];
#pragma unroll
            for (int i = 0; i < kMaxChan; ++i) {
                const int c = tid + i * kThreads;
                if (c < dim) {
#pragma unroll
                    for (int u = 0; u < kChunk; ++u) {
                        const size_t o = static_cast<size_t>(min(t0 + u, ratio - 1)) * w + c;
                        zr[i][u] = Zs[o];
                        br[i][u] = bs[o];
                        cr[i][u] = Cs[o];
                    }
                }
            }
            float a[kMaxChan][kChunk], cv[kMaxChan][kChunk];
#pragma unroll
            for (int i = 0; i < kMaxChan; ++i) {
                const bool cok = tid + i * kThreads < dim;
#pragma unroll
                for (int u = 0; u < kChunk; ++u) {
                    const bool ok = cok && t0 + u < ratio;
                    a[i][u] = ok ? __bfloat162float(zr[i][u]) + br[i][u] : -INFINITY;
                    cv[i][u] = ok ? __bfloat162float(cr[i][u]) : 0.f;
                }
            }
#pragma unroll
            for (int i = 0; i < kMaxChan; ++i) {
                float mc = a[i][0];
#pragma unroll
                for (int u = 1; u < kChunk; ++u) mc = fmaxf(mc, a[i][u]);
                const float mn = fmaxf(m[i], mc);
                const float sc = m[i] == -INFINITY ? 0.f : exp_e(m[i] - mn);
                den[i] *= sc;
                num[i] *= sc;
#pragma unroll
                for (int u = 0; u < kChunk; ++u) {
                    const float e = a[i][u] == -INFINITY ? 0.f : exp_e(a[i][u] - mn);
                    den[i] += e;
                    num[i] = fmaf(e, cv[i][u], num[i]);   // no bias on C
                }
                m[i] = mn;
            }
        }
    };
    if (in.aC) segment(in.aC, in.aZ, in.bias);          // stream a: bias columns [0, dim)
    segment(in.oC + in.own_off, in.oZ + in.own_off, in.bias + in.own_off);
#pragma unroll
    for (int i = 0; i < kMaxChan; ++i) {
        const int c = tid + i * kThreads;
        if (c < dim) y[c] = num[i] / den[i];
    }
    __syncthreads();
    entry_finish<kThreads>(in, freq, y, warp_sum);
}

// RMSNorm, RoPE and the output of an entry whose pooled channels x_c are in y[0, dim) (written
// by every thread of the CTA before a barrier). Thread t takes channels t + NT i for the
// sum of squares, as the pooling did.
template <int NT>
__device__ void entry_finish(const EntryIn& in, const double* freq, float* y, float* warp_sum) {
    const int tid = threadIdx.x;
    const int dim = in.dim;
    float sq = 0.f;
    for (int c = tid; c < dim; c += NT) sq = fmaf(y[c], y[c], sq);
    // RMSNorm: mean of x^2 over all dim channels
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
    if ((tid & 31) == 0) warp_sum[tid >> 5] = sq;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int k = 0; k < NT / 32; ++k) tot += warp_sum[k];
    const float inv = 1.0f / sqrtf(tot / static_cast<float>(dim) + in.eps);
    for (int c = tid; c < dim; c += NT) y[c] = y[c] * inv * in.gamma[c];
    __syncthreads();
    // RoPE: pair p rotates channels (d0, d0 + 1), d0 = dim - rope_dim + 2p, by pos * f_p
    for (int p = tid; p < in.rope_dim / 2; p += NT) {
        const int d0 = dim - in.rope_dim + 2 * p;
        float sn, cs;
        sincosf(reduced_angle(in.pos * freq[p]), &sn, &cs);
        const float e = y[d0], o = y[d0 + 1];
        y[d0] = e * cs - o * sn;
        y[d0 + 1] = e * sn + o * cs;
    }
    __syncthreads();
    if (in.dst)
        for (int c = tid; c < dim; c += NT) in.dst[c] = __float2bfloat16_rn(y[c]);
    if (in.dst8) {
        // FP8 E4M3 channels [0, q_dim): scale = amax / 448 over them (fp32), code =
        // E4M3(y / scale); the mixed storage keeps channels [q_dim, dim) (the RoPE part) as bf16
        const int qd = in.q_dim;
        float amax = 0.f;
        for (int c = tid; c < qd; c += NT) amax = fmaxf(amax, fabsf(y[c]));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        __syncthreads();                         // every thread has read warp_sum above
        if ((tid & 31) == 0) warp_sum[tid >> 5] = amax;
        __syncthreads();
        float m = 0.f;
#pragma unroll
        for (int k = 0; k < NT / 32; ++k) m = fmaxf(m, warp_sum[k]);
        const float sc = m > 0.f ? m / 448.0f : 1.0f;
        if (tid == 0) *in.dst_scale = sc;
        for (int c = tid; c < qd; c += NT)
            in.dst8[c] = static_cast<uint8_t>(__nv_cvt_float_to_fp8(y[c] / sc, __NV_SATFINITE, __NV_E4M3));
        if (in.dst_rope)
            for (int c = qd + tid; c < dim; c += NT) in.dst_rope[c - qd] = __float2bfloat16_rn(y[c]);
    }
}

// Long blocks (ratio >= kLongRatio, dim a multiple of 8): the pooled tokens of the channels
// [c_lo, c_lo + cn) are shared out over NT / (cn / 8) token groups, each thread taking 8
// channels (16-byte loads of C and Z, two of the bias) of every NT / (cn / 8)-th token, kRound
// tokens per round with all of a round's loads issued before any use; each group's
// online-softmax state (max, denominator, weighted sum per channel) then goes through shared
// memory and the groups are merged per channel into y[c_lo, c_lo + cn). Dependent load rounds:
// ratio / (groups * kRound) instead of ratio / kChunkLong. The channels of a softmax are
// independent, so an entry's channels may be split over several CTAs (c_lo, cn).
template <int NT, int kRound>
__device__ void pool_wide(const EntryIn& in, float* y, float* st /* [3][NT * 8] */, int c_lo, int cn) {
    const int tid = threadIdx.x;
    const int ratio = in.ratio;
    const int dim = cn;                          // the channels pooled here
    const int cg_n = cn / 8, groups = NT / cg_n;
    const int cg = tid % cg_n, tg = tid / cg_n;
    const size_t w = in.w;
    float m[8], den[8], num[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) { m[j] = -INFINITY; den[j] = 0.f; num[j] = 0.f; }
    auto segment = [&](const __nv_bfloat16* Cs, const __nv_bfloat16* Zs, const float* bs) {
        for (int t0 = tg; t0 < ratio; t0 += groups * kRound) {
            uint4 cr[kRound], zr[kRound];
            float4 b0[kRound], b1[kRound];
#pragma unroll
            for (int u = 0; u < kRound; ++u) {
                const int t = t0 + u * groups;
                const size_t o = static_cast<size_t>(t < ratio ? t : tg) * w + c_lo + cg * 8;
                cr[u] = __ldg(reinterpret_cast<const uint4*>(Cs + o));
                zr[u] = __ldg(reinterpret_cast<const uint4*>(Zs + o));
                b0[u] = __ldg(reinterpret_cast<const float4*>(bs + o));
                b1[u] = __ldg(reinterpret_cast<const float4*>(bs + o + 4));
            }
            // the round's logits; one rescale of the running sums per round
            float a[kRound][8], cv[kRound][8];
#pragma unroll
            for (int u = 0; u < kRound; ++u) {
                const bool ok = t0 + u * groups < ratio;
                const uint32_t zw[4] = {zr[u].x, zr[u].y, zr[u].z, zr[u].w};
                const uint32_t cw[4] = {cr[u].x, cr[u].y, cr[u].z, cr[u].w};
                const float bb[8] = {b0[u].x, b0[u].y, b0[u].z, b0[u].w, b1[u].x, b1[u].y, b1[u].z, b1[u].w};
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    a[u][j] = ok ? ((j & 1) ? bf16_hi(zw[j >> 1]) : bf16_lo(zw[j >> 1])) + bb[j] : -INFINITY;
                    cv[u][j] = ok ? ((j & 1) ? bf16_hi(cw[j >> 1]) : bf16_lo(cw[j >> 1])) : 0.f;
                }
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                float mc = a[0][j];
#pragma unroll
                for (int u = 1; u < kRound; ++u) mc = fmaxf(mc, a[u][j]);
                const float mn = fmaxf(m[j], mc);
                const float sc = m[j] == -INFINITY ? 0.f : exp_e(m[j] - mn);
                den[j] *= sc;
                num[j] *= sc;
#pragma unroll
                for (int u = 0; u < kRound; ++u) {
                    const float e = a[u][j] == -INFINITY ? 0.f : exp_e(a[u][j] - mn);
                    den[j] += e;
                    num[j] = fmaf(e, cv[u][j], num[j]);   // no bias on C
                }
                m[j] = mn;
            }
        }
    };
    if (tg < groups) {
        if (in.aC) segment(in.aC, in.aZ, in.bias);      // stream a: bias columns [0, dim)
        segment(in.oC + in.own_off, in.oZ + in.own_off, in.bias + in.own_off);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int c = cg * 8 + j;
            st[tg * dim + c] = m[j];
            st[NT * 8 + tg * dim + c] = den[j];
            st[2 * NT * 8 + tg * dim + c] = num[j];
        }
    }
    __syncthreads();
    // merge the groups per channel: x_c = sum_g num_g e^(m_g - M) / sum_g den_g e^(m_g - M)
    for (int c = tid; c < dim; c += NT) {
        float M = -INFINITY;
        for (int g = 0; g < groups; ++g) M = fmaxf(M, st[g * dim + c]);
        float dn = 0.f, nm = 0.f;
        for (int g = 0; g < groups; ++g) {
            const float mg = st[g * dim + c];
            const float e = mg == -INFINITY ? 0.f : exp_e(mg - M);
            dn = fmaf(st[NT * 8 + g * dim + c], e, dn);
            nm = fmaf(st[2 * NT * 8 + g * dim + c], e, nm);
        }
        y[c_lo + c] = nm / dn;
    }
    __syncthreads();
}

// entry_finish for an entry whose channels are split over the S CTAs of a cluster (CTA `part`
// holds y[c_lo, c_lo + cn)), bf16 output only: the RMSNorm's sum of squares is the one value
// that needs every channel; each CTA's partial goes into slot `part` of every CTA's s_sq
// through distributed shared memory, and a cluster barrier makes the S partials visible. The
// caller has arrived on the cluster barrier once at its start (so that every CTA of the cluster
// runs before any remote store); this function waits on that phase, then runs one more.
template <int NT, int S>
__device__ void entry_finish_split(const EntryIn& in, const double* freq, float* y, float* warp_sum,
                                   float* s_sq, int c_lo, int cn, uint32_t part) {
    const int tid = threadIdx.x;
    const int dim = in.dim;
    float sq = 0.f;
    for (int c = c_lo + tid; c < c_lo + cn; c += NT) sq = fmaf(y[c], y[c], sq);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
    if ((tid & 31) == 0) warp_sum[tid >> 5] = sq;
    __syncthreads();
    float mine = 0.f;
#pragma unroll
    for (int k = 0; k < NT / 32; ++k) mine += warp_sum[k];
    cluster_wait();                              // every CTA of the cluster has started
    if (tid < S) st_cluster_u32(cluster_map(&s_sq[part], static_cast<uint32_t>(tid)), __float_as_uint(mine));
    cluster_arrive();
    cluster_wait();                              // every CTA's partial is in s_sq
    float tot = 0.f;
#pragma unroll
    for (int r = 0; r < S; ++r) tot += s_sq[r];
    const float inv = 1.0f / sqrtf(tot / static_cast<float>(dim) + in.eps);
    for (int c = c_lo + tid; c < c_lo + cn; c += NT) y[c] = y[c] * inv * in.gamma[c];
    __syncthreads();
    // RoPE of the pairs whose first channel is here (c_lo is even: a pair is never split)
    for (int p = tid; p < in.rope_dim / 2; p += NT) {
        const int d0 = dim - in.rope_dim + 2 * p;
        if (d0 < c_lo || d0 >= c_lo + cn) continue;
        float sn, cs;
        sincosf(reduced_angle(in.pos * freq[p]), &sn, &cs);
        const float e = y[d0], o = y[d0 + 1];
        y[d0] = e * cs - o * sn;
        y[d0 + 1] = e * sn + o * cs;
    }
    __syncthreads();
    if (in.dst)
        for (int c = c_lo + tid; c < c_lo + cn; c += NT) in.dst[c] = __float2bfloat16_rn(y[c]);
}

// zero_p/zero_n16: a workspace region (16-byte words) this launch clears for the kernels after
// it (the fused decode step), so the step needs no separate memset; they read it only after
// waiting for this grid.
// NT threads; kWide: the long-block pooling of pool_wide (dim a multiple of 8; its group states
// in dynamic shared memory), else entry_math (NT = kThreads). kSplit > 1 (wide pooling, bf16
// outputs, dim a multiple of 8 * kSplit): a cluster of kSplit CTAs along x per entry, CTA r
// taking channels [r dim / kSplit, (r + 1) dim / kSplit) (grid.x = kSplit x blocks).
template <int kChunk, int kMinBlocks, int NT, bool kWide, int kSplit = 1>
__global__ void __launch_bounds__(NT, kMinBlocks)
compress_kernel(const __grid_constant__ CompressJob j0, const __grid_constant__ CompressJob j1,
                uint4* zero_p, unsigned zero_n16) {
    static_assert(kWide || NT == kThreads, "the per-channel pooling runs on kThreads threads");
    static_assert(kSplit == 1 || kWide, "only the wide pooling splits an entry's channels");
    pdl_trigger();
    {
        const unsigned nthr = gridDim.x * gridDim.y * gridDim.z * NT;
        const unsigned gt = ((blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x) * NT + threadIdx.x;
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
    const int out_fp8 = second ? j1.out_fp8 : j0.out_fp8;
    float* out_scalep = second ? j1.out_scale : j0.out_scale;
    __nv_bfloat16* out_ropep = second ? j1.out_rope : j0.out_rope;
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
    const int b = blockIdx.x / kSplit; // block (entry) within the sequence
    const uint32_t part = kSplit > 1 ? cluster_rank() : 0u;   // (the CTA's channel share)
    const int s = blockIdx.y;          // sequence
    const int tid = threadIdx.x;
    if (b >= n_blocks || s >= batch) return;

    __shared__ float y[1024];
    __shared__ float warp_sum[NT / 32];
    __shared__ float s_sq[kSplit];           // (split entries) every CTA's sum of squares
    if constexpr (kSplit > 1) cluster_arrive();   // waited on before the first remote store
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
    const int row = row_base + b;
    EntryIn in;
    in.aC = aC;
    in.aZ = aZ;
    in.oC = Cp + tok0 * w;
    in.oZ = Zp + tok0 * w;
    in.w = w;
    in.own_off = overlap ? static_cast<size_t>(dim) : 0;
    in.bias = biasp;
    in.gamma = gammap;
    in.dim = dim;
    in.ratio = ratio;
    in.rope_dim = rope_dim;
    in.eps = eps;
    in.pos = static_cast<double>(pos_s + static_cast<int64_t>(b) * ratio);
    // rows outside the destination are not written
    const bool in_range = row >= 0 && row < out_rows;
    const size_t orow = static_cast<size_t>(s) * out_rows + row;
    // mixed storage: codes of the channels without RoPE, rows of dim - rope_dim bytes
    const int q_dim = out_fp8 == 2 ? dim - (second ? j1.rope_dim : j0.rope_dim) : dim;
    in.dst = in_range && !out_fp8 ? outp + orow * dim : nullptr;
    in.dst8 = in_range && out_fp8 ? reinterpret_cast<uint8_t*>(outp) + orow * q_dim : nullptr;
    in.dst_scale = in_range && out_fp8 ? out_scalep + orow : nullptr;
    in.q_dim = q_dim;
    in.dst_rope = in_range && out_fp8 == 2 ? out_ropep + orow * (dim - q_dim) : nullptr;
    if constexpr (kSplit > 1) {
        extern __shared__ float group_state[];  // [3][NT * 8]
        const int cn = dim / kSplit;
        pool_wide<NT, kWideRound>(in, y, group_state, static_cast<int>(part) * cn, cn);
        entry_finish_split<NT, kSplit>(in, freq, y, warp_sum, s_sq, static_cast<int>(part) * cn, cn, part);
    } else if constexpr (kWide) {
        extern __shared__ float group_state[];  // [3][NT * 8]
        pool_wide<NT, kWideRound>(in, y, group_state, 0, dim);
        entry_finish<NT>(in, freq, y, warp_sum);
    } else {
        entry_math<kChunk>(in, freq, y, warp_sum);
    }
}

CompressJob make_job(const dsv4_compress_args& a) {
    CompressJob j;
    j.C = static_cast<const __nv_bfloat16*>(a.C);
    j.Z = static_cast<const __nv_bfloat16*>(a.Z);
    j.prev_C = static_cast<const __nv_bfloat16*>(a.prev_C);
    j.prev_Z = static_cast<const __nv_bfloat16*>(a.prev_Z);
    j.overlap = a.overlap;
    j.out_fp8 = a.out_fp8;
    j.out_scale = a.out_scale;
    j.out_rope = static_cast<__nv_bfloat16*>(a.out_rope);
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
    for (int p = 0; p < kMaxPairs; ++p)
        j.freq[p] = p < a.rope_dim / 2 ? std::pow(a.rope_theta, -2.0 * p / a.rope_dim) : 0.0;
    return j;
}

// ------------------------------------------------------------------ decode-time step
// One token per sequence per call. The token is staged; when it completes a block, the block
// is compressed into cache row n_comp and n_comp is bumped, all on the device, so every decode
// step runs the same launch (one captured graph serves them all).
// State per sequence s (caller-owned, zero at the start of a sequence): stage
// [2 blocks (0: in progress, 1: the previous block)][2 (C, Z)][ratio][w] bf16, fill[s] tokens of
// the block in progress, n_comp[s] entries written.
struct StepJob {
    const __nv_bfloat16* C;      // [batch, w] this step's token
    const __nv_bfloat16* Z;
    const float* bias;           // [ratio, w]
    const float* gamma;          // [dim]
    const int64_t* pos;          // [batch] the token's position
    __nv_bfloat16* stage;        // [batch, 2, 2, ratio, w]
    int32_t* fill;               // [batch]
    int32_t* n_comp;             // [batch]
    __nv_bfloat16* out;          // [batch, out_rows, dim] (or the FP8 / mixed layouts)
    int batch, dim, ratio, rope_dim, out_rows, overlap;
    float eps;
    double log2_theta;
    int out_fp8;                 // as CompressJob
    float* out_scale;
    __nv_bfloat16* out_rope;
};

__global__ void __launch_bounds__(kThreads, 2)
compress_step_kernel(const __grid_constant__ StepJob j) {
    __shared__ float y[1024];
    __shared__ float warp_sum[kThreads / 32];
    __shared__ double freq[kMaxPairs];
    const int s = blockIdx.x, tid = threadIdx.x;
    if (s >= j.batch) return;
    const size_t w = j.overlap ? 2 * static_cast<size_t>(j.dim) : static_cast<size_t>(j.dim);
    const size_t blk = 2 * static_cast<size_t>(j.ratio) * w;          // one staged block (C and Z)
    __nv_bfloat16* cur = j.stage + static_cast<size_t>(s) * 2 * blk;  // C rows, then Z rows
    __nv_bfloat16* prev = cur + blk;
    int f = j.fill[s];
    if (f < 0 || f >= j.ratio) f = 0;              // not a valid state: restart the block
    for (size_t c = tid; c < w; c += kThreads) {
        cur[static_cast<size_t>(f) * w + c] = j.C[static_cast<size_t>(s) * w + c];
        cur[(static_cast<size_t>(j.ratio) + f) * w + c] = j.Z[static_cast<size_t>(s) * w + c];
    }
    __syncthreads();                               // the staged token is visible to the CTA
    if (f + 1 < j.ratio) {
        if (tid == 0) j.fill[s] = f + 1;
        return;
    }
    const int nc = j.n_comp[s];
    if (tid < kMaxPairs)
        freq[tid] = tid < j.rope_dim / 2 ? exp2(-(2.0 * tid / j.rope_dim) * j.log2_theta) : 0.0;
    __syncthreads();
    EntryIn in;
    in.aC = j.overlap && nc > 0 ? prev : nullptr;  // the sequence's first entry has no stream a
    in.aZ = prev + static_cast<size_t>(j.ratio) * w;
    in.oC = cur;
    in.oZ = cur + static_cast<size_t>(j.ratio) * w;
    in.w = w;
    in.own_off = j.overlap ? static_cast<size_t>(j.dim) : 0;
    in.bias = j.bias;
    in.gamma = j.gamma;
    in.dim = j.dim;
    in.ratio = j.ratio;
    in.rope_dim = j.rope_dim;
    in.eps = j.eps;
    in.pos = static_cast<double>(j.pos[s] - (j.ratio - 1));   // the block's first token
    // a full cache keeps its rows: the entry is computed but not stored, n_comp stays
    const bool stored = nc >= 0 && nc < j.out_rows;
    const size_t orow = static_cast<size_t>(s) * j.out_rows + nc;
    const int q_dim = j.out_fp8 == 2 ? j.dim - j.rope_dim : j.dim;
    in.dst = stored && !j.out_fp8 ? j.out + orow * j.dim : nullptr;
    in.dst8 = stored && j.out_fp8 ? reinterpret_cast<uint8_t*>(j.out) + orow * q_dim : nullptr;
    in.dst_scale = stored && j.out_fp8 ? j.out_scale + orow : nullptr;
    in.q_dim = q_dim;
    in.dst_rope = stored && j.out_fp8 == 2 ? j.out_rope + orow * (j.dim - q_dim) : nullptr;
    entry_math<kChunkShort>(in, freq, y, warp_sum);
    if (j.overlap)                                 // this block is stream a of the next entry
        for (size_t c = tid; c < blk; c += kThreads) prev[c] = cur[c];
    if (tid == 0) {
        j.fill[s] = 0;
        if (stored) j.n_comp[s] = nc + 1;
    }
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
    const int rmax = j0.ratio > j1.ratio ? j0.ratio : j1.ratio;
    if (rmax >= kLongRatio) {
        // every job's channels in 8-channel groups (and their rows 16-byte aligned): the wide
        // pooling, its group states (3 x 512 x 8 floats) in dynamic shared memory
        const bool wide = j0.dim % 8 == 0 && (!b || j1.dim % 8 == 0);
        if (wide) {
            constexpr size_t kStateBytes = 3ull * kWideThreads * 8 * sizeof(float);
            // Few entries (the decode step's newest block: one per sequence) leave SMs idle
            // with one CTA per entry: split each entry's channels over a 2-CTA cluster when
            // the outputs are bf16 and the doubled grid still fits on the device at once.
            const int sms = sm_count() > 0 ? sm_count() : 148;
            const bool split = !j0.out_fp8 && (!b || !j1.out_fp8) && j0.dim % 16 == 0 && (!b || j1.dim % 16 == 0) &&
                               2ll * nb * bs * (b ? 2 : 1) <= sms;
            if (split) {
                if (once_per_device(reinterpret_cast<const void*>(compress_kernel<kChunkLong, 1, kWideThreads, true, 2>),
                                    kAttrLaunch, [] {
                                        return cudaFuncSetAttribute(compress_kernel<kChunkLong, 1, kWideThreads, true, 2>,
                                                                    cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                                    static_cast<int>(kStateBytes));
                                    }) != cudaSuccess)
                    return DSV4_ERR_LAUNCH;
                const dim3 g2(2u * nb, bs, b ? 2 : 1);
                return launch_cluster_k(compress_kernel<kChunkLong, 1, kWideThreads, true, 2>, g2, dim3(kWideThreads),
                                        kStateBytes, stream, false, 2u, j0, j1, static_cast<uint4*>(zero), n16) ==
                               cudaSuccess
                           ? DSV4_OK : DSV4_ERR_LAUNCH;
            }
            if (once_per_device(reinterpret_cast<const void*>(compress_kernel<kChunkLong, 1, kWideThreads, true>),
                                kAttrLaunch, [] {
                                    return cudaFuncSetAttribute(compress_kernel<kChunkLong, 1, kWideThreads, true>,
                                                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                                static_cast<int>(kStateBytes));
                                }) != cudaSuccess)
                return DSV4_ERR_LAUNCH;
            return launch_k(compress_kernel<kChunkLong, 1, kWideThreads, true>, grid, dim3(kWideThreads),
                            kStateBytes, stream, false, j0, j1, static_cast<uint4*>(zero), n16) == cudaSuccess
                       ? DSV4_OK : DSV4_ERR_LAUNCH;
        }
        return launch_k(compress_kernel<kChunkLong, 1, kThreads, false>, grid, dim3(kThreads), 0, stream, false, j0,
                        j1, static_cast<uint4*>(zero), n16) == cudaSuccess
                   ? DSV4_OK : DSV4_ERR_LAUNCH;
    }
    return launch_k(compress_kernel<kChunkShort, 2, kThreads, false>, grid, dim3(kThreads), 0, stream, false, j0, j1,
                    static_cast<uint4*>(zero), n16) == cudaSuccess
               ? DSV4_OK : DSV4_ERR_LAUNCH;
}

int launch_compress(const dsv4_compress_args& a, cudaStream_t stream) {
    return launch_compress2(&a, nullptr, stream, nullptr, 0);
}

int launch_compress_step(const dsv4_compress_step_args& a, cudaStream_t stream) {
    if (a.batch == 0) return DSV4_OK;
    StepJob j;
    j.C = static_cast<const __nv_bfloat16*>(a.C);
    j.Z = static_cast<const __nv_bfloat16*>(a.Z);
    j.bias = a.bias;
    j.gamma = a.gamma;
    j.pos = a.pos;
    j.stage = static_cast<__nv_bfloat16*>(a.stage);
    j.fill = a.fill;
    j.n_comp = a.n_comp;
    j.out = static_cast<__nv_bfloat16*>(a.out);
    j.batch = a.batch;
    j.dim = a.dim;
    j.ratio = a.ratio;
    j.rope_dim = a.rope_dim;
    j.out_rows = a.out_rows;
    j.overlap = a.overlap;
    j.eps = a.eps;
    j.log2_theta = std::log2(a.rope_theta);
    j.out_fp8 = a.out_fp8;
    j.out_scale = a.out_scale;
    j.out_rope = static_cast<__nv_bfloat16*>(a.out_rope);
    count_launch();
    return launch_k(compress_step_kernel, dim3(a.batch), dim3(kThreads), 0, stream, false, j) == cudaSuccess
               ? DSV4_OK : DSV4_ERR_LAUNCH;
}

}  // namespace dsv4

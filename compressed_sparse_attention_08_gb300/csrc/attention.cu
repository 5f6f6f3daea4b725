// Gather into the caller's fixed buffer + shared-KV MQA attention with a per-head sink.
//
// Sources: "nvfp4-megamoe-kernel: compare v0.1-e2e-working...v-c1-c2-c3-20260602",
// commit "C2" (one pre-allocated gather buffer of top_k + window rows), ARCHITECTURE_AND_
// MEMORY_AUDIT.md "B2" (CSA gathers comp_kv[topk] then the window; HCA every compressed
// entry then the window), fmha_6warp_tma_multirow_multitile.cuh "Sink bias correction" (the
// sink is one extra logit in the scaled domain that adds to the denominator only),
// PERFORMANCE_AUDIT.md "P4" (V is the gathered K row itself); "nvfp4-megamoe-kernel: compare
// master..pure-nvfp4", single_shot_inference.py eager_attention (scale = 1/sqrt(hd)).
//
// Design (decode: few queries, many rows; prefill: many queries):
//   * a gather kernel materialises the gather buffer (the caller's, or workspace): one warp
//     per row, 16-byte vector loads of whole rows with several rows in flight per warp, so
//     the random 1 KB rows stream at memory speed across every SM;
//   * the attention kernel then reads that contiguous, L2-resident buffer in 64-row chunks
//     with TMA tile loads (8 per chunk, one per 64-dim box, 128-byte swizzle) into two
//     alternating buffers; Q arrives the same way, once per CTA;
//   * the chunks of one query (compressed slots first, then window slots) are cut into
//     `n_splits` contiguous ranges and the heads into groups of 16, one CTA per (range,
//     query, head group): a 4-sequence decode still fills the GPU while each split stays
//     long enough that its fp32 partial (16 heads x D) is small next to the rows it read;
//   * bf16 tensor-core MMAs (fp32 accumulate): S = Q K^T, an online softmax in fp32,
//     O += P V with P rounded to bf16; masked slots (index -1, past the window) are excluded
//     from the softmax;
//   * a split writes (m, l, O) partials; the combine kernel merges them per (query, head)
//     and adds the sink once: o = sum_s O_s e^(m_s-M) / (sum_s l_s e^(m_s-M) + e^(sink-M)),
//     M = max(sink, m_s). With one split the CTA finishes the output itself.
#include <cmath>

#include <cuda_fp8.h>

#include "common.cuh"
#include "internal.h"

namespace dsv4 {
namespace {

constexpr int kCH = 64;      // rows per chunk
constexpr int kNT = 256;     // 8 warps

struct AttnParams {
    const float* sink;             // [H]
    const int32_t* n_comp;         // [B]
    const int32_t* idx;            // [rows, top_k] or null
    const int64_t* q_pos;          // [rows] or null
    const int32_t* win_len;        // [B]
    __nv_bfloat16* out;            // [rows, H, D]
    float* part_ml;                // [rows, n_splits, hstride, 2]
    float* part_o;                 // [rows, n_splits, hstride, D]
    uint32_t* eword;
    int rows, n_q, H, max_comp, top_k, window, win_rows, ratio, slots, comp_chunks, n_chunks,
        chunks_per_split, n_splits, oob_row;
    int n_hg, hstride;             // head groups per query, heads per partial record (n_hg*HP)
    float scale;
    const int64_t* orp;            // [rows] positions of the output's inverse RoPE, or null
    int or_pairs;                  // rotated pairs: the last 2 * or_pairs channels
    double or_log2_theta;          // log2(theta): pair j turns at theta^(-2j / rope_dim)
    // mixed FP8 / bf16 compressed KV (decode kernel only), else null
    const uint8_t* kv_nope;        // [B, max_comp, nope_dim] E4M3 codes
    const float* kv_scale;         // [B, max_comp]
    const __nv_bfloat16* kv_rope;  // [B, max_comp, D - nope_dim]
    int nope_dim;
};

// Inverse RoPE of one output pair (channels c, c + 1, c even) of query row `row`: rotated back
// by pos * f_j when the pair lies in the last 2 * or_pairs channels of a D-channel head.
__device__ __forceinline__ void inverse_rope_pair(const AttnParams& p, int row, int c, int D,
                                                  float& e, float& o) {
    const int j = (c - (D - 2 * p.or_pairs)) >> 1;
    if (!p.orp || j < 0) return;
    const double freq = exp2(-(static_cast<double>(j) / p.or_pairs) * p.or_log2_theta);
    float sn, cs;
    sincosf(reduced_angle(static_cast<double>(p.orp[row]) * freq), &sn, &cs);
    const float e0 = e, o0 = o;
    e = e0 * cs + o0 * sn;
    o = -e0 * sn + o0 * cs;
}

// Fills the inverse-RoPE fields of the kernel parameters from the call's arguments.
void set_output_rope(AttnParams& p, const dsv4_attn_args& a) {
    p.orp = a.out_rope_pos;
    p.or_pairs = a.out_rope_pos ? a.out_rope_dim / 2 : 0;
    p.or_log2_theta = a.out_rope_pos ? std::log2(a.out_rope_theta) : 0.0;
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t* r) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t* r) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];"
                 : "=r"(r[0]), "=r"(r[1]) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t* r) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(addr));
}
__device__ __forceinline__ void mma_bf16(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// Byte offset of 16-byte chunk c16 of row r in a tile stored as 64-element (128-byte) boxes of
// `rows` rows each, 128-byte swizzle (chunk ^ (row & 7)) within every box.
__device__ __forceinline__ uint32_t boxoff(int r, int c16, int rows) {
    return static_cast<uint32_t>((c16 >> 3) * rows * 128 + r * 128 + (((c16 & 7) ^ (r & 7)) << 4));
}
// Row-major 64-column bf16 tile (128-byte rows), same swizzle.
__device__ __forceinline__ uint32_t swz128(int r, int c16) {
    return static_cast<uint32_t>(r * 128 + ((c16 ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

// ------------------------------------------------------------------ gather
// Rows of the gather buffer: slot j < top_k holds comp_kv[b, idx[j]] (zeros for -1), slot
// top_k + i the i-th window row of the query (zeros past the window). One warp per row, each
// lane moving 16-byte pieces; every warp takes kRowsPerWarp rows with all loads issued before
// any store, so hundreds of random 1 KB rows are in flight per SM.
constexpr int kRowsPerWarp = 4;

template <int D>
__global__ void __launch_bounds__(256)
gather_kernel(AttnParams p, const __nv_bfloat16* __restrict__ comp_kv,
              const __nv_bfloat16* __restrict__ win, __nv_bfloat16* __restrict__ gbuf) {
    constexpr int U = D / 8;                      // 16-byte pieces per row
    constexpr int PL = (U + 31) / 32;             // pieces per lane
    pdl_trigger();
    pdl_wait();                                   // the index list comes from the kernel before
    const int lane = threadIdx.x & 31;
    const long long total = static_cast<long long>(p.rows) * p.slots;
    const long long first = (static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5)) * kRowsPerWarp;
    uint4 v[kRowsPerWarp][PL];
    long long dst_row[kRowsPerWarp];
#pragma unroll
    for (int k = 0; k < kRowsPerWarp; ++k) {
        const long long gr = first + k;
        dst_row[k] = gr < total ? gr : -1;
        const __nv_bfloat16* src = nullptr;
        if (gr < total) {
            const int row = static_cast<int>(gr / p.slots), slot = static_cast<int>(gr - static_cast<long long>(row) * p.slots);
            const int b = row / p.n_q, t = row - b * p.n_q;
            if (slot < p.top_k) {
                const int nv = row_visible(nullptr, p.n_comp, p.q_pos, p.n_q, p.ratio, p.max_comp, row, nullptr);
                int e;
                if (p.idx) {
                    e = p.idx[static_cast<size_t>(row) * p.top_k + slot];
                    if (e >= nv) { if (lane == 0) flag_error(p.eword, DSV4_EWORD_BAD_INDEX); e = -1; }
                } else {
                    e = slot < nv ? slot : -1;
                }
                if (e >= 0) src = comp_kv + (static_cast<size_t>(b) * p.max_comp + e) * D;
            } else {
                int wl = p.win_len[b];
                wl = wl < 0 ? 0 : (wl > p.win_rows ? p.win_rows : wl);
                const int w_hi = t + wl - p.n_q;
                const int w_lo = w_hi - p.window + 1 > 0 ? w_hi - p.window + 1 : 0;
                const int w_top = w_hi < wl - 1 ? w_hi : wl - 1;
                const int w_cnt = w_top >= w_lo ? w_top - w_lo + 1 : 0;
                const int wi = slot - p.top_k;
                if (wi < w_cnt) src = win + (static_cast<size_t>(b) * p.win_rows + w_lo + wi) * D;
            }
        }
#pragma unroll
        for (int j = 0; j < PL; ++j) {
            const int u = lane + 32 * j;
            v[k][j] = (src && u < U) ? __ldcs(reinterpret_cast<const uint4*>(src) + u) : make_uint4(0, 0, 0, 0);
        }
    }
#pragma unroll
    for (int k = 0; k < kRowsPerWarp; ++k) {
        if (dst_row[k] < 0) continue;
#pragma unroll
        for (int j = 0; j < PL; ++j) {
            const int u = lane + 32 * j;
            if (u < U) reinterpret_cast<uint4*>(gbuf + dst_row[k] * D)[u] = v[k][j];
        }
    }
}

template <int D, int HP>
struct Cfg {
    static constexpr int NHG = HP / 16;         // 16-head groups
    static constexpr int NRG = 8 / NHG;         // row groups of the S tile
    static constexpr int RW = kCH / NRG;        // chunk rows per warp in S
    static constexpr int NDG = 8 / NHG;         // dim groups of the O tile
    static constexpr int DW = D / NDG;          // dims per warp in O
    static constexpr int NBOX = D / 64;
    static constexpr size_t KVBUF = static_cast<size_t>(kCH) * D * 2;
    static constexpr size_t OFF_KV = static_cast<size_t>(HP) * D * 2;
    static constexpr size_t OFF_P = OFF_KV + 2 * KVBUF;
    static constexpr size_t OFF_F = OFF_P + static_cast<size_t>(HP) * 128;
    static constexpr size_t N_F = 2ull * NRG * HP + 3ull * HP;
    static constexpr size_t OFF_I = align_up(OFF_F + N_F * 4, 16);
    static constexpr size_t OFF_BAR = align_up(OFF_I + 4ull * kCH * 4, 16);
    static constexpr size_t SMEM = OFF_BAR + 3 * 8 + 1024;   // + alignment slack
    static_assert(RW % 8 == 0 && DW % 16 == 0, "tile split");
};

template <int D, int HP>
__global__ void __launch_bounds__(kNT, 1)
attn_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap gmap,
            AttnParams p) {
    using C = Cfg<D, HP>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* sm = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    uint8_t* sQ = sm;
    uint8_t* sKV = sm + C::OFF_KV;
    uint8_t* sP = sm + C::OFF_P;
    float* red_max = reinterpret_cast<float*>(sm + C::OFF_F);
    float* red_sum = red_max + C::NRG * HP;
    float* m_run = red_sum + C::NRG * HP;
    float* l_run = m_run + HP;
    float* alpha_s = l_run + HP;
    int* okf = reinterpret_cast<int*>(sm + C::OFF_I);        // [2][kCH] row is valid
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::OFF_BAR);   // q, kv0, kv1

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, tq = lane & 3;
    const int row = blockIdx.y, split = blockIdx.x, hgrp = blockIdx.z;
    const int hbase = hgrp * HP;                           // first head of this CTA
    const int Hc = p.H - hbase < HP ? p.H - hbase : HP;    // heads handled here
    const int b = row / p.n_q, t = row - b * p.n_q;
    const int nv = row_visible(nullptr, p.n_comp, p.q_pos, p.n_q, p.ratio, p.max_comp, row, nullptr);
    int wl = p.win_len[b];
    wl = wl < 0 ? 0 : (wl > p.win_rows ? p.win_rows : wl);
    const int w_hi = t + wl - p.n_q;                       // the query's own window row
    const int w_lo = w_hi - p.window + 1 > 0 ? w_hi - p.window + 1 : 0;
    const int w_top = w_hi < wl - 1 ? w_hi : wl - 1;
    const int w_cnt = w_top >= w_lo ? w_top - w_lo + 1 : 0;
    const int kc = p.top_k;                                // compressed slots
    const int c0 = split * p.chunks_per_split;
    const int c1 = c0 + p.chunks_per_split < p.n_chunks ? c0 + p.chunks_per_split : p.n_chunks;

    pdl_trigger();
    if (tid < HP) { m_run[tid] = -INFINITY; l_run[tid] = 0.f; }
    // query rows past this CTA's heads stay zero (TMA writes only the first Hc rows of a box)
    for (int i = tid; i < C::NBOX * (HP - Hc) * 8; i += kNT) {
        const int box = i / ((HP - Hc) * 8), rem = i - box * (HP - Hc) * 8;
        const int r = Hc + rem / 8, c = rem & 7;
        *reinterpret_cast<uint4*>(sQ + box * HP * 128 + r * 128 + c * 16) = make_uint4(0, 0, 0, 0);
    }
    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        mbar_init(&bars[2], 1);
        fence_barrier_init();
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    if (tid == 0) {                  // the queries are inputs: they load before the wait below
        tma_prefetch_desc(&gmap);
        mbar_arrive_expect_tx(&bars[0], static_cast<uint32_t>(Hc) * D * 2);
        for (int box = 0; box < C::NBOX; ++box)
            tma_load_2d(sQ + box * HP * 128, &qmap, &bars[0], box * 64, row * p.H + hbase);
    }

    // rows of chunk c into buffer buf: validity flags, then 64-row tile loads from the gather
    // buffer (written by the gather kernel, so it is in L2)
    auto issue = [&](int c, int buf) {
        const bool comp = c < p.comp_chunks;
        const int slot0 = comp ? c * kCH : kc + (c - p.comp_chunks) * kCH;
        if (tid < kCH) {
            int ok = 0;
            if (comp) {
                const int slot = slot0 + tid;
                if (slot < kc) {
                    if (p.idx) {
                        const int e = p.idx[static_cast<size_t>(row) * p.top_k + slot];
                        ok = e >= 0 && e < nv;
                    } else {
                        ok = slot < nv;
                    }
                }
            } else {
                ok = (c - p.comp_chunks) * kCH + tid < w_cnt ? 1 : 0;
            }
            okf[buf * kCH + tid] = ok;
        }
        __syncthreads();
        if (tid == 0) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            uint64_t* bar = &bars[1 + buf];
            mbar_arrive_expect_tx(bar, static_cast<uint32_t>(kCH) * D * 2);
            uint8_t* dst = sKV + buf * C::KVBUF;
            const int y = row * p.slots + slot0;
            for (int box = 0; box < C::NBOX; ++box)
                tma_load_2d(dst + box * kCH * 128, &gmap, bar, box * 64, y);
        }
    };

    // warp roles inside the two tiles
    const int hg = warp % C::NHG;
    const int rg = warp / C::NHG;                          // S: row group
    const int dg = warp / C::NHG;                          // O: dim group
    const int h0 = hg * 16 + g, h1 = h0 + 8;
    float o[C::DW / 8][4];
#pragma unroll
    for (int i = 0; i < C::DW / 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;

    pdl_wait();             // the index list (and the workspace) belong to the kernels before
    if (hgrp == 0 && split == 0 && tid == 0)                         // report a bad count once
        row_visible(nullptr, p.n_comp, p.q_pos, p.n_q, p.ratio, p.max_comp, row, p.eword);
    bool dead = false;      // a bounded wait ran out: keep the barrier sequence, skip the math
    if (!mbar_wait(&bars[0], 0, nullptr)) { flag_error(p.eword, DSV4_EWORD_TIMEOUT); dead = true; }
    if (c0 < c1) issue(c0, 0);
    uint32_t phase[2] = {0u, 0u};
    for (int c = c0; c < c1; ++c) {
        const int buf = (c - c0) & 1;
        if (c + 1 < c1) issue(c + 1, buf ^ 1);
        if (!dead && !mbar_wait(&bars[1 + buf], phase[buf], nullptr)) {
            flag_error(p.eword, DSV4_EWORD_TIMEOUT);
            dead = true;
        }
        phase[buf] ^= 1u;
        const uint8_t* kvb = sKV + buf * C::KVBUF;
        const int* ok = okf + buf * kCH;
        // ---- S = Q K^T for (16 heads) x (RW rows)
        float s[C::RW / 8][4];
#pragma unroll
        for (int i = 0; i < C::RW / 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
        const uint32_t qa = smem_u32(sQ), kva = smem_u32(kvb);
        if (!dead) {
#pragma unroll 4
            for (int k0 = 0; k0 < D; k0 += 16) {
                uint32_t a[4];
                ldsm_x4(qa + boxoff(hg * 16 + (lane & 15), (k0 >> 3) + (lane >> 4), HP), a);
                if constexpr (C::RW >= 16) {
#pragma unroll
                    for (int n2 = 0; n2 < C::RW / 16; ++n2) {
                        uint32_t bb[4];
                        const int rb = C::RW * rg + 16 * n2 + (lane & 7) + ((lane >> 4) << 3);
                        ldsm_x4(kva + boxoff(rb, (k0 >> 3) + ((lane >> 3) & 1), kCH), bb);
                        mma_bf16(s[2 * n2], a, bb[0], bb[1]);
                        mma_bf16(s[2 * n2 + 1], a, bb[2], bb[3]);
                    }
                } else {
                    uint32_t bb[2];
                    const int rb = C::RW * rg + (lane & 7);
                    ldsm_x2(kva + boxoff(rb, (k0 >> 3) + ((lane >> 3) & 1), kCH), bb);
                    mma_bf16(s[0], a, bb[0], bb[1]);
                }
            }
        }
        // ---- mask, scale, chunk max per head
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < C::RW / 8; ++nt) {
            const int col = C::RW * rg + 8 * nt + 2 * tq;
            const bool v0 = ok[col] && !dead, v1 = ok[col + 1] && !dead;
            s[nt][0] = v0 ? s[nt][0] * p.scale : -INFINITY;
            s[nt][1] = v1 ? s[nt][1] * p.scale : -INFINITY;
            s[nt][2] = v0 ? s[nt][2] * p.scale : -INFINITY;
            s[nt][3] = v1 ? s[nt][3] * p.scale : -INFINITY;
            mx0 = fmaxf(mx0, fmaxf(s[nt][0], s[nt][1]));
            mx1 = fmaxf(mx1, fmaxf(s[nt][2], s[nt][3]));
        }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        if (tq == 0) { red_max[rg * HP + h0] = mx0; red_max[rg * HP + h1] = mx1; }
        __syncthreads();
        float mn0 = m_run[h0], mn1 = m_run[h1];
#pragma unroll
        for (int r = 0; r < C::NRG; ++r) {
            mn0 = fmaxf(mn0, red_max[r * HP + h0]);
            mn1 = fmaxf(mn1, red_max[r * HP + h1]);
        }
        // ---- P = exp(S - m), row sums, P to shared memory as bf16
        float sum0 = 0.f, sum1 = 0.f;
#pragma unroll
        for (int nt = 0; nt < C::RW / 8; ++nt) {
            const float p0 = s[nt][0] == -INFINITY ? 0.f : expf(s[nt][0] - mn0);
            const float p1 = s[nt][1] == -INFINITY ? 0.f : expf(s[nt][1] - mn0);
            const float p2 = s[nt][2] == -INFINITY ? 0.f : expf(s[nt][2] - mn1);
            const float p3 = s[nt][3] == -INFINITY ? 0.f : expf(s[nt][3] - mn1);
            sum0 += p0 + p1;
            sum1 += p2 + p3;
            const int col = C::RW * rg + 8 * nt + 2 * tq;
            *reinterpret_cast<uint32_t*>(sP + swz128(h0, col >> 3) + (col & 7) * 2) = pack_bf16(p0, p1);
            *reinterpret_cast<uint32_t*>(sP + swz128(h1, col >> 3) + (col & 7) * 2) = pack_bf16(p2, p3);
        }
        sum0 += __shfl_xor_sync(0xffffffffu, sum0, 1);
        sum0 += __shfl_xor_sync(0xffffffffu, sum0, 2);
        sum1 += __shfl_xor_sync(0xffffffffu, sum1, 1);
        sum1 += __shfl_xor_sync(0xffffffffu, sum1, 2);
        if (tq == 0) { red_sum[rg * HP + h0] = sum0; red_sum[rg * HP + h1] = sum1; }
        __syncthreads();
        if (tid < HP) {
            const float mo = m_run[tid];
            float mn = mo, ls = 0.f;
#pragma unroll
            for (int r = 0; r < C::NRG; ++r) { mn = fmaxf(mn, red_max[r * HP + tid]); ls += red_sum[r * HP + tid]; }
            const float al = mo == -INFINITY ? 0.f : expf(mo - mn);
            l_run[tid] = l_run[tid] * al + ls;
            m_run[tid] = mn;
            alpha_s[tid] = al;
        }
        __syncthreads();
        // ---- O = O * alpha + P V for (16 heads) x (DW dims)
        {
            const float al0 = alpha_s[h0], al1 = alpha_s[h1];
#pragma unroll
            for (int i = 0; i < C::DW / 8; ++i) { o[i][0] *= al0; o[i][1] *= al0; o[i][2] *= al1; o[i][3] *= al1; }
            const uint32_t pa = smem_u32(sP);
            if (!dead) {
#pragma unroll
                for (int kk = 0; kk < kCH / 16; ++kk) {
                    uint32_t a[4];
                    ldsm_x4(pa + swz128(hg * 16 + (lane & 15), 2 * kk + (lane >> 4)), a);
#pragma unroll
                    for (int n2 = 0; n2 < C::DW / 16; ++n2) {
                        const int d0 = C::DW * dg + 16 * n2;
                        uint32_t bb[4];
                        ldsm_x4_t(kva + boxoff(16 * kk + (lane & 7) + (((lane >> 3) & 1) << 3),
                                               (d0 >> 3) + (lane >> 4), kCH), bb);
                        mma_bf16(o[2 * n2], a, bb[0], bb[1]);
                        mma_bf16(o[2 * n2 + 1], a, bb[2], bb[3]);
                    }
                }
            }
        }
        __syncthreads();
    }
    if (p.n_splits == 1) {
        // finish here: sink once, normalise, bf16
        const float* sk = p.sink;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int h = half ? h1 : h0;
            if (h >= Hc) continue;
            const float m = m_run[h], l = l_run[h], snk = sk[hbase + h];
            const float M = fmaxf(m, snk);
            const float em = m == -INFINITY ? 0.f : expf(m - M);
            const float f = em / (l * em + expf(snk - M));
            __nv_bfloat16* dst = p.out + (static_cast<size_t>(row) * p.H + hbase + h) * D;
#pragma unroll
            for (int i = 0; i < C::DW / 8; ++i) {
                const int d = C::DW * dg + 8 * i + 2 * tq;
                float e0 = o[i][2 * half] * f, o0 = o[i][2 * half + 1] * f;
                inverse_rope_pair(p, row, d, D, e0, o0);
                *reinterpret_cast<uint32_t*>(dst + d) = pack_bf16(e0, o0);
            }
        }
    } else {
        const size_t part = static_cast<size_t>(row) * p.n_splits + split;
        float* po = p.part_o + (part * p.hstride + hbase) * D;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int h = half ? h1 : h0;
#pragma unroll
            for (int i = 0; i < C::DW / 8; ++i) {
                const int d = C::DW * dg + 8 * i + 2 * tq;
                *reinterpret_cast<float2*>(po + static_cast<size_t>(h) * D + d) =
                    make_float2(o[i][2 * half], o[i][2 * half + 1]);
            }
        }
        if (tid < HP) {
            p.part_ml[(part * p.hstride + hbase + tid) * 2 + 0] = m_run[tid];
            p.part_ml[(part * p.hstride + hbase + tid) * 2 + 1] = l_run[tid];
        }
    }
}

template <int D, int HP>
__global__ void __launch_bounds__(128)
attn_combine_kernel(AttnParams p) {
    constexpr int PER = D / 128;                 // dims per thread
    constexpr int kRegSplits = 24;               // splits whose partial O is loaded up front
    __shared__ float wgt[256];
    __shared__ float red[4];
    __shared__ float bcast[1];
    const int row = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
    const int ns = p.n_splits;
    pdl_wait();
    const int HS = p.hstride;
    const float* ml = p.part_ml + static_cast<size_t>(row) * ns * HS * 2;
    const float* po = p.part_o + static_cast<size_t>(row) * ns * HS * D + static_cast<size_t>(h) * D + tid * PER;
    // every load at once: this thread's dims of the first kRegSplits splits, and the splits'
    // maxima and sums (ns <= 256: two per thread)
    float ov[kRegSplits][PER];
#pragma unroll
    for (int s = 0; s < kRegSplits; ++s) {
        if (s < ns) {
            const float* src = po + static_cast<size_t>(s) * HS * D;
            if constexpr (PER == 4) {
                const float4 v = *reinterpret_cast<const float4*>(src);
                ov[s][0] = v.x; ov[s][1] = v.y; ov[s][2] = v.z; ov[s][3] = v.w;
            } else if constexpr (PER == 2) {
                const float2 v = *reinterpret_cast<const float2*>(src);
                ov[s][0] = v.x; ov[s][1] = v.y;
            } else {
                ov[s][0] = *src;
            }
        }
    }
    const float snk = p.sink[h];
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    if (tid < ns) { m0 = ml[(tid * HS + h) * 2]; l0 = ml[(tid * HS + h) * 2 + 1]; }
    if (tid + 128 < ns) { m1 = ml[((tid + 128) * HS + h) * 2]; l1 = ml[((tid + 128) * HS + h) * 2 + 1]; }
    float M = fmaxf(m0, m1);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    if ((tid & 31) == 0) red[tid >> 5] = M;
    __syncthreads();
    M = fmaxf(fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3])), snk);
    const float e0 = m0 == -INFINITY ? 0.f : expf(m0 - M);
    const float e1 = m1 == -INFINITY ? 0.f : expf(m1 - M);
    if (tid < ns) wgt[tid] = e0;
    if (tid + 128 < ns) wgt[tid + 128] = e1;
    float den = l0 * e0 + l1 * e1;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
    __syncthreads();
    if ((tid & 31) == 0) red[tid >> 5] = den;
    __syncthreads();
    if (tid == 0) bcast[0] = 1.0f / (red[0] + red[1] + red[2] + red[3] + expf(snk - M));
    __syncthreads();
    const float inv = bcast[0];
    float acc[PER];
#pragma unroll
    for (int j = 0; j < PER; ++j) acc[j] = 0.f;
#pragma unroll
    for (int s = 0; s < kRegSplits; ++s)
        if (s < ns) {
#pragma unroll
            for (int j = 0; j < PER; ++j) acc[j] = fmaf(ov[s][j], wgt[s], acc[j]);
        }
    for (int s = kRegSplits; s < ns; ++s) {
        const float* src = po + static_cast<size_t>(s) * HS * D;
#pragma unroll
        for (int j = 0; j < PER; ++j) acc[j] = fmaf(src[j], wgt[s], acc[j]);
    }
    __nv_bfloat16* dst = p.out + (static_cast<size_t>(row) * p.H + h) * D + tid * PER;
#pragma unroll
    for (int j = 0; j < PER; ++j) acc[j] *= inv;
    if constexpr (PER == 1) {
        // one channel per thread: the pair partner is the neighbouring lane
        const float partner = __shfl_xor_sync(0xffffffffu, acc[0], 1);
        if (p.orp) {
            float e = (tid & 1) ? partner : acc[0], o = (tid & 1) ? acc[0] : partner;
            inverse_rope_pair(p, row, tid & ~1, D, e, o);
            acc[0] = (tid & 1) ? o : e;
        }
        *dst = __float2bfloat16_rn(acc[0]);
    } else {
#pragma unroll
        for (int j = 0; j < PER; j += 2) {
            inverse_rope_pair(p, row, tid * PER + j, D, acc[j], acc[j + 1]);
            *reinterpret_cast<uint32_t*>(dst + j) = pack_bf16(acc[j], acc[j + 1]);
        }
    }
}

// ------------------------------------------------------------------ decode: fused gather + tcgen05
// One CTA per (128-slot chunk, query row, group of NH heads):
//   * the chunk's rows are copied straight from the compressed cache (or the window) into a
//     shared tile laid out as D/64 boxes of [128 rows][128 B] with the 128-byte swizzle, by
//     16-byte cp.async pieces (8 warps x 16 rows; invalid slots are zero-filled). The head
//     group 0 CTA then TMA-stores the tile into the caller's gather buffer;
//   * S^T = KV Q^T on the tensor cores: M = 128 slots, N = NH heads, K = D, fp32 in TMEM;
//   * the 128 x NH scores go through shared memory once, so each thread owns one head and
//     16 slots: per-head max and sum over the chunk, P = e^(s - m) rounded to bf16 into a
//     K-major operand tile [NH heads][128 slots];
//   * O^T = V^T P^T: M = 128 dims per tile (D/128 tiles), N = NH, K = 128 slots. V^T is the
//     same shared tile read as an MN-major operand (64 dims per 128-byte row, slot rows);
//   * the chunk's (m, l, O) go to the partials; the combine kernel merges the chunks of a
//     query and adds the sink once.
constexpr int kFC = 128;          // slots per chunk (the MMA's M)
constexpr int kFT = 256;          // 8 warps

template <int D, int NH>
struct FCfg {
    static constexpr int NBOX = D / 64;
    static constexpr int MT = D / 128;                               // M tiles of O^T
    static constexpr int U = D / 8;                                  // 16-byte pieces per row
    static constexpr size_t BOX = static_cast<size_t>(kFC) * 128;    // one 64-dim box of the tile
    static constexpr size_t OFF_Q = BOX * NBOX;
    static constexpr size_t OFF_P = OFF_Q + static_cast<size_t>(NBOX) * NH * 128;
    static constexpr size_t OFF_S = OFF_P + 2ull * NH * 128;
    static constexpr size_t OFF_R = OFF_S + static_cast<size_t>(kFC) * (NH + 1) * 4;
    static constexpr size_t OFF_OK = OFF_R + 2ull * 8 * NH * 4;
    static constexpr size_t OFF_BAR = align_up(OFF_OK + kFC * 4, 16);
    static constexpr size_t SMEM = OFF_BAR + 3 * 8 + 1024;           // + alignment slack
    static constexpr uint32_t NEED = static_cast<uint32_t>(NH + MT * NH);
    static constexpr uint32_t TCOLS = NEED <= 32 ? 32 : NEED <= 64 ? 64 : NEED <= 128 ? 128 : NEED <= 256 ? 256 : 512;
    static_assert(D % 128 == 0 && (NH == 16 || NH == 32), "decode tile shape");
};

template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[N]) {
    if constexpr (N == 8) DSV4_TMEM_LD_32x32b_X8(taddr, r);
    else if constexpr (N == 16) DSV4_TMEM_LD_32x32b_X16(taddr, r);
    else DSV4_TMEM_LD_32x32b_X32(taddr, r);
}

template <int D, int NH>
__global__ void __launch_bounds__(kFT, 1)
attn_decode_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap gmap,
                   AttnParams p, const __nv_bfloat16* __restrict__ comp_kv,
                   const __nv_bfloat16* __restrict__ win, int write_gather) {
    using C = FCfg<D, NH>;
    constexpr int HC = NH / 2;                                       // TMEM columns per warp
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint32_t tmem_slot;
    __shared__ volatile int abort_flag;
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* sm = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    uint8_t* sKV = sm;
    uint8_t* sQ = sm + C::OFF_Q;
    uint8_t* sP = sm + C::OFF_P;
    float* sS = reinterpret_cast<float*>(sm + C::OFF_S);
    float* red_m = reinterpret_cast<float*>(sm + C::OFF_R);
    float* red_l = red_m + 8 * NH;
    int* okf = reinterpret_cast<int*>(sm + C::OFF_OK);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::OFF_BAR);   // q loaded, S done, O done

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int chunk = blockIdx.x, row = blockIdx.y, hgrp = blockIdx.z;
    const int hbase = hgrp * NH;
    const int Hc = p.H - hbase < NH ? p.H - hbase : NH;
    const int b = row / p.n_q, t = row - b * p.n_q;
    pdl_trigger();
    const int nv = row_visible(nullptr, p.n_comp, p.q_pos, p.n_q, p.ratio, p.max_comp, row, nullptr);
    int wl = p.win_len[b];
    wl = wl < 0 ? 0 : (wl > p.win_rows ? p.win_rows : wl);
    const int w_hi = t + wl - p.n_q;                                 // the query's own window row
    const int w_lo = w_hi - p.window + 1 > 0 ? w_hi - p.window + 1 : 0;
    const int w_top = w_hi < wl - 1 ? w_hi : wl - 1;
    const int w_cnt = w_top >= w_lo ? w_top - w_lo + 1 : 0;

    // query rows past this CTA's heads stay zero (TMA writes only the first Hc rows of a box)
    for (int i = tid; i < C::NBOX * (NH - Hc) * 8; i += kFT) {
        const int box = i / ((NH - Hc) * 8), rem = i - box * (NH - Hc) * 8;
        *reinterpret_cast<uint4*>(sQ + box * NH * 128 + (Hc + rem / 8) * 128 + (rem & 7) * 16) =
            make_uint4(0, 0, 0, 0);
    }
    if (tid == 0) {
        for (int i = 0; i < 3; ++i) mbar_init(&bars[i], 1);
        abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0) tmem_alloc(&tmem_slot, C::TCOLS);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_slot;
    if (tid == 0) {                  // the queries are inputs: they load before the wait below
        tma_prefetch_desc(&gmap);
        mbar_arrive_expect_tx(&bars[0], static_cast<uint32_t>(Hc) * D * 2);
        for (int box = 0; box < C::NBOX; ++box)
            tma_load_2d(sQ + box * NH * 128, &qmap, &bars[0], box * 64, row * p.H + hbase);
    }

    pdl_wait();                      // the index list comes from the kernel before
    if (hgrp == 0 && chunk == 0 && tid == 0)                         // report a bad count once
        row_visible(nullptr, p.n_comp, p.q_pos, p.n_q, p.ratio, p.max_comp, row, p.eword);
    // ---- gather: warp w copies slots [16w, 16w + 16) of the chunk; lanes 0..15 resolve them
    {
        const int r0 = warp * 16;
        unsigned long long src = 0;                                  // bf16 row; 0: none
        long long ent = -1;                                          // mixed storage: entry row
        float escale = 0.f;
        if (lane < 16) {
            const int slot = chunk * kFC + r0 + lane;
            if (slot < p.top_k) {
                int e;
                if (p.idx) {
                    e = p.idx[static_cast<size_t>(row) * p.top_k + slot];
                    if (e >= nv) { flag_error(p.eword, DSV4_EWORD_BAD_INDEX); e = -1; }
                } else {
                    e = slot < nv ? slot : -1;
                }
                if (e >= 0) {
                    if (p.kv_nope) {
                        ent = static_cast<long long>(b) * p.max_comp + e;
                        escale = __ldg(&p.kv_scale[ent]);
                    } else {
                        src = reinterpret_cast<unsigned long long>(comp_kv + (static_cast<size_t>(b) * p.max_comp + e) * D);
                    }
                }
            } else if (slot < p.slots) {
                const int wi = slot - p.top_k;
                if (wi < w_cnt)
                    src = reinterpret_cast<unsigned long long>(win + (static_cast<size_t>(b) * p.win_rows + w_lo + wi) * D);
            }
            okf[r0 + lane] = src != 0 || ent >= 0;
        }
        if (!p.kv_nope) {
            for (int i = lane; i < 16 * C::U; i += 32) {
                const int r = i / C::U, c = i - r * C::U;
                const unsigned long long a = __shfl_sync(0xffffffffu, src, r);
                const int rr = r0 + r;
                uint8_t* dst = sKV + (c >> 3) * C::BOX + rr * 128 + (((c & 7) ^ (rr & 7)) << 4);
                if (a) cp_async16(dst, reinterpret_cast<const uint8_t*>(a) + c * 16);
                else *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
            }
        } else {
            // mixed storage: a 16-byte bf16 piece c of a compressed row is 8 codes (piece c <
            // ncp) dequantized here, or a piece of its bf16 RoPE part; every load of the warp's
            // 16 rows is issued (codes into registers) before the first is converted
            constexpr int kPer = 16 * C::U / 32;                     // pieces per lane
            const int ncp = p.nope_dim / 8;
            const int rope_b = (D - p.nope_dim) * 2;                 // bytes of a RoPE part
            uint2 code[kPer];
#pragma unroll
            for (int k = 0; k < kPer; ++k) {
                const int i = lane + 32 * k;
                const int r = i / C::U, c = i - r * C::U;
                const unsigned long long a = __shfl_sync(0xffffffffu, src, r);
                const long long en = __shfl_sync(0xffffffffu, ent, r);
                const int rr = r0 + r;
                uint8_t* dst = sKV + (c >> 3) * C::BOX + rr * 128 + (((c & 7) ^ (rr & 7)) << 4);
                code[k] = make_uint2(0u, 0u);
                if (a) {
                    cp_async16(dst, reinterpret_cast<const uint8_t*>(a) + c * 16);
                } else if (en >= 0) {
                    if (c < ncp)
                        code[k] = __ldg(reinterpret_cast<const uint2*>(p.kv_nope + static_cast<size_t>(en) * p.nope_dim) + c);
                    else
                        cp_async16(dst, reinterpret_cast<const uint8_t*>(p.kv_rope) + static_cast<size_t>(en) * rope_b +
                                            (c - ncp) * 16);
                } else {
                    *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
                }
            }
#pragma unroll
            for (int k = 0; k < kPer; ++k) {
                const int i = lane + 32 * k;
                const int r = i / C::U, c = i - r * C::U;
                const long long en = __shfl_sync(0xffffffffu, ent, r);
                const float sc = __shfl_sync(0xffffffffu, escale, r);
                if (en >= 0 && c < ncp) {                            // (a compressed row)
                    // channel = bf16( fp32(E4M3 code) * scale ): codes in byte order
                    uint32_t o[4];
                    const uint32_t w2[2] = {code[k].x, code[k].y};
#pragma unroll
                    for (int h = 0; h < 4; ++h) {
                        const __nv_fp8x2_storage_t pr =
                            static_cast<__nv_fp8x2_storage_t>((w2[h >> 1] >> (16 * (h & 1))) & 0xFFFFu);
                        const float2 f = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(pr, __NV_E4M3)));
                        o[h] = pack_bf16(f.x * sc, f.y * sc);
                    }
                    const int rr = r0 + r;
                    uint8_t* dst = sKV + (c >> 3) * C::BOX + rr * 128 + (((c & 7) ^ (rr & 7)) << 4);
                    *reinterpret_cast<uint4*>(dst) = make_uint4(o[0], o[1], o[2], o[3]);
                }
            }
        }
    }
    cp_async_wait_all();
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
    if (tid == 0) {
        if (write_gather && hgrp == 0) {                             // the gather buffer's rows
            for (int box = 0; box < C::NBOX; ++box)
                tma_store_3d(&gmap, sKV + box * C::BOX, box * 64, chunk * kFC, row);
            bulk_commit();
        }
        // ---- S^T = KV Q^T
        if (mbar_wait(&bars[0], 0, nullptr)) {
            tc_fence_after();
            const uint32_t idesc = idesc_bf16_f32(kFC, NH);
            const uint32_t a0 = smem_u32(sKV), b0 = smem_u32(sQ);
#pragma unroll
            for (int k = 0; k < D / 16; ++k)
                umma_bf16(tmem, sdesc_kmajor_sw128(a0 + (k >> 2) * C::BOX + (k & 3) * 32),
                          sdesc_kmajor_sw128(b0 + (k >> 2) * NH * 128 + (k & 3) * 32), idesc, k > 0 ? 1u : 0u);
            umma_commit(&bars[1]);
        } else {
            flag_error(p.eword, DSV4_EWORD_TIMEOUT);
            abort_flag = 1;
        }
    }
    bool dead = !mbar_wait(&bars[1], 0, &abort_flag);
    tc_fence_after();
    // ---- scores -> shared (scaled, masked): warps w and w + 4 read TMEM lane quarter w & 3,
    //      half of the head columns each
    {
        const int q = warp & 3, half = warp >> 2;
        const int key = q * 32 + lane;
        uint32_t r[HC];
        tmem_ld_cols<HC>(tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(half * HC), r);
        tmem_wait_ld();
        const bool ok = okf[key] != 0 && !dead;
#pragma unroll
        for (int c = 0; c < HC; ++c)
            sS[key * (NH + 1) + half * HC + c] = ok ? __uint_as_float(r[c]) * p.scale : -INFINITY;
    }
    __syncthreads();
    // ---- per head (lane) over slots [16 warp, 16 warp + 16): max, P = e^(s - m), sums
    float sv[16];
    float mx = -INFINITY;
    if (lane < NH) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            sv[i] = sS[(16 * warp + i) * (NH + 1) + lane];
            mx = fmaxf(mx, sv[i]);
        }
        red_m[warp * NH + lane] = mx;
    }
    __syncthreads();
    float m = -INFINITY;
    if (lane < NH) {
#pragma unroll
        for (int j = 0; j < 8; ++j) m = fmaxf(m, red_m[j * NH + lane]);
        float l = 0.f;
        uint32_t pk[8];
#pragma unroll
        for (int i = 0; i < 16; i += 2) {
            const float p0 = sv[i] == -INFINITY ? 0.f : expf(sv[i] - m);
            const float p1 = sv[i + 1] == -INFINITY ? 0.f : expf(sv[i + 1] - m);
            l += p0 + p1;
            pk[i / 2] = pack_bf16(p0, p1);
        }
        red_l[warp * NH + lane] = l;
        // P[head][slot]: K-major, two 64-slot boxes of [NH rows][128 B], 128-byte swizzle
        uint8_t* prow = sP + (warp >> 2) * (NH * 128) + lane * 128;
        const int c0 = 2 * (warp & 3);
        *reinterpret_cast<uint4*>(prow + ((c0 ^ (lane & 7)) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        *reinterpret_cast<uint4*>(prow + (((c0 + 1) ^ (lane & 7)) << 4)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    tc_fence_before();
    __syncthreads();
    // ---- O^T = V^T P^T (V^T: the KV tile read MN-major)
    if (tid == 0 && !dead) {
        tc_fence_after();
        const uint32_t idesc = idesc_bf16_f32(kFC, NH) | (1u << 15);
        const uint32_t a0 = smem_u32(sKV), b0 = smem_u32(sP);
#pragma unroll
        for (int mt = 0; mt < C::MT; ++mt) {
#pragma unroll
            for (int kk = 0; kk < kFC / 16; ++kk)
                umma_bf16(tmem + static_cast<uint32_t>(NH + mt * NH),
                          sdesc_mnmajor_sw128(a0 + (2 * mt) * C::BOX + kk * 2048, static_cast<uint32_t>(C::BOX), 1024u),
                          sdesc_kmajor_sw128(b0 + (kk >> 2) * NH * 128 + (kk & 3) * 32), idesc, kk > 0 ? 1u : 0u);
        }
        umma_commit(&bars[2]);
    }
    const size_t part = static_cast<size_t>(row) * p.n_splits + chunk;
    if (warp == 0 && lane < Hc) {                                    // this chunk's (m, l) per head
        float l = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) l += red_l[j * NH + lane];
        p.part_ml[(part * p.hstride + hbase + lane) * 2 + 0] = dead ? -INFINITY : m;
        p.part_ml[(part * p.hstride + hbase + lane) * 2 + 1] = dead ? 0.f : l;
    }
    if (!dead && !mbar_wait(&bars[2], 0, &abort_flag)) {
        if (tid == 0) flag_error(p.eword, DSV4_EWORD_TIMEOUT);
        dead = true;
    }
    tc_fence_after();
    // ---- O^T columns -> partials: lane = dim, one column per head
    {
        const int q = warp & 3, half = warp >> 2;
        float* po = p.part_o + (part * p.hstride + hbase) * D;
        for (int task = half; task < 2 * C::MT; task += 2) {
            const int mt = task >> 1, ch = task & 1;
            uint32_t r[HC];
            tmem_ld_cols<HC>(tmem + (static_cast<uint32_t>(q * 32) << 16) +
                                 static_cast<uint32_t>(NH + mt * NH + ch * HC), r);
            tmem_wait_ld();
            const int dim = mt * 128 + q * 32 + lane;
#pragma unroll
            for (int c = 0; c < HC; ++c)
                if (ch * HC + c < Hc) po[static_cast<size_t>(ch * HC + c) * D + dim] = dead ? 0.f : __uint_as_float(r[c]);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, C::TCOLS);
    if (tid == 0) {
        if (write_gather && hgrp == 0) bulk_wait_read();             // the tile is read out
        if (abort_flag) mbar_wait(&bars[0], 0, nullptr, 100000000ull);   // the query copy landed
    }
}

struct DecodePlan { bool use; int n_chunks, nh, n_hg; };

DecodePlan decode_plan(const dsv4_attn_args& a) {
    DecodePlan d{};
    const int slots = a.top_k + a.window;
    d.n_chunks = (slots + kFC - 1) / kFC;
    d.nh = a.heads % 32 == 0 ? 32 : 16;          // every group full, or one group of <= 16
    d.n_hg = (a.heads + d.nh - 1) / d.nh;
    d.use = a.n_q == 1 && (a.dim == 128 || a.dim == 256 || a.dim == 512) && d.n_chunks >= 1 &&
            d.n_chunks <= 256;
    return d;
}

template <int D, int NH>
int run_decode(const dsv4_attn_args& a, const DecodePlan& dp, uint8_t* ws, uint32_t* eword, cudaStream_t st) {
    using C = FCfg<D, NH>;
    const int rows = a.batch * a.n_q;
    const int slots = a.top_k + a.window;
    const size_t hs = static_cast<size_t>(dp.n_hg) * NH;
    const size_t ml_b = align_up(static_cast<size_t>(rows) * dp.n_chunks * hs * 2 * 4, 256);
    CUtensorMap qmap, gmap;
    if (!encode_2d_bf16(&qmap, a.q, D, static_cast<uint64_t>(rows) * a.heads, 64, a.heads < NH ? a.heads : NH))
        return DSV4_ERR_LAUNCH;
    if (a.gather) {
        if (!encode_3d_bf16(&gmap, a.gather, D, static_cast<uint64_t>(slots), static_cast<uint64_t>(rows), 64, kFC))
            return DSV4_ERR_LAUNCH;
    } else {
        gmap = qmap;                                   // not used
    }
    AttnParams p;
    p.sink = a.sink;
    p.n_comp = a.n_comp;
    p.idx = a.idx;
    p.q_pos = a.q_pos;
    p.win_len = a.win_len;
    p.out = static_cast<__nv_bfloat16*>(a.out);
    p.eword = eword;
    p.rows = rows;
    p.n_q = a.n_q;
    p.H = a.heads;
    p.max_comp = a.max_comp;
    p.top_k = a.top_k;
    p.window = a.window;
    p.win_rows = a.win_rows;
    p.ratio = a.ratio;
    p.slots = slots;
    p.comp_chunks = 0;
    p.n_chunks = dp.n_chunks;
    p.chunks_per_split = 1;
    p.n_splits = dp.n_chunks;
    p.oob_row = 0;
    p.n_hg = dp.n_hg;
    p.hstride = static_cast<int>(hs);
    p.scale = a.scale;
    set_output_rope(p, a);
    p.kv_nope = a.kv_fp8 ? static_cast<const uint8_t*>(a.kv_nope) : nullptr;
    p.kv_scale = a.kv_fp8 ? a.kv_scale : nullptr;
    p.kv_rope = a.kv_fp8 ? static_cast<const __nv_bfloat16*>(a.kv_rope) : nullptr;
    p.nope_dim = a.kv_fp8 ? D - a.kv_rope_dim : D;
    p.part_ml = reinterpret_cast<float*>(ws);
    p.part_o = reinterpret_cast<float*>(ws + ml_b);
    static bool attr_set = false;
    if (!attr_set) {
        cudaFuncSetAttribute(attn_decode_kernel<D, NH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(C::SMEM));
        attr_set = true;
    }
    dim3 grid(dp.n_chunks, rows, dp.n_hg);
    count_launch();
    if (launch_k(attn_decode_kernel<D, NH>, grid, dim3(kFT), C::SMEM, st, true, qmap, gmap, p,
                 static_cast<const __nv_bfloat16*>(a.comp_kv), static_cast<const __nv_bfloat16*>(a.win),
                 a.gather ? 1 : 0) != cudaSuccess)
        return DSV4_ERR_LAUNCH;
    dim3 g2(rows, a.heads);
    count_launch();
    if (launch_k(attn_combine_kernel<D, 16>, g2, dim3(128), 0, st, true, p) != cudaSuccess)
        return DSV4_ERR_LAUNCH;
    return DSV4_OK;
}

struct Plan { int slots, comp_chunks, n_chunks, chunks_per_split, n_splits, hp, n_hg; };

Plan make_plan(const dsv4_attn_args& a) {
    Plan pl;
    const int rows = a.batch * a.n_q;
    pl.slots = a.top_k + a.window;
    pl.comp_chunks = (a.top_k + kCH - 1) / kCH;
    pl.n_chunks = pl.comp_chunks + (a.window + kCH - 1) / kCH;
    pl.hp = 16;                                   // heads per CTA
    pl.n_hg = (a.heads + pl.hp - 1) / pl.hp;
    const int sms = sm_count() > 0 ? sm_count() : 148;
    const int units = rows * pl.n_hg;
    int want = units > 0 ? (sms + units - 1) / units : 1;
    if (want < 1) want = 1;
    if (want > pl.n_chunks) want = pl.n_chunks;
    if (want > 256) want = 256;
    pl.chunks_per_split = pl.n_chunks > 0 ? (pl.n_chunks + want - 1) / want : 1;
    pl.n_splits = pl.n_chunks > 0 ? (pl.n_chunks + pl.chunks_per_split - 1) / pl.chunks_per_split : 1;
    return pl;
}

template <int D, int HP>
int run(const dsv4_attn_args& a, const Plan& pl, uint8_t* ws, uint32_t* eword, cudaStream_t st) {
    using C = Cfg<D, HP>;
    const int rows = a.batch * a.n_q;
    // the gather buffer: the caller's, else a workspace region after the partials
    const size_t hs = static_cast<size_t>(pl.n_hg) * HP;
    const size_t ml_b = align_up(static_cast<size_t>(rows) * pl.n_splits * hs * 2 * 4, 256);
    const size_t po_b = pl.n_splits > 1 ? align_up(static_cast<size_t>(rows) * pl.n_splits * hs * D * 4, 256) : 0;
    __nv_bfloat16* gbuf = a.gather ? static_cast<__nv_bfloat16*>(a.gather)
                                   : reinterpret_cast<__nv_bfloat16*>(ws + ml_b + po_b);
    CUtensorMap qmap, gmap;
    if (!encode_2d_bf16(&qmap, a.q, D, static_cast<uint64_t>(rows) * a.heads, 64,
                        a.heads < HP ? a.heads : HP) ||
        !encode_2d_bf16(&gmap, gbuf, D, static_cast<uint64_t>(rows) * pl.slots, 64, kCH))
        return DSV4_ERR_LAUNCH;
    AttnParams p;
    p.sink = a.sink;
    p.n_comp = a.n_comp;
    p.idx = a.idx;
    p.q_pos = a.q_pos;
    p.win_len = a.win_len;
    p.out = static_cast<__nv_bfloat16*>(a.out);
    p.eword = eword;
    p.rows = rows;
    p.n_q = a.n_q;
    p.H = a.heads;
    p.max_comp = a.max_comp;
    p.top_k = a.top_k;
    p.window = a.window;
    p.win_rows = a.win_rows;
    p.ratio = a.ratio;
    p.slots = pl.slots;
    p.comp_chunks = pl.comp_chunks;
    p.n_chunks = pl.n_chunks;
    p.chunks_per_split = pl.chunks_per_split;
    p.n_splits = pl.n_splits;
    p.oob_row = a.batch * a.max_comp;          // first row past the cache: reads as zeros
    p.n_hg = pl.n_hg;
    p.hstride = pl.n_hg * HP;
    p.scale = a.scale;
    set_output_rope(p, a);
    p.part_ml = reinterpret_cast<float*>(ws);
    p.part_o = reinterpret_cast<float*>(ws + ml_b);
    static bool attr_set = false;
    if (!attr_set) {
        cudaFuncSetAttribute(attn_kernel<D, HP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(C::SMEM));
        attr_set = true;
    }
    const long long grows = static_cast<long long>(rows) * pl.slots;
    const long long gblocks = (grows + 8 * kRowsPerWarp - 1) / (8 * kRowsPerWarp);
    count_launch();
    if (launch_k(gather_kernel<D>, dim3(static_cast<unsigned>(gblocks)), dim3(256), 0, st, true, p,
                 static_cast<const __nv_bfloat16*>(a.comp_kv), static_cast<const __nv_bfloat16*>(a.win),
                 gbuf) != cudaSuccess)
        return DSV4_ERR_LAUNCH;
    dim3 grid(pl.n_splits, rows, pl.n_hg);
    count_launch();
    if (launch_k(attn_kernel<D, HP>, grid, dim3(kNT), C::SMEM, st, true, qmap, gmap, p) != cudaSuccess)
        return DSV4_ERR_LAUNCH;
    if (pl.n_splits > 1) {
        dim3 g2(rows, a.heads);
        count_launch();
        if (launch_k(attn_combine_kernel<D, HP>, g2, dim3(128), 0, st, true, p) != cudaSuccess)
            return DSV4_ERR_LAUNCH;
    }
    return DSV4_OK;
}

}  // namespace

size_t attn_ws_bytes(const dsv4_attn_args& a) {
    const DecodePlan dp = decode_plan(a);
    if (dp.use) {
        const size_t rows = static_cast<size_t>(a.batch) * a.n_q;
        const size_t hs = static_cast<size_t>(dp.n_hg) * dp.nh;
        return align_up(rows * dp.n_chunks * hs * 2 * 4, 256) +
               align_up(rows * dp.n_chunks * hs * static_cast<size_t>(a.dim) * 4, 256);
    }
    const Plan pl = make_plan(a);
    const size_t rows = static_cast<size_t>(a.batch) * a.n_q;
    const size_t hs = static_cast<size_t>(pl.n_hg) * pl.hp;
    size_t b = align_up(rows * pl.n_splits * hs * 2 * 4, 256);
    if (pl.n_splits > 1) b += align_up(rows * pl.n_splits * hs * static_cast<size_t>(a.dim) * 4, 256);
    if (!a.gather) b += align_up(rows * pl.slots * static_cast<size_t>(a.dim) * 2, 256);
    return b;
}

int launch_attn(const dsv4_attn_args& a, uint8_t* ws, uint32_t* eword, cudaStream_t st) {
    if (a.batch * a.n_q == 0) return DSV4_OK;
    const DecodePlan dp = decode_plan(a);
    if (dp.use) {
        if (dp.nh == 16) {
            if (a.dim == 512) return run_decode<512, 16>(a, dp, ws, eword, st);
            if (a.dim == 256) return run_decode<256, 16>(a, dp, ws, eword, st);
            return run_decode<128, 16>(a, dp, ws, eword, st);
        }
        if (a.dim == 512) return run_decode<512, 32>(a, dp, ws, eword, st);
        if (a.dim == 256) return run_decode<256, 32>(a, dp, ws, eword, st);
        return run_decode<128, 32>(a, dp, ws, eword, st);
    }
    const Plan pl = make_plan(a);
    if (a.dim == 512) return run<512, 16>(a, pl, ws, eword, st);
    if (a.dim == 256) return run<256, 16>(a, pl, ws, eword, st);
    if (a.dim == 128) return run<128, 16>(a, pl, ws, eword, st);
    return DSV4_ERR_INVALID_ARG;
}

}  // namespace dsv4

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
// Design: tcgen05 kernels for decode and prefill alike. A query row's slots (its top_k
// selected compressed entries, then its window rows) are cut into 128-slot chunks, the heads
// into groups of 32 (or 16). With few query rows (decode) there is one CTA per (chunk, query
// row, head group); each CTA gathers its chunk straight from the caches into shared memory,
// scores it against the group's queries on the tensor cores and writes per-chunk (m, l, O)
// partials; the combine kernel merges the chunks of every (query, head) and adds the sink once:
//   o = sum_c O_c e^(m_c - M) / (sum_c l_c e^(m_c - M) + e^(sink - M)),  M = max(sink, m_c).
// With many query rows (prefill) one CTA per (query row, head group) walks the row's chunks
// with the same steps and a running maximum and sum, and writes the output itself.
#include <cmath>

#include <cuda_fp8.h>

#include "common.cuh"
#include "internal.h"

namespace dsv4 {
namespace {

struct AttnParams {
    const float* sink;             // [H]
    const int32_t* n_comp;         // [B]
    const int32_t* idx;            // [rows, top_k] or null
    const int64_t* q_pos;          // [rows] or null
    const int32_t* win_len;        // [B]
    __nv_bfloat16* out;            // [rows, H, D]
    float* part_ml;                // [rows, n_splits, hstride, 2]: per chunk and head (m, l)
    float* part_o;                 // [rows, n_splits, hstride, D]: per chunk and head O
    uint32_t* eword;
    int rows, n_q, H, max_comp, top_k, window, win_rows, ratio, slots, n_chunks, n_splits;
    int n_hg, hstride;             // head groups per query, heads per partial record (n_hg*NH)
    float scale;
    const int64_t* orp;            // [rows] positions of the output's inverse RoPE, or null
    int or_pairs;                  // rotated pairs: the last 2 * or_pairs channels
    double or_log2_theta;          // log2(theta): pair j turns at theta^(-2j / rope_dim)
    // mixed FP8 / bf16 compressed KV, else null
    const uint8_t* kv_nope;        // [B, max_comp, nope_dim] E4M3 codes
    const float* kv_scale;         // [B, max_comp]
    const __nv_bfloat16* kv_rope;  // [B, max_comp, D - nope_dim]
    int nope_dim;
    int fault;                     // test control: the split form does not load its query tile
    unsigned long long wait_ns;    // limit of each bounded wait
};

// (cos, sin) of the inverse RoPE's angle pos * f_j for pair j (< or_pairs) of query row `row`.
__device__ __forceinline__ float2 inverse_rope_cs(const AttnParams& p, int row, int j) {
    const double freq = exp2(-(static_cast<double>(j) / p.or_pairs) * p.or_log2_theta);
    float sn, cs;
    sincosf(reduced_angle(static_cast<double>(p.orp[row]) * freq), &sn, &cs);
    return make_float2(cs, sn);
}

// Inverse RoPE of one output pair (channels c, c + 1, c even) of query row `row`: rotated back
// by pos * f_j when the pair lies in the last 2 * or_pairs channels of a D-channel head.
__device__ __forceinline__ void inverse_rope_pair(const AttnParams& p, int row, int c, int D,
                                                  float& e, float& o) {
    const int j = (c - (D - 2 * p.or_pairs)) >> 1;
    if (!p.orp || j < 0) return;
    const float2 r = inverse_rope_cs(p, row, j);
    const float e0 = e, o0 = o;
    e = e0 * r.x + o0 * r.y;
    o = -e0 * r.y + o0 * r.x;
}

// The same rotation for the four pairs of an 8-channel piece starting at channel c0, from a
// table of every rotated pair's (cos, sin) for the CTA's one query row (filled once by
// inverse_rope_cs): the walking kernels write a row's heads x D outputs and would otherwise
// form each pair's angle once per head, its fp64 code inlined in the output loop.
__device__ __forceinline__ void inverse_rope_piece(const AttnParams& p, const float2* tab, int c0, int D,
                                                   float (&v)[8]) {
    const int lo = D - 2 * p.or_pairs;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int jj = (c0 + 2 * j - lo) >> 1;
        if (jj >= 0) {
            const float2 r = tab[jj];
            const float e0 = v[2 * j], o0 = v[2 * j + 1];
            v[2 * j] = e0 * r.x + o0 * r.y;
            v[2 * j + 1] = -e0 * r.y + o0 * r.x;
        }
    }
}

// Fills the inverse-RoPE fields of the kernel parameters from the call's arguments.
void set_output_rope(AttnParams& p, const dsv4_attn_args& a) {
    p.orp = a.out_rope_pos;
    p.or_pairs = a.out_rope_pos ? a.out_rope_dim / 2 : 0;
    p.or_log2_theta = a.out_rope_pos ? std::log2(a.out_rope_theta) : 0.0;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}

template <int D>
__global__ void __launch_bounds__(128)
attn_combine_kernel(AttnParams p) {
    constexpr int PER = D / 128;                 // dims per thread
    constexpr int kRegSplits = 24;               // splits whose partial O is loaded up front
    extern __shared__ float wgt[];               // [n_splits] e^(m_s - M)
    __shared__ float red[4];
    __shared__ float bcast[1];
    const int row = blockIdx.x, h = blockIdx.y, tid = threadIdx.x;
    const int ns = p.n_splits;
    pdl_wait();
    const int HS = p.hstride;
    const float* ml = p.part_ml + static_cast<size_t>(row) * ns * HS * 2;
    const float* po = p.part_o + static_cast<size_t>(row) * ns * HS * D + static_cast<size_t>(h) * D + tid * PER;
    // every load at once: this thread's dims of the first kRegSplits splits
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
    // the splits' maxima and sums: two per thread in registers (up to 256 splits), loaded with
    // the partials above; more splits are read again below
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    if (tid < ns) { m0 = ml[(static_cast<size_t>(tid) * HS + h) * 2]; l0 = ml[(static_cast<size_t>(tid) * HS + h) * 2 + 1]; }
    if (tid + 128 < ns) {
        m1 = ml[(static_cast<size_t>(tid + 128) * HS + h) * 2];
        l1 = ml[(static_cast<size_t>(tid + 128) * HS + h) * 2 + 1];
    }
    float M = fmaxf(m0, m1);
    for (int s = tid + 256; s < ns; s += 128) M = fmaxf(M, ml[(static_cast<size_t>(s) * HS + h) * 2]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    if ((tid & 31) == 0) red[tid >> 5] = M;
    __syncthreads();
    M = fmaxf(fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3])), snk);
    const float e0 = m0 == -INFINITY ? 0.f : exp_e(m0 - M);
    const float e1 = m1 == -INFINITY ? 0.f : exp_e(m1 - M);
    if (tid < ns) wgt[tid] = e0;
    if (tid + 128 < ns) wgt[tid + 128] = e1;
    float den = l0 * e0 + l1 * e1;
    for (int s = tid + 256; s < ns; s += 128) {
        const float m = ml[(static_cast<size_t>(s) * HS + h) * 2];
        const float e = m == -INFINITY ? 0.f : exp_e(m - M);
        wgt[s] = e;
        den = fmaf(ml[(static_cast<size_t>(s) * HS + h) * 2 + 1], e, den);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) den += __shfl_xor_sync(0xffffffffu, den, o);
    __syncthreads();
    if ((tid & 31) == 0) red[tid >> 5] = den;
    __syncthreads();
    if (tid == 0) bcast[0] = 1.0f / (red[0] + red[1] + red[2] + red[3] + exp_e(snk - M));
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
        // the thread's PER channels in one store (a warp writes one contiguous piece)
        uint32_t pk[PER / 2];
#pragma unroll
        for (int j = 0; j < PER; j += 2) {
            inverse_rope_pair(p, row, tid * PER + j, D, acc[j], acc[j + 1]);
            pk[j / 2] = pack_bf16(acc[j], acc[j + 1]);
        }
        if constexpr (PER == 4) *reinterpret_cast<uint2*>(dst) = make_uint2(pk[0], pk[1]);
        else *reinterpret_cast<uint32_t*>(dst) = pk[0];
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
    // 64 heads: the scores go through the query tile, which is dead once S^T is computed (a
    // separate score buffer would not fit beside the 128 KB KV tile)
    static constexpr bool kAliasS = NH > 32;
    static constexpr size_t OFF_Q = BOX * NBOX;
    static constexpr size_t OFF_P = OFF_Q + static_cast<size_t>(NBOX) * NH * 128;
    static constexpr size_t OFF_S = kAliasS ? OFF_Q : OFF_P + 2ull * NH * 128;
    static constexpr size_t OFF_R = kAliasS ? OFF_P + 2ull * NH * 128 : OFF_S + static_cast<size_t>(kFC) * (NH + 1) * 4;
    static constexpr size_t OFF_OK = OFF_R + 2ull * 8 * NH * 4;
    static constexpr size_t OFF_BAR = align_up(OFF_OK + kFC * 4, 16);
    static constexpr size_t SMEM = OFF_BAR + 3 * 8 + 1024;           // + alignment slack
    static constexpr uint32_t NEED = static_cast<uint32_t>(NH + MT * NH);
    static constexpr uint32_t TCOLS = NEED <= 32 ? 32 : NEED <= 64 ? 64 : NEED <= 128 ? 128 : NEED <= 256 ? 256 : 512;
    static_assert(D % 128 == 0 && (NH == 16 || NH == 32 || NH == 64), "decode tile shape");
    static_assert(!kAliasS || static_cast<size_t>(kFC) * (NH + 1) * 4 <= static_cast<size_t>(NBOX) * NH * 128,
                  "the scores fit in the query tile");
    static_assert(SMEM <= 227 * 1024, "shared memory per CTA");
};

template <int N>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t (&r)[N]) {
    if constexpr (N == 8) DSV4_TMEM_LD_32x32b_X8(taddr, r);
    else if constexpr (N == 16) DSV4_TMEM_LD_32x32b_X16(taddr, r);
    else DSV4_TMEM_LD_32x32b_X32(taddr, r);
}

// Where one slot's row comes from (lanes 0..15 of warp w hold slots 16w .. 16w + 15 of a chunk).
struct SlotSrc {
    unsigned long long src;        // a bf16 row; 0: none
    long long ent;                 // mixed storage: the entry's row; -1: none
    float escale;                  // mixed storage: the entry's scale
    int ok;                        // the slot holds a row
};

// The index-list entry of this lane's slot of chunk `chunk` (lanes 0..15; -1 elsewhere), loaded
// on its own so that the load can be issued well before its use.
__device__ __forceinline__ int load_slot_index(const AttnParams& p, int chunk, int row, int warp, int lane) {
    const int slot = chunk * kFC + warp * 16 + lane;
    return lane < 16 && p.idx && slot < p.top_k ? p.idx[static_cast<size_t>(row) * p.top_k + slot] : -1;
}

// Resolves the slots of chunk `chunk` of query row `row` from their index-list entries (or the
// dense count): the visible range (an index past it is reported and masked), the window rows.
template <int D>
__device__ __forceinline__ SlotSrc resolve_slots(const AttnParams& p, const __nv_bfloat16* __restrict__ comp_kv,
                                                 const __nv_bfloat16* __restrict__ win, int e_list, int chunk,
                                                 int b, int nv, int w_lo, int w_cnt, int warp, int lane) {
    const int r0 = warp * 16;
    unsigned long long src = 0;
    long long ent = -1;
    float escale = 0.f;
    if (lane < 16) {
        const int slot = chunk * kFC + r0 + lane;
        if (slot < p.top_k) {
            int e;
            if (p.idx) {
                e = e_list;
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
    }
    return SlotSrc{src, ent, escale, src != 0 || ent >= 0};
}

// The gather of one chunk: warp w copies its 16 resolved slots into the shared tile (cp.async
// for bf16 rows, zero fill for slots without a row; the mixed storage's codes are dequantized
// here) and marks in okf[] which slots hold a row. Every lane of the CTA must call it (the
// shuffles take all lanes). The caller waits for the copies (cp_async_wait_all) and fences
// them for the tensor cores.
template <int D, int NH>
__device__ __forceinline__ void copy_slots(const AttnParams& p, const SlotSrc& s, uint8_t* sKV, int* okf,
                                           int warp, int lane) {
    using C = FCfg<D, NH>;
    const int r0 = warp * 16;
    const unsigned long long src = s.src;
    const long long ent = s.ent;
    const float escale = s.escale;
    if (lane < 16) okf[r0 + lane] = s.ok;
    // one shuffle of a row's source per pass, U / 32 pieces per lane (D = 512: 2), or 32 / U
    // rows per pass when a row has fewer than 32 pieces
    constexpr int RPI = C::U >= 32 ? 1 : 32 / C::U;
    constexpr int PPL = C::U >= 32 ? C::U / 32 : 1;
    const int sub = C::U >= 32 ? 0 : lane / C::U;
    const int c0 = C::U >= 32 ? lane : lane - sub * C::U;
    if (!p.kv_nope) {
#pragma unroll 4
        for (int r = 0; r < 16; r += RPI) {
            const unsigned long long a = __shfl_sync(0xffffffffu, src, r + sub);
            const int rr = r0 + r + sub;
#pragma unroll
            for (int j = 0; j < PPL; ++j) {
                const int c = c0 + 32 * j;
                uint8_t* dst = sKV + (c >> 3) * C::BOX + rr * 128 + (((c & 7) ^ (rr & 7)) << 4);
                if (a) cp_async16(dst, reinterpret_cast<const uint8_t*>(a) + c * 16);
                else *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
            }
        }
    } else {
        // mixed storage: a 16-byte bf16 piece c of a compressed row is 8 codes (piece c <
        // ncp) dequantized here, or a piece of its bf16 RoPE part; every load of the warp's
        // 16 rows is issued (codes into registers) before the first is converted
        constexpr int kPer = (16 / RPI) * PPL;                   // pieces per lane
        const int ncp = p.nope_dim / 8;
        const int rope_b = (D - p.nope_dim) * 2;                 // bytes of a RoPE part
        uint2 code[kPer];
#pragma unroll
        for (int r = 0; r < 16; r += RPI) {
            const unsigned long long a = __shfl_sync(0xffffffffu, src, r + sub);
            const long long en = __shfl_sync(0xffffffffu, ent, r + sub);
            const int rr = r0 + r + sub;
#pragma unroll
            for (int j = 0; j < PPL; ++j) {
                const int k = (r / RPI) * PPL + j, c = c0 + 32 * j;
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
        }
#pragma unroll
        for (int r = 0; r < 16; r += RPI) {
            const long long en = __shfl_sync(0xffffffffu, ent, r + sub);
            const float sc = __shfl_sync(0xffffffffu, escale, r + sub);
            const int rr = r0 + r + sub;
#pragma unroll
            for (int j = 0; j < PPL; ++j) {
                const int k = (r / RPI) * PPL + j, c = c0 + 32 * j;
                if (en >= 0 && c < ncp) {                        // (a compressed row)
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
                    uint8_t* dst = sKV + (c >> 3) * C::BOX + rr * 128 + (((c & 7) ^ (rr & 7)) << 4);
                    *reinterpret_cast<uint4*>(dst) = make_uint4(o[0], o[1], o[2], o[3]);
                }
            }
        }
    }
}

template <int D, int NH>
__device__ __forceinline__ void gather_chunk(const AttnParams& p, const __nv_bfloat16* __restrict__ comp_kv,
                                             const __nv_bfloat16* __restrict__ win, uint8_t* sKV, int* okf,
                                             int chunk, int row, int b, int nv, int w_lo, int w_cnt,
                                             int warp, int lane) {
    const int e = load_slot_index(p, chunk, row, warp, lane);
    copy_slots<D, NH>(p, resolve_slots<D>(p, comp_kv, win, e, chunk, b, nv, w_lo, w_cnt, warp, lane), sKV, okf,
                      warp, lane);
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
        if (!p.fault) {              // (test control: the copy is left out, its wait runs out)
            mbar_arrive_expect_tx(&bars[0], static_cast<uint32_t>(Hc) * D * 2);
            for (int box = 0; box < C::NBOX; ++box)
                tma_load_2d(sQ + box * NH * 128, &qmap, &bars[0], box * 64, row * p.H + hbase);
        }
    }

    pdl_wait();                      // the index list comes from the kernel before
    if (hgrp == 0 && chunk == 0 && tid == 0)                         // report a bad count once
        row_visible(nullptr, p.n_comp, p.q_pos, p.n_q, p.ratio, p.max_comp, row, p.eword);
    gather_chunk<D, NH>(p, comp_kv, win, sKV, okf, chunk, row, b, nv, w_lo, w_cnt, warp, lane);
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
        if (mbar_wait(&bars[0], 0, nullptr, p.wait_ns)) {
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
    bool dead = !mbar_wait(&bars[1], 0, &abort_flag, p.wait_ns);
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
    // ---- per head over slots [16 warp, 16 warp + 16): max, P = e^(s - m), sums. Lane l
    //      owns heads l, l + 32, ... (HPL of them)
    constexpr int HPL = NH > 32 ? NH / 32 : 1;
    float sv[HPL][16];
    float m[HPL];
#pragma unroll
    for (int hh = 0; hh < HPL; ++hh) {
        const int hd = lane + 32 * hh;
        float mx = -INFINITY;
        if (hd < NH) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                sv[hh][i] = sS[(16 * warp + i) * (NH + 1) + hd];
                mx = fmaxf(mx, sv[hh][i]);
            }
            red_m[warp * NH + hd] = mx;
        }
    }
    __syncthreads();
#pragma unroll
    for (int hh = 0; hh < HPL; ++hh) {
        const int hd = lane + 32 * hh;
        m[hh] = -INFINITY;
        if (hd < NH) {
#pragma unroll
            for (int j = 0; j < 8; ++j) m[hh] = fmaxf(m[hh], red_m[j * NH + hd]);
            float l = 0.f;
            uint32_t pk[8];
#pragma unroll
            for (int i = 0; i < 16; i += 2) {
                const float p0 = sv[hh][i] == -INFINITY ? 0.f : exp_e(sv[hh][i] - m[hh]);
                const float p1 = sv[hh][i + 1] == -INFINITY ? 0.f : exp_e(sv[hh][i + 1] - m[hh]);
                l += p0 + p1;
                pk[i / 2] = pack_bf16(p0, p1);
            }
            red_l[warp * NH + hd] = l;
            // P[head][slot]: K-major, two 64-slot boxes of [NH rows][128 B], 128-byte swizzle
            // (the swizzle row is the head mod 8, the lane's too)
            uint8_t* prow = sP + (warp >> 2) * (NH * 128) + hd * 128;
            const int c0 = 2 * (warp & 3);
            *reinterpret_cast<uint4*>(prow + ((c0 ^ (lane & 7)) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            *reinterpret_cast<uint4*>(prow + (((c0 + 1) ^ (lane & 7)) << 4)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        }
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
    if (warp == 0) {                                                 // this chunk's (m, l) per head
#pragma unroll
        for (int hh = 0; hh < HPL; ++hh) {
            const int hd = lane + 32 * hh;
            if (hd < Hc) {
                float l = 0.f;
#pragma unroll
                for (int j = 0; j < 8; ++j) l += red_l[j * NH + hd];
                p.part_ml[(part * p.hstride + hbase + hd) * 2 + 0] = dead ? -INFINITY : m[hh];
                p.part_ml[(part * p.hstride + hbase + hd) * 2 + 1] = dead ? 0.f : l;
            }
        }
    }
    if (!dead && !mbar_wait(&bars[2], 0, &abort_flag, p.wait_ns)) {
        if (tid == 0) flag_error(p.eword, DSV4_EWORD_TIMEOUT);
        dead = true;
    }
    tc_fence_after();
    // ---- O^T columns -> partials: lane = dim, one column per head. 64-head CTAs stage them as
    //      fp32 [NH heads][D] in the KV tile (free once the O^T MMA and the gather buffer's copy
    //      have read it) so that they leave in 16-byte pieces of whole head rows: written one
    //      4-byte column at a time, their 128 KB took ~4.6 us (the 8K-context step: 43.9 -> 42.8
    //      us); a 32-head CTA's 64 KB gained nothing from it (the 1M-context step: +0.5 us).
    const int q = warp & 3, half = warp >> 2;
    if constexpr (NH > 32) {
        static_assert(NH * D * 4 <= C::BOX * C::NBOX, "the fp32 partial fits in the KV tile");
        if (tid == 0 && write_gather && hgrp == 0) bulk_wait_read();
        __syncthreads();
        float* sO = reinterpret_cast<float*>(sKV);
        for (int task = half; task < 2 * C::MT; task += 2) {
            const int mt = task >> 1, ch = task & 1;
            uint32_t r[HC];
            tmem_ld_cols<HC>(tmem + (static_cast<uint32_t>(q * 32) << 16) +
                                 static_cast<uint32_t>(NH + mt * NH + ch * HC), r);
            tmem_wait_ld();
            const int dim = mt * 128 + q * 32 + lane;
#pragma unroll
            for (int c = 0; c < HC; ++c) sO[(ch * HC + c) * D + dim] = dead ? 0.f : __uint_as_float(r[c]);
        }
        __syncthreads();
        float4* po4 = reinterpret_cast<float4*>(p.part_o + (part * p.hstride + hbase) * D);
        const float4* s4 = reinterpret_cast<const float4*>(sKV);
        for (int i = tid; i < Hc * (D / 4); i += kFT) po4[i] = s4[i];
    } else {
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
        if (abort_flag && !p.fault) mbar_wait(&bars[0], 0, nullptr, 100000000ull);   // the query copy landed
    }
}

// ------------------------------------------------------------------ many query rows: one CTA walks a row
// When the (query row, head group) pairs alone fill the GPU twice over, splitting rows into
// chunks only adds partials: one CTA per (query row, head group), the groups of a row side by
// side, then walks the row's chunks in order with the same gather, S^T and O^T steps, keeps
// each head's running maximum and sum (online softmax: the running O is scaled by
// e^(m_old - m_new) before the chunk's O is added), holds the running O^T in registers (each
// thread its dims for half of the group's heads), and at the end adds the sink once and
// writes the normalised output (through shared memory, in whole rows). The next chunk's
// gather starts as soon as the O^T MMA has read the tile (its index entries were loaded a
// chunk earlier), and a chunk's O^T is read out of TMEM while the next chunk's S^T MMA runs.
template <int D, int NH>
__global__ void __launch_bounds__(kFT, 1)
attn_rows_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap gmap,
                 AttnParams p, const __nv_bfloat16* __restrict__ comp_kv,
                 const __nv_bfloat16* __restrict__ win, int write_gather) {
    using C = FCfg<D, NH>;
    constexpr int HC = NH / 2;                                       // TMEM columns per warp
    static_assert(NH * D * 4 <= C::BOX * C::NBOX, "the fp32 output fits in the tile");
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint32_t tmem_slot;
    __shared__ volatile int abort_flag;
    __shared__ float s_fac[NH];      // per head: e^(m_old - m_new) of a chunk; at the end 1 / den
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
    const int hgrp = static_cast<int>(blockIdx.x % p.n_hg), row = static_cast<int>(blockIdx.x / p.n_hg);
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

    for (int i = tid; i < C::NBOX * (NH - Hc) * 8; i += kFT) {       // query rows past the heads
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
    if (tid == 0) {
        tma_prefetch_desc(&gmap);
        mbar_arrive_expect_tx(&bars[0], static_cast<uint32_t>(Hc) * D * 2);
        for (int box = 0; box < C::NBOX; ++box)
            tma_load_2d(sQ + box * NH * 128, &qmap, &bars[0], box * 64, row * p.H + hbase);
    }

    pdl_wait();                      // the index lists come from the kernel before
    if (hgrp == 0 && tid == 0) row_visible(nullptr, p.n_comp, p.q_pos, p.n_q, p.ratio, p.max_comp, row, p.eword);

    const int q4 = warp & 3, half = warp >> 2;   // TMEM lane quarter, half of the head columns
    float acc[C::MT][HC];                         // running O^T: dims mt*128 + 32*q4 + lane
#pragma unroll
    for (int mt = 0; mt < C::MT; ++mt)
#pragma unroll
        for (int c = 0; c < HC; ++c) acc[mt][c] = 0.f;
    float m_run = -INFINITY, l_run = 0.f;         // lanes < NH: head `lane` (every warp alike)
    bool dead = false;
    gather_chunk<D, NH>(p, comp_kv, win, sKV, okf, 0, row, b, nv, w_lo, w_cnt, warp, lane);
    int next_e = -1;                                 // the next chunk's index entry, loaded a chunk ahead
    // running O^T = running O^T * e^(m_old - m_new) + the last chunk's O^T (TMEM columns NH..)
    auto add_chunk_o = [&]() {
        tc_fence_after();
        uint32_t r[C::MT][HC];
#pragma unroll
        for (int mt = 0; mt < C::MT; ++mt)
            tmem_ld_cols<HC>(tmem + (static_cast<uint32_t>(q4 * 32) << 16) +
                                 static_cast<uint32_t>(NH + mt * NH + half * HC), r[mt]);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < HC; ++c) {
            const float f = s_fac[half * HC + c];
#pragma unroll
            for (int mt = 0; mt < C::MT; ++mt)
                acc[mt][c] = fmaf(acc[mt][c], f, dead ? 0.f : __uint_as_float(r[mt][c]));
        }
    };
    for (int chunk = 0; chunk < p.n_chunks; ++chunk) {
        const uint32_t ph = static_cast<uint32_t>(chunk & 1);
        cp_async_wait_all();
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        tc_fence_before();
        __syncthreads();
        if (chunk + 1 < p.n_chunks) next_e = load_slot_index(p, chunk + 1, row, warp, lane);
        if (tid == 0) {
            if (write_gather && hgrp == 0) {
                for (int box = 0; box < C::NBOX; ++box)
                    tma_store_3d(&gmap, sKV + box * C::BOX, box * 64, chunk * kFC, row);
                bulk_commit();
            }
            if (!dead && chunk == 0 && !mbar_wait(&bars[0], 0, nullptr, p.wait_ns)) dead = true;
            if (!dead) {                            // S^T = KV Q^T
                tc_fence_after();
                const uint32_t idesc = idesc_bf16_f32(kFC, NH);
                const uint32_t a0 = smem_u32(sKV), b0 = smem_u32(sQ);
#pragma unroll
                for (int k = 0; k < D / 16; ++k)
                    umma_bf16(tmem, sdesc_kmajor_sw128(a0 + (k >> 2) * C::BOX + (k & 3) * 32),
                              sdesc_kmajor_sw128(b0 + (k >> 2) * NH * 128 + (k & 3) * 32), idesc, k > 0 ? 1u : 0u);
                umma_commit(&bars[1]);
            } else if (!abort_flag) {
                flag_error(p.eword, DSV4_EWORD_TIMEOUT);
                abort_flag = 1;
            }
        }
        if (chunk > 0) add_chunk_o();                // the previous chunk's O^T, while S^T runs
        if (!dead && !mbar_wait(&bars[1], ph, &abort_flag, p.wait_ns)) {
            dead = true;
            if (tid == 0) { flag_error(p.eword, DSV4_EWORD_TIMEOUT); abort_flag = 1; }
        }
        tc_fence_after();
        {                                            // scores -> shared (scaled, masked)
            const int key = q4 * 32 + lane;
            uint32_t r[HC];
            tmem_ld_cols<HC>(tmem + (static_cast<uint32_t>(q4 * 32) << 16) + static_cast<uint32_t>(half * HC), r);
            tmem_wait_ld();
            const bool ok = okf[key] != 0 && !dead;
#pragma unroll
            for (int c = 0; c < HC; ++c)
                sS[key * (NH + 1) + half * HC + c] = ok ? __uint_as_float(r[c]) * p.scale : -INFINITY;
        }
        __syncthreads();
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
        float fac = 0.f;
        if (lane < NH) {
            float m_new = m_run;
#pragma unroll
            for (int j = 0; j < 8; ++j) m_new = fmaxf(m_new, red_m[j * NH + lane]);
            float l = 0.f;
            uint32_t pk[8];
#pragma unroll
            for (int i = 0; i < 16; i += 2) {
                const float p0 = sv[i] == -INFINITY ? 0.f : exp_e(sv[i] - m_new);
                const float p1 = sv[i + 1] == -INFINITY ? 0.f : exp_e(sv[i + 1] - m_new);
                l += p0 + p1;
                pk[i / 2] = pack_bf16(p0, p1);
            }
            red_l[warp * NH + lane] = l;
            uint8_t* prow = sP + (warp >> 2) * (NH * 128) + lane * 128;
            const int c0 = 2 * (warp & 3);
            *reinterpret_cast<uint4*>(prow + ((c0 ^ (lane & 7)) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            *reinterpret_cast<uint4*>(prow + (((c0 + 1) ^ (lane & 7)) << 4)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
            fac = m_run == -INFINITY ? 0.f : exp_e(m_run - m_new);
            if (warp == 0) s_fac[lane] = fac;
            m_run = m_new;
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        tc_fence_before();
        __syncthreads();
        if (tid == 0 && !dead) {                     // O^T = V^T P^T into fresh accumulators
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
        if (warp == 0 && lane < NH) {
            float l = 0.f;
#pragma unroll
            for (int j = 0; j < 8; ++j) l += red_l[j * NH + lane];
            l_run = l_run * fac + l;
        }
        if (!dead && !mbar_wait(&bars[2], ph, &abort_flag, p.wait_ns)) {
            dead = true;
            if (tid == 0) { flag_error(p.eword, DSV4_EWORD_TIMEOUT); abort_flag = 1; }
        }
        tc_fence_after();
        // the tile is read: the next chunk's rows go in (its S^T then runs beside this O^T's read-out)
        if (chunk + 1 < p.n_chunks) {
            if (write_gather && hgrp == 0) {
                if (tid == 0) bulk_wait_read();      // the gather buffer's copy of the tile
                __syncthreads();
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            copy_slots<D, NH>(p, resolve_slots<D>(p, comp_kv, win, next_e, chunk + 1, b, nv, w_lo, w_cnt, warp, lane),
                              sKV, okf, warp, lane);
        }
    }
    if (p.n_chunks > 0) add_chunk_o();
    tc_fence_before();
    __syncthreads();
    if (warp == 0 && lane < NH) {                    // the sink once, and 1 / denominator
        const float snk = lane < Hc ? p.sink[hbase + lane] : 0.f;
        const float M = fmaxf(m_run, snk);
        const float e = m_run == -INFINITY ? 0.f : exp_e(m_run - M);
        s_fac[lane] = e / fmaf(l_run, e, exp_e(snk - M));
    }
    // the inverse RoPE's (cos, sin) per rotated pair of this row, in the (free) score array
    float2* rtab = reinterpret_cast<float2*>(sS);
    static_assert(static_cast<size_t>(kFC) * (NH + 1) * 4 >= static_cast<size_t>(D / 2) * sizeof(float2),
                  "the RoPE table fits");
    if (p.orp)
        for (int j = tid; j < p.or_pairs; j += kFT) rtab[j] = inverse_rope_cs(p, row, j);
    if (tid == 0 && write_gather && hgrp == 0) bulk_wait_read();   // the tile's last copy out
    __syncthreads();
    // the normalised output goes through the (free) tile as fp32 [NH heads][D], then out in
    // 16-byte pieces of whole head rows, each piece's RoPE pairs rotated back in the thread
    float* sO = reinterpret_cast<float*>(sKV);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
#pragma unroll
    for (int c = 0; c < HC; ++c) {
        const int h = half * HC + c;
        const float f = s_fac[h];
#pragma unroll
        for (int mt = 0; mt < C::MT; ++mt)
            sO[h * D + mt * 128 + q4 * 32 + lane] = dead ? 0.f : acc[mt][c] * f;
    }
    __syncthreads();
    {
        __nv_bfloat16* po = p.out + (static_cast<size_t>(row) * p.H + hbase) * D;
        for (int i = tid; i < Hc * (D / 8); i += kFT) {
            const int h = i / (D / 8), k = i - h * (D / 8);
            const float4 u0 = *reinterpret_cast<const float4*>(sO + h * D + k * 8);
            const float4 u1 = *reinterpret_cast<const float4*>(sO + h * D + k * 8 + 4);
            float v[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
            if (p.orp) inverse_rope_piece(p, rtab, k * 8, D, v);
            *reinterpret_cast<uint4*>(po + static_cast<size_t>(h) * D + k * 8) =
                make_uint4(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]), pack_bf16(v[4], v[5]), pack_bf16(v[6], v[7]));
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, C::TCOLS);
    if (tid == 0) {
        if (write_gather && hgrp == 0) bulk_wait_read();
        if (abort_flag) mbar_wait(&bars[0], 0, nullptr, 100000000ull);   // the query copy landed
    }
}

// Walking form with 64 heads per CTA (D = 512). A tcgen05.mma takes about the same time to
// issue at N = 32 as at N = 64, and a chunk's gather serves every head of the CTA, so one CTA
// per (query row, 64 heads) does a chunk's work for twice the heads at little more cost than
// a 32-head CTA. The running O^T of 64 heads (4 tiles x 64 columns) does not fit in the
// registers, so it stays in TMEM and every chunk's O^T MMA accumulates into it; the online
// softmax keeps, per head, a reference maximum m that changes only when a chunk's maximum
// exceeds it by more than kRescaleTau (then the head's columns of O^T and its sum l are
// scaled by e^(m_old - m_new) through TMEM loads and stores). Every P = e^(s - m) is then at
// most e^kRescaleTau, and the result is the same softmax: the final O / l does not depend on
// which reference maximum was used. Scores, maxima and the sink are carried in base-2 units
// (times log2 e), so each P is one exp2f (with expf the softmax took 1.7 of a chunk's 5.6 us,
// with exp2f 1.0). The 128 x 64 scores are reduced in registers (a butterfly
// over the warp's 32 slots per head, then the four lane quarters through shared memory)
// rather than staged in shared memory, which with the 64 KB query tile would not fit.
constexpr float kRescaleTau = 8.f;
constexpr float kLog2e = 1.4426950408889634f;          // log2(e)
constexpr float kFastSpan = 64.f;                       // base-2 units: P below 2^64 needs no new reference

struct Rows64Cfg {
    static constexpr int D = 512, NH = 64;
    static constexpr int NBOX = D / 64, MT = D / 128;
    static constexpr size_t BOX = static_cast<size_t>(kFC) * 128;    // one 64-dim box of the KV tile
    static constexpr size_t OFF_Q = BOX * NBOX;                      // 128 KB KV tile
    static constexpr size_t OFF_P = OFF_Q + static_cast<size_t>(NBOX) * NH * 128;   // + 64 KB queries
    static constexpr size_t OFF_RM = OFF_P + static_cast<size_t>(kFC) * NH * 2;     // + 16 KB P (MN-major)
    static constexpr size_t OFF_RL = OFF_RM + 4 * NH * 4;           // per lane quarter: chunk maxima
    static constexpr size_t OFF_M = OFF_RL + 4 * NH * 4;            // per lane quarter: chunk sums
    static constexpr size_t OFF_L = OFF_M + NH * 4;                 // reference maximum per head
    static constexpr size_t OFF_F = OFF_L + NH * 4;                 // running sum per head
    static constexpr size_t OFF_OK = OFF_F + NH * 4;                // this chunk's factor per head
    static constexpr size_t OFF_BAR = align_up(OFF_OK + kFC * 4, 16);
    static constexpr size_t SMEM = OFF_BAR + 3 * 8 + 1024;          // + alignment slack
    static constexpr uint32_t TCOLS = 512;                          // S^T 64 + O^T 4 x 64 columns
    static_assert(NH * D * 4 <= BOX * NBOX, "the fp32 output fits in the KV tile");
    static_assert(SMEM <= 227 * 1024, "shared memory per CTA");
};

// Reduces 32 values per lane over the warp's 32 lanes so that lane l ends with the reduction
// of element l: at each width w, a lane keeps the half of its elements its bit w selects and
// receives the other half's partner values from lane ^ w (31 shuffles for 32 elements).
template <bool kMax>
__device__ __forceinline__ float warp_transpose_reduce(float (&v)[32], int lane) {
#pragma unroll
    for (int w = 16; w >= 1; w >>= 1) {
        const bool upper = (lane & w) != 0;
#pragma unroll
        for (int i = 0; i < w; ++i) {
            const float keep = upper ? v[i + w] : v[i];
            const float send = upper ? v[i] : v[i + w];
            const float got = __shfl_xor_sync(0xffffffffu, send, w);
            v[i] = kMax ? fmaxf(keep, got) : keep + got;
        }
    }
    return v[0];
}

__global__ void __launch_bounds__(kFT, 1)
attn_rows64_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap gmap,
                   AttnParams p, const __nv_bfloat16* __restrict__ comp_kv,
                   const __nv_bfloat16* __restrict__ win, int write_gather) {
    using C = Rows64Cfg;
    constexpr int D = C::D, NH = C::NH;
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint32_t tmem_slot;
    __shared__ volatile int abort_flag;
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* sm = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    uint8_t* sKV = sm;
    uint8_t* sQ = sm + C::OFF_Q;
    uint8_t* sP = sm + C::OFF_P;
    float* red_m = reinterpret_cast<float*>(sm + C::OFF_RM);        // [quarter][head]
    float* red_l = reinterpret_cast<float*>(sm + C::OFF_RL);
    float* s_m = reinterpret_cast<float*>(sm + C::OFF_M);
    float* s_l = reinterpret_cast<float*>(sm + C::OFF_L);
    float* s_f = reinterpret_cast<float*>(sm + C::OFF_F);
    int* okf = reinterpret_cast<int*>(sm + C::OFF_OK);
    uint64_t* bars = reinterpret_cast<uint64_t*>(sm + C::OFF_BAR);   // q loaded, S done, O done

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int hgrp = static_cast<int>(blockIdx.x % p.n_hg), row = static_cast<int>(blockIdx.x / p.n_hg);
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

    for (int i = tid; i < C::NBOX * (NH - Hc) * 8; i += kFT) {       // query rows past the heads
        const int box = i / ((NH - Hc) * 8), rem = i - box * (NH - Hc) * 8;
        *reinterpret_cast<uint4*>(sQ + box * NH * 128 + (Hc + rem / 8) * 128 + (rem & 7) * 16) =
            make_uint4(0, 0, 0, 0);
    }
    if (tid < NH) {
        s_m[tid] = -INFINITY;
        s_l[tid] = 0.f;
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
    if (tid == 0) {
        tma_prefetch_desc(&gmap);
        mbar_arrive_expect_tx(&bars[0], static_cast<uint32_t>(Hc) * D * 2);
        for (int box = 0; box < C::NBOX; ++box)
            tma_load_2d(sQ + box * NH * 128, &qmap, &bars[0], box * 64, row * p.H + hbase);
    }

    pdl_wait();                      // the index lists come from the kernel before
    if (hgrp == 0 && tid == 0) row_visible(nullptr, p.n_comp, p.q_pos, p.n_q, p.ratio, p.max_comp, row, p.eword);

    const int q4 = warp & 3, half = warp >> 2;   // TMEM lane quarter (slots / dims), head half
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(q4 * 32) << 16);
    bool dead = false;
    // this thread's slot's P summed over the chunks, per head of its half (relative to the
    // heads' current references; scaled with them), reduced over the slots once at the end
    float lacc[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) lacc[i] = 0.f;
    gather_chunk<D, NH>(p, comp_kv, win, sKV, okf, 0, row, b, nv, w_lo, w_cnt, warp, lane);
    int next_e = -1;                                 // the next chunk's index entry, loaded a chunk ahead
    for (int chunk = 0; chunk < p.n_chunks; ++chunk) {
        const uint32_t ph = static_cast<uint32_t>(chunk & 1);
        cp_async_wait_all();
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        tc_fence_before();
        __syncthreads();
        if (chunk + 1 < p.n_chunks) next_e = load_slot_index(p, chunk + 1, row, warp, lane);
        if (tid == 0) {
            if (write_gather && hgrp == 0) {
                for (int box = 0; box < C::NBOX; ++box)
                    tma_store_3d(&gmap, sKV + box * C::BOX, box * 64, chunk * kFC, row);
                bulk_commit();
            }
            if (!dead && chunk == 0 && !mbar_wait(&bars[0], 0, nullptr, p.wait_ns)) dead = true;
            if (!dead) {                            // S^T = KV Q^T into columns 0 .. NH - 1
                tc_fence_after();
                const uint32_t idesc = idesc_bf16_f32(kFC, NH);
                const uint32_t a0 = smem_u32(sKV), b0 = smem_u32(sQ);
#pragma unroll
                for (int k = 0; k < D / 16; ++k)
                    umma_bf16(tmem, sdesc_kmajor_sw128(a0 + (k >> 2) * C::BOX + (k & 3) * 32),
                              sdesc_kmajor_sw128(b0 + (k >> 2) * NH * 128 + (k & 3) * 32), idesc, k > 0 ? 1u : 0u);
                umma_commit(&bars[1]);
            } else if (!abort_flag) {
                flag_error(p.eword, DSV4_EWORD_TIMEOUT);
                abort_flag = 1;
            }
        }
        if (!dead && !mbar_wait(&bars[1], ph, &abort_flag, p.wait_ns)) {
            dead = true;
            if (tid == 0) { flag_error(p.eword, DSV4_EWORD_TIMEOUT); abort_flag = 1; }
        }
        tc_fence_after();
        // ---- the chunk's softmax: thread = slot q4 * 32 + lane, heads 32 * half .. + 31
        float v[32];
        {
            uint32_t r[32];
            DSV4_TMEM_LD_32x32b_X32(lane_base + static_cast<uint32_t>(32 * half), r);
            tmem_wait_ld();
            const bool ok = okf[q4 * 32 + lane] != 0 && !dead;
            const float sc2 = p.scale * kLog2e;      // scores in base-2 units: P = 2^(s' - m')
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = ok ? __uint_as_float(r[i]) * sc2 : -INFINITY;
        }
        // The heads' reference maxima move only when some score of the chunk exceeds its head's
        // by more than kFastSpan (base-2 units): below that, P = 2^(s' - m') stays far inside
        // the fp32 and bf16 range and the softmax is the same, so each thread checks its own
        // scores and one block-wide vote decides (the first chunk, whose references are -inf,
        // always reduces). Otherwise the chunk's per-head maxima are reduced (a butterfly over
        // the warp's 32 slots, the lane quarters through shared memory) and a head whose maximum
        // exceeds its reference by more than kRescaleTau takes it as the new reference.
        float mh[32];
#pragma unroll
        for (int i = 0; i < 32; i += 4) {
            const float4 m4 = *reinterpret_cast<const float4*>(s_m + 32 * half + i);
            mh[i] = m4.x; mh[i + 1] = m4.y; mh[i + 2] = m4.z; mh[i + 3] = m4.w;
        }
        bool over = false;
#pragma unroll
        for (int i = 0; i < 32; ++i) over |= v[i] > mh[i] + kFastSpan;
        bool any_rescale = false;
        if (__syncthreads_or(over)) {
            {
                float sv[32];                        // (the reduction consumes its input)
#pragma unroll
                for (int i = 0; i < 32; ++i) sv[i] = v[i];
                red_m[q4 * NH + 32 * half + lane] = warp_transpose_reduce<true>(sv, lane);
            }
            __syncthreads();
            // (threads 0 .. NH - 1; a first finite maximum is always taken: -inf + tau is -inf)
            bool rescale = false;
            if (tid < NH) {
                const float cm = fmaxf(fmaxf(red_m[tid], red_m[NH + tid]), fmaxf(red_m[2 * NH + tid], red_m[3 * NH + tid]));
                const float mo = s_m[tid];
                float f = 1.f;
                if (cm > mo + kRescaleTau * kLog2e) {
                    f = mo == -INFINITY ? 0.f : exp2f(mo - cm);
                    s_m[tid] = cm;
                    rescale = chunk > 0;
                }
                s_f[tid] = f;
            }
            any_rescale = __syncthreads_or(rescale) != 0;
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
                const float4 m4 = *reinterpret_cast<const float4*>(s_m + 32 * half + i);
                mh[i] = m4.x; mh[i + 1] = m4.y; mh[i + 2] = m4.z; mh[i + 3] = m4.w;
                const float4 f4 = *reinterpret_cast<const float4*>(s_f + 32 * half + i);
                lacc[i] *= f4.x; lacc[i + 1] *= f4.y; lacc[i + 2] *= f4.z; lacc[i + 3] *= f4.w;
            }
        }
        {
            // P = e^(s - m) in bf16 as the MN-major B operand of O^T: slot s's 64 heads are one
            // 128-byte row (128-byte swizzle, 8-row atoms of 1024 B); then each head's sum
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = v[i] == -INFINITY ? 0.f : exp2f(v[i] - mh[i]);
            const int s = q4 * 32 + lane;
            uint8_t* prow = sP + (s >> 3) * 1024 + (s & 7) * 128;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int c = 4 * half + j;          // 16-byte piece: heads 8c .. 8c + 7
                *reinterpret_cast<uint4*>(prow + ((c ^ (s & 7)) << 4)) =
                    make_uint4(pack_bf16(v[8 * j], v[8 * j + 1]), pack_bf16(v[8 * j + 2], v[8 * j + 3]),
                               pack_bf16(v[8 * j + 4], v[8 * j + 5]), pack_bf16(v[8 * j + 6], v[8 * j + 7]));
            }
#pragma unroll
            for (int i = 0; i < 32; ++i) lacc[i] += v[i];
        }
        if (any_rescale && !dead) {
            // the running O^T of the heads whose maximum moved, times e^(m_old - m_new) (the
            // previous chunk's O^T MMA is complete: its barrier was waited for)
            float fh[32];
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
                const float4 f4 = *reinterpret_cast<const float4*>(s_f + 32 * half + i);
                fh[i] = f4.x; fh[i + 1] = f4.y; fh[i + 2] = f4.z; fh[i + 3] = f4.w;
            }
#pragma unroll
            for (int mt = 0; mt < C::MT; ++mt) {
                uint32_t r[32];
                const uint32_t ta = lane_base + static_cast<uint32_t>(NH + mt * NH + 32 * half);
                DSV4_TMEM_LD_32x32b_X32(ta, r);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * fh[i]);
                DSV4_TMEM_ST_32x32b_X32(ta, r);
            }
            DSV4_TMEM_WAIT_ST();
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        tc_fence_before();
        __syncthreads();
        if (tid == 0 && !dead) {                     // O^T += V^T P^T (the first chunk starts it)
            tc_fence_after();
            const uint32_t idesc = idesc_bf16_f32(kFC, NH) | (1u << 15) | (1u << 16);
            const uint32_t a0 = smem_u32(sKV), b0 = smem_u32(sP);
#pragma unroll
            for (int mt = 0; mt < C::MT; ++mt) {
#pragma unroll
                for (int kk = 0; kk < kFC / 16; ++kk)
                    umma_bf16(tmem + static_cast<uint32_t>(NH + mt * NH),
                              sdesc_mnmajor_sw128(a0 + (2 * mt) * C::BOX + kk * 2048, static_cast<uint32_t>(C::BOX), 1024u),
                              sdesc_mnmajor_sw128(b0 + kk * 2048, 8192u, 1024u), idesc,
                              (chunk > 0 || kk > 0) ? 1u : 0u);
            }
            umma_commit(&bars[2]);
        }
        if (!dead && !mbar_wait(&bars[2], ph, &abort_flag, p.wait_ns)) {
            dead = true;
            if (tid == 0) { flag_error(p.eword, DSV4_EWORD_TIMEOUT); abort_flag = 1; }
        }
        tc_fence_after();
        // the tile is read: the next chunk's rows go in
        if (chunk + 1 < p.n_chunks) {
            if (write_gather && hgrp == 0) {
                if (tid == 0) bulk_wait_read();      // the gather buffer's copy of the tile
                __syncthreads();
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            copy_slots<D, NH>(p, resolve_slots<D>(p, comp_kv, win, next_e, chunk + 1, b, nv, w_lo, w_cnt, warp, lane),
                              sKV, okf, warp, lane);
        }
    }
    // each head's sum over all slots: the butterfly over the warp's 32 slots, then the quarters
    red_l[q4 * NH + 32 * half + lane] = warp_transpose_reduce<false>(lacc, lane);
    tc_fence_before();
    __syncthreads();
    if (tid < NH) s_l[tid] = (red_l[tid] + red_l[NH + tid]) + (red_l[2 * NH + tid] + red_l[3 * NH + tid]);
    __syncthreads();
    if (tid < NH) {                                  // the sink once, and 1 / denominator
        const float snk = (tid < Hc ? p.sink[hbase + tid] : 0.f) * kLog2e;    // (base-2 units)
        const float mr = s_m[tid];
        const float M = fmaxf(mr, snk);
        const float e = mr == -INFINITY ? 0.f : exp2f(mr - M);
        s_f[tid] = e / fmaf(s_l[tid], e, exp2f(snk - M));
    }
    // the inverse RoPE's (cos, sin) per rotated pair of this row, in the (free) reduction
    // arrays: 2 KB, room for every pair of a 512-channel head
    float2* rtab = reinterpret_cast<float2*>(red_m);
    static_assert(C::OFF_M - C::OFF_RM >= static_cast<size_t>(D / 2) * sizeof(float2), "the RoPE table fits");
    if (p.orp)
        for (int j = tid; j < p.or_pairs; j += kFT) rtab[j] = inverse_rope_cs(p, row, j);
    if (tid == 0 && write_gather && hgrp == 0) bulk_wait_read();   // the tile's last copy out
    __syncthreads();
    tc_fence_after();
    // the normalised O^T -> fp32 [NH heads][D] in the (free) KV tile, then out in 16-byte
    // pieces of whole head rows, each piece's RoPE pairs rotated back in the thread
    float* sO = reinterpret_cast<float*>(sKV);
    const bool have_o = p.n_chunks > 0 && !dead;
    float fo[32];                                    // this thread's heads' output factors
#pragma unroll
    for (int i = 0; i < 32; i += 4) {
        const float4 f4 = *reinterpret_cast<const float4*>(s_f + 32 * half + i);
        fo[i] = have_o ? f4.x : 0.f; fo[i + 1] = have_o ? f4.y : 0.f;
        fo[i + 2] = have_o ? f4.z : 0.f; fo[i + 3] = have_o ? f4.w : 0.f;
    }
#pragma unroll
    for (int mt = 0; mt < C::MT; ++mt) {
        uint32_t r[32] = {};
        if (have_o) {
            DSV4_TMEM_LD_32x32b_X32(lane_base + static_cast<uint32_t>(NH + mt * NH + 32 * half), r);
            tmem_wait_ld();
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) sO[(32 * half + i) * D + mt * 128 + q4 * 32 + lane] = __uint_as_float(r[i]) * fo[i];
    }
    __syncthreads();
    {
        __nv_bfloat16* po = p.out + (static_cast<size_t>(row) * p.H + hbase) * D;
        for (int i = tid; i < Hc * (D / 8); i += kFT) {
            const int h = i / (D / 8), k = i - h * (D / 8);
            const float4 u0 = *reinterpret_cast<const float4*>(sO + h * D + k * 8);
            const float4 u1 = *reinterpret_cast<const float4*>(sO + h * D + k * 8 + 4);
            float o[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
            if (p.orp) inverse_rope_piece(p, rtab, k * 8, D, o);
            *reinterpret_cast<uint4*>(po + static_cast<size_t>(h) * D + k * 8) =
                make_uint4(pack_bf16(o[0], o[1]), pack_bf16(o[2], o[3]), pack_bf16(o[4], o[5]), pack_bf16(o[6], o[7]));
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, C::TCOLS);
    if (tid == 0) {
        if (write_gather && hgrp == 0) bulk_wait_read();
        if (abort_flag) mbar_wait(&bars[0], 0, nullptr, 100000000ull);   // the query copy landed
    }
}

// (query row, head group) pairs from which one CTA walks each row. A fixed crossover measured
// on a 152-SM GB300 (the walking form took over once it had about two CTAs per SM), not a
// value derived from the device's SM count: it also fixes the workspace rule stated in the
// header (partials below it, none at or above it), which must not change from one device to
// another.
constexpr long long kRowWalkCtas = 304;

// walk: one CTA walks each (query row, head group); sized_walk: the workspace is sized for that
// (no partials), which depends on the arguments alone (the 304-pair rule in the header).
struct DecodePlan { int n_chunks, nh, n_hg; bool walk, sized_walk; };

DecodePlan decode_plan(const dsv4_attn_args& a) {
    DecodePlan d{};
    const long long slots = static_cast<long long>(a.top_k) + a.window;
    d.n_chunks = static_cast<int>((slots + kFC - 1) / kFC);
    d.nh = a.heads % 32 == 0 ? 32 : 16;          // every group full, or one group of <= 16
    d.n_hg = (a.heads + d.nh - 1) / d.nh;
    const long long pairs = static_cast<long long>(a.batch) * a.n_q * d.n_hg;
    d.sized_walk = pairs >= kRowWalkCtas;
    d.walk = d.sized_walk;
    // Rows of at most two chunks whose split CTAs (one per chunk) need a second wave on the
    // device while one CTA per pair fits in one: walking takes one wave and no merge kernel
    // (the dense HCA step: 64 sequences x 2 head groups x 2 chunks, where the split form took
    // 21 us in two waves plus 15 us of merge kernel on GB300).
    const int sms = sm_count() > 0 ? sm_count() : 148;
    if (!d.walk && d.n_chunks <= 2) {
        if (pairs <= sms && pairs * d.n_chunks > sms) d.walk = true;
    }
    // Walking rows whose 64-head CTAs alone fill the device (the prefill chunk: 2048 rows): one
    // CTA per 64 heads does a chunk for twice the heads at little more cost (attn_rows64_kernel).
    // The workspace rule above (32-head pairs) does not change.
    if (d.walk && a.dim == 512 && a.heads % 64 == 0 &&
        static_cast<long long>(a.batch) * a.n_q * (a.heads / 64) >= sms) {
        d.nh = 64;
        d.n_hg = a.heads / 64;
    }
    // Split CTAs of 32 heads that need a second wave while CTAs of 64 heads fit in one (the
    // 8K-context batch-16 step: 160 CTAs on 152 SMs, where the 8 left over took as long as
    // the first wave): one CTA per 64 heads. The partials' layout (and the workspace) does
    // not change: the same heads at the same offsets.
    if (!d.walk && a.dim == 512 && a.heads % 64 == 0) {
        const long long ctas = static_cast<long long>(a.batch) * a.n_q * d.n_chunks;
        if (ctas * (a.heads / 32) > sms && ctas * (a.heads / 64) <= sms) {
            d.nh = 64;
            d.n_hg = a.heads / 64;
        }
    }
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
    p.n_chunks = dp.n_chunks;
    p.n_splits = dp.n_chunks;
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
    const WaitCtl wc = wait_ctl(DSV4_WAIT_FAULT_ATTN_QUERY);
    p.fault = dp.walk ? 0 : wc.fault;              // the control applies to the split form only
    p.wait_ns = wc.wait_ns;
    if (once_per_device(reinterpret_cast<const void*>(attn_decode_kernel<D, NH>), kAttrLaunch, [] {
            const cudaError_t e = cudaFuncSetAttribute(attn_decode_kernel<D, NH>,
                                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                       static_cast<int>(C::SMEM));
            if (e != cudaSuccess) return e;
            if constexpr (NH > 32)
                return cudaFuncSetAttribute(attn_rows64_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            static_cast<int>(Rows64Cfg::SMEM));
            return cudaFuncSetAttribute(attn_rows_kernel<D, NH <= 32 ? NH : 32>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(C::SMEM));
        }) != cudaSuccess)
        return DSV4_ERR_LAUNCH;
    if constexpr (NH > 32) {
        if (dp.walk) {                                 // one CTA per (query row, 64 heads)
            static_assert(D == Rows64Cfg::D && NH == Rows64Cfg::NH, "64-head walk shape");
            count_launch();
            return launch_k(attn_rows64_kernel, dim3(static_cast<unsigned>(rows) * dp.n_hg), dim3(kFT),
                            Rows64Cfg::SMEM, st, true, qmap, gmap, p, static_cast<const __nv_bfloat16*>(a.comp_kv),
                            static_cast<const __nv_bfloat16*>(a.win), a.gather ? 1 : 0) == cudaSuccess
                       ? DSV4_OK
                       : DSV4_ERR_LAUNCH;
        }
    }
    if constexpr (NH <= 32) {
        if (dp.walk) {                                 // one CTA per (query row, head group)
            count_launch();
            return launch_k(attn_rows_kernel<D, NH>, dim3(static_cast<unsigned>(rows) * dp.n_hg), dim3(kFT),
                            C::SMEM, st, true, qmap, gmap, p, static_cast<const __nv_bfloat16*>(a.comp_kv),
                            static_cast<const __nv_bfloat16*>(a.win), a.gather ? 1 : 0) == cudaSuccess
                       ? DSV4_OK
                       : DSV4_ERR_LAUNCH;
        }
    }
    dim3 grid(dp.n_chunks, rows, dp.n_hg);
    count_launch();
    if (launch_k(attn_decode_kernel<D, NH>, grid, dim3(kFT), C::SMEM, st, true, qmap, gmap, p,
                 static_cast<const __nv_bfloat16*>(a.comp_kv), static_cast<const __nv_bfloat16*>(a.win),
                 a.gather ? 1 : 0) != cudaSuccess)
        return DSV4_ERR_LAUNCH;
    dim3 g2(rows, a.heads);
    count_launch();
    if (launch_k(attn_combine_kernel<D>, g2, dim3(128), static_cast<size_t>(dp.n_chunks) * 4, st, true, p) !=
        cudaSuccess)
        return DSV4_ERR_LAUNCH;
    return DSV4_OK;
}

}  // namespace

size_t attn_ws_bytes(const dsv4_attn_args& a) {
    const DecodePlan dp = decode_plan(a);
    if (dp.sized_walk) return 0;                       // no partials
    const size_t rows = static_cast<size_t>(a.batch) * a.n_q;
    const size_t hs = static_cast<size_t>(dp.n_hg) * dp.nh;
    return align_up(rows * dp.n_chunks * hs * 2 * 4, 256) +
           align_up(rows * dp.n_chunks * hs * static_cast<size_t>(a.dim) * 4, 256);
}

int launch_attn(const dsv4_attn_args& a, uint8_t* ws, uint32_t* eword, cudaStream_t st) {
    if (a.batch * a.n_q == 0) return DSV4_OK;
    const DecodePlan dp = decode_plan(a);
    if (dp.nh == 64) return run_decode<512, 64>(a, dp, ws, eword, st);
    if (dp.nh == 16) {
        if (a.dim == 512) return run_decode<512, 16>(a, dp, ws, eword, st);
        if (a.dim == 256) return run_decode<256, 16>(a, dp, ws, eword, st);
        return run_decode<128, 16>(a, dp, ws, eword, st);
    }
    if (a.dim == 512) return run_decode<512, 32>(a, dp, ws, eword, st);
    if (a.dim == 256) return run_decode<256, 32>(a, dp, ws, eword, st);
    return run_decode<128, 32>(a, dp, ws, eword, st);
}

}  // namespace dsv4

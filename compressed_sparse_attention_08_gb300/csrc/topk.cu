// Per-row top-k of fp32 scores: exact, deterministic, ties to the lower index, output in
// ascending index order padded with -1 to top_k.
//
// Sources: "nvfp4-megamoe-kernel: compare v0.1-e2e-working...v-c1-c2-c3-20260602",
// ARCHITECTURE_AND_MEMORY_AUDIT.md "F3" (tk = min(top_k, n_comp); topk over the scores);
// "nvfp4-megamoe-kernel: compare v-precision-floor-fix-20260603..pure-nvfp4",
// GETTING+CUDAGRAPH_READY.md "SECTION C" item 3 (a fixed-length index list, the invalid tail
// masked, no host read of the count).
//
// Every score becomes an order-preserving 32-bit key (-0 and +0 share a key). The k-th
// largest key T is found by radix selection (8-bit digits); the first `need_T` keys equal to
// T, in index order, complete the set. The winners are written in index order without a
// block-wide scan per element: each warp owns a contiguous run of positions, counts its
// (key > T) and (key == T) elements with ballots, one scan over the warps gives every warp
// its starting counts, and element i lands at  #greater-before(i) + min(#ties-before(i),
// need_T). Two implementations of the same rule:
//   * rows that fit in shared memory (max_comp <= kSmallCap): one CTA per row, keys in smem.
//   * long rows (1M context: 262,144 scores): one thread-block cluster of 16 CTAs per row,
//     one slice each. A histogram of the top 12 key bits per row (built by the scoring
//     kernel's epilogue when the scores come from the indexer, else by a histogram kernel)
//     gives the 12-bit bin that holds the k-th key; every CTA keeps, in index order, the
//     elements of its slice at or above that bin (a few thousand of 262,144 in all) and
//     counts bits 19..8 of the keys in that bin; counts, that second histogram and the kept
//     elements meet in the shared memory of the cluster's first CTA, so one 8-bit radix pass
//     over the short list gives the exact k-th key.
#include "common.cuh"
#include "internal.h"

namespace dsv4 {
namespace {

constexpr int kSmallCap = 32768;     // keys held in shared memory by the one-CTA path
constexpr int kBins = 4096;          // top-12-bit histogram of the long-row path
constexpr int kBinShift = 20;
constexpr int kFinalCap = 12288;     // (key, index) pairs the finalizer keeps in smem
constexpr int kMaxSlices = 64;
constexpr int kNT = 1024;
constexpr int kCl = 16;              // CTAs per row in the long-row cluster kernel (non-portable size)

// Inclusive scan over the 32 lanes of a warp.
__device__ __forceinline__ int warp_incl(int v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
    }
    return v;
}

// Shared-memory histogram increment, aggregated over the lanes of a warp that hit the same
// bin (scores cluster: without this, thousands of lanes serialise on one counter). Every
// lane of the warp must call it (active or not).
__device__ __forceinline__ void hist_add(uint32_t* hist, uint32_t bin, bool active) {
    const unsigned act = __ballot_sync(0xffffffffu, active);
    if (!active) return;
    const unsigned peers = __match_any_sync(act, bin);
    if ((threadIdx.x & 31) == static_cast<unsigned>(__ffs(peers) - 1))
        atomicAdd(&hist[bin], static_cast<uint32_t>(__popc(peers)));
}

// Radix selection among the keys whose top `known_bits` bits equal those of `prefix`
// (all keys when known_bits is 0): finds the k-th largest of them (1 <= k <= their count)
// with 8-bit digits below the known bits. On return T is that key and need_T how many keys
// equal to T belong to the top k.
template <int NT, class KeyAt>
__device__ void radix_select(int n, int k, KeyAt key_at, uint32_t* hist, int* bc,
                             uint32_t& T, int& need_T, uint32_t prefix = 0, int known_bits = 0) {
    uint32_t mask = known_bits ? ~0u << (32 - known_bits) : 0u;
    prefix &= mask;
    int need = k;
    for (int low = 32 - known_bits; low > 0;) {
        const int width = low >= 8 ? 8 : low;
        const int shift = low - width;
        const uint32_t dmask = (1u << width) - 1u;
        for (int i = threadIdx.x; i < 256; i += NT) hist[i] = 0;
        __syncthreads();
        for (int base = 0; base < n; base += NT) {
            const int i = base + threadIdx.x;
            const uint32_t key = i < n ? key_at(i) : 0u;
            const bool match = i < n && (key & mask) == prefix;
            hist_add(hist, (key >> shift) & dmask, match);
        }
        __syncthreads();
        if (threadIdx.x < 32) {
            const int lane = threadIdx.x;
            int c[8], s = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) { c[i] = static_cast<int>(hist[255 - (lane * 8 + i)]); s += c[i]; }
            const int inc = warp_incl(s);
            const int before = inc - s;
            if (before < need && inc >= need) {
                int acc = before;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if (acc + c[i] >= need) {
                        bc[0] = 255 - (lane * 8 + i);
                        bc[1] = acc;
                        break;
                    }
                    acc += c[i];
                }
            }
        }
        __syncthreads();
        const uint32_t d = static_cast<uint32_t>(bc[0]);
        need -= bc[1];
        prefix |= d << shift;
        mask |= dmask << shift;
        low = shift;
        __syncthreads();
    }
    T = prefix;
    need_T = need;
}

// Write the winners (key > T, and the first need_T keys == T) of positions 0..n-1 in
// position order: element i goes to out[#greater-before(i) + min(#ties-before(i), need_T)].
template <int NT, class KeyAt, class IdxAt>
__device__ void ordered_select(int n, uint32_t T, int need_T, KeyAt key_at, IdxAt idx_at,
                               int32_t* out, int* s_gt, int* s_tie) {
    constexpr int NW = NT / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int per = (n + NW - 1) / NW;
    const int lo = warp * per < n ? warp * per : n;
    const int hi = lo + per < n ? lo + per : n;
    int gt = 0, tie = 0;
    for (int base = lo; base < hi; base += 32) {
        const int i = base + lane;
        const uint32_t key = i < hi ? key_at(i) : 0u;
        gt += __popc(__ballot_sync(0xffffffffu, i < hi && key > T));
        tie += __popc(__ballot_sync(0xffffffffu, i < hi && key == T));
    }
    if (lane == 0) { s_gt[warp] = gt; s_tie[warp] = tie; }
    __syncthreads();
    if (warp == 0) {
        const int g = lane < NW ? s_gt[lane] : 0, t = lane < NW ? s_tie[lane] : 0;
        const int gi = warp_incl(g), ti = warp_incl(t);
        if (lane < NW) { s_gt[lane] = gi - g; s_tie[lane] = ti - t; }
    }
    __syncthreads();
    int gb = s_gt[warp], tb = s_tie[warp];
    const unsigned lt = (1u << lane) - 1u;
    for (int base = lo; base < hi; base += 32) {
        const int i = base + lane;
        const uint32_t key = i < hi ? key_at(i) : 0u;
        const bool g = i < hi && key > T, t = i < hi && key == T;
        const unsigned bg = __ballot_sync(0xffffffffu, g), bt = __ballot_sync(0xffffffffu, t);
        const int g_before = gb + __popc(bg & lt), t_before = tb + __popc(bt & lt);
        if (g || (t && t_before < need_T)) out[g_before + (t_before < need_T ? t_before : need_T)] = idx_at(i);
        gb += __popc(bg);
        tb += __popc(bt);
    }
    __syncthreads();
}

// Rows where every visible entry is selected: 0..n-1 then -1.
__device__ __forceinline__ void write_all(int32_t* out, int n, int top_k, int from, int to,
                                          int step) {
    for (int j = from; j < to && j < top_k; j += step) out[j] = j < n ? j : -1;
}

// ------------------------------------------------------------------ one CTA per row
template <int NT>
__global__ void __launch_bounds__(NT)
topk_small_kernel(TopkRows t, uint32_t* eword) {
    extern __shared__ uint32_t skeys[];
    __shared__ uint32_t hist[256];
    __shared__ int s_a[32], s_b[32];
    __shared__ int bc[2];
    pdl_trigger();
    pdl_wait();
    const int row = blockIdx.x;
    const int n = row_visible(t.n_vis, t.n_comp, t.q_pos, t.n_q, t.ratio, t.max_comp, row, eword);
    const int k = n < t.top_k ? n : t.top_k;
    int32_t* out = t.idx_out + static_cast<size_t>(row) * t.top_k;
    if (k == n) {
        write_all(out, n, t.top_k, threadIdx.x, t.top_k, NT);
        return;
    }
    for (int j = k + threadIdx.x; j < t.top_k; j += NT) out[j] = -1;
    const float* s = t.scores + static_cast<size_t>(row) * t.max_comp;
    for (int i = threadIdx.x; i < n; i += NT) skeys[i] = float_to_key(s[i]);
    __syncthreads();
    uint32_t T;
    int need_T;
    auto key_at = [&](int i) { return skeys[i]; };
    radix_select<NT>(n, k, key_at, hist, bc, T, need_T);
    ordered_select<NT>(n, T, need_T, key_at, [](int i) { return i; }, out, s_a, s_b);
}

// ------------------------------------------------------------------ long rows
struct LongWs {
    uint32_t* hist;     // [rows, kBins]: top 12 key bits (bits 31..20) of every visible key
    uint2* pairs;       // [rows, max_comp]: (key, index) survivors when they outnumber kFinalCap
};

__device__ __forceinline__ void slice_range(int n, int L, int p, int& lo, int& hi) {
    lo = p * L < n ? p * L : n;
    hi = lo + L < n ? lo + L : n;
}

// The bin of a kBins-bin histogram that holds the k-th largest key (1 <= k <= total count),
// counting from the top bin down, and how many keys lie in the bins above it: bc[0] = bin,
// bc[1] = count above, bc[2] = the bin's own count. Thread t passes in c[i] the count of bin
// kBins-1-(t*per+i). Every thread of the CTA calls it.
template <int NT>
__device__ __forceinline__ void find_bin(const int (&c)[kBins / NT], int k, int* s_a, int* bc) {
    constexpr int NW = NT / 32, per = kBins / NT;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int s = 0;
#pragma unroll
    for (int i = 0; i < per; ++i) s += c[i];
    int inc = warp_incl(s);
    if (lane == 31) s_a[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        const int v = lane < NW ? s_a[lane] : 0;
        const int vi = warp_incl(v);
        if (lane < NW) s_a[lane] = vi - v;
    }
    __syncthreads();
    inc += s_a[warp];
    const int before = inc - s;
    if (before < k && inc >= k) {
        int acc = before;
#pragma unroll
        for (int i = 0; i < per; ++i) {
            if (acc + c[i] >= k) {
                bc[0] = kBins - 1 - (static_cast<int>(threadIdx.x) * per + i);
                bc[1] = acc;
                bc[2] = c[i];
                break;
            }
            acc += c[i];
        }
    }
    __syncthreads();
}

template <int NT>
__global__ void __launch_bounds__(NT)
topk_hist_kernel(TopkRows t, LongWs w, int L, uint32_t* eword) {
    __shared__ uint32_t h[kBins];
    pdl_trigger();
    pdl_wait();
    const int row = blockIdx.x, p = blockIdx.y;
    const int n = row_visible(t.n_vis, t.n_comp, t.q_pos, t.n_q, t.ratio, t.max_comp, row, eword);
    if (n <= t.top_k) return;
    int lo, hi;
    slice_range(n, L, p, lo, hi);
    if (lo >= hi) return;
    for (int i = threadIdx.x; i < kBins; i += NT) h[i] = 0;
    __syncthreads();
    const float* s = t.scores + static_cast<size_t>(row) * t.max_comp;
    for (int i = lo + threadIdx.x; i < hi; i += NT) atomicAdd(&h[float_to_key(s[i]) >> kBinShift], 1u);
    __syncthreads();
    uint32_t* g = w.hist + static_cast<size_t>(row) * kBins;
    for (int i = threadIdx.x; i < kBins; i += NT)
        if (h[i]) atomicAdd(&g[i], h[i]);
}

// Long rows, one cluster of CL CTAs per row; CTA r takes slice r of the row. Every CTA: the
// 12-bit threshold bin tb from the row histogram; its survivors (key bin >= tb), counted;
// bits 19..8 of its keys in bin tb into a shared histogram. Through distributed shared
// memory each CTA then adds that histogram into CTA 0's and posts its count there; after a
// cluster barrier every CTA knows every count, and writes its survivors, in index order,
// straight into CTA 0's shared list at its offset (into the global list when the survivors
// outnumber the shared list). After a last cluster barrier CTA 0 finds the second-level bin,
// so one 8-bit radix pass (none when the whole sub-bin is selected) gives the exact k-th key,
// and writes the k indices. No global atomics, tickets or round trips through L2 between
// the phases.
template <int NT, int CL>
__global__ void __launch_bounds__(NT, 1)
topk_cluster_kernel(TopkRows t, LongWs w, int L, uint32_t* eword) {
    constexpr int NW = NT / 32;
    constexpr int kRegs = 16;                    // scores per lane kept in registers
    constexpr int per_bin = kBins / NT;
    extern __shared__ uint2 spairs[];           // CTA 0: the survivors (kFinalCap pairs)
    __shared__ uint32_t h2loc[kBins];           // this CTA's bits 19..8 of bin tb
    __shared__ uint32_t h2sum[kBins];           // CTA 0: the row's
    __shared__ uint32_t hist[256];
    __shared__ int s_a[32], s_b[32], s_w[32];
    __shared__ int bc[3];
    __shared__ int cl_count[CL];                // CTA 0: survivors per CTA
    __shared__ int offs[CL + 1];
    pdl_trigger();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t rank = cluster_rank();
    const int row = blockIdx.y;
    const int k = t.top_k;
    // the sums CTA 0 collects start at zero before any CTA adds into them
    for (int i = threadIdx.x; i < kBins; i += NT) { h2loc[i] = 0; h2sum[i] = 0; }
    if (threadIdx.x < CL) cl_count[threadIdx.x] = 0;
    __syncthreads();
    cluster_arrive();
    pdl_wait();
    // The row histogram, this slice's scores and the visible count do not depend on one
    // another: issue their loads together. The slice is read over its full extent (inside
    // the row's max_comp scores); entries at or past the visible count are masked below.
    const uint32_t* g1 = w.hist + static_cast<size_t>(row) * kBins;
    int c[per_bin];
#pragma unroll
    for (int i = 0; i < per_bin; ++i)
        c[i] = static_cast<int>(__ldcg(&g1[kBins - 1 - (static_cast<int>(threadIdx.x) * per_bin + i)]));
    const int slo = static_cast<int>(rank) * L < t.max_comp ? static_cast<int>(rank) * L : t.max_comp;
    const int shi = slo + L < t.max_comp ? slo + L : t.max_comp;
    const int wper = (shi - slo + NW - 1) / NW;  // warp-contiguous runs of the slice
    const int wlo = slo + (warp * wper < shi - slo ? warp * wper : shi - slo);
    const int whi = wlo + wper < shi ? wlo + wper : shi;
    const bool in_regs = wper <= 32 * kRegs;     // the same for every warp of the CTA
    const float* sc = t.scores + static_cast<size_t>(row) * t.max_comp;
    // loaded once, up front, and kept (a volatile load: the compiler may not re-issue it in
    // the two passes below)
    float v0[kRegs];
    if (in_regs) {
#pragma unroll
        for (int r = 0; r < kRegs; ++r) {
            const int i = wlo + r * 32 + lane;
            v0[r] = 0.f;
            if (i < whi) asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v0[r]) : "l"(sc + i));
        }
    }
    const int n = row_visible(t.n_vis, t.n_comp, t.q_pos, t.n_q, t.ratio, t.max_comp, row, eword);
    int32_t* out = t.idx_out + static_cast<size_t>(row) * k;
    if (n <= k) {                                // every visible entry is selected
        const int per = (k + CL - 1) / CL;
        write_all(out, n, k, static_cast<int>(rank) * per + threadIdx.x, (static_cast<int>(rank) + 1) * per, NT);
        cluster_wait();
        return;
    }
    const int hi = whi < n ? whi : n;            // visible end of this warp's run
    // 1. the 12-bit bin tb holding the k-th largest key, and how many keys lie above it
    find_bin<NT>(c, k, s_a, bc);
    const uint32_t tb = static_cast<uint32_t>(bc[0]);
    const int above = bc[1];
    // 2. count this warp's survivors (bin >= tb); keys in bin tb also go into the second
    //    histogram
    int cnt = 0;
    for (int b0 = wlo; b0 < whi; b0 += 32 * kRegs) {
#pragma unroll
        for (int r = 0; r < kRegs; ++r) {
            const int i = b0 + r * 32 + lane;
            const bool vis = i < hi;
            const uint32_t key = float_to_key(in_regs ? v0[r] : (vis ? __ldcg(&sc[i]) : 0.f));
            const uint32_t bin = key >> kBinShift;
            const unsigned bs = __ballot_sync(0xffffffffu, vis && bin >= tb);
            if (bs == 0u) continue;                 // most groups of 32 keep nothing
            cnt += __popc(bs);
            // few keys fall in bin tb, spread over 4096 sub-bins: plain atomics
            if (vis && bin == tb) atomicAdd(&h2loc[(key >> 8) & (kBins - 1)], 1u);
        }
    }
    if (lane == 0) s_w[warp] = cnt;
    __syncthreads();
    if (warp == 0) {
        const int v = lane < NW ? s_w[lane] : 0;
        const int vi = warp_incl(v);
        if (lane < NW) s_w[lane] = vi - v;       // the warp's offset within the CTA
        if (lane == NW - 1) s_b[0] = vi;         // the CTA's count
    }
    // 3. post the count and the second histogram to CTA 0 (its sums are zeroed: wait for that)
    cluster_wait();
    __syncthreads();
    if (threadIdx.x == 0) st_cluster_u32(cluster_map(&cl_count[rank], 0), static_cast<uint32_t>(s_b[0]));
    {
        const uint32_t h2r = cluster_map(h2sum, 0);
        for (int i = threadIdx.x; i < kBins; i += NT) {
            const uint32_t v = h2loc[i];
            if (v) red_cluster_add(h2r + 4u * static_cast<uint32_t>(i), v);
        }
    }
    cluster_arrive();
    cluster_wait();
    // 4. every CTA's offset in the row's list; the survivors go there in index order
    if (warp == 0) {
        const int v = lane < CL ? static_cast<int>(ld_cluster_u32(cluster_map(&cl_count[lane], 0))) : 0;
        const int vi = warp_incl(v);
        if (lane < CL) offs[lane + 1] = vi;
        if (lane == 0) offs[0] = 0;
    }
    __syncthreads();
    const int total = offs[CL];
    const bool in_smem = total <= kFinalCap;
    {
        int pos = offs[rank] + s_w[warp];
        const unsigned lt = (1u << lane) - 1u;
        const uint32_t sp0 = cluster_map(spairs, 0);
        uint2* gp = w.pairs + static_cast<size_t>(row) * t.max_comp;
        for (int b0 = wlo; b0 < whi; b0 += 32 * kRegs) {
#pragma unroll
            for (int r = 0; r < kRegs; ++r) {
                const int i = b0 + r * 32 + lane;
                const uint32_t key = float_to_key(in_regs ? v0[r] : (i < hi ? __ldcg(&sc[i]) : 0.f));
                const bool keep = i < hi && (key >> kBinShift) >= tb;
                const unsigned bk = __ballot_sync(0xffffffffu, keep);
                if (bk == 0u) continue;
                if (keep) {
                    const int at = pos + __popc(bk & lt);
                    if (in_smem) st_cluster_v2(sp0 + 8u * static_cast<uint32_t>(at), key, static_cast<uint32_t>(i));
                    else gp[at] = make_uint2(key, static_cast<uint32_t>(i));
                }
                pos += __popc(bk);
            }
        }
    }
    cluster_arrive();
    cluster_wait();
    if (rank != 0) return;
    // 5. CTA 0: the 12-bit sub-bin (bits 19..8) of bin tb holding the k-th key
    int c2[per_bin];
#pragma unroll
    for (int i = 0; i < per_bin; ++i)
        c2[i] = static_cast<int>(h2sum[kBins - 1 - (static_cast<int>(threadIdx.x) * per_bin + i)]);
    find_bin<NT>(c2, k - above, s_a, bc);
    const uint32_t prefix = (tb << kBinShift) | (static_cast<uint32_t>(bc[0]) << 8);
    const int need = k - above - bc[1];
    const bool whole_sub_bin = need == bc[2] && prefix != 0u;   // every key of the sub-bin is in
    uint32_t T;
    int need_T;
    auto finish = [&](auto key_at, auto idx_at) {
        if (whole_sub_bin) {
            // the k keys are exactly those at or above the sub-bin: no selection inside it
            T = prefix - 1u;
            need_T = 0;
        } else {
            radix_select<NT>(total, need, key_at, hist, bc, T, need_T, prefix, 32 - 8);
        }
        ordered_select<NT>(total, T, need_T, key_at, idx_at, out, s_a, s_b);
    };
    if (in_smem) {
        finish([&](int i) { return spairs[i].x; }, [&](int i) { return static_cast<int32_t>(spairs[i].y); });
    } else {
        // degenerate score distributions (huge ties): the list in global memory
        const uint2* gp = w.pairs + static_cast<size_t>(row) * t.max_comp;
        finish([&](int i) { return __ldcg(&gp[i]).x; }, [&](int i) { return static_cast<int32_t>(__ldcg(&gp[i]).y); });
    }
}

struct LongPlan { int P, L; };

LongPlan long_plan(int rows, int max_comp) {
    const int sms = sm_count() > 0 ? sm_count() : 148;
    int P = (sms + rows - 1) / (rows > 0 ? rows : 1);
    if (P < 1) P = 1;
    if (P > kMaxSlices) P = kMaxSlices;
    int L = (max_comp + P - 1) / P;
    L = (L + 1023) / 1024 * 1024;
    P = (max_comp + L - 1) / L;
    if (P < 1) P = 1;
    return {P, L};
}

}  // namespace

size_t topk_ws_bytes(int rows, int max_comp, int top_k) {
    (void)top_k;
    if (max_comp <= kSmallCap) return 0;
    size_t b = 0;
    b += align_up(static_cast<size_t>(rows) * kBins * 4, 256);   // the row histograms
    b += align_up(static_cast<size_t>(rows) * max_comp * 8, 256);
    return b;
}

uint32_t* topk_hist_buffer(uint8_t* ws) { return reinterpret_cast<uint32_t*>(ws); }
size_t topk_hist_bytes(int rows) { return static_cast<size_t>(rows) * kBins * 4; }
bool topk_uses_hist(int max_comp) { return max_comp > kSmallCap; }

int launch_topk(const TopkRows& t, uint8_t* ws, uint32_t* eword, cudaStream_t stream) {
    if (t.rows == 0) return DSV4_OK;
    if (t.max_comp <= kSmallCap) {
        const size_t smem = static_cast<size_t>(t.max_comp > 0 ? t.max_comp : 1) * 4;
        if (once_per_device(reinterpret_cast<const void*>(topk_small_kernel<kNT>), kAttrLaunch, [] {
                return cudaFuncSetAttribute(topk_small_kernel<kNT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            kSmallCap * 4);
            }) != cudaSuccess)
            return DSV4_ERR_LAUNCH;
        count_launch();
        return launch_k(topk_small_kernel<kNT>, dim3(t.rows), dim3(kNT), smem, stream, t.pdl, t, eword)
                   == cudaSuccess ? DSV4_OK : DSV4_ERR_LAUNCH;
    }
    const LongPlan pl = long_plan(t.rows, t.max_comp);
    LongWs w;
    uint8_t* p = ws;
    w.hist = reinterpret_cast<uint32_t*>(p);
    p += align_up(static_cast<size_t>(t.rows) * kBins * 4, 256);
    w.pairs = reinterpret_cast<uint2*>(p);
    if (!t.hist_zeroed &&
        cudaMemsetAsync(w.hist, 0, topk_hist_bytes(t.rows), stream) != cudaSuccess)
        return DSV4_ERR_LAUNCH;
    if (once_per_device(reinterpret_cast<const void*>(topk_cluster_kernel<kNT, kCl>), kAttrLaunch, [] {
            const cudaError_t e = cudaFuncSetAttribute(topk_cluster_kernel<kNT, kCl>,
                                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kFinalCap * 8);
            if (e != cudaSuccess || kCl <= 8) return e;
            return cudaFuncSetAttribute(topk_cluster_kernel<kNT, kCl>,
                                        cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        }) != cudaSuccess)
        return DSV4_ERR_LAUNCH;
    if (!t.hist_built) {
        count_launch();
        if (launch_k(topk_hist_kernel<kNT>, dim3(t.rows, pl.P), dim3(kNT), 0, stream, t.pdl, t, w, pl.L, eword)
            != cudaSuccess)
            return DSV4_ERR_LAUNCH;
    }
    // slices of the cluster kernel: CTA r of a row's cluster takes [r * Lc, (r + 1) * Lc)
    const int Lc = (t.max_comp + kCl - 1) / kCl;
    count_launch();
    return launch_cluster_k(topk_cluster_kernel<kNT, kCl>, dim3(kCl, t.rows), dim3(kNT), size_t(kFinalCap * 8),
                            stream, t.pdl, static_cast<unsigned>(kCl), t, w, Lc, eword) == cudaSuccess
               ? DSV4_OK : DSV4_ERR_LAUNCH;
}

}  // namespace dsv4

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
//     one slice each, its scores in registers. A histogram of the top 12 key bits per row
//     (built by the scoring kernel's epilogue when the scores come from the indexer, else by
//     a histogram kernel) gives the 12-bit bin that holds the k-th key; the counts of bits
//     19..8 of the keys in that bin, summed over the cluster, give its 24-bit prefix (an 8-bit
//     pass over the few keys sharing that prefix gives the exact key when some are left out);
//     every CTA then writes its own winners at the offset the cluster's counts give it.
#include "common.cuh"
#include "internal.h"

namespace dsv4 {
namespace {

constexpr int kSmallCap = 32768;     // keys held in shared memory by the one-CTA path
constexpr int kBins = 4096;          // top-12-bit histogram of the long-row path
constexpr int kBinShift = 20;
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

// ------------------------------------------------------------------ long rows
struct LongWs {
    uint32_t* hist;     // [rows, kBins]: top 12 key bits (bits 31..20) of every visible key
    uint32_t* h2;       // [rows, kBins]: bits 19..8 of the keys in the threshold bin
    uint32_t* h3;       // [rows, 256]: bits 7..0 of the keys sharing the k-th key's prefix
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

// ------------------------------------------------------------------ one CTA per row
// Rows up to kSmallCap keys, held in shared memory: a histogram of the top 12 key bits gives
// the bin of the k-th key, a histogram of bits 19..8 of that bin's keys its 24-bit prefix, and
// (only when some keys with that prefix are left out) one 8-bit radix pass the exact key.
template <int NT>
__global__ void __launch_bounds__(NT)
topk_small_kernel(TopkRows t, uint32_t* eword) {
    constexpr int per_bin = kBins / NT;
    extern __shared__ uint32_t skeys[];
    __shared__ uint32_t h12[kBins];
    __shared__ uint32_t hist[256];
    __shared__ int s_a[32], s_b[32];
    __shared__ int bc[3];
    pdl_trigger();
    for (int i = threadIdx.x; i < kBins; i += NT) h12[i] = 0;
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
    // 1. the top 12 bits (warp-aggregated: scores share few exponents)
    for (int base = 0; base < n; base += NT) {
        const int i = base + threadIdx.x;
        const uint32_t key = i < n ? skeys[i] : 0u;
        hist_add(h12, key >> kBinShift, i < n);
    }
    __syncthreads();
    int c[per_bin];
#pragma unroll
    for (int i = 0; i < per_bin; ++i) c[i] = static_cast<int>(h12[kBins - 1 - (static_cast<int>(threadIdx.x) * per_bin + i)]);
    find_bin<NT>(c, k, s_a, bc);                 // (its barriers: every thread has read h12)
    const uint32_t tb = static_cast<uint32_t>(bc[0]);
    const int above = bc[1];
    for (int i = threadIdx.x; i < kBins; i += NT) h12[i] = 0;
    __syncthreads();
    // 2. bits 19..8 of the keys in bin tb
    for (int base = 0; base < n; base += NT) {
        const int i = base + threadIdx.x;
        const uint32_t key = i < n ? skeys[i] : 0u;
        hist_add(h12, (key >> 8) & (kBins - 1), i < n && (key >> kBinShift) == tb);
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < per_bin; ++i) c[i] = static_cast<int>(h12[kBins - 1 - (static_cast<int>(threadIdx.x) * per_bin + i)]);
    find_bin<NT>(c, k - above, s_a, bc);
    const uint32_t prefix = (tb << kBinShift) | (static_cast<uint32_t>(bc[0]) << 8);
    const int need = k - above - bc[1];
    uint32_t T;
    int need_T;
    auto key_at = [&](int i) { return skeys[i]; };
    if (need == bc[2] && prefix != 0u) {
        T = prefix - 1u;                         // the whole sub-bin is selected
        need_T = 0;
    } else {
        radix_select<NT>(n, need, key_at, hist, bc, T, need_T, prefix, 32 - 8);
    }
    ordered_select<NT>(n, T, need_T, key_at, [](int i) { return i; }, out, s_a, s_b);
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

// Long rows, one cluster of CL CTAs per row; CTA r takes slice r of the row (its scores held
// in registers). Every CTA: the 12-bit threshold bin tb from the row histogram; bits 19..8 of
// its keys in bin tb counted in shared memory and added into the row's sub-bin counts in L2
// (global atomics spread over the L2 slices). After a cluster barrier every CTA reads the
// summed counts back (one load per thread) and finds the k-th key's 24-bit prefix itself;
// when some keys with that prefix are left out, a second round over bits 7..0 gives the
// exact key T. Each CTA then counts its keys above T and its ties at T, the counts go to
// every CTA through distributed shared memory, and after a last cluster barrier each CTA
// writes its own winners, in index order, at its offset in the row's index list (ties at T
// to the lower index: CTA order is index order). No survivor list is gathered and no CTA's
// shared memory is the target of more than a few dozen remote accesses: remote accesses
// into one SM are served one at a time, so funnelling the row's data into one CTA costs
// more than the round trips through L2.
template <int NT, int CL>
__global__ void __launch_bounds__(NT, 1)
topk_cluster_kernel(TopkRows t, LongWs w, int L, uint32_t* eword) {
    constexpr int NW = NT / 32;
    constexpr int kRegs = 16;                    // scores per lane kept in registers
    constexpr int per_bin = kBins / NT;
    __shared__ uint32_t h2loc[kBins];           // this CTA's bits 19..8 of bin tb
    __shared__ uint32_t h3loc[256];             // its bits 7..0 of the k-th key's prefix (rare)
    __shared__ int s_a[32], s_gw[32], s_tw[32], s_tot[2];
    __shared__ int bc[3];
    __shared__ uint32_t s_T[2];                 // the exact key and the ties taken (third pass)
    __shared__ int s_cnt[CL][2];                // every CTA's (keys above T, ties at T)
    pdl_trigger();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint32_t rank = cluster_rank();
    const int row = blockIdx.y;
    const int k = t.top_k;
    for (int i = threadIdx.x; i < kBins; i += NT) h2loc[i] = 0;
    for (int i = threadIdx.x; i < 256; i += NT) h3loc[i] = 0;
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
    // the passes below)
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
    if (n <= k) {                                // every visible entry is selected (every CTA)
        const int per = (k + CL - 1) / CL;
        write_all(out, n, k, static_cast<int>(rank) * per + threadIdx.x, (static_cast<int>(rank) + 1) * per, NT);
        return;
    }
    const int hi = whi < n ? whi : n;            // visible end of this warp's run
    // The passes below are bound by instruction issue (16,384 keys per SM), so each key is
    // formed once and entries past the visible end get key 0. No score has key 0 (it is a NaN
    // bit pattern; -inf is 0x007fffff), so it lies in no bin from tb on (tb >= 7), shares no
    // prefix of the k-th key and is never >= T (T > 0): no pass needs an "i < hi" test.
    uint32_t kr[kRegs];
#pragma unroll
    for (int r = 0; r < kRegs; ++r) kr[r] = wlo + r * 32 + lane < hi ? float_to_key(v0[r]) : 0u;
    // key r of this lane's run (from registers, or read again from L2 for long slices)
    auto key_of = [&](int b0, int r, int& i) -> uint32_t {
        i = b0 + r * 32 + lane;
        return in_regs ? kr[r] : (i < hi ? float_to_key(__ldcg(&sc[i])) : 0u);
    };
    // 1. the 12-bit bin tb holding the k-th largest key, and how many keys lie above it (the
    //    scan's barriers also order the zeroing of h2loc before its use); bits 19..8 of this
    //    CTA's keys in bin tb into its sub-bin counts, then into the row's in L2
    find_bin<NT>(c, k, s_a, bc);
    const uint32_t tb = static_cast<uint32_t>(bc[0]);
    const int above = bc[1];
    for (int b0 = wlo; b0 < whi; b0 += 32 * kRegs) {
#pragma unroll
        for (int r = 0; r < kRegs; ++r) {
            int i;
            const uint32_t key = key_of(b0, r, i);
            // few keys fall in bin tb, mostly spread over the 4096 sub-bins (lanes that hit
            // the same sub-bin, as heavy ties do, add once)
            hist_add(h2loc, (key >> 8) & (kBins - 1), (key >> kBinShift) == tb);
        }
    }
    __syncthreads();
    uint32_t* g2 = w.h2 + static_cast<size_t>(row) * kBins;
    for (int i = threadIdx.x; i < kBins; i += NT) {
        const uint32_t v = h2loc[i];
        if (v) atomicAdd(&g2[i], v);
    }
    cluster_arrive();                            // release: this CTA's counts are in L2
    cluster_wait();                              // acquire: so are every other CTA's
    // 2. every CTA: the sub-bin of the k-th key from the row's sums
    int c2[per_bin];
#pragma unroll
    for (int i = 0; i < per_bin; ++i)
        c2[i] = static_cast<int>(__ldcg(&g2[kBins - 1 - (static_cast<int>(threadIdx.x) * per_bin + i)]));
    find_bin<NT>(c2, k - above, s_a, bc);
    const uint32_t prefix = (tb << kBinShift) | (static_cast<uint32_t>(bc[0]) << 8);
    const int need = k - above - bc[1];
    uint32_t T;
    int need_T;
    if (need == bc[2] && prefix != 0u) {
        // the whole sub-bin is selected: the k keys are those at or above its lower edge
        T = prefix - 1u;
        need_T = 0;
    } else {
        // 3. (rare) some keys with the k-th key's 24-bit prefix are left out: bits 7..0 of
        //    those keys over the cluster give the exact key and how many of its ties are taken
        for (int b0 = wlo; b0 < whi; b0 += 32 * kRegs) {
#pragma unroll
            for (int r = 0; r < kRegs; ++r) {
                int i;
                const uint32_t key = key_of(b0, r, i);
                hist_add(h3loc, key & 255u, (key >> 8) == (prefix >> 8));
            }
        }
        __syncthreads();
        uint32_t* g3 = w.h3 + static_cast<size_t>(row) * 256;
        for (int i = threadIdx.x; i < 256; i += NT) {
            const uint32_t v = h3loc[i];
            if (v) atomicAdd(&g3[i], v);
        }
        cluster_arrive();
        cluster_wait();
        if (warp == 0) {
            int cc[8], sum = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                cc[i] = static_cast<int>(__ldcg(&g3[255 - (lane * 8 + i)]));
                sum += cc[i];
            }
            const int inc = warp_incl(sum);
            const int before = inc - sum;
            if (before < need && inc >= need) {
                int acc = before;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if (acc + cc[i] >= need) {
                        s_T[0] = prefix | static_cast<uint32_t>(255 - (lane * 8 + i));
                        s_T[1] = static_cast<uint32_t>(need - acc);
                        break;
                    }
                    acc += cc[i];
                }
            }
        }
        __syncthreads();
        T = s_T[0];
        need_T = static_cast<int>(s_T[1]);
    }
    // 4. this CTA's keys above T and ties at T, per warp and in all; the counts to every CTA
    //    (every CTA has passed the barrier above, so its shared memory may be written)
    int gt = 0, tie = 0;                         // this lane's, then the warp's
    for (int b0 = wlo; b0 < whi; b0 += 32 * kRegs) {
#pragma unroll
        for (int r = 0; r < kRegs; ++r) {
            int i;
            const uint32_t key = key_of(b0, r, i);
            gt += key > T;
            tie += key == T;
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        gt += __shfl_xor_sync(0xffffffffu, gt, o);
        tie += __shfl_xor_sync(0xffffffffu, tie, o);
    }
    if (lane == 0) { s_gw[warp] = gt; s_tw[warp] = tie; }
    __syncthreads();
    if (warp == 0) {
        const int g = lane < NW ? s_gw[lane] : 0, tt = lane < NW ? s_tw[lane] : 0;
        const int gi = warp_incl(g), ti = warp_incl(tt);
        if (lane < NW) { s_gw[lane] = gi - g; s_tw[lane] = ti - tt; }
        if (lane == NW - 1) { s_tot[0] = gi; s_tot[1] = ti; }
    }
    __syncthreads();
    if (threadIdx.x < CL) {
        st_cluster_u32(cluster_map(&s_cnt[rank][0], threadIdx.x), static_cast<uint32_t>(s_tot[0]));
        st_cluster_u32(cluster_map(&s_cnt[rank][1], threadIdx.x), static_cast<uint32_t>(s_tot[1]));
    }
    cluster_arrive();
    cluster_wait();                              // every CTA's counts are in place
    // 5. this CTA's winners in index order at its offset: keys above T before it in the row,
    //    plus the ties at T taken before it
    int gt_before = 0, tie_before = 0;
    for (int r2 = 0; r2 < static_cast<int>(rank); ++r2) { gt_before += s_cnt[r2][0]; tie_before += s_cnt[r2][1]; }
    int gb = gt_before + s_gw[warp], tbf = tie_before + s_tw[warp];
    const unsigned lt = (1u << lane) - 1u;
    for (int b0 = wlo; b0 < whi; b0 += 32 * kRegs) {
#pragma unroll
        for (int r = 0; r < kRegs; ++r) {
            int i;
            const uint32_t key = key_of(b0, r, i);
            if (__ballot_sync(0xffffffffu, key >= T) == 0u) continue;   // most groups of 32 hold none
            const bool g = key > T, tq = key == T;
            const unsigned bg = __ballot_sync(0xffffffffu, g), bt = __ballot_sync(0xffffffffu, tq);
            const int g_b = gb + __popc(bg & lt), t_b = tbf + __popc(bt & lt);
            if (g || (tq && t_b < need_T)) out[g_b + (t_b < need_T ? t_b : need_T)] = i;
            gb += __popc(bg);
            tbf += __popc(bt);
        }
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
    return align_up(topk_hist_bytes(rows), 256);   // the row histograms, all zeroed per call
}

uint32_t* topk_hist_buffer(uint8_t* ws) { return reinterpret_cast<uint32_t*>(ws); }
size_t topk_hist_bytes(int rows) { return static_cast<size_t>(rows) * (2 * kBins + 256) * 4; }
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
    w.hist = reinterpret_cast<uint32_t*>(ws);
    w.h2 = w.hist + static_cast<size_t>(t.rows) * kBins;
    w.h3 = w.h2 + static_cast<size_t>(t.rows) * kBins;
    if (!t.hist_zeroed &&
        cudaMemsetAsync(w.hist, 0, topk_hist_bytes(t.rows), stream) != cudaSuccess)
        return DSV4_ERR_LAUNCH;
    if (once_per_device(reinterpret_cast<const void*>(topk_cluster_kernel<kNT, kCl>), kAttrLaunch, [] {
            return kCl <= 8 ? cudaSuccess
                            : cudaFuncSetAttribute(topk_cluster_kernel<kNT, kCl>,
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
    return launch_cluster_k(topk_cluster_kernel<kNT, kCl>, dim3(kCl, t.rows), dim3(kNT), size_t(0),
                            stream, t.pdl, static_cast<unsigned>(kCl), t, w, Lc, eword) == cudaSuccess
               ? DSV4_OK : DSV4_ERR_LAUNCH;
}

}  // namespace dsv4

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
//   * long rows (1M context: 262,144 scores): the row is cut into P slices, one CTA each. A
//     histogram of the top 12 key bits per row (built by the scoring kernel's epilogue when
//     the scores come from the indexer, else by a histogram kernel) gives the 12-bit bin
//     that holds the k-th key; every CTA keeps, in index order, the elements of its slice at
//     or above that bin (a few thousand of 262,144 in all) and counts bits 19..8 of the keys
//     in that bin into a second histogram; the last CTA of the row to finish (atomic ticket,
//     no spinning) reads the second histogram, so one 8-bit radix pass over the short list
//     gives the exact k-th key.
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
    uint32_t* hist2;    // [rows, kBins]: bits 19..8 of the keys in the threshold bin
    uint32_t* done;     // [rows] tickets
    int32_t* counts;    // [rows, kMaxSlices]
    uint2* pairs;       // [rows, max_comp]: (key, index) survivors, slice p at p * L
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

// Long rows, P CTAs per row. Each CTA: the 12-bit threshold bin tb from the row histogram;
// the survivors of its slice (key bin >= tb) in index order into its segment of the pair
// list; bits 19..8 of the keys in bin tb into the row's second histogram. The last CTA of
// the row (atomic ticket, no spinning) finds the second-level bin from that histogram, so one
// 8-bit radix pass over the survivors gives the exact k-th key, and writes the k indices.
template <int NT>
__global__ void __launch_bounds__(NT, 1)
topk_filter_kernel(TopkRows t, LongWs w, int L, int P, uint32_t* eword) {
    constexpr int NW = NT / 32;
    constexpr int kRegs = 8;                     // scores per lane kept in registers
    constexpr int per_bin = kBins / NT;
    extern __shared__ uint2 spairs[];           // kFinalCap pairs (finalizer only)
    __shared__ uint32_t hist[256];
    __shared__ int s_a[32], s_b[32];
    __shared__ int bc[3];
    __shared__ int offs[kMaxSlices + 1];
    __shared__ int is_last;
    pdl_trigger();
    pdl_wait();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int row = blockIdx.x, p = blockIdx.y;
    const int k = t.top_k;
    // The row histogram, this slice's scores and the visible count do not depend on one
    // another: issue their loads together. The slice is read over its full extent (inside
    // the row's max_comp scores); entries at or past the visible count are masked below.
    const uint32_t* g1 = w.hist + static_cast<size_t>(row) * kBins;
    int c[per_bin];
#pragma unroll
    for (int i = 0; i < per_bin; ++i)
        c[i] = static_cast<int>(__ldcg(&g1[kBins - 1 - (static_cast<int>(threadIdx.x) * per_bin + i)]));
    const int slo = p * L;                       // < max_comp: P = ceil(max_comp / L)
    const int shi = slo + L < t.max_comp ? slo + L : t.max_comp;
    const int wper = (shi - slo + NW - 1) / NW;  // warp-contiguous runs of the slice
    const int wlo = slo + (warp * wper < shi - slo ? warp * wper : shi - slo);
    const int whi = wlo + wper < shi ? wlo + wper : shi;
    const bool in_regs = wper <= 32 * kRegs;     // the same for every warp of the CTA
    const float* sc = t.scores + static_cast<size_t>(row) * t.max_comp;
    float v0[kRegs];
    if (in_regs) {
#pragma unroll
        for (int r = 0; r < kRegs; ++r) {
            const int i = wlo + r * 32 + lane;
            v0[r] = i < whi ? __ldcg(&sc[i]) : 0.f;
        }
    }
    const int n = row_visible(t.n_vis, t.n_comp, t.q_pos, t.n_q, t.ratio, t.max_comp, row, eword);
    int32_t* out = t.idx_out + static_cast<size_t>(row) * k;
    if (n <= k) {                                // every visible entry is selected
        const int per = (k + P - 1) / P;
        write_all(out, n, k, p * per + threadIdx.x, (p + 1) * per, NT);
        return;
    }
    const int hi = whi < n ? whi : n;            // visible end of this warp's run
    // 1. the 12-bit bin tb holding the k-th largest key, and how many keys lie above it
    find_bin<NT>(c, k, s_a, bc);
    const uint32_t tb = static_cast<uint32_t>(bc[0]);
    const int above = bc[1];
    // 2. count this warp's survivors (bin >= tb); keys in bin tb also go into the second
    //    histogram
    uint32_t* g2 = w.hist2 + static_cast<size_t>(row) * kBins;
    uint2* seg = w.pairs + static_cast<size_t>(row) * t.max_comp + static_cast<size_t>(slo);
    const unsigned lt = (1u << lane) - 1u;
    int cnt = 0;
    for (int b0 = wlo; b0 < whi; b0 += 32 * kRegs) {
        uint32_t key[kRegs];
#pragma unroll
        for (int r = 0; r < kRegs; ++r) {
            const int i = b0 + r * 32 + lane;
            key[r] = float_to_key(in_regs ? v0[r] : (i < hi ? __ldcg(&sc[i]) : 0.f));
        }
#pragma unroll
        for (int r = 0; r < kRegs; ++r) {
            const int i = b0 + r * 32 + lane;
            const bool vis = i < hi;
            const uint32_t bin = key[r] >> kBinShift;
            cnt += __popc(__ballot_sync(0xffffffffu, vis && bin >= tb));
            if (vis && bin == tb) atomicAdd(&g2[(key[r] >> 8) & (kBins - 1)], 1u);
        }
    }
    if (lane == 0) s_a[warp] = cnt;              // find_bin is done with s_a
    __syncthreads();
    if (warp == 0) {
        const int v = lane < NW ? s_a[lane] : 0;
        const int vi = warp_incl(v);
        if (lane < NW) s_a[lane] = vi - v;
        if (lane == NW - 1) s_b[0] = vi;
    }
    __syncthreads();
    // 3. write them, in index order, at the warp's offset in the slice's segment
    int pos = s_a[warp];
    for (int b0 = wlo; b0 < whi; b0 += 32 * kRegs) {
        uint32_t key[kRegs];
#pragma unroll
        for (int r = 0; r < kRegs; ++r) {
            const int i = b0 + r * 32 + lane;
            key[r] = float_to_key(in_regs ? v0[r] : (i < hi ? __ldcg(&sc[i]) : 0.f));
        }
#pragma unroll
        for (int r = 0; r < kRegs; ++r) {
            const int i = b0 + r * 32 + lane;
            const bool keep = i < hi && (key[r] >> kBinShift) >= tb;
            const unsigned bk = __ballot_sync(0xffffffffu, keep);
            if (keep) seg[pos + __popc(bk & lt)] = make_uint2(key[r], static_cast<uint32_t>(i));
            pos += __popc(bk);
        }
    }
    if (threadIdx.x == 0) w.counts[static_cast<size_t>(row) * kMaxSlices + p] = s_b[0];
    // 4. the last CTA of the row to get here finishes the row (no waiting on anyone)
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned ticket = atomicAdd(&w.done[row], 1u);
        is_last = ticket == static_cast<unsigned>(P - 1);
    }
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    // slice counts, the second histogram and the first kPairRegs * 32 survivors of the
    // slices this warp copies (slices warp and warp + 32; loaded before their counts are
    // known, from inside each slice's segment), all at once
    constexpr int kPairRegs = 4;
    const uint2* rowpairs = w.pairs + static_cast<size_t>(row) * t.max_comp;
    const int32_t* rowcounts = w.counts + static_cast<size_t>(row) * kMaxSlices;
    int cnt_w[2] = {0, 0};
    uint2 pr[2][kPairRegs];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int q = warp + 32 * h;
        if (q < P) {
            if (lane == 0) cnt_w[h] = __ldcg(&rowcounts[q]);
#pragma unroll
            for (int j = 0; j < kPairRegs; ++j) {
                const int i = lane + 32 * j;
                const bool in_row = i < L && static_cast<long long>(q) * L + i < t.max_comp;
                pr[h][j] = in_row ? __ldcg(&rowpairs[static_cast<size_t>(q) * L + i]) : make_uint2(0u, 0u);
            }
        }
    }
    int c2[per_bin];
#pragma unroll
    for (int i = 0; i < per_bin; ++i)
        c2[i] = static_cast<int>(__ldcg(&g2[kBins - 1 - (static_cast<int>(threadIdx.x) * per_bin + i)]));
#pragma unroll
    for (int h = 0; h < 2; ++h) cnt_w[h] = __shfl_sync(0xffffffffu, cnt_w[h], 0);
    if (lane == 0) {
        if (warp < P) offs[warp + 1] = cnt_w[0];
        if (warp + 32 < P) offs[warp + 33] = cnt_w[1];
    }
    __syncthreads();
    if (warp < 2) {                              // inclusive scan of the P <= 64 slice counts
        int v = static_cast<int>(threadIdx.x) < P ? offs[threadIdx.x + 1] : 0;
        v = warp_incl(v);
        if (threadIdx.x == 31) s_b[1] = v;
        offs[threadIdx.x + 1] = v;
        if (threadIdx.x == 0) offs[0] = 0;
    }
    __syncthreads();
    if (threadIdx.x >= 32 && threadIdx.x < 64) offs[threadIdx.x + 1] += s_b[1];
    // the 12-bit sub-bin (bits 19..8) of bin tb holding the k-th key (its syncs publish offs)
    find_bin<NT>(c2, k - above, s_a, bc);
    const uint32_t prefix = (tb << kBinShift) | (static_cast<uint32_t>(bc[0]) << 8);
    const int need = k - above - bc[1];
    const bool whole_sub_bin = need == bc[2] && prefix != 0u;   // every key of the sub-bin is in
    const int total = offs[P];
    auto slice_of = [&](int i) {                 // slice q with offs[q] <= i < offs[q + 1]
        int a = 0, b = P - 1;
        while (a < b) {
            const int mid = (a + b + 1) >> 1;
            if (offs[mid] <= i) a = mid; else b = mid - 1;
        }
        return a;
    };
    uint32_t T;
    int need_T;
    if (total <= kFinalCap) {
        // each warp places its slices' survivors at the slices' offsets
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int q = warp + 32 * h;
            if (q < P) {
                const int base = offs[q], cnt = cnt_w[h];
#pragma unroll
                for (int j = 0; j < kPairRegs; ++j) {
                    const int i = lane + 32 * j;
                    if (i < cnt) spairs[base + i] = pr[h][j];
                }
                for (int i = kPairRegs * 32 + lane; i < cnt; i += 32)
                    spairs[base + i] = __ldcg(&rowpairs[static_cast<size_t>(q) * L + i]);
            }
        }
        __syncthreads();
        auto key_at = [&](int i) { return spairs[i].x; };
        auto idx_at = [&](int i) { return static_cast<int32_t>(spairs[i].y); };
        if (whole_sub_bin) {
            // the k keys are exactly those at or above the sub-bin: no selection inside it
            T = prefix - 1u;
            need_T = 0;
        } else {
            radix_select<NT>(total, need, key_at, hist, bc, T, need_T, prefix, 32 - 8);
        }
        ordered_select<NT>(total, T, need_T, key_at, idx_at, out, s_a, s_b);
    } else {
        // degenerate score distributions (huge ties): the same steps on the slices in place
        auto at = [&](int i) {
            const int q = slice_of(i);
            return __ldcg(&rowpairs[static_cast<size_t>(q) * L + (i - offs[q])]);
        };
        auto key_at = [&](int i) { return at(i).x; };
        auto idx_at = [&](int i) { return static_cast<int32_t>(at(i).y); };
        if (whole_sub_bin) {
            T = prefix - 1u;
            need_T = 0;
        } else {
            radix_select<NT>(total, need, key_at, hist, bc, T, need_T, prefix, 32 - 8);
        }
        ordered_select<NT>(total, T, need_T, key_at, idx_at, out, s_a, s_b);
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
    b += static_cast<size_t>(rows) * kBins * 4 * 2;       // both histograms, then
    b += align_up(static_cast<size_t>(rows) * 4, 256);    // tickets (one memset clears all three)
    b += align_up(static_cast<size_t>(rows) * kMaxSlices * 4, 256);
    b += align_up(static_cast<size_t>(rows) * max_comp * 8, 256);
    return b;
}

uint32_t* topk_hist_buffer(uint8_t* ws) { return reinterpret_cast<uint32_t*>(ws); }
size_t topk_hist_bytes(int rows) { return static_cast<size_t>(rows) * (2 * kBins + 1) * 4; }
bool topk_uses_hist(int max_comp) { return max_comp > kSmallCap; }

int launch_topk(const TopkRows& t, uint8_t* ws, uint32_t* eword, cudaStream_t stream) {
    if (t.rows == 0) return DSV4_OK;
    if (t.max_comp <= kSmallCap) {
        const size_t smem = static_cast<size_t>(t.max_comp > 0 ? t.max_comp : 1) * 4;
        static bool attr_set = false;
        if (!attr_set) {
            cudaFuncSetAttribute(topk_small_kernel<kNT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kSmallCap * 4);
            attr_set = true;
        }
        count_launch();
        return launch_k(topk_small_kernel<kNT>, dim3(t.rows), dim3(kNT), smem, stream, t.pdl, t, eword)
                   == cudaSuccess ? DSV4_OK : DSV4_ERR_LAUNCH;
    }
    const LongPlan pl = long_plan(t.rows, t.max_comp);
    LongWs w;
    uint8_t* p = ws;
    w.hist = reinterpret_cast<uint32_t*>(p);
    p += static_cast<size_t>(t.rows) * kBins * 4;
    w.hist2 = reinterpret_cast<uint32_t*>(p);
    p += static_cast<size_t>(t.rows) * kBins * 4;
    w.done = reinterpret_cast<uint32_t*>(p);
    p += align_up(static_cast<size_t>(t.rows) * 4, 256);
    w.counts = reinterpret_cast<int32_t*>(p);
    p += align_up(static_cast<size_t>(t.rows) * kMaxSlices * 4, 256);
    w.pairs = reinterpret_cast<uint2*>(p);
    if (!t.hist_zeroed &&
        cudaMemsetAsync(w.hist, 0, topk_hist_bytes(t.rows), stream) != cudaSuccess)
        return DSV4_ERR_LAUNCH;
    static bool attr_set = false;
    if (!attr_set) {
        cudaFuncSetAttribute(topk_filter_kernel<kNT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kFinalCap * 8);
        attr_set = true;
    }
    dim3 grid(t.rows, pl.P);
    if (!t.hist_built) {
        count_launch();
        if (launch_k(topk_hist_kernel<kNT>, grid, dim3(kNT), 0, stream, t.pdl, t, w, pl.L, eword) != cudaSuccess)
            return DSV4_ERR_LAUNCH;
    }
    count_launch();
    return launch_k(topk_filter_kernel<kNT>, grid, dim3(kNT), size_t(kFinalCap * 8), stream, t.pdl, t, w,
                    pl.L, pl.P, eword) == cudaSuccess ? DSV4_OK : DSV4_ERR_LAUNCH;
}

}  // namespace dsv4

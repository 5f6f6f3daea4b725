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
// largest key T is found by radix selection (four 8-bit digits); `need` more copies of T are
// taken, lowest indices first; one ordered pass (block prefix sums) writes the winners in
// index order. Two implementations of the same rule:
//   * rows that fit in shared memory (max_comp <= kSmallCap): one CTA per row, keys in smem.
//   * long rows (1M context: 262,144 scores): the row is cut into P slices. A histogram
//     kernel counts the top 12 key bits per row; a filter kernel finds the 12-bit bin that
//     holds the k-th key and keeps, in index order, every element at or above that bin
//     (a few thousand of 262,144); the last CTA of the row to finish (atomic ticket, no
//     spinning) runs the exact selection on that short list.
#include "common.cuh"
#include "internal.h"

namespace dsv4 {
namespace {

constexpr int kSmallCap = 32768;     // keys held in shared memory by the one-CTA path
constexpr int kBins = 4096;          // top-12-bit histogram of the long-row path
constexpr int kBinShift = 20;
constexpr int kFinalCap = 12288;     // (key, index) pairs the finalizer keeps in smem
constexpr int kMaxSlices = 64;

// Exclusive block prefix sum of 0/1 flags; `total` receives the block total.
template <int NT>
__device__ __forceinline__ int block_excl(bool flag, int* wsum, int& total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const unsigned m = __ballot_sync(0xffffffffu, flag);
    const int pre = __popc(m & ((1u << lane) - 1u));
    if (lane == 0) wsum[warp] = __popc(m);
    __syncthreads();
    if (warp == 0) {
        int v = lane < NT / 32 ? wsum[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, v, o);
            if (lane >= o) v += t;
        }
        wsum[lane] = v;
    }
    __syncthreads();
    const int base = warp ? wsum[warp - 1] : 0;
    total = wsum[NT / 32 - 1];
    __syncthreads();
    return base + pre;
}

// Radix selection of the k-th largest key among n (1 <= k <= n). On return T is that key
// and need_T how many keys equal to T belong to the top k.
template <int NT, class KeyAt>
__device__ void radix_select(int n, int k, KeyAt key_at, uint32_t* hist, int* bc,
                             uint32_t& T, int& need_T) {
    uint32_t prefix = 0, mask = 0;
    int need = k;
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = threadIdx.x; i < 256; i += NT) hist[i] = 0;
        __syncthreads();
        for (int i = threadIdx.x; i < n; i += NT) {
            const uint32_t key = key_at(i);
            if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
        }
        __syncthreads();
        if (threadIdx.x < 32) {
            const int lane = threadIdx.x;
            uint32_t c[8], s = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) { c[i] = hist[255 - (lane * 8 + i)]; s += c[i]; }
            uint32_t inc = s;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t t = __shfl_up_sync(0xffffffffu, inc, o);
                if (lane >= o) inc += t;
            }
            const uint32_t before = inc - s;
            if (before < static_cast<uint32_t>(need) && inc >= static_cast<uint32_t>(need)) {
                uint32_t acc = before;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if (acc + c[i] >= static_cast<uint32_t>(need)) {
                        bc[0] = 255 - (lane * 8 + i);
                        bc[1] = static_cast<int>(acc);
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
        mask |= 0xFFu << shift;
        __syncthreads();
    }
    T = prefix;
    need_T = need;
}

// Write, in position order, the index of every element with key > T and of the first
// need_T elements with key == T. Stops once k indices are out.
template <int NT, class KeyAt, class IdxAt>
__device__ void ordered_compact(int n, int k, uint32_t T, int need_T, KeyAt key_at,
                                IdxAt idx_at, int32_t* out, int* wsum) {
    int ties_before = 0, written = 0;
    for (int base = 0; base < n && written < k; base += NT) {
        const int i = base + threadIdx.x;
        const uint32_t key = i < n ? key_at(i) : 0u;
        const bool tie = i < n && key == T;
        const bool gt = i < n && key > T;
        int tot_t, tot_s;
        const int tr = block_excl<NT>(tie, wsum, tot_t);
        const bool sel = gt || (tie && ties_before + tr < need_T);
        const int pos = block_excl<NT>(sel, wsum, tot_s);
        if (sel) out[written + pos] = idx_at(i);
        ties_before += tot_t;
        written += tot_s;
    }
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
    __shared__ int wsum[32];
    __shared__ int bc[2];
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
    ordered_compact<NT>(n, k, T, need_T, key_at, [](int i) { return i; }, out, wsum);
}

// ------------------------------------------------------------------ long rows
struct LongWs {
    uint32_t* hist;     // [rows, kBins]
    int32_t* counts;    // [rows, P]
    uint32_t* done;     // [rows]
    uint2* pairs;       // [rows, max_comp]: (key, index) survivors, slice p at p * L
};

__device__ __forceinline__ void slice_range(int n, int L, int p, int& lo, int& hi) {
    lo = p * L;
    hi = lo + L < n ? lo + L : n;
}

template <int NT>
__global__ void __launch_bounds__(NT)
topk_hist_kernel(TopkRows t, LongWs w, int L, uint32_t* eword) {
    __shared__ uint32_t h[kBins];
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

template <int NT>
__global__ void __launch_bounds__(NT)
topk_filter_kernel(TopkRows t, LongWs w, int L, int P, uint32_t* eword) {
    extern __shared__ uint2 spairs[];           // kFinalCap pairs (finalizer only)
    __shared__ uint32_t hist[kBins];
    __shared__ int wsum[32];
    __shared__ int bc[2];
    __shared__ int offs[kMaxSlices + 1];
    __shared__ int is_last;
    const int row = blockIdx.x, p = blockIdx.y;
    const int n = row_visible(t.n_vis, t.n_comp, t.q_pos, t.n_q, t.ratio, t.max_comp, row, eword);
    const int top_k = t.top_k;
    int32_t* out = t.idx_out + static_cast<size_t>(row) * top_k;
    if (n <= top_k) {                            // every visible entry is selected
        const int per = (top_k + P - 1) / P;
        write_all(out, n, top_k, p * per + threadIdx.x, (p + 1) * per, NT);
        return;
    }
    const int k = top_k;
    // 1. the 12-bit bin holding the k-th largest key (same answer in every CTA of the row)
    const uint32_t* g = w.hist + static_cast<size_t>(row) * kBins;
    for (int i = threadIdx.x; i < kBins; i += NT) hist[i] = g[i];
    __syncthreads();
    {
        constexpr int per = kBins / NT;          // bins per thread, taken from the top down
        uint32_t c[per], s = 0;
#pragma unroll
        for (int i = 0; i < per; ++i) { c[i] = hist[kBins - 1 - (threadIdx.x * per + i)]; s += c[i]; }
        // inclusive block scan of s in thread order
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        uint32_t inc = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t v = __shfl_up_sync(0xffffffffu, inc, o);
            if (lane >= o) inc += v;
        }
        if (lane == 31) wsum[warp] = static_cast<int>(inc);
        __syncthreads();
        if (warp == 0) {
            int v = lane < NT / 32 ? wsum[lane] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += u;
            }
            wsum[lane] = v;
        }
        __syncthreads();
        inc += warp ? static_cast<uint32_t>(wsum[warp - 1]) : 0u;
        const uint32_t before = inc - s;
        if (before < static_cast<uint32_t>(k) && inc >= static_cast<uint32_t>(k)) {
            uint32_t acc = before;
            for (int i = 0; i < per; ++i) {
                if (acc + c[i] >= static_cast<uint32_t>(k)) { bc[0] = kBins - 1 - (threadIdx.x * per + i); break; }
                acc += c[i];
            }
        }
        __syncthreads();
    }
    const uint32_t tb = static_cast<uint32_t>(bc[0]);
    __syncthreads();
    // 2. survivors of this slice (bin >= tb), in index order
    int lo, hi;
    slice_range(n, L, p, lo, hi);
    const float* s = t.scores + static_cast<size_t>(row) * t.max_comp;
    uint2* seg = w.pairs + static_cast<size_t>(row) * t.max_comp + static_cast<size_t>(p) * L;
    int cnt = 0;
    for (int base = lo; base < hi; base += NT) {
        const int i = base + threadIdx.x;
        const uint32_t key = i < hi ? float_to_key(s[i]) : 0u;
        const bool keep = i < hi && (key >> kBinShift) >= tb;
        int tot;
        const int pos = block_excl<NT>(keep, wsum, tot);
        if (keep) seg[cnt + pos] = make_uint2(key, static_cast<uint32_t>(i));
        cnt += tot;
    }
    if (threadIdx.x == 0) w.counts[static_cast<size_t>(row) * P + p] = cnt;
    // 3. the last CTA of the row to get here finishes the row (no waiting on anyone)
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned ticket = atomicAdd(&w.done[row], 1u);
        is_last = ticket == static_cast<unsigned>(P - 1);
    }
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    if (threadIdx.x == 0) {
        int acc = 0;
        for (int q = 0; q < P; ++q) {
            offs[q] = acc;
            acc += __ldcg(&w.counts[static_cast<size_t>(row) * P + q]);
        }
        offs[P] = acc;
        w.done[row] = 0;                         // ready for the next call
    }
    __syncthreads();
    const int total = offs[P];
    const uint2* rowpairs = w.pairs + static_cast<size_t>(row) * t.max_comp;
    for (int j = k + threadIdx.x; j < top_k; j += NT) out[j] = -1;
    uint32_t T;
    int need_T;
    if (total <= kFinalCap) {
        for (int q = 0; q < P; ++q) {
            const int c = offs[q + 1] - offs[q];
            for (int i = threadIdx.x; i < c; i += NT)
                spairs[offs[q] + i] = __ldcg(&rowpairs[static_cast<size_t>(q) * L + i]);
        }
        __syncthreads();
        auto key_at = [&](int i) { return spairs[i].x; };
        auto idx_at = [&](int i) { return static_cast<int32_t>(spairs[i].y); };
        radix_select<NT>(total, k, key_at, hist, bc, T, need_T);
        ordered_compact<NT>(total, k, T, need_T, key_at, idx_at, out, wsum);
    } else {
        // degenerate score distributions (huge ties): the same steps on the slices in place
        auto at = [&](int i) {
            int q = 0;
            while (q + 1 < P && offs[q + 1] <= i) ++q;
            return __ldcg(&rowpairs[static_cast<size_t>(q) * L + (i - offs[q])]);
        };
        auto key_at = [&](int i) { return at(i).x; };
        auto idx_at = [&](int i) { return static_cast<int32_t>(at(i).y); };
        radix_select<NT>(total, k, key_at, hist, bc, T, need_T);
        ordered_compact<NT>(total, k, T, need_T, key_at, idx_at, out, wsum);
    }
}

constexpr int kNT = 512;

struct LongPlan { int P, L; };

LongPlan long_plan(int rows, int max_comp) {
    int P = (2 * 148 + rows - 1) / (rows > 0 ? rows : 1);
    if (P < 1) P = 1;
    if (P > kMaxSlices) P = kMaxSlices;
    int L = (max_comp + P - 1) / P;
    L = (L + 255) / 256 * 256;
    if (L < 1024) L = 1024;
    P = (max_comp + L - 1) / L;
    if (P < 1) P = 1;
    return {P, L};
}

}  // namespace

size_t topk_ws_bytes(int rows, int max_comp, int top_k) {
    (void)top_k;
    if (max_comp <= kSmallCap) return 0;
    const LongPlan pl = long_plan(rows, max_comp);
    size_t b = 0;
    b += align_up(static_cast<size_t>(rows) * kBins * 4, 256);
    b += align_up(static_cast<size_t>(rows) * pl.P * 4, 256);
    b += align_up(static_cast<size_t>(rows) * 4, 256);
    b += align_up(static_cast<size_t>(rows) * max_comp * 8, 256);
    return b;
}

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
        topk_small_kernel<kNT><<<t.rows, kNT, smem, stream>>>(t, eword);
        count_launch();
        return cudaGetLastError() == cudaSuccess ? DSV4_OK : DSV4_ERR_LAUNCH;
    }
    const LongPlan pl = long_plan(t.rows, t.max_comp);
    LongWs w;
    uint8_t* p = ws;
    w.hist = reinterpret_cast<uint32_t*>(p);
    p += align_up(static_cast<size_t>(t.rows) * kBins * 4, 256);
    w.counts = reinterpret_cast<int32_t*>(p);
    p += align_up(static_cast<size_t>(t.rows) * pl.P * 4, 256);
    w.done = reinterpret_cast<uint32_t*>(p);
    p += align_up(static_cast<size_t>(t.rows) * 4, 256);
    w.pairs = reinterpret_cast<uint2*>(p);
    if (cudaMemsetAsync(w.hist, 0, static_cast<size_t>(t.rows) * kBins * 4, stream) != cudaSuccess ||
        cudaMemsetAsync(w.done, 0, static_cast<size_t>(t.rows) * 4, stream) != cudaSuccess)
        return DSV4_ERR_LAUNCH;
    static bool attr_set = false;
    if (!attr_set) {
        cudaFuncSetAttribute(topk_filter_kernel<kNT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kFinalCap * 8);
        attr_set = true;
    }
    dim3 grid(t.rows, pl.P);
    topk_hist_kernel<kNT><<<grid, kNT, 0, stream>>>(t, w, pl.L, eword);
    topk_filter_kernel<kNT><<<grid, kNT, kFinalCap * 8, stream>>>(t, w, pl.L, pl.P, eword);
    count_launch(2);
    return cudaGetLastError() == cudaSuccess ? DSV4_OK : DSV4_ERR_LAUNCH;
}

}  // namespace dsv4

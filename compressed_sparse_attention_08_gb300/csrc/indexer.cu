// Lightning-indexer scoring on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
//   I[row, j] = sum_h w[row, h] * ReLU( q[row, h, :] . keys[b, j, :] )      row = b * n_q + t
//
// Sources: "nvfp4-megamoe-kernel: compare v0.1-e2e-working...v-c1-c2-c3-20260602",
// ARCHITECTURE_AND_MEMORY_AUDIT.md "F1" (one 128-wide compressed key per block, shared by
// all indexer heads: MQA) and "F3" (the scoring formula, fp32, no scale); PERFORMANCE_AUDIT.md
// "P6" (the fp32 einsum on CUDA cores is the wall at long context).
//
// Why tensor cores: every 256-byte key meets 64 heads x 128 dims = 16,384 flops, 64 flop per
// byte. Streaming keys at HBM speed needs ~430 TFLOP/s, far above the CUDA-core fp32 rate,
// so the contraction runs as a UMMA with the keys as the A operand:
//     D[128 keys x N heads] (fp32, TMEM) = K_tile[128 x 128] . Q^T[128 x N]
// Each row of D is one key's per-head dot products, so the epilogue thread that owns TMEM
// lane i reduces sum_h w_h ReLU(D[i, h]) alone, with no cross-thread reduction.
//
// CTA = 6 warps (bf16 keys, one query row per MMA), 10 or 18 (two or four query rows per MMA)
// or 14 (FP8 keys), persistent, one per SM, warp-specialised:
//   warp 0  TMA producer: key stages of 256 keys (two 128-key MMA tiles; two 128-byte-
//           swizzled boxes of 64 dims x 256 rows) into a ring of kStages 64 KB buffers; the
//           row's queries (N x 128) into the query buffer
//   warp 1  MMA issuer (one thread) and TMEM owner: per tile 8 UMMAs (K = 16 each) into one
//           of the tile accumulators of a stage slot in TMEM (two slots); one tcgen05.commit
//           publishes the stage's accumulators, another frees the stage once they are done
//   warps 2-5  epilogue: tcgen05.ld of the accumulator (thread = key), weighted ReLU sum in
//           fp32, coalesced store of the score; optionally a shared-memory histogram of the
//           scores' top 12 key bits, flushed per row into the top-k workspace (so the
//           long-row top-k needs no histogram pass of its own). FP8 keys: warps 2-13, three
//           groups of four taking the accumulators in turn; a 64 KB stage holds 512 keys, and
//           one group alone could not drain four tiles in the time the stage takes to arrive
//           (two groups scored the 1M-key rows in 38.7 us, three in 35.4, four, whose threads
//           get too few registers, in 37.0). Several query rows per MMA: one group of four
//           warps per query row, every group reading every tile.
// Why 64 KB stages: a stage stays busy from its copy until the MMA that reads it completes,
// and that hand-off adds a few hundred ns per stage; with 32 KB stages the cost took about a
// sixth of the bandwidth, with 64 KB stages it is hidden. Shared memory then holds one query
// buffer, which is all a CTA needs when it scores a single row (decode).
// Many query rows of bf16 keys (prefill, no histogram): each MMA scores a 128-key tile against
// two or four consecutive query rows of a sequence (UMMA N = 128 or 256), one epilogue group
// of four warps per query row. The keys then come from L2 (the sequence's whole cache is
// re-read per query unit), and a tcgen05.mma costs its issuing thread about the same at any
// N, so four rows per MMA halve both the key reads and the MMA instructions per score; their
// 256-column accumulators fill TMEM with two slots, and the stage shrinks to one 32 KB tile
// in a ring of four so that the four 16 KB query buffers fit.
// Launched with programmatic dependent launch: the producer waits for the preceding kernel
// (the compressor) only before a stage that holds key rows that kernel writes.
// Work: with no more rows than CTAs, every row has its own set of CTAs (every rows-th one) taking the row's
// stages in turn; with at most 48 rows (decode) only the first nine tenths of each row
// are shared out that way and the rest is claimed one stage at a time from a counter in
// the workspace header, because the SMs do not stream equally fast (a static share left the
// slowest CTA about 3 us behind the median at 1M keys per row). Otherwise each CTA takes a
// contiguous range of (row, stage) pairs. The producer hands every stage's (row, stage) to
// the MMA warp and the epilogue through a small ring of ids in shared memory, an id of -1
// ending the stream; tiles past the row's visible count are skipped.
#include "common.cuh"
#include "internal.h"

#include <cudaTypedefs.h>

namespace dsv4 {
namespace {

constexpr int kTileKeys = 128;              // UMMA M
constexpr int kDim = 128;                   // key width = UMMA K total
constexpr int kMaxHeads = 64;               // UMMA N upper bound per query
constexpr int kAccCols = 64;                // TMEM columns per accumulator and query
constexpr uint32_t kQBufBytes = kMaxHeads * kDim * 2;      // 16 KiB (bf16 queries) per query

// Key format and stage geometry. bf16 keys: two bytes per element, a 256-byte key split over two
// 64-dim boxes; FP8 E4M3: one byte, a key is one 128-byte row, the two boxes hold consecutive
// keys. A stage is two TMA boxes, 64 KiB (256 bf16 or 512 FP8 keys: 2 or 4 MMA tiles) in a
// ring of three, except with four query rows per MMA (bf16, UMMA N = 256): then a tile's
// accumulator takes 256 TMEM columns, two stage slots of one tile fill the 512, and a stage is
// one 128-key tile of 32 KiB in a ring of four. One MMA step consumes 32 bytes of K.
template <bool FP8, int QB = 1>
struct KeyFmt {
    static constexpr int kElem = FP8 ? 1 : 2;
    static constexpr bool kQuad = !FP8 && QB == 4;
    static constexpr uint32_t kStageBytes = kQuad ? 32u * 1024u : 64u * 1024u;
    static constexpr int kStages = kQuad ? 4 : 3;
    static constexpr uint32_t kBoxBytes = kStageBytes / 2;
    static constexpr int kStageKeys = static_cast<int>(kStageBytes) / (kDim * kElem);
    static constexpr int kBoxRows = FP8 ? kStageKeys / 2 : kStageKeys;   // rows of one TMA box
    static constexpr int kSub = kStageKeys / kTileKeys;
    static constexpr int kKSteps = kDim * kElem / 32;
    static constexpr int kBoxInner = 128 / kElem;          // elements per 128-byte box row
    // TMEM accumulators: two stage slots of kSub tiles each, so the MMAs of a stage wait only
    // for the epilogue of the stage two back
    static constexpr int kAccBufs = 2 * kSub;
    static constexpr size_t kSmem = 1024 + kStages * static_cast<size_t>(kStageBytes) + QB * kQBufBytes;
    static_assert(kSmem <= 227u * 1024u, "shared memory per CTA");
};
constexpr int kHistBins = 4096;             // top 12 bits of the order-preserving score key
constexpr int kIdRing = 8;                  // stage ids in flight from the producer
// stage-claim counters: words [kClaimWord, kClaimWord + rows) of the zeroed workspace header
constexpr int kClaimWord = 16;
constexpr int kMaxClaimRows = 48;

struct ScoreParams {
    const float* w;          // [rows, heads]
    const int32_t* n_comp;   // [batch]
    const int64_t* q_pos;    // [rows] or null
    float* scores;           // [rows, max_comp]
    uint32_t* hist;          // [rows, 4096] top-12-bit key histogram (zeroed), or null
    const int32_t* fresh_row0;  // [batch] first key row the preceding kernel writes, or null
    int fresh_rows;          // rows it writes per sequence (0: none)
    uint32_t* eword;
    const float* q_scale;    // FP8 keys: [rows, heads] query scales, else null
    const float* key_scale;  // FP8 keys: [batch, max_comp] key scales, else null
    uint32_t* claim;         // [rows] zeroed stage-claim counters, or null (static shares only)
    int reuse_keys;          // many rows share the keys (prefill): keep them in L2, stream the scores
    int rows, n_q, heads, max_comp, ratio, stages_per_row;
    // the walk's units: QB consecutive query rows of one sequence (QB = 1: a unit is a row)
    int units, gpb;          // units in all, units per sequence (ceil(n_q / QB))
    int fault;               // test control: the first key stage of each CTA is not loaded
    unsigned long long wait_ns;   // limit of each bounded wait
};

// The stages one CTA scores, as positions f = row * stages_per_row + stage: f = begin,
// begin + step, ... < end. With no more rows than CTAs, every row gets its own set of CTAs
// (every rows-th CTA) and they take the row's stages in turn (CTA i of n: stages i, i + n,
// ...), so a CTA keeps
// one query for the whole kernel and a row's last stage (the one the compressor may have just
// written) comes last. With more rows than CTAs (prefill), each CTA takes a contiguous range.
// Positions are 32-bit (rows x stages stays far below 2^31) and the producer steps through
// them without dividing: at kernel start its one thread spent ~1.5 us on 64-bit divisions
// before the first key copy.
struct Walk { int begin, end, step; };

__device__ __forceinline__ Walk cta_walk(int rows, int per_row) {
    const int g = static_cast<int>(gridDim.x), c = static_cast<int>(blockIdx.x);
    if (rows > g) {
        const long long total = static_cast<long long>(rows) * per_row;
        return {static_cast<int>(total * c / g), static_cast<int>(total * (c + 1) / g), 1};
    }
    // the rows interleaved over the CTAs (CTA c takes row c mod rows): consecutive CTAs land on
    // neighbouring SMs, and a row given a block of them finished up to ~1.3 us after the others
    const int r = c % rows, n_in_row = (g - r + rows - 1) / rows;
    return {r * per_row + c / rows, (r + 1) * per_row, n_in_row};
}

// NP: the heads padded to a multiple of 16 (the TMEM columns of one query's heads)
// EG: epilogue groups of four warps (threads 64 + 128 EG)
// QB: query rows scored per MMA (UMMA N = QB * NP): with QB = 2 or 4 (many rows of bf16 keys,
//     prefill) each key stage serves two or four queries, a half or a quarter of the key
//     traffic and of the MMA instructions per score
template <bool FP8, int NP, int EG, int QB>
__global__ void __launch_bounds__(64 + 128 * EG, 1)
index_score_kernel(const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap qmap, ScoreParams p) {
    using F = KeyFmt<FP8, QB>;
    constexpr int kStages = F::kStages;
    constexpr uint32_t kStageBytes = F::kStageBytes, kBoxBytes = F::kBoxBytes;
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint64_t full_bar[kStages], empty_bar[kStages];
    __shared__ uint64_t tfull_bar[2], tempty_bar[2];    // per accumulator slot (one stage)
    __shared__ uint64_t qfull_bar, qempty_bar, done_bar, epi_bar;
    __shared__ uint64_t idfull_bar[kIdRing], idempty_bar[kIdRing];
    __shared__ int2 s_id[kIdRing];                  // (row, stage) of each stage handed over
    __shared__ uint32_t tmem_slot;
    __shared__ volatile int abort_flag;
    // top-12-bit key histogram of the current row, two 16-bit counts per word (8 KB: a
    // compressor CTA still fits beside this CTA on its SM)
    // (none with QB > 1: those launches build no histogram, and the queries need the room)
    __shared__ uint32_t s_hist[QB == 1 ? kHistBins / 2 : 1];

    constexpr int kStageKeys = F::kStageKeys, kSub = F::kSub;
    constexpr int kEpiGroups = EG, kThreads = 64 + 128 * EG, kAccBufs = F::kAccBufs;
    // one epilogue group per query of the unit (QB queries per MMA): every group reads every
    // accumulator, group g its query g's columns, so a tile's queries drain at once
    constexpr bool kSplitQ = QB > 1 && EG == QB && !FP8;
    constexpr int kWq = kSplitQ ? 1 : QB;              // queries whose weights a thread holds
    constexpr int kAccColsQ = kAccCols * QB;                 // TMEM columns per accumulator
    constexpr uint32_t kTmemCols = static_cast<uint32_t>(kAccBufs * kAccColsQ);   // 256 or 512
    static_assert(!(FP8 && QB > 1) && kTmemCols <= 512, "scorer shape");
    constexpr int kFlushStages = 65535 / kStageKeys;   // a 16-bit bin count cannot overflow
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_trigger();
    // 1024-byte aligned operand buffers (the 128-byte swizzle repeats every 1024 bytes)
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* base = smem_raw + ((1024u - (raw & 1023u)) & 1023u);
    uint8_t* key_buf = base;
    uint8_t* q_buf = base + kStages * kStageBytes;

    if (threadIdx.x == 0) {
        for (int i = 0; i < kStages; ++i) { mbar_init(&full_bar[i], 1); mbar_init(&empty_bar[i], 1); }
        for (int i = 0; i < 2; ++i) {
            // every tile of the slot is released by the 128 threads of the group that drains it
            // (with split queries: of every group), whether or not the tile held visible keys
            mbar_init(&tfull_bar[i], 1);
            mbar_init(&tempty_bar[i], kSub * (kSplitQ ? 128 * kEpiGroups : 128));
        }
        mbar_init(&qfull_bar, 1);
        mbar_init(&qempty_bar, 1);
        mbar_init(&done_bar, 1);
        mbar_init(&epi_bar, 128 * kEpiGroups);
        for (int i = 0; i < kIdRing; ++i) { mbar_init(&idfull_bar[i], 1); mbar_init(&idempty_bar[i], 4 * kEpiGroups); }
        abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&kmap);
        tma_prefetch_desc(&qmap);
    }
    // query rows past `heads` stay zero for the whole kernel (TMA writes only `heads` rows)
    for (uint32_t i = threadIdx.x; i < kQBufBytes * QB / 16; i += kThreads)
        reinterpret_cast<uint4*>(q_buf)[i] = make_uint4(0, 0, 0, 0);
    for (int i = threadIdx.x; i < (QB == 1 ? kHistBins / 2 : 1); i += kThreads) s_hist[i] = 0;
    if (warp == 1) tmem_alloc(&tmem_slot, kTmemCols);
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = tmem_slot;

    const Walk wk = cta_walk(p.units, p.stages_per_row);
    const int spr = p.stages_per_row;
    const uint32_t idesc = FP8 ? idesc_e4m3_f32(kTileKeys, NP * QB) : idesc_bf16_f32(kTileKeys, NP * QB);
    const uint32_t q_half = static_cast<uint32_t>(NP * QB) * 128u;   // bf16: bytes of one 64-dim half
    // unit u: sequence u / gpb, query rows b * n_q + t0 + q for q < QB with t0 + q < n_q
    auto unit_row = [&](int u, int q) { return (u / p.gpb) * p.n_q + (u % p.gpb) * QB + q; };
    auto unit_nq = [&](int u) { const int t0 = (u % p.gpb) * QB; return min(QB, p.n_q - t0); };
    // a unit sees the keys of its last query (visibility grows with the position)
    auto unit_visible = [&](int u) {
        return row_visible(nullptr, p.n_comp, p.q_pos, p.n_q, p.ratio, p.max_comp,
                           unit_row(u, unit_nq(u) - 1), nullptr);
    };

    if (warp == 0) {
        if (lane == 0) {
            // Stage order: the CTA's share of the walk; for a row with its own set of CTAs
            // and a claim counter, only the first nine tenths of the row are shared out in
            // advance and the rest is claimed one stage at a time, so that CTAs on SMs that
            // stream faster take more and the row's CTAs finish together.
            // (claiming pays only when the row has more stages than CTAs; with at most one
            // stage each, a static share lets every CTA start before the preceding kernel ends,
            // which the first claim, on counters that kernel clears, would wait for)
            const bool dyn = p.claim != nullptr && wk.step > 1 && spr > wk.step;
            const int row0 = wk.begin / spr;
            const int cutoff = dyn ? (spr * 9 / 10) / wk.step * wk.step : spr;
            int stage = 0, qcount = 0, cur_row = -1, cur_b = 0, vis_row = -1, nv = 0, ahead = -1;
            bool waited = false, claiming = false;
            long long issued = 0, seq = 0;
            int f = wk.begin, f_row = row0, f_st = wk.begin - row0 * spr;   // position f = (f_row, f_st)
            uint32_t phase = 0;
            // decode: every key is read once (evict first); prefill: every query row re-reads
            // the same keys (evict last), while its scores stream past them
            const uint64_t stream_policy = p.reuse_keys ? l2_evict_last_policy() : l2_evict_first_policy();
            auto claim = [&]() {
                // the counters are cleared by the work before this grid
                if (!waited) { pdl_wait(); waited = true; }
                ahead = static_cast<int>(atomicAdd(&p.claim[row0], 1u));
            };
            for (;;) {
                int row, st;
                if (!claiming) {
                    if (f >= wk.end || f_st >= cutoff) {
                        if (!dyn) break;
                        claiming = true;
                        continue;
                    }
                    row = f_row;
                    st = f_st;
                    f += wk.step;
                    for (f_st += wk.step; f_st >= spr; f_st -= spr) ++f_row;
                    // before the last stage of the share: the first claim's round trip hides
                    // behind it
                    if (dyn && ahead < 0 && (f >= wk.end || f_st >= cutoff)) claim();
                } else {
                    if (ahead < 0) claim();
                    row = row0;
                    st = cutoff + ahead;
                    if (row != vis_row) {
                        nv = unit_visible(row);
                        vis_row = row;
                    }
                    if (st >= spr || st * kStageKeys >= nv) break;     // the row is all taken
                    claim();                                            // the next one, early
                }
                // The walk's first kStages stages are handed over before the row's visible count
                // is known: that load took ~1.7 us at kernel start, and the first key copy waited
                // for it. (A stage past the visible keys costs its copy; the MMA warp and the
                // epilogue skip its tiles.)
                if (issued >= kStages) {
                    if (row != vis_row) {
                        nv = unit_visible(row);
                        vis_row = row;
                    }
                    if (st * kStageKeys >= nv) continue;
                }
                {
                    // hand the stage to the MMA warp and the epilogue
                    const int slot = static_cast<int>(seq % kIdRing);
                    if (!mbar_wait(&idempty_bar[slot], static_cast<uint32_t>(((seq / kIdRing) & 1) ^ 1), &abort_flag, p.wait_ns))
                        goto fail0;
                    s_id[slot] = make_int2(row, st);
                    mbar_arrive(&idfull_bar[slot]);
                    ++seq;
                }
                if (row != cur_row) {
                    // one query buffer: the MMA warp learns of the new row from the stage id
                    // just handed over and releases the old queries once their MMAs are done
                    if (!mbar_wait(&qempty_bar, (qcount & 1) ^ 1, &abort_flag, p.wait_ns)) goto fail0;
                    const int nqu = unit_nq(row);
                    mbar_arrive_expect_tx(&qfull_bar, static_cast<uint32_t>(nqu * p.heads) * kDim * F::kElem);
                    for (int q = 0; q < nqu; ++q) {
                        // query q's heads at rows [q * NP, q * NP + heads) of the B operand
                        const int qr = unit_row(row, q) * p.heads;
                        tma_load_2d(q_buf + q * NP * 128, &qmap, &qfull_bar, 0, qr);
                        if (!FP8) tma_load_2d(q_buf + q_half + q * NP * 128, &qmap, &qfull_bar, 64, qr);
                    }
                    cur_row = row;
                    cur_b = row / p.gpb;
                    ++qcount;
                }
                if (!waited && p.fresh_rows > 0) {
                    // key rows written by the preceding kernel (the newest block's key): wait
                    // for it before streaming a stage that overlaps them
                    const int f0 = p.fresh_row0 ? p.fresh_row0[cur_b] : 0;
                    if (st * kStageKeys < f0 + p.fresh_rows && f0 < (st + 1) * kStageKeys) {
                        pdl_wait();
                        waited = true;
                    }
                }
                if (p.fault && issued == 0) {
                    // test control: this stage's copy is never issued, so the MMA warp's wait for
                    // it runs out; wait (bounded) until that warp has given up, then wind down
                    const uint64_t t0 = global_timer_ns();
                    while (!abort_flag && global_timer_ns() - t0 < 4 * p.wait_ns) {
                    }
                    goto fail0;
                }
                if (!mbar_wait(&empty_bar[stage], phase ^ 1, &abort_flag, p.wait_ns)) goto fail0;
                mbar_arrive_expect_tx(&full_bar[stage], kStageBytes);
                {
                    uint8_t* kd = key_buf + stage * kStageBytes;
                    // bf16: the two 64-dim halves of the stage's keys; FP8: two runs of 256 whole keys
                    tma_load_3d_hint(kd, &kmap, &full_bar[stage], 0, st * kStageKeys, cur_b, stream_policy);
                    tma_load_3d_hint(kd + kBoxBytes, &kmap, &full_bar[stage], FP8 ? 0 : 64,
                                     st * kStageKeys + (FP8 ? F::kBoxRows : 0), cur_b, stream_policy);
                    ++issued;
                }
                if (++stage == kStages) { stage = 0; phase ^= 1; }
            }
            {
                // end of the stream
                const int slot = static_cast<int>(seq % kIdRing);
                if (!mbar_wait(&idempty_bar[slot], static_cast<uint32_t>(((seq / kIdRing) & 1) ^ 1), &abort_flag, p.wait_ns))
                    goto fail0;
                s_id[slot] = make_int2(-1, -1);
                mbar_arrive(&idfull_bar[slot]);
            }
            if (!waited) pdl_wait();        // this grid never completes before its predecessor
            goto done0;
        fail0:
            flag_error(p.eword, DSV4_EWORD_TIMEOUT);
            abort_flag = 1;
            // let the copies this thread started land before the CTA can exit (bounded)
            for (long long i = issued > kStages ? issued - kStages : 0; i < issued; ++i)
                mbar_wait(&full_bar[i % kStages], static_cast<uint32_t>((i / kStages) & 1), nullptr, 100000000ull);
            if (qcount > 0)
                mbar_wait(&qfull_bar, static_cast<uint32_t>((qcount - 1) & 1), nullptr, 100000000ull);
            if (!waited) pdl_wait();
        done0:;
        }
    } else if (warp == 1) {
        if (lane == 0) {
            int stage = 0, qcount = 0, cur_row = -1, nv = 0;
            uint32_t phase = 0;
            for (long long seq = 0;; ++seq) {
                const int slot = static_cast<int>(seq % kIdRing);
                if (!mbar_wait(&idfull_bar[slot], static_cast<uint32_t>((seq / kIdRing) & 1), &abort_flag, p.wait_ns)) goto fail1;
                const int2 id = s_id[slot];
                if (id.x < 0) break;
                const int row = id.x, st = id.y;
                if (row != cur_row) {
                    if (cur_row >= 0) umma_commit(&qempty_bar);   // old queries free once done
                    nv = unit_visible(row);      // (its load overlaps the wait for the queries)
                    if (!mbar_wait(&qfull_bar, qcount & 1, &abort_flag, p.wait_ns)) goto fail1;
                    cur_row = row;
                    ++qcount;
                }
                if (!mbar_wait(&full_bar[stage], phase, &abort_flag, p.wait_ns)) goto fail1;
                {
                    // the stage's tiles go to accumulator slot seq & 1 once the epilogue has read
                    // out what the stage two back left there; one commit publishes them all
                    // (a wait and a commit per tile kept this thread, not the keys, the bound)
                    const int as = static_cast<int>(seq & 1);
                    if (!mbar_wait(&tempty_bar[as], static_cast<uint32_t>(((seq >> 1) & 1) ^ 1), &abort_flag, p.wait_ns))
                        goto fail1;
                    tc_fence_after();
                    const uint32_t a_stage = smem_u32(key_buf + stage * kStageBytes);
                    const uint32_t b0 = smem_u32(q_buf);
                    for (int j = 0; j < kSub; ++j) {
                        if ((st * kSub + j) * kTileKeys >= nv) break;   // tile past the visible keys
                        const uint32_t d = tmem_base + static_cast<uint32_t>((as * kSub + j) * kAccColsQ);
                        const uint32_t a0 = a_stage + static_cast<uint32_t>(j * kTileKeys * 128);
#pragma unroll
                        for (int k = 0; k < F::kKSteps; ++k) {
                            // 32 bytes of K per step; a bf16 key continues in the second box
                            const uint32_t ka = FP8 ? k * 32u : (k >> 2) * kBoxBytes + (k & 3) * 32u;
                            const uint32_t kb = FP8 ? k * 32u : (k >> 2) * q_half + (k & 3) * 32u;
                            const uint64_t ad = sdesc_kmajor_sw128(a0 + ka);
                            const uint64_t bd = sdesc_kmajor_sw128(b0 + kb);
                            if constexpr (FP8) umma_f8(d, ad, bd, idesc, k > 0 ? 1u : 0u);
                            else umma_bf16(d, ad, bd, idesc, k > 0 ? 1u : 0u);
                        }
                    }
                    umma_commit(&tfull_bar[as]);
                }
                umma_commit(&empty_bar[stage]);
                if (++stage == kStages) { stage = 0; phase ^= 1; }
            }
            goto done1;
        fail1:
            flag_error(p.eword, DSV4_EWORD_TIMEOUT);
            abort_flag = 1;
        done1:
            // every MMA issued by this thread has completed before TMEM is released
            umma_commit(&done_bar);
            if (!mbar_wait(&done_bar, 0, nullptr)) flag_error(p.eword, DSV4_EWORD_TIMEOUT);
        }
        __syncwarp();
    } else {
        // epilogue: kEpiGroups groups of 4 warps; warp -> TMEM lane quarter (warp % 4); group g
        // drains tile j of the stage with sequence number n when (n * kSub + j) % kEpiGroups == g,
        // so with several groups as many tiles drain at once (FP8: four tiles per stage, twice
        // the keys per byte of bf16)
        const int quarter = warp & 3;
        const int group = (warp - 2) >> 2;
        const int lrow = quarter * 32 + lane;
        const int etid = threadIdx.x - 64;                 // 0 .. 128 * kEpiGroups - 1
        const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
        int cur_row = -1, nv = 0;
        uint32_t fl_parity = 0;
        bool ok = true;
        // The unit's head weights (FP8: times the head's query scale). FP8 keys: three groups
        // of 448 threads leave a thread ~144 registers, too few for 64 weights beside the 64
        // accumulator columns it loads, so each warp keeps its copy in the half of the query
        // buffer that FP8 queries leave free and reads it as broadcast 16-byte loads. bf16 keys
        // keep them in registers: with four queries per MMA the broadcast loads (a wavefront per
        // 4 bytes) took more of the shared-memory data pipe than the tensor core's operand reads,
        // so those threads hold their query's 64 weights and read the accumulator 16 columns at
        // a time instead (112 registers a thread at 576 threads).
        constexpr bool kWSmem = FP8;
        constexpr bool kChunked = F::kQuad;
        static_assert(!kWSmem || 4 * kEpiGroups * NP * 4 <= static_cast<int>(kQBufBytes) / 2, "weight slots");
        float wv[kWSmem ? 1 : kWq][kWSmem ? 1 : NP];
        float* s_wv = reinterpret_cast<float*>(q_buf + kQBufBytes / 2) + (warp - 2) * NP;
        int nvq[kWq];             // keys visible to each query of the unit
        float* srow[kWq];         // each query's score row (set once per unit: no division per tile)
        const int q_lo = kSplitQ ? group : 0;      // this thread's queries: q_lo .. q_lo + kWq - 1
        int nqu = 1;              // queries in the unit
        // Every wait of the epilogue is an mbarrier wait, bounded in time and ended early once
        // any role has given up, so a failure anywhere cannot leave a thread waiting.
        auto epi_sync = [&]() -> bool {
            mbar_arrive(&epi_bar);
            const bool r = mbar_wait(&epi_bar, fl_parity, &abort_flag, p.wait_ns);
            fl_parity ^= 1;
            return r;
        };
        // The histogram is private to the CTA and flushed to the row's global histogram when
        // the row changes, and before a 16-bit count could overflow (every kFlushStages stages).
        int since_flush = 0;
        auto flush = [&](int r) {
            pdl_wait();      // the histogram may have been cleared by the preceding kernel
            if (epi_sync()) {
                uint32_t* g = p.hist + static_cast<size_t>(r) * kHistBins;
                for (int i = etid; i < (QB == 1 ? kHistBins / 2 : 0); i += 128 * kEpiGroups) {
                    const uint32_t v = s_hist[i];
                    if (v) {
                        if (v & 0xFFFFu) atomicAdd(&g[2 * i], v & 0xFFFFu);
                        if (v >> 16) atomicAdd(&g[2 * i + 1], v >> 16);
                        s_hist[i] = 0;
                    }
                }
                epi_sync();
            }
            since_flush = 0;
        };
        // the next stage's id, read one stage ahead; each warp releases the slot once read
        auto read_id = [&](long long sq, int2& id) -> bool {
            const int slot = static_cast<int>(sq % kIdRing);
            if (!mbar_wait(&idfull_bar[slot], static_cast<uint32_t>((sq / kIdRing) & 1), &abort_flag, p.wait_ns)) return false;
            const volatile int* v = reinterpret_cast<const volatile int*>(&s_id[slot]);
            id = make_int2(v[0], v[1]);
            __syncwarp();
            if (lane == 0) mbar_arrive(&idempty_bar[slot]);
            return true;
        };
        // FP8: the key scales of a stage load while the stage before it is scored (a DRAM read
        // per tile would otherwise stall the epilogue once per 128 keys). Every key scale is
        // final once the preceding kernel (which may write the newest key) has completed.
        float ks_cur[kSub], ks_next[kSub];
        int ks_row = -1;
        const float* kb = nullptr;      // the key scales of sequence ks_row / gpb
        auto load_ks = [&](int2 id) {
            if (id.x != ks_row) {
                ks_row = id.x;
                kb = p.key_scale + static_cast<size_t>(id.x / p.gpb) * p.max_comp;
            }
#pragma unroll
            for (int j = 0; j < kSub; ++j) {
                const int key = (id.y * kSub + j) * kTileKeys + lrow;
                ks_next[j] = key < p.max_comp ? __ldcg(kb + key) : 0.f;
            }
        };
        int2 id_cur = make_int2(-1, -1), id_next;
        ok = read_id(0, id_cur);
        if constexpr (FP8) {
            pdl_wait();
            if (ok && id_cur.x >= 0) load_ks(id_cur);
        }
        for (long long sq = 1; ok && id_cur.x >= 0; ++sq) {
            id_next = make_int2(-1, -1);
            if (!read_id(sq, id_next)) ok = false;
            if constexpr (FP8) {
#pragma unroll
                for (int j = 0; j < kSub; ++j) ks_cur[j] = ks_next[j];
                if (ok && id_next.x >= 0) load_ks(id_next);
            }
            const int row = id_cur.x, st = id_cur.y;
            if (row != cur_row || since_flush == kFlushStages) {
                if (p.hist && cur_row >= 0) flush(cur_row);
            }
            ++since_flush;
            if (row != cur_row) {
                nv = unit_visible(row);
                cur_row = row;
                nqu = unit_nq(row);
#pragma unroll
                for (int qi = 0; qi < kWq; ++qi) {
                    const int q = q_lo + qi;
                    const int qrow = unit_row(row, q < nqu ? q : 0);
                    nvq[qi] = QB == 1 ? nv : row_visible(nullptr, p.n_comp, p.q_pos, p.n_q, p.ratio, p.max_comp, qrow, nullptr);
                    srow[qi] = p.scores + static_cast<size_t>(qrow) * p.max_comp;
                    if constexpr (kWSmem) {
                        // FP8: the query scale folds into the head's weight (ReLU commutes with it)
                        __syncwarp();
                        for (int h = lane; h < NP; h += 32) {
                            const size_t o = static_cast<size_t>(qrow) * p.heads + h;
                            s_wv[h] = h < p.heads ? __ldg(&p.w[o]) * __ldg(&p.q_scale[o]) : 0.f;
                        }
                        __syncwarp();
                    } else {
#pragma unroll
                        for (int h = 0; h < NP; ++h) {
                            const size_t o = static_cast<size_t>(qrow) * p.heads + h;
                            wv[kWSmem ? 0 : qi][kWSmem ? 0 : h] = h < p.heads ? __ldg(&p.w[o]) : 0.f;
                        }
                    }
                }
            }
            // the stage's accumulator slot and the parity of this use of it
            const int sn = static_cast<int>(sq - 1);
            const int as = sn & 1;
            bool published = false;
            for (int j = 0; j < kSub && ok; ++j) {
                const int tile = st * kSub + j;
                if (!kSplitQ && kEpiGroups > 1 && (sn * kSub + j) % kEpiGroups != group) continue;
                if (!published) {
                    // the stage's MMAs are done (and the slot's previous use fully released)
                    if (!mbar_wait(&tfull_bar[as], static_cast<uint32_t>((sn >> 1) & 1), &abort_flag, p.wait_ns)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    published = true;
                }
                if (tile * kTileKeys >= nv) {
                    // no MMA wrote this tile (past the visible keys): the slot counts it anyway
                    mbar_arrive(&tempty_bar[as]);
                    continue;
                }
                const int key = tile * kTileKeys + lrow;
                for (int qi = 0; qi < kWq; ++qi) {
                    const int q = q_lo + qi;
                    if (q >= nqu) {
                        // (a unit's last query row may be missing: its group still frees the tile)
                        if (kSplitQ) {
                            tc_fence_before();
                            mbar_arrive(&tempty_bar[as]);
                        }
                        break;
                    }
                    const uint32_t ta0 = tmem_base + lane_addr + static_cast<uint32_t>((as * kSub + j) * kAccColsQ + q * NP);
                    if constexpr (kChunked) {
                        // 8 columns per load; four partial sums (heads h mod 4) in two packed pairs
                        uint64_t a01 = 0, a23 = 0;
#pragma unroll
                        for (int c = 0; c < NP; c += 8) {
                            uint32_t r[8];
                            DSV4_TMEM_LD_32x32b_X8(ta0 + static_cast<uint32_t>(c), r);
                            tmem_wait_ld();
#pragma unroll
                            for (int i = 0; i < 8; i += 4) {
                                fma_f32x2(a01, pack_f32x2(fmaxf(__uint_as_float(r[i + 0]), 0.f),
                                                          fmaxf(__uint_as_float(r[i + 1]), 0.f)),
                                          pack_f32x2(wv[0][c + i + 0], wv[0][c + i + 1]));
                                fma_f32x2(a23, pack_f32x2(fmaxf(__uint_as_float(r[i + 2]), 0.f),
                                                          fmaxf(__uint_as_float(r[i + 3]), 0.f)),
                                          pack_f32x2(wv[0][c + i + 2], wv[0][c + i + 3]));
                            }
                        }
                        tc_fence_before();
                        mbar_arrive(&tempty_bar[as]);
                        float s0, s1, s2, s3;
                        unpack_f32x2(a01, s0, s1);
                        unpack_f32x2(a23, s2, s3);
                        if (key < nvq[qi]) {
                            __stcs(srow[qi] + key, (s0 + s1) + (s2 + s3));
                        }
                        continue;
                    }
                    // exactly the NP columns of query q the MMA wrote (columns past them hold
                    // stale values)
                    uint32_t r[NP];
                    const uint32_t ta = ta0;
                    if constexpr (NP == 64) {
                        DSV4_TMEM_LD_32x32b_X64(ta, r);
                    } else if constexpr (NP == 32) {
                        DSV4_TMEM_LD_32x32b_X32(ta, r);
                    } else if constexpr (NP == 48) {
                        DSV4_TMEM_LD_32x32b_X32(ta, r);
                        uint32_t* r2 = r + 32;
                        DSV4_TMEM_LD_32x32b_X16(ta + 32u, r2);
                    } else {
                        DSV4_TMEM_LD_32x32b_X16(ta, r);
                    }
                    tmem_wait_ld();
                    if (kSplitQ || q == nqu - 1) {           // the accumulator is read out
                        tc_fence_before();
                        mbar_arrive(&tempty_bar[as]);
                    }
                    float s = 0.f;
                    if constexpr (FP8) {
                        // four partial sums (heads h mod 4) in two packed pairs: half the FMA
                        // instructions and a quarter of the dependent-FMA latency per key (here
                        // the epilogue, not HBM, sets the pace)
                        uint64_t a01 = 0, a23 = 0;
#pragma unroll
                        for (int h4 = 0; h4 < NP / 4; ++h4) {
                            const float4 wq = reinterpret_cast<const float4*>(s_wv)[h4];
                            fma_f32x2(a01, pack_f32x2(fmaxf(__uint_as_float(r[4 * h4 + 0]), 0.f),
                                                      fmaxf(__uint_as_float(r[4 * h4 + 1]), 0.f)),
                                      pack_f32x2(wq.x, wq.y));
                            fma_f32x2(a23, pack_f32x2(fmaxf(__uint_as_float(r[4 * h4 + 2]), 0.f),
                                                      fmaxf(__uint_as_float(r[4 * h4 + 3]), 0.f)),
                                      pack_f32x2(wq.z, wq.w));
                        }
                        float s0, s1, s2, s3;
                        unpack_f32x2(a01, s0, s1);
                        unpack_f32x2(a23, s2, s3);
                        s = ((s0 + s1) + (s2 + s3)) * ks_cur[j];
                    } else {
#pragma unroll
                        for (int h = 0; h < NP; ++h)
                            s = fmaf(wv[kWSmem ? 0 : qi][kWSmem ? 0 : h], fmaxf(__uint_as_float(r[h]), 0.f), s);
                    }
                    if (key < nvq[qi]) {
                        float* dst = srow[qi] + key;
                        if (p.reuse_keys) __stcs(dst, s);
                        else *dst = s;
                        if (QB == 1 && p.hist) {
                            const uint32_t bin = float_to_key(s) >> 20;
                            atomicAdd(&s_hist[bin >> 1], (bin & 1u) ? 0x10000u : 1u);
                        }
                    }
                }
            }
            id_cur = id_next;
        }
        if (!ok) {
            flag_error(p.eword, DSV4_EWORD_TIMEOUT);
            abort_flag = 1;
        }
        if (p.hist && cur_row >= 0) flush(cur_row);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    // looked up once (a function-local static is initialised once, even with several threads)
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
        return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
    }();
    return fn;
}

}  // namespace

bool encode_2d_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows,
                    uint32_t box_inner, uint32_t box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(inner) * 2ull};
    cuuint32_t box[2] = {box_inner, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_3d_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t mid, uint64_t outer,
                    uint32_t box_inner, uint32_t box_mid) {
    PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(mid),
                          static_cast<cuuint64_t>(outer)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(inner) * 2ull, static_cast<cuuint64_t>(inner) * mid * 2ull};
    cuuint32_t box[3] = {box_inner, box_mid, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
                  estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t index_ws_bytes(const dsv4_index_args& a) {
    const int rows = a.batch * a.n_q;
    size_t b = 0;
    b += align_up(topk_ws_bytes(rows, a.max_comp, a.top_k), 256);
    if (!a.scores_out) b += align_up(static_cast<size_t>(rows) * a.max_comp * 4, 256);
    return b;
}

size_t index_zero_bytes(const dsv4_index_args& a) {
    const int rows = a.batch * a.n_q;
    return topk_uses_hist(a.max_comp) ? topk_hist_bytes(rows) : 0;
}

namespace {
template <bool FP8, int NP, int EG, int QB>
int launch_scores_fmt(const dsv4_index_args& a, float* scores, uint32_t* hist, uint32_t* eword,
                      cudaStream_t stream, const dsv4_compress_args* fresh) {
    using F = KeyFmt<FP8, QB>;
    const int rows = a.batch * a.n_q;
    PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
    if (!encode) return DSV4_ERR_LAUNCH;
    const CUtensorMapDataType dt = FP8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    CUtensorMap kmap, qmap;
    {
        cuuint64_t dims[3] = {static_cast<cuuint64_t>(kDim), static_cast<cuuint64_t>(a.max_comp),
                              static_cast<cuuint64_t>(a.batch)};
        cuuint64_t strides[2] = {kDim * 1ull * F::kElem, static_cast<cuuint64_t>(a.max_comp) * kDim * F::kElem};
        cuuint32_t box[3] = {static_cast<cuuint32_t>(F::kBoxInner), static_cast<cuuint32_t>(F::kBoxRows), 1};
        cuuint32_t estr[3] = {1, 1, 1};
        if (encode(&kmap, dt, 3, const_cast<void*>(a.keys), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return DSV4_ERR_LAUNCH;
    }
    {
        cuuint64_t dims[2] = {static_cast<cuuint64_t>(kDim), static_cast<cuuint64_t>(rows) * a.heads};
        cuuint64_t strides[1] = {kDim * 1ull * F::kElem};
        cuuint32_t box[2] = {static_cast<cuuint32_t>(F::kBoxInner), static_cast<cuuint32_t>(a.heads)};
        cuuint32_t estr[2] = {1, 1};
        if (encode(&qmap, dt, 2, const_cast<void*>(a.q), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return DSV4_ERR_LAUNCH;
    }
    ScoreParams p;
    p.w = a.w;
    p.n_comp = a.n_comp;
    p.q_pos = a.q_pos;
    p.scores = scores;
    p.hist = hist;
    p.fresh_row0 = fresh ? fresh->out_row0 : nullptr;
    p.fresh_rows = fresh ? fresh->tokens / fresh->ratio : 0;
    p.eword = eword;
    p.q_scale = FP8 ? a.q_scale : nullptr;
    p.key_scale = FP8 ? a.key_scale : nullptr;
    p.claim = eword && rows <= kMaxClaimRows ? eword + kClaimWord : nullptr;
    p.reuse_keys = rows > sm_count() ? 1 : 0;
    p.rows = rows;
    p.n_q = a.n_q;
    p.heads = a.heads;
    p.max_comp = a.max_comp;
    p.ratio = a.ratio;
    p.stages_per_row = (a.max_comp + F::kStageKeys - 1) / F::kStageKeys;
    p.gpb = (a.n_q + QB - 1) / QB;
    p.units = a.batch * p.gpb;
    const WaitCtl wc = wait_ctl(DSV4_WAIT_FAULT_SCORER_STAGE);
    p.fault = wc.fault;
    p.wait_ns = wc.wait_ns;
    const long long total = static_cast<long long>(p.units) * p.stages_per_row;
    if (total > 0) {
        if (once_per_device(reinterpret_cast<const void*>(index_score_kernel<FP8, NP, EG, QB>), kAttrLaunch, [] {
                return cudaFuncSetAttribute(index_score_kernel<FP8, NP, EG, QB>,
                                            cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            static_cast<int>(F::kSmem));
            }) != cudaSuccess)
            return DSV4_ERR_LAUNCH;
        long long grid = sm_count();
        if (grid > total) grid = total;
        count_launch();
        if (launch_k(index_score_kernel<FP8, NP, EG, QB>, dim3(static_cast<unsigned>(grid)), dim3(64 + 128 * EG),
                     F::kSmem,
                     stream, true, kmap, qmap, p) != cudaSuccess)
            return DSV4_ERR_LAUNCH;
    }
    return DSV4_OK;
}

int launch_scores(const dsv4_index_args& a, float* scores, uint32_t* hist, uint32_t* eword,
                  cudaStream_t stream, const dsv4_compress_args* fresh) {
    const int n_pad = (a.heads + 15) / 16 * 16;
    // Three epilogue groups where the epilogue, not HBM, sets the pace: FP8 keys (512 keys per
    // stage). One group for bf16 keys, whose registers then leave room for a compressor CTA
    // beside the scoring CTA. Four (or, for two or three query rows, two) queries per MMA with
    // many rows of bf16 keys and no histogram to build (prefill), each query drained by its
    // own epilogue group: a tcgen05.mma costs its issuing thread about the same at any N, so
    // the wider MMA halves the instructions per score.
    const bool multi = static_cast<long long>(a.batch) * a.n_q > sm_count() && a.n_q >= 2 && !hist;
    const bool quad = multi && a.n_q >= 4;
#define DSV4_SCORES_NP(np)                                                               \
    if (n_pad == np)                                                                     \
        return a.key_fp8 ? launch_scores_fmt<true, np, 3, 1>(a, scores, hist, eword, stream, fresh) \
               : quad    ? launch_scores_fmt<false, np, 4, 4>(a, scores, hist, eword, stream, fresh) \
               : multi   ? launch_scores_fmt<false, np, 2, 2>(a, scores, hist, eword, stream, fresh) \
                         : launch_scores_fmt<false, np, 1, 1>(a, scores, hist, eword, stream, fresh);
    DSV4_SCORES_NP(16)
    DSV4_SCORES_NP(32)
    DSV4_SCORES_NP(48)
    DSV4_SCORES_NP(64)
#undef DSV4_SCORES_NP
    return DSV4_ERR_INVALID_ARG;
}
}  // namespace

int launch_index_score(const dsv4_index_args& a, uint32_t* eword, cudaStream_t stream) {
    if (a.batch * a.n_q == 0) return DSV4_OK;
    return launch_scores(a, a.scores_out, nullptr, eword, stream, nullptr);
}

int launch_indexer(const dsv4_index_args& a, uint8_t* ws, uint32_t* eword, cudaStream_t stream,
                   const dsv4_compress_args* fresh_keys) {
    const int rows = a.batch * a.n_q;
    if (rows == 0) return DSV4_OK;
    // workspace: [top-k workspace (its histogram first, zeroed by the caller)][scores]
    uint8_t* topk_ws = ws;
    float* scores = a.scores_out;
    if (!scores)
        scores = reinterpret_cast<float*>(ws + align_up(topk_ws_bytes(rows, a.max_comp, a.top_k), 256));
    // the top-k histogram is built by the scoring epilogue (shared-memory counts, flushed per row)
    uint32_t* hist = topk_uses_hist(a.max_comp) ? topk_hist_buffer(topk_ws) : nullptr;
    if (int rc = launch_scores(a, scores, hist, eword, stream, fresh_keys)) return rc;
    TopkRows t;
    t.scores = scores;
    t.n_vis = nullptr;
    t.n_comp = a.n_comp;
    t.q_pos = a.q_pos;
    t.n_q = a.n_q;
    t.ratio = a.ratio;
    t.idx_out = a.idx_out;
    t.rows = rows;
    t.max_comp = a.max_comp;
    t.top_k = a.top_k;
    t.hist_zeroed = true;
    t.hist_built = hist != nullptr;
    t.pdl = true;
    return launch_topk(t, topk_ws, eword, stream);
}

}  // namespace dsv4

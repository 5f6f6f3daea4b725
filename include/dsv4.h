/*
 * dsv4.h — C ABI of the GB300 (sm_103a) compressed-sparse-attention (CSA) step.
 *
 * The step of a DeepSeek-V4-style attention layer, in four stages:
 *   1. block compressor   (dsv4_compress)
 *   2. lightning indexer  (dsv4_indexer_topk: MQA scoring + per-token top-k)
 *   3. top-k on given scores (dsv4_topk: the selection stage taken alone)
 *   4. gather + sink attention (dsv4_sparse_attn_decode)
 * plus dsv4_csa_decode, which runs stages 1, 2 and 4 of one decode step back to back.
 *
 * Sources, cited by page title and section:
 *   [A] "nvfp4-megamoe-kernel: compare v0.1-e2e-working...v-c1-c2-c3-20260602"
 *   [B] "nvfp4-megamoe-kernel: compare master..pure-nvfp4"
 *   [C] "nvfp4-megamoe-kernel: compare v-precision-floor-fix-20260603..pure-nvfp4"
 *
 * Conventions for every entry point
 *   - Pointers named in an args struct are DEVICE pointers unless stated. bf16 tensors are
 *     row-major and densely packed in the stated shape. Every device pointer must be
 *     16-byte aligned.
 *   - The caller owns every buffer, the workspace included. The library never allocates,
 *     frees or synchronises, and never reads a device value on the host, so each call can
 *     be captured in a CUDA graph. Work is ordered on the given stream only.
 *   - Per-sequence counts (n_comp, win_len) are device int32 arrays, so one captured graph
 *     serves every step.
 *   - Return value: DSV4_OK, or an error code. Arguments are checked on the host before any
 *     launch (DSV4_ERR_INVALID_ARG: null pointer, misalignment, bad size, workspace too
 *     small). DSV4_ERR_LAUNCH reports a failed launch (cudaGetLastError). Errors found on
 *     the device (an index out of range, a bounded wait that ran out) are recorded in an
 *     error word at the start of the workspace and read with dsv4_read_error_word; the
 *     kernels never trap. As with any asynchronous CUDA work, a fault surfaces on a later
 *     call.
 *   - The workspace must hold dsv4_*_workspace_size(args) bytes. Its contents need no
 *     initialisation: each call clears what it uses, on the stream.
 */
#ifndef DSV4_H
#define DSV4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* dsv4_stream_t; /* a cudaStream_t; NULL = legacy default stream */

enum {
    DSV4_OK = 0,
    DSV4_ERR_INVALID_ARG = 1, /* rejected on the host before any launch */
    DSV4_ERR_LAUNCH = 2,      /* a kernel launch failed */
    DSV4_ERR_BAD_INDEX = 3,   /* device: an index outside [0, visible) was masked */
    DSV4_ERR_TIMEOUT = 4,     /* device: a bounded wait ran out; the kernel returned early */
    DSV4_ERR_UNSUPPORTED = 5  /* the device is not sm_103 (the only code the library holds) */
};

/* Device error word bits (dsv4_read_error_word). */
#define DSV4_EWORD_BAD_INDEX 0x1u
#define DSV4_EWORD_TIMEOUT   0x2u

/* ---------------------------------------------------------------------------------------
 * Stage 1. Block compressor + RMSNorm + partial RoPE.
 *
 * For sequence s, block b (tokens t = 0..ratio-1 of the block), channel c:
 *     w_t = softmax_t( Z[s, b*ratio + t, c] + bias[t, c] )
 *     x_c = sum_t w_t * C[s, b*ratio + t, c]              (the bias never touches C)
 *     y   = x / sqrt(mean_c(x_c^2) + eps) * gamma
 * then the last rope_dim channels are rotated in interleaved pairs (2j, 2j+1) by the angle
 * pos * theta^(-2j/rope_dim), pos = pos0[s] + b*ratio (the block's first token), and y is
 * rounded once to bf16.
 * [A] compressor_reduce.cu hca_compress_reduce_kernel (plain per-block softmax-reduce) and
 * apply_kv_norm_kernel (eps 1e-6); [B]/[C] commit "Fix two correctness bugs", item 1 and the
 * compressor_reduce.cu hunks (bias on the logits only); [A] PERFORMANCE_AUDIT.md "P5"
 * (interleaved-pair RoPE of the last 64 dims); [B] single_shot_inference.py eager_attention
 * (RoPE applied to the compressed entry after compression and norm).
 *
 * Arithmetic: fp32 on the device (angles in fp64), one bf16 rounding at the output.
 */
typedef struct dsv4_compress_args {
    const void* C;            /* bf16 [batch, tokens, dim]   projected KV                 */
    const void* Z;            /* bf16 [batch, tokens, dim]   gate logits                  */
    const float* bias;        /* fp32 [ratio, dim]           positional bias (logits only) */
    const float* gamma;       /* fp32 [dim]                  RMSNorm weight               */
    const int64_t* pos0;      /* int64 [batch]               position of token 0          */
    void* out;                /* bf16 [batch, out_rows, dim] destination (e.g. the cache) */
    const int32_t* out_row0;  /* int32 [batch] first destination row, or NULL for row 0   */
    int batch, tokens, dim, ratio, rope_dim;
    int out_rows;             /* rows per sequence in `out` (>= out_row0 + tokens/ratio)  */
    float eps;                /* 1e-6 on the pages                                        */
    double rope_theta;        /* 10000 on the pages                                       */
    /* Two-stream (CSA) form ([A] compressor_reduce.cu "CSA compressor reduce kernel", with
     * the bias fix above): overlap = 1 makes C and Z [batch, tokens, 2*dim] (channels
     * [0, dim) stream a, [dim, 2*dim) stream b) and bias [ratio, 2*dim]; entry b pools
     * block b-1 from stream a and block b from stream b under one softmax per channel
     * (2*ratio logits), the bias row t of each stream's half on the logits only. Entry 0
     * takes its stream-a block from prev_C / prev_Z ([batch, ratio, 2*dim]) when they are
     * given (both or neither), else pools its own block alone (the sequence's first block).
     * RMSNorm, RoPE (at the position of the entry's own first token) and the output are as
     * in the plain form. overlap = 0: the plain form; prev_C / prev_Z must be NULL. */
    int overlap;
    const void* prev_C;
    const void* prev_Z;
    /* FP8 key cache (for the FP8 indexer, see dsv4_index_args.key_fp8): out_fp8 = 1 stores each
     * entry as FP8 E4M3 codes (out: bytes [batch, out_rows, dim]) with its fp32 scale in
     * out_scale [batch, out_rows], quantized from the entry's fp32 value after RoPE exactly as
     * dsv4_quantize_rows_fp8 quantizes a row. out_fp8 = 0: bf16 entries, out_scale NULL. */
    int out_fp8;
    float* out_scale;
    /* Mixed FP8 / bf16 KV cache ([B] single_shot_inference.py eager_attention, "compressed KV
     * (mixed storage: FP8 + BF16 RoPE)"): out_fp8 = 2 stores the entry's first
     * dim - rope_dim channels as FP8 E4M3 codes in out (bytes [batch, out_rows,
     * dim - rope_dim]) with one fp32 scale per entry in out_scale (amax of those channels /
     * 448, as dsv4_quantize_rows_fp8), and its last rope_dim channels as bf16 in out_rope
     * ([batch, out_rows, rope_dim]); dsv4_attn_args.kv_fp8 reads that storage. out_rope is
     * NULL unless out_fp8 = 2. */
    void* out_rope;
} dsv4_compress_args;

int dsv4_compress(const dsv4_compress_args* args, dsv4_stream_t stream);

/* Stage 1 at decode time, one token per call: the compressor's state lives on the device, so
 * every decode step issues the same call (one captured CUDA graph serves them all) and no host
 * code has to know when a block completes ([C] GETTING+CUDAGRAPH_READY.md "SECTION C": the
 * compressor's host-side decisions are what keeps the step out of a graph; [A] commit "C1"
 * fixes the cache rows).
 *
 * Per sequence s the call stages this token's C and Z; when the staged block holds `ratio`
 * tokens it is compressed exactly as dsv4_compress would compress it (plain or two-stream form,
 * RMSNorm, RoPE at the block's first token, pos[s] - ratio + 1) into out[s, n_comp[s]], then
 * n_comp[s] is incremented and fill[s] reset. In the two-stream form the completed block is
 * kept as stream a of the next entry; the sequence's first entry (n_comp[s] == 0 when it
 * completes) has stream b only. When n_comp[s] == out_rows the entry is not stored and n_comp
 * stays. State (caller-owned, device): stage, fill and n_comp, all zero at the start of a
 * sequence (or fill zero and n_comp the cache rows already written, at a block boundary). */
typedef struct dsv4_compress_step_args {
    const void* C;            /* bf16 [batch, w]  this step's token, w = dim (plain) or 2*dim   */
    const void* Z;            /* bf16 [batch, w]                                                */
    const float* bias;        /* fp32 [ratio, w]                                                */
    const float* gamma;       /* fp32 [dim]                                                     */
    const int64_t* pos;       /* int64 [batch] position of this token                           */
    void* stage;              /* bf16 [batch, 2, 2, ratio, w] state                              */
    int32_t* fill;            /* int32 [batch] state: tokens of the block in progress           */
    int32_t* n_comp;          /* int32 [batch] state: entries written to `out`                  */
    void* out;                /* bf16 [batch, out_rows, dim] the compressed cache               */
    int batch, dim, ratio, rope_dim, out_rows, overlap;
    float eps;
    double rope_theta;
    /* Output format, as dsv4_compress_args: out_fp8 = 0 bf16 rows; 1 FP8 E4M3 rows (out:
     * bytes [batch, out_rows, dim]) with scales in out_scale [batch, out_rows]; 2 the mixed
     * KV storage (out: codes [batch, out_rows, dim - rope_dim], out_scale, out_rope bf16
     * [batch, out_rows, rope_dim]). */
    int out_fp8;
    float* out_scale;
    void* out_rope;
} dsv4_compress_step_args;
int dsv4_compress_step(const dsv4_compress_step_args* args, dsv4_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * Stage 2. Lightning-indexer score + per-token top-k.
 *
 *   I[s, t, j] = sum_h w[s, t, h] * ReLU( sum_d q[s, t, h, d] * keys[s, j, d] )
 * in fp32 (bf16 products, fp32 accumulation), over the visible entries j of query t:
 * j < n_comp[s] when q_pos is NULL (decode), else j < min(n_comp[s], (q_pos[s,t]+1)/ratio)
 * (block j, covering tokens [j*ratio, (j+1)*ratio-1], is visible when it ends at or before
 * the query position). Then idx_out[s, t, :] = the indices of the min(top_k, visible)
 * largest scores, equal scores ranked by lower index, written in ascending index order and
 * padded with -1 up to top_k.
 * [A] ARCHITECTURE_AND_MEMORY_AUDIT.md "F1" (one 128-wide key per block, shared by all 64
 * indexer heads) and "F3" (the MQA scoring formula, tk = min(top_k, n_comp), topk);
 * [A] archived_plans/NEXT_STEPS.md "Issue 2" (causal visibility of compressed entries);
 * [C] GETTING+CUDAGRAPH_READY.md "SECTION C" item 3 (fixed-length, padded index list).
 */
typedef struct dsv4_index_args {
    const void* q;            /* bf16 [batch, n_q, heads, dim]  indexer queries            */
    const float* w;           /* fp32 [batch, n_q, heads]       per-head weights           */
    const void* keys;         /* bf16 [batch, max_comp, dim]    compressed indexer keys    */
    const int32_t* n_comp;    /* int32 [batch]                  valid cache rows           */
    const int64_t* q_pos;     /* int64 [batch, n_q] query positions, or NULL (all visible) */
    int32_t* idx_out;         /* int32 [batch, n_q, top_k]                                 */
    float* scores_out;        /* fp32 [batch, n_q, max_comp] copy of the scores, or NULL    */
    int batch, n_q, heads, dim, max_comp, top_k, ratio;
    /* FP8 index keys ([B] single_shot_inference.py: "Indexer keys are stored as FP8_E4M3 in
     * the KV cache", scored on the FP8 tensor-core path). key_fp8 = 1: q and keys hold FP8
     * E4M3 codes ([batch, n_q, heads, dim] and [batch, max_comp, dim] bytes) with one fp32
     * scale per query head (q_scale [batch, n_q, heads]) and per key (key_scale
     * [batch, max_comp]), as dsv4_quantize_rows_fp8 writes them; the score is the bf16 form's
     * definition on the dequantized rows, scale * code. key_fp8 = 0: bf16 rows, scales NULL. */
    int key_fp8;
    const float* q_scale;
    const float* key_scale;
} dsv4_index_args;

size_t dsv4_indexer_topk_workspace_size(const dsv4_index_args* args);
int dsv4_indexer_topk(const dsv4_index_args* args, void* ws, size_t ws_bytes,
                      dsv4_stream_t stream);

/* The scoring half of stage 2 alone: writes I[s, t, j] for the visible j into
 * args->scores_out (required here) and leaves idx_out untouched. Same sources as above. */
size_t dsv4_index_score_workspace_size(const dsv4_index_args* args);
int dsv4_index_score(const dsv4_index_args* args, void* ws, size_t ws_bytes,
                     dsv4_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * Stage 3 alone. Top-k of caller-given fp32 scores, same rule as above.
 * scores [rows, max_comp]; n_vis [rows] visible counts; idx_out [rows, top_k].
 * Equal scores (+0.0 and -0.0 are equal) rank by lower index. Scores must not be NaN.
 */
typedef struct dsv4_topk_args {
    const float* scores;
    const int32_t* n_vis;
    int32_t* idx_out;
    int rows, max_comp, top_k;
} dsv4_topk_args;

size_t dsv4_topk_workspace_size(const dsv4_topk_args* args);
int dsv4_topk(const dsv4_topk_args* args, void* ws, size_t ws_bytes, dsv4_stream_t stream);

/* Stage 3 alone, for callers that cannot allocate device memory (for instance code running
 * inside an allocator hook, a serving loop that forbids cudaMalloc after start-up, or a
 * plug-in that receives only its input and output buffers). The pages have no counterpart
 * for this entry point: it is a convenience of this library. Same arguments, rule and
 * results as dsv4_topk, but no workspace: the scratch it needs lives in a fixed 16 MiB
 * device array that the library holds on each GPU it runs on until the process exits.
 * Calls whose scratch need (dsv4_topk_workspace_size(args)) exceeds 16 MiB return
 * DSV4_ERR_INVALID_ARG before any launch (rows of more than 32,768 entries need 33 KiB each:
 * up to 496 such rows per call).
 * The first call on a device looks up the array's device address; with lazy module loading
 * that lookup is also when the driver reserves the 16 MiB on that device, so a failure to
 * reserve it comes back from that first call as DSV4_ERR_LAUNCH. Make the first call on
 * each device at start-up, before any stream capture. Every call shares the one array, so calls that overlap on the
 * GPU (different streams, or different host threads) race and must not be issued; each call
 * clears what it needs. Device-side findings (counts out of range) are not reported by this
 * variant. No memory is allocated or freed. */
int dsv4_topk_noalloc(const dsv4_topk_args* args, dsv4_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * Stage 4. Gather into the caller's buffer + MQA attention with a per-head sink.
 *
 * Rows of query t of sequence s: the compressed rows comp_kv[s, idx[s,t,j]] for the valid
 * (>= 0) entries of idx (or, when idx is NULL — the HCA form — every visible compressed
 * row), then the sliding-window rows: win holds the most recent tokens in order with the
 * n_q query tokens last, and query t sees the `window` rows ending at its own row,
 *     [t + win_len[s] - n_q - window + 1,  t + win_len[s] - n_q]  clipped to [0, win_len[s]).
 * (Decode, n_q = 1: every one of the win_len rows; their order does not matter.)
 *   s_j = scale * q[s,t,h,:] . row_j,      m = max(max_j s_j, sink[h])
 *   out[s,t,h,:] = sum_j e^(s_j - m) row_j / (sum_j e^(s_j - m) + e^(sink[h] - m))
 * K and V are the same rows (shared-KV MQA). The sink is a logit in the scaled domain.
 * gather (optional): slot j < top_k holds comp_kv[s, idx[s,t,j]] (zeros for -1), slot
 * top_k + i the i-th window row of the query (zeros past the window).
 * [A] commit "C2" (pre-allocated gather buffer of top_k + window rows, no torch.cat);
 * [A] fmha_6warp_tma_multirow_multitile.cuh "Sink bias correction" (sink adds to the
 * denominator only, in the scaled domain); [A] PERFORMANCE_AUDIT.md "P4" (v = k);
 * [B] single_shot_inference.py eager_attention (scale = 1/sqrt(hd); CSA gathers top-k,
 * ratio > 4 gathers every compressed entry, then the window).
 * Arithmetic: bf16 tensor-core products, fp32 accumulation and softmax, bf16 output.
 */
typedef struct dsv4_attn_args {
    const void* q;            /* bf16 [batch, n_q, heads, dim]                              */
    const float* sink;        /* fp32 [heads]                                               */
    const void* comp_kv;      /* bf16 [batch, max_comp, dim]                                */
    const int32_t* n_comp;    /* int32 [batch]                                              */
    const int32_t* idx;       /* int32 [batch, n_q, top_k], or NULL: dense (top_k = max_comp) */
    const int64_t* q_pos;     /* int64 [batch, n_q] or NULL; limits the dense form          */
    const void* win;          /* bf16 [batch, win_rows, dim]                                */
    const int32_t* win_len;   /* int32 [batch]                                              */
    void* gather;             /* bf16 [batch, n_q, top_k + window, dim], or NULL            */
    void* out;                /* bf16 [batch, n_q, heads, dim]                              */
    int batch, n_q, heads, dim, max_comp, top_k, window, win_rows, ratio;
                              /* heads: 1..16, or a multiple of 16 up to 64; dim: 128/256/512 */
    float scale;              /* 1/sqrt(dim) on the pages                                   */
    /* Optional inverse RoPE of the output ([B] single_shot_inference.py eager_attention: the
     * FMHA output is rotated back at the query positions): when out_rope_pos (int64
     * [batch, n_q]) is given, the last out_rope_dim channels of every head's output are
     * rotated in pairs (2j, 2j+1) by -pos * out_rope_theta^(-2j/out_rope_dim) before the bf16
     * rounding. NULL: the output is not rotated. */
    const int64_t* out_rope_pos;
    int out_rope_dim;         /* even, 2..min(dim, 128) when out_rope_pos is given          */
    double out_rope_theta;    /* 10000 on the pages                                         */
    /* Mixed FP8 / bf16 compressed KV (dsv4_compress_args.out_fp8 = 2): with kv_fp8 = 1,
     * comp_kv is NULL and the compressed rows come from kv_nope (E4M3 codes [batch, max_comp,
     * dim - kv_rope_dim]), kv_scale (fp32 [batch, max_comp]) and kv_rope (bf16 [batch,
     * max_comp, kv_rope_dim]); each gathered row is dequantized to bf16, channel by channel
     * bf16(fp32(code) * scale), the RoPE part as stored, and that bf16 row is what the
     * attention multiplies and what the gather buffer receives. kv_rope_dim: a multiple of 8,
     * 8..dim-8. kv_fp8 = 0: the three are NULL. */
    int kv_fp8;
    const void* kv_nope;
    const float* kv_scale;
    const void* kv_rope;
    int kv_rope_dim;
} dsv4_attn_args;

/* Workspace: the 256-byte header (error word) plus, when few query rows are given (fewer than
 * 304 pairs of query row and head group; groups of 32 heads when heads is a multiple of 32,
 * else of 16), the split form's per-chunk partials: rows x ceil((top_k + window) / 128) x
 * (heads rounded up to whole groups) x (dim + 2) x 4 bytes, the (m, l) and O parts each
 * rounded up to 256. With more rows one CTA walks each row and the header alone suffices.
 * Returns 0 for a NULL args. */
size_t dsv4_sparse_attn_workspace_size(const dsv4_attn_args* args);
int dsv4_sparse_attn_decode(const dsv4_attn_args* args, void* ws, size_t ws_bytes,
                            dsv4_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * One decode step: optional compression of the newest block of the main KV and of the
 * indexer keys (written at rows out_row0 of the caches), then indexer top-k (skipped when
 * index.heads == 0: the HCA form), then gather + attention over the selected rows.
 * The stages run back to back on one stream; the workspace is shared.
 */
typedef struct dsv4_csa_args {
    const dsv4_compress_args* compress_kv;   /* or NULL */
    const dsv4_compress_args* compress_keys; /* or NULL */
    const dsv4_index_args* index;            /* or NULL for the dense (HCA) form */
    const dsv4_attn_args* attn;              /* attn->idx must equal index->idx_out */
} dsv4_csa_args;

size_t dsv4_csa_decode_workspace_size(const dsv4_csa_args* args);
int dsv4_csa_decode(const dsv4_csa_args* args, void* ws, size_t ws_bytes,
                    dsv4_stream_t stream);

/* FP8 E4M3 quantization of bf16 rows (queries or keys for the FP8 indexer): per row
 * scale = amax / 448 in fp32 (1 for an all-zero row), code = E4M3(x / scale), the division in
 * fp32, round to nearest even, saturating. x bf16 [rows, dim] -> q [rows, dim] bytes,
 * scale fp32 [rows]. dim: 32, 64, 128, 256, 512 or 1024. */
int dsv4_quantize_rows_fp8(const void* x, int rows, int dim, void* q, float* scale,
                           dsv4_stream_t stream);

/* ---------------------------------------------------------------------------------------
 * Test support: running the bounded-wait path on purpose. Not for a serving path.
 *
 * Every wait of a kernel on an asynchronous copy, or on another role of its CTA, is bounded
 * in time: when the limit runs out the kernel records DSV4_EWORD_TIMEOUT in the error word,
 * lets its own copies in flight land, frees its tensor memory and returns (the call reports
 * DSV4_ERR_TIMEOUT through dsv4_read_error_word). dsv4_test_wait_fault makes that happen
 * without any fault: from this call until the next, every launch of the named kernel leaves
 * one of its copies unissued, so the wait for that copy runs out, and every bounded wait of
 * that kernel gives up after wait_limit_us microseconds (1 .. 2,000,000; 0 keeps the default
 * of 2 s). DSV4_WAIT_FAULT_NONE restores normal launches. The setting is process-wide and is
 * read when a kernel is launched (a graph captured meanwhile keeps it). Returns
 * DSV4_ERR_INVALID_ARG for an unknown kernel or a limit out of range.
 *   DSV4_WAIT_FAULT_SCORER_STAGE: the indexer's scoring kernel (dsv4_index_score,
 *     dsv4_indexer_topk, dsv4_csa_decode) issues no copy for the first key stage of each
 *     CTA; the tensor-core warp's wait for that stage runs out.
 *   DSV4_WAIT_FAULT_ATTN_QUERY: the split-form attention kernel (decode: fewer query rows,
 *     see dsv4_sparse_attn_workspace_size) issues no copy of its query tile; the wait before
 *     its first tensor-core product runs out.
 * [A] fmha_multitile_capi.cu (errors of the device path returned through C-ABI status codes,
 * never by trapping the process).
 */
enum {
    DSV4_WAIT_FAULT_NONE = 0,
    DSV4_WAIT_FAULT_SCORER_STAGE = 1,
    DSV4_WAIT_FAULT_ATTN_QUERY = 2
};
int dsv4_test_wait_fault(int which, uint32_t wait_limit_us);

/* ---------------------------------------------------------------------------------------
 * Utilities.
 */
const char* dsv4_status_string(int status);
/* Reads (and clears) the device error word at the start of `ws`. Synchronises the stream:
 * for tests and diagnostics, never on the hot path. */
int dsv4_read_error_word(void* ws, dsv4_stream_t stream, uint32_t* out);
/* Copies `bytes` from src to dst on `stream` with one kernel (the SMs move the data), after
 * the kernel enqueued before it (programmatic dependent launch). Either pointer may be device
 * memory or pinned host memory (cudaHostAlloc / cudaHostRegister); on a Grace-Blackwell GPU
 * the SMs reach pinned host memory over the chip-to-chip link, so a decode step's inputs and
 * outputs (a few hundred kilobytes each way) move without a copy-engine transfer, which as a
 * node of a captured graph cost ~12 us for a step's 370 KB of inputs (the kernel: ~1 us,
 * measured on GB300). The pages have no counterpart for
 * this entry point: it serves the end-to-end step (inputs in, outputs out every step).
 * Both pointers 16-byte aligned, bytes a multiple of 16, ranges not overlapping, else
 * DSV4_ERR_INVALID_ARG (as for pageable host memory, which the kernel cannot address);
 * bytes = 0 does nothing. The caller keeps both buffers alive until the stream passes the
 * copy. */
int dsv4_copy_async(void* dst, const void* src, size_t bytes, dsv4_stream_t stream);
/* Number of kernel launches the last successful call on this host thread enqueued. */
int dsv4_last_launch_count(void);
/* Compressed-cache rows for a context: (max_context + ratio - 1) / ratio ([A] commit "C1"). */
int64_t dsv4_max_comp(int64_t max_context, int ratio);

#ifdef __cplusplus
}
#endif
#endif /* DSV4_H */

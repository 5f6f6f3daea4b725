// Internal launchers behind the C ABI. Arguments reaching these have been validated on the
// host (abi.cu); workspaces are sized by the matching *_ws_bytes function.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

#include "dsv4.h"

namespace dsv4 {

// Test control of the bounded waits (dsv4_test_wait_fault): for kernel `which`
// (DSV4_WAIT_FAULT_*), whether its launches leave one copy unissued, and the limit in ns of
// its bounded waits (the default unless that kernel is the one named).
struct WaitCtl {
    int fault;
    unsigned long long wait_ns;
};
WaitCtl wait_ctl(int which);

int launch_compress(const dsv4_compress_args& a, cudaStream_t stream);
// SM copy of bytes (a multiple of 16; 16-byte aligned pointers; device or pinned host memory),
// launched with programmatic dependent launch after the kernel before it.
int launch_copy(void* dst, const void* src, size_t bytes, cudaStream_t stream);
int launch_compress_step(const dsv4_compress_step_args& a, cudaStream_t stream);
// FP8 E4M3 rows: one warp per row, scale = amax / 448 (fp32), codes of x / scale.
int launch_quantize_rows_fp8(const void* x, int rows, int dim, void* q, float* scale, cudaStream_t stream);
// Up to two compressions (e.g. main KV and indexer keys) in one launch; either may be null.
// Both compressions in one launch; the launch also clears `zero_bytes` bytes at `zero` (a
// 16-byte aligned workspace region, rounded up to 16 bytes) for the kernels after it, or a
// memset does when there is nothing to compress.
int launch_compress2(const dsv4_compress_args* a, const dsv4_compress_args* b, cudaStream_t stream,
                     void* zero, size_t zero_bytes);

// Top-k over fp32 score rows. Exactly one of n_vis (an int32 [rows] array) or the indexer
// geometry (n_comp [batch], q_pos [batch, n_q] or null, ratio) gives each row's visible count.
struct TopkRows {
    const float* scores;     // [rows, max_comp]
    const int32_t* n_vis;    // [rows] or null
    const int32_t* n_comp;   // [batch] (when n_vis is null)
    const int64_t* q_pos;    // [batch, n_q] or null
    int n_q, ratio;
    int32_t* idx_out;        // [rows, top_k]
    int rows, max_comp, top_k;
    bool hist_zeroed;        // the long-row histogram was zeroed by the caller
    bool hist_built;         // ... and already filled (by the scoring epilogue)
    bool pdl;                // launch with programmatic dependent launch
};
size_t topk_ws_bytes(int rows, int max_comp, int top_k);
int launch_topk(const TopkRows& t, uint8_t* ws, uint32_t* eword, cudaStream_t stream);
// Long rows keep a top-12-bit key histogram ([rows, 4096] u32) at the start of the top-k
// workspace; a producer of scores may fill it (after it was zeroed).
bool topk_uses_hist(int max_comp);
uint32_t* topk_hist_buffer(uint8_t* topk_ws);
size_t topk_hist_bytes(int rows);

size_t index_ws_bytes(const dsv4_index_args& a);
// Bytes at the start of the indexer workspace that must be zero when the call starts (the
// long-row histograms); callers clear them together with the error word.
size_t index_zero_bytes(const dsv4_index_args& a);
// fresh_keys: the compression that writes key rows just before (its rows are waited for).
int launch_indexer(const dsv4_index_args& a, uint8_t* ws, uint32_t* eword, cudaStream_t stream,
                   const dsv4_compress_args* fresh_keys = nullptr);
// Scores only (a.scores_out required); no top-k.
int launch_index_score(const dsv4_index_args& a, uint32_t* eword, cudaStream_t stream);

// 2D bf16 tensor map, row-major [rows, inner] (inner contiguous), 128-byte swizzle, boxes of
// box_inner x box_rows elements; out-of-range boxes read as zeros. Host only, no allocation.
bool encode_2d_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows,
                    uint32_t box_inner, uint32_t box_rows);
// 3-D bf16 tensor [outer][mid][inner] (dense), box {box_inner, box_mid, 1}, 128-byte swizzle.
bool encode_3d_bf16(CUtensorMap* map, const void* base, uint64_t inner, uint64_t mid, uint64_t outer,
                    uint32_t box_inner, uint32_t box_mid);

size_t attn_ws_bytes(const dsv4_attn_args& a);
int launch_attn(const dsv4_attn_args& a, uint8_t* ws, uint32_t* eword, cudaStream_t stream);

}  // namespace dsv4

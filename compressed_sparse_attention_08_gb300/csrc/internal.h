// Internal launchers behind the C ABI. Arguments reaching these have been validated on the
// host (abi.cu); workspaces are sized by the matching *_ws_bytes function.
#pragma once

#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

#include "dsv4.h"

namespace dsv4 {

int launch_compress(const dsv4_compress_args& a, cudaStream_t stream);

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
};
size_t topk_ws_bytes(int rows, int max_comp, int top_k);
int launch_topk(const TopkRows& t, uint8_t* ws, uint32_t* eword, cudaStream_t stream);

size_t index_ws_bytes(const dsv4_index_args& a);
int launch_indexer(const dsv4_index_args& a, uint8_t* ws, uint32_t* eword, cudaStream_t stream);
// Scores only (a.scores_out required); no top-k.
int launch_index_score(const dsv4_index_args& a, uint32_t* eword, cudaStream_t stream);

size_t attn_ws_bytes(const dsv4_attn_args& a);
int launch_attn(const dsv4_attn_args& a, uint8_t* ws, uint32_t* eword, cudaStream_t stream);

}  // namespace dsv4

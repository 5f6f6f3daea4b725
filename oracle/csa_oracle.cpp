// Oracle for the compressed-sparse-attention (CSA) decode step.
//
// TEST INFRASTRUCTURE ONLY. This file is the plain, slow, single-threaded fp64
// definition of what the CUDA path computes. Only the tests, the smoke check and
// the CPU-baseline leg of the benchmark may load it. It shares no code, header,
// table or helper with the CUDA library, and the CUDA library never calls it.
//
// Sources (web pages, cited by title and section):
//   [A] "nvfp4-megamoe-kernel: compare v0.1-e2e-working...v-c1-c2-c3-20260602"
//   [B] "nvfp4-megamoe-kernel: compare master..pure-nvfp4"
//   [C] "nvfp4-megamoe-kernel: compare v-precision-floor-fix-20260603..pure-nvfp4"
//
// Every input is bf16 (raw uint16 bit patterns) or fp32, widened exactly to
// double. All arithmetic is double. Results are rounded once, to bf16 with
// round-to-nearest-even, where the step's output is bf16.
//
// Parity pins: every function below is pinned by tests/test_oracle_pins.py
// (closed forms, invariants, brute force). None is "parity unpinned".

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <vector>

namespace {

double bf16_to_double(uint16_t b) {
    uint32_t u = static_cast<uint32_t>(b) << 16;
    float f;
    std::memcpy(&f, &u, sizeof f);
    return static_cast<double>(f);
}

// Round a double to the nearest bf16 (ties to even), directly from double.
uint16_t double_to_bf16(double x) {
    if (std::isnan(x)) return 0x7FC0;
    if (x == 0.0) return std::signbit(x) ? 0x8000 : 0x0000;
    if (std::isinf(x)) return x > 0 ? 0x7F80 : 0xFF80;
    int e = std::ilogb(x);                 // |x| in [2^e, 2^(e+1))
    int ulp_exp = e - 7;                   // bf16 keeps 8 significant bits
    if (ulp_exp < -133) ulp_exp = -133;    // bf16 subnormal spacing is 2^-133
    double scaled = std::ldexp(x, -ulp_exp);
    double r = std::nearbyint(scaled);     // default rounding mode: nearest, ties to even
    double y = std::ldexp(r, ulp_exp);
    if (std::fabs(y) > 3.3895313892515355e38) return x > 0 ? 0x7F80 : 0xFF80;  // beyond bf16 max
    float f = static_cast<float>(y);       // exact: y has at most 8 significant bits
    uint32_t u;
    std::memcpy(&u, &f, sizeof u);
    return static_cast<uint16_t>(u >> 16);
}

// Number of compressed entries a query at absolute position p may see.
// [A] archived_plans/NEXT_STEPS.md, "Issue 2" fix direction: a token at position p
// attends only to compressed entries whose window ends at or before p. Block j covers
// tokens [j*r, (j+1)*r - 1], so it is visible iff (j+1)*r - 1 <= p.
int64_t visible_entries(int64_t n_comp, int64_t p, int ratio) {
    if (p < 0) return 0;
    int64_t by_pos = (p + 1) / ratio;
    return std::min<int64_t>(n_comp, by_pos);
}

// FP8 E4M3 (the OCP 8-bit floating point format, "E4M3FN"): 1 sign bit, 4 exponent bits
// (bias 7), 3 mantissa bits; exponent field 0 holds the subnormals m * 2^-9; the largest
// finite value is 1.75 * 2^8 = 448 (code 0x7E), code 0x7F is NaN, there is no infinity.
// Encoding rounds to nearest, ties to even, and saturates to +-448 (finite inputs).
uint8_t e4m3_from_double(double x) {
    if (std::isnan(x)) return 0x7F;
    const uint8_t sign = std::signbit(x) ? 0x80 : 0x00;
    const double a = std::fabs(x);
    if (a == 0.0) return sign;
    int e = std::ilogb(a);                          // a in [2^e, 2^(e+1))
    if (e < -6) e = -6;                             // below 2^-6: the subnormal spacing 2^-9
    double q = std::nearbyint(std::ldexp(a, 3 - e)); // a in units of the spacing 2^(e-3)
    if (q >= 16.0) {                                 // rounded up to the next binade
        q = 8.0;
        ++e;
    }
    if (e > 8 || (e == 8 && q > 14.0)) return static_cast<uint8_t>(sign | 0x7E);   // saturate
    if (q < 8.0) return static_cast<uint8_t>(sign | static_cast<uint8_t>(q));       // subnormal
    return static_cast<uint8_t>(sign | ((e + 7) << 3) | (static_cast<int>(q) - 8));
}

double e4m3_to_double(uint8_t c) {
    const double sign = (c & 0x80) ? -1.0 : 1.0;
    const int ef = (c >> 3) & 0xF, m = c & 7;
    if (ef == 0xF && m == 7) return std::numeric_limits<double>::quiet_NaN();
    if (ef == 0) return sign * std::ldexp(static_cast<double>(m), -9);
    return sign * std::ldexp(1.0 + m / 8.0, ef - 7);
}

}  // namespace

extern "C" {

// RMSNorm over the d channels of one entry, then RoPE on its last rope_dim channels at
// position `pos`, then one RNE rounding to bf16 (shared by both compressor forms).
static void finish_entry(double* x, int d, int rope_dim, double theta, double eps,
                         const float* gamma, double pos, uint16_t* out_row, double* out_f64_row) {
    // RMSNorm over all d channels
    double ms = 0.0;
    for (int c = 0; c < d; ++c) ms += x[c] * x[c];
    ms /= d;
    double inv = 1.0 / std::sqrt(ms + eps);
    for (int c = 0; c < d; ++c) x[c] = x[c] * inv * static_cast<double>(gamma[c]);
    // RoPE on the last rope_dim dims, pair j = (d0, d0+1), d0 = d - rope_dim + 2j
    for (int j = 0; j < rope_dim / 2; ++j) {
        const int d0 = d - rope_dim + 2 * j;
        const double freq = std::pow(theta, -2.0 * j / rope_dim);
        const double ang = pos * freq;
        const double cs = std::cos(ang), sn = std::sin(ang);
        const double e = x[d0], o = x[d0 + 1];
        x[d0] = e * cs - o * sn;
        x[d0 + 1] = e * sn + o * cs;
    }
    for (int c = 0; c < d; ++c) {
        out_row[c] = double_to_bf16(x[c]);
        if (out_f64_row) out_f64_row[c] = x[c];
    }
}

// ---------------------------------------------------------------------------
// a1/a2. Block compressor + RMSNorm + partial RoPE.
//
// [A] compressor_reduce.cu, hca_compress_reduce_kernel (plain per-block form) with the
// fix of [B]/[C] compressor_reduce.cu hunks and commit message "Fix two correctness
// bugs": the positional bias goes on the softmax logits Z + B only, never on C.
// [A] compressor_reduce.cu, apply_kv_norm_kernel: y = x / sqrt(mean(x^2) + eps) * g.
// [A] PERFORMANCE_AUDIT.md "P5": interleaved pairs (even, odd) of the last rope_dim
// dims; the inverse shown there is  e' = e c + o s,  o' = -e s + o c,  so the forward
// rotation is  e' = e c - o s,  o' = e s + o c.  [B] single_shot_inference.py
// eager_attention: RoPE is applied to the rope part of the compressed entry at its
// position after compression and norm.
//
// Layout: C, Z [B, T, d] bf16; bias [ratio, d] fp32; gamma [d] fp32; pos0 [B] int64
// (absolute position of token 0); out [B, T/ratio, d] bf16; out_f64 same shape, may be
// null. Entry b of sequence s sits at position pos0[s] + b*ratio.
// Returns 0, or -1 on bad sizes.
int oracle_compress(const uint16_t* C, const uint16_t* Z, const float* bias,
                    const float* gamma, const int64_t* pos0, int B, int T, int d,
                    int ratio, int rope_dim, double theta, double eps,
                    uint16_t* out, double* out_f64) {
    if (B < 0 || T < 0 || d <= 0 || ratio <= 0 || T % ratio != 0) return -1;
    if (rope_dim < 0 || rope_dim > d || rope_dim % 2 != 0) return -1;
    const int nb = T / ratio;
    std::vector<double> x(d);
    for (int s = 0; s < B; ++s) {
        for (int b = 0; b < nb; ++b) {
            // softmax over the ratio tokens of the block, per channel, then weighted sum of C
            for (int c = 0; c < d; ++c) {
                double m = -std::numeric_limits<double>::infinity();
                for (int t = 0; t < ratio; ++t) {
                    size_t at = (static_cast<size_t>(s) * T + static_cast<size_t>(b) * ratio + t) * d + c;
                    double a = bf16_to_double(Z[at]) + static_cast<double>(bias[static_cast<size_t>(t) * d + c]);
                    m = std::max(m, a);
                }
                double num = 0.0, den = 0.0;
                for (int t = 0; t < ratio; ++t) {
                    size_t at = (static_cast<size_t>(s) * T + static_cast<size_t>(b) * ratio + t) * d + c;
                    double a = bf16_to_double(Z[at]) + static_cast<double>(bias[static_cast<size_t>(t) * d + c]);
                    double e = std::exp(a - m);
                    den += e;
                    num += e * bf16_to_double(C[at]);   // no bias on C
                }
                x[c] = num / den;
            }
            const double pos = static_cast<double>(pos0[s] + static_cast<int64_t>(b) * ratio);
            const size_t row = static_cast<size_t>(s) * nb + b;
            finish_entry(x.data(), d, rope_dim, theta, eps, gamma, pos, out + row * d,
                         out_f64 ? out_f64 + row * d : nullptr);
        }
    }
    return 0;
}

// ---------------------------------------------------------------------------
// a1 (CSA form). Overlapped two-stream block compressor.
//
// [A] compressor_reduce.cu, "CSA compressor reduce kernel": the projections carry 2d channels,
// stream a (channels [0, d)) and stream b (channels [d, 2d)); entry i pools the ratio tokens
// of block i - 1 from stream a together with the ratio tokens of block i from stream b (entry
// 0, which has no block before it, pools only its own block from stream b), with one softmax
// over all pooled logits per channel and the weighted sum of the matching C values. The
// positional bias has 2d columns: token t of either part takes bias row t of its stream's
// half, on the logits only ([B] commit "Fix two correctness bugs", item 1). RMSNorm and RoPE
// follow as for the plain compressor, at the position of entry i's own first token.
//
// C, Z [B, T, 2d] bf16; bias [ratio, 2d] fp32; prev_C, prev_Z [B, ratio, 2d] or null: the
// block just before the first block of C (its stream a feeds entry 0); null means entry 0 is
// the sequence's first block. out [B, T/ratio, d].
int oracle_compress_overlap(const uint16_t* C, const uint16_t* Z, const uint16_t* prev_C,
                            const uint16_t* prev_Z, const float* bias, const float* gamma,
                            const int64_t* pos0, int B, int T, int d, int ratio, int rope_dim,
                            double theta, double eps, uint16_t* out, double* out_f64) {
    if (B < 0 || T < 0 || d <= 0 || ratio <= 0 || T % ratio != 0) return -1;
    if (rope_dim < 0 || rope_dim > d || rope_dim % 2 != 0) return -1;
    if ((prev_C == nullptr) != (prev_Z == nullptr)) return -1;
    const int nb = T / ratio, w = 2 * d;
    std::vector<double> x(d), lg(2 * static_cast<size_t>(ratio)), val(2 * static_cast<size_t>(ratio));
    for (int s = 0; s < B; ++s) {
        for (int i = 0; i < nb; ++i) {
            for (int c = 0; c < d; ++c) {
                int n = 0;
                // stream a: the previous block's tokens
                if (i > 0 || prev_C) {
                    for (int t = 0; t < ratio; ++t) {
                        const size_t at = i > 0
                            ? (static_cast<size_t>(s) * T + static_cast<size_t>(i - 1) * ratio + t) * w + c
                            : (static_cast<size_t>(s) * ratio + t) * w + c;
                        const uint16_t zb = i > 0 ? Z[at] : prev_Z[at];
                        const uint16_t cb = i > 0 ? C[at] : prev_C[at];
                        lg[n] = bf16_to_double(zb) + static_cast<double>(bias[static_cast<size_t>(t) * w + c]);
                        val[n] = bf16_to_double(cb);
                        ++n;
                    }
                }
                // stream b: this block's tokens
                for (int t = 0; t < ratio; ++t) {
                    const size_t at = (static_cast<size_t>(s) * T + static_cast<size_t>(i) * ratio + t) * w + d + c;
                    lg[n] = bf16_to_double(Z[at]) + static_cast<double>(bias[static_cast<size_t>(t) * w + d + c]);
                    val[n] = bf16_to_double(C[at]);
                    ++n;
                }
                double mx = -std::numeric_limits<double>::infinity();
                for (int u = 0; u < n; ++u) mx = std::max(mx, lg[u]);
                double num = 0.0, den = 0.0;
                for (int u = 0; u < n; ++u) {
                    const double e = std::exp(lg[u] - mx);
                    den += e;
                    num += e * val[u];
                }
                x[c] = num / den;
            }
            const double pos = static_cast<double>(pos0[s]) + static_cast<double>(i) * ratio;
            const size_t row = static_cast<size_t>(s) * nb + i;
            finish_entry(x.data(), d, rope_dim, theta, eps, gamma, pos, out + row * d,
                         out_f64 ? out_f64 + row * d : nullptr);
        }
    }
    return 0;
}

// ---------------------------------------------------------------------------
// a3. Lightning-indexer score (MQA form).
//
// [A] ARCHITECTURE_AND_MEMORY_AUDIT.md "F3 — The scoring einsum has the wrong algebra":
// I[t,s] = sum_h w[t,h] * ReLU(q[t,h,:] . K[s,:]), one key per compressed block shared by
// every indexer head; no scale, no softmax. [A] "F1": keys are 128 wide.
//
// Layout: q [B, n_q, H, Di] bf16; w [B, n_q, H] fp32; keys [B, max_comp, Di] bf16;
// n_comp [B]; q_pos [B, n_q] int64 or null (decode: every one of the n_comp entries is
// visible). scores [B, n_q, max_comp] double: entries at s >= n_vis are set to -inf.
// n_vis [B, n_q] receives the visible count.
int oracle_index_scores(const uint16_t* q, const float* w, const uint16_t* keys,
                        const int32_t* n_comp, const int64_t* q_pos, int B, int n_q,
                        int H, int Di, int max_comp, int ratio, double* scores,
                        int32_t* n_vis) {
    if (B < 0 || n_q < 0 || H <= 0 || Di <= 0 || max_comp < 0 || ratio <= 0) return -1;
    for (int b = 0; b < B; ++b) {
        if (n_comp[b] < 0 || n_comp[b] > max_comp) return -1;
        for (int t = 0; t < n_q; ++t) {
            const size_t row = static_cast<size_t>(b) * n_q + t;
            int64_t nv = q_pos ? visible_entries(n_comp[b], q_pos[row], ratio) : n_comp[b];
            n_vis[row] = static_cast<int32_t>(nv);
            double* out = scores + row * max_comp;
            for (int s = 0; s < max_comp; ++s) out[s] = -std::numeric_limits<double>::infinity();
            for (int64_t s = 0; s < nv; ++s) {
                const uint16_t* k = keys + (static_cast<size_t>(b) * max_comp + s) * Di;
                double total = 0.0;
                for (int h = 0; h < H; ++h) {
                    const uint16_t* qh = q + (row * H + h) * Di;
                    double dot = 0.0;
                    for (int i = 0; i < Di; ++i) dot += bf16_to_double(qh[i]) * bf16_to_double(k[i]);
                    total += static_cast<double>(w[row * H + h]) * std::max(0.0, dot);
                }
                out[s] = total;
            }
        }
    }
    return 0;
}

// ---------------------------------------------------------------------------
// a4. Per-token top-k.
//
// [A] ARCHITECTURE_AND_MEMORY_AUDIT.md "F3": tk = min(top_k, n_comp), total.topk(tk).
// [C] GETTING+CUDAGRAPH_READY.md "SECTION C" item 3: the index list has a fixed length
// top_k; entries past tk are padding and are masked, never clamped.
// Tie rule (the pages leave it open; this library fixes it): equal scores -> the lower
// index ranks first. Output order: the selected indices in ascending order, then -1.
//
// Layout: scores [rows, max_comp] (double or float); n_vis [rows]; idx [rows, top_k].
static void topk_rows_impl(const double* scores, const int32_t* n_vis, int rows,
                           int max_comp, int top_k, int32_t* idx) {
    std::vector<int32_t> order;
    for (int r = 0; r < rows; ++r) {
        const double* s = scores + static_cast<size_t>(r) * max_comp;
        const int n = n_vis[r];
        order.resize(n);
        for (int i = 0; i < n; ++i) order[i] = i;
        std::sort(order.begin(), order.end(), [s](int32_t a, int32_t b) {
            if (s[a] != s[b]) return s[a] > s[b];
            return a < b;
        });
        const int tk = std::min(top_k, n);
        std::vector<int32_t> chosen(order.begin(), order.begin() + tk);
        std::sort(chosen.begin(), chosen.end());
        int32_t* o = idx + static_cast<size_t>(r) * top_k;
        for (int j = 0; j < top_k; ++j) o[j] = j < tk ? chosen[j] : -1;
    }
}

int oracle_topk(const double* scores, const int32_t* n_vis, int rows, int max_comp,
                int top_k, int32_t* idx) {
    if (rows < 0 || max_comp < 0 || top_k <= 0) return -1;
    for (int r = 0; r < rows; ++r)
        if (n_vis[r] < 0 || n_vis[r] > max_comp) return -1;
    topk_rows_impl(scores, n_vis, rows, max_comp, top_k, idx);
    return 0;
}

// Same selection on fp32 scores (the step taken alone, on caller-given scores).
int oracle_topk_f32(const float* scores, const int32_t* n_vis, int rows, int max_comp,
                    int top_k, int32_t* idx) {
    if (rows < 0 || max_comp < 0 || top_k <= 0) return -1;
    std::vector<double> wide(static_cast<size_t>(rows) * max_comp);
    for (size_t i = 0; i < wide.size(); ++i) wide[i] = static_cast<double>(scores[i]);
    return oracle_topk(wide.data(), n_vis, rows, max_comp, top_k, idx);
}

// ---------------------------------------------------------------------------
// a5 + a6. Gather into a fixed buffer, then MQA attention with a per-head sink.
//
// Gather: [A] commit "C2": one pre-allocated buffer of (top_k + window) rows receives the
// selected compressed rows and the sliding-window rows; [A] ARCHITECTURE_AND_MEMORY_AUDIT.md
// "B2": CSA concatenates comp_kv[topk] with the window, HCA (ratio > 4) concatenates every
// compressed entry with the window.
// Attention: [A] fmha_6warp_tma_multirow_multitile.cuh, "Sink bias correction": the sink
// is one extra logit per head, already in the scaled domain, that adds to the softmax
// denominator and has no value row. [A] PERFORMANCE_AUDIT.md "P4": V is the same tensor as
// K (shared KV). [B] single_shot_inference.py eager_attention: scale = 1/sqrt(hd).
//
//   s_j = scale * q_h . kv_j,   m = max(max_j s_j, sink_h)
//   o_h = sum_j e^(s_j - m) kv_j / (sum_j e^(s_j - m) + e^(sink_h - m))
//
// Layout: q [B, n_q, H, D] bf16; sink [H] fp32; comp_kv [B, max_comp, D] bf16; n_comp [B];
// idx [B, n_q, top_k] int32 or null (dense over every visible entry; then top_k must equal
// max_comp); q_pos [B, n_q] int64 or null (decode: all n_comp visible);
// win [B, win_rows, D] bf16 holds the most recent tokens in order, the n_q query tokens
// last; win_len [B] valid rows. Query t (absolute index q_abs[t] of n_q_total, or t of n_q
// when q_abs is null) sees the `window` rows ending at its own row:
//   rows [qa + win_len - n_q_total - window + 1,  qa + win_len - n_q_total]  within [0, win_len).
// out [B, n_q, H, D] bf16; out_f64 may be null; gather [B, n_q, top_k + window, D] bf16 or
// null: slot j < top_k holds comp_kv[idx[j]] (zeros for -1), slot top_k + i holds the i-th
// window row (zeros past the window length).
int oracle_sparse_attn(const uint16_t* q, const float* sink, const uint16_t* comp_kv,
                       const int32_t* n_comp, const int32_t* idx, const int64_t* q_pos,
                       const uint16_t* win, const int32_t* win_len, const int32_t* q_abs,
                       int B, int n_q, int n_q_total, int H, int D, int max_comp, int top_k,
                       int window, int win_rows, int ratio, double scale,
                       uint16_t* out, double* out_f64, uint16_t* gather) {
    if (B < 0 || n_q < 0 || H <= 0 || D <= 0 || top_k <= 0 || window < 0 || ratio <= 0) return -1;
    if (!idx && top_k != max_comp) return -1;
    const int slots = top_k + window;
    std::vector<const uint16_t*> rows;
    std::vector<double> kv;   // widened rows, [n_rows, D]
    std::vector<double> sc;
    for (int b = 0; b < B; ++b) {
        if (n_comp[b] < 0 || n_comp[b] > max_comp) return -1;
        if (win_len[b] < 0 || win_len[b] > win_rows) return -1;
        for (int t = 0; t < n_q; ++t) {
            const size_t qrow = static_cast<size_t>(b) * n_q + t;
            const int64_t nv = q_pos ? visible_entries(n_comp[b], q_pos[qrow], ratio) : n_comp[b];
            rows.clear();
            uint16_t* g = gather ? gather + qrow * slots * static_cast<size_t>(D) : nullptr;
            if (g) std::fill(g, g + static_cast<size_t>(slots) * D, static_cast<uint16_t>(0));
            // compressed part of the gather
            for (int j = 0; j < top_k; ++j) {
                int64_t e;
                if (idx) {
                    e = idx[qrow * top_k + j];
                    if (e < 0) continue;                       // padding: masked
                    if (e >= nv) return -2;                    // not a visible entry
                } else {
                    e = j;
                    if (e >= nv) continue;
                }
                const uint16_t* src = comp_kv + (static_cast<size_t>(b) * max_comp + e) * D;
                rows.push_back(src);
                if (g) std::memcpy(g + static_cast<size_t>(j) * D, src, sizeof(uint16_t) * D);
            }
            // sliding-window part of the gather
            const int64_t qa = q_abs ? q_abs[t] : t;
            const int64_t hi = qa + win_len[b] - n_q_total;          // the query's own row
            int64_t lo = hi - window + 1;
            if (lo < 0) lo = 0;
            int slot = 0;
            for (int64_t r = lo; r <= hi && r < win_len[b] && slot < window; ++r, ++slot) {
                const uint16_t* src = win + (static_cast<size_t>(b) * win_rows + r) * D;
                rows.push_back(src);
                if (g) std::memcpy(g + static_cast<size_t>(top_k + slot) * D, src, sizeof(uint16_t) * D);
            }
            const size_t n_rows = rows.size();
            kv.assign(n_rows * D, 0.0);
            for (size_t r = 0; r < n_rows; ++r)
                for (int i = 0; i < D; ++i) kv[r * D + i] = bf16_to_double(rows[r][i]);
            sc.assign(n_rows, 0.0);
            for (int h = 0; h < H; ++h) {
                const uint16_t* qh = q + (qrow * H + h) * D;
                const double sk = static_cast<double>(sink[h]);
                double m = sk;
                for (size_t r = 0; r < n_rows; ++r) {
                    double dot = 0.0;
                    for (int i = 0; i < D; ++i) dot += bf16_to_double(qh[i]) * kv[r * D + i];
                    sc[r] = scale * dot;
                    m = std::max(m, sc[r]);
                }
                double den = std::exp(sk - m);
                std::vector<double> num(D, 0.0);
                for (size_t r = 0; r < n_rows; ++r) {
                    const double p = std::exp(sc[r] - m);
                    den += p;
                    for (int i = 0; i < D; ++i) num[i] += p * kv[r * D + i];
                }
                for (int i = 0; i < D; ++i) {
                    const double o = num[i] / den;
                    const size_t at = (qrow * H + h) * D + i;
                    out[at] = double_to_bf16(o);
                    if (out_f64) out_f64[at] = o;
                }
            }
        }
    }
    return 0;
}

// Sizing of the compressed cache for a context length.
// [A] commit "C1": max_comp = (max_context + compress_ratio - 1) // ratio.
int64_t oracle_max_comp(int64_t max_context, int ratio) {
    if (ratio <= 0 || max_context < 0) return -1;
    return (max_context + ratio - 1) / ratio;
}

// Visible count, exported so tests can pin the causal rule on its own.
int64_t oracle_visible_entries(int64_t n_comp, int64_t p, int ratio) {
    return visible_entries(n_comp, p, ratio);
}

// bf16 rounding, exported so tests can pin it against exhaustive float checks.
uint16_t oracle_double_to_bf16(double x) { return double_to_bf16(x); }

// ---------------------------------------------------------------------------
// Inverse RoPE on the attention output.
//
// [B] single_shot_inference.py eager_attention: after FMHA, "Inverse RoPE" is applied to the
// attention output at the query positions, on the last rope_dim dims of every head. The
// rotation is the inverse of the one the compressor applies ([A] PERFORMANCE_AUDIT.md "P5"
// shows it: e' = e c + o s, o' = -e s + o c, pairs (even, odd), angle pos * theta^(-2j/rope_dim)).
//
// x [rows, heads, D] double (rows = query rows, e.g. B * n_q); pos [rows] int64.
// out [rows, heads, D] bf16 bits (one RNE rounding); out_f64 may be null.
int oracle_inverse_rope(const double* x, const int64_t* pos, int rows, int heads, int D,
                        int rope_dim, double theta, uint16_t* out, double* out_f64) {
    if (rows < 0 || heads <= 0 || D <= 0 || rope_dim < 0 || rope_dim > D || rope_dim % 2 != 0) return -1;
    std::vector<double> v(D);
    for (int r = 0; r < rows; ++r) {
        for (int h = 0; h < heads; ++h) {
            const size_t base = (static_cast<size_t>(r) * heads + h) * D;
            for (int i = 0; i < D; ++i) v[i] = x[base + i];
            for (int j = 0; j < rope_dim / 2; ++j) {
                const int e0 = D - rope_dim + 2 * j;
                const double freq = std::pow(theta, -(2.0 * j) / rope_dim);
                const double ang = static_cast<double>(pos[r]) * freq;
                const double cs = std::cos(ang), sn = std::sin(ang);
                const double ev = v[e0], ov = v[e0 + 1];
                v[e0] = ev * cs + ov * sn;
                v[e0 + 1] = -ev * sn + ov * cs;
            }
            for (int i = 0; i < D; ++i) {
                out[base + i] = double_to_bf16(v[i]);
                if (out_f64) out_f64[base + i] = v[i];
            }
        }
    }
    return 0;
}

// ---------------------------------------------------------------------------
// FP8 index keys: row quantization and scoring on the quantized rows.
//
// [B] single_shot_inference.py (indexer): "Indexer keys are stored as FP8_E4M3 in the KV
// cache", scored on the FP8 tensor-core path. The pages fix no scale; the reading taken: one
// fp32 scale per row (a key row, or one head of a query), scale = amax / 448 computed in fp32
// (1 for an all-zero row), code = E4M3(x / scale) with the division in fp32, so that the codes
// are a definite function of the fp32 inputs.
//
// x [rows, dim] fp32 -> q [rows, dim] E4M3 codes, scale [rows] fp32.
int oracle_quantize_rows_e4m3(const float* x, int rows, int dim, uint8_t* q, float* scale) {
    if (rows < 0 || dim <= 0) return -1;
    for (int r = 0; r < rows; ++r) {
        const float* xr = x + static_cast<size_t>(r) * dim;
        float amax = 0.f;
        for (int i = 0; i < dim; ++i) amax = std::max(amax, std::fabs(xr[i]));
        const float sc = amax > 0.f ? amax / 448.0f : 1.0f;
        scale[r] = sc;
        for (int i = 0; i < dim; ++i) {
            const float v = xr[i] / sc;                      // fp32 division
            q[static_cast<size_t>(r) * dim + i] = e4m3_from_double(static_cast<double>(v));
        }
    }
    return 0;
}

// ---------------------------------------------------------------------------
// Mixed FP8 / bf16 compressed KV cache.
//
// [B] single_shot_inference.py eager_attention, "Compressor -> compressed KV (mixed storage:
// FP8 + BF16 RoPE)": the first dim - rope_dim channels of a compressed entry (the part
// without RoPE) are kept as FP8 E4M3 with one scale per entry, the last rope_dim channels as
// bf16, and the attention reads both parts back. The pages fix no scale rule; the readings
// taken: codes and scale of the part without RoPE as in oracle_quantize_rows_e4m3 (amax of
// that part only / 448, fp32); the RoPE part is the bf16 RNE of the fp32 entry; a gathered
// entry is dequantized to bf16 before the attention products, each channel
// bf16( fp32( e4m3(code) * scale ) ), the RoPE channels as stored.
//
// x [rows, dim] fp32 -> nope [rows, dim - rope_dim] codes, scale [rows] fp32,
// rope [rows, rope_dim] bf16 bits.
int oracle_quantize_kv_mixed(const float* x, int rows, int dim, int rope_dim, uint8_t* nope,
                             float* scale, uint16_t* rope) {
    if (rows < 0 || dim <= 0 || rope_dim < 0 || rope_dim >= dim) return -1;
    const int nd = dim - rope_dim;
    for (int r = 0; r < rows; ++r) {
        const float* xr = x + static_cast<size_t>(r) * dim;
        float amax = 0.f;
        for (int i = 0; i < nd; ++i) amax = std::max(amax, std::fabs(xr[i]));
        const float sc = amax > 0.f ? amax / 448.f : 1.f;   // as oracle_quantize_rows_e4m3
        scale[r] = sc;
        for (int i = 0; i < nd; ++i)
            nope[static_cast<size_t>(r) * nd + i] = e4m3_from_double(static_cast<double>(xr[i] / sc));
        for (int i = 0; i < rope_dim; ++i)
            rope[static_cast<size_t>(r) * rope_dim + i] = double_to_bf16(static_cast<double>(xr[nd + i]));
    }
    return 0;
}

// The bf16 rows the attention multiplies: [rows, dim] bf16 bits from the mixed storage.
int oracle_dequant_kv_mixed(const uint8_t* nope, const float* scale, const uint16_t* rope,
                            int rows, int dim, int rope_dim, uint16_t* out) {
    if (rows < 0 || dim <= 0 || rope_dim < 0 || rope_dim >= dim) return -1;
    const int nd = dim - rope_dim;
    for (int r = 0; r < rows; ++r) {
        uint16_t* o = out + static_cast<size_t>(r) * dim;
        for (int i = 0; i < nd; ++i) {
            const float v = static_cast<float>(e4m3_to_double(nope[static_cast<size_t>(r) * nd + i])) * scale[r];
            o[i] = double_to_bf16(static_cast<double>(v));      // fp32 product, then bf16
        }
        for (int i = 0; i < rope_dim; ++i) o[nd + i] = rope[static_cast<size_t>(r) * rope_dim + i];
    }
    return 0;
}

double oracle_e4m3_to_double(uint8_t c) { return e4m3_to_double(c); }
uint8_t oracle_e4m3_from_double(double x) { return e4m3_from_double(x); }

// The indexer score of the dequantized rows (the a3 definition on q_scale * q and
// k_scale * k):  I[t, j] = sum_h w[t, h] * ReLU( (q_scale[t,h] q[t,h,:]) . (k_scale[j] k[j,:]) ).
// q [B, n_q, H, Di] and k [B, max_comp, Di] E4M3 codes; q_scale [B, n_q, H], k_scale
// [B, max_comp]; the rest as oracle_index_scores.
int oracle_index_scores_fp8(const uint8_t* q, const float* q_scale, const float* w,
                            const uint8_t* keys, const float* k_scale, const int32_t* n_comp,
                            const int64_t* q_pos, int B, int n_q, int H, int Di, int max_comp,
                            int ratio, double* scores, int32_t* n_vis) {
    if (B < 0 || n_q < 0 || H <= 0 || Di <= 0 || max_comp < 0 || ratio <= 0) return -1;
    std::vector<double> qd(static_cast<size_t>(H) * Di), kd(Di);
    for (int b = 0; b < B; ++b) {
        if (n_comp[b] < 0 || n_comp[b] > max_comp) return -1;
        for (int t = 0; t < n_q; ++t) {
            const size_t row = static_cast<size_t>(b) * n_q + t;
            const int64_t nv = q_pos ? visible_entries(n_comp[b], q_pos[row], ratio) : n_comp[b];
            n_vis[row] = static_cast<int32_t>(nv);
            for (int h = 0; h < H; ++h)
                for (int i = 0; i < Di; ++i)
                    qd[static_cast<size_t>(h) * Di + i] =
                        static_cast<double>(q_scale[row * H + h]) * e4m3_to_double(q[(row * H + h) * Di + i]);
            for (int j = 0; j < max_comp; ++j) {
                double& out = scores[row * max_comp + j];
                if (j >= nv) {
                    out = -std::numeric_limits<double>::infinity();
                    continue;
                }
                const size_t kr = static_cast<size_t>(b) * max_comp + j;
                for (int i = 0; i < Di; ++i)
                    kd[i] = static_cast<double>(k_scale[kr]) * e4m3_to_double(keys[kr * Di + i]);
                double acc = 0.0;
                for (int h = 0; h < H; ++h) {
                    double dot = 0.0;
                    for (int i = 0; i < Di; ++i) dot += qd[static_cast<size_t>(h) * Di + i] * kd[i];
                    acc += static_cast<double>(w[row * H + h]) * (dot > 0.0 ? dot : 0.0);   // ReLU
                }
                out = acc;
            }
        }
    }
    return 0;
}

}  // extern "C"

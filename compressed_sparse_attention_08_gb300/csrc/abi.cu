// C ABI of the CSA library: host-side argument checks (before any CUDA call), workspace
// sizing, dispatch to the kernels on the caller's stream, and small utilities.
// No entry point allocates, frees, synchronises or reads device memory on the host,
// except dsv4_read_error_word, which exists for tests and diagnostics.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "internal.h"

namespace dsv4 {
namespace {

thread_local int g_launches = 0;
thread_local int g_last_launches = 0;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool dev_ptr_ok(const void* p) { return p != nullptr && aligned16(p); }
bool opt_ptr_ok(const void* p) { return p == nullptr || aligned16(p); }
// Memory the GPU can address: device, pinned (page-locked) host or managed memory.
bool gpu_addressable(const void* p) {
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();                      // (not a sticky error: clear it)
        return false;
    }
    return at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeHost || at.type == cudaMemoryTypeManaged;
}

// The library holds sm_103a code only: any other device is refused before a launch.
int device_check() {
    // 0 unknown, 1 ok, 2 unsupported (atomic: first calls may come from several host threads)
    static std::atomic<int> ok_for_device[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return DSV4_ERR_UNSUPPORTED;
    if (dev < 64 && ok_for_device[dev].load(std::memory_order_relaxed) == 1) return DSV4_OK;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return DSV4_ERR_UNSUPPORTED;
    const int res = major == 10 && minor == 3 ? DSV4_OK : DSV4_ERR_UNSUPPORTED;
    if (dev < 64) ok_for_device[dev].store(res == DSV4_OK ? 1 : 2, std::memory_order_relaxed);
    return res;
}

bool compress_ok(const dsv4_compress_args* a) {
    if (!a) return false;
    if (!dev_ptr_ok(a->C) || !dev_ptr_ok(a->Z) || !dev_ptr_ok(a->bias) || !dev_ptr_ok(a->gamma) ||
        !dev_ptr_ok(a->pos0) || !dev_ptr_ok(a->out) || !opt_ptr_ok(a->out_row0))
        return false;
    if (a->batch < 0 || a->tokens < 0 || a->ratio < 1 || a->dim < 2 || a->dim > 1024) return false;
    if (a->tokens % a->ratio != 0) return false;
    if (a->rope_dim < 0 || a->rope_dim > a->dim || a->rope_dim > 128 || (a->rope_dim & 1)) return false;
    if (a->out_rows < 1) return false;
    if (!a->out_row0 && a->out_rows < a->tokens / a->ratio) return false;
    if (!(a->eps >= 0.f) || !std::isfinite(a->eps) || !std::isfinite(a->rope_theta) || a->rope_theta <= 0.0)
        return false;
    if (a->overlap != 0 && a->overlap != 1) return false;
    if ((a->prev_C == nullptr) != (a->prev_Z == nullptr)) return false;
    if (a->prev_C && (!a->overlap || !dev_ptr_ok(a->prev_C) || !dev_ptr_ok(a->prev_Z))) return false;
    if (a->out_fp8 < 0 || a->out_fp8 > 2) return false;
    if (a->out_fp8 ? !dev_ptr_ok(a->out_scale) : a->out_scale != nullptr) return false;
    // mixed storage: the RoPE part in out_rope (none when rope_dim is 0)
    if (a->out_fp8 == 2 ? (a->rope_dim > 0 ? !dev_ptr_ok(a->out_rope) : a->out_rope != nullptr)
                        : a->out_rope != nullptr)
        return false;
    if (a->out_fp8 == 2 && a->rope_dim >= a->dim) return false;
    return true;
}

bool index_ok(const dsv4_index_args* a) {
    if (!a) return false;
    if (!dev_ptr_ok(a->q) || !dev_ptr_ok(a->w) || !dev_ptr_ok(a->keys) || !dev_ptr_ok(a->n_comp) ||
        !dev_ptr_ok(a->idx_out) || !opt_ptr_ok(a->q_pos) || !opt_ptr_ok(a->scores_out))
        return false;
    if (a->batch < 0 || a->n_q < 1 || a->dim != 128) return false;
    if (a->heads < 8 || a->heads > 64 || (a->heads & 7)) return false;
    if (a->max_comp < 1 || a->top_k < 1 || a->top_k > a->max_comp || a->ratio < 1) return false;
    if (static_cast<long long>(a->batch) * a->n_q > (1ll << 30)) return false;
    if (static_cast<long long>(a->batch) * a->n_q * a->heads > (1ll << 31) - 1) return false;
    if (a->key_fp8 != 0 && a->key_fp8 != 1) return false;
    if (a->key_fp8 ? (!dev_ptr_ok(a->q_scale) || !dev_ptr_ok(a->key_scale))
                   : (a->q_scale != nullptr || a->key_scale != nullptr))
        return false;
    return true;
}

bool topk_ok(const dsv4_topk_args* a) {
    if (!a) return false;
    if (!dev_ptr_ok(a->scores) || !dev_ptr_ok(a->n_vis) || !dev_ptr_ok(a->idx_out)) return false;
    if (a->rows < 0 || a->max_comp < 1 || a->top_k < 1 || a->top_k > a->max_comp) return false;
    return true;
}

bool attn_ok(const dsv4_attn_args* a) {
    if (!a) return false;
    if (!dev_ptr_ok(a->q) || !dev_ptr_ok(a->sink) || !dev_ptr_ok(a->n_comp) ||
        !dev_ptr_ok(a->win) || !dev_ptr_ok(a->win_len) || !dev_ptr_ok(a->out) ||
        !opt_ptr_ok(a->idx) || !opt_ptr_ok(a->q_pos) || !opt_ptr_ok(a->gather))
        return false;
    if (a->batch < 0 || a->n_q < 1) return false;
    if (a->dim != 128 && a->dim != 256 && a->dim != 512) return false;
    if (a->heads < 1 || a->heads > 64 || (a->heads > 16 && a->heads % 16 != 0)) return false;
    if (a->max_comp < 1 || a->top_k < 1 || a->window < 0 || a->win_rows < 1 || a->ratio < 1) return false;
    if (a->idx ? a->top_k > a->max_comp : a->top_k != a->max_comp) return false;
    if (!std::isfinite(a->scale)) return false;
    // the compressed rows: bf16 in comp_kv, or the mixed FP8 / bf16 storage
    if (a->kv_fp8 == 0) {
        if (!dev_ptr_ok(a->comp_kv) || a->kv_nope || a->kv_scale || a->kv_rope) return false;
    } else if (a->kv_fp8 == 1) {
        if (a->comp_kv || !dev_ptr_ok(a->kv_nope) || !dev_ptr_ok(a->kv_scale) || !dev_ptr_ok(a->kv_rope))
            return false;
        if (a->kv_rope_dim < 8 || a->kv_rope_dim % 8 || a->kv_rope_dim > a->dim - 8) return false;
    } else {
        return false;
    }
    if (static_cast<long long>(a->batch) * a->n_q > 65535ll) return false;   // grid.y
    if (a->out_rope_pos) {
        if (!opt_ptr_ok(a->out_rope_pos) || a->out_rope_dim < 2 || (a->out_rope_dim & 1) ||
            a->out_rope_dim > a->dim || a->out_rope_dim > 128)
            return false;
        if (!std::isfinite(a->out_rope_theta) || a->out_rope_theta <= 0.0) return false;
    }
    return true;
}

uint32_t* eword_of(void* ws) { return static_cast<uint32_t*>(ws); }
uint8_t* body_of(void* ws) { return static_cast<uint8_t*>(ws) + kWsHeader; }

struct LaunchScope {
    LaunchScope() { g_launches = 0; }
    ~LaunchScope() { g_last_launches = g_launches; }
};

}  // namespace

void count_launch(int n) { g_launches += n; }

namespace {
std::atomic<int> g_wait_fault{DSV4_WAIT_FAULT_NONE};
std::atomic<unsigned> g_wait_limit_us{0};
}  // namespace

WaitCtl wait_ctl(int which) {
    WaitCtl c{0, kDefaultWaitNs};
    if (which != DSV4_WAIT_FAULT_NONE && g_wait_fault.load() == which) {
        c.fault = 1;
        const unsigned us = g_wait_limit_us.load();
        if (us) c.wait_ns = 1000ull * us;
    }
    return c;
}

cudaError_t once_per_device(const void* kernel, int kind, const std::function<cudaError_t()>& set) {
    struct Key { const void* kernel; int dev, kind; };
    static std::mutex mu;
    static std::vector<Key> done;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) dev = -1;
    std::lock_guard<std::mutex> lock(mu);
    for (const Key& k : done)
        if (k.kernel == kernel && k.dev == dev && k.kind == kind) return cudaSuccess;
    const cudaError_t e = set();
    // a failed setting is not recorded: the next call tries again (and fails its launch)
    if (e == cudaSuccess) done.push_back(Key{kernel, dev, kind});
    else cudaGetLastError();       // the error is returned here, not left for a later launch
    return e;
}

cudaError_t prefer_max_shared(const void* kernel) {
    return once_per_device(kernel, kAttrCarveout, [kernel] {
        return cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                                    cudaSharedmemCarveoutMaxShared);
    });
}

int sm_count() {
    static std::atomic<int> cache[64] = {};   // (atomic: first calls may come from several threads)
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
    if (dev < 64) {
        const int c = cache[dev].load(std::memory_order_relaxed);
        if (c) return c;
    }
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (dev < 64) cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

}  // namespace dsv4

using namespace dsv4;

extern "C" {

int dsv4_copy_async(void* dst, const void* src, size_t bytes, dsv4_stream_t stream) {
    LaunchScope scope;
    if (bytes == 0) return DSV4_OK;
    if (!dev_ptr_ok(dst) || !dev_ptr_ok(src) || bytes % 16 != 0) return DSV4_ERR_INVALID_ARG;
    const uintptr_t d = reinterpret_cast<uintptr_t>(dst), s = reinterpret_cast<uintptr_t>(src);
    if (d < s + bytes && s < d + bytes) return DSV4_ERR_INVALID_ARG;   // overlapping ranges
    if (!gpu_addressable(dst) || !gpu_addressable(src)) return DSV4_ERR_INVALID_ARG;
    if (int rc = device_check()) return rc;
    return launch_copy(dst, src, bytes, reinterpret_cast<cudaStream_t>(stream));
}

const char* dsv4_status_string(int status) {
    switch (status) {
        case DSV4_OK: return "ok";
        case DSV4_ERR_INVALID_ARG: return "invalid argument (rejected on the host before any launch)";
        case DSV4_ERR_LAUNCH: return "kernel launch failed";
        case DSV4_ERR_BAD_INDEX: return "an index outside the visible range was masked";
        case DSV4_ERR_TIMEOUT: return "a bounded device wait ran out";
        case DSV4_ERR_UNSUPPORTED: return "unsupported device (the library is built for sm_103 only)";
        default: return "unknown status";
    }
}

int dsv4_last_launch_count(void) { return g_last_launches; }

int dsv4_test_wait_fault(int which, uint32_t wait_limit_us) {
    if (which < DSV4_WAIT_FAULT_NONE || which > DSV4_WAIT_FAULT_ATTN_QUERY || wait_limit_us > 2000000u)
        return DSV4_ERR_INVALID_ARG;
    g_wait_limit_us.store(wait_limit_us);
    g_wait_fault.store(which);
    return DSV4_OK;
}

int64_t dsv4_max_comp(int64_t max_context, int ratio) {
    if (ratio < 1 || max_context < 0) return -1;
    return (max_context + ratio - 1) / ratio;
}

int dsv4_compress(const dsv4_compress_args* a, dsv4_stream_t stream) {
    LaunchScope scope;
    if (!compress_ok(a)) return DSV4_ERR_INVALID_ARG;
    if (int rc = device_check()) return rc;
    return launch_compress(*a, reinterpret_cast<cudaStream_t>(stream));
}

int dsv4_quantize_rows_fp8(const void* x, int rows, int dim, void* q, float* scale, dsv4_stream_t stream) {
    LaunchScope scope;
    if (!dev_ptr_ok(x) || !dev_ptr_ok(q) || !dev_ptr_ok(scale) || rows < 0 || dim < 32 || dim > 1024 ||
        (dim & (dim - 1)) != 0)
        return DSV4_ERR_INVALID_ARG;
    if (int rc = device_check()) return rc;
    return launch_quantize_rows_fp8(x, rows, dim, q, scale, reinterpret_cast<cudaStream_t>(stream));
}

int dsv4_compress_step(const dsv4_compress_step_args* a, dsv4_stream_t stream) {
    LaunchScope scope;
    if (!a || !dev_ptr_ok(a->C) || !dev_ptr_ok(a->Z) || !dev_ptr_ok(a->bias) || !dev_ptr_ok(a->gamma) ||
        !dev_ptr_ok(a->pos) || !dev_ptr_ok(a->stage) || !dev_ptr_ok(a->fill) || !dev_ptr_ok(a->n_comp) ||
        !dev_ptr_ok(a->out))
        return DSV4_ERR_INVALID_ARG;
    if (a->batch < 0 || a->batch > 65535 || a->ratio < 1 || a->dim < 2 || a->dim > 1024 || a->out_rows < 1)
        return DSV4_ERR_INVALID_ARG;
    if (a->overlap != 0 && a->overlap != 1) return DSV4_ERR_INVALID_ARG;
    if (a->rope_dim < 0 || a->rope_dim > a->dim || a->rope_dim > 128 || (a->rope_dim & 1))
        return DSV4_ERR_INVALID_ARG;
    if (!(a->eps >= 0.f) || !std::isfinite(a->eps) || !std::isfinite(a->rope_theta) || a->rope_theta <= 0.0)
        return DSV4_ERR_INVALID_ARG;
    if (a->out_fp8 < 0 || a->out_fp8 > 2) return DSV4_ERR_INVALID_ARG;
    if (a->out_fp8 ? !dev_ptr_ok(a->out_scale) : a->out_scale != nullptr) return DSV4_ERR_INVALID_ARG;
    if (a->out_fp8 == 2 ? (a->rope_dim > 0 ? !dev_ptr_ok(a->out_rope) : a->out_rope != nullptr)
                        : a->out_rope != nullptr)
        return DSV4_ERR_INVALID_ARG;
    if (a->out_fp8 == 2 && a->rope_dim >= a->dim) return DSV4_ERR_INVALID_ARG;
    if (int rc = device_check()) return rc;
    return launch_compress_step(*a, reinterpret_cast<cudaStream_t>(stream));
}

size_t dsv4_indexer_topk_workspace_size(const dsv4_index_args* a) {
    if (!a) return 0;
    return kWsHeader + index_ws_bytes(*a);
}

int dsv4_indexer_topk(const dsv4_index_args* a, void* ws, size_t ws_bytes, dsv4_stream_t stream) {
    LaunchScope scope;
    if (!index_ok(a) || !dev_ptr_ok(ws) || ws_bytes < dsv4_indexer_topk_workspace_size(a))
        return DSV4_ERR_INVALID_ARG;
    if (int rc = device_check()) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(ws, 0, kWsHeader + index_zero_bytes(*a), st) != cudaSuccess) return DSV4_ERR_LAUNCH;
    return launch_indexer(*a, body_of(ws), eword_of(ws), st);
}

size_t dsv4_index_score_workspace_size(const dsv4_index_args* a) {
    (void)a;
    return kWsHeader;
}

int dsv4_index_score(const dsv4_index_args* a, void* ws, size_t ws_bytes, dsv4_stream_t stream) {
    LaunchScope scope;
    if (!index_ok(a) || !a->scores_out || !dev_ptr_ok(ws) || ws_bytes < dsv4_index_score_workspace_size(a))
        return DSV4_ERR_INVALID_ARG;
    if (int rc = device_check()) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // the header holds the error word and the scorer's stage-claim counters
    if (cudaMemsetAsync(ws, 0, kWsHeader, st) != cudaSuccess) return DSV4_ERR_LAUNCH;
    return launch_index_score(*a, eword_of(ws), st);
}

size_t dsv4_topk_workspace_size(const dsv4_topk_args* a) {
    if (!a) return 0;
    return kWsHeader + topk_ws_bytes(a->rows, a->max_comp, a->top_k);
}

int dsv4_topk(const dsv4_topk_args* a, void* ws, size_t ws_bytes, dsv4_stream_t stream) {
    LaunchScope scope;
    if (!topk_ok(a) || !dev_ptr_ok(ws) || ws_bytes < dsv4_topk_workspace_size(a))
        return DSV4_ERR_INVALID_ARG;
    if (int rc = device_check()) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(ws, 0, sizeof(uint32_t), st) != cudaSuccess) return DSV4_ERR_LAUNCH;
    TopkRows t;
    t.scores = a->scores;
    t.n_vis = a->n_vis;
    t.n_comp = nullptr;
    t.q_pos = nullptr;
    t.n_q = 1;
    t.ratio = 1;
    t.idx_out = a->idx_out;
    t.rows = a->rows;
    t.max_comp = a->max_comp;
    t.top_k = a->top_k;
    t.hist_zeroed = false;
    t.hist_built = false;
    t.pdl = true;
    return launch_topk(t, body_of(ws), eword_of(ws), st);
}

size_t dsv4_sparse_attn_workspace_size(const dsv4_attn_args* a) {
    if (!a) return 0;
    return kWsHeader + attn_ws_bytes(*a);
}

int dsv4_sparse_attn_decode(const dsv4_attn_args* a, void* ws, size_t ws_bytes, dsv4_stream_t stream) {
    LaunchScope scope;
    if (!attn_ok(a) || !dev_ptr_ok(ws) || ws_bytes < dsv4_sparse_attn_workspace_size(a))
        return DSV4_ERR_INVALID_ARG;
    if (int rc = device_check()) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(ws, 0, sizeof(uint32_t), st) != cudaSuccess) return DSV4_ERR_LAUNCH;
    return launch_attn(*a, body_of(ws), eword_of(ws), st);
}

static bool csa_ok(const dsv4_csa_args* a) {
    if (!a || !a->attn || !attn_ok(a->attn)) return false;
    if (a->compress_kv && !compress_ok(a->compress_kv)) return false;
    if (a->compress_keys && !compress_ok(a->compress_keys)) return false;
    if (a->index) {
        const dsv4_index_args& x = *a->index;
        const dsv4_attn_args& y = *a->attn;
        if (!index_ok(&x)) return false;
        if (y.idx != x.idx_out || y.top_k != x.top_k || y.batch != x.batch || y.n_q != x.n_q ||
            y.max_comp != x.max_comp || y.n_comp != x.n_comp || y.ratio != x.ratio || y.q_pos != x.q_pos)
            return false;
        // a key cache written in this step is read in the format it was written in
        const dsv4_compress_args* k = a->compress_keys;
        // (the KV cache written in this step is checked below)
        if (k && k->out == x.keys && (k->out_fp8 != x.key_fp8 || (k->out_fp8 && k->out_scale != x.key_scale)))
            return false;
    } else if (a->attn->idx) {
        return false;
    }
    // a KV cache written in this step is read in the layout it was written in
    const dsv4_compress_args* kv = a->compress_kv;
    const dsv4_attn_args& at = *a->attn;
    if (kv && (kv->out == at.comp_kv || kv->out == at.kv_nope)) {
        const bool mixed = kv->out_fp8 == 2;
        if (mixed != (at.kv_fp8 == 1) || kv->out_fp8 == 1) return false;
        if (mixed && (kv->out_scale != at.kv_scale || kv->out_rope != at.kv_rope || kv->rope_dim != at.kv_rope_dim))
            return false;
    }
    return true;
}

size_t dsv4_csa_decode_workspace_size(const dsv4_csa_args* a) {
    if (!a || !a->attn) return 0;
    size_t body = attn_ws_bytes(*a->attn);
    if (a->index) {
        const size_t b2 = index_ws_bytes(*a->index);
        body = body > b2 ? body : b2;
    }
    return kWsHeader + body;
}

int dsv4_csa_decode(const dsv4_csa_args* a, void* ws, size_t ws_bytes, dsv4_stream_t stream) {
    LaunchScope scope;
    if (!csa_ok(a) || !dev_ptr_ok(ws) || ws_bytes < dsv4_csa_decode_workspace_size(a))
        return DSV4_ERR_INVALID_ARG;
    if (int rc = device_check()) return rc;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    // the header and the top-k histograms are cleared by the compression launch (the kernels
    // after it read them only once it has completed), saving a memset in the step
    const size_t zero = kWsHeader + (a->index ? index_zero_bytes(*a->index) : 0);
    int rc = DSV4_OK;
    if ((rc = launch_compress2(a->compress_kv, a->compress_keys, st, ws, zero))) return rc;
    if (a->index && (rc = launch_indexer(*a->index, body_of(ws), eword_of(ws), st, a->compress_keys)))
        return rc;
    return launch_attn(*a->attn, body_of(ws), eword_of(ws), st);
}

int dsv4_read_error_word(void* ws, dsv4_stream_t stream, uint32_t* out) {
    if (!dev_ptr_ok(ws) || !out) return DSV4_ERR_INVALID_ARG;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    uint32_t v = 0;
    if (cudaMemcpyAsync(&v, ws, sizeof v, cudaMemcpyDeviceToHost, st) != cudaSuccess) return DSV4_ERR_LAUNCH;
    if (cudaStreamSynchronize(st) != cudaSuccess) return DSV4_ERR_LAUNCH;
    if (cudaMemsetAsync(ws, 0, sizeof v, st) != cudaSuccess) return DSV4_ERR_LAUNCH;
    if (cudaStreamSynchronize(st) != cudaSuccess) return DSV4_ERR_LAUNCH;
    *out = v;
    if (v & DSV4_EWORD_TIMEOUT) return DSV4_ERR_TIMEOUT;
    if (v & DSV4_EWORD_BAD_INDEX) return DSV4_ERR_BAD_INDEX;
    return DSV4_OK;
}

}  // extern "C"

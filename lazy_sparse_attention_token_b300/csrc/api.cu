// api.cu -- the C ABI declared in include/flashloop.h: argument checks,
// cache and workspace layout, and the order of the kernels in one loop.
//
// Loop order (rit.work page "FlashLoop: Fast and Memory-Efficient Looped
// Transformers via Lazy Updates", section "FlashLoop combines three kinds of
// saving"): early loops run in full; a later loop ranks tokens by change and
// keeps the active ones, writes their low-bit KV deltas, picks key columns
// from the previous loop's statistics and runs mass-preserving attention
// over them.
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <functional>
#include <mutex>
#include <string>
#include <vector>

#include "common.cuh"

namespace fl {

namespace {
thread_local std::string g_last_error;
std::atomic<long long> g_launches{0};

constexpr size_t kAlign = 256;
size_t align_up(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }
bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

__global__ void fill_rows_kernel(int32_t *pos, int32_t *slot, int B, int value) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b < B) {
        pos[b] = value;
        slot[b] = 0;
    }
}
}  // namespace

void note_launch(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

// ---- optional per-kernel timing ---------------------------------------------
namespace {
struct TimingRec {
    std::string name;
    cudaEvent_t ev0, ev1;
};
std::mutex g_timing_mu;
std::atomic<bool> g_timing_on{false};
std::vector<TimingRec> g_timing;
std::vector<cudaEvent_t> g_event_pool;

cudaEvent_t pooled_event() {
    if (!g_event_pool.empty()) {
        cudaEvent_t e = g_event_pool.back();
        g_event_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
}
}  // namespace

KernelTimer::KernelTimer(const char *name, cudaStream_t s) : rec_(-1), s_(s) {
    note_launch();
    if (!g_timing_on.load(std::memory_order_relaxed)) return;
    std::lock_guard<std::mutex> lock(g_timing_mu);
    TimingRec r{name, pooled_event(), pooled_event()};
    cudaEventRecord(r.ev0, s);
    g_timing.push_back(r);
    rec_ = (int)g_timing.size() - 1;
}

KernelTimer::~KernelTimer() {
    if (rec_ < 0) return;
    std::lock_guard<std::mutex> lock(g_timing_mu);
    if (rec_ < (int)g_timing.size()) cudaEventRecord(g_timing[rec_].ev1, s_);
}

flashloop_status_t set_error(flashloop_status_t st, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return st;
}

flashloop_status_t cuda_fail(cudaError_t e, const char *what) {
    return set_error(FLASHLOOP_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Every compute entry point runs only on an sm_103 device.
flashloop_status_t check_device() {
    static std::mutex mu;
    static int cached_dev = -1;
    static bool cached_ok = false;
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    std::lock_guard<std::mutex> lock(mu);
    if (dev != cached_dev) {
        int major = 0, minor = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        cached_ok = (major == 10 && minor == 3);
        cached_dev = dev;
    }
    if (!cached_ok) return set_error(FLASHLOOP_ERR_UNSUPPORTED, "device is not sm_103 (B300)");
    return FLASHLOOP_OK;
}

// A second stream per device for work of one loop that may overlap the
// caller's stream (the key selection of a lazy prefill loop), forked from and
// joined back to that stream with two events. The mutex is held while one
// call enqueues its fork and join; the stream and events live until exit.
struct SideStream {
    std::mutex mu;
    cudaStream_t s = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
    bool ok = false;
};
constexpr int kMaxSideDevices = 64;

static SideStream *side_stream() {
    static SideStream side[kMaxSideDevices];
    static std::once_flag once[kMaxSideDevices];
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxSideDevices) return nullptr;
    SideStream &ss = side[dev];
    std::call_once(once[dev], [&ss] {
        ss.ok = cudaStreamCreateWithFlags(&ss.s, cudaStreamNonBlocking) == cudaSuccess &&
                cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming) == cudaSuccess &&
                cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming) == cudaSuccess;
    });
    return ss.ok ? &ss : nullptr;
}

static bool head_dim_ok(int d) { return d == 64 || d == 96 || d == 128; }
// width of the delta codes and whether the lazy loops read an int8 base
static int code_bits_of(const flashloop_dims_t &dm) { return dm.delta_bits ? dm.delta_bits : 4; }
static bool int8_base(const flashloop_dims_t &dm) { return dm.base_bits == 8; }

static flashloop_status_t check_dims(const flashloop_dims_t *dm) {
    if (!dm) return set_error(FLASHLOOP_ERR_INVALID_ARG, "dims is NULL");
    if (dm->B < 1 || dm->N_cap < 1 || dm->H < 1 || dm->T < 1 || dm->T_dense < 1 || dm->T_dense > dm->T ||
        dm->T > FLASHLOOP_MAX_LOOPS || dm->R < 1 || dm->R > dm->N_cap || dm->K < 1 || dm->K > dm->N_cap ||
        dm->R_cap < dm->R || dm->R_cap > dm->N_cap)
        return set_error(FLASHLOOP_ERR_INVALID_ARG, "bad dims (B=%d N_cap=%d H=%d R=%d K=%d T=%d T_dense=%d R_cap=%d)",
                         dm->B, dm->N_cap, dm->H, dm->R, dm->K, dm->T, dm->T_dense, dm->R_cap);
    if (!head_dim_ok(dm->d)) return set_error(FLASHLOOP_ERR_UNSUPPORTED, "head dim %d not in {64, 96, 128}", dm->d);
    if (dm->delta_bits != 0 && (dm->delta_bits < 2 || dm->delta_bits > 4))
        return set_error(FLASHLOOP_ERR_UNSUPPORTED, "delta_bits %d not in {2, 3, 4}", dm->delta_bits);
    if (dm->base_bits != 0 && dm->base_bits != 8 && dm->base_bits != 16)
        return set_error(FLASHLOOP_ERR_UNSUPPORTED, "base_bits %d not in {8, 16}", dm->base_bits);
    return FLASHLOOP_OK;
}

struct WsLayout {
    size_t scores, kv, rows, slots, counts, total;
};

static WsLayout ws_layout(const flashloop_dims_t *dm) {
    WsLayout w;
    size_t off = 0;
    w.scores = off;
    off += align_up((size_t)dm->B * dm->N_cap * sizeof(float));
    w.kv = off;
    off += 4 * align_up((size_t)dm->B * dm->H * dm->K * dm->d * 2);
    w.rows = off;
    off += align_up((size_t)dm->B * sizeof(int32_t));
    w.slots = off;
    off += align_up((size_t)dm->B * sizeof(int32_t));
    w.counts = off;   // lazy attention: keys each row sees, [B,H,R_cap]
    off += align_up((size_t)dm->B * dm->H * dm->R_cap * sizeof(int32_t));
    w.total = off;
    return w;
}

struct CacheLayout {
    size_t dense_layer, base_codes, base_scales, idx, slot, codes, scales, total;
};

static CacheLayout cache_layout(const flashloop_dims_t *dm) {
    CacheLayout c;
    const size_t rows = (size_t)dm->B * dm->N_cap * dm->H;
    c.dense_layer = align_up(rows * dm->d * 2);
    c.base_codes = int8_base(*dm) ? align_up(rows * dm->d) : 0;
    c.base_scales = int8_base(*dm) ? align_up(rows * (dm->d / 32) * 2) : 0;
    c.idx = align_up((size_t)dm->B * dm->R_cap * 4);
    c.slot = align_up((size_t)dm->B * dm->N_cap * 4);
    c.codes = align_up((size_t)dm->B * dm->R_cap * dm->H * ((size_t)dm->d * code_bits_of(*dm) / 8));
    c.scales = align_up((size_t)dm->B * dm->R_cap * dm->H * (dm->d / 32) * 2);
    const size_t n_delta = (size_t)(dm->T - dm->T_dense);
    c.total = 2 * dm->T_dense * c.dense_layer + 2 * (c.base_codes + c.base_scales) +
              n_delta * (c.idx + c.slot + 2 * c.codes + 2 * c.scales);
    return c;
}

// Reconstruction of loop `loop` = base (last dense layer) + delta layers up to
// `loop`. `lazy` views are those the lazy loops read (appends, reconstructions,
// decode's lazy attention): with an int8 base they take it in place of the
// bf16 base layer; the dense loops' own attention reads the bf16 layers.
static DeltaView make_view(const flashloop_kv_cache_t *c, int loop, bool lazy = true) {
    DeltaView v;
    memset(&v, 0, sizeof v);
    const int td = c->dims.T_dense;
    v.code_bits = code_bits_of(c->dims);
    const bool compressed = lazy && int8_base(c->dims) && loop >= td;
    if (compressed) {
        v.k_base_codes = c->k_base_codes;
        v.v_base_codes = c->v_base_codes;
        v.k_base_scales = c->k_base_scales;
        v.v_base_scales = c->v_base_scales;
    }
    if (loop <= td) {
        v.k_base = compressed ? nullptr : c->k_dense[loop - 1];
        v.v_base = compressed ? nullptr : c->v_dense[loop - 1];
        v.n_layers = 0;
        return v;
    }
    v.k_base = compressed ? nullptr : c->k_dense[td - 1];
    v.v_base = compressed ? nullptr : c->v_dense[td - 1];
    v.n_layers = loop - td;
    for (int m = 0; m < v.n_layers; ++m) {
        v.slot[m] = c->slot[m];
        v.k_codes[m] = c->k_codes[m];
        v.k_scales[m] = c->k_scales[m];
        v.v_codes[m] = c->v_codes[m];
        v.v_scales[m] = c->v_scales[m];
    }
    return v;
}

static flashloop_status_t check_cache(const flashloop_kv_cache_t *c) {
    if (!c) return set_error(FLASHLOOP_ERR_INVALID_ARG, "cache is NULL");
    flashloop_status_t st = check_dims(&c->dims);
    if (st != FLASHLOOP_OK) return st;
    for (int t = 0; t < c->dims.T_dense; ++t)
        if (!c->k_dense[t] || !c->v_dense[t]) return set_error(FLASHLOOP_ERR_INVALID_ARG, "cache is not initialised");
    if (int8_base(c->dims) && (!c->k_base_codes || !c->v_base_codes || !c->k_base_scales || !c->v_base_scales))
        return set_error(FLASHLOOP_ERR_INVALID_ARG, "cache is not initialised (int8 base)");
    return FLASHLOOP_OK;
}

}  // namespace fl

using namespace fl;

extern "C" {

const char *flashloop_status_string(flashloop_status_t s) {
    switch (s) {
        case FLASHLOOP_OK: return "ok";
        case FLASHLOOP_ERR_INVALID_ARG: return "invalid argument";
        case FLASHLOOP_ERR_UNSUPPORTED: return "unsupported";
        case FLASHLOOP_ERR_CAPACITY: return "capacity exceeded";
        case FLASHLOOP_ERR_CUDA: return "CUDA error";
        case FLASHLOOP_ERR_WORKSPACE: return "workspace too small";
        case FLASHLOOP_ERR_DEVICE: return "device-side failure";
    }
    return "unknown status";
}

const char *flashloop_last_error(void) { return g_last_error.c_str(); }

int64_t flashloop_launch_count(void) { return g_launches.load(); }

flashloop_status_t flashloop_timing_enable(int32_t on) {
    std::lock_guard<std::mutex> lock(g_timing_mu);
    g_timing_on.store(on != 0);
    return FLASHLOOP_OK;
}

int32_t flashloop_timing_read(char *names, int32_t name_len, double *total_ms, int64_t *launches, int32_t max_kinds) {
    if (cudaDeviceSynchronize() != cudaSuccess) return -1;
    std::lock_guard<std::mutex> lock(g_timing_mu);
    std::vector<std::string> kinds;
    std::vector<double> ms;
    std::vector<int64_t> cnt;
    for (const TimingRec &r : g_timing) {
        float t = 0.f;
        cudaEventElapsedTime(&t, r.ev0, r.ev1);
        size_t k = 0;
        while (k < kinds.size() && kinds[k] != r.name) ++k;
        if (k == kinds.size()) {
            kinds.push_back(r.name);
            ms.push_back(0.0);
            cnt.push_back(0);
        }
        ms[k] += t;
        cnt[k] += 1;
        g_event_pool.push_back(r.ev0);
        g_event_pool.push_back(r.ev1);
    }
    g_timing.clear();
    const int n = (int)kinds.size() < max_kinds ? (int)kinds.size() : max_kinds;
    for (int k = 0; k < n; ++k) {
        if (names && name_len > 0) {
            strncpy(names + (size_t)k * name_len, kinds[k].c_str(), (size_t)name_len - 1);
            names[(size_t)k * name_len + name_len - 1] = 0;
        }
        if (total_ms) total_ms[k] = ms[k];
        if (launches) launches[k] = cnt[k];
    }
    return n;
}

size_t flashloop_workspace_bytes(const flashloop_dims_t *dims) {
    if (check_dims(dims) != FLASHLOOP_OK) return 0;
    return ws_layout(dims).total;
}

size_t flashloop_kv_cache_bytes(const flashloop_dims_t *dims) {
    if (check_dims(dims) != FLASHLOOP_OK) return 0;
    return cache_layout(dims).total;
}

flashloop_status_t flashloop_kv_cache_init(flashloop_kv_cache_t *cache, void *dev_buf, size_t bytes,
                                           const flashloop_dims_t *dims, flashloop_stream_t stream) {
    if (!cache || !dev_buf) return set_error(FLASHLOOP_ERR_INVALID_ARG, "cache or buffer is NULL");
    flashloop_status_t st = check_dims(dims);
    if (st != FLASHLOOP_OK) return st;
    if (reinterpret_cast<uintptr_t>(dev_buf) % kAlign)
        return set_error(FLASHLOOP_ERR_INVALID_ARG, "cache buffer must be 256-byte aligned");
    const CacheLayout L = cache_layout(dims);
    if (bytes < L.total) return set_error(FLASHLOOP_ERR_CAPACITY, "cache buffer %zu < %zu bytes", bytes, L.total);
    if ((st = check_device()) != FLASHLOOP_OK) return st;
    memset(cache, 0, sizeof *cache);
    cache->dims = *dims;
    uint8_t *p = static_cast<uint8_t *>(dev_buf);
    for (int t = 0; t < dims->T_dense; ++t) {
        cache->k_dense[t] = reinterpret_cast<uint16_t *>(p); p += L.dense_layer;
        cache->v_dense[t] = reinterpret_cast<uint16_t *>(p); p += L.dense_layer;
    }
    if (int8_base(*dims)) {
        cache->k_base_codes = reinterpret_cast<int8_t *>(p); p += L.base_codes;
        cache->v_base_codes = reinterpret_cast<int8_t *>(p); p += L.base_codes;
        cache->k_base_scales = reinterpret_cast<uint16_t *>(p); p += L.base_scales;
        cache->v_base_scales = reinterpret_cast<uint16_t *>(p); p += L.base_scales;
    }
    for (int m = 0; m < dims->T - dims->T_dense; ++m) {
        cache->idx[m] = reinterpret_cast<int32_t *>(p); p += L.idx;
        cache->slot[m] = reinterpret_cast<int32_t *>(p); p += L.slot;
        cache->k_codes[m] = p; p += L.codes;
        cache->k_scales[m] = reinterpret_cast<uint16_t *>(p); p += L.scales;
        cache->v_codes[m] = p; p += L.codes;
        cache->v_scales[m] = reinterpret_cast<uint16_t *>(p); p += L.scales;
        cudaError_t e = cudaMemsetAsync(cache->slot[m], 0xFF, (size_t)dims->B * dims->N_cap * 4, stream);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(slot)");
    }
    return FLASHLOOP_OK;
}

flashloop_status_t flashloop_select_tokens(const uint16_t *h_prev, const uint16_t *h_cur, int32_t B, int32_t N,
                                           int32_t D, int32_t R, int32_t *active_idx, float *scores,
                                           void *workspace, size_t workspace_bytes, flashloop_stream_t stream) {
    if (!h_prev || !h_cur || !active_idx) return set_error(FLASHLOOP_ERR_INVALID_ARG, "NULL pointer");
    if (!aligned16(h_prev) || !aligned16(h_cur)) return set_error(FLASHLOOP_ERR_INVALID_ARG, "inputs must be 16-byte aligned");
    if (B < 1 || N < 1 || D < 8 || D % 8 || R < 1 || R > N)
        return set_error(FLASHLOOP_ERR_INVALID_ARG, "bad sizes (B=%d N=%d D=%d R=%d)", B, N, D, R);
    float *sc = scores;
    if (!sc) {
        if (!workspace || workspace_bytes < (size_t)B * N * sizeof(float))
            return set_error(FLASHLOOP_ERR_WORKSPACE, "workspace needs %zu bytes for scores", (size_t)B * N * 4);
        sc = static_cast<float *>(workspace);
    }
    flashloop_status_t st = check_device();
    if (st != FLASHLOOP_OK) return st;
    cudaError_t e = launch_token_scores(h_prev, h_cur, B, N, D, sc, stream);
    if (e != cudaSuccess) return cuda_fail(e, "token_scores");
    e = launch_topk_rows(sc, B, N, R, active_idx, stream, "topk_tokens");
    if (e != cudaSuccess) return cuda_fail(e, "topk(tokens)");
    return FLASHLOOP_OK;
}

flashloop_status_t flashloop_gather(const void *src, int32_t B, int32_t N, int32_t row_bytes, const int32_t *idx,
                                    int32_t R, void *dst, flashloop_stream_t stream) {
    if (!src || !idx || !dst) return set_error(FLASHLOOP_ERR_INVALID_ARG, "NULL pointer");
    if (!aligned16(src) || !aligned16(dst)) return set_error(FLASHLOOP_ERR_INVALID_ARG, "src/dst must be 16-byte aligned");
    if (B < 1 || N < 1 || R < 0 || row_bytes < 16 || row_bytes % 16)
        return set_error(FLASHLOOP_ERR_INVALID_ARG, "bad sizes (B=%d N=%d R=%d row_bytes=%d)", B, N, R, row_bytes);
    flashloop_status_t st = check_device();
    if (st != FLASHLOOP_OK) return st;
    cudaError_t e = launch_gather_rows(src, B, N, row_bytes, idx, R, dst, stream);
    if (e != cudaSuccess) return cuda_fail(e, "gather");
    return FLASHLOOP_OK;
}

namespace fl {
// slots_cleared: the caller already reset the layer's slot map (at == 0), earlier
// on the stream, so that the append kernel directly follows the token selection.
static flashloop_status_t delta_append_impl(flashloop_kv_cache_t *cache, int32_t loop, const uint16_t *k_l,
                                            const uint16_t *v_l, int32_t rows_are_tokens, const int32_t *active_idx,
                                            int32_t R, int32_t at, bool slots_cleared, flashloop_stream_t stream,
                                            const int32_t *seq_exit = nullptr) {
    flashloop_status_t st = check_cache(cache);
    if (st != FLASHLOOP_OK) return st;
    const flashloop_dims_t &dm = cache->dims;
    if (loop <= dm.T_dense || loop > dm.T)
        return set_error(FLASHLOOP_ERR_INVALID_ARG, "loop %d is not a lazy loop (T_dense=%d, T=%d)", loop, dm.T_dense, dm.T);
    if (!k_l || !v_l || !active_idx) return set_error(FLASHLOOP_ERR_INVALID_ARG, "NULL pointer");
    if (!aligned16(k_l) || !aligned16(v_l)) return set_error(FLASHLOOP_ERR_INVALID_ARG, "K/V must be 16-byte aligned");
    const int m = loop - dm.T_dense - 1;
    if (R < 1 || at < 0 || (at != 0 && at != cache->count[m]))
        return set_error(FLASHLOOP_ERR_INVALID_ARG, "R=%d at=%d (layer holds %d)", R, at, cache->count[m]);
    if (at + R > dm.R_cap) return set_error(FLASHLOOP_ERR_CAPACITY, "delta layer full (%d + %d > %d)", at, R, dm.R_cap);
    if (rows_are_tokens && (cache->n_tokens < 1 || cache->n_tokens > dm.N_cap))
        return set_error(FLASHLOOP_ERR_INVALID_ARG, "rows_are_tokens needs 1 <= cache n_tokens <= N_cap");
    // every check comes before the slot map is touched: a rejected call leaves
    // the layer, its slot map and its count as they were
    if ((st = check_device()) != FLASHLOOP_OK) return st;
    if (at == 0 && !slots_cleared) {
        cudaError_t e = cudaMemsetAsync(cache->slot[m], 0xFF, (size_t)dm.B * dm.N_cap * 4, stream);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(slot)");
    }
    const DeltaView view = make_view(cache, loop - 1);
    const int src_rows = rows_are_tokens ? cache->n_tokens : R;
    cudaError_t e = launch_delta_append(view, k_l, v_l, rows_are_tokens, src_rows, active_idx, R, at, dm.B, dm.N_cap,
                                        dm.H, dm.d, dm.R_cap, cache->idx[m], cache->slot[m], cache->k_codes[m],
                                        cache->k_scales[m], cache->v_codes[m], cache->v_scales[m], stream, seq_exit);
    if (e != cudaSuccess) return cuda_fail(e, "kv_delta_append");
    cache->count[m] = at + R;
    return FLASHLOOP_OK;
}
}  // namespace fl

flashloop_status_t flashloop_kv_delta_append(flashloop_kv_cache_t *cache, int32_t loop, const uint16_t *k_l,
                                             const uint16_t *v_l, int32_t rows_are_tokens,
                                             const int32_t *active_idx, int32_t R, int32_t at,
                                             flashloop_stream_t stream) {
    return fl::delta_append_impl(cache, loop, k_l, v_l, rows_are_tokens, active_idx, R, at, false, stream);
}

flashloop_status_t flashloop_kv_dense_store(flashloop_kv_cache_t *cache, int32_t loop, const uint16_t *k,
                                            const uint16_t *v, int32_t pos0, int32_t n_rows,
                                            flashloop_stream_t stream) {
    flashloop_status_t st = check_cache(cache);
    if (st != FLASHLOOP_OK) return st;
    const flashloop_dims_t &dm = cache->dims;
    if (loop < 1 || loop > dm.T_dense)
        return set_error(FLASHLOOP_ERR_INVALID_ARG, "loop %d is not a dense loop (T_dense=%d)", loop, dm.T_dense);
    if (!k || !v || !aligned16(k) || !aligned16(v)) return set_error(FLASHLOOP_ERR_INVALID_ARG, "bad K/V pointer");
    if (pos0 < 0 || n_rows < 1 || pos0 + n_rows > dm.N_cap)
        return set_error(FLASHLOOP_ERR_CAPACITY, "rows [%d, %d) exceed N_cap=%d", pos0, pos0 + n_rows, dm.N_cap);
    if ((st = check_device()) != FLASHLOOP_OK) return st;
    const int row = dm.H * dm.d;
    cudaError_t e = launch_store_rows(k, dm.B, n_rows, row, cache->k_dense[loop - 1], dm.N_cap, pos0, stream);
    if (e == cudaSuccess) e = launch_store_rows(v, dm.B, n_rows, row, cache->v_dense[loop - 1], dm.N_cap, pos0, stream);
    if (e == cudaSuccess && int8_base(dm) && loop == dm.T_dense) {   // the base the lazy loops read, compressed
        e = launch_quantize_base(k, dm.B, n_rows, dm.H, dm.d, cache->k_base_codes, cache->k_base_scales, dm.N_cap, pos0,
                                 stream);
        if (e == cudaSuccess)
            e = launch_quantize_base(v, dm.B, n_rows, dm.H, dm.d, cache->v_base_codes, cache->v_base_scales, dm.N_cap,
                                     pos0, stream);
    }
    if (e != cudaSuccess) return cuda_fail(e, "kv_dense_store");
    return FLASHLOOP_OK;
}

namespace fl {
static flashloop_status_t select_keys_impl(const float *col_stats, int32_t B, int32_t H, int32_t N, int32_t K,
                                           int32_t n_rows, int32_t *key_idx, flashloop_stream_t stream) {
    if (!col_stats || !key_idx) return set_error(FLASHLOOP_ERR_INVALID_ARG, "NULL pointer");
    if (B < 1 || H < 1 || N < 1 || K < 1 || K > N)
        return set_error(FLASHLOOP_ERR_INVALID_ARG, "bad sizes (B=%d H=%d N=%d K=%d)", B, H, N, K);
    if (n_rows != 0 && n_rows < N)
        return set_error(FLASHLOOP_ERR_INVALID_ARG, "n_rows=%d must cover the N=%d columns", n_rows, N);
    flashloop_status_t st = check_device();
    if (st != FLASHLOOP_OK) return st;
    cudaError_t e = launch_topk_rows(col_stats, B * H, N, K, key_idx, stream, "topk_keys", n_rows);
    if (e != cudaSuccess) return cuda_fail(e, "topk(keys)");
    return FLASHLOOP_OK;
}
}  // namespace fl

flashloop_status_t flashloop_select_keys(const float *col_stats, int32_t B, int32_t H, int32_t N, int32_t K,
                                         int32_t *key_idx, void *workspace, size_t workspace_bytes,
                                         flashloop_stream_t stream) {
    (void)workspace;
    (void)workspace_bytes;
    return fl::select_keys_impl(col_stats, B, H, N, K, 0, key_idx, stream);
}

flashloop_status_t flashloop_select_keys_per_row(const float *col_stats, int32_t B, int32_t H, int32_t N, int32_t K,
                                                 int32_t n_rows, int32_t *key_idx, flashloop_stream_t stream) {
    if (n_rows < 1) return set_error(FLASHLOOP_ERR_INVALID_ARG, "n_rows=%d", n_rows);
    return fl::select_keys_impl(col_stats, B, H, N, K, n_rows, key_idx, stream);
}

flashloop_status_t flashloop_reconstruct_keys(const flashloop_kv_cache_t *cache, int32_t loop, const int32_t *key_idx,
                                              int32_t K, uint16_t *k_old, uint16_t *v_old, uint16_t *k_new,
                                              uint16_t *v_new, flashloop_stream_t stream) {
    flashloop_status_t st = check_cache(cache);
    if (st != FLASHLOOP_OK) return st;
    const flashloop_dims_t &dm = cache->dims;
    if (loop <= dm.T_dense || loop > dm.T)
        return set_error(FLASHLOOP_ERR_INVALID_ARG, "loop %d is not a lazy loop", loop);
    if (!key_idx || !k_old || !v_old || !k_new || !v_new) return set_error(FLASHLOOP_ERR_INVALID_ARG, "NULL pointer");
    if (!aligned16(k_old) || !aligned16(v_old) || !aligned16(k_new) || !aligned16(v_new))
        return set_error(FLASHLOOP_ERR_INVALID_ARG, "outputs must be 16-byte aligned");
    if (K < 1 || K > dm.N_cap) return set_error(FLASHLOOP_ERR_INVALID_ARG, "bad K=%d", K);
    if ((st = check_device()) != FLASHLOOP_OK) return st;
    cudaError_t e = launch_reconstruct_keys(make_view(cache, loop - 1), make_view(cache, loop), key_idx, dm.B, dm.H, K,
                                            dm.N_cap, dm.d, dm.R_cap, k_old, v_old, k_new, v_new, nullptr, 0,
                                            nullptr, stream);
    if (e != cudaSuccess) return cuda_fail(e, "reconstruct_keys");
    return FLASHLOOP_OK;
}

namespace fl {
// seq_exit: [B] flags or NULL; the tensor-core path leaves sequences flagged 1 unchanged.
static flashloop_status_t lazy_attention_impl(const flashloop_attn_args_t *a, flashloop_stream_t stream,
                                              const int32_t *seq_exit);
}  // namespace fl

flashloop_status_t flashloop_lazy_attention(const flashloop_attn_args_t *a, flashloop_stream_t stream) {
    return fl::lazy_attention_impl(a, stream, nullptr);
}

namespace fl {
static flashloop_status_t lazy_attention_impl(const flashloop_attn_args_t *a, flashloop_stream_t stream,
                                              const int32_t *seq_exit) {
    if (!a) return set_error(FLASHLOOP_ERR_INVALID_ARG, "args is NULL");
    flashloop_status_t st = check_cache(a->cache);
    if (st != FLASHLOOP_OK) return st;
    const flashloop_kv_cache_t *c = a->cache;
    const flashloop_dims_t &dm = c->dims;
    const bool lazy = a->mode == FLASHLOOP_ATTN_LAZY;
    if (a->mode < 0 || a->mode > 2) return set_error(FLASHLOOP_ERR_INVALID_ARG, "bad mode %d", a->mode);
    if (a->loop < 1 || a->loop > dm.T) return set_error(FLASHLOOP_ERR_INVALID_ARG, "bad loop %d", a->loop);
    if ((a->mode == FLASHLOOP_ATTN_FIRST_DENSE) != (a->loop == 1))
        return set_error(FLASHLOOP_ERR_INVALID_ARG, "FIRST_DENSE is loop 1 and only loop 1");
    if (lazy != (a->loop > dm.T_dense))
        return set_error(FLASHLOOP_ERR_INVALID_ARG, "loop %d is %s but mode is %d", a->loop,
                         a->loop > dm.T_dense ? "lazy" : "dense", a->mode);
    if (!a->q || !a->q_hat || !a->o || !a->z || !a->c) return set_error(FLASHLOOP_ERR_INVALID_ARG, "NULL state pointer");
    if (!aligned16(a->q) || !aligned16(a->q_hat) || !aligned16(a->o))
        return set_error(FLASHLOOP_ERR_INVALID_ARG, "q/q_hat/o must be 16-byte aligned");
    if (a->n_keys < 1 || a->n_keys > dm.N_cap || a->n_state < 1 || a->R < 0)
        return set_error(FLASHLOOP_ERR_INVALID_ARG, "bad n_keys/n_state/R");
    const bool few_rows = a->row_pos != nullptr && a->R <= 8;
    if (!few_rows && a->R > 0 && a->n_state != a->n_keys)
        return set_error(FLASHLOOP_ERR_INVALID_ARG, "prefill attention needs n_state == n_keys");
    if (lazy) {
        if (!a->key_idx || a->K < 1 || a->K > a->n_keys)
            return set_error(FLASHLOOP_ERR_INVALID_ARG, "lazy attention needs key_idx and 1 <= K <= n_keys");
        if (!a->row_pos && a->R > 0) return set_error(FLASHLOOP_ERR_INVALID_ARG, "lazy attention needs row_pos");
    } else if (!few_rows && a->R != a->n_keys) {
        return set_error(FLASHLOOP_ERR_INVALID_ARG, "dense prefill attention covers every row (R == n_keys)");
    }
    if ((st = check_device()) != FLASHLOOP_OK) return st;
    cudaError_t e;
    if (a->mode == FLASHLOOP_ATTN_FIRST_DENSE) {
        e = cudaMemsetAsync(a->c, 0, (size_t)dm.B * dm.H * a->n_keys * sizeof(float), stream);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(c)");
    }
    if (a->R == 0) return FLASHLOOP_OK;
    if (few_rows) {
        DecodeAttnParams p;
        memset(&p, 0, sizeof p);
        p.mode = a->mode;
        p.B = dm.B; p.H = dm.H; p.d = dm.d;
        p.n_keys = a->n_keys; p.n_state = a->n_state; p.R = a->R;
        p.row_pos = a->row_pos; p.row_slot = a->row_slot;
        p.K = lazy ? a->K : a->n_keys;
        p.key_idx = lazy ? a->key_idx : nullptr;
        p.q = a->q; p.q_hat = a->q_hat; p.o = a->o; p.z = a->z; p.c = a->c;
        p.new_view = make_view(c, a->loop, lazy);
        if (a->loop > 1) p.old_view = make_view(c, a->loop - 1, lazy);
        p.N_cap = dm.N_cap; p.R_cap = dm.R_cap;
        e = launch_decode_attention(p, stream);
        if (e == cudaErrorInvalidValue)
            return set_error(FLASHLOOP_ERR_UNSUPPORTED, "decode attention: %d keys exceed its shared-memory limit",
                             p.K);
        if (e != cudaSuccess) return cuda_fail(e, "decode_attention");
        return FLASHLOOP_OK;
    }
    TcAttnParams p;
    memset(&p, 0, sizeof p);
    p.mode = a->mode;
    p.B = dm.B; p.H = dm.H; p.d = dm.d;
    p.n_keys = a->n_keys; p.n_state = a->n_state; p.R = a->R;
    p.row_pos = lazy ? a->row_pos : nullptr;
    p.q = a->q; p.q_hat = a->q_hat; p.o = a->o; p.z = a->z; p.c = a->c;
    if (lazy) {
        const WsLayout W = ws_layout(&dm);
        if (a->K > dm.K) return set_error(FLASHLOOP_ERR_WORKSPACE, "K=%d exceeds dims.K=%d the workspace is sized for", a->K, dm.K);
        if (a->R > dm.R_cap)
            return set_error(FLASHLOOP_ERR_WORKSPACE, "R=%d exceeds dims.R_cap=%d the workspace is sized for", a->R, dm.R_cap);
        if (!a->workspace || a->workspace_bytes < W.total || reinterpret_cast<uintptr_t>(a->workspace) % kAlign)
            return set_error(FLASHLOOP_ERR_WORKSPACE, "workspace needs %zu bytes, 256-byte aligned", W.total);
        uint8_t *ws = static_cast<uint8_t *>(a->workspace) + W.kv;
        const size_t one = align_up((size_t)dm.B * dm.H * dm.K * dm.d * 2);
        uint16_t *kv[4];
        for (int i = 0; i < 4; ++i) kv[i] = reinterpret_cast<uint16_t *>(ws + i * one);
        // both reconstructions of the selected keys, and the keys each row sees
        int32_t *counts = reinterpret_cast<int32_t *>(static_cast<uint8_t *>(a->workspace) + W.counts);
        e = launch_reconstruct_keys(make_view(c, a->loop - 1), make_view(c, a->loop), a->key_idx, dm.B, dm.H, a->K,
                                    dm.N_cap, dm.d, dm.R_cap, kv[0], kv[1], kv[2], kv[3], a->row_pos, a->R, counts,
                                    stream);
        if (e != cudaSuccess) return cuda_fail(e, "reconstruct_keys");
        p.K = a->K;
        p.key_idx = a->key_idx;
        p.k_old = kv[0]; p.v_old = kv[1]; p.k_new = kv[2]; p.v_new = kv[3];
        p.kv_rows = a->K;
        p.row_cnt = counts;
    } else {
        p.K = a->n_keys;
        p.k_new = c->k_dense[a->loop - 1];
        p.v_new = c->v_dense[a->loop - 1];
        if (a->loop > 1) {
            p.k_old = c->k_dense[a->loop - 2];
            p.v_old = c->v_dense[a->loop - 2];
        }
        p.kv_rows = dm.N_cap;
    }
    p.seq_exit = seq_exit;
    e = launch_tc_attention(p, stream);
    if (e != cudaSuccess) return cuda_fail(e, "tc_attention");
    return FLASHLOOP_OK;
}
}  // namespace fl

namespace fl {
// The selection and cache half of a lazy prefill loop, shared by the fused
// step and the synthetic block: the key selection (on a side stream, forked
// from and joined back to `stream`), the token selection, then `project` (the
// block's projections of the active rows; NULL for the step, whose K/V exist
// already), then the delta append of K/V. forced: active_idx and key_idx are
// inputs and neither selection runs.
struct LazyFront {
    flashloop_kv_cache_t *c;
    int loop, n;
    const uint16_t *h_prev, *h_cur;
    float *scores;
    int32_t *active_idx, *key_idx;
    const float *col;
    int key_rank;
    bool forced;
    float exit_threshold;
    int32_t *seq_exit;
    const uint16_t *k, *v;
};

static flashloop_status_t lazy_front(const LazyFront &f, const std::function<flashloop_status_t()> &project,
                                     flashloop_stream_t stream) {
    flashloop_kv_cache_t *c = f.c;
    const flashloop_dims_t &dm = c->dims;
    flashloop_status_t st = FLASHLOOP_OK;
    if (f.key_rank != FLASHLOOP_KEYS_BY_MASS && f.key_rank != FLASHLOOP_KEYS_BY_MASS_PER_ROW)
        return set_error(FLASHLOOP_ERR_INVALID_ARG, "bad key_rank %d", f.key_rank);
    if (dm.R > f.n || dm.K > f.n)
        return set_error(FLASHLOOP_ERR_INVALID_ARG, "R=%d and K=%d must not exceed the %d tokens in the cache", dm.R, dm.K,
                         f.n);
    if (!f.forced && (!aligned16(f.h_prev) || !aligned16(f.h_cur) || (dm.H * dm.d) % 8))
        return set_error(FLASHLOOP_ERR_INVALID_ARG, "hidden states must be 16-byte aligned rows");
    {   // this loop's delta layer starts empty; cleared first so that the append
        // kernel follows the token selection kernel directly
        const int m = f.loop - dm.T_dense - 1;
        cudaError_t e = cudaMemsetAsync(c->slot[m], 0xFF, (size_t)dm.B * dm.N_cap * 4, static_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(slot)");
    }
    // The key columns depend only on the previous loop's column mass, so their
    // selection runs on a side stream while the token selection, projections
    // and K/V delta append run on the caller's; the attention waits for both.
    SideStream *ss = f.forced ? nullptr : side_stream();
    std::unique_lock<std::mutex> side_lock;
    flashloop_stream_t key_stream = stream;
    if (ss) {
        side_lock = std::unique_lock<std::mutex>(ss->mu);
        cudaError_t e = cudaEventRecord(ss->fork, static_cast<cudaStream_t>(stream));
        if (e == cudaSuccess) e = cudaStreamWaitEvent(ss->s, ss->fork, 0);
        if (e != cudaSuccess) return cuda_fail(e, "fork of the key selection");
        key_stream = ss->s;
    }
    if (!f.forced)
        st = select_keys_impl(f.col, dm.B, dm.H, f.n, dm.K, f.key_rank == FLASHLOOP_KEYS_BY_MASS_PER_ROW ? f.n : 0,
                              f.key_idx, key_stream);
    if (st == FLASHLOOP_OK && !f.forced) {
        // token selection; with exit flags, the top-k also flags sequences whose
        // largest change score is below the threshold (sticky)
        const bool upd = f.seq_exit && f.exit_threshold > 0.f;
        cudaError_t e = launch_token_scores(f.h_prev, f.h_cur, dm.B, f.n, dm.H * dm.d, f.scores, stream);
        if (e == cudaSuccess)
            e = launch_topk_rows(f.scores, dm.B, f.n, dm.R, f.active_idx, stream, "topk_tokens", 0,
                                 upd ? f.exit_threshold : 0.f, upd ? f.seq_exit : nullptr);
        if (e != cudaSuccess) st = cuda_fail(e, "token selection");
    }
    if (st == FLASHLOOP_OK && project) st = project();
    if (st == FLASHLOOP_OK)
        st = delta_append_impl(c, f.loop, f.k, f.v, 1, f.active_idx, dm.R, 0, true, stream, f.seq_exit);
    if (ss) {   // join (also on failure, so that the caller's stream is never left forked)
        cudaError_t e = cudaEventRecord(ss->join, ss->s);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(static_cast<cudaStream_t>(stream), ss->join, 0);
        side_lock.unlock();
        if (e != cudaSuccess && st == FLASHLOOP_OK) return cuda_fail(e, "join of the key selection");
    }
    return st;
}
}  // namespace fl

flashloop_status_t flashloop_loop_step(const flashloop_step_args_t *a, flashloop_stream_t stream) {
    if (!a) return set_error(FLASHLOOP_ERR_INVALID_ARG, "args is NULL");
    flashloop_status_t st = check_cache(a->cache);
    if (st != FLASHLOOP_OK) return st;
    flashloop_kv_cache_t *c = a->cache;
    const flashloop_dims_t &dm = c->dims;
    const int l = a->loop;
    if (l < 1 || l > dm.T) return set_error(FLASHLOOP_ERR_INVALID_ARG, "bad loop %d", l);
    const bool dense = l <= dm.T_dense;
    const WsLayout W = ws_layout(&dm);
    if (!a->workspace || a->workspace_bytes < W.total || reinterpret_cast<uintptr_t>(a->workspace) % kAlign)
        return set_error(FLASHLOOP_ERR_WORKSPACE, "workspace needs %zu bytes, 256-byte aligned", W.total);
    uint8_t *ws = static_cast<uint8_t *>(a->workspace);
    const int n = c->n_tokens;
    if (n < 1 || n > dm.N_cap) return set_error(FLASHLOOP_ERR_INVALID_ARG, "cache n_tokens=%d", n);

    flashloop_attn_args_t at;
    memset(&at, 0, sizeof at);
    at.loop = l;
    at.n_keys = n;
    at.q = a->q; at.q_hat = a->q_hat; at.o = a->o; at.z = a->z; at.c = a->c;
    at.cache = c;
    at.workspace = a->workspace;
    at.workspace_bytes = a->workspace_bytes;
    at.mode = l == 1 ? FLASHLOOP_ATTN_FIRST_DENSE : dense ? FLASHLOOP_ATTN_DENSE : FLASHLOOP_ATTN_LAZY;

    if (a->decode) {
        // one new token per sequence at key position n - 1; its state has one row
        const int pos = n - 1;
        int32_t *rows = reinterpret_cast<int32_t *>(ws + W.rows);
        int32_t *slots = reinterpret_cast<int32_t *>(ws + W.slots);
        {
            KernelTimer kt("fill_rows", stream);
            fill_rows_kernel<<<ceil_div(dm.B, 128), 128, 0, stream>>>(rows, slots, dm.B, pos);
        }
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return cuda_fail(e, "fill_rows");
        if (dense) {
            if ((st = flashloop_kv_dense_store(c, l, a->k, a->v, pos, 1, stream)) != FLASHLOOP_OK) return st;
        } else {
            const int m = l - dm.T_dense - 1;
            if ((st = flashloop_kv_delta_append(c, l, a->k, a->v, 0, rows, 1, c->count[m], stream)) != FLASHLOOP_OK)
                return st;
            if (!a->key_idx) return set_error(FLASHLOOP_ERR_INVALID_ARG, "key_idx is NULL");
            const int K = dm.K < n ? dm.K : n;
            if ((st = flashloop_select_keys(a->c, dm.B, dm.H, n, K, a->key_idx, nullptr, 0, stream)) != FLASHLOOP_OK)
                return st;
            at.K = K;
            at.key_idx = a->key_idx;
        }
        at.n_state = 1;
        at.R = 1;
        at.row_pos = rows;
        at.row_slot = slots;
        return flashloop_lazy_attention(&at, stream);
    }

    // prefill: every token of the sequence is a row
    at.n_state = n;
    if (dense) {
        if ((st = flashloop_kv_dense_store(c, l, a->k, a->v, 0, n, stream)) != FLASHLOOP_OK) return st;
        at.R = n;
        return flashloop_lazy_attention(&at, stream);
    }
    if (!a->h_prev || !a->h_cur || !a->active_idx || !a->key_idx)
        return set_error(FLASHLOOP_ERR_INVALID_ARG, "lazy loop needs h_prev, h_cur, active_idx and key_idx");
    if (dm.R > n || dm.K > n)
        return set_error(FLASHLOOP_ERR_INVALID_ARG, "R=%d and K=%d must not exceed the %d tokens in the cache", dm.R,
                         dm.K, n);
    LazyFront f;
    f.c = c; f.loop = l; f.n = n;
    f.h_prev = a->h_prev; f.h_cur = a->h_cur;
    f.scores = a->scores ? a->scores : reinterpret_cast<float *>(ws + W.scores);
    f.active_idx = a->active_idx; f.key_idx = a->key_idx; f.col = a->c;
    f.key_rank = a->key_rank; f.forced = false;
    f.exit_threshold = a->exit_threshold; f.seq_exit = a->seq_exit;
    f.k = a->k; f.v = a->v;
    st = lazy_front(f, nullptr, stream);
    if (st != FLASHLOOP_OK) return st;
    at.R = dm.R;
    at.row_pos = a->active_idx;
    at.K = dm.K;
    at.key_idx = a->key_idx;
    return fl::lazy_attention_impl(&at, stream, a->seq_exit);
}

namespace fl {
static flashloop_status_t gemm_impl(const uint16_t *a, int M, int K, const uint16_t *w_t, int N, const uint16_t *residual,
                                    int relu, uint16_t *const *c, int n_split, const int32_t *c_rows, int rows_per_seq,
                                    int seq_rows, flashloop_stream_t stream) {
    if (M < 0 || K < 64 || K % 64 || n_split < 1 || n_split > 3 || N < 256 * n_split || N % (256 * n_split))
        return set_error(FLASHLOOP_ERR_INVALID_ARG,
                         "gemm sizes M=%d K=%d N=%d n_split=%d (K %% 64 == 0, N %% (256 n_split) == 0)", M, K, N, n_split);
    if (!a || !w_t || !c) return set_error(FLASHLOOP_ERR_INVALID_ARG, "NULL pointer");
    if (!aligned16(a) || !aligned16(w_t) || (residual && !aligned16(residual)))
        return set_error(FLASHLOOP_ERR_INVALID_ARG, "gemm operands must be 16-byte aligned");
    for (int i = 0; i < n_split; ++i)
        if (!c[i] || !aligned16(c[i])) return set_error(FLASHLOOP_ERR_INVALID_ARG, "output %d NULL or misaligned", i);
    if (c_rows && (rows_per_seq < 1 || M % rows_per_seq || seq_rows < 1))
        return set_error(FLASHLOOP_ERR_INVALID_ARG, "scatter needs rows_per_seq >= 1 dividing M=%d and seq_rows >= 1", M);
    if (M == 0) return FLASHLOOP_OK;
    flashloop_status_t st = check_device();
    if (st != FLASHLOOP_OK) return st;
    const cudaError_t e = launch_gemm(a, M, K, w_t, N, residual, relu, c, n_split, (long long)(N / n_split), c_rows,
                                      rows_per_seq, seq_rows, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "gemm");
    return FLASHLOOP_OK;
}

struct BlockWs {
    size_t step, q, k, v, x, a, y, u, total;
};

// The step's workspace, then q/k/v in token rows, the gathered input rows x,
// the attention outputs a (bf16), y and the MLP activations u.
static BlockWs block_ws(const flashloop_dims_t *dm, int F) {
    BlockWs w;
    const size_t rows = (size_t)dm->B * dm->N_cap, D = (size_t)dm->H * dm->d;
    size_t off = ws_layout(dm).total;
    w.step = 0;
    w.q = off; off += align_up(rows * D * 2);
    w.k = off; off += align_up(rows * D * 2);
    w.v = off; off += align_up(rows * D * 2);
    w.x = off; off += align_up((size_t)dm->B * dm->R_cap * D * 2);
    w.a = off; off += align_up(rows * D * 2);
    w.y = off; off += align_up(rows * D * 2);
    w.u = off; off += align_up(rows * (size_t)F * 2);
    w.total = off;
    return w;
}

static bool block_sizes_ok(const flashloop_dims_t &dm, int F) {
    return (dm.H * dm.d) % 256 == 0 && F >= 256 && F % 256 == 0;
}
}  // namespace fl

size_t flashloop_block_workspace_bytes(const flashloop_dims_t *dims, int32_t F) {
    if (check_dims(dims) != FLASHLOOP_OK || !block_sizes_ok(*dims, F)) return 0;
    return block_ws(dims, F).total;
}

flashloop_status_t flashloop_gemm(const uint16_t *a, int32_t M, int32_t K, const uint16_t *w_t, int32_t N,
                                  const uint16_t *residual, int32_t relu, uint16_t *const *c, int32_t n_split,
                                  const int32_t *c_rows, int32_t rows_per_seq, int32_t seq_rows,
                                  flashloop_stream_t stream) {
    return gemm_impl(a, M, K, w_t, N, residual, relu, c, n_split, c_rows, rows_per_seq, seq_rows, stream);
}

flashloop_status_t flashloop_block_loop(const flashloop_block_args_t *a, flashloop_stream_t stream) {
    if (!a) return set_error(FLASHLOOP_ERR_INVALID_ARG, "args is NULL");
    flashloop_status_t st = check_cache(a->cache);
    if (st != FLASHLOOP_OK) return st;
    flashloop_kv_cache_t *c = a->cache;
    const flashloop_dims_t &dm = c->dims;
    const int l = a->loop;
    if (l < 1 || l > dm.T) return set_error(FLASHLOOP_ERR_INVALID_ARG, "bad loop %d", l);
    const flashloop_block_weights_t *wt = a->weights;
    if (!wt || !wt->w_qkv || !wt->w_o || !wt->w_1 || !wt->w_2)
        return set_error(FLASHLOOP_ERR_INVALID_ARG, "block weights missing");
    const int D = dm.H * dm.d, F = wt->F;
    if (!block_sizes_ok(dm, F))
        return set_error(FLASHLOOP_ERR_INVALID_ARG, "block needs D=%d and F=%d multiples of 256", D, F);
    const BlockWs BW = block_ws(&dm, F);
    if (!a->workspace || a->workspace_bytes < BW.total || reinterpret_cast<uintptr_t>(a->workspace) % kAlign)
        return set_error(FLASHLOOP_ERR_WORKSPACE, "block workspace needs %zu bytes, 256-byte aligned", BW.total);
    const int n = c->n_tokens;
    if (n < 1 || n > dm.N_cap) return set_error(FLASHLOOP_ERR_INVALID_ARG, "cache n_tokens=%d", n);
    if (!a->h_cur || !a->h_out || a->h_out == a->h_cur || !aligned16(a->h_cur) || !aligned16(a->h_out))
        return set_error(FLASHLOOP_ERR_INVALID_ARG, "h_cur/h_out NULL, misaligned or the same buffer");
    const bool dense = l <= dm.T_dense;
    if (!dense && (!a->active_idx || !a->key_idx || (!a->force_selection && !a->h_prev)))
        return set_error(FLASHLOOP_ERR_INVALID_ARG, "lazy loop needs active_idx, key_idx and h_prev");
    if (!dense && a->stale_idx && (a->n_stale < 0 || a->n_stale > n))
        return set_error(FLASHLOOP_ERR_INVALID_ARG, "n_stale=%d outside [0, %d]", a->n_stale, n);
    if (!dense && (dm.R > n || dm.K > n))
        return set_error(FLASHLOOP_ERR_INVALID_ARG, "R=%d and K=%d must not exceed the %d tokens in the cache", dm.R,
                         dm.K, n);
    uint8_t *ws = static_cast<uint8_t *>(a->workspace);
    uint16_t *q = a->q ? a->q : reinterpret_cast<uint16_t *>(ws + BW.q),
             *k = a->k ? a->k : reinterpret_cast<uint16_t *>(ws + BW.k),
             *v = a->v ? a->v : reinterpret_cast<uint16_t *>(ws + BW.v), *xg = reinterpret_cast<uint16_t *>(ws + BW.x),
             *ag = reinterpret_cast<uint16_t *>(ws + BW.a), *yg = reinterpret_cast<uint16_t *>(ws + BW.y),
             *ug = reinterpret_cast<uint16_t *>(ws + BW.u);
    uint16_t *qkv[3] = {q, k, v};
    if (!aligned16(q) || !aligned16(k) || !aligned16(v))
        return set_error(FLASHLOOP_ERR_INVALID_ARG, "q/k/v outputs must be 16-byte aligned");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if ((st = check_device()) != FLASHLOOP_OK) return st;

    flashloop_attn_args_t at;
    memset(&at, 0, sizeof at);
    at.loop = l;
    at.n_keys = n;
    at.n_state = n;
    at.q = q; at.q_hat = a->q_hat; at.o = a->o; at.z = a->z; at.c = a->c;
    at.cache = c;
    at.workspace = a->workspace;
    at.workspace_bytes = a->workspace_bytes;
    at.mode = l == 1 ? FLASHLOOP_ATTN_FIRST_DENSE : dense ? FLASHLOOP_ATTN_DENSE : FLASHLOOP_ATTN_LAZY;

    if (dense) {   // every token: x = H_{l-1}
        const int M = dm.B * n;
        if ((st = gemm_impl(a->h_cur, M, D, wt->w_qkv, 3 * D, nullptr, 0, qkv, 3, nullptr, 0, 0, stream)) != FLASHLOOP_OK)
            return st;
        if ((st = flashloop_kv_dense_store(c, l, k, v, 0, n, stream)) != FLASHLOOP_OK) return st;
        at.R = n;
        if ((st = lazy_attention_impl(&at, stream, nullptr)) != FLASHLOOP_OK) return st;
        cudaError_t e = launch_gather_f32_to_bf16(a->o, dm.B, n, D, nullptr, n, ag, s);
        if (e != cudaSuccess) return cuda_fail(e, "gather of the attention output");
        if ((st = gemm_impl(ag, M, D, wt->w_o, D, a->h_cur, 0, &yg, 1, nullptr, 0, 0, stream)) != FLASHLOOP_OK) return st;
        if ((st = gemm_impl(yg, M, D, wt->w_1, F, nullptr, 1, &ug, 1, nullptr, 0, 0, stream)) != FLASHLOOP_OK) return st;
        uint16_t *ho = a->h_out;
        return gemm_impl(ug, M, F, wt->w_2, D, yg, 0, &ho, 1, nullptr, 0, 0, stream);
    }

    // lazy: only the R active tokens of each sequence are recomputed
    const int R = dm.R, M = dm.B * R;
    LazyFront f;
    f.c = c; f.loop = l; f.n = n;
    f.h_prev = a->h_prev; f.h_cur = a->h_cur;
    f.scores = a->scores ? a->scores : reinterpret_cast<float *>(ws + ws_layout(&dm).scores);
    f.active_idx = a->active_idx; f.key_idx = a->key_idx; f.col = a->c;
    f.key_rank = a->key_rank; f.forced = a->force_selection != 0;
    f.exit_threshold = 0.f; f.seq_exit = nullptr;
    f.k = k; f.v = v;
    st = lazy_front(f, [&]() -> flashloop_status_t {
        // x = H_{l-1}[A]; q, k, v of the active rows, scattered to their token rows
        cudaError_t e = launch_gather_rows(a->h_cur, dm.B, n, D * 2, a->active_idx, R, xg, s);
        if (e != cudaSuccess) return cuda_fail(e, "gather of the active rows");
        return gemm_impl(xg, M, D, wt->w_qkv, 3 * D, nullptr, 0, qkv, 3, a->active_idx, R, n, stream);
    }, stream);
    if (st != FLASHLOOP_OK) return st;
    at.R = R;
    at.row_pos = a->active_idx;
    at.K = dm.K;
    at.key_idx = a->key_idx;
    if ((st = lazy_attention_impl(&at, stream, nullptr)) != FLASHLOOP_OK) return st;
    cudaError_t e = launch_gather_f32_to_bf16(a->o, dm.B, n, D, a->active_idx, R, ag, s);
    if (e != cudaSuccess) return cuda_fail(e, "gather of the attention output");
    if ((st = gemm_impl(ag, M, D, wt->w_o, D, xg, 0, &yg, 1, nullptr, 0, 0, stream)) != FLASHLOOP_OK) return st;
    if ((st = gemm_impl(yg, M, D, wt->w_1, F, nullptr, 1, &ug, 1, nullptr, 0, 0, stream)) != FLASHLOOP_OK) return st;
    // h_out = h_cur outside the active rows: bring its stale rows up to date
    // (after the token selection has read h_prev, which h_out may be)
    if (a->stale_idx)
        e = launch_copy_rows(a->h_cur, dm.B, n, D * 2, a->stale_idx, a->n_stale, a->h_out, s);
    else
        e = cudaMemcpyAsync(a->h_out, a->h_cur, (size_t)dm.B * n * D * 2, cudaMemcpyDeviceToDevice, s);
    if (e != cudaSuccess) return cuda_fail(e, "copy of the stale rows");
    uint16_t *ho = a->h_out;
    return gemm_impl(ug, M, F, wt->w_2, D, yg, 0, &ho, 1, a->active_idx, R, n, stream);
}

flashloop_status_t flashloop_set_wait_limit_ns(uint64_t ns) {
    if (ns > FLASHLOOP_WAIT_LIMIT_DEFAULT_NS)
        return set_error(FLASHLOOP_ERR_INVALID_ARG, "wait limit %llu ns exceeds the default %llu ns",
                         (unsigned long long)ns, (unsigned long long)FLASHLOOP_WAIT_LIMIT_DEFAULT_NS);
    flashloop_status_t st = check_device();
    if (st != FLASHLOOP_OK) return st;
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = static_cast<cudaError_t>(tc_attention_set_wait_limit((unsigned long long)ns));
    if (e != cudaSuccess) return cuda_fail(e, "set wait limit");
    return FLASHLOOP_OK;
}

flashloop_status_t flashloop_device_status(int32_t *word) {
    if (!word) return set_error(FLASHLOOP_ERR_INVALID_ARG, "word is NULL");
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    const int32_t tc = tc_attention_read_error(true), gm = gemm_read_error(true);
    *word = tc ? tc : gm;
    return *word ? FLASHLOOP_ERR_DEVICE : FLASHLOOP_OK;
}

}  // extern "C"

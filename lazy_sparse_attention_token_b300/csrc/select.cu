// select.cu -- token change scores and top-k selection.
//
// rit.work page "FlashLoop: Fast and Memory-Efficient Looped Transformers via
// Lazy Updates", section "FlashLoop combines three kinds of saving": later
// loops rank tokens by how much their hidden states changed and recompute
// only the active ones; keys are chosen from the previous loop's statistics.
// Both rankings keep the top-k with ties to the lower index, ascending.
#include <mutex>

#include "common.cuh"

namespace fl {
namespace {

constexpr int kScoreWarps = 8;

// score[row] = sum_x (h_cur[row,x] - h_prev[row,x])^2 in fp32. One warp per
// token row, 16-byte loads, a shuffle tree for the final sum. Pure stream:
// 2*D*2 bytes read and 4 bytes written per row.
__global__ void __launch_bounds__(kScoreWarps * 32)
token_scores_kernel(const uint16_t *__restrict__ h_prev, const uint16_t *__restrict__ h_cur,
                    long long rows, int D, float *__restrict__ score) {
    const long long row = (long long)blockIdx.x * kScoreWarps + threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const uint4 *a = reinterpret_cast<const uint4 *>(h_prev + row * D);
    const uint4 *b = reinterpret_cast<const uint4 *>(h_cur + row * D);
    const int nv = D / 8;
    float acc = 0.f;
    int v = lane;
    for (; v + 96 < nv; v += 128) {
        uint4 xa[4], xb[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            xa[u] = ldg_nc_v4(a + v + 32 * u);
            xb[u] = ldg_nc_v4(b + v + 32 * u);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            float fa[8], fb[8];
            unpack_bf16x8(xa[u], fa);
            unpack_bf16x8(xb[u], fb);
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const float dlt = fb[e] - fa[e];
                acc = fmaf(dlt, dlt, acc);
            }
        }
    }
    for (; v < nv; v += 32) {
        float fa[8], fb[8];
        unpack_bf16x8(ldg_nc_v4(a + v), fa);
        unpack_bf16x8(ldg_nc_v4(b + v), fb);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const float dlt = fb[e] - fa[e];
            acc = fmaf(dlt, dlt, acc);
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) score[row] = acc;
}

constexpr int kTopkThreads = 1024;
constexpr int kTopkWarps = kTopkThreads / 32;
constexpr int kTopkSmemMaxN = 48 * 1024;   // rows up to this length are staged in shared memory

// Exact top-k of one row of fp32 values per CTA. The k-th largest key is
// found by four 8-bit radix passes (most significant digit first) over
// order-preserving uint32 keys; then elements above it, and the first
// (lowest-index) ones equal to it, are written in ascending index order.
template <bool kStaged>
__global__ void __launch_bounds__(kTopkThreads)
topk_rows_kernel(const float *__restrict__ vals, int n, int k, int32_t *__restrict__ out) {
    extern __shared__ uint32_t staged[];
    __shared__ uint32_t hist[256];
    __shared__ uint32_t s_prefix;
    __shared__ int s_kleft;
    __shared__ unsigned long long warp_tot[kTopkWarps];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const float *row = vals + (size_t)blockIdx.x * n;
    int32_t *orow = out + (size_t)blockIdx.x * k;

    if (kStaged) {
        for (int i = tid; i < n; i += kTopkThreads) staged[i] = f32_order_key(__ldg(row + i));
    }
    auto key_at = [&](int i) -> uint32_t { return kStaged ? staged[i] : f32_order_key(__ldg(row + i)); };

    uint32_t prefix = 0, mask = 0;
    int kleft = k;
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        if (tid < 256) hist[tid] = 0;
        __syncthreads();
        for (int i = tid; i < n; i += kTopkThreads) {
            const uint32_t key = key_at(i);
            if ((key & mask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
        }
        __syncthreads();
        if (warp == 0) {
            uint32_t c[8], local = 0;
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                c[t] = hist[255 - 8 * lane - t];
                local += c[t];
            }
            uint32_t incl = local;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const uint32_t y = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += y;
            }
            const uint32_t hit = __ballot_sync(0xffffffffu, incl >= (uint32_t)kleft);
            const int first = __ffs(hit) - 1;
            if (lane == first) {
                uint32_t run = incl - local;
#pragma unroll
                for (int t = 0; t < 8; ++t) {
                    if (run + c[t] >= (uint32_t)kleft) {
                        const uint32_t bin = 255u - 8u * lane - t;
                        s_prefix = prefix | (bin << shift);
                        s_kleft = kleft - (int)run;
                        break;
                    }
                    run += c[t];
                }
            }
        }
        __syncthreads();
        prefix = s_prefix;
        kleft = s_kleft;
        mask |= 255u << shift;
    }
    const uint32_t thr = prefix;   // the k-th largest key
    const int need_eq = kleft;     // how many elements equal to it are kept

    // Each warp owns one contiguous segment; lanes walk it 32 at a time so
    // the loads stay coalesced and ballots keep index order.
    const int seg = ((n + kTopkWarps - 1) / kTopkWarps + 31) & ~31;
    const int lo = warp * seg, hi = min(n, lo + seg);
    const unsigned lt = (1u << lane) - 1u;
    uint32_t gt_cnt = 0, eq_cnt = 0;
    for (int base = lo; base < hi; base += 32) {
        const int i = base + lane;
        const uint32_t key = i < hi ? key_at(i) : 0u;
        gt_cnt += __popc(__ballot_sync(0xffffffffu, i < hi && key > thr));
        eq_cnt += __popc(__ballot_sync(0xffffffffu, i < hi && key == thr));
    }
    if (lane == 0) warp_tot[warp] = ((unsigned long long)gt_cnt << 32) | eq_cnt;
    __syncthreads();
    unsigned long long before = 0;
    for (int w = 0; w < warp; ++w) before += warp_tot[w];
    uint32_t gt_run = (uint32_t)(before >> 32), eq_run = (uint32_t)(before & 0xffffffffu);
    for (int base = lo; base < hi; base += 32) {
        const int i = base + lane;
        const uint32_t key = i < hi ? key_at(i) : 0u;
        const uint32_t gb = __ballot_sync(0xffffffffu, i < hi && key > thr);
        const uint32_t eb = __ballot_sync(0xffffffffu, i < hi && key == thr);
        const int eq_left = max(0, need_eq - (int)eq_run);
        const int eq_take = min(eq_left, __popc(eb));
        const int out_base = (int)gt_run + min((int)eq_run, need_eq);
        if (gb & (1u << lane)) {
            orow[out_base + __popc(gb & lt) + min(__popc(eb & lt), eq_take)] = i;
        } else if ((eb & (1u << lane)) && __popc(eb & lt) < eq_take) {
            orow[out_base + __popc(gb & lt) + __popc(eb & lt)] = i;
        }
        gt_run += __popc(gb);
        eq_run += __popc(eb);
    }
}

}  // namespace

cudaError_t launch_token_scores(const uint16_t *h_prev, const uint16_t *h_cur, int B, int N, int D,
                                float *scores, cudaStream_t s) {
    const long long rows = (long long)B * N;
    {
        KernelTimer kt("token_scores", s);
        token_scores_kernel<<<ceil_div(rows, kScoreWarps), kScoreWarps * 32, 0, s>>>(h_prev, h_cur, rows, D, scores);
    }
    return cudaGetLastError();
}

cudaError_t launch_topk_rows(const float *vals, int rows, int n, int k, int32_t *out, cudaStream_t s) {
    if (rows == 0) return cudaSuccess;
    if (n <= kTopkSmemMaxN) {
        const size_t smem = (size_t)n * 4;
        static bool attr_set = false;
        if (!attr_set) {
            cudaFuncSetAttribute(topk_rows_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kTopkSmemMaxN * 4);
            attr_set = true;
        }
        {
            KernelTimer kt("topk", s);
            topk_rows_kernel<true><<<rows, kTopkThreads, smem, s>>>(vals, n, k, out);
        }
    } else {
        {
            KernelTimer kt("topk", s);
            topk_rows_kernel<false><<<rows, kTopkThreads, 0, s>>>(vals, n, k, out);
        }
    }
    return cudaGetLastError();
}

}  // namespace fl

// ---------------------------------------------------------------------------
// Token selection without allocation.
//
// For callers that may not allocate device memory at all: code that runs
// inside a memory arena it does not own (a serving engine's fixed budget, a
// plugin host), or on a path where an allocation could stall or fail at the
// wrong moment. The change scores, the only scratch this step needs, live in
// a fixed array of this library instead of a caller workspace. Every device
// that loads the library holds the array until the process exits.
namespace fl {
namespace {
constexpr long long kNoAllocMaxScores = 1ll << 20;   // B * N limit: 1,048,576 fp32 scores (4 MiB)
constexpr int kNoAllocMaxDevices = 64;
static __device__ __align__(256) float g_noalloc_scores[kNoAllocMaxScores];
std::mutex g_noalloc_mu;
float *g_noalloc_ptr[kNoAllocMaxDevices] = {};
}  // namespace

}  // namespace fl

using namespace fl;

extern "C" flashloop_status_t flashloop_select_tokens_noalloc(const uint16_t *h_prev, const uint16_t *h_cur,
                                                              int32_t B, int32_t N, int32_t D, int32_t R,
                                                              int32_t *active_idx, flashloop_stream_t stream) {
    if (!h_prev || !h_cur || !active_idx) return set_error(FLASHLOOP_ERR_INVALID_ARG, "NULL pointer");
    if ((reinterpret_cast<uintptr_t>(h_prev) | reinterpret_cast<uintptr_t>(h_cur)) & 15u)
        return set_error(FLASHLOOP_ERR_INVALID_ARG, "inputs must be 16-byte aligned");
    if (B < 1 || N < 1 || D < 8 || D % 8 || R < 1 || R > N)
        return set_error(FLASHLOOP_ERR_INVALID_ARG, "bad sizes (B=%d N=%d D=%d R=%d)", B, N, D, R);
    if ((long long)B * N > kNoAllocMaxScores)
        return set_error(FLASHLOOP_ERR_CAPACITY, "B*N = %lld exceeds the fixed scratch of %lld scores",
                         (long long)B * N, kNoAllocMaxScores);
    flashloop_status_t st = check_device();
    if (st != FLASHLOOP_OK) return st;
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kNoAllocMaxDevices) return set_error(FLASHLOOP_ERR_UNSUPPORTED, "device index %d", dev);
    float *scores = nullptr;
    {
        // once per device, with that device current: the device address of the array
        std::lock_guard<std::mutex> lock(g_noalloc_mu);
        if (!g_noalloc_ptr[dev]) {
            e = cudaGetSymbolAddress(reinterpret_cast<void **>(&g_noalloc_ptr[dev]), g_noalloc_scores);
            if (e != cudaSuccess) {
                g_noalloc_ptr[dev] = nullptr;
                return cuda_fail(e, "cudaGetSymbolAddress(scratch)");
            }
        }
        scores = g_noalloc_ptr[dev];
    }
    // every score is written before it is read: nothing needs clearing
    e = launch_token_scores(h_prev, h_cur, B, N, D, scores, stream);
    if (e != cudaSuccess) return cuda_fail(e, "token_scores");
    e = launch_topk_rows(scores, B, N, R, active_idx, stream);
    if (e != cudaSuccess) return cuda_fail(e, "topk(tokens)");
    return FLASHLOOP_OK;
}

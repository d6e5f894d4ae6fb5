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
    pdl_wait();
    pdl_trigger();
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


// ---- top-k over a cluster of CTAs --------------------------------------------
// Exact top-k of each row of fp32 values: the k-th largest order-preserving
// uint32 key is found by four 8-bit radix passes (most significant digit
// first); then the keys above it, and the first (lowest-index) ones equal to
// it, are written in ascending index order. A row is split over a cluster of
// up to kTopkCluster CTAs (one row alone would otherwise run on a single SM;
// with many rows, one CTA per row already fills the GPU): each
// CTA histograms its own contiguous segment and adds the histogram into a
// fresh one on every rank of the cluster (distributed shared memory: remote
// additions that need no reply); after one cluster barrier every rank reads the
// merged histogram from its own shared memory and takes the same digit (reading
// one rank's copy remotely instead cost about 6 us per 32K-key selection). The
// output order is rank order, then warp segments, so indices stay ascending.
constexpr int kTopkCluster = 8;
constexpr int kTopkClThreads = 512;
constexpr int kTopkClWarps = kTopkClThreads / 32;
constexpr int kTopkClStageMax = 48 * 1024;   // keys per CTA staged in shared memory (192 KB)
constexpr int kTopkRowsForSingle = 128;      // with this many rows, one CTA per row fills the GPU

__device__ __forceinline__ uint32_t cl_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cl_size() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cl_map(const void *p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"((uint32_t)__cvta_generic_to_shared(p)), "r"(rank));
    return r;
}
__device__ __forceinline__ void cl_red_add(uint32_t addr, uint32_t v) {
    asm volatile("red.shared::cluster.add.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t cl_ld(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ void cl_red_max(uint32_t addr, uint32_t v) {
    asm volatile("red.shared::cluster.max.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
// Inverse of f32_order_key (for keys of finite values; -0 comes back as +0).
__device__ __forceinline__ float order_key_f32(uint32_t key) {
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}
__device__ __forceinline__ void cl_st(uint32_t addr, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
// Every thread of every CTA of the cluster passes each of these.
__device__ __forceinline__ void cl_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// norm_n > 0 ranks column i of a row by vals[i] / (norm_n - i) (IEEE fp32
// division) instead of vals[i]: a key's column mass per causal row that sees it.
// seq_exit != NULL: the row's largest value (a sequence's largest token change
// score) is found on the way, and if it is below exit_thr the row's flag is set
// to 1 (flags are only ever set here, never cleared).
template <bool kStaged>
__global__ void __launch_bounds__(kTopkClThreads)
topk_cluster_kernel(const float *__restrict__ vals, int n, int k, int32_t *__restrict__ out, int norm_n,
                    float exit_thr, int32_t *__restrict__ seq_exit) {
    extern __shared__ uint32_t staged[];
    __shared__ uint32_t whist[kTopkClWarps][256];   // one histogram per warp: keys of similar
                                                    // magnitude share a digit, so a single
                                                    // histogram would serialise on one bin
    __shared__ uint32_t g_hist[4][256];        // merged histograms: every rank adds its counts into every rank's
    __shared__ uint32_t cta_cnt[kTopkCluster][2];   // every rank's (greater, equal) counts, on every rank
    __shared__ uint32_t s_prefix;
    __shared__ int s_kleft;
    __shared__ unsigned long long warp_tot[kTopkClWarps];
    __shared__ uint32_t s_cta_max, s_row_max;   // largest key of this CTA's segment / of the row (rank 0)

    pdl_wait();
    pdl_trigger();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t rank = cl_rank(), ncta = cl_size();
    const int row_id = blockIdx.x / ncta;
    const float *row = vals + (size_t)row_id * n;
    int32_t *orow = out + (size_t)row_id * k;
    // this CTA's segment of the row, a multiple of 32 keys
    const int seg = ((n + (int)ncta - 1) / (int)ncta + 31) & ~31;
    const int lo = min(n, (int)rank * seg), hi = min(n, lo + seg), len = hi - lo;

    for (int i = tid; i < 4 * 256; i += kTopkClThreads) (&g_hist[0][0])[i] = 0u;
    if (tid == 0) {
        s_cta_max = 0u;
        s_row_max = 0u;
    }
    auto value_at = [&](int i) -> float {
        const float v = __ldg(row + lo + i);
        return norm_n > 0 ? __fdiv_rn(v, (float)(norm_n - (lo + i))) : v;
    };
    if (kStaged)
        for (int i = tid; i < len; i += kTopkClThreads) staged[i] = f32_order_key(value_at(i));
    auto key_at = [&](int i) -> uint32_t { return kStaged ? staged[i] : f32_order_key(value_at(i)); };
    cl_sync();   // rank 0's merged histograms are zero; every CTA of the cluster runs

    uint32_t prefix = 0, mask = 0;
    int kleft = k;
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        for (int i = tid; i < kTopkClWarps * 256; i += kTopkClThreads) (&whist[0][0])[i] = 0u;
        __syncthreads();
        uint32_t kmax = 0u;
        for (int i = tid; i < len; i += kTopkClThreads) {
            const uint32_t key = key_at(i);
            if ((key & mask) == prefix) atomicAdd(&whist[warp][(key >> shift) & 255u], 1u);
            kmax = max(kmax, key);
        }
        if (pass == 0 && seq_exit) {
            kmax = __reduce_max_sync(0xffffffffu, kmax);
            if (lane == 0) atomicMax(&s_cta_max, kmax);
        }
        __syncthreads();
        if (tid < 256) {
            uint32_t tot = 0;
#pragma unroll
            for (int w = 0; w < kTopkClWarps; ++w) tot += whist[w][tid];
            if (tot != 0u)
                for (uint32_t q = 0; q < ncta; ++q) cl_red_add(cl_map(&g_hist[pass][tid], q), tot);
        }
        if (pass == 0 && seq_exit && tid == 0 && len > 0) cl_red_max(cl_map(&s_row_max, 0), s_cta_max);
        cl_sync();
        if (pass == 0 && seq_exit && rank == 0 && tid == 0 && order_key_f32(s_row_max) < exit_thr)
            seq_exit[row_id] = 1;
        if (warp == 0) {
            uint32_t c[8], local = 0;
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                c[t] = g_hist[pass][255 - 8 * lane - t];
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
    const int need_eq = kleft;     // how many keys equal to it are kept

    // counts in this CTA's segment, warp by warp (each warp owns a contiguous part)
    const int wseg = ((len + kTopkClWarps - 1) / kTopkClWarps + 31) & ~31;
    const int wlo = min(len, warp * wseg), whi = min(len, wlo + wseg);
    const unsigned lt = (1u << lane) - 1u;
    uint32_t gt_cnt = 0, eq_cnt = 0;
    for (int base = wlo; base < whi; base += 32) {
        const int i = base + lane;
        const uint32_t key = i < whi ? key_at(i) : 0u;
        gt_cnt += __popc(__ballot_sync(0xffffffffu, i < whi && key > thr));
        eq_cnt += __popc(__ballot_sync(0xffffffffu, i < whi && key == thr));
    }
    if (lane == 0) warp_tot[warp] = ((unsigned long long)gt_cnt << 32) | eq_cnt;
    __syncthreads();
    if (tid == 0) {
        unsigned long long tot = 0;
        for (int w = 0; w < kTopkClWarps; ++w) tot += warp_tot[w];
        for (uint32_t q = 0; q < ncta; ++q) {
            cl_st(cl_map(&cta_cnt[rank][0], q), (uint32_t)(tot >> 32));
            cl_st(cl_map(&cta_cnt[rank][1], q), (uint32_t)(tot & 0xffffffffu));
        }
    }
    cl_sync();
    // keys before this CTA's segment (lower ranks), then before this warp's part
    uint32_t gt_run = 0, eq_run = 0;
    for (uint32_t q = 0; q < rank; ++q) {
        gt_run += cta_cnt[q][0];
        eq_run += cta_cnt[q][1];
    }
    for (int w = 0; w < warp; ++w) {
        gt_run += (uint32_t)(warp_tot[w] >> 32);
        eq_run += (uint32_t)(warp_tot[w] & 0xffffffffu);
    }
    for (int base = wlo; base < whi; base += 32) {
        const int i = base + lane;
        const uint32_t key = i < whi ? key_at(i) : 0u;
        const uint32_t gb = __ballot_sync(0xffffffffu, i < whi && key > thr);
        const uint32_t eb = __ballot_sync(0xffffffffu, i < whi && key == thr);
        const int eq_left = max(0, need_eq - (int)eq_run);
        const int eq_take = min(eq_left, __popc(eb));
        const int out_base = (int)gt_run + min((int)eq_run, need_eq);
        if (gb & (1u << lane)) {
            orow[out_base + __popc(gb & lt) + min(__popc(eb & lt), eq_take)] = lo + i;
        } else if ((eb & (1u << lane)) && __popc(eb & lt) < eq_take) {
            orow[out_base + __popc(gb & lt) + __popc(eb & lt)] = lo + i;
        }
        gt_run += __popc(gb);
        eq_run += __popc(eb);
    }
    cl_sync();   // rank 0's counts stay readable until every rank is done with them
}

}  // namespace

cudaError_t launch_token_scores(const uint16_t *h_prev, const uint16_t *h_cur, int B, int N, int D,
                                float *scores, cudaStream_t s) {
    const long long rows = (long long)B * N;
    {
        KernelTimer kt("token_scores", s);
        const cudaError_t e = launch_pdl(token_scores_kernel, dim3(ceil_div(rows, kScoreWarps)),
                                         dim3(kScoreWarps * 32), 0, s, h_prev, h_cur, rows, D, scores);
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

cudaError_t launch_topk_rows(const float *vals, int rows, int n, int k, int32_t *out, cudaStream_t s,
                             const char *name, int norm_n, float exit_thr, int32_t *seq_exit) {
    if (rows == 0) return cudaSuccess;
    const int ncta = rows >= kTopkRowsForSingle ? 1 : kTopkCluster;
    const int seg = ((n + ncta - 1) / ncta + 31) & ~31;
    const bool staged = seg <= kTopkClStageMax;
    static std::once_flag once[kMaxDevices];
    static cudaError_t attr_res[kMaxDevices];
    const cudaError_t ea = once_per_device(once, attr_res, [] {
        return cudaFuncSetAttribute(topk_cluster_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    kTopkClStageMax * 4);
    });
    if (ea != cudaSuccess) return ea;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(rows * ncta));
    cfg.blockDim = dim3(kTopkClThreads);
    cfg.dynamicSmemBytes = staged ? (size_t)seg * 4 : 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)ncta;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // see pdl_wait()
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t e;
    {
        KernelTimer kt(name, s);
        e = staged ? cudaLaunchKernelEx(&cfg, topk_cluster_kernel<true>, vals, n, k, out, norm_n, exit_thr, seq_exit)
                   : cudaLaunchKernelEx(&cfg, topk_cluster_kernel<false>, vals, n, k, out, norm_n, exit_thr, seq_exit);
    }
    return e != cudaSuccess ? e : cudaGetLastError();
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
    e = launch_topk_rows(scores, B, N, R, active_idx, stream, "topk_tokens");
    if (e != cudaSuccess) return cuda_fail(e, "topk(tokens)");
    return FLASHLOOP_OK;
}

// gemm.cu -- bf16 GEMM on the tcgen05 tensor cores for the synthetic looped
// block around the lazy step.
//
// rit.work page "FlashLoop: Fast and Memory-Efficient Looped Transformers via
// Lazy Updates", section "FlashLoop combines three kinds of saving": a later
// loop recomputes only its active tokens, the rest reuse their state. The
// block's projections and MLP therefore run on the gathered active rows only:
//   C[m, :] = act(A[m, :] W^T + residual[m, :]),   act = identity or ReLU,
// with A [M, K] bf16 (rows of the active tokens), W^T stored as [N, K] bf16
// (each output column's weights contiguous), fp32 accumulation in TMEM and a
// bf16 result (round to nearest even) written to row c_rows[m] (or m) of one
// of n_split outputs of N / n_split columns each.
//
// A persistent kernel: one CTA per SM walks the 128 x 256 output tiles
// (column tiles fastest, so CTAs running together share A rows in L2). Warp 0
// streams K-slices of 64 elements of A (128 rows) and W^T (256 rows) by TMA
// (128-byte swizzle) through a ring of kStages slots, across tile boundaries;
// warp 1 allocates TMEM and one of its threads issues the tcgen05.mma products
// (M 128, N 256, K 16, both operands K-major in shared memory) of each tile
// into one of two 256-column fp32 accumulators; warps 2..5 (one per TMEM lane
// quadrant) read a finished accumulator back 32 columns at a time, release it
// to the next tile's products, add the residual, apply the activation and
// store bf16, while the products of the next tile run. Every mbarrier wait is
// bounded (one second); a CTA that gives up records an error word, lets its
// own copies and MMAs land, frees TMEM and exits.
#include <cudaTypedefs.h>
#include <mutex>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace fl {
namespace {

using namespace ptx;

constexpr int GM = 128;              // rows of an output tile
constexpr int GN = 256;              // columns of an output tile
constexpr int GK = 64;               // K-slice per ring slot (one 128-byte swizzle atom)
constexpr int kStages = 4;
constexpr int kThreads = 192;        // warp 0 TMA, warp 1 MMA, warps 2..5 epilogue
constexpr int A_BYTES = GM * GK * 2;     // 16 KB
constexpr int B_BYTES = GN * GK * 2;     // 32 KB
constexpr int STAGE = A_BYTES + B_BYTES;
constexpr int OFF_BAR = kStages * STAGE;
constexpr int kEpiWarps = 4;
constexpr uint32_t kTmemCols = 2 * GN;   // two accumulators
// FULL[s]/EMPTY[s]: ring slot s landed / free again; ACC_FULL[b]: accumulator b
// holds a finished tile; ACC_EMPTY[b]: the epilogue has read it (one arrival
// per epilogue warp).
enum : int { BAR_FULL = 0, BAR_EMPTY = kStages, BAR_ACC_FULL = 2 * kStages, BAR_ACC_EMPTY = BAR_ACC_FULL + 2,
             BAR_DRAIN = BAR_ACC_EMPTY + 2, N_BARS = BAR_DRAIN + 1 };
constexpr int OFF_MISC = OFF_BAR + N_BARS * 8;
constexpr int SMEM = OFF_MISC + 16 + 1024;   // + room to align the base to 1024 bytes
static_assert(SMEM <= 232448, "shared memory budget");
constexpr unsigned long long kLimitNs = FLASHLOOP_WAIT_LIMIT_DEFAULT_NS;

__device__ int g_gemm_error;
constexpr int kErrWait = 0x100;      // a bounded wait gave up
constexpr int kErrRow = 0x101;       // an output row index outside [0, seq_rows): that row is not stored

struct GemmParams {
    int M, N, K, n_split, relu;
    long long c_ld;                  // row stride (elements) of each output
    const uint16_t *residual;        // [M, N] bf16 or NULL
    const int32_t *c_rows;           // [M] output row of each A row, or NULL
    int rows_per_seq, seq_rows;      // with c_rows: A row m goes to row (m / rows_per_seq) * seq_rows + c_rows[m]
    uint16_t *c[3];                  // n_split outputs
};

__device__ bool gemm_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag, bool drain) {
    if (mbar_test_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 8; ++i)
            if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
        if (!drain && *abort_flag) return false;
        if (globaltimer_ns() - t0 >= kLimitNs) {
            if (!drain) {
                *abort_flag = 1;
                atomicCAS(&g_gemm_error, 0, kErrWait);
            }
            return false;
        }
    }
}

// 2-D TMA load of a (64-element, rows) box at column c0, row c1.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, uint32_t bar, int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::
            "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1)
        : "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
gemm_kernel(const __grid_constant__ GemmParams p, const __grid_constant__ CUtensorMap tm_a,
            const __grid_constant__ CUtensorMap tm_b) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    auto bar = [&](int i) { return sbase + OFF_BAR + 8u * (uint32_t)i; };
    uint32_t *misc = reinterpret_cast<uint32_t *>(smem + OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(misc + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_k = p.K / GK;
    const int tiles_n = p.N / GN, tiles = tiles_n * ((p.M + GM - 1) / GM);

    if (threadIdx.x == 0) {
        for (int i = 0; i < N_BARS; ++i) mbar_init(bar(i), (i == BAR_ACC_EMPTY || i == BAR_ACC_EMPTY + 1) ? kEpiWarps : 1u);
        misc[1] = 0;
        mbar_fence_init();
    }
    if (warp == 1) {
        tmem_alloc(sbase + OFF_MISC, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];

    if (warp == 0 && lane == 0) {
        // ---- TMA producer: the K-slices of every tile of this CTA, through one ring ----
        prefetch_tmap(&tm_a);
        prefetch_tmap(&tm_b);
        int it = 0;   // slices issued
        bool ok = true;
        for (int tile = blockIdx.x; ok && tile < tiles; tile += gridDim.x) {
            const int n0 = (tile % tiles_n) * GN, m0 = (tile / tiles_n) * GM;
            for (int kb = 0; kb < n_k; ++kb, ++it) {
                const int s = it % kStages, use = it / kStages;
                if (!(ok = gemm_wait(bar(BAR_EMPTY + s), (use & 1) ^ 1, abort_flag, false))) break;
                const uint32_t dst = sbase + s * STAGE;
                mbar_arrive_expect_tx(bar(BAR_FULL + s), STAGE);
                tma_load_2d(dst, &tm_a, bar(BAR_FULL + s), kb * GK, m0);
                tma_load_2d(dst + A_BYTES, &tm_b, bar(BAR_FULL + s), kb * GK, n0);
            }
        }
        if (*abort_flag)   // let copies already in flight land before the CTA exits
            for (int q = max(0, it - kStages); q < it; ++q)
                gemm_wait(bar(BAR_FULL + q % kStages), (q / kStages) & 1, abort_flag, true);
    } else if (warp == 1 && lane == 0) {
        // ---- MMA issuer: tile j of this CTA into accumulator j & 1 ----
        constexpr uint32_t idesc = idesc_bf16(GM, GN, false, false, false);
        bool ok = true;
        int it = 0, j = 0;
        for (int tile = blockIdx.x; ok && tile < tiles; tile += gridDim.x, ++j) {
            const int ab = j & 1;
            // the epilogue has read this accumulator's previous tile
            if (!(ok = gemm_wait(bar(BAR_ACC_EMPTY + ab), ((j >> 1) & 1) ^ 1, abort_flag, false))) break;
            tc_fence_after();
            const uint32_t acc = tmem + (uint32_t)(ab * GN);
            for (int kb = 0; kb < n_k; ++kb, ++it) {
                const int s = it % kStages;
                if (!(ok = gemm_wait(bar(BAR_FULL + s), (it / kStages) & 1, abort_flag, false))) break;
                tc_fence_after();
                const uint64_t da = smem_desc(sbase + s * STAGE, 16, 1024, 2);
                const uint64_t db = smem_desc(sbase + s * STAGE + A_BYTES, 16, 1024, 2);
#pragma unroll
                for (int kk = 0; kk < GK / 16; ++kk)   // K = 16 per product: 32 bytes further along the atom
                    mma_bf16_ss(acc, da + 2 * kk, db + 2 * kk, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
                mma_commit(bar(BAR_EMPTY + s));
            }
            if (ok) mma_commit(bar(BAR_ACC_FULL + ab));
        }
        if (!ok) {   // drain whatever was issued before giving up
            mma_commit(bar(BAR_DRAIN));
            gemm_wait(bar(BAR_DRAIN), 0, abort_flag, true);
        }
    } else if (warp >= 2) {
        // ---- epilogue: warp w reads TMEM lane quadrant w % 4 (rows 32 (w % 4) ..) ----
        const int q = warp & 3;
        const int per = p.N / p.n_split;   // columns of each output (a multiple of GN)
        int j = 0;
        for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x, ++j) {
            const int ab = j & 1;
            const int n0 = (tile % tiles_n) * GN, m0 = (tile / tiles_n) * GM;
            const int r = q * 32 + lane, m = m0 + r;
            if (!__all_sync(0xffffffffu, gemm_wait(bar(BAR_ACC_FULL + ab), (j >> 1) & 1, abort_flag, false))) break;
            tc_fence_after();
            bool row_ok = m < p.M;
            const int out = n0 / per, nc = n0 - out * per;
            uint16_t *dst = nullptr;
            if (row_ok) {
                long long orow = m;
                if (p.c_rows) {
                    const int i = __ldg(p.c_rows + m);
                    if (i < 0 || i >= p.seq_rows) {
                        atomicCAS(&g_gemm_error, 0, kErrRow);
                        row_ok = false;
                    }
                    orow = (long long)(m / p.rows_per_seq) * p.seq_rows + i;
                }
                dst = p.c[out] + orow * p.c_ld + nc;
            }
            const uint16_t *res = row_ok && p.residual ? p.residual + (long long)m * p.N + n0 : nullptr;
            const uint32_t acc = tmem + (uint32_t)(ab * GN) + ((uint32_t)(q * 32) << 16);
#pragma unroll 1
            for (int c = 0; c < GN / 32; ++c) {
                float v[32];
                tmem_ld_32x32b_x32(acc + 32u * c, v);
                tmem_wait_ld();
                if (c == GN / 32 - 1) {   // the accumulator is read: the next tile may use it
                    tc_fence_before();
                    __syncwarp();
                    mbar_arrive_elected(bar(BAR_ACC_EMPTY + ab));
                }
                if (!row_ok) continue;
                if (res) {
                    const uint4 *r4 = reinterpret_cast<const uint4 *>(res + 32 * c);
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        float f[8];
                        unpack_bf16x8(__ldg(r4 + u), f);
#pragma unroll
                        for (int e = 0; e < 8; ++e) v[8 * u + e] = __fadd_rn(v[8 * u + e], f[e]);
                    }
                }
                if (p.relu) {
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = fmaxf(v[e], 0.f);
                }
                uint4 *d4 = reinterpret_cast<uint4 *>(dst + 32 * c);
#pragma unroll
                for (int u = 0; u < 4; ++u)
                    d4[u] = make_uint4(pack_bf16x2_rn(v[8 * u], v[8 * u + 1]), pack_bf16x2_rn(v[8 * u + 2], v[8 * u + 3]),
                                       pack_bf16x2_rn(v[8 * u + 4], v[8 * u + 5]),
                                       pack_bf16x2_rn(v[8 * u + 6], v[8 * u + 7]));
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        void *ptr = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// 2-D bf16 map of a [rows, cols] row-major array, box (64 columns, box_rows rows), 128-byte swizzle.
bool make_map_2d(CUtensorMap *map, const void *base, long long rows, long long cols, int box_rows) {
    auto enc = encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t str[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {(cuuint32_t)GK, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, str, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_gemm(const uint16_t *a, int M, int K, const uint16_t *wt, int N, const uint16_t *residual, int relu,
                        uint16_t *const *c, int n_split, long long c_ld, const int32_t *c_rows, int rows_per_seq,
                        int seq_rows, cudaStream_t s) {
    if (M == 0) return cudaSuccess;
    static std::once_flag once[kMaxDevices];
    static cudaError_t attr_res[kMaxDevices];
    const cudaError_t ea = once_per_device(once, attr_res, [] {
        return cudaFuncSetAttribute(gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    });
    if (ea != cudaSuccess) return ea;
    CUtensorMap ma, mb;
    if (!make_map_2d(&ma, a, M, K, GM) || !make_map_2d(&mb, wt, N, K, GN)) return cudaErrorInvalidValue;
    GemmParams p;
    p.M = M; p.N = N; p.K = K; p.n_split = n_split; p.relu = relu; p.c_ld = c_ld;
    p.residual = residual; p.c_rows = c_rows;
    p.rows_per_seq = rows_per_seq > 0 ? rows_per_seq : M; p.seq_rows = seq_rows;
    for (int i = 0; i < 3; ++i) p.c[i] = i < n_split ? c[i] : nullptr;
    static int sms[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (sms[dev] == 0 && cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return cudaErrorInvalidDevice;
    const long long tiles = (long long)(N / GN) * ceil_div(M, GM);
    dim3 grid((unsigned)(tiles < sms[dev] ? tiles : sms[dev]));
    {
        KernelTimer kt("gemm", s);
        const cudaError_t e = launch_pdl(gemm_kernel, grid, dim3(kThreads), (size_t)SMEM, s, p, ma, mb);
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

int32_t gemm_read_error(bool clear) {
    int v = 0;
    cudaMemcpyFromSymbol(&v, g_gemm_error, sizeof(int));
    if (clear && v) {
        int zero = 0;
        cudaMemcpyToSymbol(g_gemm_error, &zero, sizeof(int));
    }
    return v;
}

}  // namespace fl

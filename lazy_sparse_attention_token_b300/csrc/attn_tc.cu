// attn_tc.cu -- lazy (and dense) attention on the tcgen05 tensor cores.
//
// rit.work page "FlashLoop: Fast and Memory-Efficient Looped Transformers via
// Lazy Updates", section "FlashLoop combines three kinds of saving": in a lazy
// loop only active rows are recomputed, keys are chosen from the previous
// loop's statistics, and the chosen group keeps its total probability mass
// (dropping the other keys and renormalising would give the survivors too
// much weight); early loops run in full.
//
// For one (sequence b, head h, tile of 128 rows) a CTA computes, per row i
// with S_i = {j in S : j <= i}, scale s = 1/sqrt(d):
//   p_j = exp(qhat_i.k_j^(l-1) s - Z_i),  m = sum p_j,  u = sum p_j v_j^(l-1)
//   lam = logsumexp(q_i.k_j^(l) s),       Z' = lam - ln m
//   acc = -u + sum exp(q_i.k_j^(l) s - Z') v_j^(l)        (= -u + m w)
//   O_i += acc,  Z_i = Z',  qhat_i = q_i,
//   c_j += sum_i exp(q_i.k_j^(l) s - Z'_i) - p_ij         (column mass)
// in three passes over the key tiles, all with a known normaliser so no
// accumulator rescaling is ever needed:
//   pass OLD: QK_old -> p -> m, acc -= P V_old, colsum -= P
//   pass LSE: QK_new -> online max/sum -> lam
//   pass NEW: QK_new -> P' = exp(. - Z') -> acc += P' V_new, colsum += P'
// The first dense loop skips pass OLD (m = 1, u = 0).
//
// Roles (320 threads): warp 0 issues TMA loads into a K ring and a V ring
// (2 stages each; a K slot is released as soon as its QK product is done);
// warp 1 (one thread) issues tcgen05.mma into TMEM; warps 2..9 are two
// softmax warpgroups that each own one TMEM lane (= one row) and one half
// of the tile's 128 columns: they read S, do the softmax arithmetic, write
// P as bf16 into one of two shared buffers for the PV and column-sum MMAs
// (so the next tile's P never waits for the current PV), merge their row
// statistics once through TMEM, and split the epilogue. One query tile
// holds qhat for pass OLD and is reloaded with q before pass LSE. Column sums are an MMA of P^T (the same shared tile read
// MN-major) with a ones matrix, so no cross-thread reduction is needed.
// TMEM columns: S double buffer [0,256), accumulator [256,256+d), column
// sums double buffer [384,416), row-statistics exchange [448,456).
//
// Waiting threads sleep in a hinted try_wait instead of spinning. Every
// mbarrier wait is bounded (about one second); on timeout the CTA records an
// error code, stops issuing work, waits (bounded) for its own copies and
// MMAs, frees TMEM and exits.
#include <cudaTypedefs.h>
#include <float.h>
#include <mutex>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace fl {
namespace {

using namespace ptx;

constexpr int BM = 128;
constexpr int BN = 128;
constexpr int kThreads = 320;     // warp 0 TMA, warp 1 MMA, warps 2..5 and 6..9 softmax (column halves)
constexpr int kSoftmax = 256;
constexpr int kAtom = 128 * 128;  // bytes of a 128-row x 64-element bf16 tile, 128-byte swizzled
constexpr uint32_t kTmemCols = 512;
// TMEM columns: S double buffer, accumulator, column sums (double buffer), row-statistics exchange
constexpr uint32_t kColS = 0, kColAcc = 256, kColCS = 384, kColX = 448;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ int g_tc_error;

enum : int { PH_OLD = 0, PH_LSE = 1, PH_NEW = 2 };
enum : int { BAR_K_FULL = 0, BAR_K_EMPTY = 2, BAR_V_FULL = 4, BAR_V_EMPTY = 6, BAR_S_FULL = 8,
             BAR_S_EMPTY = 10, BAR_P_FULL = 12, BAR_P_EMPTY = 14, BAR_ACC = 16, BAR_STATS = 17,
             BAR_Q_READY = 18, BAR_DRAIN = 19, N_BARS = 20 };
enum : int { ERR_K_EMPTY = 1, ERR_K_FULL = 2, ERR_V_EMPTY = 3, ERR_V_FULL = 4, ERR_S_EMPTY = 5, ERR_S_FULL = 6,
             ERR_P_FULL = 7, ERR_P_EMPTY = 8, ERR_ACC = 9, ERR_STATS = 10, ERR_Q_READY = 11 };

template <int D>
struct Cfg {
    static constexpr int NA = (D + 63) / 64;        // 64-element atoms along d
    static constexpr int TB = NA * kAtom;           // one 128-row tile of Q, K or V
    static constexpr int OFF_Q = 0;                 // queries: qhat for pass OLD, then q
    static constexpr int OFF_K = TB;                // K ring: 2 stages
    static constexpr int OFF_V = 3 * TB;            // V ring: 2 stages
    static constexpr int OFF_P = 5 * TB;            // P: 2 buffers of 128 x 128 bf16
    static constexpr int OFF_ONES = OFF_P + 4 * kAtom;
    static constexpr int OFF_BAR = OFF_ONES + 512;
    static constexpr int OFF_MISC = OFF_BAR + N_BARS * 8;
    static constexpr int BYTES = OFF_MISC + 16;
    static constexpr int SMEM = BYTES + 1024;       // room to align the base to 1024 bytes
    static_assert(SMEM <= 232448, "shared memory budget");
};

struct KParams {
    int mode, H, n_keys, n_state, R, K, n_row_tiles;
    const int32_t *row_pos;
    const int32_t *key_idx;
    const uint16_t *q;
    uint16_t *q_hat;
    float *o, *z, *c;
    float sl2;   // log2(e) / sqrt(d)
};

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Bounded wait. The thread sleeps inside try_wait (hinted) rather than
// spinning; it gives up after about one second, or as soon as another role
// has given up, recording the first failure code.
__device__ __noinline__ bool wait_bar_slow(uint32_t bar, uint32_t parity, volatile int *abort_flag, int code) {
    if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 > 1000000000ull) {
            *abort_flag = 1;
            atomicCAS(&g_tc_error, 0, code);
            return false;
        }
    }
}

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int *abort_flag, int code) {
    if (mbar_test_wait(bar, parity)) return true;
    return wait_bar_slow(bar, parity, abort_flag, code);
}

// Number of entries of the ascending list S[0, n) that are <= x.
__device__ __forceinline__ int count_le(const int32_t *S, int n, int x) {
    int lo = 0, hi = n;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(S + mid) <= x) lo = mid + 1; else hi = mid;
    }
    return lo;
}

// Byte offset of 16-byte chunk `ch` (8 bf16) of row r in a 128-row tile laid
// out as 64-element atoms with the 128-byte swizzle.
__device__ __forceinline__ uint32_t swz_off(int r, int ch) {
    return (uint32_t)((ch >> 3) * kAtom + (r >> 3) * 1024 + (r & 7) * 128 + (((ch & 7) ^ (r & 7)) << 4));
}

// Gathers row r's query (qhat or q) into the swizzled query tile; the two
// softmax halves each write every other 16-byte chunk.
template <int D>
__device__ __forceinline__ void load_query_row(uint8_t *tile, const uint16_t *src_row, bool row_ok, int r, int wg) {
    const uint4 zero = make_uint4(0, 0, 0, 0);
    const uint4 *src = reinterpret_cast<const uint4 *>(src_row);
#pragma unroll
    for (int ch = wg; ch < D / 8; ch += 2)
        *reinterpret_cast<uint4 *>(tile + swz_off(r, ch)) = row_ok ? src[ch] : zero;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
tc_attention_kernel(const __grid_constant__ KParams p, const __grid_constant__ CUtensorMap tm_k_old,
                    const __grid_constant__ CUtensorMap tm_v_old, const __grid_constant__ CUtensorMap tm_k_new,
                    const __grid_constant__ CUtensorMap tm_v_new) {
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + C::OFF_BAR;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    uint32_t *misc = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(misc + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.z, h = blockIdx.y;
    const int rt = p.n_row_tiles - 1 - (int)blockIdx.x;   // heavier (later) row tiles first
    const bool dense = p.mode != FLASHLOOP_ATTN_LAZY;
    const bool first = p.mode == FLASHLOOP_ATTN_FIRST_DENSE;
    const int row0 = rt * BM;
    const int rows = min(BM, p.R - row0);
    const long long bh = (long long)b * p.H + h;
    const int32_t *S = dense ? nullptr : p.key_idx + bh * p.K;
    const int32_t *A = dense ? nullptr : p.row_pos + (long long)b * p.R + row0;
    const int min_pos = dense ? row0 : __ldg(A);
    const int max_pos = dense ? row0 + rows - 1 : __ldg(A + rows - 1);
    // Rows and keys are both ascending, so the keys a row may see are a
    // prefix of the list: row i sees the first count_le(S, i) of them.
    const int cnt = dense ? min(max_pos + 1, p.n_keys) : count_le(S, p.K, max_pos);      // last row
    const int cnt_min = dense ? min(min_pos + 1, p.n_keys) : count_le(S, p.K, min_pos);  // first row
    const int n_tiles = (cnt + BN - 1) / BN;
    if (n_tiles == 0) return;   // every row has an empty key set: state unchanged
    const int ph0 = first ? PH_LSE : PH_OLD;
    const int total = (3 - ph0) * n_tiles;
    const int kcols = dense ? p.n_keys : p.K;
    auto col_index = [&](int cc) { return cc < kcols ? (dense ? cc : __ldg(S + cc)) : INT_MAX; };

    // ---------------- set-up ----------------
    if (threadIdx.x == 0) {
        for (int i = 0; i < N_BARS; ++i) {
            uint32_t count = 1;
            if (i == BAR_S_EMPTY || i == BAR_S_EMPTY + 1 || i == BAR_P_FULL || i == BAR_P_FULL + 1 ||
                i == BAR_STATS || i == BAR_Q_READY)
                count = kSoftmax;
            mbar_init(bar(i), count);
        }
        misc[1] = 0;
        mbar_fence_init();
    }
    __syncwarp();
    if (warp == 0) {
        tmem_alloc(sbase + C::OFF_MISC, kTmemCols);
        tmem_relinquish();
    }
    if (warp == 1) {   // 16x16 bf16 ones (B operand of the column-sum MMA)
        uint4 one4 = make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
        reinterpret_cast<uint4 *>(smem + C::OFF_ONES)[lane] = one4;
        fence_proxy_async_smem();
    }
    const bool is_sm = warp >= 2;
    const int wg = is_sm ? (warp - 2) >> 2 : 0;   // column half of the softmax warps
    const int r = (warp & 3) * 32 + lane;          // tile row == TMEM lane
    const bool row_ok = is_sm && r < rows;
    const int pos = row_ok ? (dense ? row0 + r : __ldg(A + r)) : -1;
    const long long qoff = (((long long)b * p.n_state + max(pos, 0)) * p.H + h) * D;
    if (is_sm) {   // pass OLD reads qhat; the first dense loop starts with q
        load_query_row<D>(smem + C::OFF_Q, first ? p.q + qoff : p.q_hat + qoff, row_ok, r, wg);
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];

    if (warp == 0) {
        // ---------------- TMA producer: K ring and V ring ----------------
        if (lane == 0) {
            prefetch_tmap(&tm_k_old); prefetch_tmap(&tm_v_old);
            prefetch_tmap(&tm_k_new); prefetch_tmap(&tm_v_new);
            int k_issued = 0, v_issued = 0;
            int ph = ph0, t = 0;
            for (int g = 0; g < total; ++g, ++t) {
                if (t == n_tiles) { t = 0; ++ph; }
                const int key0 = t * BN;
                {
                    const int s = g & 1, use = g >> 1;
                    if (!wait_bar(bar(BAR_K_EMPTY + s), (use & 1) ^ 1, abort_flag, ERR_K_EMPTY)) break;
                    const CUtensorMap *mk = ph == PH_OLD ? &tm_k_old : &tm_k_new;
                    const uint32_t dst = sbase + C::OFF_K + C::TB * s;
                    mbar_arrive_expect_tx(bar(BAR_K_FULL + s), C::TB);
                    for (int a = 0; a < C::NA; ++a) {
                        if (dense) tma_load_4d(dst + a * kAtom, mk, bar(BAR_K_FULL + s), a * 64, h, key0, b);
                        else tma_load_4d(dst + a * kAtom, mk, bar(BAR_K_FULL + s), a * 64, key0, h, b);
                    }
                    k_issued = g + 1;
                }
                if (ph != PH_LSE) {
                    const int vi = v_issued, s = vi & 1, use = vi >> 1;
                    if (!wait_bar(bar(BAR_V_EMPTY + s), (use & 1) ^ 1, abort_flag, ERR_V_EMPTY)) break;
                    const CUtensorMap *mv = ph == PH_OLD ? &tm_v_old : &tm_v_new;
                    const uint32_t dst = sbase + C::OFF_V + C::TB * s;
                    mbar_arrive_expect_tx(bar(BAR_V_FULL + s), C::TB);
                    for (int a = 0; a < C::NA; ++a) {
                        if (dense) tma_load_4d(dst + a * kAtom, mv, bar(BAR_V_FULL + s), a * 64, h, key0, b);
                        else tma_load_4d(dst + a * kAtom, mv, bar(BAR_V_FULL + s), a * 64, key0, h, b);
                    }
                    v_issued = vi + 1;
                }
            }
            if (*abort_flag) {   // let copies already in flight land before the CTA exits
                volatile int never = 0;
                for (int g = max(0, k_issued - 2); g < k_issued; ++g)
                    wait_bar(bar(BAR_K_FULL + (g & 1)), (g >> 1) & 1, &never, ERR_K_FULL);
                for (int v = max(0, v_issued - 2); v < v_issued; ++v)
                    wait_bar(bar(BAR_V_FULL + (v & 1)), (v >> 1) & 1, &never, ERR_V_FULL);
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            constexpr uint32_t id_qk = idesc_bf16(128, 128, false, false, false);
            constexpr uint32_t id_pv_old = idesc_bf16(128, D, false, true, true);
            constexpr uint32_t id_pv_new = idesc_bf16(128, D, false, true, false);
            constexpr uint32_t id_cs_old = idesc_bf16(128, 16, true, false, true);
            constexpr uint32_t id_cs_new = idesc_bf16(128, 16, true, false, false);
            // descriptors are built once; per k-step only the start address moves
            const uint64_t d_q = smem_desc(sbase + C::OFF_Q, 16, 1024, 2);
            const uint64_t d_k = smem_desc(sbase + C::OFF_K, 16, 1024, 2);
            const uint64_t d_v = smem_desc(sbase + C::OFF_V, kAtom, 1024, 2);
            const uint64_t d_p = smem_desc(sbase + C::OFF_P, 16, 1024, 2);
            const uint64_t d_pt = smem_desc(sbase + C::OFF_P, kAtom, 1024, 2);
            const uint64_t ones = smem_desc(sbase + C::OFF_ONES, 128, 256, 0);
            constexpr uint64_t TB16 = C::TB >> 4, ATOM16 = kAtom >> 4;
            int ph_next = ph0, t_next = 0;   // phase of tile g + 1 while issuing it
            auto issue_qk = [&](int g) -> bool {
                const int s = g & 1, use = g >> 1;
                const int ph = ph_next;
                if (++t_next == n_tiles) { t_next = 0; ++ph_next; }
                if (!wait_bar(bar(BAR_K_FULL + s), use & 1, abort_flag, ERR_K_FULL)) return false;
                if (!wait_bar(bar(BAR_S_EMPTY + s), (use & 1) ^ 1, abort_flag, ERR_S_EMPTY)) return false;
                if (ph == PH_LSE && g == (PH_LSE - ph0) * n_tiles && !first) {   // queries reloaded after pass OLD
                    if (!wait_bar(bar(BAR_Q_READY), 0, abort_flag, ERR_Q_READY)) return false;
                }
                tc_fence_after();
                const uint64_t dk = d_k + TB16 * s;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t off = (kk >> 2) * ATOM16 + (kk & 3) * 2;
                    mma_bf16_ss(tmem + kColS + 128 * s, d_q + off, dk + off, id_qk, kk > 0);
                }
                mma_commit(bar(BAR_S_FULL + s));
                mma_commit(bar(BAR_K_EMPTY + s));
                return true;
            };
            bool ok = issue_qk(0);
            int pv = 0, ph = ph0, t = 0;
            for (int g = 0; ok && g < total; ++g, ++t) {
                if (t == n_tiles) { t = 0; ++ph; }
                if (g + 1 < total && !issue_qk(g + 1)) { ok = false; break; }
                if (ph == PH_LSE) continue;
                const int s = pv & 1, use = pv >> 1;   // V ring slot and P buffer share the with-V count
                if (!wait_bar(bar(BAR_V_FULL + s), use & 1, abort_flag, ERR_V_FULL)) { ok = false; break; }
                if (!wait_bar(bar(BAR_P_FULL + s), use & 1, abort_flag, ERR_P_FULL)) { ok = false; break; }
                tc_fence_after();
                const bool neg = ph == PH_OLD;
                const uint64_t dp = d_p + 2 * ATOM16 * s, dpt = d_pt + 2 * ATOM16 * s, dv = d_v + TB16 * s;
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk)   // acc += P[:, 16kk..] * V[16kk.., :]
                    mma_bf16_ss(tmem + kColAcc, dp + (kk >> 2) * ATOM16 + (kk & 3) * 2, dv + kk * 128,
                                neg ? id_pv_old : id_pv_new, (pv > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
                for (int kk = 0; kk < BM / 16; ++kk)   // colsum = P^T[:, 16kk..] * ones
                    mma_bf16_ss(tmem + kColCS + 16 * s, dpt + kk * 128, ones, neg ? id_cs_old : id_cs_new, kk > 0);
                mma_commit(bar(BAR_P_EMPTY + s));
                mma_commit(bar(BAR_V_EMPTY + s));
                ++pv;
            }
            if (ok) {
                mma_commit(bar(BAR_ACC));
            } else {   // drain whatever was issued before giving up
                mma_commit(bar(BAR_DRAIN));
                volatile int never = 0;
                wait_bar(bar(BAR_DRAIN), 0, &never, ERR_ACC);
            }
        }
    } else {
        // ---------------- softmax / epilogue: two warpgroups, one column half each ----------------
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const int half = wg * 64;
        const float zo2 = (!first && row_ok) ? __ldg(p.z + bh * p.n_state + pos) * kLog2e : 0.f;
        const int cnt_i = !row_ok ? 0 : dense ? min(pos + 1, p.n_keys) : count_le(S, p.K, pos);
        float m = 0.f, M = -INFINITY, L = 0.f, zn2 = INFINITY;
        int pv = 0;
        int col_hist[2] = {INT_MAX, INT_MAX};   // this lane's column of the last two P tiles
        bool ok = true;
        float *cb = p.c + bh * p.n_keys;
        uint32_t pk[32];   // this row's P over the half's 64 columns, bf16x2
        // column sums of P tile `idx` (done once its PV/colsum MMAs completed)
        auto flush_colsum = [&](int idx) {
            const float cs = tmem_ld_32x32b_x1(tmem + lane_base + kColCS + 16 * (idx & 1));
            tmem_wait_ld();
            const int col = col_hist[idx & 1];
            if (col != INT_MAX && cs != 0.f) atomicAdd(cb + col, cs);
        };
        int ph = ph0, t = 0;
        for (int g = 0; g < total && ok; ++g, ++t) {
            if (t == n_tiles) { t = 0; ++ph; }
            const int s = g & 1, use = g >> 1;
            if (ph == PH_LSE && t == 0 && !first) {
                // pass OLD's products are all done (their S tiles were consumed):
                // reload the query tile with this loop's q
                load_query_row<D>(smem + C::OFF_Q, p.q + qoff, row_ok, r, wg);
                fence_proxy_async_smem();
                mbar_arrive(bar(BAR_Q_READY));
            }
            if (ph == PH_NEW && t == 0) {
                // merge the two halves' row statistics through TMEM (same lane, own columns)
                tmem_st_32x32b_x4(tmem + lane_base + kColX + 4 * wg, m, M, L, 0.f);
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(bar(BAR_STATS));
                if (!wait_bar(bar(BAR_STATS), 0, abort_flag, ERR_STATS)) { ok = false; break; }
                tc_fence_after();
                float o4[4];
                tmem_ld_32x32b_x4(tmem + lane_base + kColX + 4 * (1 - wg), o4);
                tmem_wait_ld();
                const float Mx = fmaxf(M, o4[1]);
                const float Lx = (Mx > -INFINITY) ? L * ex2(M - Mx) + o4[2] * ex2(o4[1] - Mx) : 0.f;
                const float mx = first ? 1.f : m + o4[0];
                zn2 = (Mx > -INFINITY && mx >= FLT_MIN) ? Mx + __log2f(Lx) - __log2f(mx) : INFINITY;
            }
            const int c0 = t * BN;
            const bool with_v = ph != PH_LSE;
            // this lane's column of the column-sum MMA (only the first half reads sums back)
            const int jr = (with_v && wg == 0) ? col_index(c0 + r) : INT_MAX;
            // every row of the tile sees all 128 columns (uniform), else mask by the prefix count
            const bool full = c0 + BN <= cnt_min;
            const int nv = min(64, max(0, cnt_i - c0 - half));
            if (!wait_bar(bar(BAR_S_FULL + s), use & 1, abort_flag, ERR_S_FULL)) { ok = false; break; }
            tc_fence_after();
            float sv[64];
            const uint32_t sc = tmem + lane_base + kColS + 128 * s + half;
            tmem_ld_32x32b_x32(sc, sv);
            tmem_ld_32x32b_x32(sc + 32, sv + 32);
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(bar(BAR_S_EMPTY + s));
            if (!with_v) {
                // online logsumexp of this tile's new logits (log2 units)
                if (full) {
#pragma unroll
                    for (int e = 0; e < 64; ++e) sv[e] *= p.sl2;
                } else {
#pragma unroll
                    for (int e = 0; e < 64; ++e) sv[e] = e < nv ? sv[e] * p.sl2 : -INFINITY;
                }
                float c4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int e = 0; e < 64; ++e) c4[e & 3] = fmaxf(c4[e & 3], sv[e]);
                const float cmax = fmaxf(fmaxf(c4[0], c4[1]), fmaxf(c4[2], c4[3]));
                if (cmax > M) {
                    L *= ex2(M - cmax);
                    M = cmax;
                }
                float a4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int e = 0; e < 64; ++e) a4[e & 3] += ex2(sv[e] - M);
                if (M > -INFINITY) L += (a4[0] + a4[1]) + (a4[2] + a4[3]);
                continue;
            }
            // probabilities with a known normaliser: exp(logit - Z) (rows outside the
            // tile or the sequence get zero through an infinite normaliser)
            const float sub = !row_ok ? INFINITY : ph == PH_OLD ? zo2 : zn2;
            float m4[4] = {0.f, 0.f, 0.f, 0.f};
            if (full) {
#pragma unroll
                for (int e = 0; e < 64; e += 2) {
                    const float x0 = ex2(fmaf(sv[e], p.sl2, -sub));
                    const float x1 = ex2(fmaf(sv[e + 1], p.sl2, -sub));
                    m4[(e >> 1) & 3] += x0 + x1;
                    pk[e / 2] = pack_bf16x2_rn(x0, x1);
                }
            } else {
#pragma unroll
                for (int e = 0; e < 64; e += 2) {
                    const float x0 = e < nv ? ex2(fmaf(sv[e], p.sl2, -sub)) : 0.f;
                    const float x1 = e + 1 < nv ? ex2(fmaf(sv[e + 1], p.sl2, -sub)) : 0.f;
                    m4[(e >> 1) & 3] += x0 + x1;
                    pk[e / 2] = pack_bf16x2_rn(x0, x1);
                }
            }
            if (ph == PH_OLD) m += (m4[0] + m4[1]) + (m4[2] + m4[3]);
            // P buffer pb was last read by the MMAs of P tile pv - 2
            const int pb = pv & 1, puse = pv >> 1;
            if (!wait_bar(bar(BAR_P_EMPTY + pb), (puse & 1) ^ 1, abort_flag, ERR_P_EMPTY)) { ok = false; break; }
            tc_fence_after();
            if (wg == 0 && pv >= 2) flush_colsum(pv - 2);
            uint8_t *pt = smem + C::OFF_P + 2 * kAtom * pb;
#pragma unroll
            for (int q = 0; q < 8; ++q)
                *reinterpret_cast<uint4 *>(pt + swz_off(r, wg * 8 + q)) =
                    make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(bar(BAR_P_FULL + pb));
            col_hist[pb] = jr;
            ++pv;
        }
        if (ok && wg == 0) {   // column sums of the last (up to) two P tiles
            for (int idx = max(0, pv - 2); idx < pv && ok; ++idx) {
                if (!wait_bar(bar(BAR_P_EMPTY + (idx & 1)), (idx >> 1) & 1, abort_flag, ERR_P_EMPTY)) { ok = false; break; }
                tc_fence_after();
                flush_colsum(idx);
            }
        }
        if (ok && wait_bar(bar(BAR_ACC), 0, abort_flag, ERR_ACC)) {
            tc_fence_after();
            const bool update = row_ok && zn2 < INFINITY;
            const long long srow = ((long long)b * p.n_state + max(pos, 0)) * p.H + h;
            float4 *orow = reinterpret_cast<float4 *>(p.o + srow * D);
            constexpr int HALF_D = D / 2;   // accumulator columns per warpgroup
#pragma unroll
            for (int u = 0; u < HALF_D / 16; ++u) {
                float av[16];
                const int col = wg * HALF_D + 16 * u;
                tmem_ld_32x32b_x16(tmem + lane_base + kColAcc + col, av);
                tmem_wait_ld();
                if (update) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        float4 v = first ? make_float4(0.f, 0.f, 0.f, 0.f) : orow[col / 4 + e];
                        v.x += av[4 * e];
                        v.y += av[4 * e + 1];
                        v.z += av[4 * e + 2];
                        v.w += av[4 * e + 3];
                        orow[col / 4 + e] = v;
                    }
                }
            }
            if (update && wg == 0) {
                p.z[bh * p.n_state + pos] = zn2 * kLn2;
                const uint4 *src = reinterpret_cast<const uint4 *>(p.q + srow * D);
                uint4 *dst = reinterpret_cast<uint4 *>(p.q_hat + srow * D);
#pragma unroll
                for (int ch = 0; ch < D / 8; ++ch) dst[ch] = ldg_nc_v4(src + ch);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------------------
// host side

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
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

// 4-D bf16 tensor map with a (64, box1, box2, 1) box and the 128-byte swizzle.
bool make_map(CUtensorMap *map, const void *base, const cuuint64_t dims[4], const cuuint64_t strides_bytes[3],
              cuuint32_t box1, cuuint32_t box2) {
    auto enc = get_encode();
    if (!enc) return false;
    const cuuint32_t box[4] = {64, box1, box2, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(base), dims, strides_bytes, box,
                     estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int D>
cudaError_t launch_d(const TcAttnParams &p, cudaStream_t s) {
    using Cf = Cfg<D>;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaFuncSetAttribute(tc_attention_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cf::SMEM);
    });
    const bool dense = p.mode != FLASHLOOP_ATTN_LAZY;
    CUtensorMap maps[4];
    const uint16_t *src[4] = {p.k_old ? p.k_old : p.k_new, p.v_old ? p.v_old : p.v_new, p.k_new, p.v_new};
    for (int i = 0; i < 4; ++i) {
        bool ok;
        if (dense) {   // cache layer [B, N_cap, H, d]; only the first n_keys positions are read
            const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)p.H, (cuuint64_t)p.n_keys, (cuuint64_t)p.B};
            const cuuint64_t str[3] = {(cuuint64_t)D * 2, (cuuint64_t)p.H * D * 2,
                                       (cuuint64_t)p.kv_rows * p.H * D * 2};
            ok = make_map(&maps[i], src[i], dims, str, 1, BN);
        } else {       // dense selected keys [B, H, K, d]
            const cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)p.K, (cuuint64_t)p.H, (cuuint64_t)p.B};
            const cuuint64_t str[3] = {(cuuint64_t)D * 2, (cuuint64_t)p.K * D * 2, (cuuint64_t)p.H * p.K * D * 2};
            ok = make_map(&maps[i], src[i], dims, str, BN, 1);
        }
        if (!ok) return cudaErrorInvalidValue;
    }
    KParams kp;
    kp.mode = p.mode;
    kp.H = p.H;
    kp.n_keys = p.n_keys;
    kp.n_state = p.n_state;
    kp.R = p.R;
    kp.K = dense ? p.n_keys : p.K;
    kp.n_row_tiles = ceil_div(p.R, BM);
    kp.row_pos = p.row_pos;
    kp.key_idx = p.key_idx;
    kp.q = p.q;
    kp.q_hat = p.q_hat;
    kp.o = p.o;
    kp.z = p.z;
    kp.c = p.c;
    kp.sl2 = kLog2e / sqrtf((float)D);
    dim3 grid(kp.n_row_tiles, p.H, p.B);
    {
        KernelTimer kt("tc_attention", s);
        tc_attention_kernel<D><<<grid, kThreads, Cf::SMEM, s>>>(kp, maps[0], maps[1], maps[2], maps[3]);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_tc_attention(const TcAttnParams &p, cudaStream_t s) {
    if (p.R == 0) return cudaSuccess;
    switch (p.d) {
        case 64: return launch_d<64>(p, s);
        case 96: return launch_d<96>(p, s);
        case 128: return launch_d<128>(p, s);
        default: return cudaErrorInvalidValue;
    }
}

int32_t tc_attention_read_error(bool clear) {
    int v = 0;
    cudaMemcpyFromSymbol(&v, g_tc_error, sizeof(int));
    if (clear && v) {
        int zero = 0;
        cudaMemcpyToSymbol(g_tc_error, &zero, sizeof(int));
    }
    return v;
}

}  // namespace fl

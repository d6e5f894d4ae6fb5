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
//   pass OLD: QK_old -> -p -> m, acc += (-P) V_old, column sums of -P
//   pass LSE: QK_new -> online max/sum -> lam
//   pass NEW: QK_new -> P' = exp(. - Z') -> acc += P' V_new, column sums of P'
// The first dense loop skips pass OLD (m = 1, u = 0).
//
// Roles (576 threads): warp 0 issues TMA loads into a K ring (3 stages) and
// a V ring (2 stages); warp 1 (one thread) issues tcgen05.mma; warps 2..17
// are four softmax groups of four warps. A warp owns 32 TMEM lanes (= rows)
// and its group owns 32 of the tile's 128 columns. A tile's logits land in
// one of three 128-column TMEM buffers; the softmax writes the bf16
// probabilities back over the first half of the columns it has read, and the
// PV product takes them straight from TMEM (A operand in tensor memory), so P
// never touches shared memory. The probabilities are handed over before the
// column masses are formed: those are summed after the hand-off by integer
// warp reductions of a fixed-point encoding and added to c with one atomic
// per column and warp. A buffer is reused once the softmax has read it and,
// for tiles with a PV product, once that product completed. The query tile
// holds qhat for pass OLD and is reloaded with q before pass LSE; the four
// groups merge row statistics once, through shared memory.
// TMEM columns: S/P buffers [0,384), accumulator [384,384+d).
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
constexpr int BN_ = BN;
constexpr int kThreads = 576;     // warp 0 TMA, warp 1 MMA, warps 2..17 softmax (4 groups x 4 warps)
constexpr int kGroups = 4;        // softmax warpgroups, each owns 32 of a tile's 128 columns
constexpr int kGroupCols = BN_ / kGroups;
constexpr int kSoftmaxWarps = 4 * kGroups;   // softmax-side barriers take one elected arrival per warp
constexpr int kAtom = 128 * 128;  // bytes of a 128-row x 64-element bf16 tile, 128-byte swizzled
constexpr uint32_t kTmemCols = 512;
constexpr int kSBufs = 3;         // S/P buffers in TMEM, 128 columns each
constexpr uint32_t kColAcc = 384; // accumulator columns [384, 384 + d)
constexpr int kKStages = 3, kVStages = 2;
static_assert(kKStages == kSBufs, "a tile's K slot and S/P buffer share one index");
static_assert(kVStages == 2, "the MMA issuer indexes the V ring with a parity bit");
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
// Column sums are taken on integers: x*2^20 rounded into the mantissa of
// x*2^20 + 1.5*2^23 (exact while |x| < 4), so a warp reduction is exact and
// the sum of 32 lanes' offsets is removed afterwards.
constexpr float kFixScale = 1048576.0f, kFixMagic = 12582912.0f;
constexpr uint32_t kFixBits = 0x4B400000u;

__device__ int g_tc_error;

enum : int { PH_OLD = 0, PH_LSE = 1, PH_NEW = 2 };
enum : int { BAR_K_FULL = 0, BAR_K_EMPTY = 3, BAR_V_FULL = 6, BAR_V_EMPTY = 8, BAR_S_FULL = 10, BAR_S_READ = 13,
             BAR_P_FULL = 16, BAR_PV_DONE = 19, BAR_ACC = 22, BAR_STATS = 23, BAR_Q_READY = 24, BAR_DRAIN = 25,
             N_BARS = 26 };
enum : int { ERR_K_EMPTY = 1, ERR_K_FULL = 2, ERR_V_EMPTY = 3, ERR_V_FULL = 4, ERR_S_READ = 5, ERR_S_FULL = 6,
             ERR_P_FULL = 7, ERR_PV_DONE = 8, ERR_ACC = 9, ERR_STATS = 10, ERR_Q_READY = 11 };

template <int D>
struct Cfg {
    static constexpr int NA = (D + 63) / 64;        // 64-element atoms along d
    static constexpr int TB = NA * kAtom;           // one 128-row tile of Q, K or V
    static constexpr int OFF_Q = 0;                 // queries: qhat for pass OLD, then q
    static constexpr int OFF_K = TB;                // K ring
    static constexpr int OFF_V = OFF_K + kKStages * TB;   // V ring
    static constexpr int OFF_X = OFF_V + kVStages * TB;   // row-statistics exchange: [groups][128][3] fp32
    static constexpr int OFF_BAR = OFF_X + kGroups * 128 * 3 * 4;
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

// Gathers row r's query (qhat or q) into the swizzled query tile; each
// softmax group writes every kGroups-th 16-byte chunk.
template <int D>
__device__ __forceinline__ void load_query_row(uint8_t *tile, const uint16_t *src_row, bool row_ok, int r, int wg) {
    const uint4 zero = make_uint4(0, 0, 0, 0);
    const uint4 *src = reinterpret_cast<const uint4 *>(src_row);
#pragma unroll
    for (int ch = wg; ch < D / 8; ch += kGroups)
        *reinterpret_cast<uint4 *>(tile + swz_off(r, ch)) = row_ok ? src[ch] : zero;
}

// One arrival per warp: every lane's earlier shared-memory and tensor-memory
// work is ordered before lane 0 arrives.
__device__ __forceinline__ void warp_arrive(uint32_t bar, int lane) {
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(bar);
}

// TMEM column of the P values for keys [16 kk, 16 kk + 16) of an S/P buffer:
// each softmax group writes bf16 pairs over the first 16 of the 32 S columns
// it read itself (keys 32 g .. 32 g + 31 -> columns 32 g .. 32 g + 15).
__device__ __forceinline__ uint32_t p_col(int kk) { return 32u * (kk >> 1) + 8u * (kk & 1); }

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
    // Work grows with a row tile's last position (later rows see more keys), so the
    // linear CTA order runs every head's heaviest row tiles first and leaves the
    // lightest ones for the last, partial wave.
    const int b = blockIdx.z, h = (int)(blockIdx.x % p.H);
    const int rt = p.n_row_tiles - 1 - (int)(blockIdx.x / p.H);
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
            const bool many = (i >= BAR_S_READ && i < BAR_S_READ + kSBufs) || (i >= BAR_P_FULL && i < BAR_P_FULL + kSBufs) ||
                              i == BAR_STATS || i == BAR_Q_READY;
            mbar_init(bar(i), many ? (uint32_t)kSoftmaxWarps : 1u);
        }
        misc[1] = 0;
        mbar_fence_init();
    }
    __syncwarp();
    if (warp == 0) {
        tmem_alloc(sbase + C::OFF_MISC, kTmemCols);
        tmem_relinquish();
    }
    const bool is_sm = warp >= 2;
    const int wg = is_sm ? (warp - 2) >> 2 : 0;   // softmax group: columns [32 wg, 32 wg + 32) of a tile
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
        // ---------------- TMA producer: K ring (3 stages) and V ring (2 stages) ----------------
        if (lane == 0) {
            prefetch_tmap(&tm_k_old); prefetch_tmap(&tm_v_old);
            prefetch_tmap(&tm_k_new); prefetch_tmap(&tm_v_new);
            int k_issued = 0, v_issued = 0;
            int ph = ph0, t = 0;
            for (int g = 0; g < total; ++g, ++t) {
                if (t == n_tiles) { t = 0; ++ph; }
                const int key0 = t * BN;
                {
                    const int s = g % kKStages, use = g / kKStages;
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
                    const int vi = v_issued, s = vi % kVStages, use = vi / kVStages;
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
                for (int g = max(0, k_issued - kKStages); g < k_issued; ++g)
                    wait_bar(bar(BAR_K_FULL + g % kKStages), (g / kKStages) & 1, &never, ERR_K_FULL);
                for (int v = max(0, v_issued - kVStages); v < v_issued; ++v)
                    wait_bar(bar(BAR_V_FULL + v % kVStages), (v / kVStages) & 1, &never, ERR_V_FULL);
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            constexpr uint32_t id_qk = idesc_bf16(128, 128, false, false, false);
            constexpr uint32_t id_pv = idesc_bf16(128, D, false, true, false);   // A = P from TMEM
            // descriptors are built once; per k-step only the start address moves
            const uint64_t d_q = smem_desc(sbase + C::OFF_Q, 16, 1024, 2);
            const uint64_t d_k = smem_desc(sbase + C::OFF_K, 16, 1024, 2);
            const uint64_t d_v = smem_desc(sbase + C::OFF_V, kAtom, 1024, 2);
            constexpr uint64_t TB16 = C::TB >> 4, ATOM16 = kAtom >> 4;
            // Bookkeeping stays in registers: the tensor core buffers only about two
            // MMAs, so any scalar latency between MMA groups is idle tensor time.
            // Per S/P buffer (= K slot) b, bit b of: used (ever written), upar (parity
            // of its uses so far), hadv (its last tile had a PV product), pfpar (parity
            // of P-ready waits), pdpar (parity of PV-done commits).
            uint32_t used = 0, upar = 0, hadv = 0, pfpar = 0, pdpar = 0;
            int qb = 0;                      // S/P buffer and K slot of the next QK
            int ph_next = ph0, t_next = 0;   // phase and tile of the next QK
            auto issue_qk = [&](int g) -> bool {
                const int ph = ph_next;
                if (++t_next == n_tiles) { t_next = 0; ++ph_next; }
                const uint32_t bit = 1u << qb, par = (upar >> qb) & 1u;
                if (!wait_bar(bar(BAR_K_FULL + qb), par, abort_flag, ERR_K_FULL)) return false;
                if (used & bit) {   // the buffer's last S was read, and its last P consumed by PV
                    if (!wait_bar(bar(BAR_S_READ + qb), par ^ 1u, abort_flag, ERR_S_READ)) return false;
                    if ((hadv & bit) && !wait_bar(bar(BAR_PV_DONE + qb), ((pdpar >> qb) & 1u) ^ 1u, abort_flag, ERR_PV_DONE))
                        return false;
                }
                if (ph == PH_LSE && g == n_tiles && !first) {   // queries reloaded after pass OLD
                    if (!wait_bar(bar(BAR_Q_READY), 0, abort_flag, ERR_Q_READY)) return false;
                }
                tc_fence_after();
                const uint64_t dk = d_k + TB16 * (uint32_t)qb;
                const uint32_t dst = tmem + 128u * (uint32_t)qb;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t off = (kk >> 2) * ATOM16 + (kk & 3) * 2;
                    mma_bf16_ss(dst, d_q + off, dk + off, id_qk, kk > 0);
                }
                mma_commit(bar(BAR_S_FULL + qb));
                mma_commit(bar(BAR_K_EMPTY + qb));
                used |= bit;
                upar ^= bit;
                hadv = ph != PH_LSE ? (hadv | bit) : (hadv & ~bit);
                qb = qb == kSBufs - 1 ? 0 : qb + 1;
                return true;
            };
            bool ok = issue_qk(0);
            int pv = 0, ph = ph0, t = 0, pb = 0;   // pb: S/P buffer of tile g
            for (int g = 0; ok && g < total; ++g, ++t, pb = pb == kSBufs - 1 ? 0 : pb + 1) {
                if (t == n_tiles) { t = 0; ++ph; }
                if (g + 1 < total && !issue_qk(g + 1)) { ok = false; break; }
                if (ph == PH_LSE) continue;
                const int vs = pv & 1;
                const uint32_t bit = 1u << pb;
                if (!wait_bar(bar(BAR_V_FULL + vs), (pv >> 1) & 1, abort_flag, ERR_V_FULL)) { ok = false; break; }
                if (!wait_bar(bar(BAR_P_FULL + pb), (pfpar >> pb) & 1u, abort_flag, ERR_P_FULL)) { ok = false; break; }
                pfpar ^= bit;
                tc_fence_after();
                const uint64_t dv = d_v + TB16 * (uint32_t)vs;
                const uint32_t pa = tmem + 128u * (uint32_t)pb;
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk)   // acc += P[:, 16kk..] * V[16kk.., :]  (P is signed)
                    mma_bf16_ts(tmem + kColAcc, pa + p_col(kk), dv + kk * 128, id_pv, (pv > 0 || kk > 0) ? 1u : 0u);
                mma_commit(bar(BAR_PV_DONE + pb));
                pdpar ^= bit;
                mma_commit(bar(BAR_V_EMPTY + vs));
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
        // ---------------- softmax / epilogue: four groups, 32 columns each ----------------
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        const int cbase = wg * kGroupCols;
        const float zo2 = (!first && row_ok) ? __ldg(p.z + bh * p.n_state + pos) * kLog2e : 0.f;
        // every row of the tile sees the same keys when the first and last rows do
        const int cnt_i = !row_ok ? 0 : cnt_min == cnt ? cnt : dense ? min(pos + 1, p.n_keys) : count_le(S, p.K, pos);
        float m = 0.f, M = -INFINITY, L = 0.f, zn2 = INFINITY;
        bool ok = true;
        float *cb = p.c + bh * p.n_keys;
        int ph = ph0, t = 0;
        for (int g = 0; g < total && ok; ++g, ++t) {
            if (t == n_tiles) { t = 0; ++ph; }
            const int sb = g % kSBufs, suse = g / kSBufs;
            if (ph == PH_LSE && t == 0 && !first) {
                // pass OLD's products are all done (their S tiles were consumed):
                // reload the query tile with this loop's q
                load_query_row<D>(smem + C::OFF_Q, p.q + qoff, row_ok, r, wg);
                fence_proxy_async_smem();
                warp_arrive(bar(BAR_Q_READY), lane);
            }
            if (ph == PH_NEW && t == 0) {
                // merge the groups' row statistics
                float *ex = reinterpret_cast<float *>(smem + C::OFF_X);
                ex[(wg * 128 + r) * 3 + 0] = m;
                ex[(wg * 128 + r) * 3 + 1] = M;
                ex[(wg * 128 + r) * 3 + 2] = L;
                warp_arrive(bar(BAR_STATS), lane);
                if (!wait_bar(bar(BAR_STATS), 0, abort_flag, ERR_STATS)) { ok = false; break; }
                float mx = 0.f, Mx = -INFINITY, Lx = 0.f;
#pragma unroll
                for (int k = 0; k < kGroups; ++k) {
                    mx += ex[(k * 128 + r) * 3 + 0];
                    Mx = fmaxf(Mx, ex[(k * 128 + r) * 3 + 1]);
                }
                if (Mx > -INFINITY) {
#pragma unroll
                    for (int k = 0; k < kGroups; ++k)
                        Lx += ex[(k * 128 + r) * 3 + 2] * ex2(ex[(k * 128 + r) * 3 + 1] - Mx);
                }
                if (first) mx = 1.f;
                zn2 = (Mx > -INFINITY && mx >= FLT_MIN) ? Mx + __log2f(Lx) - __log2f(mx) : INFINITY;
            }
            const int c0 = t * BN;
            const bool with_v = ph != PH_LSE;
            // key position of this lane's column (for the column-mass atomics)
            const int jcol = with_v ? col_index(c0 + cbase + lane) : INT_MAX;
            // every row of the tile sees all 128 columns (uniform), else mask by the prefix count
            const bool full = c0 + BN <= cnt_min;
            const int nv = min(kGroupCols, max(0, cnt_i - c0 - cbase));
            if (!wait_bar(bar(BAR_S_FULL + sb), suse & 1, abort_flag, ERR_S_FULL)) { ok = false; break; }
            tc_fence_after();
            float sv[kGroupCols];
            tmem_ld_32x32b_x32(tmem + lane_base + 128u * sb + cbase, sv);
            tmem_wait_ld();
            warp_arrive(bar(BAR_S_READ + sb), lane);
            if (!with_v) {
                // online logsumexp of this tile's new logits (log2 units)
                if (full) {
#pragma unroll
                    for (int e = 0; e < kGroupCols; ++e) sv[e] *= p.sl2;
                } else {
#pragma unroll
                    for (int e = 0; e < kGroupCols; ++e) sv[e] = e < nv ? sv[e] * p.sl2 : -INFINITY;
                }
                float c4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int e = 0; e < kGroupCols; ++e) c4[e & 3] = fmaxf(c4[e & 3], sv[e]);
                const float cmax = fmaxf(fmaxf(c4[0], c4[1]), fmaxf(c4[2], c4[3]));
                if (cmax > M) {
                    L *= ex2(M - cmax);
                    M = cmax;
                }
                float a4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int e = 0; e < kGroupCols; ++e) a4[e & 3] += ex2(sv[e] - M);
                if (M > -INFINITY) L += (a4[0] + a4[1]) + (a4[2] + a4[3]);
                continue;
            }
            // probabilities with a known normaliser, signed by pass (OLD subtracts):
            // sign * exp(logit - Z); rows outside the tile or the sequence get zero
            // through an infinite normaliser
            const float sub = !row_ok ? INFINITY : ph == PH_OLD ? zo2 : zn2;
            const float sgn = ph == PH_OLD ? -1.f : 1.f;
            if (full) {
#pragma unroll
                for (int e = 0; e < kGroupCols; ++e) sv[e] = sgn * ex2(fmaf(sv[e], p.sl2, -sub));
            } else {
#pragma unroll
                for (int e = 0; e < kGroupCols; ++e) sv[e] = e < nv ? sgn * ex2(fmaf(sv[e], p.sl2, -sub)) : 0.f;
            }
            uint32_t pk[kGroupCols / 2];
#pragma unroll
            for (int e = 0; e < kGroupCols; e += 2) pk[e / 2] = pack_bf16x2_rn(sv[e], sv[e + 1]);
            // this tile's P, bf16, over the first half of the S columns this group just read;
            // handing it over is the PV product's critical path, the sums below are not
            tmem_st_32x32b_x16(tmem + lane_base + 128u * sb + cbase, pk);
            tmem_wait_st();
            warp_arrive(bar(BAR_P_FULL + sb), lane);
            if (ph == PH_OLD) {
                float m4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int e = 0; e < kGroupCols; ++e) m4[e & 3] += sv[e];
                m -= (m4[0] + m4[1]) + (m4[2] + m4[3]);
            }
            // column masses over the warp's 32 rows, exact on fixed-point integers
            uint32_t csum = 0u;
#pragma unroll
            for (int e = 0; e < kGroupCols; ++e) {
                const uint32_t tot = __reduce_add_sync(0xffffffffu, __float_as_uint(fmaf(sv[e], kFixScale, kFixMagic)));
                if (e == lane) csum = tot;
            }
            const int fixed = (int)(csum - 32u * kFixBits);
            if (jcol != INT_MAX && fixed != 0) atomicAdd(cb + jcol, (float)fixed * (1.0f / kFixScale));
        }
        if (ok && wait_bar(bar(BAR_ACC), 0, abort_flag, ERR_ACC)) {
            tc_fence_after();
            constexpr int GD = D / kGroups;   // accumulator columns per group (16, 24 or 32)
            float av[GD];
#pragma unroll
            for (int u = 0; u < GD / 8; ++u) tmem_ld_32x32b_x8(tmem + lane_base + kColAcc + wg * GD + 8 * u, av + 8 * u);
            tmem_wait_ld();
            const bool update = row_ok && zn2 < INFINITY;
            if (update) {
                const long long srow = ((long long)b * p.n_state + pos) * p.H + h;
                float4 *orow = reinterpret_cast<float4 *>(p.o + srow * D) + wg * (GD / 4);
                float4 ov[GD / 4];
#pragma unroll
                for (int e = 0; e < GD / 4; ++e) ov[e] = first ? make_float4(0.f, 0.f, 0.f, 0.f) : orow[e];
#pragma unroll
                for (int e = 0; e < GD / 4; ++e) {
                    ov[e].x += av[4 * e];
                    ov[e].y += av[4 * e + 1];
                    ov[e].z += av[4 * e + 2];
                    ov[e].w += av[4 * e + 3];
                    orow[e] = ov[e];
                }
                if (wg == 0) p.z[bh * p.n_state + pos] = zn2 * kLn2;
                // the query tile holds this loop's q: copy this group's chunks of it to qhat
                uint4 *dst = reinterpret_cast<uint4 *>(p.q_hat + srow * D);
#pragma unroll
                for (int ch = wg; ch < D / 8; ch += kGroups)
                    dst[ch] = *reinterpret_cast<const uint4 *>(smem + C::OFF_Q + swz_off(r, ch));
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
    dim3 grid(kp.n_row_tiles * p.H, 1, p.B);
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

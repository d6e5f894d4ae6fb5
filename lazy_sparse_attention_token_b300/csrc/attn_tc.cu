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
// Roles (608 threads): warp 0 issues TMA loads into one ring of five K/V
// tile slots, in the order the products consume them (a pass with PV products
// loads K(0), then K(t+1) before V(t); pass LSE loads keys only and so keeps
// five key tiles in flight); warp 1 issues the QK
// products and warp 2 the PV products: the tensor pipe buffers only about two
// MMAs, and a second issuer covers the barrier tests the first makes between
// its batches. Each issuing warp runs its loop with all 32 lanes and one
// elected lane issues (the arithmetic stays warp-uniform instead of taking
// issue slots from the softmax warps on the same scheduler). The QK issuer
// runs up to two tiles ahead of the softmax. Warps 3..18 are four softmax groups of
// four warps, a group owning 32 of a tile's 128 columns and a warp owning one
// 32-lane quadrant (32 rows) of TMEM.
// A softmax thread holds 4 rows x 8 columns of its group's block (two
// 16x256b TMEM loads), so row statistics stay per-thread partials that are
// merged once per pass, and a column mass is an in-thread sum over four rows
// plus a three-step butterfly over lanes. The bf16 probabilities go back to
// TMEM (two 16x128b stores) in the packed key order the PV product reads as
// its A operand, so P never touches shared memory; pass OLD's subtraction is
// the instruction descriptor's negate-A bit. Column masses are formed after
// P has been handed over and added to c with one atomic per column and warp.
// The query tile holds qhat for pass OLD and is reloaded with q (asynchronous
// copies issued under the last OLD tile's softmax) before pass LSE. TMEM columns: S buffers [0,256), P buffers [256,384), accumulator
// [384,384+d).
//
// CTAs run the (row tile, head) items heaviest first, one per SM. A lazy
// loop's items are of nearly equal size (the keys it selects sit early, so
// most row tiles see all of them), so the items past the last full wave
// would keep a few SMs busy for a whole item while the rest idle. Those run
// in a launch of their own, each split by key tiles over a cluster of up to
// four CTAs: every part runs the three passes over its own tiles, the parts'
// per-row (old mass, maximum, sum) are combined through distributed shared
// memory before pass NEW (each CTA in the same rank order, so all hold the
// same Z'), and rank 0 adds the parts' accumulators, in rank order, to O.
// That launch goes first; the main grid follows without waiting for it and
// fills the SMs it leaves free (it waits for it only before its CTAs exit).
//
// A wait tests the phase, then makes one try_wait inline (the thread is
// suspended until the phase completes or a hardware limit passes) before the
// out-of-line loop of hinted try_waits: the call would otherwise sit on the
// critical path of every hand-off. Every
// mbarrier wait is bounded (one second unless the host shortens it); on
// timeout the CTA records an error code, stops issuing work, waits (bounded,
// one second) for its own copies and MMAs, frees TMEM and exits. A softmax
// warp proceeds past a wait only when all of its lanes saw the phase. The CTAs
// of a split item meet at one cluster barrier after set-up and one before
// exit, which every CTA reaches because every wait before it is bounded.
#include <cudaTypedefs.h>
#include <float.h>
#include <mutex>
#include <type_traits>

#include "common.cuh"
#include "tc_ptx.cuh"

namespace fl {
namespace {

using namespace ptx;

constexpr int BM = 128;
constexpr int BN = 128;
constexpr int BN_ = BN;
constexpr int kThreads = 608;     // warp 0 TMA, warp 1 QK MMAs, warp 2 PV MMAs, warps 3..18 softmax (4 x 4)
constexpr int kFirstSoftmaxWarp = 3;
constexpr int kSetupBar = 1;      // named barrier of the set-up (0 is __syncthreads)
constexpr int kGroups = 4;        // softmax groups, each owns 32 of a tile's 128 columns
constexpr int kGroupCols = BN_ / kGroups;
constexpr int kSoftmaxWarps = 4 * kGroups;   // softmax-side barriers take one elected arrival per warp
constexpr int kAtom = 128 * 128;  // bytes of a 128-row x 64-element bf16 tile, 128-byte swizzled
constexpr uint32_t kTmemCols = 512;
constexpr int kSBufs = 2;         // logits S: two buffers of 128 fp32 columns, [0, 256)
constexpr uint32_t kColP = 256;   // probabilities P: two buffers of 64 columns (128 bf16), [256, 384)
constexpr uint32_t kColAcc = 384; // accumulator columns [384, 384 + d)
constexpr int kStages = 5;        // K/V tile slots of the load ring
constexpr int kMaxParts = 4;      // CTAs that may share one row tile (a cluster)
static_assert(kSBufs == 2, "S and P buffers are indexed with a parity bit");
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ int g_tc_error;
// Limit of every bounded wait on the compute path, in ns (the host may only
// shorten it, to exercise the failure path). Drains after a failure keep
// kDrainLimitNs, so that a CTA that gave up still lets its own copies and MMAs
// land before it frees TMEM and exits.
constexpr unsigned long long kWaitLimitNs = FLASHLOOP_WAIT_LIMIT_DEFAULT_NS;
constexpr unsigned long long kDrainLimitNs = FLASHLOOP_WAIT_LIMIT_DEFAULT_NS;
__device__ unsigned long long g_tc_wait_limit_ns = kWaitLimitNs;

enum : int { PH_OLD = 0, PH_LSE = 1, PH_NEW = 2 };
// PV_DONE[b] completes when the PV product that read P buffer b is done (the
// softmax may then overwrite it); the product also releases its V tile's slot.
// EMPTY[s]: ring slot s is free again (waited by the producer only).
// FULL[p % (2 kStages)]: the tile of ring position p has landed. The ring's
// tiles are consumed by two issuing threads, neither of which waits on every
// position, and a parity wait cannot tell a phase two behind from a completed
// one. With 2 kStages landed barriers the phase before position p's belongs to
// position p - 2 kStages, which is always consumed by then: a thread's
// consecutive waits are at most kStages positions apart, so the producer has
// issued p - kStages, which it does only once p - 2 kStages is consumed.
constexpr int kFullBars = 2 * kStages;
enum : int { BAR_FULL = 0, BAR_EMPTY = kFullBars, BAR_S_FULL = BAR_EMPTY + kStages, BAR_S_READ = BAR_S_FULL + 2,
             BAR_P_FULL = BAR_S_READ + 2, BAR_PV_DONE = BAR_P_FULL + 2, BAR_ACC = BAR_PV_DONE + 2,
             BAR_STATS = BAR_ACC + 1, BAR_Q_READY = BAR_STATS + 1, BAR_DRAIN = BAR_Q_READY + 1, BAR_ZN = BAR_DRAIN + 2,
             BAR_EPI = BAR_ZN + 1, BAR_XSTAT = BAR_EPI + 1, BAR_XACC = BAR_XSTAT + 1, N_BARS = BAR_XACC + 1 };
// landed barrier and its parity for ring position p
__device__ __forceinline__ int full_bar_of(int p) { return BAR_FULL + p % kFullBars; }
__device__ __forceinline__ uint32_t full_parity(int p) { return (uint32_t)(p / kFullBars) & 1u; }
enum : int { ERR_EMPTY = 1, ERR_FULL = 2, ERR_S_READ = 5, ERR_S_FULL = 6, ERR_P_FULL = 7, ERR_PV_DONE = 8,
             ERR_ACC = 9, ERR_STATS = 10, ERR_Q_READY = 11, ERR_ZN = 12, ERR_EPI = 13, ERR_XSTAT = 14, ERR_XACC = 15 };

// Ring position of a pass's loads. A pass with PV products loads K(0), then
// K(t+1) before V(t) for every t, and V(n-1) last (2n loads); pass LSE loads
// K(t) in order (n loads).
__device__ __forceinline__ int kv_pos_k(int t) { return t == 0 ? 0 : 2 * t - 1; }
__device__ __forceinline__ int kv_pos_v(int t, int n) { return t + 1 < n ? 2 * t + 2 : 2 * t + 1; }

template <int D>
struct Cfg {
    static constexpr int NA = (D + 63) / 64;        // 64-element atoms along d
    static constexpr int TB = NA * kAtom;           // one 128-row tile of Q, K or V
    static constexpr int OFF_Q = 0;                 // queries: qhat for pass OLD, then q
    static constexpr int OFF_KV = TB;               // K/V ring
    static constexpr int OFF_X = OFF_KV + kStages * TB;   // row-statistics exchange: [groups][128][3] fp32
    static constexpr int OFF_ROW = OFF_X + kGroups * 128 * 3 * 4;   // per row: key count, old and new normaliser
    static constexpr int OFF_XCL = OFF_ROW + 128 * 16;   // split items: [part][128] of (m, M, L, 0), written by every rank
    static constexpr int OFF_BAR = OFF_XCL + kMaxParts * 128 * 16;
    // epilogue: the finished accumulator rows, parked in the (then idle) ring
    static constexpr int XS = D + 4;   // padded row stride in floats
    static_assert(128 * XS * 4 <= kStages * TB, "accumulator rows fit the ring");
    static constexpr int OFF_MISC = OFF_BAR + N_BARS * 8;
    static constexpr int BYTES = OFF_MISC + 16;
    static constexpr int SMEM = BYTES + 1024;       // room to align the base to 1024 bytes
    static_assert(SMEM <= 232448, "shared memory budget");
};

struct KParams {
    int mode, H, n_keys, n_state, R, K, n_row_tiles;
    const int32_t *row_pos;
    const int32_t *row_cnt;   // lazy: keys each row sees, [B,H,R]
    const int32_t *key_idx;
    const uint16_t *q;
    uint16_t *q_hat;
    float *o, *z, *c;
    float sl2;   // log2(e) / sqrt(d)
    const int32_t *seq_exit;   // [B] or NULL: a sequence flagged 1 has stopped looping
    // Work item of CTA x: item_base + x / nparts in the heavy-first order (below).
    // nparts > 1: a cluster of nparts CTAs shares one item, CTA rank p taking key
    // tiles [p n / nparts, (p + 1) n / nparts) of its n.
    int item_base, nparts;
    // 1: this grid follows the split launch of the same loop, which it does not
    // depend on: it waits for that grid only before its CTAs exit (see below)
    int late_wait;
};

__device__ __forceinline__ float max3f(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// Packed two-lane fp32 arithmetic (one instruction for both lanes, each lane
// rounded exactly as its scalar counterpart): a * b + c and a + b.
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Bounded wait. The thread sleeps inside try_wait (hinted, at most the limit)
// rather than spinning; it gives up once `limit_ns` has passed, or as soon as
// another role has given up, recording the first failure code.
__device__ __noinline__ bool wait_bar_slow(uint32_t bar, uint32_t parity, volatile int *abort_flag, int code,
                                           unsigned long long limit_ns) {
    if (limit_ns == 0) {   // a zero limit: no waiting at all (the caller has tested the phase once)
        *abort_flag = 1;
        atomicCAS(&g_tc_error, 0, code);
        return false;
    }
    const uint64_t t0 = globaltimer_ns();
    const uint32_t hint = limit_ns < 20000ull ? (uint32_t)limit_ns : 20000u;
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 8; ++i)
            if (mbar_try_wait_sleep(bar, parity, hint)) return true;
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 >= limit_ns) {
            *abort_flag = 1;
            atomicCAS(&g_tc_error, 0, code);
            return false;
        }
    }
}

// `limit_ns` is the kernel's copy of g_tc_wait_limit_ns, read once per thread
// at the start of the kernel.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int *abort_flag, int code,
                                         unsigned long long limit_ns) {
    if (mbar_test_wait(bar, parity)) return true;
    // one try_wait inline (it suspends for up to a hardware-chosen time, and most
    // waits end within it), the bounded loop out of line
    if (limit_ns != 0 && mbar_try_wait(bar, parity)) return true;
    return wait_bar_slow(bar, parity, abort_flag, code, limit_ns);
}

// The same wait for a whole warp that goes on to warp-collective instructions
// (tcgen05.ld/st .sync.aligned, shuffles): every lane waits, and the warp
// proceeds only if all of them saw the phase complete, so that a lane that
// gave up never leaves the others alone in a collective.
__device__ __forceinline__ bool wait_bar_all(uint32_t bar, uint32_t parity, volatile int *abort_flag, int code,
                                             unsigned long long limit_ns) {
    return __all_sync(0xffffffffu, wait_bar(bar, parity, abort_flag, code, limit_ns));
}

// Wait of a drain after a failure: not cut short by the abort flag, and held to
// kDrainLimitNs whatever the compute-path limit is.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity, int code) {
    volatile int never = 0;
    if (!mbar_test_wait(bar, parity)) wait_bar_slow(bar, parity, &never, code, kDrainLimitNs);
}

// ---- a row tile split over a cluster (distributed shared memory) ----
// address of the same shared-memory location in cluster CTA `rank`
__device__ __forceinline__ uint32_t cl_map(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
__device__ __forceinline__ void cl_arrive() { asm volatile("barrier.cluster.arrive.release;" ::: "memory"); }
__device__ __forceinline__ void cl_wait() { asm volatile("barrier.cluster.wait.acquire;" ::: "memory"); }
__device__ __forceinline__ void cl_st4(uint32_t addr, float4 v) {
    asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(v.x), "f"(v.y), "f"(v.z),
                 "f"(v.w)
                 : "memory");
}
__device__ __forceinline__ float4 cl_ld4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}
// arrival on an mbarrier of another CTA of the cluster, releasing this thread's
// (and, cumulatively, what it has observed of its CTA's) shared-memory writes
__device__ __forceinline__ void cl_mbar_arrive(uint32_t remote_bar) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote_bar) : "memory");
}
// Bounded wait for a phase completed by arrivals from the cluster; acquires
// at cluster scope, so that the arriving CTAs' writes are visible after it.
__device__ __noinline__ bool wait_bar_cluster(uint32_t bar, uint32_t parity, volatile int *abort_flag, int code,
                                              unsigned long long limit_ns) {
    if (limit_ns == 0) {   // a zero limit: the phase is tested once, without waiting
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(bar), "r"(parity)
            : "memory");
        if (done) return true;
        *abort_flag = 1;
        atomicCAS(&g_tc_error, 0, code);
        return false;
    }
    const uint64_t t0 = globaltimer_ns();
    const uint32_t hint = limit_ns < 20000ull ? (uint32_t)limit_ns : 20000u;
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 8; ++i) {
            uint32_t done;
            asm volatile(
                "{\n\t.reg .pred p;\n\t"
                "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2, %3;\n\t"
                "selp.u32 %0, 1, 0, p;\n\t}"
                : "=r"(done)
                : "r"(bar), "r"(parity), "r"(hint)
                : "memory");
            if (done) return true;
        }
        if (*abort_flag) return false;
        if (globaltimer_ns() - t0 >= limit_ns) {
            *abort_flag = 1;
            atomicCAS(&g_tc_error, 0, code);
            return false;
        }
    }
}

// ---- MMA issue from a whole (converged) warp: one elected lane issues ----
// The issuing warps run their loops with all 32 lanes (so that the loop and
// descriptor arithmetic is warp-uniform) and predicate each tcgen05 instruction
// on one elected lane, always the same one (the lowest), which therefore also
// commits: a commit tracks the MMAs of the thread that executes it.
#define FL_EL "elect.sync _|e, 0xffffffff;\n\t"
#define FL_MMA_SS_E(ai, bi, n, pr) "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %" #ai ", %" #bi ", %" #n ", " #pr ";\n\t"
__device__ __forceinline__ void mma_ss_x8_el(uint32_t d_tmem, const uint64_t (&a)[8], const uint64_t (&b)[8],
                                             uint32_t idesc, uint32_t acc0) {
    asm volatile(
        "{\n\t.reg .pred p, q, e;\n\t" FL_EL
        "setp.ne.b32 p, %18, 0;\n\t"
        "setp.eq.b32 q, %17, %17;\n\t"
        FL_MMA_SS_E(1, 9, 17, p) FL_MMA_SS_E(2, 10, 17, q) FL_MMA_SS_E(3, 11, 17, q) FL_MMA_SS_E(4, 12, 17, q)
        FL_MMA_SS_E(5, 13, 17, q) FL_MMA_SS_E(6, 14, 17, q) FL_MMA_SS_E(7, 15, 17, q) FL_MMA_SS_E(8, 16, 17, q) "}"
        ::"r"(d_tmem), "l"(a[0]), "l"(a[1]), "l"(a[2]), "l"(a[3]), "l"(a[4]), "l"(a[5]), "l"(a[6]), "l"(a[7]),
        "l"(b[0]), "l"(b[1]), "l"(b[2]), "l"(b[3]), "l"(b[4]), "l"(b[5]), "l"(b[6]), "l"(b[7]), "r"(idesc), "r"(acc0)
        : "memory");
}
__device__ __forceinline__ void mma_ss_x4_el(uint32_t d_tmem, const uint64_t *a, const uint64_t *b, uint32_t idesc,
                                             uint32_t acc0) {
    asm volatile(
        "{\n\t.reg .pred p, q, e;\n\t" FL_EL
        "setp.ne.b32 p, %10, 0;\n\t"
        "setp.eq.b32 q, %9, %9;\n\t"
        FL_MMA_SS_E(1, 5, 9, p) FL_MMA_SS_E(2, 6, 9, q) FL_MMA_SS_E(3, 7, 9, q) FL_MMA_SS_E(4, 8, 9, q) "}"
        ::"r"(d_tmem), "l"(a[0]), "l"(a[1]), "l"(a[2]), "l"(a[3]), "l"(b[0]), "l"(b[1]), "l"(b[2]), "l"(b[3]),
        "r"(idesc), "r"(acc0)
        : "memory");
}
__device__ __forceinline__ void mma_ss_x2_el(uint32_t d_tmem, const uint64_t *a, const uint64_t *b, uint32_t idesc,
                                             uint32_t acc0) {
    asm volatile(
        "{\n\t.reg .pred p, q, e;\n\t" FL_EL
        "setp.ne.b32 p, %6, 0;\n\t"
        "setp.eq.b32 q, %5, %5;\n\t"
        FL_MMA_SS_E(1, 3, 5, p) FL_MMA_SS_E(2, 4, 5, q) "}"
        ::"r"(d_tmem), "l"(a[0]), "l"(a[1]), "l"(b[0]), "l"(b[1]), "r"(idesc), "r"(acc0)
        : "memory");
}
#define FL_MMA_TS_E(ai, bi, pr) "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%" #ai "], %" #bi ", %17, " #pr ";\n\t"
__device__ __forceinline__ void mma_ts_x8_el(uint32_t d_tmem, const uint32_t (&a)[8], const uint64_t (&b)[8],
                                             uint32_t idesc, uint32_t acc0) {
    asm volatile(
        "{\n\t.reg .pred p, q, e;\n\t" FL_EL
        "setp.ne.b32 p, %18, 0;\n\t"
        "setp.eq.b32 q, %17, %17;\n\t"
        FL_MMA_TS_E(1, 9, p) FL_MMA_TS_E(2, 10, q) FL_MMA_TS_E(3, 11, q) FL_MMA_TS_E(4, 12, q)
        FL_MMA_TS_E(5, 13, q) FL_MMA_TS_E(6, 14, q) FL_MMA_TS_E(7, 15, q) FL_MMA_TS_E(8, 16, q) "}"
        ::"r"(d_tmem), "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(a[4]), "r"(a[5]), "r"(a[6]), "r"(a[7]),
        "l"(b[0]), "l"(b[1]), "l"(b[2]), "l"(b[3]), "l"(b[4]), "l"(b[5]), "l"(b[6]), "l"(b[7]), "r"(idesc), "r"(acc0)
        : "memory");
}
__device__ __forceinline__ void mma_commit_el(uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t" FL_EL
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
        : "memory");
}
#undef FL_MMA_TS_E
#undef FL_MMA_SS_E
#undef FL_EL

// Byte offset of 16-byte chunk `ch` (8 bf16) of row r in a 128-row tile laid
// out as 64-element atoms with the 128-byte swizzle.
__device__ __forceinline__ uint32_t swz_off(int r, int ch) {
    return (uint32_t)((ch >> 3) * kAtom + (r >> 3) * 1024 + (r & 7) * 128 + (((ch & 7) ^ (r & 7)) << 4));
}

// Gathers the tile's query rows (qhat or q, [B, n_state, H, D] bf16) into the
// swizzled query tile. The softmax threads (index st) take consecutive 16-byte
// chunks, so a warp reads whole rows; rows past the tile's end are zero.
// Thread st takes chunks st + 512 i (i < D / 32): chunk st % (D / 8) of rows
// st / (D / 8) + (512 / (D / 8)) i. Their positions are loaded first thing in
// the kernel (query_positions), as the head of the set-up's longest chain of
// dependent loads.
template <int D>
struct QueryRows {
    static constexpr int CPR = D / 8;                      // 16-byte chunks per row
    static constexpr int N = BM * CPR / (32 * kSoftmaxWarps);
    static_assert(N * 32 * kSoftmaxWarps == BM * CPR, "the gather covers the tile exactly");
    int pos[N];                                            // -1: row outside the tile
};
template <int D>
__device__ __forceinline__ void query_positions(QueryRows<D> &qr, int st, int rows, int row0, const int32_t *A) {
#pragma unroll
    for (int i = 0; i < QueryRows<D>::N; ++i) {
        const int rr = (st + 32 * kSoftmaxWarps * i) / QueryRows<D>::CPR;
        qr.pos[i] = rr >= rows ? -1 : A ? __ldg(A + rr) : row0 + rr;
    }
}
// The same gather as 16-byte asynchronous copies (no registers held; rows
// outside the tile are zero-filled): completed by cp.async.wait_all.
template <int D>
__device__ __forceinline__ void load_query_tile_async(uint8_t *tile, const uint16_t *src, int st, int b, int h,
                                                      int H, int n_state, const QueryRows<D> &qr) {
    constexpr int CPR = QueryRows<D>::CPR;
    const uint4 *s4 = reinterpret_cast<const uint4 *>(src);
#pragma unroll
    for (int i = 0; i < QueryRows<D>::N; ++i) {
        const int c = st + 32 * kSoftmaxWarps * i;
        const int rr = c / CPR, ch = c - rr * CPR;
        const bool in = qr.pos[i] >= 0;
        const uint4 *g = in ? s4 + (((long long)b * n_state + qr.pos[i]) * H + h) * CPR + ch : s4;
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(tile + swz_off(rr, ch))), "l"(g),
                     "r"(in ? 16 : 0)
                     : "memory");
    }
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

template <int D>
__device__ __forceinline__ void load_query_tile(uint8_t *tile, const uint16_t *src, int st, int b, int h, int H,
                                                int n_state, const QueryRows<D> &qr) {
    constexpr int CPR = QueryRows<D>::CPR;
    const uint4 *s4 = reinterpret_cast<const uint4 *>(src);
    const uint64_t stream = l2_policy_evict_first();   // each query row is read by one row tile
#pragma unroll
    for (int i = 0; i < QueryRows<D>::N; ++i) {
        const int c = st + 32 * kSoftmaxWarps * i;
        const int rr = c / CPR, ch = c - rr * CPR;
        uint4 val = make_uint4(0, 0, 0, 0);
        if (qr.pos[i] >= 0)
            val = ld_global_v4_hint(s4 + (((long long)b * n_state + qr.pos[i]) * H + h) * CPR + ch, stream);
        *reinterpret_cast<uint4 *>(tile + swz_off(rr, ch)) = val;
    }
}

// One arrival per warp: every lane's earlier shared-memory and tensor-memory
// work is ordered before lane 0 arrives.
__device__ __forceinline__ void warp_arrive(uint32_t bar, int lane) {
    (void)lane;
    tc_fence_before();
    __syncwarp();
    mbar_arrive_elected(bar);
}

// Softmax fragment layout. Each softmax thread holds, per tile, rows
// rq + lane/4 + 8k (k = 0..3) of its warp's 32-lane quadrant rq and columns
// cbase + 8j + 2(lane%4) + e (j = 0..3, e = 0..1) of its group's 32 columns:
// two 16x256b loads. Index of (k, j, e) among the 32 registers:
__device__ __forceinline__ constexpr int frag(int k, int j, int e) { return 16 * (k >> 1) + 4 * j + 2 * (k & 1) + e; }

// Column sums of a fragment over the warp's 32 rows: in-thread over the four
// rows, then a transposing butterfly over the eight lanes with the same lane%4.
// Lane l ends with the sum of column 8(J/2) + 2(l%4) + J%2, J = l/4.
__device__ __forceinline__ float column_sum(const float *v, int lane) {
    float cs[8];
    auto pr = [&](int k, int j) { return make_float2(v[frag(k, j, 0)], v[frag(k, j, 1)]); };
#pragma unroll
    for (int j = 0; j < 4; ++j) {   // the two columns of a pair together
        const float2 t = add2(add2(pr(0, j), pr(1, j)), add2(pr(2, j), pr(3, j)));
        cs[2 * j] = t.x;
        cs[2 * j + 1] = t.y;
    }
#pragma unroll
    for (int w = 4; w >= 1; w >>= 1) {
        const bool up = lane & (w << 2);
#pragma unroll
        for (int e = 0; e < w; ++e) {
            const float send = up ? cs[e] : cs[e + w];
            const float keep = up ? cs[e + w] : cs[e];
            cs[e] = keep + __shfl_xor_sync(0xffffffffu, send, w << 2);
        }
    }
    return cs[0];
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
tc_attention_kernel(const __grid_constant__ KParams p, const __grid_constant__ CUtensorMap tm_k_old,
                    const __grid_constant__ CUtensorMap tm_v_old, const __grid_constant__ CUtensorMap tm_k_new,
                    const __grid_constant__ CUtensorMap tm_v_new) {
    // Every global read below depends on the kernels before this launch. A grid
    // that follows the split launch starts without waiting: that launch issued
    // its dependent launch only after all of its CTAs had waited for those
    // kernels, so their writes are visible here; and waiting for it before
    // exiting keeps the next kernel's dependency on this grid covering both.
    if (!p.late_wait) pdl_wait();
    pdl_trigger();
    const unsigned long long wlimit = g_tc_wait_limit_ns;
    if (p.seq_exit && __ldg(p.seq_exit + blockIdx.z)) {   // the whole CTA: its sequence stopped looping
        if (p.late_wait) pdl_wait();
        return;
    }
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + C::OFF_BAR;
    auto bar = [&](int i) { return bar0 + 8u * (uint32_t)i; };
    uint32_t *misc = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(misc + 1);
    int *row_cnt = reinterpret_cast<int *>(smem + C::OFF_ROW);
    float *row_zo = reinterpret_cast<float *>(smem + C::OFF_ROW + 128 * 4);
    float *row_zn = reinterpret_cast<float *>(smem + C::OFF_ROW + 128 * 8);
    int *row_pos_s = reinterpret_cast<int *>(smem + C::OFF_ROW + 128 * 12);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Work grows with a row tile's last position (later rows see more keys), so the
    // linear CTA order runs every head's heaviest row tiles first and leaves the
    // lightest ones for the last, partial wave.
    // with a cluster of nparts CTAs along x, the CTA's rank in it is x % nparts
    const bool split = p.nparts > 1;
    const int part = (int)blockIdx.x % p.nparts;
    const int item = p.item_base + (int)blockIdx.x / p.nparts;
    const int b = blockIdx.z, h = item % p.H;
    const int rt = p.n_row_tiles - 1 - item / p.H;
    const bool dense = p.mode != FLASHLOOP_ATTN_LAZY;
    const bool first = p.mode == FLASHLOOP_ATTN_FIRST_DENSE;
    const int row0 = rt * BM;
    const int rows = min(BM, p.R - row0);
    const long long bh = (long long)b * p.H + h;
    const int32_t *S = dense ? nullptr : p.key_idx + bh * p.K;
    const int32_t *A = dense ? nullptr : p.row_pos + (long long)b * p.R + row0;
    // Rows and keys are both ascending, so the keys a row may see are a
    // prefix of the list: row i sees the keys of S that are <= i, counted for
    // every lazy row before the launch.
    const int32_t *RC = dense ? nullptr : p.row_cnt + bh * p.R + row0;
    // row positions first: the query gather and the per-row loads of the set-up depend on them
    const bool is_sm = warp >= kFirstSoftmaxWarp;
    const int st = (int)threadIdx.x - 32 * kFirstSoftmaxWarp;   // softmax thread index
    const int r = (warp & 3) * 32 + lane;          // the row this thread loads and writes back
    const bool row_ok = is_sm && r < rows;
    const int pos = row_ok ? (dense ? row0 + r : __ldg(A + r)) : -1;
    QueryRows<D> qrows;
    if (is_sm) query_positions<D>(qrows, st, rows, row0, A);
    // softmax group: columns [32 wg, 32 wg + 32) of a tile; its four warps cover the four lane quadrants
    const int wg = is_sm ? (warp - kFirstSoftmaxWarp) >> 2 : 0;
    // the row's key count and old normaliser (group 0 keeps them in shared memory), issued with the gather
    const bool row_vals = row_ok && wg == 0;
    const int rc_r = row_vals && !dense ? __ldg(RC + r) : 0;
    const float z_r = row_vals && !(p.mode == FLASHLOOP_ATTN_FIRST_DENSE) ? __ldg(p.z + bh * p.n_state + pos) : 0.f;
    const int cnt = dense ? min(row0 + rows, p.n_keys) : __ldg(RC + rows - 1);   // last row
    const int cnt_min = dense ? min(row0 + 1, p.n_keys) : __ldg(RC);             // first row
    const int n_all = (cnt + BN - 1) / BN;
    if (n_all == 0) {   // every row has an empty key set: state unchanged (the whole cluster)
        if (p.late_wait) pdl_wait();
        return;
    }
    // this CTA's key tiles [t0, t0 + n_tiles); a part may get none
    const int t0 = part * n_all / p.nparts;
    const int t_end = (part + 1) * n_all / p.nparts;
    const int n_tiles = t_end - t0;
    const int ph0 = first ? PH_LSE : PH_OLD;
    const int total = (3 - ph0) * n_tiles;
    const int kcols = dense ? p.n_keys : p.K;
    auto col_index = [&](int cc) { return cc < kcols ? (dense ? cc : __ldg(S + cc)) : INT_MAX; };

    // ---------------- set-up ----------------
    if (threadIdx.x == 0) {
        for (int i = 0; i < N_BARS; ++i) {
            const bool many = (i >= BAR_S_READ && i < BAR_S_READ + kSBufs) || (i >= BAR_P_FULL && i < BAR_P_FULL + 2) ||
                              i == BAR_STATS || i == BAR_Q_READY || i == BAR_ZN || i == BAR_EPI;
            const uint32_t cnt_i = i == BAR_XSTAT ? 4u * (uint32_t)p.nparts   // the four group-0 warps of every part
                                   : i == BAR_XACC ? (uint32_t)p.nparts                  // one arrival per part
                                   : many ? (uint32_t)kSoftmaxWarps : 1u;
            mbar_init(bar(i), cnt_i);
        }
        misc[1] = 0;
        mbar_fence_init();
    }
    __syncwarp();
    // a split item: no CTA touches another's shared memory before every CTA of the
    // cluster has initialised its barriers (the cluster's CTAs start together)
    if (split) {
        cl_arrive();
        cl_wait();
    }
    if (warp == 0) {
        tmem_alloc(sbase + C::OFF_MISC, kTmemCols);
        tmem_relinquish();
    }
    // The producer needs only the barriers, so it arrives on the set-up barrier
    // without waiting and starts the K/V copies while the other warps wait for
    // the query tile and the per-row values.
    if (warp == 0) {
        tc_fence_before();
        named_bar_arrive(kSetupBar, kThreads);
    } else {
        if (is_sm) {   // pass OLD reads qhat; the first dense loop starts with q
            load_query_tile<D>(smem + C::OFF_Q, first ? p.q : p.q_hat, st, b, h, p.H, p.n_state, qrows);
            fence_proxy_async_smem();
            // the query tile is reloaded with q after pass OLD: fetch those rows into L2 now
            if (!first && row_ok && wg * 64 < D) {
                const uint16_t *qrow = p.q + (((long long)b * p.n_state + pos) * p.H + h) * D + wg * 64;
                asm volatile("prefetch.global.L2 [%0];" ::"l"(qrow));
            }
            if (wg == 0) {   // per row, shared by the four groups: key count and old normaliser (log2 units)
                row_cnt[r] = !row_ok ? 0 : cnt_min == cnt ? cnt : dense ? min(pos + 1, p.n_keys) : rc_r;
                row_zo[r] = !row_ok ? INFINITY : first ? 0.f : z_r * kLog2e;
                row_pos_s[r] = pos;
            }
        }
        tc_fence_before();
        named_bar_sync(kSetupBar, kThreads);
        tc_fence_after();
    }
    const uint32_t tmem = misc[0];   // read by warp 0 only after the closing barrier

    if (warp == 0) {
        // ---------------- TMA producer: one ring of K/V tile slots ----------------
        if (lane == 0) {
            prefetch_tmap(&tm_k_old); prefetch_tmap(&tm_v_old);
            prefetch_tmap(&tm_k_new); prefetch_tmap(&tm_v_new);
            int pos = 0;   // loads issued
            // the K/V tiles are read once per pass by every row tile of the head: keep them in
            // L2 ahead of the streamed query, output and normaliser traffic
            const uint64_t keep = l2_policy_evict_last();
            // K or V tile t of pass ph into the next slot, once its previous tile is consumed
            auto load = [&](bool is_v, int ph, int t) -> bool {
                const int s = pos % kStages, use = pos / kStages;
                if (!wait_bar(bar(BAR_EMPTY + s), (use & 1) ^ 1, abort_flag, ERR_EMPTY, wlimit)) return false;
                const CUtensorMap *m = is_v ? (ph == PH_OLD ? &tm_v_old : &tm_v_new) : (ph == PH_OLD ? &tm_k_old : &tm_k_new);
                const uint32_t dst = sbase + C::OFF_KV + C::TB * s;
                const uint32_t full = bar(full_bar_of(pos));
                mbar_arrive_expect_tx(full, C::TB);
                for (int a = 0; a < C::NA; ++a) {
                    if (dense) tma_load_4d_hint(dst + a * kAtom, m, full, a * 64, h, (t0 + t) * BN, b, keep);
                    else tma_load_4d_hint(dst + a * kAtom, m, full, a * 64, (t0 + t) * BN, h, b, keep);
                }
                ++pos;
                return true;
            };
            bool ok = true;
            for (int ph = ph0; ok && n_tiles > 0 && ph <= PH_NEW; ++ph) {   // a part may have no key tile
                if (ph == PH_LSE) {
                    for (int t = 0; ok && t < n_tiles; ++t) ok = load(false, ph, t);
                } else {   // the order kv_pos_k / kv_pos_v describe
                    ok = load(false, ph, 0);
                    for (int t = 0; ok && t < n_tiles; ++t) {
                        if (t + 1 < n_tiles) ok = load(false, ph, t + 1);
                        if (ok) ok = load(true, ph, t);
                    }
                }
            }
            if (*abort_flag) {   // let copies already in flight land before the CTA exits
                for (int q = max(0, pos - kStages); q < pos; ++q) drain_wait(bar(full_bar_of(q)), full_parity(q), ERR_FULL);
            }
        }
    } else if (warp == 1 || warp == 2) {
        // ---------------- MMA issuers (one thread each) ----------------
        // Warp 1 issues the QK products, warp 2 the PV products, and pass LSE's QK
        // products (no PV there) are split by tile parity between the two: the tensor
        // pipe buffers only about two MMAs, and each issuer's barrier tests between
        // its batches are covered by the other's MMAs. Tile g's logits go to S buffer
        // g & 1, so each buffer of pass LSE has a single issuer. The whole warp runs
        // the loop; one elected lane issues (see mma_ss_x8_el).
        {
            constexpr uint32_t id_qk = idesc_bf16(128, 128, false, false, false);
            constexpr uint32_t id_pv = idesc_bf16(128, D, false, true, false);       // A = P from TMEM
            constexpr uint32_t id_pv_neg = idesc_bf16(128, D, false, true, true);    // pass OLD subtracts
            // descriptors are built once; per k-step only the start address moves
            const uint64_t d_q = smem_desc(sbase + C::OFF_Q, 16, 1024, 2);
            const uint64_t d_k = smem_desc(sbase + C::OFF_KV, 16, 1024, 2);
            const uint64_t d_v = smem_desc(sbase + C::OFF_KV, kAtom, 1024, 2);
            constexpr uint64_t TB16 = C::TB >> 4, ATOM16 = kAtom >> 4;
            static_assert(BN / 16 == 8 && (D == 64 || D == 96 || D == 128), "MMA batch shapes");
            // start-address offset (16-byte units) of k-step kk within a 64-element-atom tile
            auto kstep_off = [](int kk) -> uint64_t { return (uint64_t)((kk >> 2) * ATOM16 + (kk & 3) * 2); };
            uint64_t aq[D / 16];   // query-tile descriptors, one per k-step
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) aq[kk] = d_q + kstep_off(kk);
            const int n_old = first ? 0 : n_tiles;   // tiles of pass OLD; pass LSE covers [n_old, n_old + n_tiles)
            const int lse0 = n_old, new0 = n_old + n_tiles;
            // ring positions of the passes' first loads
            const int base_lse = 2 * n_old, base_new = base_lse + n_tiles;
            bool q_seen = first;   // the query tile holds this loop's q (passes LSE and NEW)
            // S = Q K^T for tile g into S buffer g & 1
            auto issue_qk = [&](int g) -> bool {
                const int kp = g < lse0 ? kv_pos_k(g) : g < new0 ? base_lse + g - lse0 : base_new + kv_pos_k(g - new0);
                const int ks = kp % kStages, sb = g & 1;
                if (!wait_bar_all(bar(full_bar_of(kp)), full_parity(kp), abort_flag, ERR_FULL, wlimit)) return false;
                // the S buffer's previous tile has been read by the softmax
                if (g >= kSBufs &&
                    !wait_bar_all(bar(BAR_S_READ + sb), ((g >> 1) - 1) & 1, abort_flag, ERR_S_READ, wlimit))
                    return false;
                if (g >= lse0 && !q_seen) {   // after pass OLD, once the query tile holds this loop's q
                    if (!wait_bar_all(bar(BAR_Q_READY), 0, abort_flag, ERR_Q_READY, wlimit)) return false;
                    q_seen = true;
                }
                tc_fence_after();
                const uint64_t dk = d_k + TB16 * (uint32_t)ks;
                uint64_t bk[D / 16];
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) bk[kk] = dk + kstep_off(kk);
                const uint32_t dst = tmem + 128u * (uint32_t)sb;
                if constexpr (D == 128) {
                    mma_ss_x8_el(dst, aq, bk, id_qk, 0u);
                } else {   // d = 64: one batch of four; d = 96: four, then two
                    mma_ss_x4_el(dst, aq, bk, id_qk, 0u);
                    if constexpr (D == 96) mma_ss_x2_el(dst, aq + 4, bk + 4, id_qk, 1u);
                }
                mma_commit_el(bar(BAR_S_FULL + sb));
                mma_commit_el(bar(BAR_EMPTY + ks));
                return true;
            };
            // acc (+/-)= P V for the tile with PV index pv (P buffer pv & 1)
            auto issue_pv = [&](int pv, bool old) -> bool {
                const int pb = pv & 1;
                const int vp = pv < n_old ? kv_pos_v(pv, n_tiles) : base_new + kv_pos_v(pv - n_old, n_tiles);
                const int vs = vp % kStages;
                if (!wait_bar_all(bar(full_bar_of(vp)), full_parity(vp), abort_flag, ERR_FULL, wlimit)) return false;
                if (!wait_bar_all(bar(BAR_P_FULL + pb), (uint32_t)(pv >> 1) & 1u, abort_flag, ERR_P_FULL, wlimit))
                    return false;
                tc_fence_after();
                const uint64_t dv = d_v + TB16 * (uint32_t)vs;
                const uint32_t pa = tmem + kColP + 64u * (uint32_t)pb;
                uint32_t ap[BN / 16];
                uint64_t bv[BN / 16];
#pragma unroll
                for (int kk = 0; kk < BN / 16; ++kk) {   // acc +-= P[:, 16kk..] * V[16kk.., :]
                    ap[kk] = pa + 8u * kk;
                    bv[kk] = dv + kk * 128;
                }
                mma_ts_x8_el(tmem + kColAcc, ap, bv, old ? id_pv_neg : id_pv, pv > 0 ? 1u : 0u);
                mma_commit_el(bar(BAR_PV_DONE + pb));
                mma_commit_el(bar(BAR_EMPTY + vs));
                return true;
            };
            bool ok = true;
            if (warp == 1) {
                for (int g = 0; ok && g < lse0; ++g) ok = issue_qk(g);
                for (int g = lse0; ok && g < new0; ++g)
                    if ((g & 1) == 0) ok = issue_qk(g);
                for (int g = new0; ok && g < total; ++g) ok = issue_qk(g);
            } else {
                for (int pv = 0; ok && pv < n_old; ++pv) ok = issue_pv(pv, true);
                for (int g = lse0; ok && g < new0; ++g)
                    if ((g & 1) == 1) ok = issue_qk(g);
                for (int t = 0; ok && t < n_tiles; ++t) ok = issue_pv(n_old + t, false);
                if (ok) mma_commit_el(bar(BAR_ACC));
            }
            if (!ok) {   // drain whatever the warp's elected lane issued before giving up
                mma_commit_el(bar(BAR_DRAIN + (warp - 1)));
                drain_wait(bar(BAR_DRAIN + (warp - 1)), 0, ERR_ACC);
            }
        }
    } else {
        // ---------------- softmax / epilogue: four groups, 32 columns each ----------------
        const int rq = (warp & 3) * 32;            // the warp's TMEM lane quadrant
        const int q4 = lane & 3;
        const int rlo = rq + (lane >> 2);          // fragment rows rlo + 8k
        const int cbase = wg * kGroupCols;
        const uint32_t t_lo = tmem + ((uint32_t)rq << 16), t_hi = tmem + ((uint32_t)(rq + 16) << 16);
        // per fragment row: partial old mass, running maximum of raw logits, sum of
        // 2^((logit - Mk) sl2); key counts and normalisers are read from shared memory
        float mk[4], Mk[4], Lk[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            mk[k] = 0.f;
            Mk[k] = -INFINITY;
            Lk[k] = 0.f;
        }
        bool ok = true;
        float *cb = p.c + bh * p.n_keys;
        // this lane's column after the butterfly of column_sum()
        const int Jc = lane >> 2;
        const int mycol = cbase + 8 * (Jc >> 1) + 2 * q4 + (Jc & 1);
        int g = 0, pv = 0;   // tile index over all passes; tiles with a PV product so far

        // Waits for tile g's logits and loads this thread's fragment of them; keys
        // past a row's prefix count are masked to -inf.
        auto load_s = [&](int t, float (&v)[32]) -> bool {
            const int sb = g & 1;
            if (!wait_bar_all(bar(BAR_S_FULL + sb), (g >> 1) & 1, abort_flag, ERR_S_FULL, wlimit)) return false;
            tc_fence_after();
            tmem_ld_16x256b_x4(t_lo + 128u * sb + cbase, v);
            tmem_ld_16x256b_x4(t_hi + 128u * sb + cbase, v + 16);
            tmem_wait_ld();
            warp_arrive(bar(BAR_S_READ + sb), lane);
            const int c0 = t * BN;
            if (c0 + BN > cnt_min) {   // not every row of the tile sees all 128 columns
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int nv = row_cnt[rlo + 8 * k] - c0 - cbase - 2 * q4;
#pragma unroll
                    for (int j = 0; j < 4; ++j)
#pragma unroll
                        for (int e = 0; e < 2; ++e)
                            if (8 * j + e >= nv) v[frag(k, j, e)] = -INFINITY;
                }
            }
            return true;
        };

        // One tile of pass OLD or NEW: probabilities with a known normaliser (nz =
        // -Z in log2 units; rows outside the tile or the sequence have nz = -inf and
        // get zero), P to TMEM for the PV product, then the old mass (pass OLD) and
        // the column masses.
        auto pv_tile = [&](auto old_c, int t, const float (&nz)[4]) -> bool {
            constexpr bool OLD = decltype(old_c)::value;
            // key position of this lane's column mass, loaded before the waits below
            const int jcol = col_index(t * BN + mycol);
            float v[32];
            if (!load_s(t, v)) return false;
#pragma unroll
            for (int k = 0; k < 4; ++k)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float2 x = fma2(make_float2(v[frag(k, j, 0)], v[frag(k, j, 1)]), make_float2(p.sl2, p.sl2),
                                          make_float2(nz[k], nz[k]));
                    v[frag(k, j, 0)] = ex2(x.x);
                    v[frag(k, j, 1)] = ex2(x.y);
                }
            // P buffer pv & 1 was last read by the PV product of the V tile two before
            const int pb = pv & 1;
            if (pv >= 2 && !wait_bar_all(bar(BAR_PV_DONE + pb), (uint32_t)((pv >> 1) - 1) & 1u, abort_flag, ERR_PV_DONE, wlimit))
                return false;
            tc_fence_after();
            // bf16 pairs of adjacent keys: register pair (2i, 2i + 1) is one packed P column
            const uint32_t pcol = kColP + 64u * (uint32_t)pb + (uint32_t)(cbase >> 1);
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t pk[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) pk[i] = pack_bf16x2_rn(v[16 * half + 2 * i], v[16 * half + 2 * i + 1]);
                tmem_st_16x128b_x4((half ? t_hi : t_lo) + pcol, pk);
            }
            tmem_wait_st();
            warp_arrive(bar(BAR_P_FULL + pb), lane);
            ++pv;
            ++g;
            // after the hand-off: the old mass m and the column masses
            if constexpr (OLD) {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    float2 a2 = make_float2(v[frag(k, 0, 0)], v[frag(k, 0, 1)]);
#pragma unroll
                    for (int j = 1; j < 4; ++j) a2 = add2(a2, make_float2(v[frag(k, j, 0)], v[frag(k, j, 1)]));
                    mk[k] += a2.x + a2.y;
                }
            }
            const float cs = column_sum(v, lane);
            red_add_f32_if(cb + (jcol != INT_MAX ? jcol : 0), OLD ? -cs : cs, jcol != INT_MAX && cs != 0.f);
            return true;
        };

        // ---- pass OLD: previous-loop probabilities, subtracted ----
        if (!first) {
            float nz[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) nz[k] = -row_zo[rlo + 8 * k];
            for (int t = t0; ok && t < t_end; ++t) {
                if (t == t_end - 1) {
                    // Once the last tile's logits are ready, every QK product of pass OLD
                    // (one issuing thread, completed in order) has read the query tile:
                    // start reloading it with this loop's q under the tile's softmax.
                    ok = wait_bar_all(bar(BAR_S_FULL + (g & 1)), (g >> 1) & 1, abort_flag, ERR_S_FULL, wlimit);
                    if (ok) load_query_tile_async<D>(smem + C::OFF_Q, p.q, st, b, h, p.H, p.n_state, qrows);
                }
                if (ok) ok = pv_tile(std::true_type{}, t, nz);
            }
            if (ok && n_tiles == 0) load_query_tile_async<D>(smem + C::OFF_Q, p.q, st, b, h, p.H, p.n_state, qrows);
            cp_async_wait_all();   // also after a failure: no copy stays in flight
            if (ok) {
                fence_proxy_async_smem();
                warp_arrive(bar(BAR_Q_READY), lane);
            }
        }
        // ---- pass LSE: online logsumexp of the new logits, per fragment row ----
        for (int t = t0; ok && t < t_end; ++t) {
            float v[32];
            if (!(ok = load_s(t, v))) break;
            ++g;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float m1 = max3f(v[frag(k, 0, 0)], v[frag(k, 0, 1)], v[frag(k, 1, 0)]);
                const float m2 = max3f(v[frag(k, 1, 1)], v[frag(k, 2, 0)], v[frag(k, 2, 1)]);
                const float m3 = max3f(v[frag(k, 3, 0)], v[frag(k, 3, 1)], Mk[k]);
                const float mnew = max3f(m1, m2, m3);
                // a row that has seen no key yet keeps M = -inf and L = 0 (every term is 0)
                const float nb = mnew == -INFINITY ? 0.f : -mnew * p.sl2;
                float2 a2 = make_float2(Lk[k] * ex2(fmaf(Mk[k], p.sl2, nb)), 0.f);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const float2 x = fma2(make_float2(v[frag(k, j, 0)], v[frag(k, j, 1)]), make_float2(p.sl2, p.sl2),
                                          make_float2(nb, nb));
                    a2 = add2(a2, make_float2(ex2(x.x), ex2(x.y)));
                }
                Lk[k] = a2.x + a2.y;
                Mk[k] = mnew;
            }
        }
        // ---- merge the row statistics: Z' = lam - ln m ----
        if (ok) {
            // the epilogue reads this thread's part of its O row: fetch it into L2 now
            if (row_ok && !first && part == 0) {
                const float *orow = p.o + ((((long long)b * p.n_state + pos) * p.H + h) * D + wg * (D / kGroups));
                asm volatile("prefetch.global.L2 [%0];" ::"l"(orow));
            }
            // the four lanes of a row, then the four groups
#pragma unroll
            for (int k = 0; k < 4; ++k) {
#pragma unroll
                for (int off = 1; off <= 2; off <<= 1) {
                    const float mo = __shfl_xor_sync(0xffffffffu, mk[k], off);
                    const float Mo = __shfl_xor_sync(0xffffffffu, Mk[k], off);
                    const float Lo = __shfl_xor_sync(0xffffffffu, Lk[k], off);
                    const float Mx = fmaxf(Mk[k], Mo);
                    Lk[k] = Mx == -INFINITY ? 0.f : Lk[k] * ex2((Mk[k] - Mx) * p.sl2) + Lo * ex2((Mo - Mx) * p.sl2);
                    Mk[k] = Mx;
                    mk[k] += mo;
                }
            }
            float *ex = reinterpret_cast<float *>(smem + C::OFF_X);
            if (q4 == 0) {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    float *e = ex + (wg * 128 + rlo + 8 * k) * 3;
                    e[0] = mk[k];
                    e[1] = Mk[k];
                    e[2] = Lk[k];
                }
            }
            warp_arrive(bar(BAR_STATS), lane);
            ok = wait_bar_all(bar(BAR_STATS), 0, abort_flag, ERR_STATS, wlimit);
            if (ok && wg == 0) {
                // this CTA's old mass, maximum and sum of the row
                float mx = 0.f, Mx = -INFINITY, Lx = 0.f;
                if (r < rows) {
#pragma unroll
                    for (int k = 0; k < kGroups; ++k) {
                        mx += ex[(k * 128 + r) * 3 + 0];
                        Mx = fmaxf(Mx, ex[(k * 128 + r) * 3 + 1]);
                    }
                    if (Mx > -INFINITY) {
#pragma unroll
                        for (int k = 0; k < kGroups; ++k)
                            Lx += ex[(k * 128 + r) * 3 + 2] * ex2((ex[(k * 128 + r) * 3 + 1] - Mx) * p.sl2);
                    }
                }
                if (split) {
                    // publish them to every CTA of the cluster; each combines all parts
                    // in rank order, so every part holds the same Z' bits
                    const uint32_t xa = sbase + C::OFF_XCL + (uint32_t)(part * 128 + r) * 16u;
                    for (int q = 0; q < p.nparts; ++q) cl_st4(cl_map(xa, (uint32_t)q), make_float4(mx, Mx, Lx, 0.f));
                    __syncwarp();
                    if (lane == 0)
                        for (int q = 0; q < p.nparts; ++q) cl_mbar_arrive(cl_map(bar(BAR_XSTAT), (uint32_t)q));
                    ok = __all_sync(0xffffffffu, wait_bar_cluster(bar(BAR_XSTAT), 0, abort_flag, ERR_XSTAT, wlimit));
                    if (ok) {
                        const float4 *xc = reinterpret_cast<const float4 *>(smem + C::OFF_XCL);
                        mx = 0.f;
                        Mx = -INFINITY;
                        Lx = 0.f;
                        for (int q = 0; q < p.nparts; ++q) {
                            mx += xc[q * 128 + r].x;
                            Mx = fmaxf(Mx, xc[q * 128 + r].y);
                        }
                        if (Mx > -INFINITY)
                            for (int q = 0; q < p.nparts; ++q) Lx += xc[q * 128 + r].z * ex2((xc[q * 128 + r].y - Mx) * p.sl2);
                    }
                }
                // rows with an empty key set or no old mass keep their state (Z' = inf)
                float zn = INFINITY;
                if (r < rows && Mx > -INFINITY) {
                    if (first) mx = 1.f;
                    if (mx >= FLT_MIN) zn = Mx * p.sl2 + __log2f(Lx) - __log2f(mx);
                }
                row_zn[r] = zn;
            }
            if (ok) {
                warp_arrive(bar(BAR_ZN), lane);
                ok = wait_bar_all(bar(BAR_ZN), 0, abort_flag, ERR_ZN, wlimit);
            }
        }
        // ---- pass NEW: this loop's probabilities with the merged normaliser, added ----
        if (ok) {
            float nz[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) nz[k] = -row_zn[rlo + 8 * k];
            for (int t = t0; ok && t < t_end; ++t) ok = pv_tile(std::false_type{}, t, nz);
        }
        // Epilogue. Each warp walks whole rows so that O, Z and qhat move in full
        // lines: first its O rows are loaded (they do not depend on the accumulator,
        // so the loads overlap the last PV products); then every thread parks its
        // accumulator row in shared memory (the ring is idle by then), and the rows
        // are added to O and written back.
        constexpr int RPW = BM / kSoftmaxWarps;   // rows per warp
        const int sw = warp - kFirstSoftmaxWarp;
        const uint64_t stream = l2_policy_evict_first();   // O and qhat rows are touched once
        float4 ov[RPW];
        long long srow[RPW];
        bool upd[RPW];
#pragma unroll
        for (int i = 0; i < RPW; ++i) {
            const int rr = sw + kSoftmaxWarps * i;
            upd[i] = ok && part == 0 && rr < rows && row_zn[rr] < INFINITY;   // rank 0 writes a split item
            srow[i] = upd[i] ? ((long long)b * p.n_state + row_pos_s[rr]) * p.H + h : 0;
            ov[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (upd[i] && !first && lane < D / 4) {
                const uint4 u = ld_global_v4_hint(reinterpret_cast<const float4 *>(p.o + srow[i] * D) + lane, stream);
                ov[i] = make_float4(__uint_as_float(u.x), __uint_as_float(u.y), __uint_as_float(u.z),
                                    __uint_as_float(u.w));
            }
        }
        if (ok && wait_bar_all(bar(BAR_ACC), 0, abort_flag, ERR_ACC, wlimit)) {
            tc_fence_after();
            constexpr int GD = D / kGroups;   // accumulator columns per group (16, 24 or 32)
            float *xo = reinterpret_cast<float *>(smem + C::OFF_KV);
            const uint32_t lane_base = (uint32_t)rq << 16;
#pragma unroll
            for (int u = 0; u < GD; u += 8) {
                float av[8];
                tmem_ld_32x32b_x8(tmem + lane_base + kColAcc + wg * GD + u, av);
                tmem_wait_ld();
                if (n_tiles == 0)   // a part without key tiles: no PV product wrote the accumulator
#pragma unroll
                    for (int i = 0; i < 8; ++i) av[i] = 0.f;
                float4 *dst = reinterpret_cast<float4 *>(xo + r * C::XS + wg * GD + u);
                dst[0] = make_float4(av[0], av[1], av[2], av[3]);
                dst[1] = make_float4(av[4], av[5], av[6], av[7]);
            }
            warp_arrive(bar(BAR_EPI), lane);
            bool go = wait_bar_all(bar(BAR_EPI), 0, abort_flag, ERR_EPI, wlimit);
            if (go && split) {   // rank 0 sums the parts' parked accumulators and writes the rows
                if (st == 0) cl_mbar_arrive(cl_map(bar(BAR_XACC), 0u));
                go = part == 0 &&
                     __all_sync(0xffffffffu, wait_bar_cluster(bar(BAR_XACC), 0, abort_flag, ERR_XACC, wlimit));
                if (go && lane < D / 4) {
                    // the other parts' accumulators, added in rank order into the parked rows
                    // (each thread to the elements it writes back below), two rows at a time
                    // so that their remote loads are in flight together
#pragma unroll
                    for (int i = 0; i < RPW; i += 2) {
                        float4 rb[2][kMaxParts - 1];
#pragma unroll
                        for (int j = 0; j < 2; ++j) {
                            const int rr = sw + kSoftmaxWarps * (i + j);
                            const uint32_t xa = smem_u32(xo + rr * C::XS + 4 * lane);
#pragma unroll
                            for (int q = 1; q < kMaxParts; ++q)
                                if (rr < rows && q < p.nparts) rb[j][q - 1] = cl_ld4(cl_map(xa, (uint32_t)q));
                        }
#pragma unroll
                        for (int j = 0; j < 2; ++j) {
                            const int rr = sw + kSoftmaxWarps * (i + j);
                            if (rr >= rows) continue;
                            float4 *own = reinterpret_cast<float4 *>(xo + rr * C::XS) + lane;
                            float4 a4 = *own;
#pragma unroll
                            for (int q = 1; q < kMaxParts; ++q)
                                if (q < p.nparts) {
                                    a4.x += rb[j][q - 1].x;
                                    a4.y += rb[j][q - 1].y;
                                    a4.z += rb[j][q - 1].z;
                                    a4.w += rb[j][q - 1].w;
                                }
                            *own = a4;
                        }
                    }
                }
            }
            if (go) {
#pragma unroll
                for (int i = 0; i < RPW; ++i) {
                    if (!upd[i]) continue;
                    const int rr = sw + kSoftmaxWarps * i;
                    if (lane < D / 4) {
                        const float4 a4 = reinterpret_cast<const float4 *>(xo + rr * C::XS)[lane];
                        float4 o4 = ov[i];
                        o4.x += a4.x;
                        o4.y += a4.y;
                        o4.z += a4.z;
                        o4.w += a4.w;
                        st_global_v4_hint(reinterpret_cast<float4 *>(p.o + srow[i] * D) + lane,
                                          make_uint4(__float_as_uint(o4.x), __float_as_uint(o4.y), __float_as_uint(o4.z),
                                                     __float_as_uint(o4.w)),
                                          stream);
                    }
                    // the query tile holds this loop's q: it becomes qhat
                    if (lane < D / 8)
                        st_global_v4_hint(reinterpret_cast<uint4 *>(p.q_hat + srow[i] * D) + lane,
                                          *reinterpret_cast<const uint4 *>(smem + C::OFF_Q + swz_off(rr, lane)), stream);
                    if (lane == 0) p.z[bh * p.n_state + row_pos_s[rr]] = row_zn[rr] * kLn2;
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(misc[0], kTmemCols);
    }
    // a split item: no CTA exits while another may still read its shared memory.
    // Every wait above is bounded, so every CTA of the cluster gets here.
    if (split) {
        cl_arrive();
        cl_wait();
    }
    if (p.late_wait) pdl_wait();
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
    static std::once_flag once[kMaxDevices];
    static cudaError_t attr_res[kMaxDevices];
    const cudaError_t ea = once_per_device(once, attr_res, [] {
        return cudaFuncSetAttribute(tc_attention_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, Cf::SMEM);
    });
    if (ea != cudaSuccess) return ea;
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
    kp.row_cnt = p.row_cnt;
    kp.key_idx = p.key_idx;
    kp.q = p.q;
    kp.q_hat = p.q_hat;
    kp.o = p.o;
    kp.z = p.z;
    kp.c = p.c;
    kp.sl2 = kLog2e / sqrtf((float)D);
    kp.seq_exit = p.seq_exit;
    kp.item_base = 0;
    kp.nparts = 1;
    kp.late_wait = 0;
    if (!dense && !p.row_cnt) return cudaErrorInvalidValue;
    // One CTA per (row tile, head) item and sequence, one CTA per SM. Lazy items
    // are of nearly equal size (the selected keys sit early, so most row tiles
    // see all of them), and the items past the last full wave would leave the
    // other SMs idle for a whole item: those go to a second launch that splits
    // each over a cluster of up to four CTAs by key tiles.
    const int X = kp.n_row_tiles * p.H;
    int tail_x = 0, parts = 1;
    if (!dense) {
        int dev = 0;
        if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
        static int sms[kMaxDevices];
        if (sms[dev] == 0 && cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return cudaErrorInvalidDevice;
        const long long total = (long long)X * p.B, rem = total % sms[dev];
        if (total >= sms[dev] && rem > 0) {
            tail_x = (int)((rem + p.B - 1) / p.B);
            parts = (int)std::min<long long>(kMaxParts, sms[dev] / ((long long)tail_x * p.B));
            if (parts < 2) tail_x = 0, parts = 1;
        }
    }
    {
        // The split items go first, on an otherwise idle GPU; the main grid follows
        // without waiting for them and fills the SMs they leave free.
        KernelTimer kt("tc_attention", s);
        kp.late_wait = 0;
        if (tail_x > 0) {
            KParams kt2 = kp;
            kt2.item_base = X - tail_x;
            kt2.nparts = parts;
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(tail_x * parts, 1, p.B);
            cfg.blockDim = dim3(kThreads);
            cfg.dynamicSmemBytes = (size_t)Cf::SMEM;
            cfg.stream = s;
            cudaLaunchAttribute attr[2];
            attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[0].val.programmaticStreamSerializationAllowed = 1;
            attr[1].id = cudaLaunchAttributeClusterDimension;
            attr[1].val.clusterDim.x = (unsigned)parts;
            attr[1].val.clusterDim.y = 1;
            attr[1].val.clusterDim.z = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 2;
            const cudaError_t e =
                cudaLaunchKernelEx(&cfg, tc_attention_kernel<D>, kt2, maps[0], maps[1], maps[2], maps[3]);
            if (e != cudaSuccess) return e;
            kp.late_wait = 1;
        }
        if (X - tail_x > 0) {
            const cudaError_t e = launch_pdl(tc_attention_kernel<D>, dim3(X - tail_x, 1, p.B), dim3(kThreads),
                                             (size_t)Cf::SMEM, s, kp, maps[0], maps[1], maps[2], maps[3]);
            if (e != cudaSuccess) return e;
            if (tail_x > 0) note_launch(1);   // the timer above counted one of the two
        }
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

int32_t tc_attention_set_wait_limit(unsigned long long ns) {
    return (int32_t)cudaMemcpyToSymbol(g_tc_wait_limit_ns, &ns, sizeof ns);
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

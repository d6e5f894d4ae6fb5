// attn_decode.cu -- lazy attention for a handful of rows (decode), reading the
// base + delta cache directly.
//
// Same step as attn_tc.cu (rit.work page "FlashLoop: Fast and
// Memory-Efficient Looped Transformers via Lazy Updates", section "FlashLoop
// combines three kinds of saving": keys chosen from the previous loop's
// statistics, total probability mass of the chosen group preserved), but for
// one new query per sequence: the work is a matrix-vector product, bound by
// the bytes of the selected keys and values, so the selected K/V are
// reconstructed (base + dequantised deltas, fp32, rounded to bf16) on the fly
// instead of being materialised first.
//
// One CTA per (sequence, head, row). 16 groups of 16 lanes walk the key list;
// a lane owns an 8-element chunk of d. Pass 1 stores the old and new logits
// of every key in shared memory, the row statistics (m, lam) come from
// block reductions, pass 2 accumulates u and w and updates the column mass.
#include <float.h>
#include <mutex>

#include "common.cuh"

namespace fl {
namespace {

constexpr int kThreads = 256;
constexpr int kGroups = kThreads / 16;

__device__ __forceinline__ float group16_sum(float v) {
    v += __shfl_xor_sync(0xffffffffu, v, 8);
    v += __shfl_xor_sync(0xffffffffu, v, 4);
    v += __shfl_xor_sync(0xffffffffu, v, 2);
    v += __shfl_xor_sync(0xffffffffu, v, 1);
    return v;
}

__device__ __forceinline__ void round_bf16x8(float v[8]) {
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = __bfloat162float(__float2bfloat16_rn(v[e]));
}

// Block-wide reduction (max or sum) through shared scratch of kThreads/32 floats.
template <bool kMax>
__device__ float block_reduce(float v, float *red) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float o = __shfl_xor_sync(0xffffffffu, v, off);
        v = kMax ? fmaxf(v, o) : v + o;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    v = red[0];
    for (int w = 1; w < kThreads / 32; ++w) v = kMax ? fmaxf(v, red[w]) : v + red[w];
    return v;
}

struct DecKParams {
    int mode, H, n_keys, n_state, R, K, N_cap, R_cap;
    const int32_t *row_pos, *row_slot, *key_idx;
    const uint16_t *q;
    uint16_t *q_hat;
    float *o, *z, *c;
    DeltaView old_view, new_view;
    bool shared_base;   // old and new share the base (lazy): reconstruct incrementally
    float scale;
};

template <int D>
__global__ void __launch_bounds__(kThreads)
decode_attention_kernel(const __grid_constant__ DecKParams p) {
    extern __shared__ float sm[];
    constexpr int CH = D / 8;
    const int row = blockIdx.x % p.R;
    const long long bh = blockIdx.x / p.R;
    const int h = (int)(bh % p.H);
    const long long b = bh / p.H;
    const bool dense = p.mode != FLASHLOOP_ATTN_LAZY;
    const bool first = p.mode == FLASHLOOP_ATTN_FIRST_DENSE;
    const int pos = __ldg(p.row_pos + b * p.R + row);
    const int slot = p.row_slot ? __ldg(p.row_slot + b * p.R + row) : pos;
    const int32_t *S = dense ? nullptr : p.key_idx + bh * p.K;
    int nk;
    if (dense) {
        nk = min(pos + 1, p.n_keys);
    } else {
        int lo = 0, hi = p.K;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (__ldg(S + mid) <= pos) lo = mid + 1; else hi = mid;
        }
        nk = lo;
    }
    if (nk == 0) return;   // no key at or before the row: state unchanged

    float *sig = sm;                   // [nk] old logits (scaled)
    float *tau = sm + nk;              // [nk] new logits (scaled)
    float *red = sm + 2 * nk;          // [kThreads/32]
    float *acc = red + kThreads / 32;  // [2][kGroups][D]

    const int grp = threadIdx.x >> 4, gl = threadIdx.x & 15;
    const bool has_chunk = gl < CH;
    const int c8 = has_chunk ? gl : 0;
    const long long srow = ((b * p.n_state + slot) * p.H + h) * (long long)D;
    float qn[8], qo[8];
    unpack_bf16x8(ldg_nc_v4(p.q + srow + c8 * 8), qn);
    if (!first) unpack_bf16x8(ldg_nc_v4(p.q_hat + srow + c8 * 8), qo);

    // pass 1: logits of every key in the list. Both 16-lane groups of a warp
    // run the same number of iterations (a group past the end recomputes
    // key 0 and stores nothing) because the sums below shuffle across the
    // whole warp.
    for (int t0 = 0; t0 < nk; t0 += kGroups) {
        const int t = t0 + grp;
        const bool tv = t < nk;
        const int j = dense ? (tv ? t : 0) : __ldg(S + (tv ? t : 0));
        float kn[8], ko[8];
        float so = 0.f, sn = 0.f;
        if (p.shared_base) {
            load_base8(p.old_view.k_base, b, j, h, c8, p.H, D, p.N_cap, ko);
            apply_deltas(p.old_view, false, 0, p.old_view.n_layers, b, j, h, c8, p.H, D, p.N_cap, p.R_cap, ko);
#pragma unroll
            for (int e = 0; e < 8; ++e) kn[e] = ko[e];
            apply_deltas(p.new_view, false, p.old_view.n_layers, p.new_view.n_layers, b, j, h, c8, p.H, D, p.N_cap,
                         p.R_cap, kn);
        } else {
            load_base8(p.new_view.k_base, b, j, h, c8, p.H, D, p.N_cap, kn);
            if (!first) load_base8(p.old_view.k_base, b, j, h, c8, p.H, D, p.N_cap, ko);
        }
        round_bf16x8(kn);
        if (!first) round_bf16x8(ko);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            sn = fmaf(qn[e], kn[e], sn);
            if (!first) so = fmaf(qo[e], ko[e], so);
        }
        if (!has_chunk) sn = so = 0.f;
        sn = group16_sum(sn);
        so = group16_sum(so);
        if (tv && gl == 0) {
            tau[t] = sn * p.scale;
            sig[t] = so * p.scale;
        }
    }
    __syncthreads();

    // row statistics
    const float zo = first ? 0.f : __ldg(p.z + bh * p.n_state + slot);
    float mx = -INFINITY, ms = 0.f;
    for (int t = threadIdx.x; t < nk; t += kThreads) {
        mx = fmaxf(mx, tau[t]);
        if (!first) ms += expf(sig[t] - zo);
    }
    mx = block_reduce<true>(mx, red);
    const float m = first ? 1.f : block_reduce<false>(ms, red);
    float ls = 0.f;
    for (int t = threadIdx.x; t < nk; t += kThreads) ls += expf(tau[t] - mx);
    ls = block_reduce<false>(ls, red);
    const float lam = mx + logf(ls);
    if (!first && !(m >= FLT_MIN)) return;   // old mass underflowed: keep the row's state

    // pass 2: u = sum p v_old, w = sum a v_new, column mass
    float u[8] = {0, 0, 0, 0, 0, 0, 0, 0}, w[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    float *cb = p.c + bh * p.n_keys;
    for (int t = grp; t < nk; t += kGroups) {
        const int j = dense ? t : __ldg(S + t);
        const float a = expf(tau[t] - lam);
        const float pj = first ? 0.f : expf(sig[t] - zo);
        float vn[8], vo[8];
        if (p.shared_base) {
            load_base8(p.old_view.v_base, b, j, h, c8, p.H, D, p.N_cap, vo);
            apply_deltas(p.old_view, true, 0, p.old_view.n_layers, b, j, h, c8, p.H, D, p.N_cap, p.R_cap, vo);
#pragma unroll
            for (int e = 0; e < 8; ++e) vn[e] = vo[e];
            apply_deltas(p.new_view, true, p.old_view.n_layers, p.new_view.n_layers, b, j, h, c8, p.H, D, p.N_cap,
                         p.R_cap, vn);
        } else {
            load_base8(p.new_view.v_base, b, j, h, c8, p.H, D, p.N_cap, vn);
            if (!first) load_base8(p.old_view.v_base, b, j, h, c8, p.H, D, p.N_cap, vo);
        }
        round_bf16x8(vn);
#pragma unroll
        for (int e = 0; e < 8; ++e) w[e] = fmaf(a, vn[e], w[e]);
        if (!first) {
            round_bf16x8(vo);
#pragma unroll
            for (int e = 0; e < 8; ++e) u[e] = fmaf(pj, vo[e], u[e]);
        }
        if (gl == 0) atomicAdd(cb + j, m * a - pj);
    }
    if (has_chunk) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            acc[grp * D + c8 * 8 + e] = u[e];
            acc[(kGroups + grp) * D + c8 * 8 + e] = w[e];
        }
    }
    __syncthreads();
    for (int x = threadIdx.x; x < D; x += kThreads) {
        float us = 0.f, ws = 0.f;
        for (int g = 0; g < kGroups; ++g) {
            us += acc[g * D + x];
            ws += acc[(kGroups + g) * D + x];
        }
        const float prev = first ? 0.f : p.o[srow + x];
        p.o[srow + x] = prev - us + m * ws;
        p.q_hat[srow + x] = p.q[srow + x];
    }
    if (threadIdx.x == 0) p.z[bh * p.n_state + slot] = lam - logf(m);
}

template <int D>
cudaError_t launch_d(const DecodeAttnParams &q, cudaStream_t s) {
    int nk_max = q.mode == FLASHLOOP_ATTN_LAZY ? q.K : q.n_keys;
    const size_t smem = (size_t)(2 * nk_max + kThreads / 32 + 2 * kGroups * D) * sizeof(float);
    if (smem > 220 * 1024) return cudaErrorInvalidValue;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaFuncSetAttribute(decode_attention_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, 220 * 1024);
    });
    DecKParams p;
    p.mode = q.mode;
    p.H = q.H;
    p.n_keys = q.n_keys;
    p.n_state = q.n_state;
    p.R = q.R;
    p.K = q.K;
    p.N_cap = q.N_cap;
    p.R_cap = q.R_cap;
    p.row_pos = q.row_pos;
    p.row_slot = q.row_slot;
    p.key_idx = q.key_idx;
    p.q = q.q;
    p.q_hat = q.q_hat;
    p.o = q.o;
    p.z = q.z;
    p.c = q.c;
    p.old_view = q.old_view;
    p.new_view = q.new_view;
    p.shared_base = q.mode == FLASHLOOP_ATTN_LAZY;
    p.scale = 1.0f / sqrtf((float)D);
    const long long grid = (long long)q.B * q.H * q.R;
    {
        KernelTimer kt("decode_attention", s);
        decode_attention_kernel<D><<<(unsigned)grid, kThreads, smem, s>>>(p);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_attention(const DecodeAttnParams &p, cudaStream_t s) {
    if (p.R == 0) return cudaSuccess;
    switch (p.d) {
        case 64: return launch_d<64>(p, s);
        case 96: return launch_d<96>(p, s);
        case 128: return launch_d<128>(p, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace fl

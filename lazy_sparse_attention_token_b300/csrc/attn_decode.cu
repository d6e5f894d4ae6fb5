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
// One thread-block cluster per (sequence, head, row); its CTAs split the row's
// key list into contiguous chunks, so a long list is streamed by several SMs.
// In a CTA, 16 groups of 16 lanes walk the chunk, kU keys per group at a time.
// Every delta layer's entry of every key of the chunk is looked up once, into
// shared memory, for both passes; a step then loads its kU base rows and the
// codes of a layer together, with no dependent lookup in front.
// Pass 1 keeps the chunk's old and new logits in shared memory; the row
// statistics (old mass m, logsumexp lam) are merged across the cluster through
// distributed shared memory; pass 2 accumulates u and w and updates the column
// mass; the u and w partials are summed on cluster rank 0, which updates the
// row's state.
#include <float.h>
#include <mutex>

#include "common.cuh"

namespace fl {
namespace {

constexpr int kThreads = 256;
constexpr int kGroups = kThreads / 16;
constexpr int kU = 2;              // keys per group per step
constexpr int kMaxCluster = 8;
constexpr int kKeysPerCta = 1024;  // a CTA per this many keys, up to kMaxCluster

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

// ---- cluster helpers (distributed shared memory) --------------------------------
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
__device__ __forceinline__ void cl_st_f32(uint32_t addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ void cl_red_add_f32(uint32_t addr, float v) {
    asm volatile("red.shared::cluster.add.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
// Every thread of every CTA of the cluster passes each of these.
__device__ __forceinline__ void cl_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

struct DecKParams {
    int mode, H, n_keys, n_state, R, K, N_cap, R_cap;
    int chunk;   // keys per CTA (shared-memory sizing)
    const int32_t *row_pos, *row_slot, *key_idx;
    const uint16_t *q;
    uint16_t *q_hat;
    float *o, *z, *c;
    DeltaView old_view, new_view;
    float scale;
};

// Reconstruction (base + delta layers, fp32 in ascending layer order) of the
// 8-element chunk c8 of kU keys j, handed out twice per key: on_old(u, r) with
// the old view's layers applied, then on_new(u, r) with the new view's. One
// 8-float running value per key is live, not an old and a new copy. Every
// layer's entry of every key of the chunk was looked up once into shared
// memory (ents[m * chunk + t], t = the key's place in the chunk), so the codes
// and scales of kLayerPair layers at a time load together with no dependent
// lookup in front of them.
constexpr int kLayerPair = 1;
template <int D, class OnOld, class OnNew>
__device__ __forceinline__ void visit_rec(const DeltaView &ov, const DeltaView &nv, bool is_v, long long b,
                                          const int (&j)[kU], const int (&tt)[kU], const int *ents, int chunk, int h,
                                          int c8, int H, int N_cap, int R_cap, OnOld &&on_old, OnNew &&on_new) {
    float r[kU][8];
#pragma unroll
    for (int u = 0; u < kU; ++u) load_base8(ov, is_v, b, j[u], h, c8, H, D, N_cap, r[u]);
    for (int m0 = 0; m0 < nv.n_layers; m0 += kLayerPair) {
        int ent[kLayerPair][kU];
        uint32_t w[kLayerPair][kU];
        float s[kLayerPair][kU];
#pragma unroll
        for (int mm = 0; mm < kLayerPair; ++mm) {
            const int m = m0 + mm;
            const bool live = m < nv.n_layers;
            const uint8_t *codes = live ? (is_v ? nv.v_codes[m] : nv.k_codes[m]) : nullptr;
            const uint16_t *scales = live ? (is_v ? nv.v_scales[m] : nv.k_scales[m]) : nullptr;
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                ent[mm][u] = live ? ents[m * chunk + tt[u]] : -1;
                w[mm][u] = 0u;
                s[mm][u] = 0.f;
                if (ent[mm][u] >= 0) {
                    const long long e = (b * R_cap + ent[mm][u]) * H + h;
                    w[mm][u] = load_codes8(codes + e * (D * nv.code_bits / 8), c8, nv.code_bits);
                    s[mm][u] = __half2float(__ushort_as_half(__ldg(scales + e * (D / 32) + c8 / 4)));
                }
            }
        }
#pragma unroll
        for (int mm = 0; mm < kLayerPair; ++mm) {
            const int m = m0 + mm;
            if (m >= nv.n_layers) break;
            if (m == ov.n_layers) {
#pragma unroll
                for (int u = 0; u < kU; ++u) on_old(u, r[u]);
            }
#pragma unroll
            for (int u = 0; u < kU; ++u)
                if (ent[mm][u] >= 0) dequant_add8(r[u], w[mm][u], s[mm][u]);
        }
    }
    if (nv.n_layers <= ov.n_layers) {
#pragma unroll
        for (int u = 0; u < kU; ++u) on_old(u, r[u]);
    }
#pragma unroll
    for (int u = 0; u < kU; ++u) on_new(u, r[u]);
}

// One instantiation per mode, so that a mode's unused state (the old keys and
// values of the first dense loop, the delta entries of a dense loop) takes no
// registers. Every mode runs five CTAs per SM (48 registers): the kernel waits on
// gathers of scattered key rows, and on this part more resident warps with a few
// spilled registers beat fewer warps with more keys in flight each (two keys per
// group and one delta layer at a time, measured against four keys, two layers and
// two CTAs per SM: the 64-sequence, 16K-context decode token step 5.80 -> 4.37 ms,
// graph-replayed; four CTAs per SM for the first loop alone: 4.54 ms).
template <int D, int kMode>
__global__ void __launch_bounds__(kThreads, 5)
decode_attention_kernel(const __grid_constant__ DecKParams p) {
    extern __shared__ float sm[];
    constexpr int CH = D / 8;
    const uint32_t ncta = cl_size(), rank = cl_rank();
    const long long item = blockIdx.x / ncta;   // (sequence, head, row)
    const int row = (int)(item % p.R);
    const long long bh = item / p.R;
    const int h = (int)(bh % p.H);
    const long long b = bh / p.H;
    constexpr bool dense = kMode != FLASHLOOP_ATTN_LAZY;
    constexpr bool first = kMode == FLASHLOOP_ATTN_FIRST_DENSE;
    constexpr bool shared_base = kMode == FLASHLOOP_ATTN_LAZY;   // old and new share the base: incremental
    const int pos = __ldg(p.row_pos + b * p.R + row);
    const int slot = p.row_slot ? __ldg(p.row_slot + b * p.R + row) : pos;
    const int32_t *S = dense ? nullptr : p.key_idx + bh * p.K;
    int nk;   // keys at or before the row: a prefix of the ascending list
    if (dense) {
        nk = min(pos + 1, p.n_keys);
    } else if (__ldg(S + p.K - 1) <= pos) {
        nk = p.K;
    } else {
        int lo = 0, hi = p.K;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (__ldg(S + mid) <= pos) lo = mid + 1; else hi = mid;
        }
        nk = lo;
    }
    if (nk == 0) return;   // no key at or before the row: state unchanged (the whole cluster)

    // this CTA's chunk of the key list
    const int chunk = (nk + (int)ncta - 1) / (int)ncta;
    const int k0 = min(nk, (int)rank * chunk), cn = min(nk, k0 + chunk) - k0;

    int *idx = reinterpret_cast<int *>(sm);                  // [p.chunk] key positions (lazy)
    float *sig = sm + p.chunk;                                // [p.chunk] old logits (scaled)
    float *tau = sig + p.chunk;                               // [p.chunk] new logits (scaled)
    float *red = tau + p.chunk;                               // [kThreads/32]
    float *acc = red + kThreads / 32;                         // [2][kGroups][D]
    float *stats = acc + 2 * kGroups * D;                     // [kMaxCluster][3] (mx, ls, ms) of every rank
    float *uw = stats + kMaxCluster * 3;                      // [2][D] cluster sums of u, w (rank 0)
    int *ents = reinterpret_cast<int *>(uw + 2 * D);          // lazy: [layers][p.chunk] delta entries

    const int grp = threadIdx.x >> 4, gl = threadIdx.x & 15;
    const bool has_chunk = gl < CH;
    const int c8 = has_chunk ? gl : 0;
    const long long srow = ((b * p.n_state + slot) * p.H + h) * (long long)D;
    float qn[8], qo[8];
    unpack_bf16x8(ldg_nc_v4(p.q + srow + c8 * 8), qn);
    if (!first) unpack_bf16x8(ldg_nc_v4(p.q_hat + srow + c8 * 8), qo);
    if (!dense)
        for (int t = threadIdx.x; t < cn; t += kThreads) idx[t] = __ldg(S + k0 + t);
    if (rank == 0)
        for (int x = threadIdx.x; x < 2 * D; x += kThreads) uw[x] = 0.f;
    __syncthreads();
    if (shared_base) {   // every (layer, key) entry of the chunk, looked up once for both passes
        const int nl = p.new_view.n_layers;
        for (int x = threadIdx.x; x < nl * cn; x += kThreads) {
            const int m = x / cn, t = x - m * cn;
            ents[m * p.chunk + t] = __ldg(p.new_view.slot[m] + b * p.N_cap + idx[t]);
        }
        __syncthreads();
    }
    auto key_at = [&](int t) { return dense ? k0 + t : idx[t]; };

    // pass 1: logits of the chunk's keys. Both 16-lane groups of a warp run the
    // same number of steps (keys past the end recompute the chunk's first key and
    // store nothing) because the sums below shuffle across the whole warp.
    for (int t0 = 0; t0 < cn; t0 += kGroups * kU) {
        int jj[kU], tt[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int t = t0 + u * kGroups + grp;
            tt[u] = t < cn ? t : 0;
            jj[u] = key_at(tt[u]);
        }
        float dot_n[kU], dot_o[kU];   // this lane's part of q.k_new and qhat.k_old
        // bf16 rounding of a reconstructed chunk, then its dot product with a query chunk
        auto dot8 = [&](const float (&q8)[8], const float (&r)[8]) {
            float k8[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) k8[e] = r[e];
            round_bf16x8(k8);
            float acc8 = 0.f;
#pragma unroll
            for (int e = 0; e < 8; ++e) acc8 = fmaf(q8[e], k8[e], acc8);
            return acc8;
        };
        if constexpr (shared_base) {
            visit_rec<D>(p.old_view, p.new_view, false, b, jj, tt, ents, p.chunk, h, c8, p.H, p.N_cap, p.R_cap,
                         [&](int u, const float (&r)[8]) { dot_o[u] = dot8(qo, r); },
                         [&](int u, const float (&r)[8]) { dot_n[u] = dot8(qn, r); });
        } else {   // dense layers: every key's rows are requested before any is used
            float kn[kU][8], ko[kU][8];
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                load_base8(p.new_view.k_base, b, jj[u], h, c8, p.H, D, p.N_cap, kn[u]);
                if (!first) load_base8(p.old_view.k_base, b, jj[u], h, c8, p.H, D, p.N_cap, ko[u]);
            }
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                dot_n[u] = dot8(qn, kn[u]);
                dot_o[u] = first ? 0.f : dot8(qo, ko[u]);
            }
        }
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            float sn = dot_n[u], so = first ? 0.f : dot_o[u];
            if (!has_chunk) sn = so = 0.f;
            sn = group16_sum(sn);
            so = group16_sum(so);
            const int t = t0 + u * kGroups + grp;
            if (t < cn && gl == 0) {
                tau[t] = sn * p.scale;
                sig[t] = so * p.scale;
            }
        }
    }
    __syncthreads();

    // row statistics of the chunk, then of the row (merged over the cluster)
    const float zo = first ? 0.f : __ldg(p.z + bh * p.n_state + slot);
    float mx = -INFINITY;
    for (int t = threadIdx.x; t < cn; t += kThreads) mx = fmaxf(mx, tau[t]);
    mx = block_reduce<true>(mx, red);
    float ls = 0.f, ms = 0.f;
    for (int t = threadIdx.x; t < cn; t += kThreads) {
        ls += mx > -INFINITY ? expf(tau[t] - mx) : 0.f;
        if (!first) ms += expf(sig[t] - zo);
    }
    ls = block_reduce<false>(ls, red);
    ms = first ? 0.f : block_reduce<false>(ms, red);
    if (ncta > 1) {
        if (threadIdx.x < ncta) {
            cl_st_f32(cl_map(&stats[rank * 3 + 0], threadIdx.x), mx);
            cl_st_f32(cl_map(&stats[rank * 3 + 1], threadIdx.x), ls);
            cl_st_f32(cl_map(&stats[rank * 3 + 2], threadIdx.x), ms);
        }
        cl_sync();
    } else {
        if (threadIdx.x == 0) {
            stats[0] = mx;
            stats[1] = ls;
            stats[2] = ms;
        }
        __syncthreads();
    }
    float gmx = -INFINITY, gls = 0.f, m = 0.f;
    for (uint32_t r = 0; r < ncta; ++r) gmx = fmaxf(gmx, stats[r * 3]);
    for (uint32_t r = 0; r < ncta; ++r) {
        if (stats[r * 3] > -INFINITY) gls += stats[r * 3 + 1] * expf(stats[r * 3] - gmx);
        m += stats[r * 3 + 2];
    }
    if (first) m = 1.f;
    const float lam = gmx + logf(gls);
    if (!first && !(m >= FLT_MIN)) return;   // old mass underflowed: keep the row's state (the whole cluster)

    // pass 2: u = sum p v_old, w = sum a v_new over the chunk, column mass
    float u_[8] = {0, 0, 0, 0, 0, 0, 0, 0}, w[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    float *cb = p.c + bh * p.n_keys;
    for (int t0 = 0; t0 < cn; t0 += kGroups * kU) {
        int jj[kU], tt[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int t = t0 + u * kGroups + grp;
            tt[u] = t < cn ? t : 0;
            jj[u] = key_at(tt[u]);
        }
        // probabilities of the step's keys: new (a) and old (pj); keys past the end add nothing
        float a[kU], pj[kU];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
            const int t = t0 + u * kGroups + grp;
            const bool valid = t < cn;
            a[u] = valid ? expf(tau[t] - lam) : 0.f;
            pj[u] = valid && !first ? expf(sig[t] - zo) : 0.f;
        }
        // u += pj v_old and w += a v_new with the bf16-rounded reconstructions, key by key
        auto acc8 = [&](float (&dst)[8], float coef, const float (&r)[8]) {
            float v8[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) v8[e] = r[e];
            round_bf16x8(v8);
#pragma unroll
            for (int e = 0; e < 8; ++e) dst[e] = fmaf(coef, v8[e], dst[e]);
        };
        if constexpr (shared_base) {
            visit_rec<D>(p.old_view, p.new_view, true, b, jj, tt, ents, p.chunk, h, c8, p.H, p.N_cap, p.R_cap,
                         [&](int u, const float (&r)[8]) {
                             if (t0 + u * kGroups + grp < cn) acc8(u_, pj[u], r);
                         },
                         [&](int u, const float (&r)[8]) {
                             if (t0 + u * kGroups + grp < cn) acc8(w, a[u], r);
                         });
        } else {   // dense layers: every key's rows are requested before any is used
            float vn[kU][8], vo[kU][8];
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                load_base8(p.new_view.v_base, b, jj[u], h, c8, p.H, D, p.N_cap, vn[u]);
                if (!first) load_base8(p.old_view.v_base, b, jj[u], h, c8, p.H, D, p.N_cap, vo[u]);
            }
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                if (t0 + u * kGroups + grp >= cn) continue;
                acc8(w, a[u], vn[u]);
                if (!first) acc8(u_, pj[u], vo[u]);
            }
        }
#pragma unroll
        for (int u = 0; u < kU; ++u)
            if (t0 + u * kGroups + grp < cn && gl == 0) atomicAdd(cb + jj[u], m * a[u] - pj[u]);
    }
    if (has_chunk) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            acc[grp * D + c8 * 8 + e] = u_[e];
            acc[(kGroups + grp) * D + c8 * 8 + e] = w[e];
        }
    }
    __syncthreads();
    // the chunk's u and w, summed over the groups, into rank 0's cluster sums
    for (int x = threadIdx.x; x < D; x += kThreads) {
        float us = 0.f, ws = 0.f;
        for (int g = 0; g < kGroups; ++g) {
            us += acc[g * D + x];
            ws += acc[(kGroups + g) * D + x];
        }
        if (ncta > 1) {
            cl_red_add_f32(cl_map(&uw[x], 0), us);
            cl_red_add_f32(cl_map(&uw[D + x], 0), ws);
        } else {
            uw[x] = us;
            uw[D + x] = ws;
        }
    }
    if (ncta > 1) cl_sync(); else __syncthreads();
    if (rank != 0) return;
    for (int x = threadIdx.x; x < D; x += kThreads) {
        const float prev = first ? 0.f : p.o[srow + x];
        p.o[srow + x] = prev - uw[x] + m * uw[D + x];
        p.q_hat[srow + x] = p.q[srow + x];
    }
    if (threadIdx.x == 0) p.z[bh * p.n_state + slot] = lam - logf(m);
}

template <int D>
cudaError_t launch_d(const DecodeAttnParams &q, cudaStream_t s) {
    const int nk_max = q.mode == FLASHLOOP_ATTN_LAZY ? q.K : q.n_keys;
    const int ncta = max(1, min(kMaxCluster, (nk_max + kKeysPerCta - 1) / kKeysPerCta));
    const int chunk = (nk_max + ncta - 1) / ncta;
    const int n_ent = q.mode == FLASHLOOP_ATTN_LAZY ? q.new_view.n_layers * chunk : 0;   // delta entries
    const size_t smem =
        (size_t)(3 * chunk + kThreads / 32 + 2 * kGroups * D + kMaxCluster * 3 + 2 * D + n_ent) * sizeof(float);
    if (smem > 220 * 1024) return cudaErrorInvalidValue;
    static std::once_flag once[kMaxDevices];
    static cudaError_t attr_res[kMaxDevices];
    const cudaError_t ea = once_per_device(once, attr_res, [] {
        cudaError_t e = cudaFuncSetAttribute(decode_attention_kernel<D, FLASHLOOP_ATTN_FIRST_DENSE>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, 220 * 1024);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(decode_attention_kernel<D, FLASHLOOP_ATTN_DENSE>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, 220 * 1024);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(decode_attention_kernel<D, FLASHLOOP_ATTN_LAZY>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, 220 * 1024);
        return e;
    });
    if (ea != cudaSuccess) return ea;
    DecKParams p;
    p.mode = q.mode;
    p.H = q.H;
    p.n_keys = q.n_keys;
    p.n_state = q.n_state;
    p.R = q.R;
    p.K = q.K;
    p.N_cap = q.N_cap;
    p.R_cap = q.R_cap;
    p.chunk = chunk;
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
    p.scale = 1.0f / sqrtf((float)D);
    const long long grid = (long long)q.B * q.H * q.R * ncta;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)ncta;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e;
    {
        KernelTimer kt("decode_attention", s);
        e = q.mode == FLASHLOOP_ATTN_FIRST_DENSE
                ? cudaLaunchKernelEx(&cfg, decode_attention_kernel<D, FLASHLOOP_ATTN_FIRST_DENSE>, p)
            : q.mode == FLASHLOOP_ATTN_DENSE ? cudaLaunchKernelEx(&cfg, decode_attention_kernel<D, FLASHLOOP_ATTN_DENSE>, p)
                                             : cudaLaunchKernelEx(&cfg, decode_attention_kernel<D, FLASHLOOP_ATTN_LAZY>, p);
    }
    return e != cudaSuccess ? e : cudaGetLastError();
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

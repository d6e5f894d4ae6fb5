// kvcache.cu -- dense gathers and the base + int4-delta KV cache.
//
// rit.work page "FlashLoop: Fast and Memory-Efficient Looped Transformers via
// Lazy Updates":
//   section "Later loops change only part of the state": neighbouring KV sets
//   differ less than whole states, so store a base plus small deltas;
//   section "FlashLoop combines three kinds of saving": the cache is a
//   compressed base plus a sequence of compressed deltas, a low-bit delta is
//   written for active tokens and none for inactive ones (4-bit in the main
//   experiments), and selected data is gathered into dense buffers.
//
// Arithmetic that must agree bit for bit with any other implementation of
// the same definition is written with explicit IEEE intrinsics: fp32
// reconstruction adds scale*code layer by layer in ascending order, the
// delta is one fp32 subtraction, scale = fp16_rne(amax / 7) with an IEEE
// divide, and code = rint_even(delta / scale) clamped to [-7, 7]. Codes
// become floats, and quotients codes, through exact fp32 bit tricks rather
// than the conversion unit.
#include "common.cuh"

namespace fl {
namespace {

constexpr int kCopyWarps = 8;

// dst[b, r, :] = src[b, idx[b, r], :]; one warp per row, 16-byte vectors.
__global__ void __launch_bounds__(kCopyWarps * 32)
gather_rows_kernel(const uint4 *__restrict__ src, int N, int vecs, const int32_t *__restrict__ idx,
                   int R, long long rows, uint4 *__restrict__ dst) {
    const long long row = (long long)blockIdx.x * kCopyWarps + threadIdx.x / 32;
    if (row >= rows) return;
    const long long b = row / R;
    const int i = __ldg(idx + row);
    if ((unsigned)i >= (unsigned)N) return;   // outside the sequence: the row is not gathered
    const uint4 *s = src + (b * N + i) * (long long)vecs;
    uint4 *d = dst + row * (long long)vecs;
    for (int v = threadIdx.x & 31; v < vecs; v += 32) d[v] = ldg_nc_v4(s + v);
}

// dst[b, idx[b, r], :] = src[b, idx[b, r], :]; one warp per row, 16-byte vectors.
__global__ void __launch_bounds__(kCopyWarps * 32)
copy_rows_kernel(const uint4 *__restrict__ src, int N, int vecs, const int32_t *__restrict__ idx, int R,
                 long long rows, uint4 *__restrict__ dst) {
    pdl_wait();
    pdl_trigger();
    const long long row = (long long)blockIdx.x * kCopyWarps + threadIdx.x / 32;
    if (row >= rows) return;
    const long long b = row / R;
    const int i = __ldg(idx + row);
    if ((unsigned)i >= (unsigned)N) return;   // outside the sequence: nothing to copy
    const long long off = (b * N + i) * (long long)vecs;
    for (int v = threadIdx.x & 31; v < vecs; v += 32) dst[off + v] = __ldg(src + off + v);
}

// dst[b * R + r, :] = bf16_rne(src[b, idx[b, r], :]) (idx NULL: src row r): one
// warp per row, 8 fp32 in, 8 bf16 (16 bytes) out per lane step.
__global__ void __launch_bounds__(kCopyWarps * 32)
gather_f32_bf16_kernel(const float *__restrict__ src, int N, int elems, const int32_t *__restrict__ idx, int R,
                       long long rows, uint16_t *__restrict__ dst) {
    pdl_wait();
    pdl_trigger();
    const long long row = (long long)blockIdx.x * kCopyWarps + threadIdx.x / 32;
    if (row >= rows) return;
    const long long b = row / R;
    const int i = idx ? __ldg(idx + row) : (int)(row - b * R);
    if ((unsigned)i >= (unsigned)N) return;   // outside the sequence: the row is not gathered
    const float4 *s = reinterpret_cast<const float4 *>(src + (b * N + i) * (long long)elems);
    uint4 *d = reinterpret_cast<uint4 *>(dst + row * (long long)elems);
    for (int v = threadIdx.x & 31; v < elems / 8; v += 32) {
        const float4 a = __ldg(s + 2 * v), c = __ldg(s + 2 * v + 1);
        d[v] = make_uint4(pack_bf16x2_rn(a.x, a.y), pack_bf16x2_rn(a.z, a.w), pack_bf16x2_rn(c.x, c.y),
                          pack_bf16x2_rn(c.z, c.w));
    }
}

// dst[b, pos0 + r, :] = src[b, r, :] for r < n_rows.
__global__ void __launch_bounds__(kCopyWarps * 32)
store_rows_kernel(const uint4 *__restrict__ src, int n_rows, int vecs, uint4 *__restrict__ dst,
                  int dst_rows, int pos0, long long rows) {
    const long long row = (long long)blockIdx.x * kCopyWarps + threadIdx.x / 32;
    if (row >= rows) return;
    const long long b = row / n_rows, r = row % n_rows;
    const uint4 *s = src + row * (long long)vecs;
    uint4 *d = dst + (b * dst_rows + pos0 + r) * (long long)vecs;
    for (int v = threadIdx.x & 31; v < vecs; v += 32) d[v] = ldg_nc_v4(s + v);
}

// One thread per (sequence, entry, head, 32-element quantisation group): the
// group's four 8-element chunks of the loop-l row and of the base row are
// loaded together, each earlier delta layer costs one slot lookup, one codes
// load (4 * BITS bytes) and one scale load for the whole group, and the
// group's 32 codes go out as BITS 32-bit words. blockIdx.y: 0 = K, 1 = V.
// Four 256-thread blocks per SM (64 registers): the kernel waits on chains of
// dependent gathers (one per earlier delta layer), so resident warps matter more
// than a few spilled registers.
template <int BITS>
__global__ void __launch_bounds__(256, 4)
delta_append_kernel(DeltaView view, const uint16_t *__restrict__ k_l, const uint16_t *__restrict__ v_l,
                    int rows_are_tokens, int src_rows, const int32_t *__restrict__ active, int R, int at,
                    int H, int d, int N_cap, int R_cap, long long total, int32_t *__restrict__ out_idx,
                    int32_t *__restrict__ out_slot, uint8_t *__restrict__ k_codes,
                    uint16_t *__restrict__ k_scales, uint8_t *__restrict__ v_codes,
                    uint16_t *__restrict__ v_scales, const int32_t *__restrict__ seq_exit) {
    pdl_wait();
    pdl_trigger();
    // 32-bit index arithmetic (the launcher checks that total fits): 64-bit
    // division and remainder are long instruction sequences
    const uint32_t t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= (uint32_t)total) return;
    const bool is_v = blockIdx.y == 1;
    const uint32_t gpr = (uint32_t)d / 32u;   // quantisation groups per (row, head)
    const uint32_t rest = t / gpr;
    const int g = (int)(t - rest * gpr);
    const uint32_t be32 = rest / (uint32_t)H;   // b * R + e
    const int h = (int)(rest - be32 * (uint32_t)H);
    const uint32_t b32 = be32 / (uint32_t)R;
    const int e = (int)(be32 - b32 * (uint32_t)R);
    const long long be = be32, b = b32;
    const int i = __ldg(active + be);
    const long long src_row = rows_are_tokens ? (long long)i : (long long)e;

    constexpr int RB = BITS * 4;              // bytes of one group's codes
    constexpr float QMAX = (float)((1 << (BITS - 1)) - 1);
    const uint16_t *x_l = (is_v ? v_l : k_l) + ((b * src_rows + src_row) * H + h) * (long long)d + g * 32;
    uint4 xv[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) xv[c] = ldg_nc_v4(x_l + c * 8);
    float x[32], rec[32];
#pragma unroll
    for (int c = 0; c < 4; ++c) load_base8(view, is_v, b, i, h, 4 * g + c, H, d, N_cap, rec + 8 * c);
#pragma unroll
    for (int c = 0; c < 4; ++c) unpack_bf16x8(xv[c], x + 8 * c);
    // the previous loop's reconstruction: base plus each earlier layer's deltas, in order
    for (int m = 0; m < view.n_layers; ++m) {
        const int en = __ldg(view.slot[m] + b * N_cap + i);
        if (en < 0) continue;
        const long long ent = (b * R_cap + en) * H + h;
        const uint8_t *codes = is_v ? view.v_codes[m] : view.k_codes[m];
        const uint16_t *scales = is_v ? view.v_scales[m] : view.k_scales[m];
        const uint8_t *crow = codes + ent * (d * BITS / 8);
        uint32_t w[4];
        if constexpr (BITS == 4) {
            const uint4 w4 = __ldg(reinterpret_cast<const uint4 *>(crow + g * RB));
            w[0] = w4.x; w[1] = w4.y; w[2] = w4.z; w[3] = w4.w;
        } else {
#pragma unroll
            for (int c = 0; c < 4; ++c) w[c] = load_codes8(crow, 4 * g + c, BITS);
        }
        const float sc = __half2float(__ushort_as_half(__ldg(scales + ent * (d / 32) + g)));
#pragma unroll
        for (int c = 0; c < 4; ++c) dequant_add8(rec + 8 * c, w[c], sc);
    }

    float amax = 0.f;
#pragma unroll
    for (int u = 0; u < 32; ++u) {
        x[u] = __fsub_rn(x[u], rec[u]);   // the delta
        amax = fmaxf(amax, fabsf(x[u]));
    }
    // a sequence that has stopped looping keeps its K/V: its entries are zero deltas
    if (seq_exit && __ldg(seq_exit + b)) amax = 0.f;
    const __half sh = __float2half_rn(__fdiv_rn(amax, QMAX));   // the scale is exact: fp16(fp32(amax / qmax))
    const float s = __half2float(sh);
    // code = rint(delta / scale): the quotient is taken as delta * (1 / scale), within
    // about one ulp of the divided one, so a code can only differ where the quotient
    // lies within ~1e-6 of a rounding boundary (n + 1/2)
    const float inv = s > 0.f ? __frcp_rn(s) : 0.f;
    // the group's codes as a little-endian bit string of BITS-bit fields
    uint32_t packed[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int k = 0; k < 32; ++k) {
        // rint is monotone and fixes +-qmax, so clamping before rounding gives the
        // same integer; adding 1.5 * 2^23 rounds the clamped quotient to an
        // integer (ties to even) in the low mantissa bits, whose low BITS bits are
        // then the code in two's complement
        const float r = fminf(QMAX, fmaxf(-QMAX, __fmul_rn(x[k], inv)));
        const uint32_t code = __float_as_uint(__fadd_rn(r, 12582912.0f)) & ((1u << BITS) - 1u);
        const int bit = BITS * k;
        packed[bit >> 5] |= code << (bit & 31);
        if ((bit & 31) + BITS > 32) packed[(bit >> 5) + 1] |= code >> (32 - (bit & 31));
    }
    const long long ent = (b * R_cap + at + e) * H + h;
    uint8_t *codes = is_v ? v_codes : k_codes;
    uint16_t *scales = is_v ? v_scales : k_scales;
    uint32_t *dst = reinterpret_cast<uint32_t *>(codes + ent * (d * BITS / 8) + g * RB);
    if constexpr (BITS == 4) {
        *reinterpret_cast<uint4 *>(dst) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    } else {
#pragma unroll
        for (int w = 0; w < BITS; ++w) dst[w] = packed[w];
    }
    scales[ent * (d / 32) + g] = __half_as_ushort(sh);
    if (!is_v && h == 0 && g == 0) {
        out_idx[b * R_cap + at + e] = i;
        out_slot[b * N_cap + i] = at + e;
    }
}

// 32 fp32 values as bf16 (RNE), four 16-byte stores.
__device__ __forceinline__ void store_group_bf16(const float (&rec)[32], uint16_t *dst) {
    uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
    for (int c = 0; c < 4; ++c)
        d4[c] = make_uint4(pack_bf16x2_rn(rec[8 * c + 0], rec[8 * c + 1]), pack_bf16x2_rn(rec[8 * c + 2], rec[8 * c + 3]),
                           pack_bf16x2_rn(rec[8 * c + 4], rec[8 * c + 5]), pack_bf16x2_rn(rec[8 * c + 6], rec[8 * c + 7]));
}

// For each selected key j = key_idx[b,h,r]: reconstruction at the old loop
// (old_layers deltas) and at the new loop (new_layers deltas), bf16 RNE,
// written densely as [B, H, K, d]. A selected key of one head is one lane
// group of d/4 lanes (a warp for d = 128, 96; two keys per warp for d = 64):
// each lane owns one 16-byte chunk (8 elements) of the K or the V row, so
// base rows and the dense copies move as whole rows. The dependent loads run
// in two rounds per four delta layers: every layer's slot entry of the key at
// once, then every entry's codes and scale at once, then the fp32 sums in
// ascending layer order.
//
// The first n_count_blocks blocks instead count, for every (b, h) and row i,
// the keys that row sees: #{r : key_idx[b,h,r] <= row_pos[b,i]} (both lists
// ascending), by binary search over the head's key list staged in shared
// memory (or read from global memory when the list is longer than the stage).
constexpr int kRecThreads = 256;
constexpr int kCountSplit = 4;            // counting blocks per (b, h)
constexpr int kCountStageMax = 12288;     // keys staged in shared memory (48 KB)
constexpr int kLayerBatch = 4;            // delta layers whose loads are issued together
// Six blocks per SM (40 registers, no spills): the key gathers are latency-bound,
// and the extra resident warps take the 32K launch from 28.9 to 25.4 us.
template <int D>
__global__ void __launch_bounds__(kRecThreads, 6)
reconstruct_keys_kernel(DeltaView view, int old_layers, int new_layers, const int32_t *__restrict__ key_idx,
                        int H, int K, int N_cap, int R_cap, int n_keys_total,
                        uint16_t *__restrict__ k_old, uint16_t *__restrict__ v_old,
                        uint16_t *__restrict__ k_new, uint16_t *__restrict__ v_new,
                        const int32_t *__restrict__ row_pos, int R, int n_count_blocks,
                        int32_t *__restrict__ row_cnt) {
    pdl_wait();
    pdl_trigger();
    extern __shared__ int32_t s_keys[];
    if ((int)blockIdx.x < n_count_blocks) {
        const int bh = (int)blockIdx.x / kCountSplit, part = (int)blockIdx.x % kCountSplit;
        const int b = bh / H;
        const int32_t *S = key_idx + (long long)bh * K;
        const bool staged = K <= kCountStageMax;
        if (staged)
            for (int i = threadIdx.x; i < K; i += kRecThreads) s_keys[i] = __ldg(S + i);
        __syncthreads();
        const int per = (R + kCountSplit - 1) / kCountSplit;
        const int i0 = part * per, i1 = min(R, i0 + per);
        for (int i = i0 + (int)threadIdx.x; i < i1; i += kRecThreads) {
            const int x = __ldg(row_pos + (long long)b * R + i);
            int lo = 0, hi = K;
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if ((staged ? s_keys[mid] : __ldg(S + mid)) <= x) lo = mid + 1; else hi = mid;
            }
            row_cnt[(long long)bh * R + i] = lo;
        }
        return;
    }
    constexpr int d = D;
    constexpr int cpr = D / 8;              // 16-byte chunks per row of one tensor
    constexpr int lpk = 2 * cpr;            // lanes per key: K chunks, then V chunks
    constexpr int kpw = 32 / lpk;           // keys per warp
    const int lane = threadIdx.x & 31, sub = lane / lpk, c = lane - sub * lpk;
    // 32-bit index arithmetic (the launcher checks that the key count fits):
    // 64-bit division is a long instruction sequence
    const uint32_t key = ((uint32_t)(blockIdx.x - n_count_blocks) * (kRecThreads / 32) + threadIdx.x / 32) * kpw + sub;
    if (sub >= kpw || key >= (uint32_t)n_keys_total) return;
    const bool is_v = c >= cpr;
    const int ch = is_v ? c - cpr : c;      // elements 8 ch .. 8 ch + 7, quantisation group ch / 4
    const uint32_t bh = key / (uint32_t)K;
    const uint32_t b32 = bh / (uint32_t)H;
    const int h = (int)(bh - b32 * (uint32_t)H);
    const long long b = b32;
    const int j = __ldg(key_idx + key);
    const long long tok = b * N_cap + j;
    float rec[8];
    load_base8(view, is_v, b, j, h, ch, H, d, N_cap, rec);
    uint16_t *o_old = (is_v ? v_old : k_old) + (long long)key * d + ch * 8;
    uint16_t *o_new = (is_v ? v_new : k_new) + (long long)key * d + ch * 8;
    auto store8 = [&](uint16_t *dst) {
        *reinterpret_cast<uint4 *>(dst) = make_uint4(pack_bf16x2_rn(rec[0], rec[1]), pack_bf16x2_rn(rec[2], rec[3]),
                                                     pack_bf16x2_rn(rec[4], rec[5]), pack_bf16x2_rn(rec[6], rec[7]));
    };
    for (int m0 = 0; m0 < new_layers; m0 += kLayerBatch) {
        int en[kLayerBatch];
#pragma unroll
        for (int u = 0; u < kLayerBatch; ++u) en[u] = m0 + u < new_layers ? __ldg(view.slot[m0 + u] + tok) : -1;
        uint32_t w[kLayerBatch];
        float sc[kLayerBatch];
#pragma unroll
        for (int u = 0; u < kLayerBatch; ++u) {
            w[u] = 0u;
            sc[u] = 0.f;
            if (en[u] >= 0) {
                const int m = m0 + u;
                const long long ent = (b * R_cap + en[u]) * H + h;
                const uint8_t *codes = is_v ? view.v_codes[m] : view.k_codes[m];
                const uint16_t *scales = is_v ? view.v_scales[m] : view.k_scales[m];
                w[u] = load_codes8(codes + ent * (d * view.code_bits / 8), ch, view.code_bits);
                sc[u] = __half2float(__ushort_as_half(__ldg(scales + ent * (d / 32) + ch / 4)));
            }
        }
#pragma unroll
        for (int u = 0; u < kLayerBatch; ++u) {
            if (m0 + u == old_layers) store8(o_old);
            if (en[u] >= 0) dequant_add8(rec, w[u], sc[u]);
        }
    }
    if (new_layers <= old_layers) store8(o_old);
    store8(o_new);
}

// The int8 base of stored rows: one thread per (sequence, row, head, 32-element
// group), the same quantiser as the deltas with qmax = 127.
__global__ void __launch_bounds__(256)
quantize_base_kernel(const uint16_t *__restrict__ src, int n_rows, int H, int d, int8_t *__restrict__ codes,
                     uint16_t *__restrict__ scales, int N_cap, int pos0, long long total) {
    pdl_wait();
    pdl_trigger();
    const long long t = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= total) return;
    const int gpr = d / 32;
    const long long rest = t / gpr;
    const int g = (int)(t - rest * gpr);
    const long long brh = rest;                 // (b * n_rows + r) * H + h
    const long long br = brh / H;
    const int h = (int)(brh - br * H);
    const long long b = br / n_rows;
    const int r = (int)(br - b * n_rows);
    const uint16_t *x = src + brh * d + g * 32;
    float v[32];
#pragma unroll
    for (int c = 0; c < 4; ++c) unpack_bf16x8(ldg_nc_v4(x + 8 * c), v + 8 * c);
    float amax = 0.f;
#pragma unroll
    for (int k = 0; k < 32; ++k) amax = fmaxf(amax, fabsf(v[k]));
    const __half sh = __float2half_rn(__fdiv_rn(amax, 127.0f));
    const float s = __half2float(sh);
    const float inv = s > 0.f ? __frcp_rn(s) : 0.f;
    uint32_t packed[8];
#pragma unroll
    for (int w = 0; w < 8; ++w) {
        packed[w] = 0u;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float q = fminf(127.f, fmaxf(-127.f, __fmul_rn(v[4 * w + k], inv)));
            packed[w] |= (__float_as_uint(__fadd_rn(q, 12582912.0f)) & 0xFFu) << (8 * k);
        }
    }
    const long long drow = (b * N_cap + pos0 + r) * H + h;
    uint4 *dst = reinterpret_cast<uint4 *>(codes + drow * d + g * 32);
    dst[0] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    dst[1] = make_uint4(packed[4], packed[5], packed[6], packed[7]);
    scales[drow * (d / 32) + g] = __half_as_ushort(sh);
}

}  // namespace

cudaError_t launch_quantize_base(const uint16_t *src, int B, int n_rows, int H, int d, int8_t *codes,
                                 uint16_t *scales, int N_cap, int pos0, cudaStream_t s) {
    const long long total = (long long)B * n_rows * H * (d / 32);
    if (total == 0) return cudaSuccess;
    {
        KernelTimer kt("quantize_base", s);
        const cudaError_t e = launch_pdl(quantize_base_kernel, dim3(ceil_div(total, 256)), dim3(256), 0, s, src, n_rows,
                                         H, d, codes, scales, N_cap, pos0, total);
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

cudaError_t launch_gather_rows(const void *src, int B, int N, int row_bytes, const int32_t *idx, int R,
                               void *dst, cudaStream_t s) {
    const long long rows = (long long)B * R;
    if (rows == 0) return cudaSuccess;
    {
        KernelTimer kt("gather", s);
        gather_rows_kernel<<<ceil_div(rows, kCopyWarps), kCopyWarps * 32, 0, s>>>(
        static_cast<const uint4 *>(src), N, row_bytes / 16, idx, R, rows, static_cast<uint4 *>(dst));
    }
    return cudaGetLastError();
}

cudaError_t launch_copy_rows(const void *src, int B, int N, int row_bytes, const int32_t *idx, int R, void *dst,
                             cudaStream_t s) {
    const long long rows = (long long)B * R;
    if (rows == 0) return cudaSuccess;
    {
        KernelTimer kt("copy_rows", s);
        const cudaError_t e = launch_pdl(copy_rows_kernel, dim3(ceil_div(rows, kCopyWarps)), dim3(kCopyWarps * 32), 0,
                                         s, static_cast<const uint4 *>(src), N, row_bytes / 16, idx, R, rows,
                                         static_cast<uint4 *>(dst));
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

cudaError_t launch_gather_f32_to_bf16(const float *src, int B, int N, int elems, const int32_t *idx, int R,
                                      uint16_t *dst, cudaStream_t s) {
    const long long rows = (long long)B * R;
    if (rows == 0) return cudaSuccess;
    {
        KernelTimer kt("gather_f32_bf16", s);
        const cudaError_t e = launch_pdl(gather_f32_bf16_kernel, dim3(ceil_div(rows, kCopyWarps)), dim3(kCopyWarps * 32),
                                         0, s, src, N, elems, idx, R, rows, dst);
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

cudaError_t launch_store_rows(const uint16_t *src, int B, int n_rows, int row_elems, uint16_t *dst,
                              int dst_rows, int pos0, cudaStream_t s) {
    const long long rows = (long long)B * n_rows;
    if (rows == 0) return cudaSuccess;
    {
        KernelTimer kt("store_rows", s);
        store_rows_kernel<<<ceil_div(rows, kCopyWarps), kCopyWarps * 32, 0, s>>>(
        reinterpret_cast<const uint4 *>(src), n_rows, row_elems / 8, reinterpret_cast<uint4 *>(dst), dst_rows,
        pos0, rows);
    }
    return cudaGetLastError();
}

cudaError_t launch_delta_append(const DeltaView &view, const uint16_t *k_l, const uint16_t *v_l,
                                int rows_are_tokens, int src_rows, const int32_t *active, int R, int at,
                                int B, int N_cap, int H, int d, int R_cap, int32_t *out_idx,
                                int32_t *out_slot, uint8_t *k_codes, uint16_t *k_scales, uint8_t *v_codes,
                                uint16_t *v_scales, cudaStream_t s, const int32_t *seq_exit) {
    const long long total = (long long)B * R * H * (d / 32);
    if (total == 0) return cudaSuccess;
    if (total > 0x7fffffffLL - 256) return cudaErrorInvalidValue;   // the kernel indexes in 32 bits
    dim3 grid(ceil_div(total, 256), 2);
    {
        KernelTimer kt("delta_append", s);
        auto kern = view.code_bits == 2 ? delta_append_kernel<2> : view.code_bits == 3 ? delta_append_kernel<3>
                                                                                         : delta_append_kernel<4>;
        const cudaError_t e = launch_pdl(kern, grid, dim3(256), 0, s, view, k_l, v_l,
                                         rows_are_tokens, src_rows, active, R, at, H, d, N_cap, R_cap, total,
                                         out_idx, out_slot, k_codes, k_scales, v_codes, v_scales, seq_exit);
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

cudaError_t launch_reconstruct_keys(const DeltaView &old_view, const DeltaView &new_view,
                                    const int32_t *key_idx, int B, int H, int K, int N_cap, int d,
                                    int R_cap, uint16_t *k_old, uint16_t *v_old, uint16_t *k_new,
                                    uint16_t *v_new, const int32_t *row_pos, int R, int32_t *row_cnt,
                                    cudaStream_t s) {
    const long long n_keys = (long long)B * H * K;
    const int n_count = row_cnt && R > 0 ? B * H * kCountSplit : 0;
    if (n_keys == 0 && n_count == 0) return cudaSuccess;
    if (n_keys > 0x7fffffffLL) return cudaErrorInvalidValue;
    if (d != 64 && d != 96 && d != 128) return cudaErrorInvalidValue;
    const int kpw = 32 / (2 * (d / 8));                         // keys per warp
    const long long keys_per_block = (long long)(kRecThreads / 32) * kpw;
    const int n_rec = ceil_div(n_keys, keys_per_block);
    const size_t smem = n_count && K <= kCountStageMax ? (size_t)K * sizeof(int32_t) : 0;
    auto kern = d == 64 ? reconstruct_keys_kernel<64> : d == 96 ? reconstruct_keys_kernel<96> : reconstruct_keys_kernel<128>;
    {
        KernelTimer kt("reconstruct_keys", s);
        const cudaError_t e = launch_pdl(kern, dim3(n_count + n_rec), dim3(kRecThreads), smem, s, new_view,
                                         old_view.n_layers, new_view.n_layers, key_idx, H, K, N_cap, R_cap,
                                         (int)n_keys, k_old, v_old, k_new, v_new, row_pos, R, n_count, row_cnt);
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

}  // namespace fl

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
    const uint4 *s = src + (b * N + i) * (long long)vecs;
    uint4 *d = dst + row * (long long)vecs;
    for (int v = threadIdx.x & 31; v < vecs; v += 32) d[v] = ldg_nc_v4(s + v);
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
// loaded together, each earlier delta layer costs one slot lookup, one
// 16-byte codes load and one scale load for the whole group, and the group's
// 32 codes (16 bytes) go out in one store. blockIdx.y: 0 = K, 1 = V.
// Four 256-thread blocks per SM (64 registers): the kernel waits on chains of
// dependent gathers (one per earlier delta layer), so resident warps matter more
// than a few spilled registers.
__global__ void __launch_bounds__(256, 4)
delta_append_kernel(DeltaView view, const uint16_t *__restrict__ k_l, const uint16_t *__restrict__ v_l,
                    int rows_are_tokens, int src_rows, const int32_t *__restrict__ active, int R, int at,
                    int H, int d, int N_cap, int R_cap, long long total, int32_t *__restrict__ out_idx,
                    int32_t *__restrict__ out_slot, uint8_t *__restrict__ k_codes,
                    uint16_t *__restrict__ k_scales, uint8_t *__restrict__ v_codes,
                    uint16_t *__restrict__ v_scales) {
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

    const uint16_t *x_l = (is_v ? v_l : k_l) + ((b * src_rows + src_row) * H + h) * (long long)d + g * 32;
    const uint16_t *base = (is_v ? view.v_base : view.k_base) + ((b * N_cap + i) * H + h) * (long long)d + g * 32;
    uint4 xv[4], bv[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) xv[c] = ldg_nc_v4(x_l + c * 8);
#pragma unroll
    for (int c = 0; c < 4; ++c) bv[c] = ldg_nc_v4(base + c * 8);
    float x[32], rec[32];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        unpack_bf16x8(xv[c], x + 8 * c);
        unpack_bf16x8(bv[c], rec + 8 * c);
    }
    // the previous loop's reconstruction: base plus each earlier layer's deltas, in order
    for (int m = 0; m < view.n_layers; ++m) {
        const int en = __ldg(view.slot[m] + b * N_cap + i);
        if (en < 0) continue;
        const long long ent = (b * R_cap + en) * H + h;
        const uint8_t *codes = is_v ? view.v_codes[m] : view.k_codes[m];
        const uint16_t *scales = is_v ? view.v_scales[m] : view.k_scales[m];
        const uint4 w4 = __ldg(reinterpret_cast<const uint4 *>(codes + ent * (d / 2) + g * 16));
        const float sc = __half2float(__ushort_as_half(__ldg(scales + ent * (d / 32) + g)));
        const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
        for (int c = 0; c < 4; ++c) dequant_add8(rec + 8 * c, w[c], sc);
    }

    float amax = 0.f;
#pragma unroll
    for (int u = 0; u < 32; ++u) {
        x[u] = __fsub_rn(x[u], rec[u]);   // the delta
        amax = fmaxf(amax, fabsf(x[u]));
    }
    const __half sh = __float2half_rn(__fdiv_rn(amax, 7.0f));   // the scale is exact: fp16(fp32(amax / 7))
    const float s = __half2float(sh);
    // code = rint(delta / scale): the quotient is taken as delta * (1 / scale), within
    // about one ulp of the divided one, so a code can only differ where the quotient
    // lies within ~1e-6 of a rounding boundary (n + 1/2)
    const float inv = s > 0.f ? __frcp_rn(s) : 0.f;
    uint32_t packed[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        packed[c] = 0u;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            // rint is monotone and fixes +-7, so clamping before rounding gives the
            // same integer; adding 1.5 * 2^23 rounds the clamped quotient to an
            // integer (ties to even) in the low mantissa bits, whose low nibble is
            // then the code in two's complement
            const float r = fminf(7.f, fmaxf(-7.f, __fmul_rn(x[8 * c + k], inv)));
            packed[c] |= (__float_as_uint(__fadd_rn(r, 12582912.0f)) & 0xFu) << (4 * k);
        }
    }
    const long long ent = (b * R_cap + at + e) * H + h;
    uint8_t *codes = is_v ? v_codes : k_codes;
    uint16_t *scales = is_v ? v_scales : k_scales;
    *reinterpret_cast<uint4 *>(codes + ent * (d / 2) + g * 16) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
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
// written densely as [B, H, K, d]. One thread per 32-element group of a
// selected row: its four base chunks load together and each delta layer is
// one slot lookup, one 16-byte codes load and one scale load for the group.
// blockIdx.y: 0 = K, 1 = V.
//
// The first n_count_blocks blocks of the K half instead count, for every
// (b, h) and row i, the keys that row sees: #{r : key_idx[b,h,r] <= row_pos[b,i]}
// (both lists ascending), by binary search over the head's key list.
constexpr int kRecThreads = 256;
__global__ void __launch_bounds__(kRecThreads)
reconstruct_keys_kernel(DeltaView view, int old_layers, int new_layers, const int32_t *__restrict__ key_idx,
                        int H, int K, int d, int N_cap, int R_cap, long long total,
                        uint16_t *__restrict__ k_old, uint16_t *__restrict__ v_old,
                        uint16_t *__restrict__ k_new, uint16_t *__restrict__ v_new,
                        const int32_t *__restrict__ row_pos, int R, long long count_total, int n_count_blocks,
                        int32_t *__restrict__ row_cnt) {
    pdl_wait();
    pdl_trigger();
    if ((int)blockIdx.x < n_count_blocks) {
        if (blockIdx.y != 0) return;
        const uint32_t t = blockIdx.x * kRecThreads + threadIdx.x;
        if (t >= (uint32_t)count_total) return;
        const uint32_t bh32 = t / (uint32_t)R;
        const int i = (int)(t - bh32 * (uint32_t)R);
        const long long bh = bh32, b = bh32 / (uint32_t)H;
        const int32_t *S = key_idx + bh * K;
        const int x = __ldg(row_pos + b * R + i);
        int lo = 0, hi = K;
        while (lo < hi) {
            const int mid = (lo + hi) >> 1;
            if (__ldg(S + mid) <= x) lo = mid + 1; else hi = mid;
        }
        row_cnt[bh * R + i] = lo;
        return;
    }
    const uint32_t t = (blockIdx.x - (uint32_t)n_count_blocks) * kRecThreads + threadIdx.x;   // 32-bit, as above
    if (t >= (uint32_t)total) return;
    const bool is_v = blockIdx.y == 1;
    const uint32_t gpr = (uint32_t)d / 32u;
    const uint32_t bhr32 = t / gpr;          // (b * H + h) * K + r
    const int g = (int)(t - bhr32 * gpr);
    const uint32_t bh32 = bhr32 / (uint32_t)K;
    const uint32_t b32 = bh32 / (uint32_t)H;
    const int h = (int)(bh32 - b32 * (uint32_t)H);
    const long long bhr = bhr32, b = b32;
    const int j = __ldg(key_idx + bhr);
    const uint16_t *base = (is_v ? view.v_base : view.k_base) + ((b * N_cap + j) * H + h) * (long long)d + g * 32;
    uint4 bv[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) bv[c] = ldg_nc_v4(base + c * 8);
    float rec[32];
#pragma unroll
    for (int c = 0; c < 4; ++c) unpack_bf16x8(bv[c], rec + 8 * c);
    for (int m = 0; m < new_layers; ++m) {
        if (m == old_layers) store_group_bf16(rec, (is_v ? v_old : k_old) + bhr * d + g * 32);
        const int en = __ldg(view.slot[m] + b * N_cap + j);
        if (en < 0) continue;
        const long long ent = (b * R_cap + en) * H + h;
        const uint8_t *codes = is_v ? view.v_codes[m] : view.k_codes[m];
        const uint16_t *scales = is_v ? view.v_scales[m] : view.k_scales[m];
        const uint4 w4 = __ldg(reinterpret_cast<const uint4 *>(codes + ent * (d / 2) + g * 16));
        const float sc = __half2float(__ushort_as_half(__ldg(scales + ent * (d / 32) + g)));
        const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
        for (int c = 0; c < 4; ++c) dequant_add8(rec + 8 * c, w[c], sc);
    }
    if (new_layers <= old_layers) store_group_bf16(rec, (is_v ? v_old : k_old) + bhr * d + g * 32);
    store_group_bf16(rec, (is_v ? v_new : k_new) + bhr * d + g * 32);
}

}  // namespace

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
                                uint16_t *v_scales, cudaStream_t s) {
    const long long total = (long long)B * R * H * (d / 32);
    if (total == 0) return cudaSuccess;
    if (total > 0x7fffffffLL - 256) return cudaErrorInvalidValue;   // the kernel indexes in 32 bits
    dim3 grid(ceil_div(total, 256), 2);
    {
        KernelTimer kt("delta_append", s);
        const cudaError_t e = launch_pdl(delta_append_kernel, grid, dim3(256), 0, s, view, k_l, v_l,
                                         rows_are_tokens, src_rows, active, R, at, H, d, N_cap, R_cap, total,
                                         out_idx, out_slot, k_codes, k_scales, v_codes, v_scales);
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

cudaError_t launch_reconstruct_keys(const DeltaView &old_view, const DeltaView &new_view,
                                    const int32_t *key_idx, int B, int H, int K, int N_cap, int d,
                                    int R_cap, uint16_t *k_old, uint16_t *v_old, uint16_t *k_new,
                                    uint16_t *v_new, const int32_t *row_pos, int R, int32_t *row_cnt,
                                    cudaStream_t s) {
    const long long total = (long long)B * H * K * (d / 32);
    const long long count_total = row_cnt ? (long long)B * H * R : 0;
    const int n_count = ceil_div(count_total, kRecThreads);
    if (total == 0 && n_count == 0) return cudaSuccess;
    if (total + count_total > 0x7fffffffLL - 2 * kRecThreads) return cudaErrorInvalidValue;   // 32-bit indexing
    dim3 grid(n_count + ceil_div(total, kRecThreads), 2);
    {
        KernelTimer kt("reconstruct_keys", s);
        const cudaError_t e = launch_pdl(reconstruct_keys_kernel, grid, dim3(kRecThreads), 0, s, new_view,
                                         old_view.n_layers, new_view.n_layers, key_idx, H, K, d, N_cap, R_cap,
                                         total, k_old, v_old, k_new, v_new, row_pos, R, count_total, n_count,
                                         row_cnt);
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

}  // namespace fl

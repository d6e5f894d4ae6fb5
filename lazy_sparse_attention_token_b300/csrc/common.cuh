// common.cuh -- helpers shared by the FlashLoop CUDA sources (sm_103a only).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "device_once.h"
#include "flashloop.h"

#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ != 1030)
#error "this library is written for sm_103a only"
#endif

namespace fl {

// Kernel attributes belong to one device's context: `set` runs once per
// device (the current one) and its cudaError_t is returned on every later
// call from that device (device_once.h).
template <class Set>
inline cudaError_t once_per_device(std::once_flag (&once)[kMaxDevices], cudaError_t (&res)[kMaxDevices], Set &&set) {
    return once_per_device_with(once, res, [](int *dev) { return cudaGetDevice(dev); }, cudaErrorInvalidDevice,
                                static_cast<Set &&>(set));
}

// ---- host bookkeeping (api.cu) -------------------------------------------
void note_launch(int n = 1);

// Brackets one kernel launch with CUDA events on its stream while timing is
// enabled (flashloop_timing_enable); counts the launch either way.
class KernelTimer {
  public:
    KernelTimer(const char *name, cudaStream_t s);
    ~KernelTimer();
  private:
    int rec_;
    cudaStream_t s_;
};
flashloop_status_t set_error(flashloop_status_t st, const char *fmt, ...);
flashloop_status_t check_launch(const char *what);
flashloop_status_t check_device();
flashloop_status_t cuda_fail(cudaError_t e, const char *what);

constexpr int kMaxLoops = FLASHLOOP_MAX_LOOPS;

// Device view of the delta layers needed to reconstruct one loop.
struct DeltaView {
    const uint16_t *k_base;            // [B, N_cap, H, d] bf16, or NULL for an int8 base
    const uint16_t *v_base;
    const int8_t *k_base_codes;        // int8 base [B, N_cap, H, d] (when k_base is NULL)
    const int8_t *v_base_codes;
    const uint16_t *k_base_scales;     // [B, N_cap, H, d/32] fp16
    const uint16_t *v_base_scales;
    int code_bits;                     // width of the delta codes: 2, 3 or 4
    int n_layers;                      // delta layers applied, ascending
    const int32_t *slot[kMaxLoops];    // [B, N_cap]
    const uint8_t *k_codes[kMaxLoops]; // [B, R_cap, H, d * code_bits / 8]
    const uint16_t *k_scales[kMaxLoops];
    const uint8_t *v_codes[kMaxLoops];
    const uint16_t *v_scales[kMaxLoops];
};

// ---- launchers (one per kernel family) -----------------------------------
// select.cu
cudaError_t launch_token_scores(const uint16_t *h_prev, const uint16_t *h_cur, int B, int N, int D,
                                float *scores, cudaStream_t s);
// `name` labels the launch in the per-kernel timing ("topk_tokens", "topk_keys").
// norm_n > 0 ranks column i by vals[i] / (norm_n - i) (requires n <= norm_n).
// seq_exit != NULL sets seq_exit[row] = 1 when the row's largest value is below exit_thr.
cudaError_t launch_topk_rows(const float *vals, int rows, int n, int k, int32_t *out, cudaStream_t s,
                             const char *name, int norm_n = 0, float exit_thr = 0.f, int32_t *seq_exit = nullptr);
// kvcache.cu
cudaError_t launch_gather_rows(const void *src, int B, int N, int row_bytes, const int32_t *idx, int R,
                               void *dst, cudaStream_t s);
cudaError_t launch_store_rows(const uint16_t *src, int B, int n_rows, int row_elems, uint16_t *dst,
                              int dst_rows, int pos0, cudaStream_t s);
// int8 base of rows src [B, n_rows, H, d] bf16 at positions pos0.. of codes
// [B, N_cap, H, d] and scales [B, N_cap, H, d/32]: one fp16 scale per 32
// elements, scale = fp16_rne(amax / 127), code = rint_even(x / scale) in [-127, 127].
cudaError_t launch_quantize_base(const uint16_t *src, int B, int n_rows, int H, int d, int8_t *codes,
                                 uint16_t *scales, int N_cap, int pos0, cudaStream_t s);
cudaError_t launch_delta_append(const DeltaView &view, const uint16_t *k_l, const uint16_t *v_l,
                                int rows_are_tokens, int src_rows, const int32_t *active, int R, int at,
                                int B, int N_cap, int H, int d, int R_cap, int32_t *out_idx,
                                int32_t *out_slot, uint8_t *k_codes, uint16_t *k_scales, uint8_t *v_codes,
                                uint16_t *v_scales, cudaStream_t s, const int32_t *seq_exit = nullptr);
// Reconstruction of the selected keys at the old and the new loop into
// [B, H, K, d]; with row_cnt set, the same launch also counts the keys each of
// the R rows at row_pos sees, into row_cnt [B, H, R].
cudaError_t launch_reconstruct_keys(const DeltaView &old_view, const DeltaView &new_view,
                                    const int32_t *key_idx, int B, int H, int K, int N_cap, int d,
                                    int R_cap, uint16_t *k_old, uint16_t *v_old, uint16_t *k_new,
                                    uint16_t *v_new, const int32_t *row_pos, int R, int32_t *row_cnt,
                                    cudaStream_t s);
// attn_tc.cu (tensor-core prefill / dense attention)
struct TcAttnParams {
    int mode;            // flashloop_attn_mode_t
    int B, H, d;
    int n_keys;          // key positions
    int n_state;         // state rows per sequence
    int R;               // rows per sequence
    const int32_t *row_pos;   // [B,R] or NULL (dense: row = key position)
    int K;               // key columns per (b,h) (dense: n_keys)
    const int32_t *key_idx;   // [B,H,K] or NULL (dense)
    int32_t *row_cnt;         // lazy: keys each row sees [B,H,R], filled before the launch
    const uint16_t *q;
    uint16_t *q_hat;
    float *o, *z, *c;
    // key/value sources: lazy = dense [B,H,K,d] buffers; dense = cache layers [B,N_cap,H,d]
    const uint16_t *k_old, *v_old, *k_new, *v_new;
    int kv_rows;         // rows of the source arrays per (b[,h]) (K or N_cap)
    const int32_t *seq_exit;  // [B] or NULL: sequences flagged 1 are left unchanged
};
cudaError_t launch_tc_attention(const TcAttnParams &p, cudaStream_t s);
int32_t tc_attention_read_error(bool clear);
int32_t tc_attention_set_wait_limit(unsigned long long ns);   // cudaError_t
// attn_decode.cu (few-row attention reading the cache directly)
struct DecodeAttnParams {
    int mode;
    int B, H, d;
    int n_keys, n_state, R;
    const int32_t *row_pos, *row_slot;
    int K;
    const int32_t *key_idx;   // NULL for dense modes (all keys)
    const uint16_t *q;
    uint16_t *q_hat;
    float *o, *z, *c;
    DeltaView old_view, new_view;   // reconstructions at loop-1 and loop
    int N_cap, R_cap;
    float *scratch;           // [B, H, R, K] x 2 logits
};
cudaError_t launch_decode_attention(const DecodeAttnParams &p, cudaStream_t s);
// gemm.cu: C = act(A W^T + residual), bf16 in and out, fp32 accumulation (see the file).
// c_rows (or NULL): A row m is written to row (m / rows_per_seq) * seq_rows + c_rows[m].
cudaError_t launch_gemm(const uint16_t *a, int M, int K, const uint16_t *wt, int N, const uint16_t *residual, int relu,
                        uint16_t *const *c, int n_split, long long c_ld, const int32_t *c_rows, int rows_per_seq,
                        int seq_rows, cudaStream_t s);
int32_t gemm_read_error(bool clear);
// kvcache.cu: dst[b, idx[b, r], :] = src[b, idx[b, r], :] for rows of row_bytes (% 16 == 0).
cudaError_t launch_copy_rows(const void *src, int B, int N, int row_bytes, const int32_t *idx, int R, void *dst,
                             cudaStream_t s);
// kvcache.cu: dst[b * R + r, :] = bf16_rne(src[b, idx[b, r], :]) for fp32 rows of `elems`
// (idx NULL: rows r of src in order, R = rows per sequence).
cudaError_t launch_gather_f32_to_bf16(const float *src, int B, int N, int elems, const int32_t *idx, int R,
                                      uint16_t *dst, cudaStream_t s);

// ---- device helpers -------------------------------------------------------
__device__ __forceinline__ float bf16_bits_to_f32(uint32_t h) { return __uint_as_float(h << 16); }

__device__ __forceinline__ void unpack_bf16x8(const uint4 &v, float *f) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

__device__ __forceinline__ uint32_t pack_bf16x2_rn(float lo, float hi) {
    __nv_bfloat162 t = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&t);
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// Order-preserving map of a finite fp32 to uint32 (larger float -> larger
// key); -0 is folded onto +0 so equal values compare equal.
__device__ __forceinline__ uint32_t f32_order_key(float f) {
    uint32_t u = __float_as_uint(f);
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Code t (bits [4t, 4t + 4) of w, two's complement in [-8, 7]) as an exact fp32.
// Offset by 8 the code is a nibble in [0, 15]; written into the low mantissa
// bits of 2^23 it gives the float 2^23 + 8 + code, and subtracting 2^23 + 8
// (exact: both are integers below 2^24) leaves the code. This keeps the
// conversion on the integer and fp32 pipes rather than the slower
// integer-to-float conversion unit.
__device__ __forceinline__ float code_f32(uint32_t w, int t) {
    return __fsub_rn(__uint_as_float(((w >> (4 * t)) & 0xFu) ^ 0x4B000008u), 8388616.0f);
}

// r[t] += s * code t of w (t = 0..7), two elements per packed fp32 instruction:
// code_f32's exact subtraction, the exact product and the rounded sum, each
// lane rounded exactly as the scalar __fadd_rn(r, __fmul_rn(s, code_f32(w, t))).
__device__ __forceinline__ void dequant_add8(float *r, uint32_t w, float s) {
#pragma unroll
    for (int t = 0; t < 8; t += 2) {
        const uint32_t n0 = ((w >> (4 * t)) & 0xFu) ^ 0x4B000008u;
        const uint32_t n1 = ((w >> (4 * t + 4)) & 0xFu) ^ 0x4B000008u;
        asm("{\n\t.reg .b64 c, k, m, a;\n\t"
            "mov.b64 c, {%2, %3};\n\t"
            "mov.b64 k, {%5, %5};\n\t"
            "mov.b64 m, {%4, %4};\n\t"
            "sub.rn.f32x2 c, c, k;\n\t"
            "mul.rn.f32x2 c, c, m;\n\t"
            "mov.b64 a, {%0, %1};\n\t"
            "add.rn.f32x2 a, a, c;\n\t"
            "mov.b64 {%0, %1}, a;\n\t}"
            : "+f"(r[t]), "+f"(r[t + 1])
            : "r"(n0), "r"(n1), "f"(s), "f"(8388616.0f));
    }
}

// Adds scale*code of every delta layer of `view` that holds token i to the
// 8 fp32 values of chunk c8 (elements 8*c8 .. 8*c8+7) of head h.
__device__ __forceinline__ void apply_deltas(const DeltaView &view, bool is_v, int m0, int m1, long long b,
                                             int i, int h, int c8, int H, int d, int N_cap, int R_cap,
                                             float rec[8]) {
    for (int m = m0; m < m1; ++m) {
        const int e = __ldg(view.slot[m] + b * N_cap + i);
        if (e < 0) continue;
        const long long ent = (b * R_cap + e) * H + h;
        const uint8_t *codes = is_v ? view.v_codes[m] : view.k_codes[m];
        const uint16_t *scales = is_v ? view.v_scales[m] : view.k_scales[m];
        const uint32_t w = __ldg(reinterpret_cast<const uint32_t *>(codes + ent * (d / 2)) + c8);
        const float s = __half2float(__ushort_as_half(__ldg(scales + ent * (d / 32) + c8 / 4)));
        dequant_add8(rec, w, s);
    }
}

__device__ __forceinline__ void load_base8(const uint16_t *base, long long b, int i, int h, int c8, int H,
                                           int d, int N_cap, float rec[8]) {
    const uint4 v = ldg_nc_v4(base + ((b * N_cap + i) * H + h) * (long long)d + c8 * 8);
    unpack_bf16x8(v, rec);
}

// The base's 8 fp32 values of chunk c8 of token i, head h: bf16 rows, or an
// int8 base's scale * code (exact in fp32: an 8-bit code times an fp16 scale).
__device__ __forceinline__ void load_base8(const DeltaView &view, bool is_v, long long b, int i, int h, int c8,
                                           int H, int d, int N_cap, float rec[8]) {
    const uint16_t *bf = is_v ? view.v_base : view.k_base;
    if (bf) {
        load_base8(bf, b, i, h, c8, H, d, N_cap, rec);
        return;
    }
    const long long row = (b * N_cap + i) * H + h;
    const int8_t *codes = is_v ? view.v_base_codes : view.k_base_codes;
    const uint16_t *scales = is_v ? view.v_base_scales : view.k_base_scales;
    const uint2 c = __ldg(reinterpret_cast<const uint2 *>(codes + row * d) + c8);
    const float s = __half2float(__ushort_as_half(__ldg(scales + row * (d / 32) + c8 / 4)));
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const int code = (int)(int8_t)(((e < 4 ? c.x : c.y) >> (8 * (e & 3))) & 0xFFu);
        rec[e] = __fmul_rn(s, (float)code);
    }
}

// The 8 codes of chunk c8 (elements 8 c8 .. 8 c8 + 7) of a row of `bits`-bit
// two's-complement codes (a little-endian bit string), returned as eight 4-bit
// two's-complement nibbles (code t in bits [4t, 4t + 4)) of the same values, the
// form dequant_add8 takes. `row` is 4-byte aligned (a row holds d * bits / 8
// bytes, a multiple of 4 for d a multiple of 32).
__device__ __forceinline__ uint32_t load_codes8(const uint8_t *row, int c8, int bits) {
    const uint32_t *w = reinterpret_cast<const uint32_t *>(row);
    if (bits == 4) return __ldg(w + c8);
    const int off = 8 * bits * c8;            // first bit of the chunk
    const int wi = off >> 5, sh = off & 31;
    uint32_t v = __ldg(w + wi) >> sh;
    if (sh + 8 * bits > 32) v |= __ldg(w + wi + 1) << (32 - sh);
    const uint32_t mask = (1u << bits) - 1u, sign = 1u << (bits - 1);
    uint32_t out = 0u;
#pragma unroll
    for (int t = 0; t < 8; ++t) {
        uint32_t c = (v >> (bits * t)) & mask;
        if (c & sign) c |= 0xFu & ~mask;      // sign-extend to four bits
        out |= c << (4 * t);
    }
    return out;
}

inline int ceil_div(long long a, long long b) { return (int)((a + b - 1) / b); }

// Programmatic dependent launch. A kernel launched with launch_pdl may have its
// CTAs scheduled while the previous kernel on the stream is still finishing;
// pdl_wait() blocks until that kernel has completed and its writes are visible
// (a no-op for a normal launch), so it comes before any global memory access.
// pdl_trigger() lets the next such kernel be scheduled once every CTA of this
// grid has started.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace fl

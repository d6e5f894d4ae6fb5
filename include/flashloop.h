/*
 * flashloop.h -- C ABI of the FlashLoop lazy loop step on one B300 (sm_103a).
 *
 * The operations follow the rit.work page "FlashLoop: Fast and
 * Memory-Efficient Looped Transformers via Lazy Updates" (a summary of the
 * Yang & Liu preprint):
 *   - section "Later loops change only part of the state": every loop of a
 *     looped transformer makes its own KV cache; few tokens keep changing and
 *     that group narrows and nests; a small, stable group of keys drives the
 *     loop-to-loop change of attention; neighbouring KV sets differ less than
 *     whole states, so a base plus small deltas compresses better;
 *   - section "FlashLoop combines three kinds of saving": early loops run in
 *     full; later loops rank tokens by how much their hidden state changed
 *     and recompute only the active ones (the rest reuse state and KV
 *     entries); keys are chosen from the previous loop's statistics and the
 *     chosen group keeps its total probability mass; the KV cache is a
 *     compressed base plus a sequence of compressed deltas, a low-bit delta
 *     for active tokens and no entry for inactive ones (4-bit deltas); the
 *     selected data is gathered into dense buffers.
 *
 * Conventions for every call below
 *   - Pointers are DEVICE pointers owned by the caller, 16-byte aligned, to
 *     contiguous row-major arrays with the shapes given. bf16 and fp16
 *     values travel as uint16_t bit patterns.
 *   - No call allocates, frees or synchronises the device unless its comment
 *     says so. Work is enqueued on `stream` (a cudaStream_t; NULL = legacy
 *     default stream) and the call returns.
 *   - Host-side validation failures return an error status and enqueue
 *     nothing. A failed launch returns FLASHLOOP_ERR_CUDA. The detail of the
 *     last failure on the calling thread is in flashloop_last_error().
 *   - Index lists are int32, ascending, and ties in every ranking go to the
 *     lower index.
 *   - Calls are reentrant; calls that write the same buffers on different
 *     streams without ordering race.
 */
#ifndef FLASHLOOP_H
#define FLASHLOOP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *flashloop_stream_t; /* same type as cudaStream_t */

typedef enum {
    FLASHLOOP_OK = 0,
    FLASHLOOP_ERR_INVALID_ARG = -1, /* null/misaligned pointer, bad size or count */
    FLASHLOOP_ERR_UNSUPPORTED = -2, /* head dim not in {64, 96, 128}, or not an sm_103 device */
    FLASHLOOP_ERR_CAPACITY = -3,    /* cache or delta layer too small for the request */
    FLASHLOOP_ERR_CUDA = -4,        /* a CUDA runtime call or kernel launch failed */
    FLASHLOOP_ERR_WORKSPACE = -5,   /* workspace missing or smaller than required */
    FLASHLOOP_ERR_DEVICE = -6       /* a kernel reported a failure (see flashloop_device_status) */
} flashloop_status_t;

#define FLASHLOOP_MAX_LOOPS 32

/* Default limit of every bounded wait inside the attention kernel (ns). */
#define FLASHLOOP_WAIT_LIMIT_DEFAULT_NS 1000000000ull

/* Problem sizes. B sequences, N_cap key positions per sequence (prefill
 * tokens plus room for decode tokens), H heads of dimension d (64, 96 or
 * 128), D = H*d. R active tokens per sequence and K key columns per
 * (sequence, head) per lazy loop. T loops of which the first T_dense are
 * dense. R_cap = entries per delta layer and sequence (>= R).
 * Cache format ("a compressed base plus a sequence of compressed deltas";
 * 4-bit deltas in the page's main experiments, lower widths degrade quality):
 *   delta_bits  width of the delta codes: 4 (or 0), 3 or 2; symmetric codes
 *               in [-qmax, qmax], qmax = 2^(delta_bits-1) - 1
 *   base_bits   16 (or 0): the base is the last dense loop's bf16 layer;
 *               8: the lazy loops read an int8 copy of it instead (one fp16
 *               scale per 32 elements, scale = fp16(amax/127)), made when
 *               that layer is stored; the dense loops still attend over bf16. */
typedef struct {
    int32_t B, N_cap, H, d;
    int32_t R, K;
    int32_t T, T_dense;
    int32_t R_cap;
    int32_t delta_bits, base_bits;
} flashloop_dims_t;

/* Per-loop KV cache ("a compressed base plus a sequence of compressed
 * deltas"). Dense loop t (1..T_dense) owns a full bf16 layer; the base is
 * layer T_dense (with base_bits = 8 also held as int8 codes [B, N_cap, H, d]
 * with fp16 scales [B, N_cap, H, d/32], which the lazy loops read). Lazy
 * loop l (T_dense < l <= T) owns delta layer l - T_dense - 1 holding, per
 * sequence b, count[] entries:
 *   idx    [B, R_cap]            token index of each entry, ascending
 *   slot   [B, N_cap]            entry of each token, -1 = no entry
 *   codes  [B, R_cap, H, d*w/8]  two's-complement codes of w = delta_bits
 *                                bits; element x occupies bits [x*w, x*w + w)
 *                                of its row read as a little-endian bit
 *                                string (w = 4: element 2t is the low nibble
 *                                of byte t)
 *   scales [B, R_cap, H, d/32]   fp16 scale of each 32-element group
 * for K and V separately. The reconstruction of token j at loop l is the
 * base (scale*code for an int8 base) plus, in ascending loop order,
 * scale*code of every delta layer up to l that holds j, summed in fp32
 * without fused multiply-add.
 * All pointers are carved from one caller buffer by flashloop_kv_cache_init;
 * `count` and `n_tokens` are host-side and updated by the calls that append. */
typedef struct {
    flashloop_dims_t dims;
    int32_t n_tokens;                        /* key positions in use */
    uint16_t *k_dense[FLASHLOOP_MAX_LOOPS];  /* [B, N_cap, H, d] bf16 */
    uint16_t *v_dense[FLASHLOOP_MAX_LOOPS];
    int32_t *idx[FLASHLOOP_MAX_LOOPS];
    int32_t *slot[FLASHLOOP_MAX_LOOPS];
    uint8_t *k_codes[FLASHLOOP_MAX_LOOPS];
    uint16_t *k_scales[FLASHLOOP_MAX_LOOPS];
    uint8_t *v_codes[FLASHLOOP_MAX_LOOPS];
    uint16_t *v_scales[FLASHLOOP_MAX_LOOPS];
    int32_t count[FLASHLOOP_MAX_LOOPS];
    int8_t *k_base_codes, *v_base_codes;     /* base_bits = 8: [B, N_cap, H, d] */
    uint16_t *k_base_scales, *v_base_scales; /* base_bits = 8: [B, N_cap, H, d/32] fp16 */
} flashloop_kv_cache_t;

/* How a lazy prefill loop ranks key columns for its selection. */
typedef enum {
    FLASHLOOP_KEYS_BY_MASS = 0,         /* column mass c_j */
    FLASHLOOP_KEYS_BY_MASS_PER_ROW = 1  /* c_j / (N - j): mass per causal row that sees key j */
} flashloop_key_rank_t;

typedef enum {
    FLASHLOOP_ATTN_FIRST_DENSE = 0, /* loop 1: every row and key, no previous state (m = 1, u = 0) */
    FLASHLOOP_ATTN_DENSE = 1,       /* a later dense loop: every row and key, previous state used */
    FLASHLOOP_ATTN_LAZY = 2         /* listed rows, selected key columns, preserved mass */
} flashloop_attn_mode_t;

/* Lazy attention with preserved probability mass. For every listed row i
 * (key position pos_i, state slot s) and head h, with S_i = {j in S : j <= i}
 * and scale 1/sqrt(d):
 *   p_j   = exp(qhat_s . k_j^(l-1) * scale - Z_s)        previous-loop probability
 *   m     = sum_{S_i} p_j,   u = sum_{S_i} p_j v_j^(l-1)
 *   tau_j = q_s . k_j^(l) * scale,  lam = logsumexp_{S_i} tau
 *   w     = sum_{S_i} exp(tau_j - lam) v_j^(l)
 *   O_s <- O_s - u + m w,  Z_s <- lam - ln m,  qhat_s <- q_s,
 *   c_j += m exp(tau_j - lam) - p_j  for j in S_i.
 * k^(t), v^(t) are the cache's reconstructions rounded to bf16. Rows with
 * S_i empty, or with m below FLT_MIN, keep O, Z and qhat. FIRST_DENSE uses
 * m = 1, u = 0, p = 0 and overwrites c with the column sums. DENSE and
 * FIRST_DENSE take every key and every row (row_pos is ignored, R = n_state
 * = n_keys). The dense layer of loop `loop` must already hold K/V.
 * Precision: bf16 operands, fp32 accumulation and softmax.
 * LAZY with more than 8 rows uses `workspace` (flashloop_workspace_bytes of
 * the cache's dims) for the gathered keys and the per-row key counts, and
 * needs K <= dims.K and R <= dims.R_cap; otherwise FLASHLOOP_ERR_WORKSPACE. */
typedef struct {
    int32_t mode;             /* flashloop_attn_mode_t */
    int32_t loop;             /* l, 1-based */
    int32_t n_keys;           /* key positions 0..n_keys-1 of the cache */
    int32_t n_state;          /* state rows per sequence */
    int32_t R;                /* listed rows per sequence */
    const int32_t *row_pos;   /* [B, R] key position of each row, ascending */
    const int32_t *row_slot;  /* [B, R] state row of each row; NULL = row_pos */
    int32_t K;                /* selected key columns per (b, h) (LAZY) */
    const int32_t *key_idx;   /* [B, H, K] ascending (LAZY) */
    const uint16_t *q;        /* [B, n_state, H, d] bf16, loop-l queries */
    uint16_t *q_hat;          /* [B, n_state, H, d] bf16 state (in/out) */
    float *o;                 /* [B, n_state, H, d] state (in/out) */
    float *z;                 /* [B, H, n_state] log-normaliser state (in/out) */
    float *c;                 /* [B, H, n_keys] column mass (in/out) */
    const flashloop_kv_cache_t *cache;
    void *workspace;
    size_t workspace_bytes;
} flashloop_attn_args_t;

/* One loop of the looped model, fused: for a dense loop (l <= T_dense) it
 * stores K/V as dense layer l and runs dense attention; for a lazy loop it
 * runs select_tokens on (h_prev, h_cur), kv_delta_append of K and V for the
 * active tokens, select_keys on c, and lazy attention. `decode` = 1 runs the
 * same loop for ONE new token per sequence at key position cache->n_tokens-1
 * (the caller counts it in n_tokens before loop 1): state arrays then have
 * one row, the token is always active, and h_prev/h_cur are unused.
 * In a lazy prefill loop the key selection runs on a library-owned stream
 * forked from `stream` with an event and joined back to it before the
 * attention, so every piece of the loop is ordered on `stream` as usual (and
 * the call can be captured into a CUDA graph from `stream`). */
typedef struct {
    int32_t loop;
    int32_t decode;
    const uint16_t *h_prev;   /* [B, N, D] bf16, loop l-1 hidden states (prefill, lazy) */
    const uint16_t *h_cur;    /* [B, N, D] bf16, loop l hidden states */
    const uint16_t *q;        /* [B, N, H, d] bf16 (decode: [B, 1, H, d]) */
    const uint16_t *k;
    const uint16_t *v;
    uint16_t *q_hat;          /* state, as in flashloop_attn_args_t */
    float *o;
    float *z;
    float *c;                 /* [B, H, n_keys] */
    flashloop_kv_cache_t *cache;
    int32_t *active_idx;      /* [B, R] out (prefill lazy loops) */
    int32_t *key_idx;         /* [B, H, K] out (lazy loops) */
    float *scores;            /* [B, N] out, or NULL */
    void *workspace;
    size_t workspace_bytes;
    int32_t key_rank;         /* flashloop_key_rank_t of the key selection (prefill lazy loops) */
    /* Early exit of a sequence by state difference (prefill lazy loops; NULL
     * seq_exit = off). seq_exit [B] int32 device flags, caller-owned, zero at
     * the start: a sequence flagged 1 has stopped looping, and every later lazy
     * loop leaves it unchanged (its delta entries are zero deltas, its rows
     * keep O, Z and qhat, its column masses stay). With exit_threshold > 0 the
     * loop first sets the flag of every sequence whose largest token change
     * score (squared L2 norm of h_cur - h_prev, the one the token selection
     * ranks by) is below it, in fp32; flags are never cleared by the library. */
    float exit_threshold;
    int32_t *seq_exit;
} flashloop_step_args_t;

/* Weights of the synthetic looped block (one weight-shared block applied every
 * loop; random weights stand in for a trained looped model). Each matrix is
 * stored transposed, [out features, in features] row-major bf16, so that the
 * weights of one output feature are contiguous:
 *   w_qkv [3D, D]  rows 0..D-1 give q, D..2D-1 k, 2D..3D-1 v, each in
 *                  (head, dim) order, the layout of a [B, N, H, d] row
 *   w_o   [D, D]   attention output projection
 *   w_1   [F, D]   MLP up projection (ReLU)
 *   w_2   [D, F]   MLP down projection
 * D = H*d and F must be multiples of 256. */
typedef struct {
    const uint16_t *w_qkv, *w_o, *w_1, *w_2;
    int32_t F;
} flashloop_block_weights_t;

/* One loop l of the synthetic looped block around the lazy step (rit.work
 * page "FlashLoop: Fast and Memory-Efficient Looped Transformers via Lazy
 * Updates", section "FlashLoop combines three kinds of saving": a later loop
 * recomputes only its active tokens, the others reuse their state). With
 * x_i = H_{l-1}[i] (bf16) and bf16() = round to nearest even:
 *   q_i, k_i, v_i = bf16(x_i W_q), bf16(x_i W_k), bf16(x_i W_v)
 *   (the loop's attention as in flashloop_loop_step, giving O_i)
 *   y_i = bf16(x_i + bf16(O_i) W_o)
 *   u_i = bf16(relu(y_i W_1))
 *   H_l[i] = bf16(y_i + u_i W_2)
 * for every token i of a dense loop, and only for the active tokens i of a
 * lazy loop, whose other tokens keep H_l[i] = H_{l-1}[i]. Products accumulate
 * in fp32. The active tokens of a lazy loop are the top-R of the change
 * score on (h_prev = H_{l-2}, h_cur = H_{l-1}) as in flashloop_select_tokens;
 * its keys the top-K of c as in flashloop_select_keys (key_rank chooses the
 * ranking as in flashloop_step_args_t). */
typedef struct {
    int32_t loop;
    const uint16_t *h_prev;   /* [B, N, D] H_{l-2} (lazy loops) */
    const uint16_t *h_cur;    /* [B, N, D] H_{l-1}, the loop's input */
    /* [B, N, D] out: H_l. In a lazy loop only the rows that can differ from
     * h_cur are written: on entry every row not listed in stale_idx must
     * already hold h_cur's value. stale_idx [B, n_stale] (NULL: every row is
     * stale and is copied from h_cur) is typically the previous lazy loop's
     * active_idx when h_out is the buffer of h_prev (buffers then alternate:
     * the next loop's h_prev is this h_cur and its h_out this h_cur's buffer).
     * h_out may be h_prev; it must not be h_cur. Dense loops write every row.
     * Indices outside [0, N) in stale_idx are skipped. */
    uint16_t *h_out;
    const int32_t *stale_idx;
    int32_t n_stale;
    uint16_t *q_hat;          /* state, as in flashloop_attn_args_t */
    float *o;
    float *z;
    float *c;                 /* [B, H, n_keys] */
    flashloop_kv_cache_t *cache;
    int32_t *active_idx;      /* [B, R] out (in with force_selection) (lazy loops) */
    int32_t *key_idx;         /* [B, H, K] out (in with force_selection) (lazy loops) */
    int32_t force_selection;  /* 1: active_idx and key_idx are inputs, no selection runs */
    int32_t key_rank;         /* flashloop_key_rank_t */
    float *scores;            /* [B, N] out, or NULL */
    const flashloop_block_weights_t *weights;
    /* [B, N, H, d] bf16 each, out, or NULL (then they live in the workspace):
     * the loop's q, k, v (a lazy loop writes the active tokens' rows only) */
    uint16_t *q, *k, *v;
    void *workspace;          /* flashloop_block_workspace_bytes(dims, F), 256-byte aligned */
    size_t workspace_bytes;
} flashloop_block_args_t;

/* ---- sizes and set-up ------------------------------------------------- */

/* Bytes of workspace every call below needs for these dims (prefill and
 * decode). Returns 0 for invalid dims. */
size_t flashloop_workspace_bytes(const flashloop_dims_t *dims);

/* Bytes of workspace flashloop_block_loop needs for these dims and MLP
 * width F (the step's workspace plus the block's q/k/v and row buffers).
 * Returns 0 for invalid dims or F. */
size_t flashloop_block_workspace_bytes(const flashloop_dims_t *dims, int32_t F);

/* Bytes of the single device buffer that holds the whole KV cache. */
size_t flashloop_kv_cache_bytes(const flashloop_dims_t *dims);

/* Carves `dev_buf` (>= flashloop_kv_cache_bytes, 256-byte aligned) into the
 * cache layers and enqueues the reset of every slot map to -1 on `stream`.
 * Counts and n_tokens start at zero. */
flashloop_status_t flashloop_kv_cache_init(flashloop_kv_cache_t *cache, void *dev_buf, size_t bytes,
                                           const flashloop_dims_t *dims, flashloop_stream_t stream);

/* ---- the steps of a lazy loop ----------------------------------------- */

/* Token selection ("rank tokens by how much their hidden states changed
 * and recompute only the active ones"): score_i = sum_x (h_cur - h_prev)^2
 * in fp32 over the D features of token i, then the R largest per sequence
 * (ties to the lower index), ascending.
 * h_prev, h_cur [B, N, D] bf16; active_idx [B, R] out; scores [B, N] out
 * or NULL. Workspace: flashloop_workspace_bytes (holds the scores when
 * `scores` is NULL). 1 <= R <= N; D % 8 == 0. */
flashloop_status_t flashloop_select_tokens(const uint16_t *h_prev, const uint16_t *h_cur,
                                           int32_t B, int32_t N, int32_t D, int32_t R,
                                           int32_t *active_idx, float *scores,
                                           void *workspace, size_t workspace_bytes,
                                           flashloop_stream_t stream);

/* Token selection that allocates nothing (no counterpart in the paper; an
 * interface for callers that may not allocate device memory: code running
 * inside a memory arena it does not own, such as a serving engine's fixed
 * budget or a plugin host, or on a path where an allocation could stall or
 * fail at the wrong moment). Same operation and result as
 * flashloop_select_tokens, but the B*N change scores live in a fixed array
 * of this library (at most 1,048,576 scores, 4 MiB, held on every device
 * that loads the library until the process exits) instead of a caller
 * workspace; larger B*N returns FLASHLOOP_ERR_CAPACITY. The first call on
 * each device looks up the array's device address (no allocation), so make
 * that first call before any stream capture. All calls share the array:
 * calls whose work may overlap on the device (different streams, or
 * different host threads) race and must be serialised by the caller. */
flashloop_status_t flashloop_select_tokens_noalloc(const uint16_t *h_prev, const uint16_t *h_cur,
                                                   int32_t B, int32_t N, int32_t D, int32_t R,
                                                   int32_t *active_idx, flashloop_stream_t stream);

/* Gather of selected rows into a dense buffer ("the selected data is
 * gathered into dense buffers"): dst[b, r, :] = src[b, idx[b, r], :].
 * src [B, N, row_bytes], idx [B, R] in [0, N), dst [B, R, row_bytes];
 * row_bytes % 16 == 0. A row whose index lies outside [0, N) is skipped
 * (its dst row is left as it was). */
flashloop_status_t flashloop_gather(const void *src, int32_t B, int32_t N, int32_t row_bytes,
                                    const int32_t *idx, int32_t R, void *dst,
                                    flashloop_stream_t stream);

/* Delta append ("for tokens that stay active, write a low-bit difference
 * from the previous state; inactive tokens get no new entry"; 4-bit). For
 * lazy loop `loop` and every active token i and head: delta = bf16 input
 * minus the loop-(l-1) reconstruction (fp32); per 32-element group
 * scale = fp16_rne(amax / 7) and code = rint_even(delta / scale) clamped to
 * [-7, 7] (zero scale gives zero codes). Writes entries [at, at + R) of
 * the loop's K and V delta layers, their idx and slot entries, and sets
 * count = at + R. at == 0 starts the layer afresh (its slot map is reset
 * first); at == count appends (decode). k_l, v_l are bf16, either
 * [B, n_tokens, H, d] indexed by token (rows_are_tokens = 1) or [B, R, H, d]
 * with one row per listed token (rows_are_tokens = 0, as for a decode token). */
flashloop_status_t flashloop_kv_delta_append(flashloop_kv_cache_t *cache, int32_t loop,
                                             const uint16_t *k_l, const uint16_t *v_l,
                                             int32_t rows_are_tokens,
                                             const int32_t *active_idx, int32_t R, int32_t at,
                                             flashloop_stream_t stream);

/* Stores K/V rows as (part of) dense layer `loop` (loop <= T_dense):
 * layer[b, pos0 + r] = k[b, r] for r < n_rows. k, v [B, n_rows, H, d].
 * With base_bits = 8, storing into the base layer (loop = T_dense) also
 * writes those rows' int8 codes and scales. */
flashloop_status_t flashloop_kv_dense_store(flashloop_kv_cache_t *cache, int32_t loop,
                                            const uint16_t *k, const uint16_t *v,
                                            int32_t pos0, int32_t n_rows, flashloop_stream_t stream);

/* Key-column selection ("keys are chosen from the previous loop's
 * statistics"): the K largest col_stats per (b, h), ties to the lower index,
 * ascending. col_stats [B, H, N] fp32; key_idx [B, H, K] out. */
flashloop_status_t flashloop_select_keys(const float *col_stats, int32_t B, int32_t H, int32_t N, int32_t K,
                                         int32_t *key_idx, void *workspace, size_t workspace_bytes,
                                         flashloop_stream_t stream);

/* Key-column selection by column mass per causal row: another reading of
 * "keys are chosen from the previous loop's statistics" (same page and
 * section as flashloop_select_keys): the K largest col_stats[b, h, j] / (n_rows - j) per
 * (b, h), the quotient an IEEE fp32 division, ties to the lower index,
 * ascending. In a prefill of n_rows tokens, n_rows - j rows see key j, so a
 * key that late rows see is not outranked only for being seen by fewer rows.
 * col_stats [B, H, N] fp32; key_idx [B, H, K] out. N <= n_rows. */
flashloop_status_t flashloop_select_keys_per_row(const float *col_stats, int32_t B, int32_t H, int32_t N, int32_t K,
                                                 int32_t n_rows, int32_t *key_idx, flashloop_stream_t stream);

/* Reconstruct-gather of the selected keys: for j = key_idx[b, h, r],
 * k_old/v_old[b, h, r, :] = bf16_rne(reconstruction at loop-1) and
 * k_new/v_new[b, h, r, :] = bf16_rne(reconstruction at loop). Outputs
 * [B, H, K, d] bf16 each. */
flashloop_status_t flashloop_reconstruct_keys(const flashloop_kv_cache_t *cache, int32_t loop,
                                              const int32_t *key_idx, int32_t K,
                                              uint16_t *k_old, uint16_t *v_old,
                                              uint16_t *k_new, uint16_t *v_new,
                                              flashloop_stream_t stream);

/* Lazy (or dense) attention, see flashloop_attn_args_t. */
flashloop_status_t flashloop_lazy_attention(const flashloop_attn_args_t *args, flashloop_stream_t stream);

/* One fused loop, see flashloop_step_args_t. Graph-capturable: it only
 * enqueues kernels and memsets on `stream`. */
flashloop_status_t flashloop_loop_step(const flashloop_step_args_t *args, flashloop_stream_t stream);

/* bf16 GEMM on the tcgen05 tensor cores, the projections of the synthetic
 * looped block: for every row m < M,
 *   C[m, :] = act(A[m, :] W^T + residual[m, :])   act = ReLU if relu else identity,
 * A [M, K] bf16, w_t = W^T [N, K] bf16, residual [M, N] bf16 or NULL, fp32
 * accumulation, the residual added in fp32, then one round to bf16 (nearest
 * even). Columns [s*N/n_split, (s+1)*N/n_split) go to output c[s]
 * (c: a host array of n_split device pointers), whose rows are N/n_split
 * elements long. Row m goes to output row m, or with c_rows [M] (device) to
 * row (m / rows_per_seq) * seq_rows + c_rows[m] (a scatter to token rows of
 * sequences of seq_rows rows; M % rows_per_seq == 0). An index outside
 * [0, seq_rows) stores nothing for that row and sets the device status word
 * (flashloop_device_status) to 0x101. Requires K % 64 == 0, 1 <= n_split <= 3,
 * N % (256 * n_split) == 0, 16-byte aligned pointers. M = 0 enqueues nothing. */
flashloop_status_t flashloop_gemm(const uint16_t *a, int32_t M, int32_t K, const uint16_t *w_t, int32_t N,
                                  const uint16_t *residual, int32_t relu, uint16_t *const *c, int32_t n_split,
                                  const int32_t *c_rows, int32_t rows_per_seq, int32_t seq_rows,
                                  flashloop_stream_t stream);

/* One loop of the synthetic looped block, see flashloop_block_args_t.
 * Prefill only (every token of the cache's n_tokens is a row); no early exit.
 * Graph-capturable like flashloop_loop_step. */
flashloop_status_t flashloop_block_loop(const flashloop_block_args_t *args, flashloop_stream_t stream);

/* ---- diagnostics -------------------------------------------------------- */

/* Name of a status code ("ok", "invalid argument", ...), or "unknown status"
 * for a value outside flashloop_status_t. A static string: do not free it. */
const char *flashloop_status_string(flashloop_status_t status);

/* Message of the most recent failing call made by the calling thread (which
 * argument, size or CUDA call failed). Successful calls leave it unchanged;
 * the pointer stays valid until that thread's next failing call. Owned by the
 * library: do not free it. Empty before the thread's first failure. */
const char *flashloop_last_error(void);

/* Reads and clears the device-side failure word (0 = none) that kernels set
 * when a bounded wait gives up: codes below 0x100 come from the attention
 * kernel, 0x100 from the GEMM, 0x101 is the GEMM's out-of-range output row
 * (the attention's word is reported first when both are set; both are
 * cleared). SYNCHRONISES the current device. */
flashloop_status_t flashloop_device_status(int32_t *word);

/* Sets the limit, in ns, of the bounded waits inside the tensor-core
 * attention kernel on the current device (failure handling, not part of the
 * method: for tests and diagnosis of the give-up path). A wait that runs past
 * it makes the CTA record an error word (see flashloop_device_status), stop
 * issuing work, let its own copies and MMAs land (drains keep the default
 * limit) and exit; the launch still completes and the context stays usable.
 * 0 <= ns <= FLASHLOOP_WAIT_LIMIT_DEFAULT_NS (the limit can only be
 * shortened; pass the default to restore it), else FLASHLOOP_ERR_INVALID_ARG.
 * With 0 a wait does not wait at all: it gives up unless its phase has
 * already completed when first tested. Call it between launches: it
 * SYNCHRONISES the current device. */
flashloop_status_t flashloop_set_wait_limit_ns(uint64_t ns);

/* Number of kernel launches this library has enqueued from the calling
 * process (a counter for benchmarks). */
int64_t flashloop_launch_count(void);

/* Per-kernel timing for benchmarks. While enabled, every kernel launch of
 * this library is bracketed by two CUDA events recorded on the launch's own
 * stream. */
flashloop_status_t flashloop_timing_enable(int32_t on);

/* SYNCHRONISES the current device, then reports, per kernel family, its
 * name (written to names + k*name_len, NUL-terminated), the summed event
 * time in ms and the number of launches since the previous read, and
 * clears the records. Returns the number of families written (at most
 * max_kinds), or -1 if the synchronisation failed. */
int32_t flashloop_timing_read(char *names, int32_t name_len, double *total_ms, int64_t *launches,
                              int32_t max_kinds);

#ifdef __cplusplus
}
#endif
#endif /* FLASHLOOP_H */

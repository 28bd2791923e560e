/*
 * sinkkv.h -- C ABI of libsinkkv: sink + sliding-window KV attention with RoPE/YaRN
 * on one NVIDIA GB300 (sm_103a).
 *
 * The operations follow the problem statement of these pages:
 *   [RoPE]   "RoPE, scaling, sliding window, attention sinks" (mlinterviewnotes)
 *   [MIXED]  "Inference & 128K Long Context" / "KV-Cache Engineering" (GPT-OSS-Lite)
 *   [DYN]    "#2961 rope: --rope-scaling dynamic" (strata pull request)
 *   [SINK]   "Attention Sink 与 Streaming KV Cache" (llm-glossary)
 *
 * Conventions for every call
 *   - Ownership: the caller owns every tensor, cache, state array and workspace.
 *     The library owns only sk_rope_table objects (host and device memory).
 *   - Pointers named "device" are CUDA device pointers of the current device;
 *     "host" pointers are ordinary host memory.  `stream` is a cudaStream_t
 *     (NULL = legacy default stream).  Every call is asynchronous on `stream`
 *     except table create/rebuild, which synchronise `stream` before returning.
 *   - Layouts are dense, row-major, innermost last, with no padding.
 *   - Errors: host-side argument checks run before any launch and return an
 *     sk_status; nothing is launched on error.  Conditions that depend on device
 *     state (a position past the table, a global layer past its capacity) are
 *     detected by the kernel, which then leaves that sequence untouched and ORs a
 *     bit into the layer's device error word `err` (SK_DEVERR_*), if given.
 *     Launch failures return SK_ERR_CUDA.  No call aborts or traps the GPU.
 */
#ifndef SINKKV_H
#define SINKKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Exported symbols (the library is built with hidden default visibility). */
#if defined(__GNUC__)
#define SK_API __attribute__((visibility("default")))
#else
#define SK_API
#endif

typedef enum {
    SK_OK = 0,
    SK_ERR_ARG = 1,             /* a null pointer, bad shape or inconsistent argument */
    SK_ERR_CAPACITY = 2,        /* a cache cannot hold what was asked */
    SK_ERR_POSITION_RANGE = 3,  /* a position at or past the table's max_positions */
    SK_ERR_UNSUPPORTED = 4,     /* a valid combination this build does not implement */
    SK_ERR_CUDA = 5             /* a CUDA runtime call or launch failed */
} sk_status;

typedef enum { SK_BF16 = 0, SK_F32 = 1, SK_I8 = 2 } sk_dtype;

typedef enum { SK_LAYER_RING = 0, SK_LAYER_GLOBAL = 1 } sk_layer_kind;

/* Bits of a device error word (uint32_t, caller-owned, zeroed by the caller). */
#define SK_DEVERR_POSITION_RANGE 0x1u  /* a position >= max_positions was skipped   */
#define SK_DEVERR_CAPACITY       0x2u  /* a global-layer append past capacity was skipped */
#define SK_DEVERR_TIMEOUT        0x4u  /* a bounded in-kernel wait gave up (never expected) */
#define SK_DEVERR_BLOCK_TABLE    0x8u  /* a paged block id outside [0, n_blocks) was met  */
#define SK_DEVERR_STATE          0x10u /* a prefill's prior cache did not hold its prefix */

/*
 * Rotary configuration.  [RoPE] "Let d_h be the head dimension, r <= d_h the rotary
 * dimension ... b the base"; the frequencies omega_i = theta^(-2i/r) (the
 * _compute_inv_freq listing); NeoX pairs (j, j + r/2), GPT-J pairs (2j, 2j+1).
 * yarn_factor <= 1 means plain RoPE; otherwise the YaRN blend of [RoPE] "YaRN,
 * precisely" with original context yarn_orig_ctx, beta_fast / beta_slow, and the
 * mscale mu = 0.1 ln s + 1 folded into both cos and sin.
 * Constraints: rotary_dim even, 16 <= rotary_dim <= head_dim, head_dim in {64, 128},
 * rotary_dim a multiple of 16; max_positions >= 1.
 */
typedef struct {
    int32_t head_dim;
    int32_t rotary_dim;
    int32_t neox;            /* 1 = NeoX pairing, 0 = GPT-J pairing */
    int32_t reserved0;
    double theta;            /* rope_theta, > 1 */
    double yarn_factor;      /* <= 1: plain RoPE */
    int64_t yarn_orig_ctx;   /* L0, used when yarn_factor > 1 */
    double beta_fast;        /* default 32 */
    double beta_slow;        /* default 1 */
    int64_t max_positions;   /* table rows: positions 0 .. max_positions-1 */
} sk_rope_config;

/* Opaque, library-owned cos/sin table.  Its device buffer is
 * float2[max_positions][rotary_dim/2] = (mu cos(P omega_j), mu sin(P omega_j)),
 * computed in float64 on the host and rounded to float32 ([RoPE] "Hybrid models
 * break the uniform-spec assumption", the walk of one decode token: the rotation
 * gathers table rows and does no trigonometry). */
typedef struct sk_rope_table sk_rope_table;

/*
 * One layer's KV cache for a batch of sequences.  All pointers are device pointers
 * owned by the caller.
 *   kind = SK_LAYER_RING   ([MIXED] "Windowed layers - ring buffer", extended with
 *     [SINK]'s pinned sinks): slots [0, sinks) hold positions 0..sinks-1 and are
 *     never overwritten; slots [sinks, sinks+window) are a ring with state
 *     head[b] in [0, window) and count[b] in [0, window]; capacity = sinks + window.
 *   kind = SK_LAYER_GLOBAL ([MIXED] "Global layers"): slot = position, rows [0, pos[b])
 *     are valid; capacity = rows allocated per (sequence, kv head).
 *   k, v:    [batch][n_kv_heads][capacity][head_dim] of k_dtype / v_dtype
 *   k_scale: [batch][n_kv_heads][capacity] float, one scale per int8 K row (k_dtype
 *            SK_I8 only, else NULL)
 *   head, count: int32 [batch] (ring only; may be NULL for global layers)
 *   pos:     int64 [batch], tokens seen so far = the next absolute position
 *   err:     uint32 device error word, may be NULL
 * k_dtype in {SK_BF16, SK_F32, SK_I8}; v_dtype in {SK_BF16, SK_F32}.
 */
typedef struct {
    int32_t kind;
    int32_t k_dtype;
    int32_t v_dtype;
    int32_t batch;
    int32_t n_kv_heads;
    int32_t head_dim;
    int32_t sinks;
    int32_t window;
    int64_t capacity;
    void* k;
    void* v;
    float* k_scale;
    int32_t* head;
    int32_t* count;
    int64_t* pos;
    uint32_t* err;
} sk_kv_layer;

/*
 * One layer's paged KV cache for a batch of requests ("vLLM, from the inside out",
 * PagedAttention: a shared pool of fixed-size blocks and a per-request block table
 * from logical block to physical block; [RoPE] "Hybrid models break the uniform-spec
 * assumption": static sink blocks put in front of every block table).  All pointers
 * are device pointers owned by the caller; the caller allocates and frees blocks.
 *   k_pool, v_pool: [n_blocks][n_kv_heads][block_size][head_dim] of k_dtype / v_dtype
 *   block_table: int32 [batch][max_blocks]; request block j holds the request's tokens
 *     [j*block_size, (j+1)*block_size).  Entries of blocks that hold no visible key may
 *     be anything (freed blocks, e.g. -1): they are never read.
 *   sink_block_ids: int32 [n_sink_blocks] static sink blocks, the same for every
 *     request, or NULL when n_sink_blocks = 0.
 *   seq_lens: int64 [batch], the request's own tokens so far (static sink tokens not
 *     counted) = the RoPE position of its next token.
 *   err: uint32 device error word, may be NULL.
 * Attention of a request sees the logical key sequence "static sink tokens
 * (n_sink_blocks * block_size of them), then the request's tokens", of length
 * L = sink_len + seq_len (0 when seq_len = 0), and within it the first `sinks` keys
 * and the last `window` keys (every key when window <= 0): the visible set V(L - 1)
 * of a cache with capacity sinks + window ([SINK] "可见集合与容量定义").  With static
 * sink blocks, sinks = their token count gives them the role of the pinned sinks;
 * without, sinks = S keeps the request's own first S tokens (StreamingLLM on paged
 * memory).
 * k_dtype, v_dtype: SK_BF16 or SK_F32 (the same for both).  block_size a power of two
 * in [4, 1024].
 */
typedef struct {
    int32_t k_dtype;
    int32_t v_dtype;
    int32_t batch;
    int32_t n_kv_heads;
    int32_t head_dim;
    int32_t block_size;
    int32_t max_blocks;
    int32_t n_sink_blocks;
    int32_t sinks;
    int32_t window;
    int64_t n_blocks;
    void* k_pool;
    void* v_pool;
    const int32_t* block_table;
    const int32_t* sink_block_ids;
    int64_t* seq_lens;
    uint32_t* err;
} sk_paged_layer;

/* ---- RoPE table (host float64 build, device float32 copy) ---------------------- */

/* Build the table for `cfg` on the current device.  Allocates the device buffer;
 * on success *out owns it.  Synchronises `stream`.  Errors: SK_ERR_ARG for a bad
 * config or NULL pointer, SK_ERR_CUDA if the allocation or copy fails. */
SK_API sk_status sk_rope_table_create(const sk_rope_config* cfg, void* stream, sk_rope_table** out);

/* Rebuild the table in place for a new YaRN factor: same device pointer, so CUDA
 * graphs captured against it read the new angles ([DYN] "What it does", the table).
 * The entries are computed independently on host threads, so the result is bitwise
 * that of sk_rope_table_create with the new factor.  Ordered on `stream`
 * (kernels already queued on it finish first) and synchronises it. */
SK_API sk_status sk_rope_table_rebuild(sk_rope_table* table, double new_yarn_factor, void* stream);

/* Free the table (device and host memory).  NULL is ignored.  The caller must
 * ensure no queued kernel still reads it. */
SK_API void sk_rope_table_destroy(sk_rope_table* table);

/* Read back the table's config and its device buffer (float2 [max_positions][r/2]).
 * Either output may be NULL. */
SK_API sk_status sk_rope_table_info(const sk_rope_table* table, sk_rope_config* cfg_out,
                             const void** device_cos_sin);

/* Fill a host buffer with the table for `cfg` without any device: out is float
 * [max_positions][rotary_dim/2][2] (cos, sin pairs, the layout of the device table),
 * 8-byte aligned, owned by the caller.  n_threads host threads (0 = automatic); every entry is
 * computed on its own, so the bits do not depend on n_threads ([DYN] "Measured on
 * this branch": the threaded build equals the single-thread one bit for bit).
 * Each entry is computed in float64 as cos/sin of its block's anchor P0 w (P0 a
 * multiple of 64) combined with cos/sin of the offset (P - P0) w by angle addition,
 * then scaled by mu and rounded to float32.
 * Errors: SK_ERR_ARG for a bad config, NULL or misaligned out, or n_threads outside
 * [0, 256]. */
SK_API sk_status sk_rope_table_fill_host(const sk_rope_config* cfg, int32_t n_threads, float* out);

/* ---- Dynamic YaRN factor ------------------------------------------------------------ */

/* [DYN] "What it does", the factor: 1 while total_positions <= orig_ctx (the trained
 * context L0); beyond it (total_positions / orig_ctx) rounded up to a multiple of
 * `step`, then capped at `cap`.  Host only.  Errors: SK_ERR_ARG for
 * total_positions < 0, orig_ctx < 1, step <= 0, cap < 1 or NULL factor_out. */
SK_API sk_status sk_rope_dynamic_factor(int64_t total_positions, int64_t orig_ctx, double step, double cap,
                                        double* factor_out);

/* A table whose YaRN factor follows the dialog's length, and which turns the cached
 * keys when the factor changes ([DYN] "What it does": the factor, the cached keys,
 * the table).  Opaque, library-owned: a live table (the one to pass to
 * sk_kv_append / sk_rope_apply; its device pointer never changes) and a spare of
 * the same size. */
typedef struct sk_rope_dynamic sk_rope_dynamic;

/* cfg->yarn_factor is the starting factor (<= 1: plain RoPE), cfg->yarn_orig_ctx is
 * L0 and cfg's beta_fast / beta_slow shape every later factor; `step` > 0 is the
 * rounding step; cap <= 0 means max_positions / L0 (the most positions the table
 * holds, over the trained ones).  Allocates two device tables of max_positions x
 * rotary_dim/2 float2 each and synchronises `stream`.  Errors: SK_ERR_ARG for a bad
 * config (checked at the starting factor and at factor max(2, cap)), SK_ERR_CUDA. */
SK_API sk_status sk_rope_dynamic_create(const sk_rope_config* cfg, double step, double cap, void* stream,
                                        sk_rope_dynamic** out);

/* The live table (stable for the object's lifetime); NULL for a NULL handle. */
SK_API const sk_rope_table* sk_rope_dynamic_table(const sk_rope_dynamic* dyn);

/* The factor the live table and the turned keys hold (1 = plain RoPE). */
SK_API double sk_rope_dynamic_current_factor(const sk_rope_dynamic* dyn);

/* Pick the factor for a dialog that now spans total_positions positions (the
 * prompt's length at prefill, the grown length in decode).  If it differs from the
 * current one: build the new factor's table on host threads into the spare, turn
 * every cached key of `layers` (host array of n_layers descriptors; as
 * sk_kv_rerotate) from the live factor to the new one, copy the spare over the live
 * table's device buffer, and synchronise `stream`; the live table then equals, bit
 * for bit, sk_rope_table_create at the new factor.  If the factor is unchanged
 * nothing is launched.  *factor_out (may be NULL) gets the factor now in force,
 * *switched_out (may be NULL) 1 if it changed.  Errors: SK_ERR_POSITION_RANGE if
 * total_positions exceeds max_positions (nothing changes), SK_ERR_ARG, the errors of
 * sk_kv_rerotate, SK_ERR_CUDA. */
SK_API sk_status sk_rope_dynamic_update(sk_rope_dynamic* dyn, int64_t total_positions,
                                        const sk_kv_layer* layers, int32_t n_layers, void* stream,
                                        double* factor_out, int32_t* switched_out);

/* Free both tables.  NULL is ignored.  No queued kernel may still read them. */
SK_API void sk_rope_dynamic_destroy(sk_rope_dynamic* dyn);

/* ---- RoPE apply ------------------------------------------------------------------ */

/* Rotate x in place: x [n_tok][n_heads][head_dim] (dtype SK_BF16 or SK_F32, device),
 * row t at absolute position positions[t] (device int64 [n_tok]).
 * [RoPE] the rotation listing: o1 = x1 cos - x2 sin, o2 = x2 cos + x1 sin, times mu;
 * dims [r, d_h) untouched.  A row whose position is < 0 or >= max_positions is left
 * unchanged and sets SK_DEVERR_POSITION_RANGE in *err (device, may be NULL).
 * n_tok = 0 launches nothing and returns SK_OK; x and positions may then be NULL. */
SK_API sk_status sk_rope_apply(const sk_rope_table* table, void* x, int32_t dtype, int64_t n_tok,
                        int32_t n_heads, const int64_t* positions, uint32_t* err, void* stream);

/* ---- Fused RoPE + KV append -------------------------------------------------------- */

/* Append T new tokens per sequence to `layer`, rotating Q and K on the way.
 *   table: the RoPE table; NULL when k is already rotated (a chunk rotated with
 *      sk_rope_apply for sk_prefill_attention with a prior): k is then written as
 *      given, q must be NULL, and head_dim must be 64 or 128.
 *   q: [batch][T][n_q_heads][head_dim] of io_dtype, device, may be NULL; rotated in place.
 *   k: [batch][T][n_kv_heads][head_dim] of io_dtype, device; rotated in place, then
 *      written to the cache (quantised per row for an int8 K cache).
 *   v: [batch][T][n_kv_heads][head_dim] of io_dtype, device; written as is.
 * Token t of sequence b has absolute position P = pos[b] + t: the same counter gives
 * the angle and the slot ([RoPE] "Where the positions come from").
 * Ring layers ([MIXED] MixedKVCache.append, with [SINK] sinks): P < sinks goes to
 * slot P; of the remaining n tokens, n >= window keeps the last `window` at ring slots
 * 0..window-1 with head = 0, count = window; otherwise they go to ring slot
 * (head + u) % window, head = (head + n) % window, count = min(window, count + n).
 * Global layers: slot = P; pos[b] + T > capacity skips the sequence and sets
 * SK_DEVERR_CAPACITY.  pos[b] += T.  pos[b] + T > max_positions skips the sequence
 * and sets SK_DEVERR_POSITION_RANGE.
 * io_dtype: SK_BF16 or SK_F32.  Supported (io, k cache, v cache): (F32,F32,F32),
 * (BF16,BF16,BF16), (BF16,I8,BF16); others return SK_ERR_UNSUPPORTED.
 * n_q_heads must be a multiple of n_kv_heads when q is given.
 * T = 0 checks the layer, launches nothing (the state stays as it is) and returns
 * SK_OK; q, k and v may then be NULL. */
SK_API sk_status sk_kv_append(const sk_rope_table* table, const sk_kv_layer* layer, void* q,
                       int32_t n_q_heads, void* k, const void* v, int32_t io_dtype, int32_t T,
                       void* stream);

/* ---- Decode attention (split-K over the visible set) ------------------------------ */

/* Workspace bytes sk_decode_attention needs for `layer` and n_q_heads. */
SK_API size_t sk_decode_workspace_bytes(const sk_kv_layer* layer, int32_t n_q_heads);

/* One decode query per sequence against the visible set of its cache, after its own
 * append.  [SINK] "可见集合与容量定义": V(P) = 0..P when P < C, else sinks 0..S-1 and
 * max(S, P-W+1)..P; in a ring layer these are exactly the occupied slots
 * [0, min(pos, S) + count).  Global layers read rows [0, pos).
 * q head h reads kv head h / (n_q_heads / n_kv_heads) ([MIXED] 5.5 repeat_kv, done as an
 * in-register broadcast).  scores = q.k / sqrt(d_h), softmax, out = sum p v
 * ([SINK] the experiment's incremental_sink).
 *   q_rot: [batch][n_q_heads][head_dim] of io_dtype (device); out: same shape and dtype.
 *   sink_logits: NULL, or device float32 [n_q_heads], 4-byte aligned: learned sinks
 *   ([RoPE] "Hybrid models break the uniform-spec assumption": a trained per-head
 *   scalar in the softmax denominator that holds no cache rows).  Head h's weights
 *   become exp(s_j) / (sum_i exp(s_i) + exp(z_h)) with s the scaled scores and
 *   z_h = sink_logits[h] clamped to [-10, 15] in the kernel ([MIXED] "Sink clamp
 *   cache").  The same value serves every sequence.
 *   workspace: device, >= sk_decode_workspace_bytes(layer, n_q_heads) bytes, 16-byte
 *   aligned; its contents need no initialisation.
 * Supported: io SK_F32 with an F32/F32 cache, io SK_BF16 with a BF16/BF16 cache, and io
 * SK_BF16 with an I8/BF16 cache (int8 K codes and one fp32 scale per row in k_scale, as
 * sk_kv_append and sk_kv_rerotate write them; head_dim 128): a key is code * scale.
 * n_q_heads / n_kv_heads in {1, 2, 4} for head_dim 128 and {1, 2, 4, 8} for 64. */
SK_API sk_status sk_decode_attention(const sk_kv_layer* layer, const void* q_rot, int32_t n_q_heads,
                                     int32_t io_dtype, const float* sink_logits, void* out,
                                     void* workspace, size_t ws_bytes, void* stream);

/* ---- Decode attention without any allocation -------------------------------------- */

/* Bytes of the library's built-in decode scratch (see below). */
#define SK_DECODE_NOALLOC_SCRATCH_BYTES (4u << 20)

/* sk_decode_attention for callers that cannot allocate device memory.
 * The source pages have no counterpart to this call: it exists for callers that
 * must not call cudaMalloc or any allocating routine, for example a serving loop
 * whose device memory is fully carved up by its own pool at start-up, a plug-in that
 * runs inside a host application that owns all device allocations, or a runtime
 * with a no-allocation rule on its steady-state path.  It does the same work with
 * the same arguments, minus the workspace: the scratch comes from one fixed
 * SK_DECODE_NOALLOC_SCRATCH_BYTES (4 MiB) array in device memory that the library
 * declares statically, so every GPU that loads the library holds those 4 MiB until
 * the process exits.
 *   - Set-up: the first call on each device (with that device current) looks up the
 *     array's device address once; make that first call before any stream capture.
 *   - Limit: the scratch needed grows with batch * n_kv_heads (about
 *     (152 + batch * n_kv_heads) * n_q_heads/n_kv_heads * (head_dim + 2) * 4 bytes);
 *     when it exceeds the array the call launches nothing and returns
 *     SK_ERR_CAPACITY.  Use sk_decode_attention with your own workspace then.
 *   - Sharing: every call uses the same array.  Calls that may overlap on the GPU
 *     (on different streams without ordering) race on it and give wrong results;
 *     serialise them on one stream.  Each call writes every scratch word it reads,
 *     so the contents left by an earlier call never matter.
 * Allocates nothing: no cudaMalloc, cudaFree or allocating library routine. */
SK_API sk_status sk_decode_attention_noalloc(const sk_kv_layer* layer, const void* q_rot,
                                             int32_t n_q_heads, int32_t io_dtype,
                                             const float* sink_logits, void* out, void* stream);

/* ---- Decode step: RoPE + append + attention in two kernels ------------------------- */

/* Workspace bytes sk_decode_step needs for `layer` and n_q_heads (0: unsupported). */
SK_API size_t sk_decode_step_workspace_bytes(const sk_kv_layer* layer, int32_t n_q_heads);

/* One decode token per sequence: sk_kv_append with T = 1 followed by
 * sk_decode_attention, with the append folded into the attention's two kernels, so a
 * step is one split kernel and one combine instead of three launches ([MIXED] 4.3-4.4:
 * at decode the step is bound by the KV bytes it streams; the separate append was a
 * launch and a hand-off of its own for a few KB).  The results are the same bits as
 * those two calls: the key is rotated and stored with the append's arithmetic and its
 * state rules (slot, head, count, pos, the SK_DEVERR_POSITION_RANGE and
 * SK_DEVERR_CAPACITY refusals), q is rotated the same way, and the attention reads the
 * same rows in the same order.  Differences: q and k are NOT rotated in place (they are
 * read only), and a ring head outside [0, window) is refused with SK_DEVERR_STATE
 * instead of being written through.
 *   table: the RoPE table (head_dim as the layer's); NULL: q and k come rotated and are
 *      used as given (no position limit but the counter's own).
 *   q: [batch][n_q_heads][head_dim] of io_dtype, device, read only.
 *   k, v: [batch][n_kv_heads][head_dim] of io_dtype, device, read only.
 *   out: [batch][n_q_heads][head_dim] of io_dtype, device; may alias q.
 *   sink_logits, workspace: as sk_decode_attention, with
 *      sk_decode_step_workspace_bytes(layer, n_q_heads) bytes of workspace.
 * The state (head, count, pos) changes in the second kernel; until the call's work is
 * done on the stream nothing else may read or write this layer.
 * Supported: ring and global layers with io SK_BF16 and a BF16/BF16 cache, or io
 * SK_F32 and an F32/F32 cache (int8 K caches: sk_kv_append + sk_decode_attention);
 * n_q_heads / n_kv_heads as sk_decode_attention. */
SK_API sk_status sk_decode_step(const sk_rope_table* table, const sk_kv_layer* layer, const void* q,
                                int32_t n_q_heads, const void* k, const void* v, int32_t io_dtype,
                                const float* sink_logits, void* out, void* workspace, size_t ws_bytes,
                                void* stream);

/* ---- Prefill attention (causal + window + sinks) ---------------------------------- */

/* Keys a chunk starting at position p0 takes from a prior cache: with window > 0 the
 * first s0 = min(sinks, p0) positions and then the last min(window - 1, p0 - s0)
 * positions before p0 (all its queries can see); with window <= 0 all p0 of them.
 * -1 for p0 < 0 or sinks < 0. */
SK_API int64_t sk_prefill_prior_keys(int64_t p0, int32_t sinks, int32_t window);

/* Workspace bytes sk_prefill_attention needs: with prior_keys > 0 (sk_prefill_prior_keys
 * of a call that passes a prior) a copy of the prior's keys and values, padded with zero
 * rows to a multiple of 64 (the chunk's own keys and values are read in place); without
 * a prior, or with T = 0, no scratch is used and the answer is a token 16 bytes.  0 for
 * an unsupported shape. */
SK_API size_t sk_prefill_workspace_bytes(int32_t batch, int32_t T, int32_t n_kv_heads, int32_t head_dim,
                                         int64_t prior_keys);

/* Masked attention of a prompt chunk on the tensor cores, over the chunk itself and,
 * optionally, over the keys a prior cache holds for the same sequences.
 *   q_rot: [batch][T][n_q_heads][head_dim], k_rot, v: [batch][T][n_kv_heads][head_dim],
 *   out: [batch][T][n_q_heads][head_dim]; all SK_BF16, device, 16-byte aligned.
 *   sink_logits: NULL, or device float32 [n_q_heads] learned sinks, as for
 *   sk_decode_attention (clamped to [-10, 15], denominator only).
 * Chunk index t has absolute position p0 + t.  A query at position P sees a key at
 * position k iff k <= P and (k < sinks or P - k < window) ([MIXED] 5.5: idx_q >= idx_k
 * and idx_q - idx_k < window; [SINK] sink + recent).  window <= 0 means a global layer
 * (causal only).  Only key tiles the mask leaves at least partly visible are visited.
 * q head h reads kv head h / (n_q_heads / n_kv_heads).
 *   prior: NULL, or the layer whose cache holds positions [0, p0) of every sequence
 *   (pos[b] == p0; the chunk has not been appended yet).  The keys before p0 come
 *   from it ([MIXED] 5.5: a multi-token chunk over a cached prefix, query index offset
 *   by T_k - T_q).  Without a prior, keys before p0 are not seen.  A ring prior must
 *   have the call's sinks and window (window > 0) and a count of
 *   min(window, p0 - min(sinks, p0)), as appends through this library leave it; a
 *   global prior needs p0 <= capacity (SK_ERR_CAPACITY otherwise).  K and V bf16, same
 *   batch, n_kv_heads and head_dim.
 *   A device state that does not match p0 sets SK_DEVERR_STATE in *err; the result
 *   is then undefined, and every read stays inside the cache.
 *   workspace: device, >= sk_prefill_workspace_bytes(batch, T, n_kv_heads, head_dim,
 *   prior ? sk_prefill_prior_keys(p0, sinks, window) : 0) bytes, 16-byte aligned, no
 *   initialisation needed.  err: device error word (SK_DEVERR_TIMEOUT if a bounded
 *   in-kernel wait gave up, SK_DEVERR_STATE as above), may be NULL.
 * Supported: head_dim 128, SK_BF16, T + prior keys (padded to a multiple of 64) <= 2^30.  T = 0 checks the other
 * arguments, launches nothing and returns SK_OK; q_rot, k_rot, v, out and workspace
 * may then be NULL. */
SK_API sk_status sk_prefill_attention(const void* q_rot, const void* k_rot, const void* v, int32_t batch,
                                      int32_t T, int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim,
                                      int64_t p0, int32_t sinks, int32_t window, const sk_kv_layer* prior,
                                      const float* sink_logits, void* out, void* workspace, size_t ws_bytes,
                                      uint32_t* err, void* stream);

/* ---- Cached-key rerotation on a factor change ------------------------------------ */

/* Turn every cached key of `layers` (host array of n_layers descriptors, device
 * buffers) from table `from` (factor A) to table `to` (factor B), in place:
 * each rotary pair at position P is turned by P (omega_B - omega_A) and scaled by
 * mu_B / mu_A, computed from the two tables' entries with R_a R_b = R_{a+b}
 * ([DYN] "The cached keys follow a change"; [SINK] RoPE section).  The tail dims
 * are unchanged.  An int8 K row is dequantised (code * scale), turned and
 * requantised with a new scale = max|x| / 127 and codes rint(x * (127 / max|x|))
 * (half to even), clamped to [-127, 127].
 * Positions come from the layer state: global slot s < pos[b] holds position s;
 * ring sink slot s < min(pos, S) holds s; ring slot j < count holds
 * pos - 1 - ((head - 1 - j) mod window).  Both tables must share head_dim,
 * rotary_dim, pairing and theta, and cover every cached position (else
 * SK_DEVERR_POSITION_RANGE for the row, which stays unchanged).
 * k_dtype SK_BF16 or SK_I8.  n_layers <= 128. */
SK_API sk_status sk_kv_rerotate(const sk_kv_layer* layers, int32_t n_layers, const sk_rope_table* from,
                         const sk_rope_table* to, void* stream);

/* ---- Paged caches ------------------------------------------------------------------ */

/* sk_kv_append for a paged layer: rotate q (optional, in place) and k (in place) at
 * positions seq_lens[b] + t and write k, v into the pool slots the block table gives
 * (block block_table[b][P / block_size], row P % block_size of each kv head);
 * seq_lens[b] += T.  The blocks for the new tokens must be in the table.  A request
 * whose seq_lens[b] + T exceeds max_blocks * block_size, or whose positions pass the
 * table, is skipped with SK_DEVERR_CAPACITY / SK_DEVERR_POSITION_RANGE; a token whose
 * block id is outside [0, n_blocks) is not stored and sets SK_DEVERR_BLOCK_TABLE.
 * Layouts, dtypes and T = 0 as sk_kv_append. */
SK_API sk_status sk_paged_append(const sk_rope_table* table, const sk_paged_layer* layer, void* q,
                                 int32_t n_q_heads, const void* k, const void* v, int32_t io_dtype, int32_t T,
                                 void* stream);

/* Workspace bytes sk_paged_decode_attention needs. */
SK_API size_t sk_paged_decode_workspace_bytes(const sk_paged_layer* layer, int32_t n_q_heads);

/* sk_decode_attention over a paged layer: one query per request (after its own
 * append) against the visible keys of its logical key sequence (see sk_paged_layer),
 * gathered block by block.  Only blocks holding visible keys are read; a visible key
 * whose block id is outside [0, n_blocks) reads block 0 instead and sets
 * SK_DEVERR_BLOCK_TABLE.  A request with seq_lens[b] = 0 gets zeros.  Arguments,
 * dtypes, learned sink logits and workspace rules as sk_decode_attention. */
SK_API sk_status sk_paged_decode_attention(const sk_paged_layer* layer, const void* q_rot, int32_t n_q_heads,
                                           int32_t io_dtype, const float* sink_logits, void* out,
                                           void* workspace, size_t ws_bytes, void* stream);

/* ---- Local-position caches: turn the recent keys on a window slide ---------------- */

/* Turn every occupied recent (ring) key of the ring layers `layers` (host array of
 * n_layers descriptors, device buffers) by `delta` positions, in place: each rotary
 * pair is multiplied by R(delta w_j) of `table`'s frequencies, with no mscale change;
 * sink slots [0, sinks), empty ring slots, the tail dims and all values are left
 * untouched.  This is the rerotation a cache needs when it feeds attention local
 * positions in [0, C-1] and its window slides: recent keys move from local p to
 * p - 1, i.e. delta = -(keys evicted), while the sink keys keep their local
 * positions ([SINK] "RoPE：absolute positions 与 local rerotation 是两种实现",
 * R_a R_b = R_{a+b}: no raw key needed).  A cache holding absolute positions (the
 * rest of this library) never needs it.  int8 rows are requantised as in
 * sk_kv_rerotate.  Errors: SK_ERR_ARG for a global layer or bad descriptors,
 * SK_ERR_POSITION_RANGE if |delta| >= table max_positions; delta = 0 launches
 * nothing.  k_dtype SK_BF16 or SK_I8, n_layers <= 128. */
SK_API sk_status sk_kv_shift_recent(const sk_kv_layer* layers, int32_t n_layers, const sk_rope_table* table,
                                    int32_t delta, void* stream);

/* ---- Misc ------------------------------------------------------------------------ */

/* Read a device error word after the work queued on `stream` (synchronises it).
 * *bits_out (may be NULL) gets the SK_DEVERR_* bits; with clear != 0 the word is reset
 * to zero afterwards.  Returns SK_OK when no bit is set, else the status of the most
 * specific condition: SK_ERR_CAPACITY, SK_ERR_POSITION_RANGE, SK_ERR_ARG (a paged block
 * id outside the pool, or a prefill's prior cache state that did not match its p0),
 * SK_ERR_CUDA (a bounded in-kernel wait gave up), in that order.
 * [MIXED] "KV-Cache Engineering", 4.6: a cache overflow fails loudly, never by silent
 * truncation; this is how a C caller hears it. */
SK_API sk_status sk_sync_check(uint32_t* err, int32_t clear, void* stream, uint32_t* bits_out);

/* Diagnostic: launch one thread that waits, through the library's bounded in-kernel
 * wait, on an mbarrier that never completes.  After the wait's limit (about one
 * second) it gives up, ORs SK_DEVERR_TIMEOUT into *err (device) and exits: the same
 * path every pipelined kernel takes if a copy never lands, so a caller can check that
 * such a failure is reported and leaves the context usable.  Asynchronous on
 * `stream`; SK_ERR_ARG for err == NULL. */
SK_API sk_status sk_selftest_bounded_wait(uint32_t* err, void* stream);

/* Diagnostic: run sk_prefill_attention's pipeline on a global causal chunk (p0 = 0, no
 * sinks, no window, no prior) in which the softmax warps never signal that P of tile
 * stall_tile (0-based, in each block's visiting order) is ready.  Every block that
 * visits that tile stalls: its P.V issuer's bounded wait gives up after about one
 * second, every later wait of the block gives up within a few polls, the MMAs and
 * copies already issued drain (each drain wait bounded), the block frees its tensor
 * memory and ORs SK_DEVERR_TIMEOUT into *err (device).  Blocks with fewer tiles finish
 * normally.  The output is undefined.  Same arguments, layouts and checks as
 * sk_prefill_attention (workspace >= sk_prefill_workspace_bytes(batch, T, n_kv_heads,
 * head_dim, 0)); SK_ERR_ARG for err == NULL or stall_tile < 0.  Asynchronous on
 * `stream`. */
SK_API sk_status sk_selftest_prefill_stall(const void* q_rot, const void* k_rot, const void* v, int32_t batch,
                                           int32_t T, int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim,
                                           void* out, void* workspace, size_t ws_bytes, int32_t stall_tile,
                                           uint32_t* err, void* stream);

/* A static, human-readable name for a status code. */
SK_API const char* sk_status_str(sk_status status);

/* Library version as major*10000 + minor*100 + patch. */
SK_API int32_t sk_version(void);

#ifdef __cplusplus
}
#endif

#endif /* SINKKV_H */

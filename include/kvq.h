/*
 * kvq.h -- C ABI of the rotated 4-bit KV-cache decode path (GB300, sm_103a).
 *
 * Method: "Serving Kolibri-1 with a 4-bit KV cache" (sevren.ai), section "What we do":
 * every key of a full-attention layer is rotated by a fixed randomized Hadamard matrix
 * R = H diag(s)/sqrt(128) after its RMS norm, stored as 4-bit codes with one fp16 scale
 * and one fp16 offset per token and head (4.25 bits per number); values are stored the
 * same way without rotation; queries are rotated by the same R with both QK-norm gains
 * folded in, and decode attention reads the 4-bit codes directly. The 40 sliding-window
 * layers (window 513) keep a stock FP8 e4m3 cache, read by the same kernel family.
 *
 * Conventions for every entry point:
 *  - All pointers are owned by the caller; the library allocates nothing. Pointers
 *    documented as "device" must be device-accessible memory of the current device;
 *    "host" pointers are ordinary CPU memory.
 *  - Calls taking a stream are asynchronous on that stream and never synchronise.
 *  - Host-side checks run first; on failure the call returns a non-zero kvq_status and
 *    launches nothing.
 *  - Problems only visible on the device (a block-table entry outside the page pool, a
 *    position beyond capacity, a non-finite input, an fp16 scale or offset that had to
 *    saturate, a bounded wait that gave up) are OR-ed into *dev_err as KVQ_DEVERR_* bits;
 *    the affected token-heads or pages are skipped. Kernels never trap and never spin
 *    without a time limit. The caller reads *dev_err after synchronising.
 *  - Kernels are launched with programmatic stream serialisation, so a call's first kernel
 *    may start while the previous kernel on the stream is still running. Until that kernel
 *    has completed it reads none of the call's inputs except the folded prologue weights
 *    (Mq, Mk and their FWHT multipliers), which the int4 calls stage on chip first. Those
 *    must be complete when the call is made: written by a host copy, by an ordinary kernel,
 *    or by a kernel that allows dependent launch only after writing them. Within a call each
 *    kernel waits for the one before it before reading anything that kernel writes.
 *  - Fixed geometry: head_dim 128, 64 tokens per page.
 *  - Thread-safe: no mutable global state beyond per-device attribute caches and the
 *    test-only wait limit of kvq_set_stage_wait_limit_ns.
 */
#ifndef KVQ_H
#define KVQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The same type as cudaStream_t; 0 is the legacy default stream. */
typedef struct CUstream_st* kvq_stream_t;

typedef enum kvq_status {
  KVQ_OK = 0,
  KVQ_ERR_INVALID_ARG = 1, /* null pointer, bad size, misaligned buffer, workspace too small */
  KVQ_ERR_UNSUPPORTED = 2, /* head_dim != 128, page_size != 64, S outside 1..8, too many rows */
  KVQ_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed */
  KVQ_ERR_SCRATCH_TOO_SMALL = 4 /* kvq_decode_attn_int4_noalloc: request needs more than its fixed scratch */
} kvq_status;

typedef enum kvq_dtype { KVQ_F32 = 0, KVQ_BF16 = 1 } kvq_dtype;

#define KVQ_HEAD_DIM 128
#define KVQ_PAGE_SIZE 64
#define KVQ_MAX_SEQS 1024

/* bits of *dev_err */
#define KVQ_DEVERR_PAGE 0x1      /* block-table entry outside [0, num_pages) */
#define KVQ_DEVERR_POS 0x2       /* sequence id or position outside the cache */
#define KVQ_DEVERR_NONFINITE 0x4 /* NaN/Inf in a key, value or query row (row skipped) */
#define KVQ_DEVERR_RANGE 0x8     /* fp16 scale or offset saturated at +-65504 */
#define KVQ_DEVERR_TIMEOUT 0x10  /* a bounded wait on a copy gave up (results invalid) */

/*
 * Paged int4 cache of one full-attention layer.
 * Physical layout: one contiguous 8704-byte block per (page, KV head), so that one bulk copy
 * moves a page of one head into shared memory:
 *   pages: [num_pages][num_kv_heads][8704] bytes (device, 16-byte aligned); within a block
 *     bytes    0..4095  K codes [64 tokens][64 bytes]
 *     bytes 4096..8191  V codes [64 tokens][64 bytes]
 *     bytes 8192..8447  K meta  [64 tokens] uint32
 *     bytes 8448..8703  V meta  [64 tokens] uint32
 *   A K record: byte b holds code 2b in its low nibble and code 2b+1 in its high nibble; its
 *     four 16-byte chunks are stored in XOR order: logical chunk c of token slot t at physical
 *     chunk c ^ (((t >> 1) & 1) | ((t >> 2) & 2)).
 *   A V record: 32 little-endian 16-bit elements; element l holds dims 4l..4l+3, each code c
 *     as a sign bit (c < 8) and a 3-bit magnitude e (7 - c if the sign is set, else c - 8),
 *     so that c - 7.5 = (sign ? -1 : 1) * (e + 0.5). Field bits (e, sign) per dim:
 *     dim 4l: 1-3, 15; dim 4l+1: 4-6, 14; dim 4l+2: 11-13, 7; dim 4l+3: 8-10, 0. With these
 *     positions one lop3 on the element, on it shifted left by 1, on its bytes swapped, or on
 *     those shifted left by 7, gives an f16 subnormal of (c - 7.5) times a power of two.
 *   In V records the four 16-byte chunks of token slot t (0..63)
 *   are stored in XOR order: logical chunk c at physical chunk c ^ ((t >> 1) & 3), so a
 *   transposing shared-memory read of eight consecutive tokens touches eight bank groups.
 *   A meta word: bits 0..15 the fp16 scale, bits 16..31 the fp16 offset; value = code*scale + offset.
 *   block_table: [num_seqs][max_pages_per_seq] int32 (device): physical page of logical
 *     page p of sequence q; position `pos` lives in page pos/64, slot pos%64.
 */
#define KVQ_INT4_BLOCK_BYTES 8704

typedef struct kvq_int4_cache {
  uint8_t* pages;
  const int32_t* block_table;
  int32_t num_seqs;
  int32_t max_pages_per_seq;
  int32_t num_pages;
  int32_t num_kv_heads;
  int32_t page_size; /* must be 64 */
  int32_t head_dim;  /* must be 128 */
} kvq_int4_cache;

/*
 * FP8 e4m3 ring cache of one sliding-window layer (stock format: one fp32 scale per
 * tensor). Position `pos` of sequence q, head h lives in slot pos % capacity. The ring is
 * stored in blocks of 64 slots, keys then values, one contiguous 16384-byte block each:
 *   data: [num_seqs][num_kv_heads][capacity/64][2 (K, V)][64 slots][128] bytes (device,
 *   16-byte aligned); the eight 16-byte chunks of the record in slot t are stored at
 *   physical chunk c ^ (t & 7).
 * capacity must be a multiple of 64 and at least window + S - 1 for the calls using it.
 */
typedef struct kvq_fp8_ring {
  uint8_t* data;
  int32_t num_seqs;
  int32_t num_kv_heads;
  int32_t capacity;
  int32_t head_dim; /* must be 128 */
} kvq_fp8_ring;

/* Human-readable name of a status code (static string). */
const char* kvq_status_string(kvq_status status);

/*
 * kvq_build_rotation -- section "What we do": R = H diag(s)/sqrt(128), H the Sylvester
 * Hadamard matrix, s a random sign per column: s[j] = +1 when the top bit of the j-th
 * output of splitmix64 seeded with `seed` is 0, else -1. Entries computed in fp64 and
 * rounded to fp32.
 *   s_out: host int8[head_dim] (may be NULL); R_out: host float[head_dim*head_dim], row-major.
 * Returns KVQ_ERR_UNSUPPORTED unless head_dim == 128, KVQ_ERR_INVALID_ARG if R_out is NULL.
 */
kvq_status kvq_build_rotation(uint64_t seed, int head_dim, int8_t* s_out, float* R_out);

/*
 * kvq_fold_qk -- section "What we do", QK-norm gain folding: scores depend only on q.k,
 * so g_k moves to the query side and the cache holds R n(k):
 *   M_q = R diag(g_q * g_k)  (each entry the fp64 product R[j][i]*(g_q[i]*g_k[i]) rounded
 *   once to fp32),  M_k = R.
 *   R, g_q, g_k: host inputs (row-major R); Mq_out, Mk_out: host float[128*128] outputs.
 */
kvq_status kvq_fold_qk(const float* R, const float* g_q, const float* g_k, int head_dim, float* Mq_out,
                       float* Mk_out);

/*
 * kvq_fold_qk_fwht -- the same rotation and gain fold for the fast Walsh-Hadamard prologue
 * (kvq_rotate_quant_append_fwht, kvq_decode_attn_int4_fwht). Because R = H diag(s)/sqrt(128),
 * R n = H (s n)/sqrt(128) and R diag(g_q g_k) n = H (s g_q g_k n)/sqrt(128): the folded form is
 * one multiplier per channel in front of H.
 *   s: host int8[128] of +1/-1 (from kvq_build_rotation); g_q, g_k: host float[128].
 *   wq_out[i] = s[i]*g_q[i]*g_k[i] (fp64 product rounded once to fp32); wk_out[i] = s[i].
 * Returns KVQ_ERR_INVALID_ARG for a NULL pointer or an s entry other than +1/-1.
 */
kvq_status kvq_fold_qk_fwht(const int8_t* s, const float* g_q, const float* g_k, int head_dim, float* wq_out,
                            float* wk_out);

/*
 * kvq_rotate_quant_append -- section "What we do": keys rotated (with their RMS norm) by
 * M_k and values unrotated, each quantised to 4-bit codes with fp16 scale/offset per
 * token and head, written into the page slot of (seq_ids[t], positions[t]).
 *   Mk:        device float[128*128] row-major (y = M_k n(k)).
 *   k, v:      device [T][num_kv_heads][128] of `dtype` (pre-norm keys, raw values).
 *   seq_ids, positions: device int32[T].
 * Arithmetic (bit-exact specification, fp32, IEEE operations in this order):
 *   lanes l=0..31 hold x[4l..4l+3]; t_l = fma(x3,x3,fma(x2,x2,fma(x1,x1,x0*x0)));
 *   t_l <- t_l + t_(l^o) for o = 16,8,4,2,1; inv = 1/sqrt(t/128 + eps); n = x*inv;
 *   y_j = fma chain over i=0..127 of M[j][i]*n_i;
 *   o = fp16 toward -inf of min(y); s = fp16 toward +inf of (max(y)-o)/15 (a zero o or s is
 *   stored as +0; an o below -65504 or an s above 65504 saturates there, KVQ_DEVERR_RANGE);
 *   code_i = 0 if s == 0 else clamp(round_half_even((y_i - o)/s), 0, 15).
 * Values use the same quantiser on the raw row. T == 0 is a no-op.
 */
kvq_status kvq_rotate_quant_append(const kvq_int4_cache* cache, const float* Mk, const void* k, const void* v,
                                   kvq_dtype dtype, int T, const int32_t* seq_ids, const int32_t* positions,
                                   float eps, int32_t* dev_err, kvq_stream_t stream);

/*
 * kvq_rotate_quant_append_fwht -- kvq_rotate_quant_append with the second prologue
 * specification: y = c FWHT(wk n(k)), c = fp32(1/sqrt(128)) (R n(k) up to rounding).
 *   wk: device float[128], 16-byte aligned (kvq_fold_qk_fwht's wk_out).
 * Arithmetic (bit-exact specification, fp32): n(k) as in kvq_rotate_quant_append; u_i = wk_i*n_i;
 *   for h = 1, 2, 4, ..., 64 and every i with (i & h) == 0: (u_i, u_i+h) <- (u_i + u_i+h, u_i - u_i+h);
 *   y_j = c*u_j; then the same quantiser. Values as in kvq_rotate_quant_append.
 */
kvq_status kvq_rotate_quant_append_fwht(const kvq_int4_cache* cache, const float* wk, const void* k, const void* v,
                                        kvq_dtype dtype, int T, const int32_t* seq_ids, const int32_t* positions,
                                        float eps, int32_t* dev_err, kvq_stream_t stream);

/*
 * Bytes of device workspace needed by kvq_decode_attn_int4 / kvq_decode_attn_fp8_swa for
 * B sequences, S query rows each, num_q_heads query heads over num_kv_heads KV heads.
 * Returns 0 for arguments no call would accept.
 */
size_t kvq_decode_workspace_bytes(int B, int S, int num_q_heads, int num_kv_heads);

/*
 * kvq_decode_attn_int4 -- split-K flash-decoding attention over the int4 cache (section
 * "What we do": decode reads the 4-bit codes directly, nothing is rotated back).
 *   Sequence b (0..B-1) uses block-table row b and has ctx_len[b] cached positions.
 *   Query row r (0..S-1) sits at position ctx_len[b] + r and attends causally to
 *   positions 0..ctx_len[b]+r (a speculative-decoding verify block when S > 1).
 *   q:        device [B][S][num_q_heads][128] of `dtype`, pre-norm queries; the call applies
 *             q~ = M_q n(q) with the prologue arithmetic above. Query head hq reads KV head
 *             hq / (num_q_heads/num_kv_heads).
 *   k_new, v_new: device [B][S][num_kv_heads][128] of `dtype`, or both NULL. When given, the
 *             S rows are rotated, quantised and appended at positions ctx_len[b]+r first.
 *   Mq, Mk:   device float[128*128] (Mk only read when k_new is given).
 *   sm_scale: softmax scale applied to q~.k (1/sqrt(128) for the model).
 *   out:      device float [B][S][num_q_heads][128], the normalised attention output.
 *   workspace: device, >= kvq_decode_workspace_bytes(B, S, num_q_heads, num_kv_heads),
 *             256-byte aligned; contents need no initialisation.
 *   q_rot_out: optional device float [B][S][num_q_heads][128] copy of q~ (NULL to skip).
 * Requires 1 <= B <= KVQ_MAX_SEQS, 1 <= S <= 8, S*(num_q_heads/num_kv_heads) <= 48.
 */
kvq_status kvq_decode_attn_int4(const kvq_int4_cache* cache, const float* Mq, const float* Mk, const void* q,
                                kvq_dtype dtype, int B, int S, int num_q_heads, const int32_t* ctx_len,
                                const void* k_new, const void* v_new, float sm_scale, float eps, float* out,
                                void* workspace, size_t workspace_bytes, float* q_rot_out, int32_t* dev_err,
                                kvq_stream_t stream);

/*
 * kvq_decode_attn_int4_fwht -- kvq_decode_attn_int4 with the FWHT prologue for the queries
 * (q~ = c FWHT(wq n(q)) in the fp32 order of kvq_rotate_quant_append_fwht) and, when
 * k_new/v_new are given, for the appended keys. The cache must have been filled with the FWHT
 * prologue too (kvq_rotate_quant_append_fwht) for the scores to match R's rotation on both sides.
 *   wq, wk: device float[128], 16-byte aligned (kvq_fold_qk_fwht); wk only read with k_new.
 * All other arguments, limits and errors as kvq_decode_attn_int4.
 */
kvq_status kvq_decode_attn_int4_fwht(const kvq_int4_cache* cache, const float* wq, const float* wk, const void* q,
                                     kvq_dtype dtype, int B, int S, int num_q_heads, const int32_t* ctx_len,
                                     const void* k_new, const void* v_new, float sm_scale, float eps, float* out,
                                     void* workspace, size_t workspace_bytes, float* q_rot_out, int32_t* dev_err,
                                     kvq_stream_t stream);

/*
 * kvq_fp8_append -- stock FP8 cache write of the sliding-window layers: code =
 * e4m3(x / scale) with an IEEE fp32 division, round-to-nearest-even, saturating to +-448,
 * into slot positions[t] % capacity of sequence seq_ids[t]. Rows with a non-finite entry
 * are skipped (KVQ_DEVERR_NONFINITE).
 *   k, v: device [T][num_kv_heads][128] of `dtype`; seq_ids, positions: device int32[T].
 */
kvq_status kvq_fp8_append(const kvq_fp8_ring* ring, const void* k, const void* v, kvq_dtype dtype, int T,
                          const int32_t* seq_ids, const int32_t* positions, float k_scale, float v_scale,
                          int32_t* dev_err, kvq_stream_t stream);

/*
 * kvq_decode_attn_fp8_swa -- sliding-window attention over the FP8 ring (the stock path of
 * the 40 window-513 layers). Row r of sequence b sits at position pos0[b] + r and attends
 * to positions max(0, pos0[b]+r-window+1) .. pos0[b]+r, dequantised as e4m3(c)*k_scale and
 * e4m3(c)*v_scale. q is used as given (no prologue).
 *   q: device [B][S][num_q_heads][128] of `dtype`; out: device float [B][S][num_q_heads][128].
 *   k_new, v_new: device [B][S][num_kv_heads][128] of `dtype` or both NULL; when given they
 *     are written (kvq_fp8_append arithmetic) at positions pos0[b]+r before attending.
 *   workspace: as for kvq_decode_attn_int4.
 * Requires 1 <= B <= KVQ_MAX_SEQS, 1 <= S <= 8, window >= 1, capacity >= window + S - 1.
 */
kvq_status kvq_decode_attn_fp8_swa(const kvq_fp8_ring* ring, const void* q, kvq_dtype dtype, int B, int S,
                                   int num_q_heads, const int32_t* pos0, int window, const void* k_new,
                                   const void* v_new, float k_scale, float v_scale, float sm_scale, float* out,
                                   void* workspace, size_t workspace_bytes, int32_t* dev_err,
                                   kvq_stream_t stream);

/*
 * kvq_fp8_swa_plan -- the launch shape kvq_decode_attn_fp8_swa takes for these sizes on the
 * calling thread's current device; no launch, nothing allocated (reads device attributes and
 * the kernel's occupancy, cached per device).
 *   out[0]: CTAs per (sequence, KV head): the cluster size of the one-launch path, which
 *           appends and attends in one kernel and merges on chip; 1 also for the
 *           one-CTA-per-pair shape taken when the call has at least as many (sequence, KV head)
 *           pairs as the device has SMs; 0 where the one-launch path does not fit (rings
 *           beyond one cluster; 40 or more query rows per KV head with fewer pairs than SMs),
 *           which takes a separate append, the split-K kernel and its combine pass.
 *   out[1]: unit streams (warps per query-tile group) per CTA; out[2]: copy stages per stream;
 *   out[3]: 32-slot ring units per stream (the largest; 0 with out[0] = 0).
 * Returns KVQ_ERR_INVALID_ARG / KVQ_ERR_UNSUPPORTED under the same conditions on these
 * arguments as kvq_decode_attn_fp8_swa (capacity a positive multiple of 64).
 */
kvq_status kvq_fp8_swa_plan(int capacity, int B, int S, int num_q_heads, int num_kv_heads, int32_t out[4]);

/*
 * kvq_set_stage_wait_limit_ns -- test hook for the failure path of the bounded waits: sets, for
 * every later launch in the process, how long the split-K attention kernel of
 * kvq_decode_attn_int4 (and of the window path's split-K form) waits for a page's copy into a
 * shared-memory stage, and for a stage to be released, before it gives up, sets
 * KVQ_DEVERR_TIMEOUT and abandons the call's remaining pages (outputs then invalid). ns = 0 gives
 * up at the first unsuccessful check. The wait for copies still in flight before a CTA exits
 * always keeps the default. Default 2000000000 (2 s); the default is what a caller should run
 * with. Always returns KVQ_OK.
 */
kvq_status kvq_set_stage_wait_limit_ns(uint64_t ns);

/*
 * kvq_decode_attn_int4_noalloc -- the same computation as kvq_decode_attn_int4 for callers
 * that cannot allocate device memory at decode time (an engine that hands all free GPU
 * memory to its KV pool at start-up, a thread that must not touch the device allocator, an
 * environment where cudaMalloc or a framework allocator is unavailable). The paper has no
 * counterpart: this is a packaging variant of the workspace handling only.
 * The workspace comes from a fixed scratch array inside this library's device image, of
 * KVQ_NOALLOC_SCRATCH_BYTES. The call allocates nothing; the caller still passes every input
 * and output.
 *   - Arguments, checks and results are those of kvq_decode_attn_int4 without (workspace,
 *     workspace_bytes): the same status for the same bad argument.
 *   - Requests with valid arguments whose workspace (kvq_decode_workspace_bytes) exceeds the
 *     scratch return KVQ_ERR_SCRATCH_TOO_SMALL and launch nothing.
 *   - When the memory is taken: under lazy module loading (the CUDA default) the first call on
 *     a device loads the module holding the array, and so allocates its 16 MiB there, while
 *     looking up its device address (with that device current); under eager loading the
 *     library's load does. The device keeps it until the process exits. Make the first call on
 *     each device before reserving the memory pool the engine hands out, and before any
 *     stream capture.
 *   - Every call looks the address up again (cheap once loaded), so calls stay valid across a
 *     cudaDeviceReset.
 *   - All calls on a device share the one scratch array, which keeps the last call's
 *     contents (no call needs it zeroed). Calls whose execution overlaps on the GPU race on
 *     it: serialise them (one stream, or explicit ordering between streams and threads).
 */
#define KVQ_NOALLOC_SCRATCH_BYTES (16u << 20)

kvq_status kvq_decode_attn_int4_noalloc(const kvq_int4_cache* cache, const float* Mq, const float* Mk, const void* q,
                                        kvq_dtype dtype, int B, int S, int num_q_heads, const int32_t* ctx_len,
                                        const void* k_new, const void* v_new, float sm_scale, float eps, float* out,
                                        float* q_rot_out, int32_t* dev_err, kvq_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H */

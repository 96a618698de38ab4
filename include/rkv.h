/*
 * rkv.h - C ABI of librkv, the ResidualKV cache codec for one GB300 (sm_103a).
 *
 * Method: "ResidualKV:基于参考向量与残差的 KV Cache 压缩" (study notes on
 * arXiv 2602.08005v2), cited as "ResidualKV notes §x".  The cache keeps a
 * sparse pool of reference tokens in FP8 and, for every other token, a short
 * quantised latent residual.  Writing a token retrieves its k nearest
 * references, averages them and stores z = f_c(kv) - f_c(mean) quantised per
 * group; reading a token restores KV_hat = dequant(z) W_d + mean, splits it
 * into K and V and applies RoPE to K at the token's own position.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - Pointers marked (device) are CUDA device pointers on the current device;
 *   pointers marked (host) are ordinary host memory read before the call
 *   returns.  No signature uses a framework type.
 * - Ownership: the caller allocates and frees the weights, the storage
 *   tensors (rkv_storage), all inputs and all outputs.  The library owns only
 *   the context, its repacked weight copies, RoPE tables, scratch and a
 *   pinned staging buffer; rkv_free releases exactly those.
 * - Streams: `stream` is a cudaStream_t passed as void* (NULL = legacy
 *   default stream).  Every call enqueues its work on that stream and returns
 *   without synchronising, except rkv_create and rkv_get_status.
 * - Errors: a negative rkv_status means nothing was launched (the message is
 *   available from rkv_last_error).  Problems only the device can see (an
 *   out-of-range selected position, a never-written token, a timed-out wait,
 *   an FP16 overflow of a group extreme) never trap: the kernel clamps or
 *   skips the row, writes zeros for it, and ORs a bit into the context's
 *   device status word, read by rkv_get_status.
 * - All dimensions are in elements unless a name ends in _bytes.
 */
#ifndef RKV_H
#define RKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  RKV_OK = 0,
  RKV_EINVAL = -1,      /* bad argument: shape, dtype, range, ordering       */
  RKV_EALIGN = -2,      /* a pointer is not 16-byte aligned                  */
  RKV_ECAPACITY = -3,   /* more tokens / references than the config allows   */
  RKV_EEMPTYPOOL = -4,  /* a non-reference token whose pool has no reference */
  RKV_ECUDA = -5,       /* a CUDA runtime call or kernel launch failed       */
  RKV_EDEVICE = -6,     /* rkv_get_status: the device status word is set     */
  RKV_ETIMEOUT = -7     /* rkv_get_status: a kernel wait gave up             */
} rkv_status;

/* element types */
enum { RKV_F32 = 0, RKV_BF16 = 1 };

/* bits of the device status word (rkv_get_status) */
enum {
  RKV_FLAG_TIMEOUT = 1,      /* a bounded spin-wait expired; the CTA stopped  */
  RKV_FLAG_BAD_INDEX = 2,    /* a selected (seq, pos) was out of range        */
  RKV_FLAG_UNWRITTEN = 4,    /* a selected token was never written            */
  RKV_FLAG_FP16_SAT = 8,     /* a group extreme saturated at +-65504          */
  RKV_FLAG_BAD_SLOT = 16     /* a pool slot outside [0, max_refs)             */
};

/*
 * Codec configuration.  Shapes follow ResidualKV notes §2.1 (d_k = N*D, the
 * joint vector kv_i has 2*d_k entries), §2.3 (d_c, d_ff), §2.4 (g, b) and §2.6
 * (the reference schedule, fixed or dynamic stride).  Limits of this build: head_dim in {64, 128}; 2*d_k a
 * multiple of 256; d_c a multiple of 64 and at most 512 (the decoder keeps a token
 * tile's z~ in tensor memory); d_ff a multiple of 128; topk in 1..4; group = 32; bits in {4, 2, 16} (16 =
 * quantisation off, z kept as bf16).
 */
typedef struct {
  int32_t n_kv_heads;        /* N                                              */
  int32_t head_dim;          /* D                                              */
  int32_t d_c;               /* latent code width                              */
  int32_t d_ff;              /* SwiGLU hidden width                            */
  int32_t topk;              /* k (the page's default is 4)                    */
  int32_t group;             /* g = 32                                         */
  int32_t bits;              /* 4, 2 or 16                                     */
  int32_t ref_stride;        /* s_0: the stride of the reference schedule      */
  int32_t kv_dtype;          /* RKV_F32 or RKV_BF16: input kv rows             */
  int32_t out_dtype;         /* RKV_F32 or RKV_BF16: restored K and V          */
  double rope_base;          /* theta_j = rope_base^(-2j/D)                    */
  int32_t batch;             /* number of sequences B                          */
  int32_t max_tokens;        /* T_cap: positions per sequence                  */
  int32_t max_refs;          /* R_cap: pool slots per sequence, at least the
                                schedule's positions below T_cap (0 = exactly
                                that many)                                    */
  int32_t max_rows;          /* rows one compress pass handles (0 = 32768);
                                larger calls are processed in passes          */
  double ref_alpha;          /* alpha >= 0: growth of the dynamic stride (0 =
                                fixed stride)                                 */
  int32_t ref_sink;          /* n_sink >= 0: sink tokens                       */
  int32_t mean_precompute;   /* 0: the encoder maps each token's reference mean
                                row (GEMM-1/2 over kv and mean rows); 1: it takes
                                the mean's pre-activations from the references'
                                own, kept beside the pool (mean W = (1/k) sum
                                r_j W, §2.3): rkv_pool_append computes
                                r [W_c1 | W_c2] in fp32 for each appended
                                reference (a context-owned table, 8 d_ff bytes
                                per pool slot), and rkv_compress's GEMM-1/2 runs
                                on kv rows only.  The mean is then never rounded
                                to a bf16 operand, so codes can differ from mode
                                0 by one near rounding boundaries.            */
} rkv_config;
/*
 * Reference schedule (ResidualKV notes §2.6): a position is a reference iff it
 * is one of the sink tokens 0 .. n_sink-1 or one of p_0 = n_sink,
 * p_{m+1} = p_m + s_0 + floor(alpha * (p_m - n_sink)) (the product in binary64).
 * alpha = 0, n_sink = 0 is the fixed stride: pos % s_0 == 0.  Pool slot m of a
 * sequence holds its m-th reference position.
 */

/*
 * Cache storage, allocated by the caller on the device and zero-filled or
 * not (rkv_create initialises what needs it).  Sizes in bytes are given by
 * rkv_storage_bytes.  All row-major; "row" = seq * T_cap + pos for token
 * tables and seq * R_cap + slot for pool tables.
 *   pool_fp8   [B, R_cap, 2d_k]  E4M3 references (ResidualKV notes §2.4, §3.3)
 *   pool_norm2 [B, R_cap]  fp32  squared norm of each decoded reference
 *   pool_pos   [B, R_cap]  int32 position of each reference, INT32_MAX = empty
 *   codes      [B, T_cap, code_bytes]  packed codes (d_c*b/8 bytes; 2*d_c
 *                                for bits = 16)
 *   meta       [B, T_cap, d_c/g, 2]  FP16 (min, max) of each group
 *   ref_idx    [B, T_cap, topk] int32  retrieved pool slots, nearest first,
 *                                -1 padded; a reference token stores
 *                                [its slot, -1, ...]
 */
typedef struct {
  void* pool_fp8;
  float* pool_norm2;
  int32_t* pool_pos;
  void* codes;
  void* meta;
  int32_t* ref_idx;
} rkv_storage;

/* Byte sizes of the six storage tensors, in the order of rkv_storage. */
rkv_status rkv_storage_bytes(const rkv_config* cfg, size_t sizes[6]);

/*
 * The reference positions of cfg's schedule below max_tokens (ResidualKV notes
 * §2.6; see rkv_config), in increasing order: the positions a caller passes to
 * rkv_pool_append, every other position going to rkv_compress.
 *   pos (host, caller-owned) receives the first min(capacity, count) positions;
 *   it may be NULL when capacity is 0.  *count (host) receives their number.
 * Errors: RKV_EINVAL (invalid cfg, capacity < 0, NULL count or NULL pos with
 * capacity > 0).  No device work.
 */
rkv_status rkv_reference_positions(const rkv_config* cfg, int32_t* pos, int32_t capacity,
                                   int32_t* count);

typedef struct rkv_ctx rkv_ctx;

/*
 * Create a codec context on the current device.
 *   Wc1, Wc2 (device, bf16) [2d_k, d_ff]; Wc3 (device, bf16) [d_ff, d_c];
 *   Wd (device, bf16) [d_c, 2d_k] - row-major, the row-vector convention of
 *   ResidualKV notes §2.3 (f_c) and §2.5 (f_d(z) = z W_d).  The library keeps
 *   its own repacked copies; the caller's weights may be freed afterwards.
 *   st: device storage (see rkv_storage); pointers must stay valid for the
 *   context's lifetime.  rkv_create marks every pool slot empty, every token
 *   row unwritten (ref_idx = -1) and synchronises `stream`.
 * Returns RKV_EINVAL for an unsupported config, RKV_EALIGN for a pointer not
 * 16-byte aligned, RKV_ECUDA if allocation or a launch fails.
 */
rkv_status rkv_create(const rkv_config* cfg, const void* Wc1, const void* Wc2,
                      const void* Wc3, const void* Wd, const rkv_storage* st,
                      void* stream, rkv_ctx** out);

/*
 * Append reference tokens to their sequences' pools (ResidualKV notes §2.6
 * reference schedule; §2.4 and §3.3: references are stored directly, in FP8).
 *   kv (device) rows of 2*d_k elements of cfg.kv_dtype; row r of the call
 *     reads kv + src_rows[r] * kv_row_stride (src_rows NULL: row r).
 *   src_rows, seq, pos (host) [n]; every pos must be a position of the
 *     schedule (see rkv_config), and per sequence the positions must continue
 *     the sequence's references in order (slot m = the m-th schedule position).
 * Writes pool_fp8/pool_norm2/pool_pos at the position's slot (and the context's
 * bf16 copy of the reference, see rkv_pool_cache) and the
 * token's own row: ref_idx = [slot, -1, ...], codes = 0, meta = 0.
 * Errors (nothing launched): RKV_EINVAL (range, not a reference position,
 * out of order), RKV_ECAPACITY (slot >= R_cap).
 */
rkv_status rkv_pool_append(rkv_ctx* ctx, const void* kv, int64_t kv_row_stride,
                           const int32_t* src_rows, const int32_t* seq,
                           const int32_t* pos, int32_t n, void* stream);

/*
 * Encode non-reference tokens (ResidualKV notes §2.2 retrieval and mean,
 * §2.3 z = f_c(kv) - f_c(mean), §2.4 group quantisation).
 *   kv, kv_row_stride, src_rows, seq, pos: as for rkv_pool_append; every pos
 *     must NOT be a reference position, and every reference of the sequence
 *     before pos must already have been appended (stream order).
 * Token i uses the references with position < pos_i, k_i = min(k, count),
 * ties to the smaller slot.  Writes ref_idx, codes and meta of each token.
 * Errors: RKV_EINVAL, RKV_EEMPTYPOOL (no reference before pos), RKV_ECAPACITY.
 */
rkv_status rkv_compress(rkv_ctx* ctx, const void* kv, int64_t kv_row_stride,
                        const int32_t* src_rows, const int32_t* seq,
                        const int32_t* pos, int32_t n, void* stream);

/*
 * Restore selected tokens (ResidualKV notes §2.5 KV_hat = z~ W_d + mean,
 * §2.1 K/V split and RoPE at the token's own position, §2.7 sparse read).
 *   seq, pos (device, int32) [n_sel]: the selected tokens, any order,
 *     duplicates allowed.
 *   k_out, v_out (device) [n_sel, N, D] of cfg.out_dtype: K (rotated) and V;
 *     32-byte aligned (RKV_EALIGN otherwise).  Only their first n_sel rows are
 *     written.
 * An out-of-range (seq, pos) or a never-written token yields zero rows and a
 * status bit (RKV_FLAG_BAD_INDEX / RKV_FLAG_UNWRITTEN).  n_sel = 0 is a no-op.
 */
rkv_status rkv_reconstruct(rkv_ctx* ctx, const int32_t* seq, const int32_t* pos,
                           int32_t n_sel, void* k_out, void* v_out, void* stream);

/*
 * Restore the selections of several contexts in one launch (ResidualKV notes §2.5,
 * §2.7: the same computation as one rkv_reconstruct per context).  Meant for the
 * layers of one decode step whose selections are all known before their restores
 * run (an index set chosen once per step for a group of sparse layers, as in the
 * OmniKV combination, or independent selections); a layer whose selection depends
 * on an earlier layer's attention must be restored by its own call.  One launch
 * saves each further restore its own start-up and tail.
 *   ctxs [n]: contexts of equal shape (N, D, d_c, topk, bits, batch, max_tokens,
 *     max_refs, out_dtype, rope_base) on one device; each restores from its own
 *     storage and W_d.  1 <= n <= 32.
 *   seq[i], pos[i] (device, int32) [n_sel[i]], k_out[i], v_out[i] (device)
 *     [n_sel[i], N, D]: as for rkv_reconstruct; n_sel[i] = 0 skips problem i.
 * Bad selections raise the status bits of their own context; a kernel wait that
 * times out is reported on ctxs[0].  The launch's timing is ctxs[0]'s; a call with
 * one non-empty problem runs rkv_reconstruct's kernel on that context.
 * Errors (nothing launched): RKV_EINVAL (NULL, n, mismatched contexts), RKV_EALIGN;
 * RKV_ECUDA.
 */
rkv_status rkv_reconstruct_multi(rkv_ctx* const* ctxs, int32_t n, const int32_t* const* seq,
                                 const int32_t* const* pos, const int32_t* n_sel,
                                 void* const* k_out, void* const* v_out, void* stream);

/*
 * Sparse-layer attention over restored K/V (ResidualKV notes §2.7, the output
 * equation o = softmax(q K_hat^T / sqrt(D)) V_hat over the selected tokens I_t).
 *   q (device, fp32) [n_q_heads, D]: the decode query, already rotated at its own
 *     position; query head h reads key/value head h / (n_q_heads / N).
 *   k, v (device, cfg.out_dtype) [n, N, D]: rows of rkv_reconstruct's outputs
 *     (the selected tokens of one sequence), 16-byte aligned.
 *   out (device, fp32) [n_q_heads, D].
 *   n_q_heads: a multiple of N, at most 8 N;  n in [1, 262144].
 * The softmax is fp32 with a per-chunk maximum; the library's workspace holds the
 * chunk partials, so calls on one context must not run concurrently.
 * Errors (nothing launched): RKV_EINVAL (sizes, NULL), RKV_EALIGN; RKV_ECUDA.
 */
rkv_status rkv_sparse_attention(rkv_ctx* ctx, const float* q, int32_t n_q_heads,
                                const void* k, const void* v, int32_t n, float* out,
                                void* stream);

/*
 * Restore fused into the sparse layer's attention (ResidualKV notes §2.7, Fig. 7: the
 * selected tokens I_t are restored and attended in one pass, o = softmax(q K_hat^T /
 * sqrt(D)) V_hat); the same result as rkv_reconstruct followed by rkv_sparse_attention,
 * without writing K_hat / V_hat to memory.
 *   seq, pos (device, int32) [n_sel]: the selected tokens (as for rkv_reconstruct).
 *   q (device, fp32) [n_q_heads, D]: the decode query, already rotated; query head h
 *     reads key/value head h / (n_q_heads / N).  8-byte aligned.
 *   out (device, fp32) [n_q_heads, D].
 *   n_q_heads: a multiple of N, at most 8 N;  n_sel in [1, min(262144, B * max_tokens)].
 * Needs head_dim = 128 and out_dtype = bf16: K_hat and V_hat are rounded to bf16 where
 * rkv_reconstruct would store them, the scores and the weights reach the tensor core as
 * bf16 high + low parts (relative error below 2^-16), sums are fp32.  The library's
 * workspace holds per-tile partials, so calls on one context must not run concurrently.
 * Bad selections raise the same status bits as rkv_reconstruct (their rows count as
 * zero K_hat / V_hat rows).
 * Errors (nothing launched): RKV_EINVAL (shape, dtype, sizes, NULL), RKV_EALIGN; RKV_ECUDA.
 */
rkv_status rkv_restore_attend(rkv_ctx* ctx, const int32_t* seq, const int32_t* pos,
                              int32_t n_sel, const float* q, int32_t n_q_heads, float* out,
                              void* stream);

/*
 * The context's bf16 copy of the reference pool: [B, R_cap, 2d_k], row
 * s * R_cap + slot holding the decoded E4M3 reference of that slot exactly (every E4M3
 * value is a bf16 value).  It is the tensor-core operand of retrieval, a compute cache
 * that rkv_pool_append keeps in step with pool_fp8, not part of the cache's storage;
 * the context owns it and rkv_free releases it.  *ptr (device) and *bytes receive its
 * address and size; read it only in stream order after the appends that wrote it.
 * Errors: RKV_EINVAL (NULL argument).
 */
rkv_status rkv_pool_cache(rkv_ctx* ctx, void** ptr, size_t* bytes);

/*
 * Forget everything written for one sequence (seq >= 0) or for all (seq = -1):
 * its pool slots become empty and its token rows unwritten, so the slot can
 * hold a new sequence (stream-ordered; codes and extremes are overwritten by
 * later writes).  Errors: RKV_EINVAL for seq out of range.
 */
rkv_status rkv_reset(rkv_ctx* ctx, int32_t seq, void* stream);

/*
 * Read and clear the device status word (stream-ordered copy, then the
 * stream is synchronised).  *flags receives the RKV_FLAG_* bits.  Returns
 * RKV_OK if no bit was set, RKV_ETIMEOUT if RKV_FLAG_TIMEOUT was set,
 * RKV_EDEVICE for any other bit, RKV_ECUDA if the copy failed.
 */
rkv_status rkv_get_status(rkv_ctx* ctx, int32_t* flags, void* stream);

/* Message of the last non-OK status returned on this thread. */
const char* rkv_last_error(void);

/* Release the context; NULL is allowed.  Never frees caller storage. */
void rkv_free(rkv_ctx* ctx);

/*
 * Retrieval that allocates nothing.  The page has no counterpart to this entry point:
 * it exists for callers that must not call the CUDA allocator - a serving runtime that
 * reserves all device memory up front in its own arena, or a step that must not pay
 * cudaMalloc's implicit device synchronisation.  Such callers cannot create a context
 * (rkv_create allocates), yet can run the retrieval step on buffers they own.
 *
 * Computes, for one sequence, what the retrieval of rkv_compress computes (ResidualKV
 * notes §2.2): for each query row i, the topk pool slots j with pool_pos[j] < q_pos[i]
 * nearest in squared L2 distance, nearest first, ties to the smaller slot, -1 padded.
 *   queries    (device, bf16)  [n, d]   the query rows (bf16 joint K/V rows)
 *   q_pos      (device, int32) [n]      their positions
 *   pool       (device, bf16)  [R, d]   the decoded reference rows (for a context's
 *                                      sequence s: rkv_pool_cache rows s * R_cap ..)
 *   pool_norm2 (device, fp32)  [R]      their squared norms (rkv_storage.pool_norm2)
 *   pool_pos   (device, int32) [R]      their positions; INT32_MAX marks an empty slot
 *   out_idx    (device, int32) [n, topk]  output
 *   flags      (device, int32) or NULL: RKV_FLAG_* bits are ORed into it (the caller
 *              clears it).  If a wait of the kernel gives up (RKV_FLAG_TIMEOUT), every
 *              slot of out_idx is written as -1.  With NULL, the call uses a status word
 *              of its own inside the library's scratch, cleared at the start of the
 *              call, with the same effect on out_idx.
 * d must be a multiple of 64, topk in 1..4, queries and pool 16-byte aligned.
 * Scratch: a fixed 4 MiB device array inside the library (every GPU that loads the
 * library holds it until the process exits), enough for ceil(n/128)*ceil(R/256) <= 1024
 * tiles, e.g. n <= 2048 queries against R <= 16384 references; larger calls return
 * RKV_ECAPACITY before any launch.  Nothing in the array needs to start at zero: each
 * call writes every entry it later reads.  All calls share the array, so calls whose
 * kernels overlap on the GPU (different streams, no ordering) race and must not be made.
 * The first call on a device looks up the array's device address (cudaGetSymbolAddress
 * with that device current); make that first call before any stream capture.  A failed
 * look-up returns RKV_ECUDA and is tried again by the next call.  No call allocates or
 * frees memory.
 */
rkv_status rkv_retrieve_noalloc(const void* queries, const int32_t* q_pos, int32_t n,
                                const void* pool, const float* pool_norm2,
                                const int32_t* pool_pos, int32_t R, int32_t d, int32_t topk,
                                int32_t* out_idx, int32_t* flags, void* stream);

/* ---------------------------------------------------------------------------
 * Instrumentation (not part of the method).
 * rkv_set_timing(ctx, 1) records CUDA events around every kernel launch on
 * the launching stream; rkv_get_timing returns, per kernel name, the number
 * of launches and the summed event time since the last reset (it
 * synchronises on the recorded events).  rkv_launch_count counts every
 * kernel the context has launched.
 * ------------------------------------------------------------------------- */
typedef struct {
  char name[48];
  int64_t launches;
  double total_ms;
} rkv_kernel_timing;

rkv_status rkv_set_timing(rkv_ctx* ctx, int32_t enable);
int32_t rkv_get_timing(rkv_ctx* ctx, rkv_kernel_timing* out, int32_t max_entries,
                       int32_t reset);
int64_t rkv_launch_count(rkv_ctx* ctx);

/*
 * Test hook: device address and size of a scratch tensor of the last
 * compress pass.  M and D are in dense order (the pass's rows grouped by
 * sequence, stably), Q in retrieval order (the same groups, each padded to a
 * multiple of 128); for a pass over one sequence, row q of each is the pass's
 * row q:
 *   0 = M, bf16 [rows, 2d_k]: the mean of each row's retrieved references;
 *   1 = D, bf16 [rows, 2*d_ff]: row q = [hi | lo], the fp32 difference of the
 *       SwiGLU hidden rows h(kv_q) - h(mean_q) as two bf16 parts (hi = its bf16
 *       rounding, lo = the bf16 rounding of the rest);
 *   2 = Q, bf16 [rows, parts*2d_k]: the query rows, whose first 2d_k columns
 *       are bf16(kv) (parts = 1 for bf16 kv, 3 for fp32: hi, mid, lo pieces);
 *   3 = P (mean_precompute only), fp32 [B R_cap rounded up to 128, 2*d_ff]:
 *       row s R_cap + slot = r [W_c1 | W_c2] of that reference r, the columns
 *       of each 256-column block being 128 W_c1 columns then the same 128 W_c2
 *       columns (block n: hidden units 128 n .. 128 n + 127).
 * Valid until the next call on the context.
 */
rkv_status rkv_debug_scratch(rkv_ctx* ctx, int32_t which, void** ptr, size_t* bytes);

/*
 * Test hook for failure detection: launches one block that waits on an
 * mbarrier nothing ever arrives at.  The wait is bounded like every pipeline
 * wait in this library; after about a second it sets RKV_FLAG_TIMEOUT in the
 * device status word and the kernel returns.  No fault, no hang: the context
 * stays usable.  rkv_get_status then reports RKV_ETIMEOUT.  The page has no
 * counterpart.
 */
rkv_status rkv_debug_timeout_probe(rkv_ctx* ctx, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* RKV_H */

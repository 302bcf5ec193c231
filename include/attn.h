/*
 * attn.h -- C ABI of the GB300 (sm_103a) attention-forward library.
 *
 * Computes O = softmax(scale * Q K^T + mask) V and the per-row log-sum-exp with the
 * flash-attention online-softmax recurrence ("Flash-Attention: Context (CTE)",
 * section "The online-softmax recurrence"; minfer "03 - 8n FA-style tiled prefill
 * attention", section 2.1 "Online softmax"), for prefill (many queries) and for decode
 * (a few new queries against a flat or paged KV cache).
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library never
 *     frees, keeps or allocates device memory during a call.  Scratch memory that a
 *     call needs is passed in by the caller (see attn_decode_workspace_bytes).
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).
 *     Every compute entry point only enqueues work on it and returns; results are
 *     valid once the stream has reached that point.
 *   - Arguments are checked on the host before anything is enqueued.  An invalid call
 *     returns ATTN_ERR_INVALID_ARG or ATTN_ERR_UNSUPPORTED and enqueues nothing.
 *   - A failed launch returns ATTN_ERR_CUDA; the library clears the pending CUDA error
 *     (cudaGetLastError) before returning so the caller's stream is not poisoned
 *     (minfer 8n, section 3.3, on the shared-memory opt-in failure).
 *   - Faults found by a kernel (a page index past the pool, a wait that never ended)
 *     never trap: the kernel sets a device error word, skips the faulty access, and the
 *     caller reads the word with attn_get_device_error() after synchronising.
 *   - bf16 is IEEE bfloat16 (the top half of an fp32); fp32 is IEEE binary32.
 *   - All entry points are thread-safe with respect to each other on distinct streams.
 */
#ifndef ATTN_GB300_ATTN_H
#define ATTN_GB300_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1,    /* a pointer, size or value violates the contract */
    ATTN_ERR_UNSUPPORTED = 2,    /* valid in principle, not implemented (e.g. d = 96) */
    ATTN_ERR_CUDA = 3,           /* a CUDA runtime call or launch failed */
    ATTN_ERR_PAGE_OOB = 4,       /* device: a block-table entry >= num_pages was met */
    ATTN_ERR_DEVICE_TIMEOUT = 5, /* device: a pipeline wait exceeded its limit */
    ATTN_ERR_WORKSPACE = 6,      /* workspace NULL, misaligned or too small */
    ATTN_ERR_CACHE_LEN = 7       /* device: a cache_len outside [s_active, max_cache_len] */
} attn_status;

typedef enum { ATTN_BF16 = 0, ATTN_F32 = 1 } attn_dtype;

/* Element type of a decode KV cache (attn_opts.kv_dtype). */
typedef enum { ATTN_KV_BF16 = 0, ATTN_KV_E4M3 = 1 } attn_kv_dtype;

/*
 * attn_opts -- optional features of attn_fwd_prefill_ex and attn_fwd_decode_ex.  Pass
 * NULL, or a zero-initialised struct, for the behaviour of the plain calls.  The struct
 * is read on the host during the call and may be reused or freed afterwards.
 *
 *   sink : attention sink ("Flash-Attention: Context (CTE)", "Algorithm - the
 *          per-section max update" and "Algorithm - fused exp and the running sum";
 *          "Flash-Attention: Decode (TKG)", one sink per query head broadcast over the
 *          batch).  A DEVICE array of fp32 [hq], one logit per query head, in the units
 *          of the scaled scores s_j = scale * q.k_j.  The sink joins every row's maximum
 *          and sum as one more logit without a value row:
 *            O   = sum_{allowed j} exp(s_j - M) V_j / (sum_{allowed j} exp(s_j - M) + exp(sink - M))
 *            LSE = M + ln(sum_{allowed j} exp(s_j - M) + exp(sink - M)),
 *            M   = max(max_{allowed j} s_j, sink);
 *          a row with no allowed key gets O = 0 and LSE = sink.  A logit of -inf is no
 *          sink for that head.  Values must be finite or -inf (+inf or NaN give
 *          unspecified results).  NULL = no sink.  Must be 4-byte aligned.
 *
 *   kv_dtype, k_scale, v_scale : decode only (attn_fwd_prefill_ex rejects a kv_dtype other
 *          than ATTN_KV_BF16 with ATTN_ERR_UNSUPPORTED).  ATTN_KV_E4M3 declares k_cache
 *          and v_cache as FP8-e4m3 caches ("Flash-Attention: Decode (TKG)", "Decode (TKG)
 *          vs context (CTE) - the diff"): one byte per element (1 sign, 4 exponent bits
 *          with bias 7, 3 mantissa bits; no infinities, NaN at S.1111.111), same layouts
 *          as the bf16 caches with the byte as the element.  Element x of K stands for
 *          e4m3(x) * k_scale and of V for e4m3(x) * v_scale; both scales must be finite.
 *          With an e4m3 cache d must be 128 or 256.  Slots past cache_len may hold any
 *          byte, NaN codes included; they contribute exactly zero.
 *
 *   window : decode only (prefill has its own window argument).  window > 0 gives new
 *          token t (q_pos = cache_len - s_active + t) the keys j with
 *          q_pos - window + 1 <= j <= q_pos: the prefill window band (AGENTS.md "Sliding
 *          window"; "Flash-Attention: Decode (TKG)", "gen_mask_tkg" type B is that band
 *          at the cache end).  Tiles wholly before every new token's window are not read,
 *          so block-table entries for them may hold anything.  0 = no window.
 *   circular : decode and attn_append_kv, flat caches only.  The flat cache is a ring of
 *          max_cache_len rows: logical position j lives in row j mod max_cache_len, so
 *          cache_len may exceed max_cache_len (type B's wrapped case).  Decode then needs
 *          window > 0, window + s_active - 1 <= max_cache_len (the band fits in the
 *          ring) and max_cache_len a multiple of 32.
 *   rope_inv_freq : a DEVICE fp32 array [d/2] or NULL.  Decode rotates each query row by
 *          rotary position embedding at its q_pos before the product, and attn_append_kv
 *          rotates each new K row at its position ("Flash-Attention: Decode (TKG)",
 *          "Algorithm", step 0; "New-token K/V append"), in half-split form: for i < d/2,
 *          theta = pos * rope_inv_freq[i],
 *            x'[i] = x[i] cos theta - x[i + d/2] sin theta,
 *            x'[i + d/2] = x[i + d/2] cos theta + x[i] sin theta.
 *          Keys already in the cache are used as stored (rotated when they were
 *          appended).  The rotated query is rounded to bf16 before the product.  Must be
 *          4-byte aligned.
 *
 *   cu_seqlens_q, cu_seqlens_k, nseq : prefill only, packed sequences ("Flash-Attention:
 *          Context (CTE)", "Algorithm - the dynamic range_select family": per-row key
 *          bounds for sequence packing and a dynamic prefix length).  DEVICE int32 arrays
 *          [nseq + 1], non-decreasing from 0 to sq and to skv: sequence s holds query rows
 *          [cu_seqlens_q[s], cu_seqlens_q[s+1]) and key rows [cu_seqlens_k[s],
 *          cu_seqlens_k[s+1]) of the one batch (b must be 1).  Each sequence is its own
 *          problem: its queries sit at the tail of its keys (more keys than queries is a
 *          cached prefix), the causal and window masks apply inside it, and no row sees a
 *          key of another sequence.  Offsets that break these rules give unspecified
 *          results but no out-of-range access.  NULL = one problem per (batch, head).
 *   prefill_workspace, prefill_workspace_bytes : packed prefill only; NULL / 0 otherwise.
 *          A DEVICE scratch buffer of at least attn_prefill_workspace_bytes(sq) bytes,
 *          4-byte aligned, owned by the caller and not read by it until the stream has
 *          passed the call.  With it, a small pass first writes a work order of the query
 *          tiles.  Head_dim <= 128: grouped by sequence, most KV tiles first within one, and
 *          the persistent CTAs draw the tiles from a counter the pass resets (kept after
 *          the order), so the tiles in flight share one or two sequences' K/V and the CTAs
 *          stay balanced.  Head_dim 256: ordered by KV-tile count, most first, for the
 *          persistent kernel's fixed zig-zag.  Results are the same with or without it
 *          (each tile is computed the same way wherever it runs); without it the tiles
 *          keep their index order.  Ignored for more than 8192 units of work.
 */
typedef struct {
    const float* sink;
    int kv_dtype;
    float k_scale;
    float v_scale;
    int window;
    int circular;
    const float* rope_inv_freq;
    const int32_t* cu_seqlens_q;
    const int32_t* cu_seqlens_k;
    int nseq;
    void* prefill_workspace;
    size_t prefill_workspace_bytes;
} attn_opts;

/*
 * attn_fwd_prefill -- fused attention forward for sq queries against skv keys.
 *
 * Defines ("Flash-Attention: Context (CTE)", Abstract and "The masking"; optimum-neuron
 * attention AGENTS.md, "Sliding window"; minfer 8n, section 2.1):
 *   kv(h)     = h / (hq / hkv)                         (GQA, CTE "GQA and multi-head")
 *   q_pos(i)  = i + (skv - sq)                         (queries sit at the key tail)
 *   allowed   = j < skv  and (!causal or j <= q_pos(i))
 *                        and (window == 0 or j >= q_pos(i) - window + 1)
 *   s_j       = scale * sum_x Q[b,h,i,x] K[b,kv(h),j,x]
 *   O[b,h,i]  = sum_{allowed j} exp(s_j - M) V[b,kv(h),j] / sum_{allowed j} exp(s_j - M)
 *   LSE[b,h,i]= M + ln sum_{allowed j} exp(s_j - M),   M = max_{allowed j} s_j
 * A row with no allowed key gets O = 0 and LSE = -inf (minfer 8n: rows with l == 0
 * stay 0).  Computed with the online-softmax recurrence: whole KV tiles outside the
 * causal/window band are skipped ("CTE", "Algorithm - compute-skip"), the mask is applied
 * only on tiles that straddle a band edge, exp is evaluated as exp2 with scale*log2(e)
 * folded into one multiply-add, and the accumulator is rescaled lazily.
 *
 * Layouts (row-major, contiguous, 16-byte aligned base pointers):
 *   q : bf16 [b, hq,  sq,  d]      k, v : bf16 [b, hkv, skv, d]
 *   o : [b, hq, sq, d] in o_dtype (ATTN_BF16 rounds to nearest-even, or ATTN_F32)
 *   lse : fp32 [b, hq, sq], natural-log units of the scaled scores; may be NULL.
 * Sizes: b, hq, hkv >= 1, hq % hkv == 0, sq >= 0 (0 = nothing to do), skv >= 0,
 *   d in {64, 128, 256}, window >= 0 and window > 0 only with causal != 0,
 *   scale finite.  Rows, heads and batches up to 2^31 - 1 elements per dimension.
 * Errors: INVALID_ARG / UNSUPPORTED before launch; CUDA if a launch fails;
 *   a device timeout is reported by attn_get_device_error().
 */
attn_status attn_fwd_prefill(const void* q, const void* k, const void* v, void* o, float* lse,
                             int b, int hq, int hkv, int sq, int skv, int d, float scale,
                             int causal, int window, attn_dtype o_dtype, void* stream);

/*
 * attn_fwd_prefill_ex -- attn_fwd_prefill with the options of attn_opts (NULL = none):
 * same arguments, layouts, semantics and errors, plus ATTN_ERR_INVALID_ARG for an
 * invalid option (a misaligned sink pointer; packed sequences with b != 1, nseq < 1 or
 * a missing or misaligned offset array; a prefill workspace without packed sequences,
 * misaligned or smaller than attn_prefill_workspace_bytes(sq)) and ATTN_ERR_UNSUPPORTED
 * for a decode option (an e4m3 kv_dtype, window, circular or rope_inv_freq).
 */
attn_status attn_fwd_prefill_ex(const void* q, const void* k, const void* v, void* o, float* lse,
                                int b, int hq, int hkv, int sq, int skv, int d, float scale,
                                int causal, int window, attn_dtype o_dtype,
                                const attn_opts* opts, void* stream);

/*
 * attn_prefill_workspace_bytes -- bytes of the optional packed-prefill scratch
 * (attn_opts.prefill_workspace) for sq query rows: 4 bytes per 128-row query tile.
 * Returns 0 for sq <= 0.
 */
size_t attn_prefill_workspace_bytes(int sq);

/*
 * attn_decode_workspace_bytes -- bytes of caller-provided scratch that attn_fwd_decode
 * needs for these sizes: split-KV partial outputs [b*hq*s_active][slots][d] fp32 and
 * their (max, sum) pairs, slots = ceil(max_cache_len / kv_chunk) + 1, then one int per
 * (sequence, head).  kv_chunk as for attn_fwd_decode (0 = library default).  Returns 0
 * for invalid sizes.
 */
size_t attn_decode_workspace_bytes(int b, int hq, int s_active, int d, int max_cache_len,
                                   int kv_chunk);

/*
 * attn_fwd_decode -- attention of s_active new tokens per sequence against its KV cache.
 *
 * Defines ("Flash-Attention: Decode (TKG)", "The single-query decode attention",
 * "KV-cache layouts and access", "gen_mask_tkg"):
 *   the cache of sequence b holds cache_len[b] tokens, the last s_active of which are the
 *   new tokens' own K/V (already appended by the caller);
 *   new token t sits at q_pos = cache_len[b] - s_active + t and attends cache position j
 *   iff j <= q_pos (the validity cut j < cache_len plus the tril block among the new
 *   tokens); the softmax runs over the cache axis; GQA as in attn_fwd_prefill.
 * It runs as a split-KV pass followed by a log-sum-exp combine.  The split pass is one
 * wave of CTAs that share the KV tiles of all (sequence, kv head) pairs evenly, each CTA
 * reading at least kv_chunk tokens (unless it reads the last ones); every piece of a pair
 * that one CTA reads keeps its own running max, sum and unnormalised output.
 *
 * Layouts:
 *   q : bf16 [b, hq, s_active, d]        o : [b, hq, s_active, d] in o_dtype
 *   lse : fp32 [b, hq, s_active] (may be NULL)
 *   cache_len : int32 [b]
 *   paged cache (block_table != NULL): k_cache, v_cache bf16 [num_pages, hkv, page_size, d];
 *     block_table uint32 [b, max_pages_per_seq]; logical token j of sequence b lives in
 *     page block_table[b][j / page_size], slot j % page_size ("Paged / block cache").
 *     Entries past ceil(cache_len/page_size) are never read.
 *   flat cache (block_table == NULL): k_cache, v_cache bf16 [b, hkv, max_cache_len, d].
 *   Slots past cache_len may hold anything (even NaN); they contribute exactly zero.
 * Sizes: hq % hkv == 0; (hq / hkv) * s_active <= 16; d in {64, 128, 256};
 *   1 <= s_active; cache_len[b] in [s_active, max_cache_len];
 *   paged: page_size a power of two in [16, 256], max_cache_len <=
 *   max_pages_per_seq * page_size, num_pages >= 1; kv_chunk = 0 or a positive multiple of
 *   32 (and of page_size when page_size > 32).  kv_chunk = 0 picks the largest power of two
 *   in [256, 4096] not above b * max_cache_len / 128; attn_decode_workspace_bytes applies
 *   the same rule.  A larger kv_chunk needs less scratch; below the even share of the
 *   tiles it does not change how the work is split.
 * Workspace: device scratch of at least attn_decode_workspace_bytes(...), 16-byte aligned,
 *   owned by the caller, not read before it is written; calls that share it must not
 *   overlap on the device.
 * Errors: INVALID_ARG / UNSUPPORTED / WORKSPACE before launch; CUDA on launch failure.
 *   A block-table entry >= num_pages or a cache_len outside its range is reported by
 *   attn_get_device_error() (ATTN_ERR_PAGE_OOB / ATTN_ERR_CACHE_LEN); the offending page
 *   is not read and the affected outputs are unspecified.
 */
attn_status attn_fwd_decode(const void* q, const void* k_cache, const void* v_cache,
                            const uint32_t* block_table, const int32_t* cache_len, int b, int hq,
                            int hkv, int d, int s_active, int page_size, int max_pages_per_seq,
                            int num_pages, int max_cache_len, float scale, void* o, float* lse,
                            attn_dtype o_dtype, int kv_chunk, void* workspace,
                            size_t workspace_bytes, void* stream);

/*
 * attn_fwd_decode_ex -- attn_fwd_decode with the options of attn_opts (NULL = none):
 * same arguments (opts sits after kv_chunk), layouts, workspace, semantics and errors,
 * plus ATTN_ERR_INVALID_ARG for an invalid option (a misaligned sink or rope_inv_freq
 * pointer, an unknown kv_dtype, a non-finite scale of an e4m3 cache, a negative window, a
 * circular paged cache or a circular cache whose window does not fit) and
 * ATTN_ERR_UNSUPPORTED for an e4m3 cache with d = 64 or a prefill option (packed
 * sequences or a prefill workspace).  With circular, cache_len[b] may
 * exceed max_cache_len.  The sink is applied where the split-KV chunks are merged and the
 * scales are folded into the chunk pass, so the workspace size is the same for every
 * option.
 */
attn_status attn_fwd_decode_ex(const void* q, const void* k_cache, const void* v_cache,
                               const uint32_t* block_table, const int32_t* cache_len, int b,
                               int hq, int hkv, int d, int s_active, int page_size,
                               int max_pages_per_seq, int num_pages, int max_cache_len,
                               float scale, void* o, float* lse, attn_dtype o_dtype, int kv_chunk,
                               const attn_opts* opts, void* workspace, size_t workspace_bytes,
                               void* stream);

/*
 * attn_append_kv -- write the new tokens' K and V into a bf16 cache ("Flash-Attention:
 * Decode (TKG)", "New-token K/V append": the kernel's persistent store of the new K).
 * New token t of sequence b goes to logical position cache_len[b] - s_active + t (cache_len
 * already counts the new tokens, as for attn_fwd_decode), through the block table or, for
 * a flat cache, at row j (row j mod max_cache_len with opts->circular).  With
 * opts->rope_inv_freq its K row is rotated at position j first (see attn_opts) and rounded
 * to bf16; V is copied as is.  Other options are ignored.
 *
 * Layouts: k_new, v_new bf16 [b, hkv, s_active, d]; caches and block_table as for
 *   attn_fwd_decode (bf16 only).  Only the new tokens' cache rows are written.
 * Sizes: as attn_fwd_decode, d in {64, 128, 256}; circular only with a flat cache.
 * Errors: INVALID_ARG / UNSUPPORTED before launch; CUDA on launch failure; a block-table
 *   entry >= num_pages (that row is not written) or a cache_len outside its range is
 *   reported by attn_get_device_error().
 */
attn_status attn_append_kv(const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                           const uint32_t* block_table, const int32_t* cache_len, int b, int hkv,
                           int d, int s_active, int page_size, int max_pages_per_seq,
                           int num_pages, int max_cache_len, const attn_opts* opts, void* stream);

/*
 * attn_fwd_decode_static_ws -- attn_fwd_decode for callers that cannot allocate device
 * memory.  The pages have no counterpart to this entry point; it exists for callers that
 * must not call cudaMalloc or any other allocator when they run attention: code held to
 * a fixed device-memory budget set up once at start-up, plug-ins hosted by a runtime that
 * owns every device allocation, real-time loops that must stay out of the allocator.
 *
 * Same arguments, layouts, semantics and results as attn_fwd_decode, minus the workspace:
 * the split-KV scratch is a fixed 64 MiB device array compiled into the library (present
 * on every GPU that loads the library until the process exits).  A call whose scratch,
 * attn_decode_workspace_bytes(b, hq, s_active, d, max_cache_len, kv_chunk), exceeds
 * 64 MiB is rejected with ATTN_ERR_WORKSPACE and enqueues nothing.  All calls share the
 * array, so calls that overlap on the GPU (on different streams, or from host threads
 * without ordering between them) race and give unspecified results; order them on one
 * stream.  The array needs no clearing: each call writes every part it later reads.
 * Each call made while `stream` is not being captured looks up the array's device
 * address on the current device (cudaGetSymbolAddress) and remembers it; a call made
 * during a capture uses the remembered address, so make the first call on each device
 * before any stream capture begins (otherwise: ATTN_ERR_CUDA).  After a device reset the
 * next call outside a capture finds the array's new address.
 * Allocates nothing: no cudaMalloc, cudaFree or allocating library routine is called.
 */
attn_status attn_fwd_decode_static_ws(const void* q, const void* k_cache, const void* v_cache,
                                      const uint32_t* block_table, const int32_t* cache_len,
                                      int b, int hq, int hkv, int d, int s_active, int page_size,
                                      int max_pages_per_seq, int num_pages, int max_cache_len,
                                      float scale, void* o, float* lse, attn_dtype o_dtype,
                                      int kv_chunk, void* stream);

/*
 * attn_gen_mask_decode -- materialise the decode 0/1 mask that attn_fwd_decode applies
 * in registers ("Flash-Attention: Decode (TKG)", "gen_mask_tkg": type A `index <
 * cache length` and type C, the tril(ones(s_active)) block of the new tokens):
 *   mask[b, h, t, j] = 1 iff j < cache_len[b] and j <= cache_len[b] - s_active + t.
 * It is evaluated by the same device predicate the decode kernel uses.
 * mask_out: uint8 [b, hq, s_active, max_len] (device).  cache_len must lie in
 * [s_active, max_len]; rows of a sequence outside it are left all-zero and flagged
 * (ATTN_ERR_CACHE_LEN via attn_get_device_error).
 */
attn_status attn_gen_mask_decode(const int32_t* cache_len, int b, int hq, int s_active,
                                 int max_len, uint8_t* mask_out, void* stream);

/*
 * attn_check_wait_timeout -- a test export of the failure path.  The library's kernels
 * never trap: every pipeline wait is bounded, and a wait that runs out sets a device error
 * word and unwinds.  This call launches one thread that waits, with the same bounded wait,
 * on an mbarrier phase that nothing completes, gives up after wait_cycles SM clock cycles
 * (1 .. 2^33), sets the timeout word and returns.  attn_get_device_error() then reports
 * ATTN_ERR_DEVICE_TIMEOUT and the context stays usable.  Returns INVALID_ARG for a
 * wait_cycles outside its range, CUDA if the launch fails.
 */
attn_status attn_check_wait_timeout(long long wait_cycles, void* stream);

/*
 * attn_get_device_error -- synchronise `stream`, then read and clear the device error
 * words of every kernel in the library on the current device.  Returns ATTN_OK, or the
 * most severe of ATTN_ERR_DEVICE_TIMEOUT, ATTN_ERR_PAGE_OOB, ATTN_ERR_CACHE_LEN; returns
 * ATTN_ERR_CUDA if the synchronisation itself failed.
 */
attn_status attn_get_device_error(void* stream);

/* attn_status_string -- static, human-readable name of a status code. */
const char* attn_status_string(attn_status status);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_ATTN_H */

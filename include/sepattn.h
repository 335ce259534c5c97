/*
 * sepattn.h -- C ABI of the B300 (sm_103a) SepLLM attention library.
 *
 * The method: "SepLLM: Accelerate Large Language Models by Compressing One
 * Segment into One Separator" (arXiv 2412.12094).  Each query attends to the
 * first `a` tokens, every preceding separator token (. , ? ! ; : space tab
 * newline) and its `n` nearest tokens, itself included; every other pair is
 * masked (anthology record lit-748, Key takeaways, "The mask"; pith.science
 * review, key_machinery).  Streaming generation keeps four KV blocks
 * (initial, separator, past window, local window) under a capacity c, moves
 * the past window's separators into the separator block when the cache is
 * full, and applies RoPE at positions inside the cache (pith.science review,
 * key_machinery; paperhub rebuttal, reply A1 to the second reviewer).
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Pointers are DEVICE pointers unless the argument says "host".
 *  - The caller allocates and owns every buffer; the library never allocates
 *    device memory and keeps no state between calls other than the device
 *    status word described at sep_get_device_status().
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  All work
 *    is enqueued asynchronously on it; calls do not synchronise, except
 *    sep_cache_export / sep_cache_import / sep_get_device_status, which say so.
 *  - Tensors are dense row-major ("[B, H, L, d]" means d is contiguous) and
 *    16-byte aligned.  bf16 is IEEE bfloat16 stored as uint16.
 *  - Host-side argument checks return an error before anything is enqueued.
 *    Errors found on the device (a corrupt index, an inconsistent cache, a
 *    bounded wait that expired) are written to the device status word; no
 *    kernel traps.  A CUDA launch error returns SEP_ERR_CUDA.
 *  - Thread safety: calls on different buffers may run concurrently; calls
 *    that touch the same buffer must be ordered by the caller.
 */
#ifndef SEPATTN_H
#define SEPATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SEP_OK = 0,
  SEP_ERR_INVALID_ARG = 1,   /* a null pointer, a bad size or a misaligned buffer */
  SEP_ERR_UNSUPPORTED = 2,   /* a valid request this build does not implement */
  SEP_ERR_CAPACITY = 3,      /* streaming capacities violate a + s + w < c */
  SEP_ERR_CUDA = 4,          /* a CUDA runtime call failed */
  SEP_ERR_TIMEOUT = 5,       /* device: a bounded wait expired */
  SEP_ERR_DEVICE_BOUNDS = 6, /* device: an index or count was out of range */
  SEP_ERR_WORKSPACE = 7,     /* workspace / buffer smaller than the size query */
  SEP_ERR_TOO_LARGE = 8      /* request exceeds the fixed scratch of sep_attn_fwd_static */
} sep_status;

typedef enum { SEP_F32 = 0, SEP_BF16 = 1 } sep_dtype;

/* Largest separator-id list accepted by the calls that take one. */
#define SEP_MAX_SEP_IDS 64
/* Query-tile height of the block lists the attention kernels consume. */
#define SEP_BLOCK_M 128

/* ======================================================================
 * Index: separator detection, keep-token compaction, block lists
 * ====================================================================== */

/* Bytes of the index buffer for B sequences of length L and query tiles of
 * block_m rows (0 if an argument is out of range). */
size_t sep_index_bytes(int B, int L, int block_m);

/* sep_build_index -- separator flags, keep-token prefix scan and compaction,
 * and per-query-tile block lists for a batch of token-id sequences.
 *
 * Defines: sep[b,j] = ids[b,j] in sep_ids; keep[b,j] = (j < a) or sep[b,j]
 * (the tokens a query still sees once they have left its n-token window:
 * anthology record lit-748, "The mask"; paperhub rebuttal, reply A1 to the
 * first reviewer, for the separator set).
 *
 *   ids        device int32 [B, L] token ids.
 *   sep_ids    HOST int32 [n_sep_ids] separator ids (0 <= n_sep_ids <=
 *              SEP_MAX_SEP_IDS; 0 ids gives StreamingLLM's sink + window).
 *   a          number of initial (attention-sink) tokens, >= 0.
 *   n          neighbour window, >= 1; row i's window is [i-n+1, i].
 *   block_m    query-tile height of the block lists; must be SEP_BLOCK_M.
 *   index_buf  device buffer of index_bytes >= sep_index_bytes(B, L, block_m),
 *              256-byte aligned, written by this call (every field below
 *              but the keep_pos entries past each count).  Its fields
 *              are reached with sep_index_views(); the attention calls read
 *              a, n, B and L from it.
 *
 * Fields (all int32 unless stated):
 *   keep_prefix [B, L+1]   number of keep tokens in [0, j)
 *   keep_pos    [B, L]     ascending positions of keep tokens; only the
 *                          entries below keep_count[b] are written
 *   keep_count  [B]
 *   blocks      [B, T, 4]  T = ceil(L / block_m); for tile t with first row
 *                          i0 = t*block_m and W = max(0, i0-n+1):
 *                          {n_gather = keep_prefix[W], dense_lo = W,
 *                           dense_hi = min(L, i0+block_m), flags = (W < a)}
 *   keep_bits   uint32 [B, ceil(L/32)]  bit j%32 of word j/32 = keep[j]
 * Every visible pair (i, j) of a tile's rows is covered exactly once: by
 * the first n_gather keep tokens, or by the dense range [dense_lo, dense_hi)
 * under the element mask j <= i and (keep[j] or j >= i-n+1).
 * Errors: SEP_ERR_INVALID_ARG (B, L < 1, a < 0, n < 1, bad n_sep_ids, null
 * or misaligned pointers), SEP_ERR_UNSUPPORTED (block_m != SEP_BLOCK_M),
 * SEP_ERR_WORKSPACE (index_bytes too small), SEP_ERR_CUDA. */
sep_status sep_build_index(const int32_t* ids, int B, int L,
                           const int32_t* sep_ids, int n_sep_ids,
                           int a, int n, int block_m,
                           void* index_buf, size_t index_bytes, void* stream);

/* sep_build_index_fixed -- the index of the FixLLM control: the same
 * fields and block lists as sep_build_index, with the separators replaced
 * by one kept token per interval of `delta` positions (anthology record
 * lit-748, Key takeaways, "What is ablated": FixLLM keeps one token at fixed
 * intervals instead of separators).  keep[j] = (j < a) or ((j + 1) % delta
 * == 0); no token ids are read.  sep_attn_fwd / sep_attn_bwd consume the
 * result unchanged.  delta = 1 keeps every token (full causal attention).
 * Errors: SEP_ERR_INVALID_ARG (B, L < 1, a < 0, n < 1, delta < 1, null or
 * misaligned index_buf), SEP_ERR_UNSUPPORTED, SEP_ERR_WORKSPACE, SEP_ERR_CUDA. */
sep_status sep_build_index_fixed(int B, int L, int a, int n, int delta, int block_m,
                                 void* index_buf, size_t index_bytes, void* stream);

/* sep_build_index_varlen -- the index of a PACK: B sequences of different
 * lengths stored one after another, as a training step packs documents.
 * The mask is defined per sequence (anthology record lit-748, "The mask",
 * "Training from scratch"); the pages say nothing of packing, so each
 * sequence of a pack is treated as a sequence of its own: its positions
 * restart at 0, its first `a` tokens are its sinks, and no query sees a key
 * of another sequence.
 *
 *   ids         device int32 [total] token ids of all sequences, packed.
 *   cu_seqlens  device int32 [B + 1] sequence starts: sequence b is packed
 *               rows [cu_seqlens[b], cu_seqlens[b+1]); cu_seqlens[0] = 0 and
 *               cu_seqlens[B] = total.  Empty sequences are allowed.
 *   max_len     the longest sequence length (>= 1); every per-sequence
 *               field of the index is padded to it.  Size the buffer with
 *               sep_index_bytes(B, max_len, block_m).
 *   other arguments as sep_build_index.
 * The fields (sep_index_views with L = max_len) hold, for each sequence, what
 * sep_build_index gives for that sequence alone in local positions, padded:
 * keep_prefix[b][j] = keep_count[b] for j >= len_b, keep_pos written below
 * the count only, empty block records {0, 0, 0, 0} for tiles at or past len_b, zero
 * keep bits past len_b.
 * Errors: SEP_ERR_INVALID_ARG, SEP_ERR_UNSUPPORTED, SEP_ERR_WORKSPACE,
 * SEP_ERR_CUDA; device: SEP_ERR_DEVICE_BOUNDS if cu_seqlens is not a valid
 * partition of [0, total) into lengths <= max_len (the offending sequences
 * index as empty). */
sep_status sep_build_index_varlen(const int32_t* ids, const int32_t* cu_seqlens, int B,
                                  int total, int max_len, const int32_t* sep_ids,
                                  int n_sep_ids, int a, int n, int block_m, void* index_buf,
                                  size_t index_bytes, void* stream);

/* Device pointers to the fields of an index buffer (pure pointer arithmetic,
 * no device access).  Any output pointer may be NULL. */
sep_status sep_index_views(void* index_buf, int B, int L, int block_m,
                           int32_t** keep_prefix, int32_t** keep_pos,
                           int32_t** keep_count, int32_t** blocks,
                           uint32_t** keep_bits);

/* ======================================================================
 * Sep-Attention forward and backward (prefill / training)
 * ====================================================================== */

/* Workspace bytes for sep_attn_fwd (backward = 0) or sep_attn_bwd
 * (backward = 1).  The forward uses it for the gathered keep-token K/V; the
 * backward also for row statistics and keep-token gradient accumulators. */
size_t sep_attn_workspace_bytes(int B, int Hq, int Hkv, int L, int d,
                                sep_dtype dtype, int backward);

/* sep_attn_fwd -- O = softmax(Q K^T * scale + log M) V under the SepLLM
 * mask M of the index (anthology record lit-748, "The mask"; masked pairs
 * get -inf before the softmax), plus the natural-log row partition LSE.
 *
 *   index_buf  built by sep_build_index for the same B and L.
 *   q          [B, Hq, L, d]; k, v [B, Hkv, L, d]; element type `dtype`.
 *   o          [B, Hq, L, d] output, element type `dtype`.
 *   lse        float32 [B, Hq, L] output: log sum_j exp(S_ij) over visible j.
 *   Hq % Hkv == 0; q head h reads kv head h / (Hq / Hkv).
 *   d          64 or 128.
 *   dtype      SEP_BF16 (tcgen05 tensor-core kernel, fp32 accumulation, P
 *              rounded to bf16 for the P.V product) or SEP_F32 (CUDA-core
 *              kernel, fp32 throughout).
 *   scale      softmax scale; <= 0 selects 1/sqrt(d).
 *   ws         workspace of ws_bytes >= sep_attn_workspace_bytes(.., 0),
 *              256-byte aligned.
 * Errors: SEP_ERR_INVALID_ARG, SEP_ERR_UNSUPPORTED (d, dtype),
 * SEP_ERR_WORKSPACE, SEP_ERR_CUDA; device: SEP_ERR_DEVICE_BOUNDS if the
 * index does not match B and L, SEP_ERR_TIMEOUT. */
sep_status sep_attn_fwd(const void* index_buf, const void* q, const void* k,
                        const void* v, void* o, float* lse,
                        int B, int Hq, int Hkv, int L, int d, sep_dtype dtype,
                        float scale, void* ws, size_t ws_bytes, void* stream);

/* sep_attn_bwd -- gradients of the masked attention (the pages train with
 * the mask: anthology record lit-748, "The mask" and "Training from
 * scratch").  Textbook recomputation: P = exp(S*scale - LSE),
 * Delta = rowsum(dO o O), dS = P o (dO V^T - Delta), dV = P^T dO,
 * dQ = dS K * scale, dK = dS^T Q * scale; with Hq > Hkv, dK and dV of a kv
 * head sum over its q heads.
 *
 *   o, lse     outputs of sep_attn_fwd for the same inputs.
 *   dout       [B, Hq, L, d] gradient of O.
 *   dq         [B, Hq, L, d] output; dk, dv [B, Hkv, L, d] outputs.
 *   dtype      SEP_BF16 only (SEP_ERR_UNSUPPORTED otherwise).
 *   d          64 or 128.
 *   ws         ws_bytes >= sep_attn_workspace_bytes(.., 1).
 * Errors: as sep_attn_fwd. */
sep_status sep_attn_bwd(const void* index_buf, const void* q, const void* k,
                        const void* v, const void* o, const float* lse,
                        const void* dout, void* dq, void* dk, void* dv,
                        int B, int Hq, int Hkv, int L, int d, sep_dtype dtype,
                        float scale, void* ws, size_t ws_bytes, void* stream);

/* sep_attn_fwd_hybrid / sep_attn_bwd_hybrid -- hybrid heads: some kv groups
 * attend with full causal attention, the others under the index's mask.
 * The pages evaluate this layout two ways:
 *  - as a baseline with some heads on a sliding window and the rest on
 *    full attention (paperhub rebuttal page, reply A5 to the third
 *    reviewer).  Build the index with no separator ids and a = 0 for
 *    those window heads;
 *  - with the first, or first and last, layers on full attention
 *    (anthology record lit-748, "Training from scratch").
 *
 * Bit g of full_groups (g < Hkv <= 64) puts kv group g -- q heads
 * g*(Hq/Hkv) .. (g+1)*(Hq/Hkv)-1 and kv head g -- on the causal mask
 * j <= i, exactly the index's mask with a window n >= L.  The other groups
 * use the index's mask.  full_groups = 0 is sep_attn_fwd / sep_attn_bwd.
 * All other arguments, layouts, workspaces and errors are those of
 * sep_attn_fwd and sep_attn_bwd with dtype SEP_BF16.  Bits at or above Hkv
 * give SEP_ERR_INVALID_ARG. */
sep_status sep_attn_fwd_hybrid(const void* index_buf, const void* q, const void* k,
                               const void* v, void* o, float* lse,
                               int B, int Hq, int Hkv, int L, int d,
                               unsigned long long full_groups, float scale,
                               void* ws, size_t ws_bytes, void* stream);
sep_status sep_attn_bwd_hybrid(const void* index_buf, const void* q, const void* k,
                               const void* v, const void* o, const float* lse,
                               const void* dout, void* dq, void* dk, void* dv,
                               int B, int Hq, int Hkv, int L, int d,
                               unsigned long long full_groups, float scale,
                               void* ws, size_t ws_bytes, void* stream);

/* Workspace bytes of sep_attn_fwd_varlen (backward = 0) and
 * sep_attn_bwd_varlen (backward = 1) for a pack of B sequences of at most
 * max_len rows in `total` rows (0 if the shape is invalid). */
size_t sep_attn_workspace_bytes_varlen(int B, int total, int max_len, int Hq, int Hkv, int d,
                                       int backward);

/* sep_attn_fwd_varlen / sep_attn_bwd_varlen -- sep_attn_fwd and
 * sep_attn_bwd over a pack indexed by sep_build_index_varlen: the mask of
 * each sequence on its own, no pair across sequences.
 *
 *   q, o, dout, dq  [Hq, total, d] bf16: per head, the sequences' rows packed
 *                   in the order of cu_seqlens.
 *   k, v, dk, dv    [Hkv, total, d] bf16.
 *   lse             float32 [Hq, total].
 *   B, total, max_len  as given to sep_build_index_varlen.
 *   ws              ws_bytes >= sep_attn_workspace_bytes_varlen(..).
 * Everything else (GQA mapping, d in {64, 128}, scale, errors) as
 * sep_attn_fwd / sep_attn_bwd with dtype SEP_BF16.  total = 0 does nothing.
 * Device: SEP_ERR_DEVICE_BOUNDS if the index is not a pack index of these
 * B, max_len and total. */
sep_status sep_attn_fwd_varlen(const void* index_buf, const void* q, const void* k,
                               const void* v, void* o, float* lse, int B, int total,
                               int max_len, int Hq, int Hkv, int d, float scale, void* ws,
                               size_t ws_bytes, void* stream);
sep_status sep_attn_bwd_varlen(const void* index_buf, const void* q, const void* k,
                               const void* v, const void* o, const float* lse,
                               const void* dout, void* dq, void* dk, void* dv, int B, int total,
                               int max_len, int Hq, int Hkv, int d, float scale, void* ws,
                               size_t ws_bytes, void* stream);

/* Size of the fixed device scratch array behind sep_attn_fwd_static. */
#define SEP_STATIC_SCRATCH_BYTES (64u << 20)

/* sep_attn_fwd_static -- sep_attn_fwd for callers that cannot allocate.
 *
 * The paper has no counterpart to this call; it exists for library users.
 * Some callers cannot call cudaMalloc or any allocating routine: code inside
 * an allocator callback or out-of-memory handler, a plug-in whose host
 * framework owns all device memory, a real-time loop that allocates nothing
 * after start-up.  sep_attn_fwd needs a caller-provided workspace; this call
 * needs none.  It computes exactly what sep_attn_fwd computes for
 * dtype = SEP_BF16, with the gathered keep-token K/V rows held in a fixed
 * device array of SEP_STATIC_SCRATCH_BYTES (64 MiB) inside the library.
 * It calls no cudaMalloc, cudaFree or other allocating routine.
 *
 * Arguments, layouts and the index are those of sep_attn_fwd (bf16 only;
 * d 64 or 128).  The caller still allocates q, k, v, o, lse and the index.
 * Limit: the forward workspace, sep_attn_workspace_bytes(B, Hq, Hkv, L, d,
 * SEP_BF16, 0) (4 * B * Hkv * L' * d bytes with L' = L rounded up to a
 * multiple of 128), must not exceed
 * SEP_STATIC_SCRATCH_BYTES; larger shapes return SEP_ERR_TOO_LARGE before
 * any device work.
 *
 * The scratch array:
 *  - is held by every GPU that loads the library, until the process exits;
 *  - is found on each device by the first call made with that device
 *    current (cudaGetSymbolAddress); make that first call before any stream
 *    capture;
 *  - is shared by every call and keeps the last call's contents.  Calls do
 *    not depend on them: every scratch row a call reads, it first writes.
 *    Calls that overlap on the GPU (other streams, unordered host threads)
 *    race on it, so the caller must order them.
 * Errors: SEP_ERR_INVALID_ARG, SEP_ERR_UNSUPPORTED, SEP_ERR_TOO_LARGE,
 * SEP_ERR_CUDA; device errors as sep_attn_fwd. */
sep_status sep_attn_fwd_static(const void* index_buf, const void* q, const void* k,
                               const void* v, void* o, float* lse,
                               int B, int Hq, int Hkv, int L, int d, float scale,
                               void* stream);

/* ======================================================================
 * Streaming four-block KV cache and decode attention
 * ====================================================================== */

/* Shape of a batch of S streaming caches. */
typedef struct {
  int S;            /* sequences */
  int Hkv;          /* kv heads, 1..64 */
  int d;            /* head dim, 128 (64 also accepted) */
  int a;            /* initial (sink) block capacity */
  int s;            /* separator block capacity */
  int w;            /* local window capacity */
  int c;            /* total capacity, <= 1024; requires a + s + w < c */
  float rope_theta; /* RoPE base; <= 0 selects 500000 */
} sep_cache_params;

/* Bytes of one cache buffer (0 if the shape is invalid). */
size_t sep_cache_bytes(const sep_cache_params* p);

/* sep_cache_init -- empty caches and the RoPE cos/sin table (rotate-half
 * pairing, inv_freq_i = theta^(-2i/d), positions 0..c-1).
 *   p          HOST params; cache_buf device buffer of `bytes` >=
 *              sep_cache_bytes(p), 256-byte aligned.
 * Errors: SEP_ERR_INVALID_ARG, SEP_ERR_CAPACITY (a + s + w >= c),
 * SEP_ERR_UNSUPPORTED (Hkv > 64, c > 1024, d not 64/128), SEP_ERR_WORKSPACE,
 * SEP_ERR_CUDA.  Synchronous on `stream` for the table upload. */
sep_status sep_cache_init(const sep_cache_params* p, void* cache_buf,
                          size_t bytes, void* stream);

/* sep_cache_step -- one streaming step for every sequence: update the cache
 * with the new token, then (if q and out are non-NULL) attend from the new
 * token's queries over the whole cache, the new token included.
 *
 * Update (pith.science review, key_machinery): when the cache holds exactly
 * c entries, the past window's separators move, oldest first, into the
 * separator block (its oldest entries beyond s are dropped) and the rest of
 * the past window is dropped; then the token enters the initial block if it
 * has fewer than a entries, else the local window, whose oldest entry moves
 * to the past window once it holds more than w.
 * Attention (paperhub rebuttal, reply A1 to the second reviewer): entry k
 * of the logical order initial + separator + past + local is rotated by
 * RoPE at position k; the new token (last entry) at position N-1.
 *
 *   q        [S, Hq, d] bf16 queries of the new tokens (NULL: update only).
 *   k_new, v_new [S, Hkv, d] bf16 un-rotated keys / values of the new tokens.
 *   ids_new  int32 [S] token ids of the new tokens.
 *   sep_ids  HOST int32 [n_sep_ids] separator ids (<= SEP_MAX_SEP_IDS).
 *   out      [S, Hq, d] bf16 (NULL: update only).
 *   Hq       q heads: Hq / Hkv must be 1, 2, 4 or 8.
 *   scale    <= 0 selects 1/sqrt(d).
 * Errors: SEP_ERR_INVALID_ARG, SEP_ERR_UNSUPPORTED, SEP_ERR_CUDA; device:
 * SEP_ERR_DEVICE_BOUNDS if the stored counters are inconsistent. */
sep_status sep_cache_step(const sep_cache_params* p, void* cache_buf,
                          const void* q, const void* k_new, const void* v_new,
                          const int32_t* ids_new, const int32_t* sep_ids,
                          int n_sep_ids, void* out, int Hq, float scale,
                          void* stream);

/* Bytes of the workspace sep_cache_prefill needs for a prompt of T tokens
 * (0 if the shape is invalid). */
size_t sep_cache_prefill_workspace_bytes(const sep_cache_params* p, int T);

/* sep_cache_prefill -- append a whole prompt of T tokens to EMPTY caches in
 * one launch.  The result is the state T update-only sep_cache_step calls
 * (q = out = NULL) would leave: the same export image, and every later step
 * gives the same outputs.  Under the update rule of sep_cache_step the
 * cache holds, in text order, the first a tokens, the newest <= s
 * separators among the tokens the window has left and the window itself
 * (pith.science review, key_machinery), so only the window start depends on
 * the step-by-step history; it is replayed from a separator prefix count.
 *
 *   k_prompt, v_prompt [T, S, Hkv, d] bf16 (the T step inputs stacked).
 *   ids      int32 [T, S] token ids.
 *   sep_ids  HOST int32 [n_sep_ids].
 *   ws       device workspace >= sep_cache_prefill_workspace_bytes(p, T),
 *            256-byte aligned.
 * Errors: SEP_ERR_INVALID_ARG, SEP_ERR_UNSUPPORTED, SEP_ERR_CAPACITY,
 * SEP_ERR_WORKSPACE, SEP_ERR_CUDA; device: SEP_ERR_DEVICE_BOUNDS if a cache
 * is not empty (its counters are left untouched). */
sep_status sep_cache_prefill(const sep_cache_params* p, void* cache_buf, const void* k_prompt,
                             const void* v_prompt, const int32_t* ids, int T,
                             const int32_t* sep_ids, int n_sep_ids, void* ws, size_t ws_bytes,
                             void* stream);

/* Bytes of the host image written by sep_cache_export. */
size_t sep_cache_export_bytes(const sep_cache_params* p);

/* sep_cache_export -- copy the caches to a HOST buffer in logical order
 * (synchronises `stream`).  Layout (little-endian):
 *   int32 header[8] = {0x53455043 ('SEPC'), S, Hkv, d, a, s, w, c}
 *   per sequence, int32 counts[8] = {n_init, n_sep, n_past, n_win, total,
 *                                    next_text_position, 0, 0}
 *   int32  pos[S][c]            text positions, logical order, -1 past total
 *   uint8  is_sep[S][c]         separator flags, 0 past total
 *   uint16 k[S][c][Hkv][d]      raw bf16 keys (un-rotated), 0 past total
 *   uint16 v[S][c][Hkv][d]      bf16 values, 0 past total
 * Errors: SEP_ERR_INVALID_ARG, SEP_ERR_WORKSPACE, SEP_ERR_CUDA. */
sep_status sep_cache_export(const sep_cache_params* p, const void* cache_buf,
                            void* host_dst, size_t bytes, void* stream);

/* sep_cache_import -- load an image written by sep_cache_export (synchronous).
 * A cache imported from an export continues bit-identically: same contents
 * and, because attention reduces in logical order, the same outputs.
 * Errors: SEP_ERR_INVALID_ARG (header or counts inconsistent with p),
 * SEP_ERR_WORKSPACE, SEP_ERR_CUDA. */
sep_status sep_cache_import(const sep_cache_params* p, void* cache_buf,
                            const void* host_src, size_t bytes, void* stream);

/* ======================================================================
 * Status
 * ====================================================================== */

/* Read and clear the device status word of the current device (SEP_OK if no
 * kernel reported an error since the last call).  Synchronises the device. */
sep_status sep_get_device_status(void);

/* sep_profile_events -- timing hook for benchmarks (no counterpart in the
 * paper).  Registers up to SEP_MAX_PROFILE_EVENTS cudaEvent_t handles for
 * the calling host thread; while registered, sep_attn_fwd and sep_attn_bwd
 * record them on their stream around the kernels they launch, so a caller
 * can time each kernel with cudaEventElapsedTime (also inside a CUDA-graph
 * capture, where the records become graph nodes).  n_events = 0 clears.
 *   sep_attn_fwd (bf16): [0] before the keep gather, [1] before the
 *                        attention kernel, [2] after it.
 *   sep_attn_bwd:        [0] before the prep kernel (keep gather, Delta and
 *                        the dK/dV work schedule), [1] before the dK/dV
 *                        kernel, [2] before the dQ kernel (which also writes
 *                        the keep tokens' dK / dV rows), [3] after it.
 * Indices past n_events are skipped.  The handles stay owned by the caller
 * and must outlive their registration.
 * Errors: SEP_ERR_INVALID_ARG (n_events out of range, or events NULL with
 * n_events > 0). */
#define SEP_MAX_PROFILE_EVENTS 8
sep_status sep_profile_events(void* const* events, int n_events);

/* sep_selftest_wait_timeout -- exercises the failure path every kernel's
 * bounded waits share (no counterpart in the paper).  Launches one thread
 * that waits on a shared-memory mbarrier whose arrival never comes; after
 * limit_us microseconds (1 .. 1000000) the wait gives up, the kernel writes
 * SEP_ERR_TIMEOUT to the device status word and returns.  Nothing traps and
 * the context stays usable: sep_get_device_status() then returns
 * SEP_ERR_TIMEOUT (and clears it).  Asynchronous on `stream`.
 * Errors: SEP_ERR_INVALID_ARG, SEP_ERR_CUDA. */
sep_status sep_selftest_wait_timeout(int limit_us, void* stream);

/* Static English text for a status code. */
const char* sep_status_string(sep_status s);

#ifdef __cplusplus
}
#endif

#endif /* SEPATTN_H */

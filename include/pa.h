/*
 * pa.h -- C ABI of the paged-attention library (libpa.so) for GB300 (sm_103a).
 *
 * Exact causal grouped-query attention over a paged KV cache.  The hot path:
 *   pa_write_kv        scatter new K/V rows into their pages,
 *   pa_prefill         causal prefill of a packed batch of prompts (tcgen05 / TMEM),
 *   pa_decode          one query per sequence over its whole cache (split-KV + LSE merge).
 * Around it:
 *   pa_prefill_cached  prefill of query chunks over a cached prefix (chunked prefill),
 *   pa_write_kv_rope   rotary embedding of K fused into the scatter,
 *   pa_prefill_rope    pa_prefill_cached with rotary embedding of Q in the kernel's prologue,
 *   pa_alloc_pages, pa_release_slots   page allocation on the device, table in place,
 *   pa_prefill_backward  gradients of the prefill (tcgen05 / TMEM),
 *   pa_decode_noalloc  pa_decode with the library's fixed scratch instead of a workspace,
 *   pa_page_bytes, pa_decode_workspace_size, pa_status_string   sizes and messages,
 *   pa_debug_hold_first_copy  diagnostic that makes a kernel's bounded wait run out (tests).
 *
 * The problem statement follows these web pages (cited by title and section):
 *  - jaehun.me, "6. KV cache 를 16토큰 블록으로 쪼개기 -- block table 로 비연속 블록을
 *    읽는 법" (tiny-vllm part 6): page layout ("블록 하나가 담는 것: K 는 앞, V 는
 *    V_OFFSET 뒤"), block table ("block table: slot·레이어·논리 블록 세 항목의 배열"),
 *    address and length rule ("논리 블록 → 물리 블록 → 바이트 주소"), in-place output
 *    ("출력은 입력 자리에: in-place").
 *  - jaehun.me, "3. The prefill path: flowing the entire prompt at once"
 *    (tiny-vllm part 3): K/V scatter ("Distributing K/V into paged blocks"), GQA
 *    ("Per-head attention scores and GQA"), causal mask and merge rule
 *    ("causalMask and online softmax").
 *  - base.kaita.kr, "플래시어텐션-2: 더 나은 병렬화" (FlashAttention-2 explainer):
 *    deferred normalisation and L = m + log l ("단계별 설명 (순전파의 두 가지 손질)"),
 *    causal tile skipping ("인과 마스크 처리"), GQA by index ("4. MQA · GQA 지원").
 *
 * Memory layout (all bf16 = IEEE binary32 upper half, little-endian):
 *   page (block) of 16 tokens: K[16][KV_DIM] then V[16][KV_DIM], KV_DIM = Hkv * d;
 *     page bytes = 64 * KV_DIM (32768 for 8 x 64); V starts 32 * KV_DIM bytes in.
 *     Token t of page p, kv head h, dim k: K at p*page_bytes + t*KV_DIM*2 + h*d*2 + k*2.
 *   pool: num_blocks pages, contiguous.
 *   block_table: int32 [num_slots][n_layers][max_blocks_per_seq], -1 = unassigned;
 *     token pos of (slot, layer) lives in page block_table[slot][layer][pos / 16].
 *   q, o (prefill): [total_tokens][Hq][d] bf16, sequence b owns rows
 *     cu_seqlens[b] .. cu_seqlens[b+1]-1; q, o (decode): [batch][Hq][d] bf16.
 *   lse: fp32, prefill [total_tokens][Hq], decode [batch][Hq]; natural-log
 *     log-sum-exp of the scaled scores, L = m + ln l.
 *   GQA: q head h reads kv head h / (Hq / Hkv).
 *
 * Ownership: the caller allocates and owns every buffer (device memory unless
 * stated).  The library keeps no state between calls and allocates no memory,
 * with two exceptions described at their calls: pa_decode_noalloc's fixed
 * scratch, and the few MB of scratch pa_prefill_cached takes for a
 * key-split last wave from a stream-ordered memory pool of the library's
 * own.
 * All calls are asynchronous on `stream`; they return after validating the
 * arguments and enqueueing the kernels.
 *
 * Errors:
 *   synchronous   -- the return value (PA_ERR_INVALID_ARG, PA_ERR_UNSUPPORTED,
 *                    PA_ERR_CUDA); nothing is enqueued when it is not PA_OK.
 *   asynchronous  -- kernels report data errors through *err_flag (device int32):
 *                    PA_ERR_BAD_BLOCK for a table entry that is -1 or >= num_blocks
 *                    where a page is needed, a slot outside [0, num_slots), a
 *                    position beyond 16 * max_blocks_per_seq, or lengths that do
 *                    not fit the call; PA_ERR_TIMEOUT if a bounded wait inside a
 *                    kernel ran out; PA_ERR_OUT_OF_PAGES if a page allocation
 *                    would take more pages than the free stack holds.  The offending page or row is skipped (its
 *                    output is unspecified) and the kernel never traps.  The caller
 *                    zeroes *err_flag before the call and reads it after
 *                    synchronising; the first error code written is kept.
 */
#ifndef PA_H
#define PA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* pa_stream_t;

typedef enum pa_status {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1,  /* null pointer, bad size, misaligned or aliased buffer */
    PA_ERR_UNSUPPORTED = 2,  /* valid request outside what the kernels implement */
    PA_ERR_CUDA = 3,         /* a CUDA runtime call or kernel launch failed */
    PA_ERR_BAD_BLOCK = 4,    /* device-reported through err_flag (see above) */
    PA_ERR_TIMEOUT = 5,      /* device-reported through err_flag (see above) */
    PA_ERR_OUT_OF_PAGES = 6  /* device-reported: the free stack ran short (or would overflow) */
} pa_status;

/* Tokens per page; fixed ("BLOCK_SIZE = 16", tiny-vllm part 6, page layout). */
#define PA_BLOCK_TOKENS 16

/* Cache geometry, validated on every call. */
typedef struct pa_geom {
    int32_t num_q_heads;        /* Hq > 0, a multiple of Hkv */
    int32_t num_kv_heads;       /* Hkv > 0 */
    int32_t head_dim;           /* d: 64 or 128 for attention; any multiple of 8 for write */
    int32_t n_layers;           /* table dimension 1 */
    int32_t num_slots;          /* table dimension 0 */
    int32_t max_blocks_per_seq; /* table dimension 2 */
    int64_t num_blocks;         /* pages in the pool */
} pa_geom;

/* Bytes of one page: 2 (K, V) * 16 tokens * Hkv * d * 2 bytes.  0 for a NULL
 * or invalid geometry. */
size_t pa_page_bytes(const pa_geom* geom);

/*
 * pa_write_kv -- scatter n_tokens new K/V rows into their pages.
 * Definition: row i of k_new / v_new (each [n_tokens][KV_DIM] bf16, row-major)
 * is copied to the K / V row of token tok_pos[i] of (tok_slot[i], layer):
 *   pool + blk * page_bytes + (pos % 16) * KV_DIM * 2      (K)
 *   ... + 32 * KV_DIM                                      (V)
 * with blk = block_table[slot][layer][pos / 16] (tiny-vllm part 6, page
 * layout; part 3, "Distributing K/V into paged blocks").  Bytes of the pool
 * not named by a valid row are left untouched; the copy is bit-exact.
 * Arguments: tok_slot, tok_pos: device int32 [n_tokens]; pool, k_new, v_new:
 * device, 16-byte aligned; k_new / v_new must not overlap the pool.  Pages
 * are not allocated here: the caller fills block_table first.  Two rows with
 * the same (slot, layer, pos) in one call leave either row's bytes.
 * Rows with an invalid slot, position or table entry are skipped and set
 * *err_flag = PA_ERR_BAD_BLOCK.  n_tokens == 0 is a no-op.
 */
pa_status pa_write_kv(const pa_geom* geom, void* pool, const int32_t* block_table,
                      int32_t layer, int32_t n_tokens, const int32_t* tok_slot,
                      const int32_t* tok_pos, const void* k_new, const void* v_new,
                      int32_t* err_flag, pa_stream_t stream);

/*
 * pa_write_kv_rope -- pa_write_kv with RoPE applied to K on the way into the
 * pages (jaehun.me tiny-vllm part 3, "RoPE: a rotation that references a
 * table"): in every kv head, element i and element i + head_dim/2 of row t's
 * K form a pair rotated by the angle of position tok_pos[t],
 *   x1' = x1 c - x2 s,   x2' = x1 s + x2 c,
 * with c = cos_table[tok_pos[t]][i], s = sin_table[tok_pos[t]][i], computed in
 * fp32 with every product and sum rounded on its own, then rounded to bf16
 * (nearest even).  V is stored unchanged, exactly as pa_write_kv.
 * Arguments: as pa_write_kv, plus cos_table, sin_table: device fp32
 * [max_pos][head_dim/2], 16-byte aligned, read only (the caller fills them,
 * e.g. with cos/sin of pos * base^(-2i/head_dim) and any frequency scaling its
 * model uses).  Rows with tok_pos >= max_pos are skipped and set
 * PA_ERR_BAD_BLOCK like an invalid table entry.  Requires head_dim % 16 == 0.
 */
pa_status pa_write_kv_rope(const pa_geom* geom, void* pool, const int32_t* block_table,
                           int32_t layer, int32_t n_tokens, const int32_t* tok_slot,
                           const int32_t* tok_pos, const void* k_new, const void* v_new,
                           const float* cos_table, const float* sin_table, int32_t max_pos,
                           int32_t* err_flag, pa_stream_t stream);

/*
 * pa_prefill -- causal prefill of a packed batch of fresh prompts.
 * Definition: for sequence b of length n_b = cu_seqlens[b+1] - cu_seqlens[b]
 * (slot slots[b]), query row i (0 <= i < n_b) of q head h attends keys 0..i of
 * (slots[b], layer), kv head h / (Hq/Hkv):
 *   s_j = scale * <q_i, k_j>,  m = max_j s_j,  l = sum_j e^(s_j - m),
 *   o_i = sum_j e^(s_j - m) v_j / l,   lse_i = m + ln l.
 * (FlashAttention-2 explainer, "단계별 설명"; tiny-vllm part 3, "Per-head
 * attention scores and GQA" and "causalMask and online softmax".)
 * Arguments: q, o: device bf16 [total_tokens][Hq][d], 16-byte aligned; o may
 * alias q (each output row is written only after every read of its query
 * row).  lse: device fp32 [total_tokens][Hq] or NULL.  cu_seqlens: device int32
 * [batch+1], cu_seqlens[0] = 0, non-decreasing, cu_seqlens[batch] <=
 * total_tokens.  slots: device int32 [batch].  max_seqlen: host upper bound on
 * every n_b (sizes the grid; longer sequences set PA_ERR_BAD_BLOCK).
 * total_tokens: host row count of q / o.  scale: finite and > 0 (else
 * PA_ERR_INVALID_ARG).  Requires d in {64, 128}.  Rows of q not covered by
 * cu_seqlens are neither read for output nor written.
 */
pa_status pa_prefill(const pa_geom* geom, const void* q, const void* pool,
                     const int32_t* block_table, int32_t layer, int32_t batch,
                     const int32_t* cu_seqlens, const int32_t* slots, int32_t max_seqlen,
                     int32_t total_tokens, float scale, void* o, float* lse,
                     int32_t* err_flag, pa_stream_t stream);

/*
 * pa_prefill_cached -- causal prefill of query chunks over a cached prefix
 * (chunked prefill).
 * Definition: the cache of (slots[b], layer) already holds prefix_lens[b]
 * tokens followed by the K/V of sequence b's n_b = cu_seqlens[b+1] -
 * cu_seqlens[b] new tokens (written with pa_write_kv before this call); the
 * i-th query row of sequence b sits at position prefix_lens[b] + i and
 * attends keys 0..prefix_lens[b] + i, with the scores, softmax, o and lse of
 * pa_prefill.  This is the decode's rule that a query reads the cache up to
 * and including its own token (tiny-vllm part 6, "논리 블록 → 물리 블록 →
 * 바이트 주소") applied to every query of the chunk, with the prompt's causal
 * mask inside the chunk (part 3, "causalMask and online softmax").
 * prefix_lens == NULL means all zero (pa_prefill); a chunk of one query at
 * prefix seq_len - 1 is pa_decode's result for that sequence.
 * Arguments: as pa_prefill, plus prefix_lens: device int32 [batch] or NULL,
 * each >= 0 with prefix_lens[b] + n_b <= 16 * max_blocks_per_seq (larger or
 * negative values set PA_ERR_BAD_BLOCK and leave that sequence's output
 * unspecified).  max_seqlen bounds the chunk lengths n_b only.
 * With a prefix array, work items that would leave the GPU's last wave
 * partly idle run as two halves of their key range whose fp32 partials are
 * combined by the LSE rule (part 3, "causalMask and online softmax"): the
 * result is deterministic and agrees with the NULL-prefix call to rounding,
 * not bit for bit.  Those halves take a few MB of scratch from a stream-
 * ordered memory pool of the library's own, allocated and freed on `stream`
 * (kept for the process); if it cannot be had, the call runs without it.
 */
pa_status pa_prefill_cached(const pa_geom* geom, const void* q, const void* pool,
                            const int32_t* block_table, int32_t layer, int32_t batch,
                            const int32_t* cu_seqlens, const int32_t* prefix_lens,
                            const int32_t* slots, int32_t max_seqlen, int32_t total_tokens,
                            float scale, void* o, float* lse, int32_t* err_flag,
                            pa_stream_t stream);

/*
 * pa_prefill_rope -- pa_prefill_cached with RoPE applied to the queries in the
 * kernel's prologue (jaehun.me tiny-vllm part 3, "RoPE: a rotation that
 * references a table": the program turns Q and K with the same tables before
 * the scores; K turns on its way into the pages, pa_write_kv_rope).
 * Definition: the i-th query row of sequence b sits at position
 * prefix_lens[b] + i (prefix_lens NULL: 0), the position its K row was
 * written at; in each q head, element k and element k + head_dim/2 turn by
 * the angle of that position exactly as pa_write_kv_rope turns K (fp32, every
 * product and sum rounded on its own, then bf16 nearest even), and the scores,
 * softmax, o and lse are pa_prefill_cached's on the turned rows.  q itself is
 * not modified; o may alias q.
 * Arguments: as pa_prefill_cached, plus cos_table, sin_table: device fp32
 * [max_pos][head_dim/2], 16-byte aligned (the tables given to
 * pa_write_kv_rope).  max_pos >= 0 (else PA_ERR_INVALID_ARG).  A query row
 * whose position is >= max_pos sets PA_ERR_BAD_BLOCK (its output is then
 * unspecified).
 */
pa_status pa_prefill_rope(const pa_geom* geom, const void* q, const void* pool,
                          const int32_t* block_table, int32_t layer, int32_t batch,
                          const int32_t* cu_seqlens, const int32_t* prefix_lens,
                          const int32_t* slots, int32_t max_seqlen, int32_t total_tokens,
                          float scale, const float* cos_table, const float* sin_table,
                          int32_t max_pos, void* o, float* lse, int32_t* err_flag,
                          pa_stream_t stream);

/*
 * pa_prefill_backward -- gradients of pa_prefill's output with respect to q
 * and to the K / V rows it read from the pages (training only).
 * Definition: with s_ij = scale <q_i, k_j> (j <= i), p_ij = e^(s_ij - L_i)
 * recomputed from the stored L = lse (FlashAttention-2 explainer, "전체
 * 흐름": the backward rebuilds P from L), do = dout and o the forward output:
 *   D_i = <do_i, o_i>,  dp_ij = <do_i, v_j>,  ds_ij = p_ij (dp_ij - D_i),
 *   dv_j = sum_i p_ij do_i,  dk_j = scale sum_i ds_ij q_i,  dq_i = scale sum_j ds_ij k_j,
 * with dk, dv summed over the q heads of each kv head's group ("4. MQA · GQA
 * 지원").  Work is split by key blocks, dq contributions are added atomically
 * ("2. 시퀀스 길이 방향으로도 병렬화", item 4), so dq's low bits vary from run
 * to run; dk and dv do not.
 * Arguments: q, pool, block_table, layer, batch, cu_seqlens, slots,
 * max_seqlen, total_tokens, scale: exactly those of the pa_prefill call whose
 * gradients are wanted (the pages must still hold the same K/V).  o: device
 * bf16 [total_tokens][Hq][d] and lse: device fp32 [total_tokens][Hq], that
 * call's outputs.  dout: device bf16 [total_tokens][Hq][d].  delta: device fp32
 * workspace of 2 * total_tokens * Hq floats (overwritten: -L log2 e, then -D).  dq: device fp32
 * [total_tokens][Hq][d], set to zero first (every row).  dk, dv: device fp32
 * [total_tokens][Hkv][d], row t is the gradient of the K / V row written for
 * token t; rows not covered by cu_seqlens are not written.  q, o, dout, dq,
 * dk, dv and pool 16-byte aligned; lse, delta 4-byte aligned.  Requires d in
 * {64, 128} and max_seqlen <= 4194240.  Bad lengths, slots or table entries
 * set PA_ERR_BAD_BLOCK (the gradients of that sequence are then unspecified).
 */
pa_status pa_prefill_backward(const pa_geom* geom, const void* q, const void* pool,
                              const int32_t* block_table, int32_t layer, int32_t batch,
                              const int32_t* cu_seqlens, const int32_t* slots, int32_t max_seqlen,
                              int32_t total_tokens, float scale, const void* o, const float* lse,
                              const void* dout, float* delta, float* dq, float* dk, float* dv,
                              int32_t* err_flag, pa_stream_t stream);

/*
 * pa_decode_workspace_size -- bytes of device workspace pa_decode needs for
 * up to `batch` sequences of up to `max_seq_len` tokens.  Depends only on the
 * geometry and these two numbers (not on the device).  0 for invalid input.
 */
size_t pa_decode_workspace_size(const pa_geom* geom, int32_t batch, int32_t max_seq_len);

/*
 * pa_decode -- one query per sequence over its whole cache.
 * Definition: query b (q[b], slot slots[b]) sits at position seq_lens[b]-1 and
 * attends keys 0..seq_lens[b]-1; the length includes the token just written
 * (tiny-vllm part 6, "논리 블록 → 물리 블록 → 바이트 주소").  Same scores,
 * softmax, o and lse as pa_prefill; seq_lens[b] == 0 gives o = 0, lse = -inf.
 * The keys of long sequences are split across CTAs; partial results are
 * merged by the rule m = max(m_a, m_b), l = l_a e^(m_a - m) + l_b e^(m_b - m)
 * (tiny-vllm part 3, "causalMask and online softmax"), applied to the
 * accumulated outputs as well.  The split depends only on the lengths and the
 * launch shape, never on physical page ids, so results are bit-identical
 * under any page permutation and from run to run.
 * Arguments: q, o: device bf16 [batch][Hq][d], 16-byte aligned; o may alias q.
 * lse: device fp32 [batch][Hq] or NULL.  seq_lens, slots: device int32
 * [batch].  max_seq_len: host upper bound on every seq_len (sizes the grid
 * and the workspace; lengths beyond 16 * max_blocks_per_seq set
 * PA_ERR_BAD_BLOCK).  workspace: device, 16-byte aligned, at least
 * pa_decode_workspace_size(geom, batch, max_seq_len) bytes, contents need not
 * be initialised, not shared with a concurrent call.  scale: finite and > 0
 * (else PA_ERR_INVALID_ARG).  Requires d in {64, 128}, Hq/Hkv in {1, 2, 4, 8},
 * Hkv <= 8 and a page of at most 64 KiB (else PA_ERR_UNSUPPORTED).
 */
pa_status pa_decode(const pa_geom* geom, const void* q, const void* pool,
                    const int32_t* block_table, int32_t layer, int32_t batch,
                    const int32_t* seq_lens, const int32_t* slots, int32_t max_seq_len,
                    float scale, void* o, float* lse, void* workspace, size_t workspace_bytes,
                    int32_t* err_flag, pa_stream_t stream);

/*
 * PA_DECODE_STATIC_SCRATCH_BYTES / pa_decode_noalloc -- decode without a
 * caller-provided workspace.  The paper has no counterpart to this call; it
 * exists for callers that cannot allocate device memory at the point where
 * they decode: for example a plugin inside a host application that reserves
 * all device memory up front for its own allocator, or a serving loop that
 * must not call cudaMalloc (which can synchronise the device) between steps.
 *
 * Same arguments, definition and results as pa_decode, minus the workspace.
 * The split partials go to a fixed scratch array of
 * PA_DECODE_STATIC_SCRATCH_BYTES that lives inside libpa.so's device code:
 * every GPU on which the library's kernels are loaded holds these bytes until
 * the process exits.  The call allocates nothing.
 *   - Size limit: a request whose pa_decode_workspace_size(geom, batch,
 *     max_seq_len) exceeds PA_DECODE_STATIC_SCRATCH_BYTES is rejected with
 *     PA_ERR_UNSUPPORTED before anything is enqueued (use pa_decode then).
 *   - Set-up: the first call on each device (with that device current) looks
 *     up the scratch array's device address; make that first call before any
 *     stream capture.  The address is kept for the life of the process: after
 *     a cudaDeviceReset (or anything else that destroys and re-creates the
 *     device's primary context) the kept address is stale, so do not call
 *     pa_decode_noalloc on that device again in the same process.
 *   - Checks: the arguments are checked exactly as pa_decode checks them
 *     (same status codes, an empty batch is a no-op) before the size check
 *     and the set-up.
 *   - Sharing: every call on a device uses the same scratch, which keeps the
 *     previous call's contents (nothing in it needs to start at zero).  Calls
 *     that can overlap on the GPU -- on different streams without ordering,
 *     or from different host threads -- race on it; serialise them.
 */
#define PA_DECODE_STATIC_SCRATCH_BYTES (16u << 20)

pa_status pa_decode_noalloc(const pa_geom* geom, const void* q, const void* pool,
                            const int32_t* block_table, int32_t layer, int32_t batch,
                            const int32_t* seq_lens, const int32_t* slots, int32_t max_seq_len,
                            float scale, void* o, float* lse, int32_t* err_flag,
                            pa_stream_t stream);

/*
 * Page lifetime on the device (NEXT to the hot path: keeps the block table
 * resident instead of copying it from the host after every change).
 * The free stack is free_pages[0 .. *free_count - 1] (device int32
 * [num_blocks] and a device int32), its top last; the caller fills it once
 * (e.g. with 0 .. num_blocks - 1) and owns both buffers.  Calls that touch the
 * same stack or table must not overlap on the GPU (they race).
 *
 * pa_alloc_pages -- every logical block that positions 0 .. seq_lens[b] - 1 of
 * slots[b] need, in every layer, whose table entry is -1 takes the page on top
 * of the stack, walking sequences in order, then layers, then logical blocks
 * (tiny-vllm part 6, "물리 블록의 수명: free_blocks 가 관리한다": a page is
 * popped when a logical block's entry is -1, a prompt's blocks at prefill and a
 * new block when a decode step's token starts one).  Entries below
 * old_lens[b] / 16 are not looked at (old_lens: device int32 [batch] or NULL
 * for 0).  All or nothing: if the stack holds fewer pages than needed, nothing
 * changes and *err_flag gets PA_ERR_OUT_OF_PAGES; an invalid slot or length
 * sets PA_ERR_BAD_BLOCK, also with nothing changed, as does a slot named
 * twice in one call.  slots, seq_lens: device int32 [batch]; block_table:
 * device, the layout of pa_write_kv.  Both calls require geom->num_slots <=
 * PA_PAGES_MAX_SLOTS (else PA_ERR_UNSUPPORTED before anything is enqueued):
 * the kernels keep one bit per slot in shared memory to refuse a slot named
 * twice.
 *
 * pa_release_slots -- every page held by slots[0 .. n-1], in every layer, goes
 * back on the stack in the same walking order and its entry becomes -1 (the
 * pages' slot-end loop).  Nothing changes (PA_ERR_OUT_OF_PAGES) if the stack
 * would grow past num_blocks, which means a page was freed twice.
 */
#define PA_PAGES_MAX_SLOTS 65536

pa_status pa_alloc_pages(const pa_geom* geom, int32_t* block_table, int32_t batch,
                         const int32_t* slots, const int32_t* old_lens, const int32_t* seq_lens,
                         int32_t* free_pages, int32_t* free_count, int32_t* err_flag,
                         pa_stream_t stream);
pa_status pa_release_slots(const pa_geom* geom, int32_t* block_table, int32_t n,
                           const int32_t* slots, int32_t* free_pages, int32_t* free_count,
                           int32_t* err_flag, pa_stream_t stream);

/*
 * pa_debug_hold_first_copy -- diagnostic for the bounded waits inside the
 * kernels (tests only; the pages have no counterpart).  While enabled, the
 * first CTA of every later pa_prefill / pa_prefill_cached / pa_prefill_rope /
 * pa_decode launch arms the barrier of its first tensor copy (the query tiles
 * of the prefill, the first page of the decode) without issuing the copy, so
 * that barrier's phase never completes and the roles waiting on it give up
 * after the kernels' wait limit of about 2 seconds.  That CTA then records
 * PA_ERR_TIMEOUT in *err_flag, tells its other roles to stop, lets every copy
 * it did issue land, frees its tensor memory and returns; no kernel traps and
 * the context stays usable.  The outputs of that call are unspecified; other
 * CTAs run normally.  Process-wide, not to be changed while a call is being
 * enqueued on another thread.  enable = 0 restores normal operation (the
 * default).  Returns PA_OK.
 */
pa_status pa_debug_hold_first_copy(int32_t enable);

/* Static, NUL-terminated description of a status code. */
const char* pa_status_string(pa_status status);

#ifdef __cplusplus
}
#endif
#endif /* PA_H */

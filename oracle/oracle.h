/*
 * oracle.h -- plain fp64 CPU oracle for causal grouped-query attention over a
 * paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this code; it exists so that tests, the smoke check and the timed CPU
 * baseline have an independent statement of what the GPU path must compute.
 * It shares no header, constant or helper with the CUDA sources.
 *
 * Sources (web pages; sections quoted by their headings):
 *  [TV3] jaehun.me, "3. The prefill path: flowing the entire prompt at once"
 *        (tiny-vllm series, part 3), sections "Distributing K/V into paged
 *        blocks", "Per-head attention scores and GQA", "causalMask and online
 *        softmax".
 *  [TV6] jaehun.me, "6. KV cache 를 16토큰 블록으로 쪼개기 -- block table 로
 *        비연속 블록을 읽는 법" (tiny-vllm series, part 6), sections
 *        "블록 하나가 담는 것: K 는 앞, V 는 V_OFFSET 뒤" (page layout),
 *        "block table: slot·레이어·논리 블록 세 항목의 배열" (table index),
 *        "논리 블록 → 물리 블록 → 바이트 주소" (address / length rule),
 *        "online softmax: 블록을 훑으며 가중 평균".
 *  [FA2] base.kaita.kr, "플래시어텐션-2: 더 나은 병렬화" (FlashAttention-2
 *        explainer), sections "단계별 설명 (순전파의 두 가지 손질)" (deferred
 *        normalisation, L = m + log l), "숫자로 해 보기 (해설용, 점수 4개 · 값
 *        4개를 2블록으로)" (worked example), "인과 마스크 처리" (causal mask),
 *        "4. MQA · GQA 지원".
 *
 * Parity status: every function here is pinned by tests/test_oracle_pins.py
 * (worked example, closed forms, invariants, a library SDPA on tiny cases).
 */
#ifndef PA_ORACLE_H
#define PA_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Cache geometry.  A block (page) holds 16 tokens; KV_DIM = num_kv_heads *
 * head_dim; a page is K[16][KV_DIM] followed by V[16][KV_DIM], bf16. */
typedef struct {
    int32_t num_q_heads;
    int32_t num_kv_heads;
    int32_t head_dim;
    int32_t n_layers;
    int32_t num_slots;
    int32_t max_blocks_per_seq;
    int64_t num_blocks;
} orc_geom;

/* Status codes returned by the oracle. */
#define ORC_OK 0
#define ORC_BAD_ARG (-1)
#define ORC_BAD_BLOCK (-2)

/* Byte scatter of new K/V rows into their pages [TV3 "Distributing K/V into
 * paged blocks"; TV6 page layout].  Rows whose slot, position or table entry
 * is invalid are skipped; the return value is the number of skipped rows
 * (>= 0) or ORC_BAD_ARG. */
int64_t orc_write_kv(const orc_geom* g, uint8_t* pool, const int32_t* block_table,
                     int32_t layer, int64_t n_tokens, const int32_t* tok_slot,
                     const int32_t* tok_pos, const uint16_t* k_new, const uint16_t* v_new);

/* Page lifetime on a free stack [TV6 "물리 블록의 수명: free_blocks 가
 * 관리한다"].  free_pages[0..*free_count-1] is the stack, its top last.
 * orc_alloc_pages: every logical block of positions 0..seq_lens[b]-1 of
 * slots[b], in every layer, whose entry is -1 pops the top page, walking
 * sequences, then layers, then logical blocks in order (entries below
 * old_lens[b] / 16 are not looked at; old_lens may be NULL); all or nothing
 * when the stack runs short.  orc_release_slots: every page held by the
 * slots goes back (push) in the same walking order and its entry becomes -1.
 * Both return the number of pages moved, or ORC_BAD_ARG with nothing
 * changed (also when a slot is named twice in one call). */
int64_t orc_alloc_pages(const orc_geom* g, int32_t* block_table, int32_t batch, const int32_t* slots,
                        const int32_t* old_lens, const int32_t* seq_lens, int32_t* free_pages,
                        int32_t* free_count);
int64_t orc_release_slots(const orc_geom* g, int32_t* block_table, int32_t n, const int32_t* slots,
                          int32_t* free_pages, int32_t* free_count);

/* orc_write_kv with K rotated by RoPE at each row's position [TV3 "RoPE: a
 * rotation that references a table"]: in every kv head, element i and
 * element i + head_dim/2 are rotated as
 *   x1' = x1 cos - x2 sin,   x2' = x1 sin + x2 cos
 * with cos/sin read from caller tables [max_pos][head_dim/2] fp32 at the row's
 * position, in fp32 with each product and sum rounded separately, then
 * rounded to bf16 (nearest even).  V is copied unchanged.  Rows at a position
 * >= max_pos count as skipped. */
int64_t orc_write_kv_rope(const orc_geom* g, uint8_t* pool, const int32_t* block_table,
                          int32_t layer, int64_t n_tokens, const int32_t* tok_slot,
                          const int32_t* tok_pos, const uint16_t* k_new, const uint16_t* v_new,
                          const float* cos_tab, const float* sin_tab, int32_t max_pos);

/* Query rows of a packed batch rotated by RoPE [TV3 "RoPE: a rotation that
 * references a table": Q and K are rotated with the same tables before the
 * scores].  The i-th query row of sequence b (rows cu_seqlens[b] ..
 * cu_seqlens[b+1]-1 of q[T][Hq][d], bf16 bits) sits at position
 * prefix_lens[b] + i (prefix_lens NULL: 0); each q head is rotated as
 * orc_write_kv_rope rotates a kv head of K, then rounded to bf16.  Writes
 * q_rot[T][Hq][d].  Returns ORC_OK, or ORC_BAD_ARG for a position >= max_pos
 * or bad lengths.  RoPE-Q prefill = orc_rope_q, then orc_prefill_cached on
 * q_rot. */
int orc_rope_q(const orc_geom* g, const uint16_t* q, int32_t batch, const int32_t* cu_seqlens,
               const int32_t* prefix_lens, const float* cos_tab, const float* sin_tab, int32_t max_pos,
               uint16_t* q_rot);

/* Gather the first n tokens of (slot, layer) into K[n][Hkv][d], V[n][Hkv][d]
 * (fp64) through the block table [TV6 address rule].  Returns ORC_OK or
 * ORC_BAD_BLOCK / ORC_BAD_ARG. */
int orc_gather_kv(const orc_geom* g, const uint8_t* pool, const int32_t* block_table,
                  int32_t layer, int32_t slot, int32_t n, double* K, double* V);

/* Softmax of one score row s[0..n) (entries may be -INFINITY = masked), as
 * the plain two-pass definition: m = max s, l = sum exp(s - m), w = exp(s - m)/l.
 * Writes w[n] (may be NULL), *m, *l.  n == 0 or all-masked gives l = 0. */
void orc_softmax_row(const double* s, int32_t n, double* w, double* m, double* l);

/* Un-normalised partial over one key subset [FA2 "단계별 설명"]: m = max s,
 * l = sum exp(s - m), acc[k] = sum exp(s_j - m) * v[j][k]; v is [n][dv]. */
void orc_partial(const double* s, const double* v, int32_t n, int32_t dv,
                 double* m, double* l, double* acc);

/* Merge of partials by their maxima [TV3 "causalMask and online softmax"
 * merge rule; FA2 worked example, block 2]: m* = max m_i,
 * l* = sum l_i e^(m_i - m*), acc* = sum acc_i e^(m_i - m*).  Outputs the
 * merged (m*, l*, acc*) and the normalised O = acc* / l*, L = m* + ln l*. */
void orc_merge(int32_t nparts, const double* m, const double* l, const double* acc,
               int32_t dv, double* m_out, double* l_out, double* acc_out,
               double* o, double* lse);

/* Causal prefill of a packed batch.  Sequence b owns query rows
 * cu_seqlens[b] .. cu_seqlens[b+1]-1 of q[T][Hq][d] (bf16 bits) and the cache
 * of slots[b]; query row i of a sequence attends keys 0..i.  Outputs
 * o[T][Hq][d] and lse[T][Hq] (fp64).  nthreads <= 0 means all cores.
 * Returns ORC_OK or an error status (nothing useful is written then). */
int orc_prefill(const orc_geom* g, const uint16_t* q, const uint8_t* pool,
                const int32_t* block_table, int32_t layer, int32_t batch,
                const int32_t* cu_seqlens, const int32_t* slots, float scale,
                double* o, double* lse, int32_t nthreads);

/* Same definition, evaluated only at nsamp (row, q head) pairs; rows index
 * the packed q.  o[nsamp][d], lse[nsamp]. */
int orc_prefill_rows(const orc_geom* g, const uint16_t* q, const uint8_t* pool,
                     const int32_t* block_table, int32_t layer, int32_t batch,
                     const int32_t* cu_seqlens, const int32_t* slots, float scale,
                     int64_t nsamp, const int64_t* rows, const int32_t* heads,
                     double* o, double* lse, int32_t nthreads);

/* Causal prefill of query chunks over a cached prefix.  The cache of slots[b]
 * already holds prefix_lens[b] tokens followed by the K/V of sequence b's
 * queries (rows cu_seqlens[b] .. cu_seqlens[b+1]-1); the i-th of them sits at
 * position prefix_lens[b] + i and attends keys 0..prefix_lens[b] + i (the
 * decode's "length includes the token just written" rule applied to every
 * query of the chunk [TV6 "논리 블록 → 물리 블록 → 바이트 주소"], with the
 * prompt's causal mask inside the chunk [TV3 "causalMask and online
 * softmax"]).  prefix_lens == NULL or all zero is orc_prefill; a chunk of one
 * query at prefix seq_len - 1 is orc_decode.  Outputs as orc_prefill. */
int orc_prefill_cached(const orc_geom* g, const uint16_t* q, const uint8_t* pool,
                       const int32_t* block_table, int32_t layer, int32_t batch,
                       const int32_t* cu_seqlens, const int32_t* prefix_lens, const int32_t* slots,
                       float scale, double* o, double* lse, int32_t nthreads);

/* orc_prefill_cached at nsamp (row, q head) pairs, as orc_prefill_rows. */
int orc_prefill_cached_rows(const orc_geom* g, const uint16_t* q, const uint8_t* pool,
                            const int32_t* block_table, int32_t layer, int32_t batch,
                            const int32_t* cu_seqlens, const int32_t* prefix_lens,
                            const int32_t* slots, float scale, int64_t nsamp, const int64_t* rows,
                            const int32_t* heads, double* o, double* lse, int32_t nthreads);

/* Gradients of the causal prefill (orc_prefill's definition) with respect to
 * q and to the K/V rows it reads, given the output gradient dout[T][Hq][d]
 * (bf16 bits): dq[T][Hq][d], and dk, dv[T][Hkv][d] for the prompt tokens in
 * packed row order, kv head h of row t holding the sum over the q heads that
 * read it [FA2 "4. MQA · GQA 지원"].  fp64, from the chain rule through the
 * softmax with p recomputed from the scores [FA2, 전체 흐름]. */
int orc_prefill_backward(const orc_geom* g, const uint16_t* q, const uint8_t* pool,
                         const int32_t* block_table, int32_t layer, int32_t batch,
                         const int32_t* cu_seqlens, const int32_t* slots, float scale,
                         const uint16_t* dout, double* dq, double* dk, double* dv, int32_t nthreads);

/* orc_prefill_backward at sampled outputs: dq[s] = dq of (q_rows[s],
 * q_heads[s]) for s < n_q, and dk[t], dv[t] = dk, dv of (k_rows[t], kv head
 * k_heads[t]) for t < n_k (rows in packed order), equal bit for bit to the
 * full call's entries; each row's statistics are computed once per (sequence,
 * q head) that a k sample needs. */
int orc_prefill_backward_rows(const orc_geom* g, const uint16_t* q, const uint8_t* pool,
                              const int32_t* block_table, int32_t layer, int32_t batch,
                              const int32_t* cu_seqlens, const int32_t* slots, float scale,
                              const uint16_t* dout, int64_t n_q, const int64_t* q_rows,
                              const int32_t* q_heads, double* dq, int64_t n_k, const int64_t* k_rows,
                              const int32_t* k_heads, double* dk, double* dv, int32_t nthreads);

/* Single-query decode [TV6 "논리 블록 → 물리 블록 → 바이트 주소"]: query b
 * (q[B][Hq][d]) attends keys 0..seq_lens[b]-1 of slots[b]; the length
 * includes the token just written.  seq_len 0 gives O = 0, L = -inf.
 * Outputs o[B][Hq][d], lse[B][Hq]. */
int orc_decode(const orc_geom* g, const uint16_t* q, const uint8_t* pool,
               const int32_t* block_table, int32_t layer, int32_t batch,
               const int32_t* seq_lens, const int32_t* slots, float scale,
               double* o, double* lse, int32_t nthreads);

/* Threads the oracle would use for nthreads <= 0. */
int32_t orc_default_threads(void);

#ifdef __cplusplus
}
#endif
#endif

/*
 * oracle.c -- plain fp64 CPU oracle for causal grouped-query attention over a
 * paged KV cache.  TEST INFRASTRUCTURE ONLY (tests, the smoke check and the
 * timed CPU baseline call it; the product library never does).
 *
 * It is the plain definition written out, with no tiling, fusion or
 * reordering beyond what the definition states:
 *   1. gather K/V of a sequence from its pages through the block table into
 *      contiguous fp64 arrays;
 *   2. scores s_j = scale * <q, k_j> for every key j, with keys j > i masked to
 *      -inf for query row i (causal);
 *   3. two-pass softmax: m = max_j s_j, l = sum_j e^(s_j - m),
 *      O = sum_j e^(s_j - m) v_j / l, L = m + ln l.
 * Citations name the web page and section; see oracle.h for the page list.
 * Readings taken where the pages are silent or garbled:
 *   - masked scores are exactly -inf (weight 0), not a finite sentinel;
 *   - L uses the natural log of the *scaled* scores (the FA2 worked example
 *     gives L = 3 + ln 1.553 = 3.440);
 *   - the GQA map is consecutive: kv head = q head / (Hq / Hkv);
 *   - KV_DIM = Hkv * head_dim in general (the pages fix 8 x 64 = 512).
 */
#define _DEFAULT_SOURCE
#include "oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* "BLOCK_SIZE = 16 tokens" [TV6 "블록 하나가 담는 것"]. */
#define TOKENS_PER_BLOCK 16

/* ---------------------------------------------------------------- layout */

/* KV_DIM: elements of one token's K (or V) row = kv heads x head dim
 * [TV6 "블록 하나가 담는 것": KV_DIM = 8 x 64 = 512]. */
static int64_t kv_dim(const orc_geom* g) { return (int64_t)g->num_kv_heads * g->head_dim; }

/* V_OFFSET = BLOCK_SIZE * KV_DIM * sizeof(bf16); BLOCK_BYTES = 2 * V_OFFSET
 * [TV6 "블록 하나가 담는 것": 16384 and 32768 bytes for KV_DIM 512]. */
static int64_t v_offset(const orc_geom* g) { return (int64_t)TOKENS_PER_BLOCK * kv_dim(g) * 2; }
static int64_t block_bytes(const orc_geom* g) { return 2 * v_offset(g); }

/* bf16 is the upper 16 bits of an IEEE binary32; the conversion is exact. */
static double bf16_to_double(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static int geom_ok(const orc_geom* g) {
    if (!g) return 0;
    if (g->num_q_heads <= 0 || g->num_kv_heads <= 0 || g->head_dim <= 0) return 0;
    if (g->num_q_heads % g->num_kv_heads != 0) return 0;
    if (g->n_layers <= 0 || g->num_slots <= 0 || g->max_blocks_per_seq <= 0) return 0;
    if (g->num_blocks <= 0) return 0;
    return 1;
}

/* Physical block holding token `pos` of (slot, layer), or -1 when the slot,
 * layer, position or table entry is out of range.  The flat table index is
 * slot * N_LAYERS * MAX_BLOCKS_PER_SEQ + layer * MAX_BLOCKS_PER_SEQ + block_idx
 * [TV6 "block table: slot·레이어·논리 블록 세 항목의 배열"]; -1 marks an
 * unassigned entry. */
static int64_t block_of(const orc_geom* g, const int32_t* block_table, int32_t slot,
                        int32_t layer, int64_t pos) {
    if (slot < 0 || slot >= g->num_slots) return -1;
    if (layer < 0 || layer >= g->n_layers) return -1;
    if (pos < 0) return -1;
    int64_t logical_block = pos / TOKENS_PER_BLOCK;
    if (logical_block >= g->max_blocks_per_seq) return -1;
    int64_t idx = (int64_t)slot * g->n_layers * g->max_blocks_per_seq +
                  (int64_t)layer * g->max_blocks_per_seq + logical_block;
    int32_t physical_block = block_table[idx];
    if (physical_block < 0 || physical_block >= g->num_blocks) return -1;
    return physical_block;
}

/* ----------------------------------------------------------- write_kv */

/* New token's K at kv_cache + block*BLOCK_BYTES + token_in_block*KV_DIM*2 and
 * V at the same address + V_OFFSET [TV6 "블록 하나가 담는 것", decode
 * write; TV3 "Distributing K/V into paged blocks" for the prefill chunks]. */
int64_t orc_write_kv(const orc_geom* g, uint8_t* pool, const int32_t* block_table,
                     int32_t layer, int64_t n_tokens, const int32_t* tok_slot,
                     const int32_t* tok_pos, const uint16_t* k_new, const uint16_t* v_new) {
    if (!geom_ok(g) || n_tokens < 0) return ORC_BAD_ARG;
    if (n_tokens == 0) return 0;
    if (!pool || !block_table || !tok_slot || !tok_pos || !k_new || !v_new) return ORC_BAD_ARG;
    const int64_t row_bytes = kv_dim(g) * 2;
    int64_t skipped = 0;
    for (int64_t t = 0; t < n_tokens; ++t) {
        int64_t blk = block_of(g, block_table, tok_slot[t], layer, tok_pos[t]);
        if (blk < 0) {
            ++skipped;
            continue;
        }
        int64_t token_in_block = tok_pos[t] % TOKENS_PER_BLOCK;
        uint8_t* k_dst = pool + blk * block_bytes(g) + token_in_block * row_bytes;
        uint8_t* v_dst = k_dst + v_offset(g);
        memcpy(k_dst, (const uint8_t*)k_new + t * row_bytes, (size_t)row_bytes);
        memcpy(v_dst, (const uint8_t*)v_new + t * row_bytes, (size_t)row_bytes);
    }
    return skipped;
}

/* bf16 bits of a float, round to nearest even (NaN stays a quiet NaN). */
static uint16_t float_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x0040u);
    const uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

static float bf16_to_float(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* RoPE of one row of `heads` heads (a K row: the kv heads; a query row: the
 * q heads) [TV3 "RoPE: a rotation that references a table"]: in each head,
 * element i and element i + d/2 form a pair rotated by the angle of the
 * token's position, read from caller tables cos/sin[pos][d/2]:
 *   x1' = x1 c - x2 s,   x2' = x1 s + x2 c,
 * in fp32 with every product and sum rounded on its own (this file is built
 * as ISO C, so nothing is contracted into an FMA), then rounded to bf16. */
static void rope_row(const orc_geom* g, int32_t heads, const uint16_t* k, const float* cos_row,
                     const float* sin_row, uint16_t* out) {
    const int32_t d = g->head_dim, half = d / 2;
    for (int32_t h = 0; h < heads; ++h) {
        const uint16_t* x = k + (int64_t)h * d;
        uint16_t* y = out + (int64_t)h * d;
        for (int32_t i = 0; i < half; ++i) {
            const float x1 = bf16_to_float(x[i]), x2 = bf16_to_float(x[i + half]);
            const float c = cos_row[i], s = sin_row[i];
            const float a = x1 * c, b = x2 * s, e = x1 * s, f = x2 * c;
            const float y1 = a - b, y2 = e + f;
            y[i] = float_to_bf16(y1);
            y[i + half] = float_to_bf16(y2);
        }
    }
}

/* orc_write_kv with K rotated by RoPE at each row's position; V is copied.
 * Rows with a position >= max_pos are skipped like invalid table entries. */
int64_t orc_write_kv_rope(const orc_geom* g, uint8_t* pool, const int32_t* block_table,
                          int32_t layer, int64_t n_tokens, const int32_t* tok_slot,
                          const int32_t* tok_pos, const uint16_t* k_new, const uint16_t* v_new,
                          const float* cos_tab, const float* sin_tab, int32_t max_pos) {
    if (!geom_ok(g) || n_tokens < 0 || max_pos < 0 || (g->head_dim & 1)) return ORC_BAD_ARG;
    if (n_tokens == 0) return 0;
    if (!pool || !block_table || !tok_slot || !tok_pos || !k_new || !v_new || !cos_tab || !sin_tab)
        return ORC_BAD_ARG;
    const int64_t row_bytes = kv_dim(g) * 2;
    const int32_t half = g->head_dim / 2;
    uint16_t* rot = (uint16_t*)malloc((size_t)row_bytes);
    if (!rot) return ORC_BAD_ARG;
    int64_t skipped = 0;
    for (int64_t t = 0; t < n_tokens; ++t) {
        int64_t blk = block_of(g, block_table, tok_slot[t], layer, tok_pos[t]);
        if (blk < 0 || tok_pos[t] >= max_pos) {
            ++skipped;
            continue;
        }
        rope_row(g, g->num_kv_heads, k_new + t * kv_dim(g), cos_tab + (int64_t)tok_pos[t] * half,
                 sin_tab + (int64_t)tok_pos[t] * half, rot);
        int64_t token_in_block = tok_pos[t] % TOKENS_PER_BLOCK;
        uint8_t* k_dst = pool + blk * block_bytes(g) + token_in_block * row_bytes;
        uint8_t* v_dst = k_dst + v_offset(g);
        memcpy(k_dst, rot, (size_t)row_bytes);
        memcpy(v_dst, (const uint8_t*)v_new + t * row_bytes, (size_t)row_bytes);
    }
    free(rot);
    return skipped;
}

/* Query rows of a packed batch rotated at their positions [TV3 "RoPE: a
 * rotation that references a table": the program rotates Q and K with the
 * same kernel and tables before the scores].  The i-th query row of sequence
 * b sits at position prefix[b] + i (prefix NULL: 0), the position its K row
 * was written at; each of its q heads turns exactly as a kv head of K. */
int orc_rope_q(const orc_geom* g, const uint16_t* q, int32_t batch, const int32_t* cu_seqlens,
               const int32_t* prefix_lens, const float* cos_tab, const float* sin_tab, int32_t max_pos,
               uint16_t* q_rot) {
    if (!geom_ok(g) || batch < 0 || !cu_seqlens || max_pos < 0 || (g->head_dim & 1)) return ORC_BAD_ARG;
    if (cu_seqlens[0] != 0) return ORC_BAD_ARG;
    const int32_t half = g->head_dim / 2;
    const int64_t row = (int64_t)g->num_q_heads * g->head_dim;
    for (int32_t b = 0; b < batch; ++b) {
        const int32_t pre = prefix_lens ? prefix_lens[b] : 0;
        if (cu_seqlens[b + 1] < cu_seqlens[b] || pre < 0) return ORC_BAD_ARG;
        for (int64_t t = cu_seqlens[b]; t < cu_seqlens[b + 1]; ++t) {
            const int64_t pos = (int64_t)pre + (t - cu_seqlens[b]);
            if (pos >= max_pos || !q || !q_rot || !cos_tab || !sin_tab) return ORC_BAD_ARG;
            rope_row(g, g->num_q_heads, q + t * row, cos_tab + pos * half, sin_tab + pos * half, q_rot + t * row);
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------ page lifetime */

/* Every logical block that positions 0..seq_lens[b]-1 of slots[b] need gets a
 * physical page, in every layer: a table entry that is -1 takes the page on
 * top of the free stack (pop_back), walking sequences in order, then layers,
 * then logical blocks [TV6 "물리 블록의 수명: free_blocks 가 관리한다": prefill
 * takes a page when its logical block is -1, decode when a new block starts].
 * Entries below old_lens[b] / 16 (old_lens may be NULL) are not looked at.
 * All or nothing: when the stack holds fewer pages than needed nothing
 * changes and ORC_BAD_ARG is returned.  Returns the number of pages taken. */
int64_t orc_alloc_pages(const orc_geom* g, int32_t* block_table, int32_t batch, const int32_t* slots,
                        const int32_t* old_lens, const int32_t* seq_lens, int32_t* free_pages,
                        int32_t* free_count) {
    if (!geom_ok(g) || batch < 0 || !block_table || !free_pages || !free_count) return ORC_BAD_ARG;
    if (batch > 0 && (!slots || !seq_lens)) return ORC_BAD_ARG;
    for (int32_t b = 0; b < batch; ++b) /* a slot named twice is refused */
        for (int32_t c = 0; c < b; ++c)
            if (slots[c] == slots[b]) return ORC_BAD_ARG;
    const int32_t mb = g->max_blocks_per_seq;
    int64_t need = 0;
    for (int pass = 0; pass < 2; ++pass) {
        int32_t top = *free_count;
        for (int32_t b = 0; b < batch; ++b) {
            const int32_t slot = slots[b], len = seq_lens[b];
            if (slot < 0 || slot >= g->num_slots || len < 0 || len > mb * TOKENS_PER_BLOCK) return ORC_BAD_ARG;
            const int32_t lo = old_lens ? old_lens[b] / TOKENS_PER_BLOCK : 0;
            const int32_t hi = (len + TOKENS_PER_BLOCK - 1) / TOKENS_PER_BLOCK;
            for (int32_t layer = 0; layer < g->n_layers; ++layer)
                for (int32_t lb = lo < 0 ? 0 : lo; lb < hi; ++lb) {
                    int32_t* e = block_table + ((int64_t)slot * g->n_layers + layer) * mb + lb;
                    if (*e != -1) continue;
                    if (pass == 0) {
                        ++need;
                    } else {
                        *e = free_pages[--top]; /* pop_back */
                    }
                }
        }
        if (pass == 0 && need > *free_count) return ORC_BAD_ARG;
        if (pass == 1) *free_count = top;
    }
    return need;
}

/* Every page held by slots[0..n-1], in every layer, goes back on the free
 * stack (push_back), walking slots in order, then layers, then logical
 * blocks, and its table entry becomes -1 [TV6 "물리 블록의 수명: free_blocks
 * 가 관리한다": the loop that ends a slot].  Returns the pages returned, or
 * ORC_BAD_ARG (nothing changes) when the stack would overflow num_blocks. */
int64_t orc_release_slots(const orc_geom* g, int32_t* block_table, int32_t n, const int32_t* slots,
                          int32_t* free_pages, int32_t* free_count) {
    if (!geom_ok(g) || n < 0 || !block_table || !free_pages || !free_count) return ORC_BAD_ARG;
    if (n > 0 && !slots) return ORC_BAD_ARG;
    for (int32_t i = 0; i < n; ++i) /* a slot named twice is refused */
        for (int32_t c = 0; c < i; ++c)
            if (slots[c] == slots[i]) return ORC_BAD_ARG;
    const int32_t mb = g->max_blocks_per_seq;
    int64_t held = 0;
    for (int32_t i = 0; i < n; ++i) {
        if (slots[i] < 0 || slots[i] >= g->num_slots) return ORC_BAD_ARG;
        for (int64_t k = 0; k < (int64_t)g->n_layers * mb; ++k)
            if (block_table[(int64_t)slots[i] * g->n_layers * mb + k] != -1) ++held;
    }
    if (*free_count + held > g->num_blocks) return ORC_BAD_ARG;
    int32_t top = *free_count;
    for (int32_t i = 0; i < n; ++i)
        for (int32_t layer = 0; layer < g->n_layers; ++layer)
            for (int32_t lb = 0; lb < mb; ++lb) {
                int32_t* e = block_table + ((int64_t)slots[i] * g->n_layers + layer) * mb + lb;
                if (*e == -1) continue;
                free_pages[top++] = *e; /* push_back */
                *e = -1;
            }
    *free_count = top;
    return held;
}

/* -------------------------------------------------------------- gather */

/* Element (token, kv head, dim) of K lives at
 * block*BLOCK_BYTES + token*KV_DIM*2 + kv_head*HEAD_DIM*2 + dim*2, and of V at
 * the same address + V_OFFSET; a block holds min(n - 16*lb, 16) valid tokens
 * [TV6 "논리 블록 → 물리 블록 → 바이트 주소"]. */
int orc_gather_kv(const orc_geom* g, const uint8_t* pool, const int32_t* block_table,
                  int32_t layer, int32_t slot, int32_t n, double* K, double* V) {
    if (!geom_ok(g) || n < 0 || !pool || !block_table || (n > 0 && (!K || !V)))
        return ORC_BAD_ARG;
    const int32_t hkv = g->num_kv_heads, d = g->head_dim;
    for (int32_t t = 0; t < n; ++t) {
        int64_t blk = block_of(g, block_table, slot, layer, t);
        if (blk < 0) return ORC_BAD_BLOCK;
        int64_t token_in_block = t % TOKENS_PER_BLOCK;
        for (int32_t h = 0; h < hkv; ++h) {
            for (int32_t k = 0; k < d; ++k) {
                int64_t addr = blk * block_bytes(g) + token_in_block * kv_dim(g) * 2 +
                               (int64_t)h * d * 2 + (int64_t)k * 2;
                uint16_t kb, vb;
                memcpy(&kb, pool + addr, 2);
                memcpy(&vb, pool + addr + v_offset(g), 2);
                K[((int64_t)t * hkv + h) * d + k] = bf16_to_double(kb);
                V[((int64_t)t * hkv + h) * d + k] = bf16_to_double(vb);
            }
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------- softmax */

/* Plain two-pass softmax of one row: m = max s, l = sum e^(s - m),
 * w = e^(s - m) / l.  Masked entries are -inf and get weight exactly 0. */
void orc_softmax_row(const double* s, int32_t n, double* w, double* m_out, double* l_out) {
    double m = -INFINITY;
    for (int32_t j = 0; j < n; ++j)
        if (s[j] > m) m = s[j];
    double l = 0.0;
    if (m == -INFINITY) {
        if (w)
            for (int32_t j = 0; j < n; ++j) w[j] = 0.0;
        *m_out = m;
        *l_out = 0.0;
        return;
    }
    for (int32_t j = 0; j < n; ++j) l += exp(s[j] - m);
    if (w)
        for (int32_t j = 0; j < n; ++j) w[j] = exp(s[j] - m) / l;
    *m_out = m;
    *l_out = l;
}

/* Un-normalised output and statistics of one key subset: keep O~ and l,
 * divide once at the end [FA2 "단계별 설명 (순전파의 두 가지 손질)"]. */
void orc_partial(const double* s, const double* v, int32_t n, int32_t dv, double* m,
                 double* l, double* acc) {
    orc_softmax_row(s, n, NULL, m, l);
    for (int32_t k = 0; k < dv; ++k) acc[k] = 0.0;
    if (*m == -INFINITY) return;
    for (int32_t j = 0; j < n; ++j) {
        double p = exp(s[j] - *m);
        for (int32_t k = 0; k < dv; ++k) acc[k] += p * v[(int64_t)j * dv + k];
    }
}

/* Merge rule m = max(m_a, m_b), d = d_a e^(m_a - m) + d_b e^(m_b - m)
 * [TV3 "causalMask and online softmax"], applied to every partial; the
 * accumulated outputs are rescaled the same way [FA2 worked example, block 2:
 * O~ = 0.368 * 23.68 + 30].  L = m + ln l [FA2 "단계별 설명"]. */
void orc_merge(int32_t nparts, const double* m, const double* l, const double* acc,
               int32_t dv, double* m_out, double* l_out, double* acc_out, double* o,
               double* lse) {
    double ms = -INFINITY;
    for (int32_t i = 0; i < nparts; ++i)
        if (m[i] > ms) ms = m[i];
    double ls = 0.0;
    for (int32_t k = 0; k < dv; ++k) acc_out[k] = 0.0;
    if (ms != -INFINITY) {
        for (int32_t i = 0; i < nparts; ++i) {
            if (m[i] == -INFINITY) continue; /* an empty part contributes nothing */
            double c = exp(m[i] - ms);
            ls += l[i] * c;
            for (int32_t k = 0; k < dv; ++k) acc_out[k] += acc[(int64_t)i * dv + k] * c;
        }
    }
    *m_out = ms;
    *l_out = ls;
    if (ls > 0.0) {
        for (int32_t k = 0; k < dv; ++k) o[k] = acc_out[k] / ls;
        *lse = ms + log(ls);
    } else {
        for (int32_t k = 0; k < dv; ++k) o[k] = 0.0;
        *lse = -INFINITY;
    }
}

/* ----------------------------------------------------------- attention */

/* One output row: query qv[d] against keys 0..nkeys-1 of kv head hk, with
 * keys j > last_key masked (causal).  s_buf has room for nkeys scores.
 * Q head h reads kv head h / (Hq/Hkv) [TV3 "Per-head attention scores and
 * GQA"; FA2 "4. MQA · GQA 지원"]. */
static void attend_row(const orc_geom* g, const double* qv, const double* K, const double* V,
                       int32_t hk, int32_t nkeys, int32_t last_key, double scale,
                       double* s_buf, double* o, double* lse) {
    const int32_t hkv = g->num_kv_heads, d = g->head_dim;
    for (int32_t j = 0; j < nkeys; ++j) {
        if (j > last_key) {
            s_buf[j] = -INFINITY; /* causal mask: column after the row */
            continue;
        }
        const double* kj = K + ((int64_t)j * hkv + hk) * d;
        double dot = 0.0;
        for (int32_t k = 0; k < d; ++k) dot += qv[k] * kj[k];
        s_buf[j] = scale * dot;
    }
    double m, l;
    orc_softmax_row(s_buf, nkeys, NULL, &m, &l);
    if (l == 0.0) {
        for (int32_t k = 0; k < d; ++k) o[k] = 0.0;
        *lse = -INFINITY;
        return;
    }
    for (int32_t k = 0; k < d; ++k) {
        double acc = 0.0;
        for (int32_t j = 0; j < nkeys; ++j) {
            if (s_buf[j] == -INFINITY) continue;
            acc += exp(s_buf[j] - m) * V[((int64_t)j * hkv + hk) * d + k];
        }
        o[k] = acc / l;
    }
    *lse = m + log(l);
}

/* ------------------------------------------------------ thread helpers */

int32_t orc_default_threads(void) {
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    return n > 0 ? (int32_t)n : 1;
}

typedef struct {
    void (*fn)(void* ctx, int64_t item, double* scratch);
    void* ctx;
    int64_t n_items;
    int64_t next; /* shared work counter */
    int64_t scratch_len;
} pool_job;

static void* pool_worker(void* arg) {
    pool_job* job = (pool_job*)arg;
    double* scratch = (double*)malloc(sizeof(double) * (size_t)(job->scratch_len + 1));
    if (!scratch) return NULL;
    for (;;) {
        int64_t item = __atomic_fetch_add(&job->next, 1, __ATOMIC_RELAXED);
        if (item >= job->n_items) break;
        job->fn(job->ctx, item, scratch);
    }
    free(scratch);
    return NULL;
}

/* Runs fn(ctx, item, scratch) for every item on nthreads threads. */
static void run_items(void (*fn)(void*, int64_t, double*), void* ctx, int64_t n_items,
                      int64_t scratch_len, int32_t nthreads) {
    if (nthreads <= 0) nthreads = orc_default_threads();
    if (nthreads > n_items) nthreads = (int32_t)(n_items > 0 ? n_items : 1);
    pool_job job = {fn, ctx, n_items, 0, scratch_len};
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
    int32_t started = 0;
    for (int32_t i = 1; i < nthreads && th; ++i)
        if (pthread_create(&th[started], NULL, pool_worker, &job) == 0) ++started;
    pool_worker(&job);
    for (int32_t i = 0; i < started; ++i) pthread_join(th[i], NULL);
    free(th);
}

/* ------------------------------------------------------------- prefill */

typedef struct {
    const orc_geom* g;
    const uint16_t* q;
    const int32_t* cu;
    const int32_t* prefix; /* cached tokens before each sequence's queries (NULL: none) */
    double scale;
    double** K; /* per sequence gathered keys (NULL when not needed) */
    double** V;
    int32_t batch;
    /* full prefill */
    double* o;
    double* lse;
    /* sampled rows */
    const int64_t* rows;
    const int32_t* heads;
} prefill_ctx;

static int32_t seq_of_row(const int32_t* cu, int32_t batch, int64_t row) {
    for (int32_t b = 0; b < batch; ++b)
        if (row >= cu[b] && row < cu[b + 1]) return b;
    return -1;
}

/* One (packed row, q head) output.  The i-th query of sequence b sits at
 * position prefix[b] + i of its sequence, after the prefix[b] cached tokens,
 * and attends keys 0..prefix[b] + i: the causal rule of a fresh prompt, with
 * the cache read up to and including the query's own token, whose K/V were
 * written first [TV6 "논리 블록 → 물리 블록 → 바이트 주소"; TV3 "causalMask
 * and online softmax"].  Without a prefix this is the fresh-prompt prefill. */
static void prefill_one(const prefill_ctx* c, int64_t row, int32_t hq, double* scratch,
                        double* o, double* lse) {
    const orc_geom* g = c->g;
    const int32_t d = g->head_dim, hq_n = g->num_q_heads;
    const int32_t group = g->num_q_heads / g->num_kv_heads;
    int32_t b = seq_of_row(c->cu, c->batch, row);
    int32_t pre = c->prefix ? c->prefix[b] : 0;
    int32_t n = c->cu[b + 1] - c->cu[b];
    int32_t i = (int32_t)(row - c->cu[b]); /* index of this query among its sequence's queries */
    double* qv = scratch;                  /* d doubles, then pre + n scores */
    for (int32_t k = 0; k < d; ++k) qv[k] = bf16_to_double(c->q[(row * hq_n + hq) * d + k]);
    attend_row(g, qv, c->K[b], c->V[b], hq / group, pre + n, pre + i, c->scale, scratch + d, o, lse);
}

static void prefill_item(void* ctx, int64_t item, double* scratch) {
    const prefill_ctx* c = (const prefill_ctx*)ctx;
    const int32_t hq_n = c->g->num_q_heads, d = c->g->head_dim;
    int64_t row = item / hq_n;
    int32_t hq = (int32_t)(item % hq_n);
    prefill_one(c, row, hq, scratch, c->o + (row * hq_n + hq) * d, c->lse + row * hq_n + hq);
}

static void prefill_rows_item(void* ctx, int64_t item, double* scratch) {
    const prefill_ctx* c = (const prefill_ctx*)ctx;
    const int32_t d = c->g->head_dim;
    prefill_one(c, c->rows[item], c->heads[item], scratch, c->o + item * d, c->lse + item);
}

static int check_batch(const orc_geom* g, int32_t batch, const int32_t* cu, const int32_t* slots,
                       int32_t layer) {
    if (!geom_ok(g) || batch < 0 || !cu || !slots) return 0;
    if (layer < 0 || layer >= g->n_layers) return 0;
    if (cu[0] != 0) return 0;
    for (int32_t b = 0; b < batch; ++b)
        if (cu[b + 1] < cu[b]) return 0;
    return 1;
}

/* Gathers the sequences flagged in `need` (all when need == NULL). */
static int gather_all(const orc_geom* g, const uint8_t* pool, const int32_t* bt, int32_t layer,
                      int32_t batch, const int32_t* lens, const int32_t* slots,
                      const char* need, double** K, double** V) {
    const int64_t row = kv_dim(g);
    for (int32_t b = 0; b < batch; ++b) {
        K[b] = V[b] = NULL;
        if (need && !need[b]) continue;
        int64_t n = lens[b];
        K[b] = (double*)malloc(sizeof(double) * (size_t)(n * row + 1));
        V[b] = (double*)malloc(sizeof(double) * (size_t)(n * row + 1));
        if (!K[b] || !V[b]) return ORC_BAD_ARG;
        int st = orc_gather_kv(g, pool, bt, layer, slots[b], (int32_t)n, K[b], V[b]);
        if (st != ORC_OK) return st;
    }
    return ORC_OK;
}

static void free_all(int32_t batch, double** K, double** V) {
    for (int32_t b = 0; b < batch; ++b) {
        free(K[b]);
        free(V[b]);
    }
    free(K);
    free(V);
}

static int prefill_common(const orc_geom* g, const uint16_t* q, const uint8_t* pool,
                          const int32_t* bt, int32_t layer, int32_t batch, const int32_t* cu,
                          const int32_t* prefix, const int32_t* slots, float scale, int64_t nsamp,
                          const int64_t* rows, const int32_t* heads, double* o, double* lse,
                          int32_t nthreads) {
    if (!check_batch(g, batch, cu, slots, layer) || !pool || !bt || !o || !lse) return ORC_BAD_ARG;
    const int64_t T = cu[batch];
    if (T > 0 && !q) return ORC_BAD_ARG;
    int32_t* lens = (int32_t*)malloc(sizeof(int32_t) * (size_t)(batch + 1));
    char* need = (char*)calloc((size_t)batch + 1, 1);
    double** K = (double**)calloc((size_t)batch + 1, sizeof(double*));
    double** V = (double**)calloc((size_t)batch + 1, sizeof(double*));
    if (!lens || !need || !K || !V) {
        free(lens); free(need); free(K); free(V);
        return ORC_BAD_ARG;
    }
    int32_t nmax = 0;
    int st = ORC_OK;
    for (int32_t b = 0; b < batch; ++b) {
        /* keys of sequence b: its cached prefix, then its queries' own tokens */
        const int64_t nk = (int64_t)(prefix ? prefix[b] : 0) + (cu[b + 1] - cu[b]);
        if ((prefix && prefix[b] < 0) || nk > 0x7FFFFFFF) st = ORC_BAD_ARG;
        lens[b] = (int32_t)(nk > 0x7FFFFFFF ? 0 : nk);
        if (lens[b] > nmax) nmax = lens[b];
    }
    if (rows) {
        for (int64_t s = 0; s < nsamp; ++s) {
            int32_t b = (rows[s] >= 0 && rows[s] < T) ? seq_of_row(cu, batch, rows[s]) : -1;
            if (b < 0 || heads[s] < 0 || heads[s] >= g->num_q_heads) st = ORC_BAD_ARG;
            else need[b] = 1;
        }
    }
    if (st == ORC_OK) st = gather_all(g, pool, bt, layer, batch, lens, slots, rows ? need : NULL, K, V);
    if (st == ORC_OK) {
        prefill_ctx c = {g, q, cu, prefix, (double)scale, K, V, batch, o, lse, rows, heads};
        if (rows)
            run_items(prefill_rows_item, &c, nsamp, (int64_t)g->head_dim + nmax, nthreads);
        else
            run_items(prefill_item, &c, T * g->num_q_heads, (int64_t)g->head_dim + nmax, nthreads);
    }
    free_all(batch, K, V);
    free(lens);
    free(need);
    return st;
}

int orc_prefill(const orc_geom* g, const uint16_t* q, const uint8_t* pool,
                const int32_t* block_table, int32_t layer, int32_t batch,
                const int32_t* cu_seqlens, const int32_t* slots, float scale, double* o,
                double* lse, int32_t nthreads) {
    return prefill_common(g, q, pool, block_table, layer, batch, cu_seqlens, NULL, slots, scale, 0,
                          NULL, NULL, o, lse, nthreads);
}

int orc_prefill_cached(const orc_geom* g, const uint16_t* q, const uint8_t* pool,
                       const int32_t* block_table, int32_t layer, int32_t batch,
                       const int32_t* cu_seqlens, const int32_t* prefix_lens, const int32_t* slots,
                       float scale, double* o, double* lse, int32_t nthreads) {
    return prefill_common(g, q, pool, block_table, layer, batch, cu_seqlens, prefix_lens, slots, scale,
                          0, NULL, NULL, o, lse, nthreads);
}

int orc_prefill_rows(const orc_geom* g, const uint16_t* q, const uint8_t* pool,
                     const int32_t* block_table, int32_t layer, int32_t batch,
                     const int32_t* cu_seqlens, const int32_t* slots, float scale,
                     int64_t nsamp, const int64_t* rows, const int32_t* heads, double* o,
                     double* lse, int32_t nthreads) {
    if (nsamp < 0 || (nsamp > 0 && (!rows || !heads))) return ORC_BAD_ARG;
    static const int64_t no_rows = 0;
    return prefill_common(g, q, pool, block_table, layer, batch, cu_seqlens, NULL, slots, scale,
                          nsamp, rows ? rows : &no_rows, heads, o, lse, nthreads);
}

int orc_prefill_cached_rows(const orc_geom* g, const uint16_t* q, const uint8_t* pool,
                            const int32_t* block_table, int32_t layer, int32_t batch,
                            const int32_t* cu_seqlens, const int32_t* prefix_lens,
                            const int32_t* slots, float scale, int64_t nsamp, const int64_t* rows,
                            const int32_t* heads, double* o, double* lse, int32_t nthreads) {
    if (nsamp < 0 || (nsamp > 0 && (!rows || !heads))) return ORC_BAD_ARG;
    static const int64_t no_rows = 0;
    return prefill_common(g, q, pool, block_table, layer, batch, cu_seqlens, prefix_lens, slots, scale,
                          nsamp, rows ? rows : &no_rows, heads, o, lse, nthreads);
}

/* ------------------------------------------------------------ backward */

typedef struct {
    const orc_geom* g;
    const uint16_t* q;
    const uint16_t* dout;
    const int32_t* cu;
    double scale;
    double** K;
    double** V;
    double* dq;
    double* dk;
    double* dv;
    int32_t batch;
} backward_ctx;

/* One query row i of sequence b, q head h: the scores s_j = scale q_i . k_j
 * (j <= i), m = max_j s_j, l = sum_j e^(s_j - m), p_j = e^(s_j - m) / l,
 * dp_j = do_i . v_j, D = sum_j p_j dp_j and ds_j = p_j (dp_j - D), with p
 * recomputed from the scores as the FA2 backward recomputes it from the stored
 * L [FA2, 전체 흐름: "L로 P 재계산"].  Fills qv, dov (the row's q and do),
 * p[0..i], ds[0..i]; returns m, l, D; dq_i = scale sum_j ds_j k_j into dqi
 * when it is not NULL. */
static void backward_row(const backward_ctx* c, int32_t b, int32_t h, int32_t i, double* qv,
                         double* dov, double* p, double* ds, double* m_out, double* l_out,
                         double* D_out, double* dqi) {
    const orc_geom* g = c->g;
    const int32_t hq_n = g->num_q_heads, hkv = g->num_kv_heads, d = g->head_dim;
    const int32_t hk = h / (hq_n / hkv);
    const int64_t row = c->cu[b] + i;
    const double* K = c->K[b];
    const double* V = c->V[b];
    for (int32_t k = 0; k < d; ++k) {
        qv[k] = bf16_to_double(c->q[(row * hq_n + h) * d + k]);
        dov[k] = bf16_to_double(c->dout[(row * hq_n + h) * d + k]);
    }
    double m = -INFINITY;
    for (int32_t j = 0; j <= i; ++j) {
        const double* kj = K + ((int64_t)j * hkv + hk) * d;
        double dot = 0.0;
        for (int32_t k = 0; k < d; ++k) dot += qv[k] * kj[k];
        p[j] = c->scale * dot;
        if (p[j] > m) m = p[j];
    }
    double l = 0.0;
    for (int32_t j = 0; j <= i; ++j) l += exp(p[j] - m);
    double D = 0.0;
    for (int32_t j = 0; j <= i; ++j) {
        p[j] = exp(p[j] - m) / l;
        const double* vj = V + ((int64_t)j * hkv + hk) * d;
        double dp = 0.0;
        for (int32_t k = 0; k < d; ++k) dp += dov[k] * vj[k];
        ds[j] = dp;
        D += p[j] * dp;
    }
    for (int32_t j = 0; j <= i; ++j) ds[j] = p[j] * (ds[j] - D);
    if (dqi) {
        for (int32_t k = 0; k < d; ++k) dqi[k] = 0.0;
        for (int32_t j = 0; j <= i; ++j) {
            const double* kj = K + ((int64_t)j * hkv + hk) * d;
            for (int32_t k = 0; k < d; ++k) dqi[k] += c->scale * ds[j] * kj[k];
        }
    }
    *m_out = m;
    *l_out = l;
    *D_out = D;
}

/* Gradients of the causal prefill of sequence b for the q heads of kv head hk
 * (one work item: it alone writes these dQ rows and these dK / dV rows).  The
 * definition, by the chain rule through o_i = sum_j p_ij v_j and the softmax
 * p_ij = e^(s_ij) / sum_k e^(s_ik), s_ij = scale q_i . k_j, j <= i:
 *   dv_j += sum_i p_ij do_i          dp_ij = do_i . v_j
 *   D_i   = sum_j p_ij dp_ij         ds_ij = p_ij (dp_ij - D_i)
 *   dq_i  = scale sum_j ds_ij k_j    dk_j += scale sum_i ds_ij q_i
 * with dk, dv summed over the q heads that read kv head hk [FA2 "4. MQA · GQA
 * 지원": the gradients of the implicitly repeated heads are added]. */
static void backward_item(void* ctx, int64_t item, double* scratch) {
    const backward_ctx* c = (const backward_ctx*)ctx;
    const orc_geom* g = c->g;
    const int32_t hq_n = g->num_q_heads, hkv = g->num_kv_heads, d = g->head_dim;
    const int32_t group = hq_n / hkv;
    const int32_t b = (int32_t)(item / hkv), hk = (int32_t)(item % hkv);
    const int64_t r0 = c->cu[b];
    const int32_t n = c->cu[b + 1] - c->cu[b];
    double* qv = scratch;        /* d */
    double* dov = qv + d;        /* d */
    double* p = dov + d;         /* n */
    double* ds = p + n;          /* n */
    for (int32_t r = 0; r < group; ++r) {
        const int32_t h = hk * group + r;
        for (int32_t i = 0; i < n; ++i) {
            double m, l, D;
            backward_row(c, b, h, i, qv, dov, p, ds, &m, &l, &D, c->dq + ((r0 + i) * hq_n + h) * d);
            for (int32_t j = 0; j <= i; ++j) {
                double* dkj = c->dk + ((r0 + j) * hkv + hk) * d;
                double* dvj = c->dv + ((r0 + j) * hkv + hk) * d;
                for (int32_t k = 0; k < d; ++k) {
                    dkj[k] += c->scale * ds[j] * qv[k];
                    dvj[k] += p[j] * dov[k];
                }
            }
        }
    }
}

int orc_prefill_backward(const orc_geom* g, const uint16_t* q, const uint8_t* pool,
                         const int32_t* block_table, int32_t layer, int32_t batch,
                         const int32_t* cu_seqlens, const int32_t* slots, float scale,
                         const uint16_t* dout, double* dq, double* dk, double* dv, int32_t nthreads) {
    if (!check_batch(g, batch, cu_seqlens, slots, layer) || !pool || !block_table || !dq || !dk || !dv)
        return ORC_BAD_ARG;
    const int64_t T = cu_seqlens[batch];
    if (T > 0 && (!q || !dout)) return ORC_BAD_ARG;
    int32_t* lens = (int32_t*)malloc(sizeof(int32_t) * (size_t)(batch + 1));
    double** K = (double**)calloc((size_t)batch + 1, sizeof(double*));
    double** V = (double**)calloc((size_t)batch + 1, sizeof(double*));
    if (!lens || !K || !V) {
        free(lens); free(K); free(V);
        return ORC_BAD_ARG;
    }
    int32_t nmax = 0;
    for (int32_t b = 0; b < batch; ++b) {
        lens[b] = cu_seqlens[b + 1] - cu_seqlens[b];
        if (lens[b] > nmax) nmax = lens[b];
    }
    const int64_t kv = kv_dim(g);
    for (int64_t x = 0; x < T * g->num_q_heads * g->head_dim; ++x) dq[x] = 0.0;
    for (int64_t x = 0; x < T * kv; ++x) dk[x] = dv[x] = 0.0;
    int st = gather_all(g, pool, block_table, layer, batch, lens, slots, NULL, K, V);
    if (st == ORC_OK) {
        backward_ctx c = {g, q, dout, cu_seqlens, (double)scale, K, V, dq, dk, dv, batch};
        run_items(backward_item, &c, (int64_t)batch * g->num_kv_heads, 2 * (int64_t)g->head_dim + 2 * nmax,
                  nthreads);
    }
    free_all(batch, K, V);
    free(lens);
    return st;
}

/* ------------------------------------------------ backward at sampled rows */

typedef struct {
    backward_ctx base;
    int32_t n_pairs;            /* (sequence, q head) pairs whose row statistics are needed */
    const int32_t* pair_b;
    const int32_t* pair_h;
    const int64_t* pair_first;  /* first stats item of each pair; [n_pairs + 1] */
    double** stats;             /* per pair: m, l, D of every row, [3 n] */
    int64_t n_q;
    const int64_t* q_rows;
    const int32_t* q_heads;
    double* dq;                 /* [n_q][d] */
    const int64_t* k_rows;
    const int32_t* k_heads;
    const int32_t* k_pair0;     /* stats pair of (sequence of k row, first q head of its group) */
    double* dk;                 /* [n_k][d] */
    double* dv;
} backward_rows_ctx;

static void backward_stats_item(void* ctx, int64_t item, double* scratch) {
    const backward_rows_ctx* c = (const backward_rows_ctx*)ctx;
    int32_t k = 0;
    while (item >= c->pair_first[k + 1]) ++k;
    const int32_t i = (int32_t)(item - c->pair_first[k]);
    const int32_t d = c->base.g->head_dim;
    const int32_t n = c->base.cu[c->pair_b[k] + 1] - c->base.cu[c->pair_b[k]];
    double* st = c->stats[k] + 3 * (int64_t)i;
    backward_row(&c->base, c->pair_b[k], c->pair_h[k], i, scratch, scratch + d, scratch + 2 * d,
                 scratch + 2 * d + n, &st[0], &st[1], &st[2], NULL);
}

/* Sample s < n_q: dq of (row, q head), the row computation of
 * orc_prefill_backward.  Sample n_q + t: dk, dv of key row k_rows[t], kv head
 * k_heads[t]: the terms of orc_prefill_backward's sums that land on that key,
 * in its order (q heads of the group, then query rows i >= j), each p_ij and
 * ds_ij rebuilt from row i's m, l and D as that row computes them. */
static void backward_sample_item(void* ctx, int64_t item, double* scratch) {
    const backward_rows_ctx* c = (const backward_rows_ctx*)ctx;
    const backward_ctx* bc = &c->base;
    const orc_geom* g = bc->g;
    const int32_t hq_n = g->num_q_heads, hkv = g->num_kv_heads, d = g->head_dim;
    const int32_t group = hq_n / hkv;
    if (item < c->n_q) {
        const int64_t row = c->q_rows[item];
        const int32_t b = seq_of_row(bc->cu, bc->batch, row);
        const int32_t n = bc->cu[b + 1] - bc->cu[b];
        double m, l, D;
        backward_row(bc, b, c->q_heads[item], (int32_t)(row - bc->cu[b]), scratch, scratch + d,
                     scratch + 2 * d, scratch + 2 * d + n, &m, &l, &D, c->dq + item * d);
        return;
    }
    const int64_t t = item - c->n_q;
    const int64_t row = c->k_rows[t];
    const int32_t hk = c->k_heads[t];
    const int32_t b = seq_of_row(bc->cu, bc->batch, row);
    const int64_t r0 = bc->cu[b];
    const int32_t n = bc->cu[b + 1] - bc->cu[b];
    const int32_t j = (int32_t)(row - r0);
    const double* kj = bc->K[b] + ((int64_t)j * hkv + hk) * d;
    const double* vj = bc->V[b] + ((int64_t)j * hkv + hk) * d;
    double* dkj = c->dk + t * d;
    double* dvj = c->dv + t * d;
    double* qv = scratch;
    double* dov = scratch + d;
    for (int32_t k = 0; k < d; ++k) dkj[k] = dvj[k] = 0.0;
    for (int32_t r = 0; r < group; ++r) {
        const int32_t h = hk * group + r;
        const double* st = c->stats[c->k_pair0[t] + r];
        for (int32_t i = j; i < n; ++i) {
            const int64_t qrow = r0 + i;
            for (int32_t k = 0; k < d; ++k) {
                qv[k] = bf16_to_double(bc->q[(qrow * hq_n + h) * d + k]);
                dov[k] = bf16_to_double(bc->dout[(qrow * hq_n + h) * d + k]);
            }
            double dot = 0.0;
            for (int32_t k = 0; k < d; ++k) dot += qv[k] * kj[k];
            const double pij = exp(bc->scale * dot - st[3 * i]) / st[3 * i + 1];
            double dp = 0.0;
            for (int32_t k = 0; k < d; ++k) dp += dov[k] * vj[k];
            const double dsij = pij * (dp - st[3 * i + 2]);
            for (int32_t k = 0; k < d; ++k) {
                dkj[k] += bc->scale * dsij * qv[k];
                dvj[k] += pij * dov[k];
            }
        }
    }
}

int orc_prefill_backward_rows(const orc_geom* g, const uint16_t* q, const uint8_t* pool,
                              const int32_t* block_table, int32_t layer, int32_t batch,
                              const int32_t* cu_seqlens, const int32_t* slots, float scale,
                              const uint16_t* dout, int64_t n_q, const int64_t* q_rows,
                              const int32_t* q_heads, double* dq, int64_t n_k, const int64_t* k_rows,
                              const int32_t* k_heads, double* dk, double* dv, int32_t nthreads) {
    if (!check_batch(g, batch, cu_seqlens, slots, layer) || !pool || !block_table || n_q < 0 || n_k < 0)
        return ORC_BAD_ARG;
    if ((n_q > 0 && (!q_rows || !q_heads || !dq)) || (n_k > 0 && (!k_rows || !k_heads || !dk || !dv)))
        return ORC_BAD_ARG;
    const int64_t T = cu_seqlens[batch];
    if (T > 0 && (!q || !dout)) return ORC_BAD_ARG;
    const int32_t hq_n = g->num_q_heads, hkv = g->num_kv_heads, group = hq_n / hkv;
    int st = ORC_OK;
    int32_t* lens = (int32_t*)malloc(sizeof(int32_t) * (size_t)(batch + 1));
    char* need = (char*)calloc((size_t)batch + 1, 1);
    int32_t* pair_of = (int32_t*)malloc(sizeof(int32_t) * (size_t)((int64_t)batch * hq_n + 1));
    int32_t* pair_b = (int32_t*)malloc(sizeof(int32_t) * (size_t)((int64_t)batch * hq_n + 1));
    int32_t* pair_h = (int32_t*)malloc(sizeof(int32_t) * (size_t)((int64_t)batch * hq_n + 1));
    int64_t* pair_first = (int64_t*)malloc(sizeof(int64_t) * (size_t)((int64_t)batch * hq_n + 2));
    int32_t* k_pair0 = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n_k + 1));
    double** stats = (double**)calloc((size_t)((int64_t)batch * hq_n + 1), sizeof(double*));
    double** K = (double**)calloc((size_t)batch + 1, sizeof(double*));
    double** V = (double**)calloc((size_t)batch + 1, sizeof(double*));
    if (!lens || !need || !pair_of || !pair_b || !pair_h || !pair_first || !k_pair0 || !stats || !K || !V) {
        st = ORC_BAD_ARG;
        goto done;
    }
    int32_t nmax = 0;
    for (int32_t b = 0; b < batch; ++b) {
        lens[b] = cu_seqlens[b + 1] - cu_seqlens[b];
        if (lens[b] > nmax) nmax = lens[b];
    }
    for (int64_t x = 0; x < (int64_t)batch * hq_n; ++x) pair_of[x] = -1;
    for (int64_t s = 0; s < n_q; ++s) {
        const int32_t b = (q_rows[s] >= 0 && q_rows[s] < T) ? seq_of_row(cu_seqlens, batch, q_rows[s]) : -1;
        if (b < 0 || q_heads[s] < 0 || q_heads[s] >= hq_n) st = ORC_BAD_ARG;
        else need[b] = 1;
    }
    int32_t n_pairs = 0;
    for (int64_t t = 0; t < n_k && st == ORC_OK; ++t) {
        const int32_t b = (k_rows[t] >= 0 && k_rows[t] < T) ? seq_of_row(cu_seqlens, batch, k_rows[t]) : -1;
        if (b < 0 || k_heads[t] < 0 || k_heads[t] >= hkv) {
            st = ORC_BAD_ARG;
            break;
        }
        need[b] = 1;
        /* the group's q heads get consecutive pair numbers */
        const int64_t key = (int64_t)b * hq_n + (int64_t)k_heads[t] * group;
        if (pair_of[key] < 0) {
            for (int32_t r = 0; r < group; ++r) {
                pair_of[key + r] = n_pairs;
                pair_b[n_pairs] = b;
                pair_h[n_pairs] = k_heads[t] * group + r;
                ++n_pairs;
            }
        }
        k_pair0[t] = pair_of[key];
    }
    if (st == ORC_OK) st = gather_all(g, pool, block_table, layer, batch, lens, slots, need, K, V);
    if (st == ORC_OK) {
        pair_first[0] = 0;
        for (int32_t k = 0; k < n_pairs; ++k) {
            const int32_t n = lens[pair_b[k]];
            pair_first[k + 1] = pair_first[k] + n;
            stats[k] = (double*)malloc(sizeof(double) * (size_t)(3 * (int64_t)n + 1));
            if (!stats[k]) st = ORC_BAD_ARG;
        }
    }
    if (st == ORC_OK) {
        backward_rows_ctx c;
        memset(&c, 0, sizeof(c));
        c.base.g = g;
        c.base.q = q;
        c.base.dout = dout;
        c.base.cu = cu_seqlens;
        c.base.scale = (double)scale;
        c.base.K = K;
        c.base.V = V;
        c.base.batch = batch;
        c.n_pairs = n_pairs;
        c.pair_b = pair_b;
        c.pair_h = pair_h;
        c.pair_first = pair_first;
        c.stats = stats;
        c.n_q = n_q;
        c.q_rows = q_rows;
        c.q_heads = q_heads;
        c.dq = dq;
        c.k_rows = k_rows;
        c.k_heads = k_heads;
        c.k_pair0 = k_pair0;
        c.dk = dk;
        c.dv = dv;
        const int64_t scratch = 2 * (int64_t)g->head_dim + 2 * (int64_t)nmax;
        if (n_pairs > 0) run_items(backward_stats_item, &c, pair_first[n_pairs], scratch, nthreads);
        run_items(backward_sample_item, &c, n_q + n_k, scratch, nthreads);
    }
done:
    if (stats)
        for (int64_t k = 0; k < (int64_t)batch * hq_n; ++k) free(stats[k]);
    free(stats);
    if (K && V) free_all(batch, K, V);
    else {
        free(K);
        free(V);
    }
    free(lens);
    free(need);
    free(pair_of);
    free(pair_b);
    free(pair_h);
    free(pair_first);
    free(k_pair0);
    return st;
}

/* -------------------------------------------------------------- decode */

typedef struct {
    const orc_geom* g;
    const uint16_t* q;
    const uint8_t* pool;
    const int32_t* bt;
    int32_t layer;
    const int32_t* lens;
    const int32_t* slots;
    double scale;
    double* o;
    double* lse;
    int status; /* first error seen (written under the atomic below) */
} decode_ctx;

/* Query b sits at position seq_len - 1 and sees keys 0..seq_len-1: the length
 * already counts the token just written, so nothing in the future is read
 * [TV6 "논리 블록 → 물리 블록 → 바이트 주소"]. */
static void decode_item(void* ctx, int64_t b, double* scratch) {
    decode_ctx* c = (decode_ctx*)ctx;
    const orc_geom* g = c->g;
    const int32_t d = g->head_dim, hq_n = g->num_q_heads, hkv = g->num_kv_heads;
    const int32_t group = hq_n / hkv;
    const int32_t n = c->lens[b];
    double* out = c->o + b * hq_n * d;
    double* lse = c->lse + b * hq_n;
    if (n <= 0) {
        for (int32_t k = 0; k < hq_n * d; ++k) out[k] = 0.0;
        for (int32_t h = 0; h < hq_n; ++h) lse[h] = -INFINITY;
        return;
    }
    double* K = (double*)malloc(sizeof(double) * (size_t)n * (size_t)kv_dim(g));
    double* V = (double*)malloc(sizeof(double) * (size_t)n * (size_t)kv_dim(g));
    int st = (K && V) ? orc_gather_kv(g, c->pool, c->bt, c->layer, c->slots[b], n, K, V)
                      : ORC_BAD_ARG;
    if (st != ORC_OK) {
        int expected = ORC_OK;
        __atomic_compare_exchange_n(&c->status, &expected, st, 0, __ATOMIC_RELAXED,
                                    __ATOMIC_RELAXED);
    } else {
        double* qv = scratch;
        for (int32_t h = 0; h < hq_n; ++h) {
            for (int32_t k = 0; k < d; ++k)
                qv[k] = bf16_to_double(c->q[((int64_t)b * hq_n + h) * d + k]);
            attend_row(g, qv, K, V, h / group, n, n - 1, c->scale, scratch + d, out + h * d,
                       lse + h);
        }
    }
    free(K);
    free(V);
}

int orc_decode(const orc_geom* g, const uint16_t* q, const uint8_t* pool,
               const int32_t* block_table, int32_t layer, int32_t batch,
               const int32_t* seq_lens, const int32_t* slots, float scale, double* o,
               double* lse, int32_t nthreads) {
    if (!geom_ok(g) || batch < 0 || layer < 0 || layer >= g->n_layers) return ORC_BAD_ARG;
    if (batch == 0) return ORC_OK;
    if (!q || !pool || !block_table || !seq_lens || !slots || !o || !lse) return ORC_BAD_ARG;
    int32_t nmax = 0;
    for (int32_t b = 0; b < batch; ++b)
        if (seq_lens[b] > nmax) nmax = seq_lens[b];
    decode_ctx c = {g, q, pool, block_table, layer, seq_lens, slots, (double)scale, o, lse, ORC_OK};
    run_items(decode_item, &c, batch, (int64_t)g->head_dim + nmax, nthreads);
    return c.status;
}

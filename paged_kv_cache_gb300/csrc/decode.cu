// decode.cu -- single-query attention over a paged KV cache, split across CTAs.
//
// What is computed (jaehun.me tiny-vllm part 6, "논리 블록 → 물리 블록 → 바이트
// 주소" and "online softmax: 블록을 훑으며 가중 평균"): query b attends the first
// seq_lens[b] tokens of its slot; logical page lp lives in physical page
// block_table[slot][layer][lp]; the last page holds min(n - 16 lp, 16) tokens.
// Partial results over disjoint key ranges are merged by
//   m = max(m_a, m_b),  l = l_a e^(m_a - m) + l_b e^(m_b - m)
// (part 3, "causalMask and online softmax"), applied to the outputs as well.
//
// GB300 design (the series' kernel is one 64-thread CTA per (slot, q head)
// walking tokens with two __syncthreads each; that is prior art only):
//  * Work split.  All pages of all sequences form one flat list of T pages;
//    CTA c of G takes pages [c T / G, (c+1) T / G).  Every CTA gets the same
//    number of pages (+-1) whatever the length mix, and a CTA's range may
//    cover the tail of one sequence, whole sequences and the head of another.
//    Each (sequence, CTA) piece is a unit: a unit that is the whole sequence
//    writes o / lse directly; otherwise it writes a normalised partial
//    (o_i, L_i) to slot b + c of the workspace (unique, because the pieces
//    form a monotone staircase in (b, c)), and a second kernel merges them.
//    The split depends only on the lengths and G, never on page ids.
//  * Memory pipeline.  Warp 0 is the producer: it walks the CTA's pages,
//    prefetches 32 block-table entries per warp load, and streams each whole
//    page (K half and V half, contiguous: 32 KiB for 8 x 64) into a shared-
//    memory stage with one cp.async.bulk (two for a partial last page, which
//    copies only its valid rows), plus the sequence's query row at the start
//    of a unit.  Several stages stay in flight per SM, so HBM sees long
//    sequential reads with enough bytes outstanding to cover its latency.
//  * Compute.  One consumer warp per KV head (two when the GQA group is 8)
//    packs the group's query heads: each lane owns 16 dims of one token row,
//    so a warp covers 8 (d 64) or 4 (d 128) tokens per pass; dot products
//    reduce over 4 or 8 lanes with xor-shuffles; each token subgroup keeps its
//    own online-softmax state (m, l, acc) in registers and the subgroups merge
//    once per unit.  The running max is only moved when a score exceeds it by
//    more than 2^8 (exact: o and l share the same reference m).
#include <math_constants.h>

#include <mutex>

#include "pa_internal.cuh"

namespace pa {
namespace {

constexpr int kMaxConsumerWarps = 8;
constexpr int kMaxGrid = 1024;
constexpr int kSmemBudget = 200 * 1024;
constexpr int kMaxStages = 8;
constexpr int kCtlBytes = 1024;  // barriers + control words before the stages

enum : int { kFirst = 1, kLast = 2, kWhole = 4, kSkip = 8 };

struct StageHeader {
    int b;         // sequence of the page
    int ntok;      // tokens present in the stage (0 when the page is skipped)
    int flags;     // kFirst / kLast / kWhole / kSkip
    int slot_idx;  // workspace slot of a partial unit (b + cta)
};

struct DecodeParams {
    KGeom g;
    const uint8_t* q;     // bf16 [batch][hq][d]
    const uint8_t* pool;  // pages
    const int32_t* bt;
    int layer;
    int batch;
    const int32_t* seq_lens;
    const int32_t* slots;
    float scale_log2;     // scale * log2(e): scores kept in the base-2 domain
    __nv_bfloat16* o;
    float* lse;
    uint8_t* ws;
    long long ws_meta;    // int2 [batch]: first and last CTA of each sequence
    long long ws_lse;     // float [nslots][hq]: partial L (natural log)
    long long ws_o;       // float [nslots][hq][d]: partial normalised outputs
    int32_t* err;
    int attend_grid;      // CTAs of the attend kernel (G)
    int nst;              // pipeline stages
    int stage_bytes;      // page + q row + header, 128-byte multiple
    int q_bytes;          // hq * d * 2
    int wph;              // consumer warps per kv head
};

__host__ __device__ inline long long align_up(long long x, long long a) { return (x + a - 1) / a * a; }

struct WsLayout {
    long long meta, lse, o, total;
};

__host__ __device__ inline WsLayout ws_layout(int batch, long long nslots, int hq, int d) {
    WsLayout w;
    w.meta = 256;  // [0, 256): header, total page count at offset 0
    w.lse = align_up(w.meta + 8ll * batch, 256);
    w.o = align_up(w.lse + 4ll * nslots * hq, 256);
    w.total = align_up(w.o + 4ll * nslots * hq * d, 256);
    return w;
}

inline long long grid_cap(int batch, int max_seq_len) {
    long long upper = static_cast<long long>(batch) * ((max_seq_len + kBlockTokens - 1) / kBlockTokens);
    if (upper < 1) upper = 1;
    return upper < kMaxGrid ? upper : kMaxGrid;
}

__device__ __forceinline__ int pages_of(int len) { return len > 0 ? (len + kBlockTokens - 1) / kBlockTokens : 0; }

// First page of CTA c when T pages are split over G CTAs.
__device__ __forceinline__ long long range_start(long long c, long long T, long long G) { return c * T / G; }

// CTA owning flat page p.
__device__ __forceinline__ long long owner_of(long long p, long long T, long long G) {
    return ((p + 1) * G - 1) / T;
}

// Block-wide sum of one value per thread (all threads must call).
__device__ long long block_sum(long long v, long long* red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    if (lane == 0) red[warp] = v;
    __syncthreads();
    long long t = 0;
    for (int i = 0; i < nw; ++i) t += red[i];
    __syncthreads();
    return t;
}

// Block-wide inclusive scan of one value per thread; returns the inclusive
// prefix and the block total (all threads must call).
__device__ long long block_scan(long long v, long long* red, long long* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        long long u = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += u;
    }
    if (lane == 31) red[warp] = v;
    __syncthreads();
    long long before = 0, t = 0;
    for (int i = 0; i < nw; ++i) {
        if (i < warp) before += red[i];
        t += red[i];
    }
    __syncthreads();
    *total = t;
    return v + before;
}

template <int D, int GW>
__global__ void __launch_bounds__(32 * (1 + kMaxConsumerWarps), 1)
decode_attend_kernel(const DecodeParams p) {
    constexpr int LPT = D / 16;        // lanes per token row (16 dims each)
    constexpr int TPP = 32 / LPT;      // tokens per warp pass
    constexpr int PASSES = kBlockTokens / TPP;

    extern __shared__ __align__(1024) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + kMaxStages;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 256);
    long long* ctl = reinterpret_cast<long long*>(smem + 512);  // scan scratch and results
    long long* red = ctl + 8;                                   // per-warp partials
    uint8_t* stages = smem + kCtlBytes;

    const KGeom& g = p.g;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n_consumers = (blockDim.x >> 5) - 1;
    const long long G = gridDim.x, c = blockIdx.x;

    if (tid == 0) {
        for (int s = 0; s < p.nst; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], n_consumers);
        }
        *abort_flag = 0;
        mbar_init_fence();
    }

    // ---- this CTA's page range: total pages, then the sequence holding p_begin
    long long local = 0;
    for (int i = tid; i < p.batch; i += blockDim.x) {
        int len = p.seq_lens[i];
        if (len < 0) set_error(p.err, PA_ERR_BAD_BLOCK);
        local += pages_of(len);
    }
    const long long T = block_sum(local, red);
    const long long p_begin = T > 0 ? range_start(c, T, G) : 0;
    const long long p_end = T > 0 ? range_start(c + 1, T, G) : 0;
    if (c == 0 && tid == 0) *reinterpret_cast<long long*>(p.ws) = T;
    if (tid == 0) {
        ctl[0] = -1;  // first sequence of the range
        ctl[1] = 0;   // its first flat page
    }
    __syncthreads();
    if (p_begin < p_end) {
        long long carry = 0;
        for (int base = 0; base < p.batch; base += blockDim.x) {
            const int i = base + tid;
            const long long pg = i < p.batch ? pages_of(p.seq_lens[i]) : 0;
            long long chunk_total;
            const long long incl = block_scan(pg, red, &chunk_total) + carry;
            const long long excl = incl - pg;
            if (pg > 0 && excl <= p_begin && p_begin < incl) {
                ctl[0] = i;
                ctl[1] = excl;
            }
            carry += chunk_total;
            __syncthreads();
            if (ctl[0] >= 0) break;
        }
    }
    __syncthreads();
    const long long n_pages = p_end - p_begin;
    const int b_first = static_cast<int>(ctl[0]);
    const long long sp_first = ctl[1];
    if (n_pages <= 0 || b_first < 0) return;

    const long long row_bytes = static_cast<long long>(g.kv_dim) * 2;
    const long long half_page = g.page_bytes / 2;

    if (warp == 0) {
        // ------------------------------------------------------ producer
        int b = b_first;
        long long sp = sp_first;  // flat index of page 0 of sequence b
        int len_b = p.seq_lens[b];
        int pages_b = pages_of(len_b);
        int slot_b = p.slots[b];
        bool slot_ok = slot_b >= 0 && slot_b < g.num_slots;
        long long tbase = (static_cast<long long>(slot_ok ? slot_b : 0) * g.n_layers + p.layer) * g.maxb;
        long long win_base = -1;
        int win_val = -1;
        bool whole = false;
        long long k = 0;
        bool stop = false;
        for (long long pg = p_begin; pg < p_end; ++pg, ++k) {
            while (pg >= sp + pages_b) {  // next sequence with pages
                sp += pages_b;
                ++b;
                len_b = p.seq_lens[b];
                pages_b = pages_of(len_b);
                slot_b = p.slots[b];
                slot_ok = slot_b >= 0 && slot_b < g.num_slots;
                tbase = (static_cast<long long>(slot_ok ? slot_b : 0) * g.n_layers + p.layer) * g.maxb;
                win_base = -1;
            }
            const long long lp = pg - sp;
            if (win_base < 0 || lp >= win_base + 32) {
                win_base = lp;
                const long long idx = lp + lane;
                win_val = -1;
                if (slot_ok && idx < pages_b && idx < g.maxb) win_val = __ldg(p.bt + tbase + idx);
            }
            const int entry = __shfl_sync(0xffffffffu, win_val, static_cast<int>(lp - win_base));
            const bool bad = !slot_ok || lp >= g.maxb || entry < 0 || entry >= g.nblocks;
            const bool first = (pg == p_begin) || lp == 0;
            const bool last = (pg == p_end - 1) || lp == pages_b - 1;
            if (first) whole = (lp == 0) && (sp + pages_b <= p_end);
            const int ntok = (lp == pages_b - 1) ? len_b - static_cast<int>(lp) * kBlockTokens : kBlockTokens;
            const int st = static_cast<int>(k % p.nst);
            if (k >= p.nst &&
                !mbar_wait(&empty[st], static_cast<uint32_t>((k / p.nst - 1) & 1), abort_flag, p.err)) {
                stop = true;
                break;
            }
            if (lane == 0) {
                uint8_t* stage = stages + static_cast<long long>(st) * p.stage_bytes;
                StageHeader* hdr = reinterpret_cast<StageHeader*>(stage + g.page_bytes + p.q_bytes);
                if (lp == 0) {  // this CTA holds the sequence's first page: record its CTA span
                    int2 meta;
                    meta.x = static_cast<int>(c);
                    meta.y = static_cast<int>(owner_of(sp + pages_b - 1, T, G));
                    *reinterpret_cast<int2*>(p.ws + p.ws_meta + 8ll * b) = meta;
                }
                if (bad) set_error(p.err, PA_ERR_BAD_BLOCK);
                hdr->b = b;
                hdr->ntok = bad ? 0 : ntok;
                hdr->flags = (first ? kFirst : 0) | (last ? kLast : 0) | (whole ? kWhole : 0) | (bad ? kSkip : 0);
                hdr->slot_idx = static_cast<int>(b + c);
                const uint32_t kv_bytes = bad ? 0u : static_cast<uint32_t>(2ll * ntok * row_bytes);
                mbar_arrive_expect_tx(&full[st], kv_bytes + (first ? static_cast<uint32_t>(p.q_bytes) : 0u));
                if (!bad) {
                    const uint8_t* src = p.pool + static_cast<long long>(entry) * g.page_bytes;
                    if (ntok == kBlockTokens) {
                        bulk_g2s(stage, src, static_cast<uint32_t>(g.page_bytes), &full[st]);
                    } else {
                        const uint32_t part = static_cast<uint32_t>(ntok * row_bytes);
                        bulk_g2s(stage, src, part, &full[st]);
                        bulk_g2s(stage + half_page, src + half_page, part, &full[st]);
                    }
                }
                if (first)
                    bulk_g2s(stage + g.page_bytes, p.q + static_cast<long long>(b) * p.q_bytes,
                             static_cast<uint32_t>(p.q_bytes), &full[st]);
            }
            __syncwarp();
        }
        // Drain: the copies of the last stages must land before the CTA exits.
        if (stop && lane == 0) {
            const long long k0 = k > p.nst ? k - p.nst : 0;
            for (long long i = k0; i < k; ++i)
                mbar_drain(&full[i % p.nst], static_cast<uint32_t>((i / p.nst) & 1));
        }
        return;
    }

    // ---------------------------------------------------------- consumers
    const int cw = warp - 1;
    const int h = cw / p.wph;                 // kv head
    const int slice = cw % p.wph;             // which GW query heads of the group
    const int hq0 = h * g.group + slice * GW; // first query head of this warp
    const int sub = lane / LPT;               // token subgroup
    const int part = lane % LPT;              // 16-dim slice of the row

    float q[GW][16], acc[GW][16], m[GW], l[GW];
#pragma unroll
    for (int j = 0; j < GW; ++j) {
        m[j] = -CUDART_INF_F;
        l[j] = 0.f;
#pragma unroll
        for (int e = 0; e < 16; ++e) acc[j][e] = 0.f, q[j][e] = 0.f;
    }

    for (long long k = 0; k < n_pages; ++k) {
        const int st = static_cast<int>(k % p.nst);
        if (!mbar_wait(&full[st], static_cast<uint32_t>((k / p.nst) & 1), abort_flag, p.err)) break;
        const uint8_t* stage = stages + static_cast<long long>(st) * p.stage_bytes;
        const StageHeader hdr = *reinterpret_cast<const StageHeader*>(stage + g.page_bytes + p.q_bytes);

        if (hdr.flags & kFirst) {
            const uint8_t* qs = stage + g.page_bytes;
#pragma unroll
            for (int j = 0; j < GW; ++j) {
                const uint4* src = reinterpret_cast<const uint4*>(qs + ((hq0 + j) * D + part * 16) * 2);
                const uint4 a = src[0], bq = src[1];
                const uint32_t w[8] = {a.x, a.y, a.z, a.w, bq.x, bq.y, bq.z, bq.w};
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    q[j][2 * e] = bf16lo(w[e]);
                    q[j][2 * e + 1] = bf16hi(w[e]);
                }
                m[j] = -CUDART_INF_F;
                l[j] = 0.f;
#pragma unroll
                for (int e = 0; e < 16; ++e) acc[j][e] = 0.f;
            }
        }

        const uint8_t* kbase = stage + (h * D + part * 16) * 2;
#pragma unroll
        for (int pass = 0; pass < PASSES; ++pass) {
            const int t = pass * TPP + sub;
            const bool valid = t < hdr.ntok;
            float dot[GW];
            uint32_t vw[8];
#pragma unroll
            for (int j = 0; j < GW; ++j) dot[j] = 0.f;
            if (valid) {
                const uint4* kp = reinterpret_cast<const uint4*>(kbase + t * row_bytes);
                const uint4* vp = reinterpret_cast<const uint4*>(kbase + half_page + t * row_bytes);
                // neighbouring token rows sit 2*KV_DIM bytes apart (same banks): odd
                // subgroups read their second 16-byte chunk first so a quarter-warp
                // touches every bank once
                const int f = sub & 1;
                const uint4 ka = kp[f], kb = kp[f ^ 1], va = vp[f], vb = vp[f ^ 1];
                const uint4 k0 = f ? kb : ka, k1 = f ? ka : kb, v0 = f ? vb : va, v1 = f ? va : vb;
                const uint32_t kw[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
                vw[0] = v0.x; vw[1] = v0.y; vw[2] = v0.z; vw[3] = v0.w;
                vw[4] = v1.x; vw[5] = v1.y; vw[6] = v1.z; vw[7] = v1.w;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float x0 = bf16lo(kw[e]), x1 = bf16hi(kw[e]);
#pragma unroll
                    for (int j = 0; j < GW; ++j) dot[j] = fmaf(q[j][2 * e + 1], x1, fmaf(q[j][2 * e], x0, dot[j]));
                }
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) vw[e] = 0u;
            }
#pragma unroll
            for (int off = 1; off < LPT; off <<= 1)
#pragma unroll
                for (int j = 0; j < GW; ++j) dot[j] += __shfl_xor_sync(0xffffffffu, dot[j], off);
            if (valid) {
#pragma unroll
                for (int j = 0; j < GW; ++j) {
                    const float s = dot[j] * p.scale_log2;
                    if (s > m[j] + 8.f) {  // move the reference max (rare after the first token)
                        const float corr = ex2_approx(m[j] - s);
                        l[j] *= corr;
#pragma unroll
                        for (int e = 0; e < 16; ++e) acc[j][e] *= corr;
                        m[j] = s;
                    }
                    const float pw = ex2_approx(s - m[j]);
                    l[j] += pw;
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        acc[j][2 * e] = fmaf(pw, bf16lo(vw[e]), acc[j][2 * e]);
                        acc[j][2 * e + 1] = fmaf(pw, bf16hi(vw[e]), acc[j][2 * e + 1]);
                    }
                }
            }
        }

        if (hdr.flags & kLast) {
            // merge the token subgroups (lanes LPT, 2 LPT, ... apart)
#pragma unroll
            for (int off = LPT; off < 32; off <<= 1) {
#pragma unroll
                for (int j = 0; j < GW; ++j) {
                    const float mo = __shfl_xor_sync(0xffffffffu, m[j], off);
                    const float lo = __shfl_xor_sync(0xffffffffu, l[j], off);
                    const float mn = fmaxf(m[j], mo);
                    const float a = (m[j] == -CUDART_INF_F) ? 0.f : ex2_approx(m[j] - mn);
                    const float bw = (mo == -CUDART_INF_F) ? 0.f : ex2_approx(mo - mn);
                    l[j] = l[j] * a + lo * bw;
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const float ao = __shfl_xor_sync(0xffffffffu, acc[j][e], off);
                        acc[j][e] = acc[j][e] * a + ao * bw;
                    }
                    m[j] = mn;
                }
            }
            if (sub == 0) {
#pragma unroll
                for (int j = 0; j < GW; ++j) {
                    const int hq = hq0 + j;
                    const bool any = l[j] > 0.f;
                    const float inv = any ? 1.f / l[j] : 0.f;
                    const float L = any ? (m[j] + lg2_approx(l[j])) * kLn2 : -CUDART_INF_F;
                    if (hdr.flags & kWhole) {
                        uint32_t w[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) w[e] = pack_bf16x2(acc[j][2 * e] * inv, acc[j][2 * e + 1] * inv);
                        uint4* dst = reinterpret_cast<uint4*>(p.o + (static_cast<long long>(hdr.b) * g.hq + hq) * D + part * 16);
                        dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
                        dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
                        if (part == 0 && p.lse) p.lse[static_cast<long long>(hdr.b) * g.hq + hq] = L;
                    } else {
                        float4* dst = reinterpret_cast<float4*>(
                            p.ws + p.ws_o + ((static_cast<long long>(hdr.slot_idx) * g.hq + hq) * D + part * 16) * 4);
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            dst[e] = make_float4(acc[j][4 * e] * inv, acc[j][4 * e + 1] * inv,
                                                 acc[j][4 * e + 2] * inv, acc[j][4 * e + 3] * inv);
                        if (part == 0)
                            reinterpret_cast<float*>(p.ws + p.ws_lse)[static_cast<long long>(hdr.slot_idx) * g.hq + hq] = L;
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
    }
}

// Merges the partial units of every split sequence; writes o = 0, lse = -inf
// for empty sequences.  One CTA per sequence, one thread per (head, 8 dims).
template <int D>
__global__ void __launch_bounds__(256) decode_merge_kernel(const DecodeParams p) {
    const KGeom& g = p.g;
    const int b = blockIdx.x;
    const int len = p.seq_lens[b];
    const int chunks = g.hq * (D / 8);
    if (len <= 0) {
        for (int w = threadIdx.x; w < chunks; w += blockDim.x) {
            uint4* dst = reinterpret_cast<uint4*>(p.o + static_cast<long long>(b) * g.hq * D) + w;
            *dst = make_uint4(0u, 0u, 0u, 0u);
        }
        if (p.lse)
            for (int h = threadIdx.x; h < g.hq; h += blockDim.x) p.lse[static_cast<long long>(b) * g.hq + h] = -CUDART_INF_F;
        return;
    }
    const int2 meta = *reinterpret_cast<const int2*>(p.ws + p.ws_meta + 8ll * b);
    const long long G = p.attend_grid;
    if (meta.x < 0 || meta.y >= G || meta.x > meta.y) {  // attend kernel gave up early
        if (threadIdx.x == 0) set_error(p.err, PA_ERR_TIMEOUT);
        return;
    }
    if (meta.x == meta.y) return;  // one unit: the attend kernel wrote the result
    const long long T = *reinterpret_cast<const long long*>(p.ws);
    const float* lse_part = reinterpret_cast<const float*>(p.ws + p.ws_lse);
    const float* o_part = reinterpret_cast<const float*>(p.ws + p.ws_o);
    for (int w = threadIdx.x; w < chunks; w += blockDim.x) {
        const int hq = w / (D / 8);
        const int e0 = (w % (D / 8)) * 8;
        float M = -CUDART_INF_F, S = 0.f, acc[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = 0.f;
        for (long long cc = meta.x; cc <= meta.y; ++cc) {
            if (range_start(cc, T, G) == range_start(cc + 1, T, G)) continue;  // CTA without pages
            const long long slot = b + cc;
            const float Lc = lse_part[slot * g.hq + hq];
            if (Lc == -CUDART_INF_F) continue;
            const float4* src = reinterpret_cast<const float4*>(o_part + (slot * g.hq + hq) * D + e0);
            const float4 x0 = src[0], x1 = src[1];
            const float Mn = fmaxf(M, Lc);
            const float a = (M == -CUDART_INF_F) ? 0.f : ex2_approx((M - Mn) * kLog2e);
            const float wgt = ex2_approx((Lc - Mn) * kLog2e);
            S = S * a + wgt;
            const float xv[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = acc[e] * a + xv[e] * wgt;
            M = Mn;
        }
        const float inv = S > 0.f ? 1.f / S : 0.f;
        uint32_t packed[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) packed[e] = pack_bf16x2(acc[2 * e] * inv, acc[2 * e + 1] * inv);
        *reinterpret_cast<uint4*>(p.o + (static_cast<long long>(b) * g.hq + hq) * D + e0) =
            make_uint4(packed[0], packed[1], packed[2], packed[3]);
        if (e0 == 0 && p.lse)
            p.lse[static_cast<long long>(b) * g.hq + hq] = S > 0.f ? M + lg2_approx(S) * kLn2 : -CUDART_INF_F;
    }
}

struct LaunchShape {
    int gw, wph, nw, nst, stage_bytes, q_bytes, smem;
};

bool decode_shape(const KGeom& g, LaunchShape* s) {
    if (g.d != 64 && g.d != 128) return false;
    if (g.group != 1 && g.group != 2 && g.group != 4 && g.group != 8) return false;
    s->gw = g.group < 4 ? g.group : 4;
    s->wph = g.group / s->gw;
    s->nw = g.hkv * s->wph;
    if (s->nw > kMaxConsumerWarps) return false;
    s->q_bytes = g.hq * g.d * 2;
    const long long stage = align_up(g.page_bytes + s->q_bytes + static_cast<long long>(sizeof(StageHeader)), 128);
    if (stage > 64 * 1024 + 16 * 1024) return false;
    s->stage_bytes = static_cast<int>(stage);
    int nst = static_cast<int>((kSmemBudget - kCtlBytes) / stage);
    if (nst > kMaxStages) nst = kMaxStages;
    if (nst < 2) return false;
    s->nst = nst;
    s->smem = kCtlBytes + nst * s->stage_bytes;
    return true;
}

template <int D, int GW>
cudaError_t launch_attend(const DecodeParams& p, const LaunchShape& s, int grid, cudaStream_t stream) {
    auto kern = decode_attend_kernel<D, GW>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, s.smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, 32 * (1 + s.nw), s.smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

bool decode_supported(const KGeom& g) {
    LaunchShape s;
    return decode_shape(g, &s);
}

size_t decode_workspace_bytes(const KGeom& g, int batch, int max_seq_len) {
    const long long nslots = batch + grid_cap(batch, max_seq_len) - 1;
    return static_cast<size_t>(ws_layout(batch, nslots, g.hq, g.d).total);
}

cudaError_t launch_decode(const KGeom& g, const void* q, const void* pool, const int32_t* block_table,
                          int layer, int batch, const int32_t* seq_lens, const int32_t* slots,
                          int max_seq_len, float scale, void* o, float* lse, void* workspace,
                          int32_t* err, cudaStream_t stream) {
    LaunchShape s;
    if (!decode_shape(g, &s)) return cudaErrorInvalidValue;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    long long grid = grid_cap(batch, max_seq_len);
    if (grid > sms) grid = sms;
    const long long nslots = batch + grid_cap(batch, max_seq_len) - 1;
    const WsLayout w = ws_layout(batch, nslots, g.hq, g.d);

    DecodeParams p;
    p.g = g;
    p.q = static_cast<const uint8_t*>(q);
    p.pool = static_cast<const uint8_t*>(pool);
    p.bt = block_table;
    p.layer = layer;
    p.batch = batch;
    p.seq_lens = seq_lens;
    p.slots = slots;
    p.scale_log2 = scale * kLog2e;
    p.o = static_cast<__nv_bfloat16*>(o);
    p.lse = lse;
    p.ws = static_cast<uint8_t*>(workspace);
    p.ws_meta = w.meta;
    p.ws_lse = w.lse;
    p.ws_o = w.o;
    p.err = err;
    p.nst = s.nst;
    p.stage_bytes = s.stage_bytes;
    p.q_bytes = s.q_bytes;
    p.wph = s.wph;

    const int gi = static_cast<int>(grid);
    p.attend_grid = gi;
    if (g.d == 64) {
        e = s.gw == 1 ? launch_attend<64, 1>(p, s, gi, stream)
          : s.gw == 2 ? launch_attend<64, 2>(p, s, gi, stream)
                      : launch_attend<64, 4>(p, s, gi, stream);
        if (e != cudaSuccess) return e;
        decode_merge_kernel<64><<<batch, 256, 0, stream>>>(p);
    } else {
        e = s.gw == 1 ? launch_attend<128, 1>(p, s, gi, stream)
          : s.gw == 2 ? launch_attend<128, 2>(p, s, gi, stream)
                      : launch_attend<128, 4>(p, s, gi, stream);
        if (e != cudaSuccess) return e;
        decode_merge_kernel<128><<<batch, 256, 0, stream>>>(p);
    }
    return cudaGetLastError();
}

}  // namespace pa

// ---------------------------------------------------------------------------
// Allocation-free decode (pa_decode_noalloc, declared in pa.h).
//
// For callers that cannot allocate device memory where they decode -- a
// plugin whose host application has already reserved the device memory for
// its own allocator, or a serving loop that must not call cudaMalloc between
// steps -- the split partials go to this fixed array instead of a caller
// workspace.  It is part of the library's device code, so every GPU that
// loads these kernels holds it until the process exits.  Nothing in it has to
// start at zero: every byte the merge kernel reads is written earlier in the
// same call.  Calls that overlap on the GPU share it and race.
namespace pa {
namespace {

constexpr size_t kStaticScratchBytes = PA_DECODE_STATIC_SCRATCH_BYTES;
static __device__ __align__(256) uint8_t g_decode_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;

// Device address of g_decode_scratch on the current device, looked up once
// per device (in host code the array's name is only a host-side stand-in).
cudaError_t static_scratch(void** out) {
    static std::mutex mu;
    static void* addr[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (addr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (e != cudaSuccess) return e;
        addr[dev] = p;
    }
    *out = addr[dev];
    return cudaSuccess;
}

}  // namespace
}  // namespace pa

extern "C" __attribute__((visibility("default"))) pa_status pa_decode_noalloc(
    const pa_geom* geom, const void* q, const void* pool, const int32_t* block_table, int32_t layer,
    int32_t batch, const int32_t* seq_lens, const int32_t* slots, int32_t max_seq_len, float scale,
    void* o, float* lse, int32_t* err_flag, pa_stream_t stream) {
    if (pa_decode_workspace_size(geom, batch, max_seq_len) > pa::kStaticScratchBytes)
        return PA_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    if (pa::static_scratch(&scratch) != cudaSuccess) return PA_ERR_CUDA;
    return pa_decode(geom, q, pool, block_table, layer, batch, seq_lens, slots, max_seq_len, scale, o,
                     lse, scratch, pa::kStaticScratchBytes, err_flag, stream);
}


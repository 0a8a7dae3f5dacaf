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
//    prefetches 32 block-table entries per warp load, and moves each page
//    (32 KiB for 8 x 64) into a shared-memory stage with two TMA tensor copies,
//    one for the K half and one for the V half.  The tensor map views the
//    pool as [64 dims][rows of 2*KV_DIM bytes][KV_DIM/64 column blocks of 128
//    bytes]: one {64, 16, KV_DIM/64} box is a whole half page, laid down as
//    128-byte lines (column block major, token minor) with the 128-byte
//    swizzle, so the 16-byte pieces of 8 consecutive token rows sit in 8
//    different bank groups.  The sequence's query row rides along at the start
//    of a unit.  Two CTAs per SM, two stages each, keep enough bytes in
//    flight for HBM; the page is read front to back in two large requests.
//  * Compute.  One consumer warp per KV head; the GQA group's query heads are
//    the rows of a 16-row warp-level MMA (mma.sync m16n8k16, bf16 in, fp32
//    accumulate; rows past the group are zero): per page S = Q K^T is 8 MMAs
//    (d 64) with K fragments from ldmatrix, the online softmax runs on the
//    accumulator fragments (one row per lane quad, a 2-step xor-shuffle max),
//    and P goes straight from those fragments into the A operand of O += P V
//    (V fragments from ldmatrix.trans, addresses following the swizzle).  The
//    running max is only moved when a page's max exceeds it by more than 2^8
//    (exact: o and l share the same reference m).
#include <math_constants.h>

#include <mutex>

#include "pa_internal.cuh"

// Profiling build only (PA_DECODE_TRACE, libpa_trace.so): globaltimer marks of
// every attend CTA (start, first page in shared memory, end, SM) and every
// merge CTA (past the grid dependency, end), read back by
// paged_kv_cache_gb300/decode_trace.py.  The product library has none of it.
#ifndef PA_DECODE_TRACE
#define PA_DECODE_TRACE 0
#endif
#if PA_DECODE_TRACE
namespace pa {
constexpr int kTraceAttend = 1024, kTraceMerge = 8192;
__device__ unsigned long long g_trace[kTraceAttend * 4 + kTraceMerge * 2];
__device__ __forceinline__ void trace_set(int i, unsigned long long v) { g_trace[i] = v; }
__device__ __forceinline__ void trace_max(int i, unsigned long long v) { atomicMax(&g_trace[i], v); }
}  // namespace pa
#define PA_TRACE(stmt) stmt
#else
#define PA_TRACE(stmt)
#endif

namespace pa {
namespace {

constexpr int kMaxConsumerWarps = 8;
constexpr int kMaxGrid = 1024;
constexpr int kSmemBudget = 112 * 1024;  // per CTA: two CTAs share an SM
constexpr int kCtasPerSm = 2;
constexpr int kMaxStages = 8;
// Stages per CTA: two measured faster than three (256 mixed-length sequences
// 160 -> 154 us, 64 sequences of 128..2048 tokens 43.3 -> 42.3 us): with 304
// CTAs, two 32 KiB pages each already keep ~19 MB in flight, and fewer
// requests queued in the memory system even out the CTAs' service.
constexpr int kStagesWanted = 2;
constexpr int kCtlBytes = 1024;  // barriers + control words, then the q slots, then the stages

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
    long long ws_lse;     // float [nslots][hq]: partial L (natural log)
    long long ws_o;       // float [nslots][hq][d]: partial normalised outputs
    int32_t* err;
    int attend_grid;      // CTAs of the attend kernel (G)
    int nst;              // pipeline stages
    int kv_stage_bytes;   // 64 * kv_dim: a whole page, K half then V half
    int q_bytes;          // hq * d * 2
    int qslot_bytes;      // q row + stage header, 64-byte multiple
    int stages_off;       // offset of the (1024-aligned) page stages in shared memory
    int hold_first_copy;  // diagnostic: CTA 0 arms its first page copy without issuing it
};

__host__ __device__ inline long long align_up(long long x, long long a) { return (x + a - 1) / a * a; }

struct WsLayout {
    long long lse, o, total;
};

__host__ __device__ inline WsLayout ws_layout(int batch, long long nslots, int hq, int d) {
    WsLayout w;
    (void)batch;
    w.lse = 0;
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

template <int D>
__global__ void __launch_bounds__(32 * (1 + kMaxConsumerWarps), D == 64 ? kCtasPerSm : 1)
decode_attend_kernel(const __grid_constant__ CUtensorMap kvmap, const DecodeParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);  // swizzled stages want 1024 B
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    uint64_t* empty = full + kMaxStages;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 256);
    long long* ctl = reinterpret_cast<long long*>(smem + 512);  // scan scratch and results
    long long* red = ctl + 8;                                   // per-warp partials
    uint8_t* qslots = smem + kCtlBytes;                         // per stage: q row, header
    uint8_t* stages = smem + p.stages_off;

    const KGeom& g = p.g;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n_consumers = (blockDim.x >> 5) - 1;
    const long long G = gridDim.x, c = blockIdx.x;
    // The merge grid may be scheduled now: its CTAs wait (griddepcontrol.wait)
    // until this grid has finished and its writes are visible.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    PA_TRACE(if (tid == 0 && blockIdx.x < kTraceAttend) {
        unsigned smid;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
        trace_set(blockIdx.x * 4 + 0, global_timer_ns());
        trace_set(blockIdx.x * 4 + 3, smid);
    })

    if (tid == 0) {
        for (int s = 0; s < p.nst; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], n_consumers);
        }
        *abort_flag = 0;
        mbar_init_fence();
    }

    // ---- this CTA's page range: total pages, then the sequence holding p_begin
    // (the slots of the first blockDim sequences are loaded with their lengths,
    // so that the first table row needs no further round trip)
    long long local = 0;
    int my_slot = -1;
    for (int i = tid; i < p.batch; i += blockDim.x) {
        int len = p.seq_lens[i];
        if (i == tid) my_slot = p.slots[i];
        if (len < 0) set_error(p.err, PA_ERR_BAD_BLOCK);
        local += pages_of(len);
    }
    const long long T = block_sum(local, red);
    const long long p_begin = T > 0 ? range_start(c, T, G) : 0;
    const long long p_end = T > 0 ? range_start(c + 1, T, G) : 0;
    if (tid == 0) {
        ctl[0] = -1;  // first sequence of the range
        ctl[1] = 0;   // its first flat page
        ctl[2] = -1;  // its slot
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
                ctl[2] = base == 0 ? my_slot : p.slots[i];
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
    const int slot_first = static_cast<int>(ctl[2]);
    if (n_pages <= 0 || b_first < 0) return;


    if (warp == 0) {
        // ------------------------------------------------------ producer
        int b = b_first;
        long long sp = sp_first;  // flat index of page 0 of sequence b
        int len_b = p.seq_lens[b];
        int pages_b = pages_of(len_b);
        int slot_b = slot_first;
        bool slot_ok = slot_b >= 0 && slot_b < g.num_slots;
        long long tbase = (static_cast<long long>(slot_ok ? slot_b : 0) * g.n_layers + p.layer) * g.maxb;
        long long win_base = -1;
        int win_val = -1;
        // the first 32 table entries of the next sequence, loaded ahead so that
        // crossing into it does not wait on the table (valid when nxt_b >= 0)
        int nxt_b = -1, nxt_val = -1;
        auto preload = [&](int bb) {
            nxt_b = -1;
            if (bb >= p.batch) return;
            const int s2 = p.slots[bb];
            const int pg2 = pages_of(p.seq_lens[bb]);
            if (s2 < 0 || s2 >= g.num_slots || pg2 <= 0) return;
            const long long tb2 = (static_cast<long long>(s2) * g.n_layers + p.layer) * g.maxb;
            nxt_val = (lane < pg2 && lane < g.maxb) ? __ldg(p.bt + tb2 + lane) : -1;
            nxt_b = bb;
        };
        if (sp + pages_b < p_end) preload(b + 1);  // the range goes past this sequence
        const bool hold = p.hold_first_copy && c == 0;
        bool whole = false;
        long long k = 0;
        for (long long pg = p_begin; pg < p_end; ++pg, ++k) {
            if (pg >= sp + pages_b) {
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
                if (b == nxt_b) {  // entries 0..31 of this sequence are already here
                    win_base = 0;
                    win_val = nxt_val;
                }
                nxt_b = -1;
                if (sp + pages_b < p_end) preload(b + 1);
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
            if (k >= p.nst && !mbar_wait(&empty[st], static_cast<uint32_t>((k / p.nst - 1) & 1), abort_flag, p.err))
                break;  // a consumer stopped the CTA, or the wait ran out
            if (lane == 0) {
                uint8_t* stage = stages + static_cast<long long>(st) * p.kv_stage_bytes;
                uint8_t* qslot = qslots + st * p.qslot_bytes;
                StageHeader* hdr = reinterpret_cast<StageHeader*>(qslot + p.q_bytes);
                if (bad) set_error(p.err, PA_ERR_BAD_BLOCK);
                hdr->b = b;
                hdr->ntok = bad ? 0 : ntok;
                hdr->flags = (first ? kFirst : 0) | (last ? kLast : 0) | (whole ? kWhole : 0) | (bad ? kSkip : 0);
                hdr->slot_idx = static_cast<int>(b + c);
                const uint32_t kv_bytes = bad ? 0u : static_cast<uint32_t>(p.kv_stage_bytes);
                mbar_arrive_expect_tx(&full[st], kv_bytes + (first ? static_cast<uint32_t>(p.q_bytes) : 0u));
                // the diagnostic hold: the first page's copy is armed, not issued
                if (!bad && !(hold && k == 0)) {  // whole K half and whole V half (a partial page's tail is not used)
                    tma_load_3d(stage, &kvmap, 0, entry * 32, 0, &full[st]);
                    tma_load_3d(stage + p.kv_stage_bytes / 2, &kvmap, 0, entry * 32 + 16, 0, &full[st]);
                }
                if (first)
                    bulk_g2s(qslot, p.q + static_cast<long long>(b) * p.q_bytes, static_cast<uint32_t>(p.q_bytes),
                             &full[st]);
            }
            __syncwarp();
        }
        // Drain: the copies of the last stages land before the CTA exits,
        // whichever role stopped it (phases already complete return at once).
        if (lane == 0) {
            const long long k0 = k > p.nst ? k - p.nst : 0;
            for (long long i = k0; i < k; ++i)
                if (!(hold && i == 0)) mbar_drain(&full[i % p.nst], static_cast<uint32_t>((i / p.nst) & 1));
        }
        return;
    }

    // ---------------------------------------------------------- consumers
    const int h = warp - 1;                   // kv head of this warp
    const int gid = lane >> 2, tq = lane & 3; // MMA fragment row group / column pair
    const bool row_real = gid < g.group;      // fragment row gid is a real query head
    const int hq_row = h * g.group + gid;
    const int mi = lane >> 3, rr = lane & 7;  // ldmatrix: matrix and row this lane addresses
    // Address of 16-byte piece (token t, dims d0..d0+7 of this warp's head) in a
    // half page: line = 16 * (column block) + t, piece swizzled by t % 8.
    auto piece = [&](int t, int d0) -> uint32_t {
        const int col = h * D + d0;
        return static_cast<uint32_t>((((col >> 6) * 16 + t) << 7) + ((((col & 63) >> 3) ^ (t & 7)) << 4));
    };
    const int half = p.kv_stage_bytes / 2;
    const float sl2 = p.scale_log2;

    uint32_t qa[D / 16][2];  // A fragments of Q (rows gid; the rows gid+8 are zero)
    float oacc[D / 8][4];    // O accumulator fragments, 8 dims per tile
    float m_ref = -CUDART_INF_F, l_part = 0.f;
#pragma unroll
    for (int ks = 0; ks < D / 16; ++ks) qa[ks][0] = qa[ks][1] = 0u;
#pragma unroll
    for (int nt = 0; nt < D / 8; ++nt) oacc[nt][0] = oacc[nt][1] = oacc[nt][2] = oacc[nt][3] = 0.f;

    for (long long k = 0; k < n_pages; ++k) {
        const int st = static_cast<int>(k % p.nst);
        if (!mbar_wait(&full[st], static_cast<uint32_t>((k / p.nst) & 1), abort_flag, p.err)) break;
        PA_TRACE(if (k == 0 && warp == 1 && lane == 0 && blockIdx.x < kTraceAttend)
                     trace_set(blockIdx.x * 4 + 1, global_timer_ns());)
        uint8_t* stage = stages + static_cast<long long>(st) * p.kv_stage_bytes;
        const uint8_t* qslot = qslots + st * p.qslot_bytes;
        const StageHeader hdr = *reinterpret_cast<const StageHeader*>(qslot + p.q_bytes);
        const uint32_t kbase = smem_u32(stage), vbase = kbase + half;

        if (hdr.flags & kFirst) {
            const uint8_t* qrow = qslot + hq_row * D * 2;
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                qa[ks][0] = row_real ? *reinterpret_cast<const uint32_t*>(qrow + (16 * ks + 2 * tq) * 2) : 0u;
                qa[ks][1] = row_real ? *reinterpret_cast<const uint32_t*>(qrow + (16 * ks + 8 + 2 * tq) * 2) : 0u;
            }
            m_ref = -CUDART_INF_F;
            l_part = 0.f;
#pragma unroll
            for (int nt = 0; nt < D / 8; ++nt) oacc[nt][0] = oacc[nt][1] = oacc[nt][2] = oacc[nt][3] = 0.f;
        }

        if (!(hdr.flags & kSkip)) {
            const int ntok = hdr.ntok;
            if (ntok < kBlockTokens) {  // rows past the end: zero this head's V lines (0 x NaN guard)
                constexpr int LINES = D / 64;  // 128-byte lines per token row of one head
                for (int idx = lane; idx < (kBlockTokens - ntok) * LINES * 8; idx += 32) {
                    const int t = ntok + idx / (LINES * 8);
                    const int blk = (idx / 8) % LINES;
                    *reinterpret_cast<uint4*>(stage + half + (((h * LINES + blk) * 16 + t) << 7) + ((idx & 7) << 4)) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
                __syncwarp();
            }
            // S = Q K^T: two 8-token tiles; matrices (tokens 0-7 | 8-15) x (dims +0 | +8)
            float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                uint32_t kb[4];
                ldmatrix_x4(kb, kbase + piece((mi >> 1) * 8 + rr, 16 * ks + (mi & 1) * 8));
                const uint32_t a[4] = {qa[ks][0], 0u, qa[ks][1], 0u};
                mma_bf16_16816(s0, a, kb[0], kb[1]);
                mma_bf16_16816(s1, a, kb[2], kb[3]);
            }
            // this lane's scores: row gid, tokens 2tq, 2tq+1, 8+2tq, 9+2tq
            float x0 = s0[0], x1 = s0[1], x2 = s1[0], x3 = s1[1];
            if (ntok < kBlockTokens) {
                if (2 * tq >= ntok) x0 = -CUDART_INF_F;
                if (2 * tq + 1 >= ntok) x1 = -CUDART_INF_F;
                if (8 + 2 * tq >= ntok) x2 = -CUDART_INF_F;
                if (9 + 2 * tq >= ntok) x3 = -CUDART_INF_F;
            }
            float mx = fmaxf(fmaxf(x0, x1), fmaxf(x2, x3));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const float m_tile = mx * sl2;
            if (m_tile > m_ref + 8.f) {  // move the reference max (same decision across the quad)
                const float corr = ex2_approx(m_ref - m_tile);
                l_part *= corr;
#pragma unroll
                for (int nt = 0; nt < D / 8; ++nt) {
                    oacc[nt][0] *= corr;
                    oacc[nt][1] *= corr;
                }
                m_ref = m_tile;
            }
            float e0, e1, e2, e3;
            ffma2(e0, e1, x0, x1, sl2, sl2, -m_ref, -m_ref);
            ffma2(e2, e3, x2, x3, sl2, sl2, -m_ref, -m_ref);
            const float p0 = ex2_approx(e0), p1 = ex2_approx(e1), p2 = ex2_approx(e2), p3 = ex2_approx(e3);
            l_part += (p0 + p1) + (p2 + p3);
            const uint32_t pa[4] = {pack_bf16x2(p0, p1), 0u, pack_bf16x2(p2, p3), 0u};
            // O += P V
#pragma unroll
            for (int np = 0; np < D / 16; ++np) {  // matrices (tokens 0-7 | 8-15) x (dims +0 | +8)
                uint32_t vb[4];
                ldmatrix_x4_trans(vb, vbase + piece((mi & 1) * 8 + rr, 16 * np + (mi >> 1) * 8));
                mma_bf16_16816(oacc[2 * np], pa, vb[0], vb[1]);
                mma_bf16_16816(oacc[2 * np + 1], pa, vb[2], vb[3]);
            }
            if (ntok < kBlockTokens) fence_proxy_async_smem();  // our zeros before the next TMA copy
        }

        if (hdr.flags & kLast) {
            float l = l_part + __shfl_xor_sync(0xffffffffu, l_part, 1);
            l += __shfl_xor_sync(0xffffffffu, l, 2);
            if (row_real) {
                const bool any = l > 0.f;
                const float inv = any ? 1.f / l : 0.f;
                const float L = any ? (m_ref + lg2_approx(l)) * kLn2 : -CUDART_INF_F;
                if (hdr.flags & kWhole) {
                    __nv_bfloat16* dst = p.o + (static_cast<long long>(hdr.b) * g.hq + hq_row) * D + 2 * tq;
#pragma unroll
                    for (int nt = 0; nt < D / 8; ++nt)
                        *reinterpret_cast<uint32_t*>(dst + 8 * nt) = pack_bf16x2(oacc[nt][0] * inv, oacc[nt][1] * inv);
                    if (tq == 0 && p.lse) p.lse[static_cast<long long>(hdr.b) * g.hq + hq_row] = L;
                } else {
                    float* dst = reinterpret_cast<float*>(p.ws + p.ws_o) +
                                 (static_cast<long long>(hdr.slot_idx) * g.hq + hq_row) * D + 2 * tq;
#pragma unroll
                    for (int nt = 0; nt < D / 8; ++nt)
                        *reinterpret_cast<float2*>(dst + 8 * nt) = make_float2(oacc[nt][0] * inv, oacc[nt][1] * inv);
                    if (tq == 0)
                        reinterpret_cast<float*>(p.ws + p.ws_lse)[static_cast<long long>(hdr.slot_idx) * g.hq + hq_row] = L;
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
    }
    PA_TRACE(if (lane == 0 && blockIdx.x < kTraceAttend) trace_max(blockIdx.x * 4 + 2, global_timer_ns());)
}

// The CTAs of the attend grid that hold sequence b, from the lengths and the
// grid size alone (the same split the attend kernel makes): first and last
// CTA, the page count T and whether the span is empty.  All threads of the
// block call it; it reads only seq_lens.
struct SeqSpan {
    long long T, c0, c1;
    int len;
};

__device__ SeqSpan seq_span(const DecodeParams& p, int b, long long G, long long* red) {
    long long tot = 0, before = 0;
    for (int i = threadIdx.x; i < p.batch; i += blockDim.x) {
        const long long pg = pages_of(p.seq_lens[i]);
        tot += pg;
        if (i < b) before += pg;
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        tot += __shfl_xor_sync(0xffffffffu, tot, off);
        before += __shfl_xor_sync(0xffffffffu, before, off);
    }
    if (lane == 0) {
        red[2 * warp] = tot;
        red[2 * warp + 1] = before;
    }
    __syncthreads();
    SeqSpan s;
    s.T = 0;
    long long sp = 0;
    for (int w = 0; w < nw; ++w) {
        s.T += red[2 * w];
        sp += red[2 * w + 1];
    }
    s.len = p.seq_lens[b];
    const int pages_b = pages_of(s.len);
    s.c0 = pages_b > 0 ? owner_of(sp, s.T, G) : 0;
    s.c1 = pages_b > 0 ? owner_of(sp + pages_b - 1, s.T, G) : 0;
    return s;
}

// Merges the partial units of every split sequence; writes o = 0, lse = -inf
// for empty sequences.  One CTA per (sequence, 8 q heads), one warp per head.
// Launched as a programmatic dependent of the attend kernel: the span of the
// sequence comes from the lengths before griddepcontrol.wait, and everything
// the attend kernel writes is read after it, in one round of loads per
// kMergeBatch pieces: lane k takes piece k's L for the max and the weights of
// the LSE rule while every lane loads its dims of the pieces' rows.
constexpr int kMergeHeadsPerCta = 8;
constexpr int kMergeThreads = 32 * kMergeHeadsPerCta;
constexpr int kMergeBatch = 16;  // pieces whose loads are all in flight at once

template <int D>
__global__ void __launch_bounds__(kMergeThreads) decode_merge_kernel(const DecodeParams p) {
    constexpr int PER = D / 32;  // dims per lane
    __shared__ long long red[2 * (kMergeThreads / 32)];
    const KGeom& g = p.g;
    const int b = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int hq = blockIdx.y * kMergeHeadsPerCta + warp;
    const long long G = p.attend_grid;
    const SeqSpan sp = seq_span(p, b, G, red);
    asm volatile("griddepcontrol.wait;" ::: "memory");
    PA_TRACE(const int trace_id = blockIdx.y * gridDim.x + blockIdx.x;
             if (threadIdx.x == 0 && trace_id < kTraceMerge)
                 trace_set(kTraceAttend * 4 + trace_id * 2, global_timer_ns());
             struct TraceEnd {
                 int id;
                 __device__ ~TraceEnd() {
                     if ((threadIdx.x & 31) == 0 && id < kTraceMerge)
                         trace_max(kTraceAttend * 4 + id * 2 + 1, global_timer_ns());
                 }
             } trace_end{trace_id};)
    if (hq >= g.hq) return;
    const long long row = static_cast<long long>(b) * g.hq + hq;
    if (sp.len <= 0) {
#pragma unroll
        for (int e = 0; e < PER; ++e) p.o[row * D + lane * PER + e] = __float2bfloat16_rn(0.f);
        if (lane == 0 && p.lse) p.lse[row] = -CUDART_INF_F;
        return;
    }
    if (sp.c0 == sp.c1) return;  // one unit: the attend kernel wrote the result
    const long long T = sp.T;
    const int P = static_cast<int>(sp.c1 - sp.c0 + 1);  // pieces
    const float* lse_part = reinterpret_cast<const float*>(p.ws + p.ws_lse);
    const float* o_part = reinterpret_cast<const float*>(p.ws + p.ws_o);
    // CTAs of the attend grid whose page range is empty wrote nothing
    auto has_pages = [&](long long cc) { return range_start(cc, T, G) != range_start(cc + 1, T, G); };
    auto load_row = [&](long long cc, float* v) {
        const float* src = o_part + ((b + cc) * g.hq + hq) * D + lane * PER;
        if (PER == 2) {
            const float2 x = *reinterpret_cast<const float2*>(src);
            v[0] = x.x;
            v[PER - 1] = x.y;
        } else {
            const float4 x = *reinterpret_cast<const float4*>(src);
            v[0] = x.x;
            v[1 % PER] = x.y;
            v[2 % PER] = x.z;
            v[3 % PER] = x.w;
        }
    };

    float acc[PER], S = 0.f;
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] = 0.f;
    float M = -CUDART_INF_F;
    // Batches of kMergeBatch pieces, each in one round of loads: lane k takes
    // piece k's L while every lane loads its dims of all the batch's rows.
    // With more than one batch the max comes first, in a pass of its own.
    const bool one_batch = P <= kMergeBatch;
    if (!one_batch) {
        for (long long cc = sp.c0 + lane; cc <= sp.c1; cc += 32)
            if (has_pages(cc)) M = fmaxf(M, lse_part[(b + cc) * g.hq + hq]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    }
    for (long long c0 = sp.c0; c0 <= sp.c1; c0 += kMergeBatch) {
        const int n = static_cast<int>(min(static_cast<long long>(kMergeBatch), sp.c1 - c0 + 1));
        float v[kMergeBatch][PER];
#pragma unroll
        for (int k = 0; k < kMergeBatch; ++k)
            if (k < n) load_row(c0 + k, v[k]);
        const bool mine = lane < n && has_pages(c0 + lane);
        const float Lm = mine ? lse_part[(b + c0 + lane) * g.hq + hq] : -CUDART_INF_F;
        if (one_batch) {
            M = Lm;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
        }
        const float w = (M == -CUDART_INF_F || Lm == -CUDART_INF_F) ? 0.f : ex2_approx((Lm - M) * kLog2e);
        S += w;
#pragma unroll
        for (int k = 0; k < kMergeBatch; ++k) {
            const float wk = __shfl_sync(0xffffffffu, w, k);
            if (k < n && wk != 0.f) {
#pragma unroll
                for (int e = 0; e < PER; ++e) acc[e] = fmaf(wk, v[k][e], acc[e]);
            }
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) S += __shfl_xor_sync(0xffffffffu, S, off);

    // 3. the row
    const float inv = S > 0.f ? 1.f / S : 0.f;
#pragma unroll
    for (int e = 0; e < PER; ++e) p.o[row * D + lane * PER + e] = __float2bfloat16_rn(acc[e] * inv);
    if (lane == 0 && p.lse) p.lse[row] = S > 0.f ? M + lg2_approx(S) * kLn2 : -CUDART_INF_F;
}

// The same merge with one CTA per (sequence, q head): its 8 warps take the
// partials in turn and add their sums through shared memory.  Used when the
// batch has few (sequence, head) rows, so that long sequences, which the
// attend grid splits into many pieces, do not leave one warp walking all of
// them while most SMs idle.
template <int D>
__global__ void __launch_bounds__(kMergeThreads) decode_merge_split_kernel(const DecodeParams p) {
    constexpr int PER = D / 32;
    constexpr int W = kMergeThreads / 32;
    __shared__ long long red[2 * W];
    __shared__ float red_m[W];
    __shared__ float red_s[W];
    __shared__ float red_o[W][D];
    const KGeom& g = p.g;
    const int b = blockIdx.x, hq = blockIdx.y;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const long long G = p.attend_grid;
    const SeqSpan sp = seq_span(p, b, G, red);
    asm volatile("griddepcontrol.wait;" ::: "memory");
    PA_TRACE(const int trace_id = blockIdx.y * gridDim.x + blockIdx.x;
             if (threadIdx.x == 0 && trace_id < kTraceMerge)
                 trace_set(kTraceAttend * 4 + trace_id * 2, global_timer_ns());
             struct TraceEnd {
                 int id;
                 __device__ ~TraceEnd() {
                     if ((threadIdx.x & 31) == 0 && id < kTraceMerge)
                         trace_max(kTraceAttend * 4 + id * 2 + 1, global_timer_ns());
                 }
             } trace_end{trace_id};)
    const long long row = static_cast<long long>(b) * g.hq + hq;
    if (sp.len <= 0) {
        if (warp == 0) {
#pragma unroll
            for (int e = 0; e < PER; ++e) p.o[row * D + lane * PER + e] = __float2bfloat16_rn(0.f);
            if (lane == 0 && p.lse) p.lse[row] = -CUDART_INF_F;
        }
        return;
    }
    if (sp.c0 == sp.c1) return;  // one unit: the attend kernel wrote the result
    const long long T = sp.T;
    const float* lse_part = reinterpret_cast<const float*>(p.ws + p.ws_lse);
    const float* o_part = reinterpret_cast<const float*>(p.ws + p.ws_o);
    auto has_pages = [&](long long cc) { return range_start(cc, T, G) != range_start(cc + 1, T, G); };

    // 1. max of the partial L over the whole CTA
    float M = -CUDART_INF_F;
    for (long long cc = sp.c0 + threadIdx.x; cc <= sp.c1; cc += kMergeThreads)
        if (has_pages(cc)) M = fmaxf(M, lse_part[(b + cc) * g.hq + hq]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    if (lane == 0) red_m[warp] = M;
    __syncthreads();
#pragma unroll
    for (int w = 0; w < W; ++w) M = fmaxf(M, red_m[w]);

    // 2. warp w sums partials sp.c0 + w, + W, ... (lanes over dims)
    float acc[PER], S = 0.f;
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] = 0.f;
    if (M != -CUDART_INF_F) {
#pragma unroll 4
        for (long long cc = sp.c0 + warp; cc <= sp.c1; cc += W) {
            if (!has_pages(cc)) continue;
            const float Lc = lse_part[(b + cc) * g.hq + hq];
            const float wk = (Lc == -CUDART_INF_F) ? 0.f : ex2_approx((Lc - M) * kLog2e);
            S += wk;
            const float* src = o_part + ((b + cc) * g.hq + hq) * D + lane * PER;
            if (PER == 2) {
                const float2 v = *reinterpret_cast<const float2*>(src);
                acc[0] = fmaf(wk, v.x, acc[0]);
                acc[PER - 1] = fmaf(wk, v.y, acc[PER - 1]);
            } else {
                const float4 v = *reinterpret_cast<const float4*>(src);
                acc[0] = fmaf(wk, v.x, acc[0]);
                acc[1 % PER] = fmaf(wk, v.y, acc[1 % PER]);
                acc[2 % PER] = fmaf(wk, v.z, acc[2 % PER]);
                acc[3 % PER] = fmaf(wk, v.w, acc[3 % PER]);
            }
        }
    }
    if (lane == 0) red_s[warp] = S;
#pragma unroll
    for (int e = 0; e < PER; ++e) red_o[warp][lane * PER + e] = acc[e];
    __syncthreads();

    // 3. the row
    if (warp == 0) {
        float St = 0.f;
#pragma unroll
        for (int w = 0; w < W; ++w) St += red_s[w];
        const float inv = St > 0.f ? 1.f / St : 0.f;
#pragma unroll
        for (int e = 0; e < PER; ++e) {
            float a = 0.f;
#pragma unroll
            for (int w = 0; w < W; ++w) a += red_o[w][lane * PER + e];
            p.o[row * D + lane * PER + e] = __float2bfloat16_rn(a * inv);
        }
        if (lane == 0 && p.lse) p.lse[row] = St > 0.f ? M + lg2_approx(St) * kLn2 : -CUDART_INF_F;
    }
}

template <int D>
cudaError_t launch_merge(const DecodeParams& p, int batch, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    // few (sequence, head) rows: a CTA per row; else a warp per row
    const bool split = static_cast<long long>(batch) * p.g.hq <= 4ll * p.attend_grid;
    cfg.gridDim = split ? dim3(static_cast<unsigned>(batch), static_cast<unsigned>(p.g.hq), 1)
                        : dim3(static_cast<unsigned>(batch),
                               static_cast<unsigned>((p.g.hq + kMergeHeadsPerCta - 1) / kMergeHeadsPerCta), 1);
    cfg.blockDim = dim3(kMergeThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return split ? cudaLaunchKernelEx(&cfg, decode_merge_split_kernel<D>, p)
                 : cudaLaunchKernelEx(&cfg, decode_merge_kernel<D>, p);
}

struct LaunchShape {
    int nw, nst, kv_stage_bytes, q_bytes, qslot_bytes, stages_off, smem;
};

bool decode_shape(const KGeom& g, LaunchShape* s) {
    if (g.d != 64 && g.d != 128) return false;
    if (g.group != 1 && g.group != 2 && g.group != 4 && g.group != 8) return false;
    s->nw = g.hkv;  // one consumer warp per kv head
    if (s->nw > kMaxConsumerWarps) return false;
    if (g.kv_dim / 64 > 256) return false;  // TMA box dimension
    s->q_bytes = g.hq * g.d * 2;
    s->qslot_bytes = static_cast<int>(align_up(s->q_bytes + static_cast<long long>(sizeof(StageHeader)), 64));
    s->kv_stage_bytes = static_cast<int>(g.page_bytes);
    if (s->kv_stage_bytes > 64 * 1024) return false;
    // 1024 B of slack to align the dynamic base, control words, q slots, stages
    int nst = kStagesWanted;
    for (; nst >= 2; --nst) {
        const long long off = align_up(kCtlBytes + static_cast<long long>(nst) * s->qslot_bytes, 1024);
        if (1024 + off + static_cast<long long>(nst) * s->kv_stage_bytes <= kSmemBudget) break;
    }
    if (nst < 2) return false;
    s->nst = nst;
    s->stages_off = static_cast<int>(align_up(kCtlBytes + static_cast<long long>(nst) * s->qslot_bytes, 1024));
    s->smem = 1024 + s->stages_off + nst * s->kv_stage_bytes;
    return true;
}

// The pool as a 3D tensor {64 dims, pages*32 rows of 2*KV_DIM bytes,
// KV_DIM/64 column blocks of 128 bytes}; one box {64, 16, KV_DIM/64} is a
// half page (16 token rows, all heads).
bool encode_pool_map(CUtensorMap* map, const KGeom& g, const void* pool) {
    EncodeTiledFn fn = tensor_map_encoder();
    if (!fn) return false;
    const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(g.nblocks) * 32, static_cast<cuuint64_t>(g.kv_dim / 64)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(g.kv_dim) * 2, 128};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(kBlockTokens), static_cast<cuuint32_t>(g.kv_dim / 64)};
    const cuuint32_t estr[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(pool), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
cudaError_t launch_attend(const CUtensorMap& map, const DecodeParams& p, const LaunchShape& s, int grid,
                          cudaStream_t stream) {
    auto kern = decode_attend_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, s.smem);
    if (e != cudaSuccess) return e;
    kern<<<grid, 32 * (1 + s.nw), s.smem, stream>>>(map, p);
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
    if (grid > static_cast<long long>(kCtasPerSm) * sms) grid = static_cast<long long>(kCtasPerSm) * sms;
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
    p.ws_lse = w.lse;
    p.ws_o = w.o;
    p.err = err;
    p.nst = s.nst;
    p.kv_stage_bytes = s.kv_stage_bytes;
    p.q_bytes = s.q_bytes;
    p.qslot_bytes = s.qslot_bytes;
    p.stages_off = s.stages_off;
    p.hold_first_copy = debug_hold_first_copy();
    CUtensorMap map;
    if (!encode_pool_map(&map, g, pool)) return cudaErrorInvalidValue;

    const int gi = static_cast<int>(grid);
    p.attend_grid = gi;
    if (g.d == 64) {
        e = launch_attend<64>(map, p, s, gi, stream);
        if (e != cudaSuccess) return e;
        e = launch_merge<64>(p, batch, stream);
        if (e != cudaSuccess) return e;
    } else {
        e = launch_attend<128>(map, p, s, gi, stream);
        if (e != cudaSuccess) return e;
        e = launch_merge<128>(p, batch, stream);
        if (e != cudaSuccess) return e;
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

#if PA_DECODE_TRACE
// Profiling build only: clear the marks / copy them to host memory.
extern "C" __attribute__((visibility("default"))) int pa_trace_decode_reset(void) {
    static unsigned long long zero[pa::kTraceAttend * 4 + pa::kTraceMerge * 2];
    return cudaMemcpyToSymbol(pa::g_trace, zero, sizeof(zero)) == cudaSuccess ? 0 : 1;
}
extern "C" __attribute__((visibility("default"))) int pa_trace_decode_read(void* host, size_t bytes) {
    if (bytes < sizeof(pa::g_trace)) return 1;
    return cudaMemcpyFromSymbol(host, pa::g_trace, sizeof(pa::g_trace)) == cudaSuccess ? 0 : 1;
}
#endif

extern "C" __attribute__((visibility("default"))) pa_status pa_decode_noalloc(
    const pa_geom* geom, const void* q, const void* pool, const int32_t* block_table, int32_t layer,
    int32_t batch, const int32_t* seq_lens, const int32_t* slots, int32_t max_seq_len, float scale,
    void* o, float* lse, int32_t* err_flag, pa_stream_t stream) {
    // the arguments are checked as pa_decode checks them before the scratch
    // lookup (a runtime call), so a bad call returns the same status
    bool no_work = false;
    const pa_status st = pa::decode_args(geom, q, pool, block_table, layer, batch, seq_lens, slots, max_seq_len,
                                         scale, o, err_flag, &no_work);
    if (st != PA_OK || no_work) return st;
    if (pa_decode_workspace_size(geom, batch, max_seq_len) > pa::kStaticScratchBytes)
        return PA_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    if (pa::static_scratch(&scratch) != cudaSuccess) return PA_ERR_CUDA;
    return pa_decode(geom, q, pool, block_table, layer, batch, seq_lens, slots, max_seq_len, scale, o,
                     lse, scratch, pa::kStaticScratchBytes, err_flag, stream);
}


// pages.cu -- page lifetime on the device: a free stack of physical pages,
// allocation for new sequence lengths and release of whole slots, with the
// block table kept resident (no copy of the table from the host).
//
// The pages' program keeps free_blocks on the host: a page is taken with
// pop_back when a logical block's entry is -1 (a prompt's blocks, or a decode
// step whose token starts a new block) and a slot that ends pushes back every
// page it holds, walking layers then logical blocks, resetting the entries to
// -1; the whole table is then copied to the device again (jaehun.me
// tiny-vllm part 6, "물리 블록의 수명: free_blocks 가 관리한다").  Here the
// stack and the table stay on the device and one kernel does each step, in
// the same walking order (sequences, then layers, then logical blocks), so
// the result is the pages' result exactly.
//
// One CTA of 1024 threads per call, one warp per (sequence, layer) item, its
// lanes over consecutive logical blocks (8 x 32 entries loaded at a time): the items' pages are counted, an
// exclusive scan over the warps gives each item its place on the stack, and
// the item's warp moves its pages in order (ballot and population count).
// An allocation that gives old_lens (a decode step: a block or two per item)
// takes one thread per item instead, 1024 items per round.  A first counting pass checks the stack
// height, so a call that would run short (or overflow on release) changes
// nothing and reports through err_flag.
#include "pa_internal.cuh"

namespace pa {
namespace {

constexpr int kThreads = 1024;
// One bit per slot a call names, so that a slot named twice is refused; the
// C ABI refuses geometries with more slots than the bitmap covers.
constexpr int kSlotBitmapWords = PA_PAGES_MAX_SLOTS / 32;
static_assert(kSlotBitmapWords * 32 == PA_PAGES_MAX_SLOTS, "one bit per slot");

// Marks slot (already checked to lie in [0, num_slots)) as seen; returns true
// if it already was.
__device__ __forceinline__ bool seen_before(uint32_t* bitmap, int slot) {
    const uint32_t bit = 1u << (slot & 31);
    return (atomicOr(&bitmap[slot >> 5], bit) & bit) != 0;
}

__device__ __forceinline__ void clear_bitmap(uint32_t* bitmap) {
    for (int w = threadIdx.x; w < kSlotBitmapWords; w += kThreads) bitmap[w] = 0u;
}

constexpr int kWarps = kThreads / 32;

// Exclusive scan over the CTA's warps of one value per warp (every lane of a
// warp passes the same v); *total receives the sum.
__device__ __forceinline__ long long warps_exclusive_scan(long long v, long long* total) {
    __shared__ long long sums[kWarps];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) sums[warp] = v;
    __syncthreads();
    if (warp == 0) {
        long long w = sums[lane];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const long long y = __shfl_up_sync(0xffffffffu, w, off);
            if (lane >= off) w += y;
        }
        sums[lane] = w;  // inclusive
    }
    __syncthreads();
    const long long before = warp == 0 ? 0 : sums[warp - 1];
    *total = sums[kWarps - 1];
    __syncthreads();  // sums is reused by the next call
    return before;
}

// A warp walks a table row kUnroll x 32 entries at a time: all the loads of a
// stretch are issued before any of them is used, so a long row costs a few
// memory latencies rather than one per 32 entries.
constexpr int kUnroll = 8;

// One warp walks the logical blocks [lo, hi) of a table row in order; `take`
// says whether an entry moves.  Returns the number that do.
template <typename Take>
__device__ __forceinline__ int warp_count(const int32_t* row, int lo, int hi, Take take) {
    const int lane = threadIdx.x & 31;
    int n = 0;
    for (int s0 = lo; s0 < hi; s0 += 32 * kUnroll) {
        int32_t v[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int lb = s0 + 32 * u + lane;
            v[u] = lb < hi ? row[lb] : 0;
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
            n += __popc(__ballot_sync(0xffffffffu, s0 + 32 * u + lane < hi && take(v[u])));
    }
    return n;
}

struct RowRange {
    int32_t* row;
    int lo, hi;
};

// The table row of item k = (sequence b, layer) of an allocation and the
// blocks it looks at; row is null for an invalid slot or length.
__device__ __forceinline__ RowRange alloc_row(const KGeom& g, int32_t* table, const int32_t* slots,
                                              const int32_t* old_lens, const int32_t* seq_lens, long long k) {
    RowRange it;
    const int b = static_cast<int>(k / g.n_layers), layer = static_cast<int>(k % g.n_layers);
    const int slot = slots[b], len = seq_lens[b];
    const bool ok = slot >= 0 && slot < g.num_slots && len >= 0 && len <= g.maxb * kBlockTokens;
    const int lo = old_lens ? old_lens[b] / kBlockTokens : 0;
    it.lo = lo < 0 ? 0 : lo;
    it.hi = (len + kBlockTokens - 1) / kBlockTokens;
    it.row = ok ? table + (static_cast<long long>(slot) * g.n_layers + layer) * g.maxb : nullptr;
    return it;
}

__global__ void __launch_bounds__(kThreads) alloc_pages_kernel(KGeom g, int32_t* table, int batch,
                                                               const int32_t* slots, const int32_t* old_lens,
                                                               const int32_t* seq_lens, int32_t* free_pages,
                                                               int32_t* free_count, int32_t* err) {
    __shared__ int s_bad;
    __shared__ uint32_t s_seen[kSlotBitmapWords];
    if (threadIdx.x == 0) s_bad = 0;
    clear_bitmap(s_seen);
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const long long items = static_cast<long long>(batch) * g.n_layers;
    auto free_entry = [](int32_t e) { return e == -1; };
    // pass 1: count (and validate); item k goes to warp k % kWarps of chunk k / kWarps
    long long need = 0;
    for (long long c0 = 0; c0 < items; c0 += kWarps) {
        const long long k = c0 + warp;
        int cnt = 0;
        if (k < items) {
            const RowRange it = alloc_row(g, table, slots, old_lens, seq_lens, k);
            if (!it.row) {
                if (lane == 0) s_bad = 1;
            } else {
                if (lane == 0 && k % g.n_layers == 0 && seen_before(s_seen, slots[k / g.n_layers])) s_bad = 1;
                cnt = warp_count(it.row, it.lo, it.hi, free_entry);
            }
        }
        long long total;
        warps_exclusive_scan(cnt, &total);
        need += total;
    }
    __syncthreads();
    const int top = *free_count;
    if (s_bad || need > top || top > g.nblocks) {
        if (threadIdx.x == 0) set_error(err, s_bad ? PA_ERR_BAD_BLOCK : PA_ERR_OUT_OF_PAGES);
        return;
    }
    // pass 2: the r-th page the walk needs is the one r places below the top
    long long base = 0;
    for (long long c0 = 0; c0 < items; c0 += kWarps) {
        const long long k = c0 + warp;
        RowRange it;
        it.row = nullptr;
        int cnt = 0;
        if (k < items) {
            it = alloc_row(g, table, slots, old_lens, seq_lens, k);
            cnt = warp_count(it.row, it.lo, it.hi, free_entry);
        }
        long long total;
        long long r = base + warps_exclusive_scan(cnt, &total);
        if (it.row) {
            for (int s0 = it.lo; s0 < it.hi; s0 += 32 * kUnroll) {
                int32_t v[kUnroll];
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    const int lb = s0 + 32 * u + lane;
                    v[u] = lb < it.hi ? it.row[lb] : 0;
                }
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    const int lb = s0 + 32 * u + lane;
                    const bool take = lb < it.hi && v[u] == -1;
                    const uint32_t m = __ballot_sync(0xffffffffu, take);
                    if (take) it.row[lb] = free_pages[top - 1 - (r + __popc(m & ((1u << lane) - 1u)))];
                    r += __popc(m);
                }
            }
        }
        base += total;
    }
    if (threadIdx.x == 0) *free_count = static_cast<int32_t>(top - need);
}

// Exclusive scan of v over the CTA's threads; *total receives the sum.
__device__ __forceinline__ long long threads_exclusive_scan(int v, long long* total) {
    __shared__ int wsum[kWarps];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off) x += y;
    }
    if (lane == 31) wsum[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = wsum[lane];
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, w, off);
            if (lane >= off) w += y;
        }
        wsum[lane] = w;  // inclusive
    }
    __syncthreads();
    const long long before = (warp == 0 ? 0 : wsum[warp - 1]) + x - v;
    *total = wsum[kWarps - 1];
    __syncthreads();  // wsum is reused by the next call
    return before;
}

// The same allocation with one thread per item (1024 items per round): for
// calls that give old_lens, where each item looks at a block or two (a decode
// step), so rounds, not rows, are what costs.
__global__ void __launch_bounds__(kThreads) alloc_pages_short_kernel(KGeom g, int32_t* table, int batch,
                                                                     const int32_t* slots, const int32_t* old_lens,
                                                                     const int32_t* seq_lens, int32_t* free_pages,
                                                                     int32_t* free_count, int32_t* err) {
    __shared__ int s_bad;
    __shared__ uint32_t s_seen[kSlotBitmapWords];
    if (threadIdx.x == 0) s_bad = 0;
    clear_bitmap(s_seen);
    __syncthreads();
    const long long items = static_cast<long long>(batch) * g.n_layers;
    long long need = 0;
    for (long long c0 = 0; c0 < items; c0 += kThreads) {
        const long long k = c0 + threadIdx.x;
        int cnt = 0;
        if (k < items) {
            const RowRange it = alloc_row(g, table, slots, old_lens, seq_lens, k);
            if (!it.row || (k % g.n_layers == 0 && seen_before(s_seen, slots[k / g.n_layers]))) {
                s_bad = 1;
            } else {
                for (int lb = it.lo; lb < it.hi; ++lb) cnt += it.row[lb] == -1;
            }
        }
        long long total;
        threads_exclusive_scan(cnt, &total);
        need += total;
    }
    __syncthreads();
    const int top = *free_count;
    if (s_bad || need > top || top > g.nblocks) {
        if (threadIdx.x == 0) set_error(err, s_bad ? PA_ERR_BAD_BLOCK : PA_ERR_OUT_OF_PAGES);
        return;
    }
    long long base = 0;
    for (long long c0 = 0; c0 < items; c0 += kThreads) {
        const long long k = c0 + threadIdx.x;
        RowRange it;
        it.row = nullptr;
        int cnt = 0;
        if (k < items) {
            it = alloc_row(g, table, slots, old_lens, seq_lens, k);
            for (int lb = it.lo; lb < it.hi; ++lb) cnt += it.row[lb] == -1;
        }
        long long total;
        long long r = base + threads_exclusive_scan(cnt, &total);
        if (it.row)
            for (int lb = it.lo; lb < it.hi; ++lb)
                if (it.row[lb] == -1) it.row[lb] = free_pages[top - 1 - r++];
        base += total;
    }
    if (threadIdx.x == 0) *free_count = static_cast<int32_t>(top - need);
}

__global__ void __launch_bounds__(kThreads) release_slots_kernel(KGeom g, int32_t* table, int n,
                                                                 const int32_t* slots, int32_t* free_pages,
                                                                 int32_t* free_count, int32_t* err) {
    __shared__ int s_bad;
    __shared__ uint32_t s_seen[kSlotBitmapWords];
    if (threadIdx.x == 0) s_bad = 0;
    clear_bitmap(s_seen);
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const long long items = static_cast<long long>(n) * g.n_layers;
    auto row_of = [&](long long k) -> int32_t* {
        const int i = static_cast<int>(k / g.n_layers), layer = static_cast<int>(k % g.n_layers);
        const int slot = slots[i];
        if (slot < 0 || slot >= g.num_slots) return nullptr;
        return table + (static_cast<long long>(slot) * g.n_layers + layer) * g.maxb;
    };
    auto held_entry = [](int32_t e) { return e != -1; };
    long long held = 0;
    for (long long c0 = 0; c0 < items; c0 += kWarps) {
        const long long k = c0 + warp;
        int cnt = 0;
        if (k < items) {
            int32_t* row = row_of(k);
            if (!row) {
                if (lane == 0) s_bad = 1;
            } else {
                if (lane == 0 && k % g.n_layers == 0 && seen_before(s_seen, slots[k / g.n_layers])) s_bad = 1;
                cnt = warp_count(row, 0, g.maxb, held_entry);
            }
        }
        long long total;
        warps_exclusive_scan(cnt, &total);
        held += total;
    }
    __syncthreads();
    const int top = *free_count;
    if (s_bad || top < 0 || top + held > g.nblocks) {
        if (threadIdx.x == 0) set_error(err, s_bad ? PA_ERR_BAD_BLOCK : PA_ERR_OUT_OF_PAGES);
        return;
    }
    long long base = 0;
    for (long long c0 = 0; c0 < items; c0 += kWarps) {
        const long long k = c0 + warp;
        int32_t* row = nullptr;
        int cnt = 0;
        if (k < items) {
            row = row_of(k);
            cnt = warp_count(row, 0, g.maxb, held_entry);
        }
        long long total;
        long long r = base + warps_exclusive_scan(cnt, &total);
        if (row) {
            for (int s0 = 0; s0 < g.maxb; s0 += 32 * kUnroll) {
                int32_t v[kUnroll];
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    const int lb = s0 + 32 * u + lane;
                    v[u] = lb < g.maxb ? row[lb] : -1;
                }
#pragma unroll
                for (int u = 0; u < kUnroll; ++u) {
                    const int lb = s0 + 32 * u + lane;
                    const bool give = v[u] != -1;
                    const uint32_t m = __ballot_sync(0xffffffffu, give);
                    if (give) {
                        free_pages[top + r + __popc(m & ((1u << lane) - 1u))] = v[u];
                        row[lb] = -1;
                    }
                    r += __popc(m);
                }
            }
        }
        base += total;
    }
    if (threadIdx.x == 0) *free_count = static_cast<int32_t>(top + held);
}

}  // namespace

cudaError_t launch_alloc_pages(const KGeom& g, int32_t* table, int batch, const int32_t* slots,
                               const int32_t* old_lens, const int32_t* seq_lens, int32_t* free_pages,
                               int32_t* free_count, int32_t* err, cudaStream_t stream) {
    // same result either way; the layout only decides how fast the rows are walked
    if (old_lens)
        alloc_pages_short_kernel<<<1, kThreads, 0, stream>>>(g, table, batch, slots, old_lens, seq_lens, free_pages,
                                                             free_count, err);
    else
        alloc_pages_kernel<<<1, kThreads, 0, stream>>>(g, table, batch, slots, old_lens, seq_lens, free_pages,
                                                       free_count, err);
    return cudaGetLastError();
}

cudaError_t launch_release_slots(const KGeom& g, int32_t* table, int n, const int32_t* slots, int32_t* free_pages,
                                 int32_t* free_count, int32_t* err, cudaStream_t stream) {
    release_slots_kernel<<<1, kThreads, 0, stream>>>(g, table, n, slots, free_pages, free_count, err);
    return cudaGetLastError();
}

}  // namespace pa

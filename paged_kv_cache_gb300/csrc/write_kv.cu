// write_kv.cu -- scatter of new K/V rows into their pages.
//
// The pages write a new token's K at
//   kv_cache + block * BLOCK_BYTES + token_in_block * KV_DIM * 2
// and its V at the same address + V_OFFSET, the block coming from
// block_table[slot][layer][pos / 16] (jaehun.me tiny-vllm part 6, "블록 하나가
// 담는 것: K 는 앞, V 는 V_OFFSET 뒤"; part 3, "Distributing K/V into paged
// blocks").  The series issues one device-to-device memcpy per page per layer;
// here one launch moves every row of the call: each thread moves 8 chunks of 16
// bytes of one row (4 or 1 when the row's chunk count does not divide), a
// row's threads taking consecutive chunks in each pass, so that every load and
// store instruction of a warp covers whole contiguous runs of k_new/v_new and
// of the page row.
#include "pa_internal.cuh"

namespace pa {
namespace {

// CPT 16-byte chunks of one K or V row per thread, a row's chunks/CPT threads
// apart (CPT divides the row's chunk count).  The row's data is read before its page is looked up,
// so the two global latencies overlap instead of adding up.
// V_ONLY: the V rows alone, for the RoPE scatter, which turns K in a kernel of
// its own (rows at a position >= max_pos are skipped there too); this launch
// lets that one start at once (it reads nothing this one writes).
template <int CPT, bool V_ONLY>
__global__ void __launch_bounds__(256) write_kv_kernel(KGeom g, uint8_t* __restrict__ pool,
                                                       const int32_t* __restrict__ block_table,
                                                       int layer, int n_tokens,
                                                       const int32_t* __restrict__ tok_slot,
                                                       const int32_t* __restrict__ tok_pos,
                                                       const uint4* __restrict__ k_new,
                                                       const uint4* __restrict__ v_new,
                                                       int max_pos, int32_t* err) {
    if (V_ONLY) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int chunks = g.kv_dim / 8;  // 16-byte chunks per K (or V) row
    const int groups = chunks / CPT;  // threads per K (or V) row
    const int per_row = V_ONLY ? groups : 2 * groups;
    const long long total = static_cast<long long>(n_tokens) * per_row;
    const long long half_page = g.page_bytes / 2;  // V_OFFSET
    const long long row_bytes = static_cast<long long>(g.kv_dim) * 2;
    for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long row = idx / per_row;
        const int rem = static_cast<int>(idx - row * per_row);
        const int is_v = V_ONLY || rem >= groups;
        const int c = V_ONLY ? rem : is_v ? rem - groups : rem;  // chunks c, c + groups, c + 2 groups, ...
        const uint4* src = (is_v ? v_new : k_new) + row * chunks + c;
        uint4 val[CPT];
#pragma unroll
        for (int x = 0; x < CPT; ++x)
            asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                         : "=r"(val[x].x), "=r"(val[x].y), "=r"(val[x].z), "=r"(val[x].w)
                         : "l"(src + x * groups));
        const int slot = __ldg(tok_slot + row);
        const int pos = __ldg(tok_pos + row);
        long long blk = -1;
        if (slot >= 0 && slot < g.num_slots && pos >= 0 && pos / kBlockTokens < g.maxb && (!V_ONLY || pos < max_pos)) {
            const long long tidx =
                (static_cast<long long>(slot) * g.n_layers + layer) * g.maxb + pos / kBlockTokens;
            const int e = __ldg(block_table + tidx);
            if (e >= 0 && e < g.nblocks) blk = e;
        }
        if (blk < 0) {
            if (rem == 0) set_error(err, PA_ERR_BAD_BLOCK);
            continue;
        }
        uint4* dst = reinterpret_cast<uint4*>(pool + blk * g.page_bytes + (is_v ? half_page : 0) +
                                              static_cast<long long>(pos % kBlockTokens) * row_bytes) + c;
#pragma unroll
        for (int x = 0; x < CPT; ++x) dst[x * groups] = val[x];
    }
}

// Streaming 16-byte load (read once: not kept in L1).
__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// The same scatter with K rotated by RoPE on the way (jaehun.me tiny-vllm part
// 3, "RoPE: a rotation that references a table"): in each kv head, element i
// and element i + d/2 form a pair turned by the angle of the row's position,
//   x1' = x1 c - x2 s,   x2' = x1 s + x2 c,
// with c, s from caller tables [max_pos][d/2] fp32.  Each product and sum is
// rounded on its own (no FMA contraction), then to bf16 nearest-even (rope8).
// Threads work on groups of kRopeRows rows: the group's K threads first (8
// pairs, 16 bytes of each half, in each of KPT heads Hkv/KPT apart, which
// share one angle row), then its V threads (VPT 16-byte chunks each, a row's
// V threads taking consecutive chunks in each pass), so that a warp runs
// either the rotation or the copy.
// Every thread reads its row's data, then the position, then the page entry
// and (K) the angle rows together, so that the latencies overlap.

constexpr int kRopeRows = 8;  // rows per thread group of the RoPE scatter

template <int KPT, int VPT, bool K_ONLY>
__global__ void __launch_bounds__(256) write_kv_rope_kernel(KGeom g, uint8_t* __restrict__ pool,
                                                            const int32_t* __restrict__ block_table, int layer,
                                                            int n_tokens, const int32_t* __restrict__ tok_slot,
                                                            const int32_t* __restrict__ tok_pos,
                                                            const uint4* __restrict__ k_new,
                                                            const uint4* __restrict__ v_new,
                                                            const float* __restrict__ cos_tab,
                                                            const float* __restrict__ sin_tab, int max_pos,
                                                            int32_t* err) {
    const int hc = g.d / 16;            // pair chunks per head (8 pairs each)
    const int kt = g.hkv / KPT * hc;    // K threads per row
    const int vc = g.kv_dim / 8;        // 16-byte V chunks per row
    const int vt = vc / VPT;            // V threads per row
    const int k_threads = kRopeRows * kt;
    const int per_group = k_threads + (K_ONLY ? 0 : kRopeRows * vt);
    const long long total = static_cast<long long>((n_tokens + kRopeRows - 1) / kRopeRows) * per_group;
    const long long half_page = g.page_bytes / 2;  // V_OFFSET
    const long long row_bytes = static_cast<long long>(g.kv_dim) * 2;
    for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long grp = idx / per_group;
        const int rem = static_cast<int>(idx - grp * per_group);
        const bool is_k = K_ONLY || rem < k_threads;
        const int local = is_k ? rem / kt : (rem - k_threads) / vt;
        const int c = is_k ? rem % kt : (rem - k_threads) % vt;  // K: (first head, pair chunk); V: first chunk
        const int c8 = 8 * (c % hc);                             // K: first pair element within the head
        const long long row = grp * kRopeRows + local;
        if (row >= n_tokens) continue;
        // the row's data first: its latency overlaps the lookups
        uint4 lo[KPT], hi[KPT], vv[VPT];
        if (is_k) {
#pragma unroll
            for (int x = 0; x < KPT; ++x) {
                const long long e_lo = static_cast<long long>(c / hc + x * (g.hkv / KPT)) * g.d + c8;
                lo[x] = ld_stream(k_new + (row * g.kv_dim + e_lo) / 8);
                hi[x] = ld_stream(k_new + (row * g.kv_dim + e_lo + g.d / 2) / 8);
            }
        } else {
#pragma unroll
            for (int x = 0; x < VPT; ++x) vv[x] = ld_stream(v_new + row * vc + c + x * vt);
        }
        const int slot = __ldg(tok_slot + row);
        const int pos = __ldg(tok_pos + row);
        const bool pos_ok = pos >= 0 && pos < max_pos && pos / kBlockTokens < g.maxb;
        // the angle row is read beside the page entry, not after it
        float4 cs[4];
        if (is_k && pos_ok) {
            const long long a = static_cast<long long>(pos) * (g.d / 2) + c8;
            const float4* ct = reinterpret_cast<const float4*>(cos_tab + a);
            const float4* st = reinterpret_cast<const float4*>(sin_tab + a);
            cs[0] = __ldg(ct);
            cs[1] = __ldg(ct + 1);
            cs[2] = __ldg(st);
            cs[3] = __ldg(st + 1);
        }
        long long blk = -1;
        if (slot >= 0 && slot < g.num_slots && pos_ok) {
            const long long tidx =
                (static_cast<long long>(slot) * g.n_layers + layer) * g.maxb + pos / kBlockTokens;
            const int e = __ldg(block_table + tidx);
            if (e >= 0 && e < g.nblocks) blk = e;
        }
        if (blk < 0) {
            if (rem == local * kt) set_error(err, PA_ERR_BAD_BLOCK);  // the row's first K thread
            continue;
        }
        uint8_t* dst_row = pool + blk * g.page_bytes + static_cast<long long>(pos % kBlockTokens) * row_bytes;
        if (is_k) {
#pragma unroll
            for (int x = 0; x < KPT; ++x) {
                const long long e_lo = static_cast<long long>(c / hc + x * (g.hkv / KPT)) * g.d + c8;
                rope8(lo[x], hi[x], cs[0], cs[1], cs[2], cs[3]);
                *reinterpret_cast<uint4*>(dst_row + e_lo * 2) = lo[x];
                *reinterpret_cast<uint4*>(dst_row + (e_lo + g.d / 2) * 2) = hi[x];
            }
        } else {
            uint4* dv = reinterpret_cast<uint4*>(dst_row + half_page) + c;
#pragma unroll
            for (int x = 0; x < VPT; ++x) dv[x * vt] = vv[x];
        }
    }
    // K_ONLY runs as a programmatic dependent of the V copy: it leaves only once
    // that launch is complete, so the call is, in stream order, when this is.
    if (K_ONLY) asm volatile("griddepcontrol.wait;" ::: "memory");
}

}  // namespace

cudaError_t launch_write_kv_rope(const KGeom& g, void* pool, const int32_t* block_table, int layer,
                                 int n_tokens, const int32_t* tok_slot, const int32_t* tok_pos,
                                 const void* k_new, const void* v_new, const float* cos_tab,
                                 const float* sin_tab, int max_pos, int32_t* err, cudaStream_t stream) {
    // V rows by the plain scatter (few registers, many bytes in flight), then
    // K turned by the RoPE kernel in a launch that runs beside it; KPT heads'
    // pairs per thread, KPT dividing the kv head count
    const int threads = 256;
    {
        const int chunks = g.kv_dim / 8;
        const int cpt = chunks % 8 == 0 ? 8 : chunks % 4 == 0 ? 4 : 1;
        const long long total = static_cast<long long>(n_tokens) * (chunks / cpt);
        long long blocks = (total + threads - 1) / threads;
        if (blocks > (1ll << 30)) blocks = 1ll << 30;  // grid-stride covers the rest
        auto kern = cpt == 8 ? write_kv_kernel<8, true> : cpt == 4 ? write_kv_kernel<4, true> : write_kv_kernel<1, true>;
        kern<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
            g, static_cast<uint8_t*>(pool), block_table, layer, n_tokens, tok_slot, tok_pos,
            static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), max_pos, err);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    const int kpt = g.hkv % 4 == 0 ? 4 : g.hkv % 2 == 0 ? 2 : 1;
    const int hc = g.d / 16;
    const int per_group = kRopeRows * (g.hkv / kpt * hc);
    const long long total = static_cast<long long>((n_tokens + kRopeRows - 1) / kRopeRows) * per_group;
    long long blocks = (total + threads - 1) / threads;
    if (blocks > (1ll << 30)) blocks = 1ll << 30;
    auto kern = kpt == 4 ? write_kv_rope_kernel<4, 8, true>
                         : kpt == 2 ? write_kv_rope_kernel<2, 4, true> : write_kv_rope_kernel<1, 2, true>;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
    cfg.blockDim = dim3(threads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, g, static_cast<uint8_t*>(pool), block_table, layer, n_tokens, tok_slot,
                              tok_pos, static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), cos_tab,
                              sin_tab, max_pos, err);
}

cudaError_t launch_write_kv(const KGeom& g, void* pool, const int32_t* block_table, int layer,
                            int n_tokens, const int32_t* tok_slot, const int32_t* tok_pos,
                            const void* k_new, const void* v_new, int32_t* err,
                            cudaStream_t stream) {
    const int chunks = g.kv_dim / 8;
    const int cpt = chunks % 8 == 0 ? 8 : chunks % 4 == 0 ? 4 : 1;
    const long long total = static_cast<long long>(n_tokens) * 2 * (chunks / cpt);
    const int threads = 256;
    long long blocks = (total + threads - 1) / threads;
    if (blocks > (1ll << 30)) blocks = 1ll << 30;  // grid-stride covers the rest
    if (cpt == 8)
        write_kv_kernel<8, false><<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
            g, static_cast<uint8_t*>(pool), block_table, layer, n_tokens, tok_slot, tok_pos,
            static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), 0, err);
    else if (cpt == 4)
        write_kv_kernel<4, false><<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
            g, static_cast<uint8_t*>(pool), block_table, layer, n_tokens, tok_slot, tok_pos,
            static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), 0, err);
    else
        write_kv_kernel<1, false><<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
            g, static_cast<uint8_t*>(pool), block_table, layer, n_tokens, tok_slot, tok_pos,
            static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), 0, err);
    return cudaGetLastError();
}

}  // namespace pa

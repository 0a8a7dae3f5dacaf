// write_kv.cu -- scatter of new K/V rows into their pages.
//
// The pages write a new token's K at
//   kv_cache + block * BLOCK_BYTES + token_in_block * KV_DIM * 2
// and its V at the same address + V_OFFSET, the block coming from
// block_table[slot][layer][pos / 16] (jaehun.me tiny-vllm part 6, "블록 하나가
// 담는 것: K 는 앞, V 는 V_OFFSET 뒤"; part 3, "Distributing K/V into paged
// blocks").  The series issues one device-to-device memcpy per page per layer;
// here one launch moves every row of the call: one thread per 16-byte chunk,
// consecutive threads on consecutive chunks of a row, so reads of k_new/v_new
// and writes of each 2*KV_DIM-byte row are fully coalesced 16-byte accesses.
#include "pa_internal.cuh"

namespace pa {
namespace {

__global__ void __launch_bounds__(256) write_kv_kernel(KGeom g, uint8_t* __restrict__ pool,
                                                       const int32_t* __restrict__ block_table,
                                                       int layer, int n_tokens,
                                                       const int32_t* __restrict__ tok_slot,
                                                       const int32_t* __restrict__ tok_pos,
                                                       const uint4* __restrict__ k_new,
                                                       const uint4* __restrict__ v_new,
                                                       int32_t* err) {
    const int chunks = g.kv_dim / 8;  // 16-byte chunks per K (or V) row
    const long long total = static_cast<long long>(n_tokens) * 2 * chunks;
    const long long half_page = g.page_bytes / 2;  // V_OFFSET
    const long long row_bytes = static_cast<long long>(g.kv_dim) * 2;
    for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long row = idx / (2 * chunks);
        const int rem = static_cast<int>(idx - row * 2 * chunks);
        const int is_v = rem >= chunks;
        const int c = is_v ? rem - chunks : rem;
        const int slot = __ldg(tok_slot + row);
        const int pos = __ldg(tok_pos + row);
        long long blk = -1;
        if (slot >= 0 && slot < g.num_slots && pos >= 0 && pos / kBlockTokens < g.maxb) {
            const long long tidx =
                (static_cast<long long>(slot) * g.n_layers + layer) * g.maxb + pos / kBlockTokens;
            const int e = __ldg(block_table + tidx);
            if (e >= 0 && e < g.nblocks) blk = e;
        }
        if (blk < 0) {
            if (rem == 0) set_error(err, PA_ERR_BAD_BLOCK);
            continue;
        }
        const uint4* src = (is_v ? v_new : k_new) + row * chunks + c;
        uint4 val;
        asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                     : "=r"(val.x), "=r"(val.y), "=r"(val.z), "=r"(val.w)
                     : "l"(src));
        uint8_t* dst = pool + blk * g.page_bytes + (is_v ? half_page : 0) +
                       static_cast<long long>(pos % kBlockTokens) * row_bytes +
                       static_cast<long long>(c) * 16;
        *reinterpret_cast<uint4*>(dst) = val;
    }
}

}  // namespace

cudaError_t launch_write_kv(const KGeom& g, void* pool, const int32_t* block_table, int layer,
                            int n_tokens, const int32_t* tok_slot, const int32_t* tok_pos,
                            const void* k_new, const void* v_new, int32_t* err,
                            cudaStream_t stream) {
    const long long total = static_cast<long long>(n_tokens) * 2 * (g.kv_dim / 8);
    const int threads = 256;
    long long blocks = (total + threads - 1) / threads;
    if (blocks > (1ll << 30)) blocks = 1ll << 30;  // grid-stride covers the rest
    write_kv_kernel<<<static_cast<unsigned>(blocks), threads, 0, stream>>>(
        g, static_cast<uint8_t*>(pool), block_table, layer, n_tokens, tok_slot, tok_pos,
        static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), err);
    return cudaGetLastError();
}

}  // namespace pa

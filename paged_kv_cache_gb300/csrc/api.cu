// api.cu -- the C ABI of libpa.so (declared in include/pa.h): argument
// validation, then one asynchronous launch sequence per call.  No memory is
// allocated and no state is kept between calls.
#include <atomic>
#include <cmath>
#include <cstdint>

#include "pa_internal.cuh"

#define PA_API extern "C" __attribute__((visibility("default")))

namespace pa {
namespace {
std::atomic<int> g_hold_first_copy{0};
}
int debug_hold_first_copy() { return g_hold_first_copy.load(std::memory_order_relaxed); }

EncodeTiledFn tensor_map_encoder() {
    // looked up once, by the first call from any thread (a function-local
    // static is initialised exactly once, so concurrent first calls do not race)
    static const EncodeTiledFn fn = [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<EncodeTiledFn>(ptr);
        return static_cast<EncodeTiledFn>(nullptr);
    }();
    return fn;
}
}  // namespace pa

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Geometry fields that every call needs.
bool geom_valid(const pa_geom* g) {
    if (!g) return false;
    if (g->num_q_heads <= 0 || g->num_kv_heads <= 0 || g->head_dim <= 0) return false;
    if (g->num_q_heads % g->num_kv_heads != 0) return false;
    if (g->head_dim % 8 != 0) return false;  // rows move in 16-byte chunks
    if (g->n_layers <= 0 || g->num_slots <= 0 || g->max_blocks_per_seq <= 0) return false;
    if (g->num_blocks <= 0) return false;
    const long long kv_dim = static_cast<long long>(g->num_kv_heads) * g->head_dim;
    if (kv_dim > (1 << 20)) return false;
    return true;
}

pa::KGeom kgeom(const pa_geom* g) {
    pa::KGeom k;
    k.hq = g->num_q_heads;
    k.hkv = g->num_kv_heads;
    k.d = g->head_dim;
    k.group = g->num_q_heads / g->num_kv_heads;
    k.n_layers = g->n_layers;
    k.num_slots = g->num_slots;
    k.maxb = g->max_blocks_per_seq;
    k.kv_dim = g->num_kv_heads * g->head_dim;
    k.nblocks = g->num_blocks;
    k.page_bytes = 64ll * k.kv_dim;
    return k;
}

bool ranges_overlap(const void* a, size_t a_len, const void* b, size_t b_len) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
    return a0 < b0 + b_len && b0 < a0 + a_len;
}

pa_status cuda_status(cudaError_t e) { return e == cudaSuccess ? PA_OK : PA_ERR_CUDA; }

}  // namespace

PA_API size_t pa_page_bytes(const pa_geom* geom) {
    if (!geom_valid(geom)) return 0;
    return static_cast<size_t>(kgeom(geom).page_bytes);
}

PA_API pa_status pa_write_kv(const pa_geom* geom, void* pool, const int32_t* block_table,
                             int32_t layer, int32_t n_tokens, const int32_t* tok_slot,
                             const int32_t* tok_pos, const void* k_new, const void* v_new,
                             int32_t* err_flag, pa_stream_t stream) {
    if (!geom_valid(geom)) return PA_ERR_INVALID_ARG;
    if (layer < 0 || layer >= geom->n_layers || n_tokens < 0) return PA_ERR_INVALID_ARG;
    if (n_tokens == 0) return PA_OK;
    if (!pool || !block_table || !tok_slot || !tok_pos || !k_new || !v_new || !err_flag)
        return PA_ERR_INVALID_ARG;
    if (!aligned16(pool) || !aligned16(k_new) || !aligned16(v_new)) return PA_ERR_INVALID_ARG;
    const pa::KGeom g = kgeom(geom);
    const size_t pool_len = static_cast<size_t>(g.nblocks) * static_cast<size_t>(g.page_bytes);
    const size_t rows_len = static_cast<size_t>(n_tokens) * g.kv_dim * 2;
    if (ranges_overlap(k_new, rows_len, pool, pool_len) ||
        ranges_overlap(v_new, rows_len, pool, pool_len))
        return PA_ERR_INVALID_ARG;
    return cuda_status(pa::launch_write_kv(g, pool, block_table, layer, n_tokens, tok_slot,
                                           tok_pos, k_new, v_new, err_flag,
                                           reinterpret_cast<cudaStream_t>(stream)));
}


PA_API pa_status pa_write_kv_rope(const pa_geom* geom, void* pool, const int32_t* block_table,
                                  int32_t layer, int32_t n_tokens, const int32_t* tok_slot,
                                  const int32_t* tok_pos, const void* k_new, const void* v_new,
                                  const float* cos_table, const float* sin_table, int32_t max_pos,
                                  int32_t* err_flag, pa_stream_t stream) {
    if (!geom_valid(geom)) return PA_ERR_INVALID_ARG;
    if (layer < 0 || layer >= geom->n_layers || n_tokens < 0 || max_pos < 0) return PA_ERR_INVALID_ARG;
    if (geom->head_dim % 16 != 0) return PA_ERR_UNSUPPORTED;
    if (n_tokens == 0) return PA_OK;
    if (!pool || !block_table || !tok_slot || !tok_pos || !k_new || !v_new || !cos_table || !sin_table ||
        !err_flag)
        return PA_ERR_INVALID_ARG;
    if (!aligned16(pool) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(cos_table) ||
        !aligned16(sin_table))
        return PA_ERR_INVALID_ARG;
    const pa::KGeom g = kgeom(geom);
    const size_t pool_len = static_cast<size_t>(g.nblocks) * static_cast<size_t>(g.page_bytes);
    const size_t rows_len = static_cast<size_t>(n_tokens) * g.kv_dim * 2;
    if (ranges_overlap(k_new, rows_len, pool, pool_len) ||
        ranges_overlap(v_new, rows_len, pool, pool_len))
        return PA_ERR_INVALID_ARG;
    return cuda_status(pa::launch_write_kv_rope(g, pool, block_table, layer, n_tokens, tok_slot, tok_pos,
                                                k_new, v_new, cos_table, sin_table, max_pos, err_flag,
                                                reinterpret_cast<cudaStream_t>(stream)));
}

namespace {
// The checks of pa_prefill_cached (shared with pa_prefill_rope); *no_work is
// set when the call has nothing to enqueue and the status is PA_OK.
pa_status prefill_args(const pa_geom* geom, const void* q, const void* pool, const int32_t* block_table,
                       int32_t layer, int32_t batch, const int32_t* cu_seqlens, const int32_t* slots,
                       int32_t max_seqlen, int32_t total_tokens, float scale, const void* o,
                       const int32_t* err_flag, bool* no_work) {
    *no_work = false;
    if (!geom_valid(geom)) return PA_ERR_INVALID_ARG;
    if (layer < 0 || layer >= geom->n_layers) return PA_ERR_INVALID_ARG;
    if (batch < 0 || max_seqlen < 0 || total_tokens < 0 || !std::isfinite(scale) || !(scale > 0.f))
        return PA_ERR_INVALID_ARG;
    if (geom->head_dim != 64 && geom->head_dim != 128) return PA_ERR_UNSUPPORTED;
    if (batch == 0 || total_tokens == 0 || max_seqlen == 0) {
        *no_work = true;
        return PA_OK;
    }
    if (!q || !pool || !block_table || !cu_seqlens || !slots || !o || !err_flag)
        return PA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(o) || !aligned16(pool)) return PA_ERR_INVALID_ARG;
    // TMA coordinates are int32: pool rows (32 per page) and q rows must fit.
    if (kgeom(geom).nblocks * 32 >= (1ll << 31)) return PA_ERR_UNSUPPORTED;
    return PA_OK;
}
}  // namespace

PA_API pa_status pa_prefill_cached(const pa_geom* geom, const void* q, const void* pool,
                                   const int32_t* block_table, int32_t layer, int32_t batch,
                                   const int32_t* cu_seqlens, const int32_t* prefix_lens,
                                   const int32_t* slots, int32_t max_seqlen, int32_t total_tokens,
                                   float scale, void* o, float* lse, int32_t* err_flag,
                                   pa_stream_t stream) {
    bool no_work = false;
    const pa_status st = prefill_args(geom, q, pool, block_table, layer, batch, cu_seqlens, slots, max_seqlen,
                                      total_tokens, scale, o, err_flag, &no_work);
    if (st != PA_OK || no_work) return st;
    return cuda_status(pa::launch_prefill(kgeom(geom), q, pool, block_table, layer, batch, cu_seqlens,
                                          prefix_lens, slots, max_seqlen, total_tokens, scale, o,
                                          lse, err_flag, reinterpret_cast<cudaStream_t>(stream)));
}

PA_API pa_status pa_prefill_rope(const pa_geom* geom, const void* q, const void* pool,
                                 const int32_t* block_table, int32_t layer, int32_t batch,
                                 const int32_t* cu_seqlens, const int32_t* prefix_lens,
                                 const int32_t* slots, int32_t max_seqlen, int32_t total_tokens,
                                 float scale, const float* cos_table, const float* sin_table,
                                 int32_t max_pos, void* o, float* lse, int32_t* err_flag,
                                 pa_stream_t stream) {
    if (max_pos < 0) return PA_ERR_INVALID_ARG;
    bool no_work = false;
    const pa_status st = prefill_args(geom, q, pool, block_table, layer, batch, cu_seqlens, slots, max_seqlen,
                                      total_tokens, scale, o, err_flag, &no_work);
    if (st != PA_OK || no_work) return st;
    if (!cos_table || !sin_table || !aligned16(cos_table) || !aligned16(sin_table)) return PA_ERR_INVALID_ARG;
    return cuda_status(pa::launch_prefill(kgeom(geom), q, pool, block_table, layer, batch, cu_seqlens,
                                          prefix_lens, slots, max_seqlen, total_tokens, scale, o, lse, err_flag,
                                          reinterpret_cast<cudaStream_t>(stream), cos_table, sin_table, max_pos));
}

PA_API pa_status pa_prefill(const pa_geom* geom, const void* q, const void* pool,
                            const int32_t* block_table, int32_t layer, int32_t batch,
                            const int32_t* cu_seqlens, const int32_t* slots, int32_t max_seqlen,
                            int32_t total_tokens, float scale, void* o, float* lse,
                            int32_t* err_flag, pa_stream_t stream) {
    return pa_prefill_cached(geom, q, pool, block_table, layer, batch, cu_seqlens, nullptr, slots,
                             max_seqlen, total_tokens, scale, o, lse, err_flag, stream);
}

PA_API pa_status pa_prefill_backward(const pa_geom* geom, const void* q, const void* pool,
                                     const int32_t* block_table, int32_t layer, int32_t batch,
                                     const int32_t* cu_seqlens, const int32_t* slots, int32_t max_seqlen,
                                     int32_t total_tokens, float scale, const void* o, const float* lse,
                                     const void* dout, float* delta, float* dq, float* dk, float* dv,
                                     int32_t* err_flag, pa_stream_t stream) {
    if (!geom_valid(geom)) return PA_ERR_INVALID_ARG;
    if (layer < 0 || layer >= geom->n_layers) return PA_ERR_INVALID_ARG;
    if (batch < 0 || max_seqlen < 0 || total_tokens < 0 || !std::isfinite(scale) || !(scale > 0.f))
        return PA_ERR_INVALID_ARG;
    if (geom->head_dim != 64 && geom->head_dim != 128) return PA_ERR_UNSUPPORTED;
    if (total_tokens == 0) return PA_OK;
    if (!q || !pool || !o || !lse || !dout || !delta || !dq || !dk || !dv || !err_flag)
        return PA_ERR_INVALID_ARG;
    if (batch > 0 && (!block_table || !cu_seqlens || !slots)) return PA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(o) || !aligned16(dout) || !aligned16(dq) || !aligned16(dk) ||
        !aligned16(dv) || !aligned16(pool) || (reinterpret_cast<uintptr_t>(lse) & 3) ||
        (reinterpret_cast<uintptr_t>(delta) & 3))
        return PA_ERR_INVALID_ARG;
    if (max_seqlen > 64 * 65535) return PA_ERR_UNSUPPORTED;
    const pa::KGeom kg = kgeom(geom);
    if (kg.nblocks * 32 >= (1ll << 31)) return PA_ERR_UNSUPPORTED;  // TMA row coordinates are int32
    return cuda_status(pa::launch_prefill_backward(kg, q, pool, block_table, layer, batch, cu_seqlens,
                                                   slots, max_seqlen, total_tokens, scale, o, lse, dout, delta,
                                                   dq, dk, dv, err_flag, reinterpret_cast<cudaStream_t>(stream)));
}

PA_API size_t pa_decode_workspace_size(const pa_geom* geom, int32_t batch, int32_t max_seq_len) {
    if (!geom_valid(geom) || batch < 0 || max_seq_len < 0) return 0;
    return pa::decode_workspace_bytes(kgeom(geom), batch, max_seq_len);
}

namespace pa {
// Every check of pa_decode except those on the workspace, in the same order
// (shared with pa_decode_noalloc); *no_work is set when the call has nothing
// to enqueue (an empty batch) and the status is PA_OK.
pa_status decode_args(const pa_geom* geom, const void* q, const void* pool, const int32_t* block_table,
                      int32_t layer, int32_t batch, const int32_t* seq_lens, const int32_t* slots,
                      int32_t max_seq_len, float scale, const void* o, const int32_t* err_flag, bool* no_work) {
    *no_work = false;
    if (!geom_valid(geom)) return PA_ERR_INVALID_ARG;
    if (layer < 0 || layer >= geom->n_layers) return PA_ERR_INVALID_ARG;
    if (batch < 0 || max_seq_len < 0 || !std::isfinite(scale) || !(scale > 0.f)) return PA_ERR_INVALID_ARG;
    if (!decode_supported(kgeom(geom))) return PA_ERR_UNSUPPORTED;
    if (batch == 0) {
        *no_work = true;
        return PA_OK;
    }
    if (!q || !pool || !block_table || !seq_lens || !slots || !o || !err_flag) return PA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(o) || !aligned16(pool)) return PA_ERR_INVALID_ARG;
    return PA_OK;
}
}  // namespace pa

PA_API pa_status pa_decode(const pa_geom* geom, const void* q, const void* pool,
                           const int32_t* block_table, int32_t layer, int32_t batch,
                           const int32_t* seq_lens, const int32_t* slots, int32_t max_seq_len,
                           float scale, void* o, float* lse, void* workspace,
                           size_t workspace_bytes, int32_t* err_flag, pa_stream_t stream) {
    bool no_work = false;
    const pa_status st = pa::decode_args(geom, q, pool, block_table, layer, batch, seq_lens, slots, max_seq_len,
                                         scale, o, err_flag, &no_work);
    if (st != PA_OK || no_work) return st;
    const pa::KGeom g = kgeom(geom);
    if (!workspace || !aligned16(workspace)) return PA_ERR_INVALID_ARG;
    if (workspace_bytes < pa::decode_workspace_bytes(g, batch, max_seq_len))
        return PA_ERR_INVALID_ARG;
    return cuda_status(pa::launch_decode(g, q, pool, block_table, layer, batch, seq_lens, slots,
                                         max_seq_len, scale, o, lse, workspace, err_flag,
                                         reinterpret_cast<cudaStream_t>(stream)));
}

PA_API pa_status pa_alloc_pages(const pa_geom* geom, int32_t* block_table, int32_t batch,
                                const int32_t* slots, const int32_t* old_lens, const int32_t* seq_lens,
                                int32_t* free_pages, int32_t* free_count, int32_t* err_flag,
                                pa_stream_t stream) {
    if (!geom_valid(geom) || batch < 0) return PA_ERR_INVALID_ARG;
    if (geom->num_slots > PA_PAGES_MAX_SLOTS) return PA_ERR_UNSUPPORTED;
    if (!block_table || !free_pages || !free_count || !err_flag) return PA_ERR_INVALID_ARG;
    if (batch > 0 && (!slots || !seq_lens)) return PA_ERR_INVALID_ARG;
    if (batch == 0) return PA_OK;
    return cuda_status(pa::launch_alloc_pages(kgeom(geom), block_table, batch, slots, old_lens, seq_lens,
                                              free_pages, free_count, err_flag,
                                              reinterpret_cast<cudaStream_t>(stream)));
}

PA_API pa_status pa_release_slots(const pa_geom* geom, int32_t* block_table, int32_t n,
                                  const int32_t* slots, int32_t* free_pages, int32_t* free_count,
                                  int32_t* err_flag, pa_stream_t stream) {
    if (!geom_valid(geom) || n < 0) return PA_ERR_INVALID_ARG;
    if (geom->num_slots > PA_PAGES_MAX_SLOTS) return PA_ERR_UNSUPPORTED;
    if (!block_table || !free_pages || !free_count || !err_flag) return PA_ERR_INVALID_ARG;
    if (n > 0 && !slots) return PA_ERR_INVALID_ARG;
    if (n == 0) return PA_OK;
    return cuda_status(pa::launch_release_slots(kgeom(geom), block_table, n, slots, free_pages, free_count,
                                                err_flag, reinterpret_cast<cudaStream_t>(stream)));
}

PA_API pa_status pa_debug_hold_first_copy(int32_t enable) {
    pa::g_hold_first_copy.store(enable ? 1 : 0, std::memory_order_relaxed);
    return PA_OK;
}

PA_API const char* pa_status_string(pa_status status) {
    switch (status) {
        case PA_OK: return "PA_OK: success";
        case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG: invalid argument";
        case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED: configuration not supported";
        case PA_ERR_CUDA: return "PA_ERR_CUDA: CUDA runtime or launch error";
        case PA_ERR_BAD_BLOCK: return "PA_ERR_BAD_BLOCK: invalid page, slot, position or length";
        case PA_ERR_TIMEOUT: return "PA_ERR_TIMEOUT: a bounded wait inside a kernel ran out";
        case PA_ERR_OUT_OF_PAGES: return "PA_ERR_OUT_OF_PAGES: the free page stack ran short (or would overflow)";
    }
    return "unknown pa_status";
}

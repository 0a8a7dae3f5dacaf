// prefill.cu -- causal prefill over a paged KV cache on the sm_103a tensor
// cores (tcgen05.mma, accumulators in tensor memory, operands staged by TMA).
//
// What is computed: query row i of a sequence attends keys 0..i; scores
// s = scale q.k (jaehun.me tiny-vllm part 3, "Per-head attention scores and
// GQA"), masked above the diagonal ("causalMask and online softmax"), softmax
// with the FlashAttention-2 deferred normalisation: keep the unnormalised
// output and l, divide once at the end, store L = m + ln l (base.kaita.kr,
// "플래시어텐션-2: 더 나은 병렬화", "단계별 설명 (순전파의 두 가지 손질)").
// Tiles whose keys all lie after their rows are skipped and only the diagonal
// tile is masked ("인과 마스크 처리").  Q head h reads kv head h / (Hq / Hkv)
// without copying K/V ("4. MQA · GQA 지원").
//
// GB300 mapping (prior art on the pages: cuBLAS per head + separate mask and
// softmax kernels; FA2's warp split on A100):
//  * One CTA per SM-sized work item: a 128-row query tile of a sequence for two
//    q heads of the same GQA group (tiles A and B; one head when the group size
//    is odd).  Both tiles read the same K/V tiles, staged once.  Items are
//    launched heaviest first (the last row tiles own the most key tiles).
//  * Warp 0 (TMA producer): the two Q tiles with one 2D tensor copy per 64-dim
//    chunk; each 128-key K/V tile as 8 pages, each page one {64 x 16} box per
//    chunk for K and one for V, rows addressed through the block table -- the
//    pool is one 2D tensor [pages * 32 rows][KV_DIM], page p's K rows at 32p,
//    V rows at 32p + 16.  128-byte swizzled boxes stack into the canonical
//    K-major (Q, K) / MN-major (V) operand layouts of the tensor core.  Pages
//    past the sequence end are read at an out-of-range row, which the copy
//    engine fills with zeros.  Three K/V stages at d 64, two at d 128.
//  * Warp 1 (single-thread MMA issuer): S = Q K^T (M 128, N 128, K 16 steps)
//    into TMEM; after a softmax warpgroup hands back P, O += P V with P read
//    straight from TMEM (M 128, N 64 per 64-dim chunk, K 16).  Issue order
//    PV_A(j), QK_A(j+1), PV_B(j), QK_B(j+1): while one tile's softmax runs, the
//    tensor core works on the other tile.
//  * Warps 4-7 and 8-11 (softmax, one warpgroup per tile): thread r owns query
//    row r, i.e. TMEM lane r; scores stream out of TMEM 32 columns at a time;
//    P = 2^(s*scale*log2e - m) is formed with packed fp32 FMAs and the SFU
//    exp2, packed to bf16 into TMEM; l stays in a register.  The reference max
//    only moves when a row max exceeds it by more than 2^8; then the thread
//    rescales its O row in TMEM (exact, since the final division uses the same
//    m).  The epilogue divides by l, writes o (bf16) and L = ln2 (m + log2 l).
//  * TMEM (512 columns): S_A, S_B, O_A, O_B, and P_A, P_B in their own columns
//    at d 64; at d 128 P overwrites the S it came from.
//  * A partial last page has its V rows past the sequence end zeroed in shared
//    memory before the PV product (masked P is exactly 0, but 0 x NaN is not).
#include <math_constants.h>

#include "pa_internal.cuh"

namespace pa {
namespace {

constexpr int BM = 128;               // query rows per tile (TMEM lanes)
constexpr int BN = 128;               // keys per K/V tile
constexpr int kPagesPerTile = BN / kBlockTokens;
constexpr int kThreads = 384;         // TMA warp, MMA warp, 2 idle, 2 softmax warpgroups
constexpr int kChunkBytes = 128 * 128;  // 128 rows x 128 bytes: one 64-dim chunk of a tile
constexpr int kTmemCols = 512;

template <int D>
struct Cfg {
    static constexpr int KCH = D / 64;
    static constexpr int Q_BYTES = KCH * kChunkBytes;  // one query tile
    static constexpr int K_BYTES = KCH * kChunkBytes;
    static constexpr int STAGE_BYTES = 2 * K_BYTES;
    static constexpr int NST = D == 64 ? 3 : 2;
    static constexpr int SMEM = 1024 + 2 * Q_BYTES + NST * STAGE_BYTES + 1024;
    // tensor memory: S_A S_B (128 columns each), O_A O_B (d each), P_A P_B (64
    // each) -- at d 128 there is no room left, so P overwrites the S it came from
    static constexpr bool P_ALIAS = D == 128;
    static __device__ __forceinline__ uint32_t s_col(int t) { return 128u * t; }
    static __device__ __forceinline__ uint32_t o_col(int t) { return 256u + D * t; }
    static __device__ __forceinline__ uint32_t p_col(int t) { return P_ALIAS ? 128u * t : 384u + 64u * t; }
};

struct PrefillParams {
    KGeom g;
    const int32_t* bt;
    int layer;
    int batch;
    const int32_t* cu;
    const int32_t* slots;
    int max_seqlen;
    int total_tokens;
    int n_row_tiles;
    int pair;             // 1: a CTA takes two q heads of one GQA group
    float scale_log2;
    __nv_bfloat16* o;
    float* lse;
    int32_t* err;
};

// Softmax of one tile for the calling thread's query row r (= its TMEM lane).
// The 128 scores are streamed from TMEM 32 columns at a time, the next chunk's
// load in flight while the current one is processed.  On the diagonal tile the
// keys after the row are masked to -inf.

// Row max of the raw scores.
template <bool DIAG>
__device__ __forceinline__ float tile_row_max(uint32_t tS, int r) {
    uint32_t b0[32], b1[32];
    float mx = -CUDART_INF_F;
    tmem_ld_x32_nowait(tS, b0);
    tmem_wait_ld_dep(b0);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t(&cur)[32] = (q & 1) ? b1 : b0;
        uint32_t(&nxt)[32] = (q & 1) ? b0 : b1;
        if (q < 3) tmem_ld_x32_nowait(tS + 32 * (q + 1), nxt);
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
            float s0 = __uint_as_float(cur[e]), s1 = __uint_as_float(cur[e + 1]);
            if (DIAG) {
                if (32 * q + e > r) s0 = -CUDART_INF_F;
                if (32 * q + e + 1 > r) s1 = -CUDART_INF_F;
            }
            mx = fmax3(mx, s0, s1);
        }
        if (q < 3) tmem_wait_ld_dep(nxt);
    }
    return mx;
}

// P = 2^(s * sc - m_ref) as bf16 pairs into the 64 TMEM columns at tP (one
// packed FMA per two scores, one ex2 each); returns the sum of the fp32 P and,
// through mx, the raw row max of the tile (tracked in the same pass).
template <bool DIAG>
__device__ __forceinline__ float tile_row_p(uint32_t tS, uint32_t tP, int r, float sc, float m_ref, float& mx) {
    const float nm = -m_ref;
    float ls[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};  // 4 independent pair sums
    float m = -CUDART_INF_F;
    uint32_t b0[32], b1[32];
    tmem_ld_x32_nowait(tS, b0);
    tmem_wait_ld_dep(b0);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t(&cur)[32] = (q & 1) ? b1 : b0;
        uint32_t(&nxt)[32] = (q & 1) ? b0 : b1;
        if (q < 3) tmem_ld_x32_nowait(tS + 32 * (q + 1), nxt);
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            float s0 = __uint_as_float(cur[2 * e]), s1 = __uint_as_float(cur[2 * e + 1]);
            if (DIAG) {
                if (32 * q + 2 * e > r) s0 = -CUDART_INF_F;
                if (32 * q + 2 * e + 1 > r) s1 = -CUDART_INF_F;
            }
            m = fmax3(m, s0, s1);
            float x0, x1;
            ffma2(x0, x1, s0, s1, sc, sc, nm, nm);
            const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
            const int a = 2 * (e & 3);
            fadd2(ls[a], ls[a + 1], ls[a], ls[a + 1], p0, p1);
            pk[e] = pack_bf16x2(p0, p1);
        }
        tmem_st_x16_nowait(tP + 16 * q, pk);
        if (q < 3) tmem_wait_ld_dep(nxt);
    }
    tmem_wait_st();
    mx = m;
    return ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
}

// Softmax role of one query tile: the warpgroup's thread r owns query row r
// (TMEM lane r).  O in TMEM holds sum_t P_t V_t with every P_t relative to one
// reference m_o (log2 units of the scaled score); l_run is relative to the same
// m_o.  With a separate P region (d 64) P_j is formed against the current m_o in
// one pass that also finds the tile max; only the first tile or a jump of more
// than 2^64 takes a separate max pass.  With P over S (d 128) the max pass
// always comes first.  When a tile max exceeds m_o by more than 2^8 the
// reference moves up: l_run at once, the O row before the next PV product
// (or in the epilogue).  Exact: o = O / l uses a single reference.
template <int D>
__device__ __forceinline__ void softmax_role(uint32_t tS, uint32_t tO, uint32_t tP, int r, int i, int nkv, int n,
                                             int cu0, int hq, bool zero_tail_owner, uint8_t* sKV, uint64_t* s_full,
                                             uint64_t* p_full, uint64_t* o_done, uint64_t* kv_full,
                                             volatile int* abort_flag, const PrefillParams& p) {
    using C = Cfg<D>;
    const KGeom& g = p.g;
    const float sc = p.scale_log2;
    const int row_in_seq = i * BM + r;
    float m_o = -CUDART_INF_F, l_run = 0.f;
    float o_pending = 1.f;  // factor O still owes for a move of m_o
    bool ok = true;
    const int last_lp = (n + kBlockTokens - 1) / kBlockTokens - 1;
    const int tail_valid = n - last_lp * kBlockTokens;
    const bool zero_tail = zero_tail_owner && (i == (n - 1) / BM) && tail_valid < kBlockTokens;
    for (int j = 0; j < nkv; ++j) {
        if (!__all_sync(0xffffffffu, mbar_wait(s_full, j & 1, abort_flag, p.err))) {
            ok = false;
            break;
        }
        tc_fence_after_sync();
        const bool diag = (j == i);
        float mx, lsum;
        if (C::P_ALIAS || j == 0) {
            const float m_tile = sc * (diag ? tile_row_max<true>(tS, r) : tile_row_max<false>(tS, r));
            if (j == 0) {
                m_o = m_tile;
            } else if (m_tile > m_o + 8.f) {  // move the reference before this product
                const float f = ex2_approx(m_o - m_tile);
                l_run *= f;
                o_pending *= f;
                m_o = m_tile;
            }
            lsum = diag ? tile_row_p<true>(tS, tP, r, sc, m_o, mx) : tile_row_p<false>(tS, tP, r, sc, m_o, mx);
        } else {
            lsum = diag ? tile_row_p<true>(tS, tP, r, sc, m_o, mx) : tile_row_p<false>(tS, tP, r, sc, m_o, mx);
            const float m_tile = mx * sc;
            if (__any_sync(0xffffffffu, m_tile > m_o + 64.f)) {  // rare: redo against the new max
                const float m_new = fmaxf(m_o, m_tile);
                const float f = ex2_approx(m_o - m_new);
                l_run *= f;
                o_pending *= f;
                m_o = m_new;
                lsum = diag ? tile_row_p<true>(tS, tP, r, sc, m_o, mx) : tile_row_p<false>(tS, tP, r, sc, m_o, mx);
            }
        }
        if (j > 0 && __any_sync(0xffffffffu, o_pending != 1.f)) {
            // O must follow the reference before this tile's PV product
            if (!__all_sync(0xffffffffu, mbar_wait(o_done, (j - 1) & 1, abort_flag, p.err))) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
#pragma unroll
            for (int c = 0; c < C::KCH; ++c) {
                uint32_t ov[64];
                tmem_ld_x64(tO + 64 * c, ov);
#pragma unroll
                for (int e = 0; e < 64; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * o_pending);
                tmem_st_x64(tO + 64 * c, ov);
            }
            o_pending = 1.f;
        }
        l_run += lsum;
        if (!C::P_ALIAS) {
            const float m_tile = mx * sc;
            if (m_tile > m_o + 8.f) {  // move the reference up; O follows after this product
                const float f = ex2_approx(m_o - m_tile);
                l_run *= f;
                o_pending = f;
                m_o = m_tile;
            }
        }
        if (diag && zero_tail) {
            const int st = j % C::NST;
            if (!__all_sync(0xffffffffu, mbar_wait(&kv_full[st], (j / C::NST) & 1, abort_flag, p.err))) {
                ok = false;
                break;
            }
            uint8_t* sV = sKV + st * C::STAGE_BYTES + C::K_BYTES;
            const int kk = last_lp - j * kPagesPerTile;  // page of the tile
            const int nz = (kBlockTokens - tail_valid) * 8 * C::KCH;  // 16-byte pieces
            for (int t = r; t < nz; t += 128) {
                const int piece = t & 7;
                const int c = (t >> 3) % C::KCH;
                const int row = tail_valid + (t >> 3) / C::KCH;
                *reinterpret_cast<uint4*>(sV + c * kChunkBytes + (kk * kBlockTokens + row) * 128 + piece * 16) =
                    make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();
        }
        tc_fence_before_sync();
        mbar_arrive(p_full);
    }
    if (ok && __all_sync(0xffffffffu, mbar_wait(o_done, (nkv - 1) & 1, abort_flag, p.err))) {
        tc_fence_after_sync();
        const bool store = row_in_seq < n;
        const float inv = l_run > 0.f ? o_pending / l_run : 0.f;
        const long long orow = static_cast<long long>(cu0 + row_in_seq) * g.hq + hq;
#pragma unroll
        for (int c = 0; c < C::KCH; ++c) {
            uint32_t ov[64];
            tmem_ld_x64(tO + 64 * c, ov);
            if (store) {
                uint4* dst = reinterpret_cast<uint4*>(p.o + orow * D + 64 * c);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    uint4 v;
                    v.x = pack_bf16x2(__uint_as_float(ov[8 * e + 0]) * inv, __uint_as_float(ov[8 * e + 1]) * inv);
                    v.y = pack_bf16x2(__uint_as_float(ov[8 * e + 2]) * inv, __uint_as_float(ov[8 * e + 3]) * inv);
                    v.z = pack_bf16x2(__uint_as_float(ov[8 * e + 4]) * inv, __uint_as_float(ov[8 * e + 5]) * inv);
                    v.w = pack_bf16x2(__uint_as_float(ov[8 * e + 6]) * inv, __uint_as_float(ov[8 * e + 7]) * inv);
                    dst[e] = v;
                }
            }
        }
        if (store && p.lse) p.lse[orow] = l_run > 0.f ? (m_o + lg2_approx(l_run)) * kLn2 : -CUDART_INF_F;
    }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
prefill_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kvmap,
               const PrefillParams p) {
    using C = Cfg<D>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);  // 1024-aligned operand tiles
    uint8_t* sQ = smem;                                            // tile A, then tile B
    uint8_t* sKV = smem + 2 * C::Q_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sKV + C::NST * C::STAGE_BYTES);
    uint64_t* q_full = bars;
    uint64_t* kv_full = bars + 1;
    uint64_t* kv_empty = bars + 1 + C::NST;
    uint64_t* s_full = bars + 1 + 2 * C::NST;  // [2]
    uint64_t* p_full = s_full + 2;             // [2]
    uint64_t* o_done = s_full + 4;             // [2]
    uint64_t* mma_done = s_full + 6;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 24);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 25);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const KGeom& g = p.g;

    // ---- work item: row tile (heaviest first), sequence, q head (pair)
    const int units = p.pair ? g.hq / 2 : g.hq;
    const int per_tile = p.batch * units;
    const int item = blockIdx.x;
    const int i = p.n_row_tiles - 1 - item / per_tile;
    const int rem = item % per_tile;
    const int b = rem / units;
    const int u = rem % units;
    const int hq_a = p.pair ? 2 * u : u;
    const bool has_b = p.pair != 0;
    const int hq_b = hq_a + 1;
    const int hk = hq_a / g.group;
    const int cu0 = p.cu[b], cu1 = p.cu[b + 1];
    const int n = cu1 - cu0;
    const bool bad_len = cu0 < 0 || n < 0 || cu1 > p.total_tokens || n > p.max_seqlen;
    if (i == 0 && u == 0 && tid == 0 && bad_len) set_error(p.err, PA_ERR_BAD_BLOCK);
    if (cu0 < 0 || n <= 0 || cu1 > p.total_tokens) return;
    if (i * BM >= n) return;
    const int slot = p.slots[b];
    const bool slot_ok = slot >= 0 && slot < g.num_slots;
    if (!slot_ok && tid == 0) set_error(p.err, PA_ERR_BAD_BLOCK);
    const int nkv = i + 1;  // causal: key tiles 0..i
    const int pages_b = (n + kBlockTokens - 1) / kBlockTokens;
    const long long tbase = (static_cast<long long>(slot_ok ? slot : 0) * g.n_layers + p.layer) * g.maxb;

    if (tid == 0) {
        mbar_init(q_full, 1);
        for (int s = 0; s < C::NST; ++s) {
            mbar_init(&kv_full[s], 1);
            mbar_init(&kv_empty[s], 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(&s_full[t], 1);
            mbar_init(&p_full[t], 128);
            mbar_init(&o_done[t], 1);
        }
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        mbar_init_fence();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            prefetch_tensor_map(&qmap);
            prefetch_tensor_map(&kvmap);
            mbar_arrive_expect_tx(q_full, (has_b ? 2 : 1) * C::Q_BYTES);
#pragma unroll
            for (int c = 0; c < C::KCH; ++c) {
                tma_load_2d(sQ + c * kChunkBytes, &qmap, hq_a * D + 64 * c, cu0 + i * BM, q_full);
                if (has_b)
                    tma_load_2d(sQ + C::Q_BYTES + c * kChunkBytes, &qmap, hq_b * D + 64 * c, cu0 + i * BM, q_full);
            }
        }
        const int oob_row = static_cast<int>(g.nblocks * 32);  // first row past the pool: zero fill
        int issued = 0;
        bool stop = false;
        for (int j = 0; j < nkv; ++j) {
            const int st = j % C::NST;
            if (j >= C::NST &&
                !__all_sync(0xffffffffu, mbar_wait(&kv_empty[st], ((j / C::NST) - 1) & 1, abort_flag, p.err))) {
                stop = true;
                break;
            }
            // lanes 0..7 fetch the tile's page ids
            const int lp = j * kPagesPerTile + lane;
            int row = -1;
            if (lane < kPagesPerTile && lp < pages_b) {
                if (slot_ok && lp < g.maxb) {
                    const int e = __ldg(p.bt + tbase + lp);
                    if (e >= 0 && e < g.nblocks) row = e * 32;
                }
                if (row < 0) set_error(p.err, PA_ERR_BAD_BLOCK);
            }
            uint8_t* sK = sKV + st * C::STAGE_BYTES;
            uint8_t* sV = sK + C::K_BYTES;
            if (lane == 0) mbar_arrive_expect_tx(&kv_full[st], C::STAGE_BYTES);
#pragma unroll
            for (int k = 0; k < kPagesPerTile; ++k) {
                const int rr = __shfl_sync(0xffffffffu, row, k);
                if (lane == 0) {
                    const int y = rr < 0 ? oob_row : rr;
#pragma unroll
                    for (int c = 0; c < C::KCH; ++c) {
                        tma_load_2d(sK + c * kChunkBytes + k * 2048, &kvmap, hk * D + 64 * c, y, &kv_full[st]);
                        tma_load_2d(sV + c * kChunkBytes + k * 2048, &kvmap, hk * D + 64 * c, y + 16, &kv_full[st]);
                    }
                }
            }
            ++issued;
        }
        if (stop && lane == 0) {  // let every copy in flight land before leaving
            mbar_drain(q_full, 0);
            for (int jj = issued > C::NST ? issued - C::NST : 0; jj < issued; ++jj)
                mbar_drain(&kv_full[jj % C::NST], (jj / C::NST) & 1);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // Tile A's softmax runs while the tensor core works on tile B and the
        // reverse: PV_A(j), QK_A(j+1), PV_B(j), QK_B(j+1), ...
        if (lane == 0) {
            constexpr uint32_t idesc_qk = umma_idesc_bf16(BM, BN, false);
            constexpr uint32_t idesc_pv = umma_idesc_bf16(BM, 64, true);
            const uint32_t sq = smem_u32(sQ);
            auto qk = [&](int t, int st) {
                const uint32_t sK = smem_u32(sKV + st * C::STAGE_BYTES);
                const uint32_t sqt = sq + t * C::Q_BYTES;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t off = (ks / 4) * kChunkBytes + (ks % 4) * 32;
                    umma_ss(tmem + C::s_col(t), umma_sdesc_sw128(sqt + off, 16, 1024),
                            umma_sdesc_sw128(sK + off, 16, 1024), idesc_qk, ks > 0 ? 1u : 0u);
                }
                umma_commit(&s_full[t]);
            };
            auto pv = [&](int t, int st, bool acc) {
                const uint32_t sV = smem_u32(sKV + st * C::STAGE_BYTES) + C::K_BYTES;
#pragma unroll
                for (int ks = 0; ks < BN / 16; ++ks) {
#pragma unroll
                    for (int c = 0; c < C::KCH; ++c)
                        umma_ts(tmem + C::o_col(t) + 64 * c, tmem + C::p_col(t) + ks * 8,
                                umma_sdesc_sw128(sV + c * kChunkBytes + ks * 2048, 1024, 1024), idesc_pv,
                                (acc || ks > 0) ? 1u : 0u);
                }
                umma_commit(&o_done[t]);
            };
            bool ok = mbar_wait(q_full, 0, abort_flag, p.err) && mbar_wait(&kv_full[0], 0, abort_flag, p.err);
            if (ok) {
                tc_fence_after_sync();
                qk(0, 0);
                if (has_b) qk(1, 0);
            }
            for (int j = 0; ok && j < nkv; ++j) {
                const int st = j % C::NST;
                const int st1 = (j + 1) % C::NST;
                const bool more = j + 1 < nkv;
                if (!mbar_wait(&p_full[0], j & 1, abort_flag, p.err)) break;
                tc_fence_after_sync();
                pv(0, st, j > 0);
                if (more) {
                    if (!mbar_wait(&kv_full[st1], ((j + 1) / C::NST) & 1, abort_flag, p.err)) break;
                    tc_fence_after_sync();
                    qk(0, st1);
                }
                if (has_b) {
                    if (!mbar_wait(&p_full[1], j & 1, abort_flag, p.err)) break;
                    tc_fence_after_sync();
                    pv(1, st, j > 0);
                }
                umma_commit(&kv_empty[st]);
                if (has_b && more) qk(1, st1);
            }
            umma_commit(mma_done);  // every MMA of this CTA done before TMEM is freed
            mbar_drain(mma_done, 0);
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ------------------------------------------------------------ softmax
        const int t = (warp - 4) >> 2;  // 0: tile A (warps 4-7), 1: tile B (warps 8-11)
        if (t == 0 || has_b) {
            const int r = (warp & 3) * 32 + lane;
            const uint32_t lane_base = tmem_lane_base(warp);
            softmax_role<D>(tmem + lane_base + C::s_col(t), tmem + lane_base + C::o_col(t),
                            tmem + lane_base + C::p_col(t), r, i, nkv, n, cu0, t ? hq_b : hq_a, t == 0, sKV,
                            &s_full[t], &p_full[t], &o_done[t], kv_full, abort_flag, p);
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

// 2D bf16 tensor [rows][cols] with row pitch `pitch_bytes`, box {64, box_rows},
// 128-byte swizzle, zero fill out of range.
bool encode_2d(CUtensorMap* map, const void* base, unsigned long long cols, unsigned long long rows,
               unsigned long long pitch_bytes, unsigned box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {pitch_bytes};
    const cuuint32_t box[2] = {64, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
cudaError_t launch(const CUtensorMap& qmap, const CUtensorMap& kvmap, const PrefillParams& p, cudaStream_t stream) {
    auto kern = prefill_kernel<D>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D>::SMEM);
    if (e != cudaSuccess) return e;
    const long long grid = static_cast<long long>(p.n_row_tiles) * p.batch * (p.pair ? p.g.hq / 2 : p.g.hq);
    if (grid > 0x7FFFFFFFll) return cudaErrorInvalidConfiguration;
    kern<<<static_cast<unsigned>(grid), kThreads, Cfg<D>::SMEM, stream>>>(qmap, kvmap, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill(const KGeom& g, const void* q, const void* pool, const int32_t* block_table, int layer,
                           int batch, const int32_t* cu_seqlens, const int32_t* slots, int max_seqlen,
                           int total_tokens, float scale, void* o, float* lse, int32_t* err, cudaStream_t stream) {
    CUtensorMap qmap, kvmap;
    if (!encode_2d(&qmap, q, static_cast<unsigned long long>(g.hq) * g.d, static_cast<unsigned long long>(total_tokens),
                   static_cast<unsigned long long>(g.hq) * g.d * 2, BM))
        return cudaErrorInvalidValue;
    if (!encode_2d(&kvmap, pool, static_cast<unsigned long long>(g.kv_dim),
                   static_cast<unsigned long long>(g.nblocks) * 32, static_cast<unsigned long long>(g.kv_dim) * 2,
                   kBlockTokens))
        return cudaErrorInvalidValue;
    PrefillParams p;
    p.g = g;
    p.bt = block_table;
    p.layer = layer;
    p.batch = batch;
    p.cu = cu_seqlens;
    p.slots = slots;
    p.max_seqlen = max_seqlen;
    p.total_tokens = total_tokens;
    p.n_row_tiles = (max_seqlen + BM - 1) / BM;
    p.pair = (g.group % 2 == 0) ? 1 : 0;
    p.scale_log2 = scale * kLog2e;
    p.o = static_cast<__nv_bfloat16*>(o);
    p.lse = lse;
    p.err = err;
    return g.d == 64 ? launch<64>(qmap, kvmap, p, stream) : launch<128>(qmap, kvmap, p, stream);
}

}  // namespace pa

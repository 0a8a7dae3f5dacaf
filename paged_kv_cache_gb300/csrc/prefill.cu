// prefill.cu -- causal prefill over a paged KV cache on the sm_103a tensor
// cores (tcgen05.mma, accumulators in tensor memory, operands staged by TMA).
//
// What is computed: query row i of a sequence attends keys 0..i; scores
// s = scale q.k (jaehun.me tiny-vllm part 3, "Per-head attention scores and
// GQA"), masked above the diagonal ("causalMask and online softmax"), softmax
// with the FlashAttention-2 deferred normalisation: keep the unnormalised
// output and l, divide once at the end, store L = m + ln l (base.kaita.kr,
// "플래시어텐션-2: 더 나은 병렬화", "단계별 설명 (순전파의 두 가지 손질)").
// Key tiles that lie wholly after a row tile are skipped and only the tiles
// that cross the diagonal are masked ("인과 마스크 처리").  Q head h reads kv
// head h / (Hq / Hkv) without copying K/V ("4. MQA · GQA 지원").
//
// GB300 mapping (prior art on the pages: cuBLAS per head + separate mask and
// softmax kernels; FA2's warp split on A100):
//  * One CTA per work item: a 128-row query tile of a sequence for T q heads of
//    one GQA group (T = 4 at d 64, 2 at d 128 when the group size allows; 1
//    otherwise).  The T tiles read the same K/V, staged once.  Items are
//    launched heaviest first (the last row tiles own the most key tiles).
//  * Warp 4T (TMA producer): the T query tiles with one 2D tensor copy per
//    64-dim chunk; each 64-key K/V tile as 4 pages, each page one {64 x 16} box
//    per chunk for K and one for V, rows addressed through the block table --
//    the pool is one 2D tensor [pages * 32 rows][KV_DIM], page p's K rows at
//    32p, V rows at 32p + 16.  128-byte swizzled boxes stack into the canonical
//    K-major (Q, K) / MN-major (V) operand layouts of the tensor core.  Pages
//    past the sequence end are read at an out-of-range row, which the copy
//    engine fills with zeros.
//  * Warps 4T+1 (and 4T+2 when T >= 2) issue the MMAs; the whole warp runs
//    the loop and one elected lane issues.  S_t = Q_t K^T (M 128, N 64, K 16
//    steps) into TMEM; after tile t's softmax hands back P_t, O_t += P_t V (M
//    128, N 64 per 64-dim chunk, K 16, P read from TMEM), then the next S_t.
//    The tiles take turns, so the tensor core works on the others while one
//    tile's softmax runs; with two issuing warps, tile t belongs to warp t % 2.
//    Where tensor memory holds two score buffers per tile (T <= 2: d 128, and
//    the two-head launches at d 64) S of key tile j + 1 is computed while the
//    softmax works on tile j, and P of tile j is followed in its buffer by S
//    of tile j + 2.
//  * Warps 4t..4t+3 (softmax of tile t): thread r owns query row r, i.e. TMEM
//    lane r, and all 64 scores of the key tile, read as two 32-key halves.  A
//    half whose max exceeds the reference max by more than 2^8 moves it (l
//    at once, the first half's P and partial sums in registers if the second
//    half moves it, its O row in TMEM in place -- with one score buffer no PV
//    product is in flight then; with two it first waits for the last one).
//    P = 2^(s*scale*log2e - m) comes from packed fp32 FMAs and the SFU exp2,
//    packed to bf16.  The epilogue divides by l, writes o (bf16) and
//    L = ln2 (m + log2 l).  Exact: o = O / l uses the one reference.
//  * TMEM: tile t owns NB 64 + d columns from t (NB 64 + d): NB score buffers
//    S (each 32-key half holds its P in its first 16 columns), then O.
//  * A partial last page has its V rows past the sequence end zeroed in shared
//    memory before the PV products (masked P is exactly 0, but 0 x NaN is not).
//  * RoPE on the queries (pa_prefill_rope; tiny-vllm part 3, "RoPE: a rotation
//    that references a table": Q turns with the tables K turned with): once
//    the query tiles have landed, each softmax thread turns its own row of its
//    tile in shared memory, following the 128-byte swizzle, with the angle
//    row of the query's position (loaded before the tiles arrive), and the
//    first QK product waits for every row to be turned.
#include <math_constants.h>

#include <mutex>

#include "pa_internal.cuh"

namespace pa {
namespace {

constexpr int BM = 128;                 // query rows per tile (TMEM lanes)
constexpr int BN = 64;                  // keys per K/V tile
constexpr int kPagesPerTile = BN / kBlockTokens;
constexpr int kQChunkBytes = BM * 128;  // 128 rows x 128 bytes: one 64-dim chunk of a query tile
constexpr int kKChunkBytes = BN * 128;  // 64 keys x 128 bytes: one 64-dim chunk of a K or V tile
constexpr float kMoveAbove = 8.f;       // the reference max moves when a 32-key half exceeds it by 2^8

template <int D, int T>
struct Cfg {
    static constexpr int KCH = D / 64;
    static constexpr int PRODUCER_WARP = 4 * T;
    static constexpr int MMA_WARPS = T >= 2 ? 2 : 1;  // tile t is issued by MMA warp t % MMA_WARPS
    static constexpr int MMA_WARP = 4 * T + 1;        // the first one; it also owns the TMEM allocation
    static constexpr int THREADS = 32 * (4 * T + 1 + MMA_WARPS);
    static constexpr int Q_BYTES = KCH * kQChunkBytes;  // one query tile
    static constexpr int K_BYTES = KCH * kKChunkBytes;
    static constexpr int STAGE_BYTES = 2 * K_BYTES;
    static constexpr int CTL_BYTES = 1024;
    static constexpr int NST_FIT = (220 * 1024 - T * Q_BYTES - CTL_BYTES - 1024) / STAGE_BYTES;
    static constexpr int NST = NST_FIT > 8 ? 8 : NST_FIT;
    static constexpr int SMEM = 1024 + T * Q_BYTES + NST * STAGE_BYTES + CTL_BYTES;
    // score buffers per tile: two where tensor memory holds them (S of key
    // tile j + 1 is then computed while the softmax works on S of tile j)
    static constexpr int NB = T * (2 * BN + D) <= 512 ? 2 : 1;
    static constexpr int TILE_COLS = NB * BN + D;
    static constexpr uint32_t TMEM_COLS = T * TILE_COLS <= 128 ? 128u : T * TILE_COLS <= 256 ? 256u : 512u;
    static_assert(T * TILE_COLS <= 512, "tensor memory holds S and O of every tile");
    static_assert(NST >= 2, "two K/V stages at least");
    static_assert(NB == 1 || NST >= 3, "a K/V stage for each score buffer in flight and one more");
    static_assert(1 + 2 * NST + 2 * NB * T + 2 * T + MMA_WARPS + 1 <= 64, "barriers fit below the TMEM slot");
    static __device__ __forceinline__ uint32_t s_col(int t, int b) {
        return static_cast<uint32_t>(TILE_COLS * t + BN * b);
    }
    static __device__ __forceinline__ uint32_t o_col(int t) { return static_cast<uint32_t>(TILE_COLS * t + NB * BN); }
    // P columns of key step ks (16 keys) in score buffer b of tile t: the 32
    // keys of each half of the tile put their P over the first 16 of their
    // own score columns
    static __device__ __forceinline__ uint32_t p_col(int t, int b, int ks) {
        return s_col(t, b) + 32u * (ks >> 1) + 8u * (ks & 1);
    }
};

struct PrefillParams {
    KGeom g;
    const int32_t* bt;
    int layer;
    int batch;
    const int32_t* cu;
    const int32_t* prefix;  // cached tokens before each sequence's queries, or null
    const int32_t* slots;
    int max_seqlen;
    int total_tokens;
    int n_row_tiles;
    int heads_per_cta;    // T
    float scale_log2;
    __nv_bfloat16* o;
    bool o_32b;           // o is 32-byte aligned: rows go out in whole 32-byte sectors
    float* lse;
    int32_t* err;
    const float* cos_tab;  // RoPE-Q: angle tables [max_pos][d/2] (null without RoPE)
    const float* sin_tab;
    int max_pos;
    int hold_first_copy;   // diagnostic: CTA 0 arms its query copy without issuing it
    int item_base;         // work item of this launch's CTA 0
    int tail;              // launched as a programmatic dependent of the launch before it
    int has_tail;          // a tail launch follows this one
    // Key split (a tail launch only): CTA 2k + h takes half h of the key tiles
    // of item item_base + k and leaves its partial (O not yet divided by l,
    // with its m and l) in ws_o / ws_ml; the second of the two to finish, as
    // counted in ws_cnt[k], combines both.
    int ksplit;
    float* ws_o;    // [items][2][T][BM][D]
    float2* ws_ml;  // [items][2][T][BM]: (m in scaled log2 units, l)
    int* ws_cnt;    // [items], zero before the launch
};

// Barrier among the first `threads` threads of the CTA (the softmax warps) on
// hardware barrier 1; barrier 0 is the CTA-wide one.
__device__ __forceinline__ void softmax_barrier(int threads) {
    asm volatile("bar.sync 1, %0;" ::"r"(threads) : "memory");
}

// One float twice, as the 64-bit pair operand of the packed fp32 ops.
__device__ __forceinline__ uint64_t pair2(float a) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %1};" : "=l"(r) : "f"(a));
    return r;
}

// P = 2^(s * sc + nm) of 32 scores, packed to bf16 pairs; adds the fp32 P to
// ls (FIRST: the first half of the tile, whose first four pairs start ls).
// sc and nm enter the packed FMAs as pairs formed once per call.
template <bool FIRST>
__device__ __forceinline__ void p_chunk(const uint32_t (&v)[32], float sc, float nm, float (&ls)[8],
                                        uint32_t (&pk)[16]) {
    const uint64_t sc2 = pair2(sc), nm2 = pair2(nm);
#pragma unroll
    for (int e = 0; e < 16; ++e) {
        float x0, x1;
        asm("{\n\t.reg .b64 a2, d2;\n\t"
            "mov.b64 a2, {%2, %3};\n\t"
            "fma.rn.f32x2 d2, a2, %4, %5;\n\t"
            "mov.b64 {%0, %1}, d2;\n\t}"
            : "=f"(x0), "=f"(x1)
            : "f"(__uint_as_float(v[2 * e])), "f"(__uint_as_float(v[2 * e + 1])), "l"(sc2), "l"(nm2));
        const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
        const int a = 2 * (e & 3);
        if (FIRST && e < 4) {
            ls[a] = p0;
            ls[a + 1] = p1;
        } else {
            fadd2(ls[a], ls[a + 1], ls[a], ls[a + 1], p0, p1);
        }
        pk[e] = pack_bf16x2(p0, p1);
    }
}

// Scores of keys after the row become -inf: element e sits at key c0 + e
// relative to the first row of the tile.
__device__ __forceinline__ void mask_chunk(uint32_t (&v)[32], int c0, int r) {
#pragma unroll
    for (int e = 0; e < 32; ++e)
        if (c0 + e > r) v[e] = __float_as_uint(-CUDART_INF_F);
}

// Max of 32 scores in 16 three-input max operations: four chains over
// seven scores each, then their results with the four left over.
__device__ __forceinline__ float chunk_max16(const uint32_t (&v)[32]) {
    auto x = [&](int e) { return __uint_as_float(v[e]); };
    float c[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        c[k] = fmax3(x(8 * k), x(8 * k + 1), x(8 * k + 2));
        c[k] = fmax3(c[k], x(8 * k + 3), x(8 * k + 4));
        c[k] = fmax3(c[k], x(8 * k + 5), x(8 * k + 6));
    }
    const float a = fmax3(c[0], c[1], x(7));
    const float b = fmax3(c[2], c[3], x(15));
    return fmaxf(fmax3(a, x(23), x(31)), b);
}

// RoPE of row r of one query tile in shared memory (the tile's 64-dim chunks
// are 128 rows of 128 bytes, 16-byte pieces swizzled by row % 8): pair (e,
// e + D/2) of every 8-element group turns by the angle row of position pos.
// The angle rows are requested before the tile is waited for.  Returns false
// if the wait for the tile gave up.
template <int D>
__device__ __forceinline__ bool rope_q_row(uint8_t* tile, int r, bool turn, long long pos, uint64_t* q_full,
                                           volatile int* abort_flag, const PrefillParams& p) {
    constexpr int NG = D / 16;             // groups of 8 pairs
    constexpr int GB = NG < 4 ? NG : 4;    // groups whose angles are in registers at once
    float4 cs[GB][4];
    auto load = [&](int g0) {
#pragma unroll
        for (int gg = 0; gg < GB; ++gg) {
            const long long a = pos * (D / 2) + 8 * (g0 + gg);
            const float4* ct = reinterpret_cast<const float4*>(p.cos_tab + a);
            const float4* st = reinterpret_cast<const float4*>(p.sin_tab + a);
            cs[gg][0] = __ldg(ct);
            cs[gg][1] = __ldg(ct + 1);
            cs[gg][2] = __ldg(st);
            cs[gg][3] = __ldg(st + 1);
        }
    };
    if (turn) load(0);
    if (!__all_sync(0xffffffffu, mbar_wait(q_full, 0, abort_flag, p.err))) return false;
    auto piece = [&](int e) -> uint4* {  // the 16 bytes holding elements e .. e + 7 of row r
        return reinterpret_cast<uint4*>(tile + (e / 64) * kQChunkBytes + r * 128 + ((((e % 64) / 8) ^ (r & 7)) * 16));
    };
    if (turn) {
#pragma unroll
        for (int g0 = 0; g0 < NG; g0 += GB) {
            if (g0 > 0) load(g0);
#pragma unroll
            for (int gg = 0; gg < GB; ++gg) {
                const int e = 8 * (g0 + gg);
                uint4 lo = *piece(e), hi = *piece(e + D / 2);
                rope8(lo, hi, cs[gg][0], cs[gg][1], cs[gg][2], cs[gg][3]);
                *piece(e) = lo;
                *piece(e + D / 2) = hi;
            }
        }
        fence_proxy_async_smem();  // the turned rows before the tensor core reads them
    }
    return true;
}

// Softmax of query tile t: the warp's thread owns row r (TMEM lane r) and
// reads each 32-key half of a key tile's scores from tensor memory once.
// SPLIT: the instance may run as one half of a key split (not the RoPE-Q one).
template <int D, int T, bool SPLIT>
__device__ __forceinline__ void softmax_role(int t, int r, uint32_t tmem_lane, int i, int j0, int j1, int n,
                                             int pos0, int kv_len, int cu0, int hq,
                                             uint8_t* sKV, uint64_t* s_full, uint64_t* p_full, uint64_t* o_done,
                                             uint64_t* pv_done, uint64_t* kv_full, volatile int* abort_flag,
                                             int* split_flag,
                                             bool ok, const PrefillParams& p) {
    using C = Cfg<D, T>;
    const KGeom& g = p.g;
    const float sc = p.scale_log2;
    const uint32_t tO = tmem_lane + C::o_col(t);
    const int row = i * BM + r;  // query row within the chunk; its position is pos0 + r
    const int last_lp = (kv_len + kBlockTokens - 1) / kBlockTokens - 1;
    const int tail_valid = kv_len - last_lp * kBlockTokens;
    // every tile zeroes the V tail itself before its P is handed over: the
    // tiles' PV products are issued by different warps in no fixed order
    const int j_tail = tail_valid < kBlockTokens ? last_lp / kPagesPerTile : -1;
    float m_o = -CUDART_INF_F, l = 0.f;
    // -m_o (0 while m_o is -inf), kept in a register and set when the
    // reference moves: 0.8 % faster at d 64, 0.6 % at d 128 than forming it
    // from m_o before each use
    float nm_reg = 0.f;
    // the move test in raw score units (scale > 0): a half whose raw max
    // exceeds thr_raw = (m_o + 2^8) / sc moves the reference.  One multiply
    // and one add fewer between a half's max and its exp2: 1077 -> 1092
    // TFLOP/s at d 64, the same bits.
    const float move_raw = kMoveAbove / sc;
    float thr_raw = -CUDART_INF_F;
    if constexpr (!SPLIT) ok = true;  // outside a key split the role is entered only when ok
    for (int j = j0; (!SPLIT || ok) && j < j1; ++j) {
        const int jj = j - j0;  // key tiles of this CTA so far: barrier phases and stages count from j0
        const int sb = jj % C::NB;  // this key tile's score buffer
        const uint32_t tS = tmem_lane + C::s_col(t, sb);
        if (!__all_sync(0xffffffffu, mbar_wait(&s_full[sb], (jj / C::NB) & 1, abort_flag, p.err))) {
            ok = false;
            break;
        }
        tc_fence_after_sync();
        const int rel = BN * j - pos0;  // first key of the tile relative to the first row's position
        const bool diag = rel > -BN;      // the tile crosses the diagonal
        float f = 1.f;  // factor for l and this row of O when the reference moves
        bool moved = false;  // the reference moved in this tile
        // this tile's sums of P, started with its first half's values instead
        // of adding those to zeros (d 64 1090 -> 1094 TFLOP/s, the same bits)
        float ls[8];
        // this row of O follows the reference (with one score buffer no PV
        // product is in flight here)
        auto rescale_o = [&]() {
            if (jj > 0 && __any_sync(0xffffffffu, moved)) {
                // with two score buffers the PV product of key tile jj - 1 may
                // still be adding into O: wait for it (bounded)
                if constexpr (C::NB == 2) {
                    if (!__all_sync(0xffffffffu, mbar_wait(pv_done, (jj - 1) & 1, abort_flag, p.err))) return;
                }
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t ov[32];
                    tmem_ld_x32(tO + 32 * c, ov);
#pragma unroll
                    for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * f);
                    tmem_st_x32(tO + 32 * c, ov);
                }
            }
        };
        // one read of each 32-key half: the first half's max may move the
        // reference and its P waits in registers; should the second half
        // move it again (by more than 2^8, rare past the first tile), that
        // P and the partial sums follow the new reference in registers
        uint32_t pa[16];
        {
            uint32_t va[32];
            tmem_ld_x32(tS, va);
            if (diag) mask_chunk(va, rel, r);
            const float ma_raw = chunk_max16(va);
            if (ma_raw > thr_raw) {
                const float m_a = sc * ma_raw;
                thr_raw = ma_raw + move_raw;
                moved = true;
                f = ex2_approx(m_o - m_a);  // 0 from -inf
                l *= f;
                m_o = m_a;
                nm_reg = -m_o;
            }
            p_chunk<true>(va, sc, nm_reg, ls, pa);
        }
        {
            uint32_t vb[32], pk[16];
            tmem_ld_x32(tS + 32, vb);
            if (diag) mask_chunk(vb, rel + 32, r);
            const float mb_raw = chunk_max16(vb);
            if (mb_raw > thr_raw) {
                const float m_b = sc * mb_raw;
                thr_raw = mb_raw + move_raw;
                moved = true;
                const float f2 = ex2_approx(m_o - m_b);
                f *= f2;
                l *= f2;
                m_o = m_b;
                nm_reg = -m_o;
#pragma unroll
                for (int e = 0; e < 8; ++e) ls[e] *= f2;
#pragma unroll
                for (int e = 0; e < 16; ++e) pa[e] = pack_bf16x2(bf16lo(pa[e]) * f2, bf16hi(pa[e]) * f2);
            }
            p_chunk<false>(vb, sc, nm_reg, ls, pk);
            tmem_st_x16_nowait(tS + 32, pk);
        }
        tmem_st_x16_nowait(tS, pa);
        rescale_o();
        l += ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
        if (j == j_tail) {
            // V rows past the sequence end in the last page: zero (0 x NaN is NaN)
            const int st = jj % C::NST;
            if (!__all_sync(0xffffffffu, mbar_wait(&kv_full[st], (jj / C::NST) & 1, abort_flag, p.err))) {
                ok = false;
                break;
            }
            uint8_t* sV = sKV + st * C::STAGE_BYTES + C::K_BYTES;
            const int kk = last_lp % kPagesPerTile;  // page within the tile
            const int nz = (kBlockTokens - tail_valid) * 8 * C::KCH;  // 16-byte pieces
            for (int x = r; x < nz; x += BM) {
                const int piece = x & 7;
                const int c = (x >> 3) % C::KCH;
                const int rr = tail_valid + (x >> 3) / C::KCH;
                *reinterpret_cast<uint4*>(sV + c * kKChunkBytes + (kk * kBlockTokens + rr) * 128 + piece * 16) =
                    make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();
        }
        tmem_wait_st();
        tc_fence_before_sync();
        mbar_arrive(&p_full[sb]);
    }
    const bool empty = SPLIT && j1 <= j0;  // a key-split half with no key tile: O = 0, l = 0
    // `have`: this warp's O and l are complete.  In a key split every softmax
    // warp goes on from here whatever it says (the split's barriers count on it).
    const bool have = ok && (empty || __all_sync(0xffffffffu, mbar_wait(o_done, 0, abort_flag, p.err)));
    if (SPLIT || have) {
        tc_fence_after_sync();
        const bool store = row < n;
        const long long orow = static_cast<long long>(cu0 + row) * g.hq + hq;
        // this row of O, not yet divided by l: from TMEM, or 0 for an empty half
        auto load_o = [&](int c, uint32_t (&ov)[32]) {
            if (empty) {
#pragma unroll
                for (int e = 0; e < 32; ++e) ov[e] = 0u;
            } else {
                tmem_ld_x32(tO + 32 * c, ov);
            }
        };
        float m_fin = m_o, l_fin = l;       // the row's reference max and sum
        float a_own = 1.f, a_other = 0.f;  // weights of this half's O and of the other half's
        const float* o_other = nullptr;
        if constexpr (SPLIT) {
            // leave this half's partial; the second half to finish combines both
            const int k = static_cast<int>(blockIdx.x >> 1), h = static_cast<int>(blockIdx.x & 1);
            const long long prow = ((static_cast<long long>(k) * 2 + h) * T + t) * BM + r;
            const long long qrow = ((static_cast<long long>(k) * 2 + (h ^ 1)) * T + t) * BM + r;
            if (have) {
                float4* wo = reinterpret_cast<float4*>(p.ws_o + prow * D);
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t ov[32];
                    load_o(c, ov);
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        wo[8 * c + e] = make_float4(__uint_as_float(ov[4 * e]), __uint_as_float(ov[4 * e + 1]),
                                                    __uint_as_float(ov[4 * e + 2]), __uint_as_float(ov[4 * e + 3]));
                }
                p.ws_ml[prow] = make_float2(m_o, l);
                __threadfence();
            }
            // the CTA's softmax warps, all of them: every partial of this half is out
            softmax_barrier(4 * T * 32);
            if (t == 0 && r == 0) *split_flag = atomicAdd(p.ws_cnt + k, 1);
            softmax_barrier(4 * T * 32);
            if (*split_flag != 1 || !have) return;  // the other half combines (or this one stopped)
            __threadfence();
            const float2 mlq = __ldcg(p.ws_ml + qrow);
            // the same expression whichever half combines: half 0's terms first
            const float m0 = h == 0 ? m_o : mlq.x, l0 = h == 0 ? l : mlq.y;
            const float m1 = h == 0 ? mlq.x : m_o, l1 = h == 0 ? mlq.y : l;
            m_fin = fmaxf(m0, m1);
            const float a0 = m0 == -CUDART_INF_F ? 0.f : ex2_approx(m0 - m_fin);
            const float a1 = m1 == -CUDART_INF_F ? 0.f : ex2_approx(m1 - m_fin);
            l_fin = __fadd_rn(__fmul_rn(l0, a0), __fmul_rn(l1, a1));
            a_own = h == 0 ? a0 : a1;
            a_other = h == 0 ? a1 : a0;
            o_other = p.ws_o + qrow * D;
            if (t == 0 && r == 0) p.ws_cnt[k] = 0;  // ready for the next call
        }
        const float inv = l_fin > 0.f ? 1.f / l_fin : 0.f;
        uint4* dst = reinterpret_cast<uint4*>(p.o + orow * D);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
            uint32_t ov[32];
            load_o(c, ov);
            if (SPLIT && o_other) {
                // two rounded products and their sum, never fused: the same
                // bits whichever half adds them
                const float4* oq = reinterpret_cast<const float4*>(o_other) + 8 * c;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float4 w = __ldcg(oq + e);
                    const float x[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        ov[4 * e + q] = __float_as_uint(__fadd_rn(__fmul_rn(__uint_as_float(ov[4 * e + q]), a_own),
                                                                  __fmul_rn(x[q], a_other)));
                }
            }
            if (store && p.o_32b) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    uint32_t v[8];
#pragma unroll
                    for (int w = 0; w < 8; ++w)
                        v[w] = pack_bf16x2(__uint_as_float(ov[16 * e + 2 * w]) * inv,
                                           __uint_as_float(ov[16 * e + 2 * w + 1]) * inv);
                    st_global_v8(dst + 4 * c + 2 * e, v);
                }
            } else if (store) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    uint4 v;
                    v.x = pack_bf16x2(__uint_as_float(ov[8 * e + 0]) * inv, __uint_as_float(ov[8 * e + 1]) * inv);
                    v.y = pack_bf16x2(__uint_as_float(ov[8 * e + 2]) * inv, __uint_as_float(ov[8 * e + 3]) * inv);
                    v.z = pack_bf16x2(__uint_as_float(ov[8 * e + 4]) * inv, __uint_as_float(ov[8 * e + 5]) * inv);
                    v.w = pack_bf16x2(__uint_as_float(ov[8 * e + 6]) * inv, __uint_as_float(ov[8 * e + 7]) * inv);
                    dst[4 * c + e] = v;
                }
            }
        }
        if (store && p.lse) p.lse[orow] = l_fin > 0.f ? (m_fin + lg2_approx(l_fin)) * kLn2 : -CUDART_INF_F;
    }
}

// SPLIT: the instance that runs the halves of a key split (never with ROPE);
// the other instances compile without any of its steps.
template <int D, int T, bool ROPE, bool SPLIT>
__global__ void __launch_bounds__(Cfg<D, T>::THREADS, 1)
prefill_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kvmap,
               const PrefillParams p) {
    using C = Cfg<D, T>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);  // 1024-aligned operand tiles
    uint8_t* sQ = smem;                                            // T query tiles
    uint8_t* sKV = smem + T * C::Q_BYTES;
    uint8_t* ctl = sKV + C::NST * C::STAGE_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(ctl);
    uint64_t* q_full = bars;
    uint64_t* kv_full = bars + 1;                 // [NST]
    uint64_t* kv_empty = bars + 1 + C::NST;       // [NST]
    uint64_t* s_full = bars + 1 + 2 * C::NST;     // [T][NB] scores of a tile in a TMEM buffer
    uint64_t* p_full = s_full + C::NB * T;        // [T][NB] P of a tile in that buffer
    uint64_t* o_done = s_full + 2 * C::NB * T;    // [T] the last PV product of a tile done
    uint64_t* mma_done = o_done + T;              // [MMA_WARPS]
    uint64_t* q_ready = mma_done + C::MMA_WARPS;  // RoPE-Q: every query row turned
    uint64_t* pv_done = q_ready + 1;              // [T] (NB = 2) each PV product of a tile done
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 64);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 65);
    int* split_flag = reinterpret_cast<int*>(bars + 66);  // key split: this half finished second

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const KGeom& g = p.g;
    // A launch of the tail items may be scheduled once every CTA of this one
    // has started: it then fills the SMs this launch's last wave leaves idle.
    if (p.has_tail) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // The tail launch reads nothing the launch before it writes; its CTAs only
    // wait for that launch to finish before they leave (tail_wait at every
    // exit), so that the call is complete, in stream order, when the tail
    // launch is.
    auto tail_wait = [&p]() {
        if (p.tail) asm volatile("griddepcontrol.wait;" ::: "memory");
    };

    // ---- work item: row tile (heaviest first), sequence, kv head, group of T q heads
    const int qgroups = g.group / T;
    const int units = g.hkv * qgroups;
    const int per_tile = p.batch * units;
    const int item = (SPLIT ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x)) + p.item_base;
    const int i = p.n_row_tiles - 1 - item / per_tile;
    const int rem = item % per_tile;
    const int b = rem / units;
    const int u = rem % units;
    const int hk = u / qgroups;
    const int hq0 = hk * g.group + (u % qgroups) * T;
    const int cu0 = p.cu[b], cu1 = p.cu[b + 1];
    const int n = cu1 - cu0;
    const int pre = p.prefix ? p.prefix[b] : 0;
    const bool bad_len = cu0 < 0 || n < 0 || cu1 > p.total_tokens || n > p.max_seqlen || pre < 0 ||
                         static_cast<long long>(pre) + n > static_cast<long long>(g.maxb) * kBlockTokens;
    if (i == 0 && u == 0 && tid == 0 && bad_len) set_error(p.err, PA_ERR_BAD_BLOCK);
    if (bad_len || n <= 0 || i * BM >= n) {
        tail_wait();
        return;
    }
    const int slot = p.slots[b];
    const bool slot_ok = slot >= 0 && slot < g.num_slots;
    if (!slot_ok && tid == 0) set_error(p.err, PA_ERR_BAD_BLOCK);
    // causal: key tiles up to the one holding the last row's key pre + BM (i + 1) - 1,
    // and none past the cached sequence
    const int kv_len = pre + n;
    const int nkv = min((pre + BM * (i + 1) + BN - 1) / BN, (kv_len + BN - 1) / BN);
    // this CTA's key tiles [j0, j1): all of them, or one half of a key split
    // (the second half holds the diagonal and the sequence's last page)
    const int j0 = SPLIT && (blockIdx.x & 1) ? nkv / 2 : 0;
    const int j1 = SPLIT && !(blockIdx.x & 1) ? nkv / 2 : nkv;
    const int nk = j1 - j0;
    const int pages_b = (kv_len + kBlockTokens - 1) / kBlockTokens;
    const long long tbase = (static_cast<long long>(slot_ok ? slot : 0) * g.n_layers + p.layer) * g.maxb;

    if (tid == 0) {
        mbar_init(q_full, 1);
        for (int s = 0; s < C::NST; ++s) {
            mbar_init(&kv_full[s], 1);
            mbar_init(&kv_empty[s], C::MMA_WARPS);
        }
        for (int t = 0; t < T; ++t) {
            for (int b = 0; b < C::NB; ++b) {
                mbar_init(&s_full[C::NB * t + b], 1);
                mbar_init(&p_full[C::NB * t + b], BM);
            }
            mbar_init(&o_done[t], 1);
            if (C::NB == 2) mbar_init(&pv_done[t], 1);
        }
        for (int m = 0; m < C::MMA_WARPS; ++m) mbar_init(&mma_done[m], 1);
        if (ROPE) mbar_init(q_ready, 4 * T);  // one arrive per softmax warp
        *abort_flag = 0;
        mbar_init_fence();
    }
    if (warp == C::MMA_WARP) {
        tmem_alloc(tmem_slot, C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    int producer_issued = 0;       // K/V tiles the producer issued (its lane 0 drains them on an abort)
    bool producer_held_q = false;  // the diagnostic hold kept the query copy back

    if (warp == C::PRODUCER_WARP) {
        // ------------------------------------------------------------ TMA producer
        // the diagnostic hold: the query tiles' barrier is armed but no copy is
        // issued, so its phase never completes and the waits on it run out
        // (an empty half of a key split copies nothing)
        const bool hold_q = (p.hold_first_copy && blockIdx.x == 0) || (SPLIT && nk == 0);
        if (lane == 0) {
            prefetch_tensor_map(&qmap);
            prefetch_tensor_map(&kvmap);
            mbar_arrive_expect_tx(q_full, T * C::Q_BYTES);
            if (!hold_q) {
#pragma unroll
                for (int t = 0; t < T; ++t)
#pragma unroll
                    for (int c = 0; c < C::KCH; ++c)
                        tma_load_2d(sQ + t * C::Q_BYTES + c * kQChunkBytes, &qmap, (hq0 + t) * D + 64 * c,
                                    cu0 + i * BM, q_full);
            }
        }
        const int oob_row = static_cast<int>(g.nblocks * 32);  // first row past the pool: zero fill
        int issued = 0;
        for (int j = j0; j < j1; ++j) {
            const int jj = j - j0;
            const int st = jj % C::NST;
            if (jj >= C::NST &&
                !__all_sync(0xffffffffu, mbar_wait(&kv_empty[st], ((jj / C::NST) - 1) & 1, abort_flag, p.err)))
                break;  // another role stopped the CTA, or the wait ran out (then *abort_flag is set)
            // lanes 0..3 fetch the tile's page ids
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
                        tma_load_2d(sK + c * kKChunkBytes + k * 2048, &kvmap, hk * D + 64 * c, y, &kv_full[st]);
                        tma_load_2d(sV + c * kKChunkBytes + k * 2048, &kvmap, hk * D + 64 * c, y + 16, &kv_full[st]);
                    }
                }
            }
            ++issued;
        }
        producer_issued = issued;
        producer_held_q = hold_q;
    } else if (warp >= C::MMA_WARP) {
        // ------------------------------------------------------------ MMA issuers
        // Per key tile j, for each of this warp's query tiles in turn: once its
        // P is in TMEM, O_t += P_t V_j, then S_t = Q_t K_{j+1}^T over the same
        // columns (the tensor core runs one thread's products in order, so PV
        // has read P before QK overwrites it).  While tile t waits for its
        // softmax, the products of the other tiles keep the tensor core busy.
        // Two warps share the tiles so that the issue of one warp's products
        // overlaps the other warp's waits; a K/V stage is released once both
        // have committed their last product on it.  (At T = 2, one warp issuing
        // both tiles' products spent ~44 cycles an instruction, about 1400 of
        // the ~2400 cycles of a key step at d 128.)
        const int mw = warp - C::MMA_WARP;
        constexpr uint32_t idesc_qk = umma_idesc_bf16(BM, BN, false);
        constexpr uint32_t idesc_pv = umma_idesc_bf16(BM, 64, true);
        const uint32_t sq = smem_u32(sQ);
        auto wait_all = [&](uint64_t* bar, uint32_t parity) {
            return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, p.err));
        };
        auto qk = [&](int t, int st, int b) {
            const uint32_t sK = smem_u32(sKV + st * C::STAGE_BYTES);
            const uint32_t sqt = sq + t * C::Q_BYTES;
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
                umma_ss_elect(tmem + C::s_col(t, b),
                              umma_sdesc_sw128(sqt + (ks / 4) * kQChunkBytes + (ks % 4) * 32, 16, 1024),
                              umma_sdesc_sw128(sK + (ks / 4) * kKChunkBytes + (ks % 4) * 32, 16, 1024), idesc_qk,
                              ks > 0 ? 1u : 0u);
            umma_commit_elect(&s_full[C::NB * t + b]);
        };
        auto pv = [&](int t, int st, int b, bool acc) {
            const uint32_t sV = smem_u32(sKV + st * C::STAGE_BYTES) + C::K_BYTES;
#pragma unroll
            for (int ks = 0; ks < BN / 16; ++ks)
#pragma unroll
                for (int c = 0; c < C::KCH; ++c)
                    umma_ts_elect(tmem + C::o_col(t) + 64 * c, tmem + C::p_col(t, b, ks),
                                  umma_sdesc_sw128(sV + c * kKChunkBytes + ks * 2048, 1024, 1024), idesc_pv,
                                  (acc || ks > 0) ? 1u : 0u);
        };
        bool ok = (!SPLIT || nk > 0) && wait_all(ROPE ? q_ready : q_full, 0) && wait_all(&kv_full[0], 0);
        if (ok) {
            tc_fence_after_sync();
#pragma unroll
            for (int t = 0; t < T; ++t)
                if (t % C::MMA_WARPS == mw) qk(t, 0, 0);
        }
        if constexpr (C::NB == 2) {
            // the second buffer: scores of key tile 1 before any P is back
            if (ok && nk > 1) {
                ok = wait_all(&kv_full[1], 0);
                if (ok) {
                    tc_fence_after_sync();
#pragma unroll
                    for (int t = 0; t < T; ++t)
                        if (t % C::MMA_WARPS == mw) qk(t, 1, 1);
                }
            }
        }
        for (int jj = 0; (!SPLIT || C::NB == 2 || ok) && jj < nk; ++jj) {
            if (C::NB == 2 && !ok) break;
            const int st = jj % C::NST;
            const int b = jj % C::NB;  // the buffer holding P of key tile jj
            const int jn = jj + C::NB;  // the key tile whose scores go into that buffer next
            const int stn = jn % C::NST;
            const bool more = jn < nk;
#pragma unroll
            for (int t = 0; t < T; ++t) {
                if (t % C::MMA_WARPS != mw) continue;
                if (!wait_all(&p_full[C::NB * t + b], (jj / C::NB) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                pv(t, st, b, jj > 0);
                if constexpr (C::NB == 2) umma_commit_elect(&pv_done[t]);  // O may be rescaled once it is done
                if (t + C::MMA_WARPS >= T) umma_commit_elect(&kv_empty[st]);  // this warp's last tile
                if (more) {
                    if (t < C::MMA_WARPS) {  // this warp's first tile
                        if (!wait_all(&kv_full[stn], (jn / C::NST) & 1)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after_sync();
                    }
                    qk(t, stn, b);
                } else if (C::NB == 1 || jj == nk - 1) {
                    umma_commit_elect(&o_done[t]);
                }
            }
        }
        umma_commit_elect(&mma_done[mw]);  // every MMA of this warp done before TMEM is freed
        mbar_drain(&mma_done[mw], 0);
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax
        const int t = warp >> 2;
        const int r = (warp & 3) * 32 + lane;  // query row = TMEM lane
        bool ok = true;
        if constexpr (ROPE) {
            const long long pos = static_cast<long long>(pre) + BM * i + r;
            const bool in_chunk = BM * i + r < n;
            const bool turn = in_chunk && pos < p.max_pos;
            if (in_chunk && !turn) set_error(p.err, PA_ERR_BAD_BLOCK);
            ok = rope_q_row<D>(sQ + t * C::Q_BYTES, r, turn, pos, q_full, abort_flag, p);
            __syncwarp();
            if (ok) mbar_arrive_elect(q_ready);
        }
        // in a key split every softmax warp enters, whatever `ok` says: the
        // split's barriers count on it
        if (SPLIT || ok)
            softmax_role<D, T, SPLIT>(t, r, tmem + tmem_lane_base(warp), i, j0, j1, n, pre + BM * i, kv_len,
                                             cu0, hq0 + t, sKV, &s_full[C::NB * t], &p_full[C::NB * t], &o_done[t],
                                             &pv_done[t], kv_full,
                                             abort_flag, split_flag, ok, p);
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == C::MMA_WARP) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
    // Without an abort every copy issued was waited for by the role that uses
    // it.  After one, the copies still in flight land before the CTA leaves
    // (phases already complete return at once).
    if (warp == C::PRODUCER_WARP && lane == 0 && *abort_flag) {
        if (!producer_held_q) mbar_drain(q_full, 0);
        for (int jj = producer_issued > C::NST ? producer_issued - C::NST : 0; jj < producer_issued; ++jj)
            mbar_drain(&kv_full[jj % C::NST], (jj / C::NST) & 1);
    }
    tail_wait();
}

// 2D bf16 tensor [rows][cols] with row pitch `pitch_bytes`, box {64, box_rows},
// 128-byte swizzle, zero fill out of range.
bool encode_2d(CUtensorMap* map, const void* base, unsigned long long cols, unsigned long long rows,
               unsigned long long pitch_bytes, unsigned box_rows) {
    EncodeTiledFn fn = tensor_map_encoder();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {pitch_bytes};
    const cuuint32_t box[2] = {64, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Work items [first, first + count) of the T-heads-per-CTA numbering; `tail`
// launches them as a programmatic dependent of the launch before.
template <int D, int T>
cudaError_t launch(const CUtensorMap& qmap, const CUtensorMap& kvmap, PrefillParams p, long long first,
                   long long count, bool tail, bool has_tail, cudaStream_t stream) {
    using C = Cfg<D, T>;
    auto kern = p.cos_tab ? prefill_kernel<D, T, true, false>
                          : (p.ksplit ? prefill_kernel<D, T, false, true> : prefill_kernel<D, T, false, false>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    if (count <= 0) return cudaSuccess;
    if (first + count > 0x7FFFFFFFll) return cudaErrorInvalidConfiguration;
    p.heads_per_cta = T;
    p.item_base = static_cast<int>(first);
    p.tail = tail ? 1 : 0;
    p.has_tail = has_tail ? 1 : 0;
    const unsigned grid = static_cast<unsigned>(p.ksplit ? 2 * count : count);  // key split: two CTAs an item
    if (!tail) {
        kern<<<grid, C::THREADS, C::SMEM, stream>>>(qmap, kvmap, p);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid, 1, 1);
    cfg.blockDim = dim3(C::THREADS, 1, 1);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, qmap, kvmap, p);
}

// Scratch of a key-split launch, from a memory pool of the library's own per
// device (kept for the process, never released to the system, so that a call
// allocates and frees in stream order at the cost of a pool lookup).
cudaError_t split_scratch(size_t bytes, cudaStream_t stream, void** out) {
    static std::mutex mu;
    static cudaMemPool_t pools[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    cudaMemPool_t pool;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!pools[dev]) {
            cudaMemPoolProps props = {};
            props.allocType = cudaMemAllocationTypePinned;
            props.location.type = cudaMemLocationTypeDevice;
            props.location.id = dev;
            e = cudaMemPoolCreate(&pools[dev], &props);
            if (e != cudaSuccess) return e;
            uint64_t keep = ~0ull;
            e = cudaMemPoolSetAttribute(pools[dev], cudaMemPoolAttrReleaseThreshold, &keep);
            if (e != cudaSuccess) return e;
        }
        pool = pools[dev];
    }
    return cudaMallocFromPoolAsync(out, bytes, pool, stream);
}

// The call's work items with T q heads per CTA, heaviest first.  When they
// make only a few waves over the SMs and the last one is partial, the items of
// that last wave run in a second launch that starts while the first one's last
// wave runs:
// - with a cached prefix (long key ranges) each item as two CTAs of T heads,
//   one per half of its key tiles, whose partials the later one combines;
// - otherwise (or if its scratch cannot be had) with T/2 heads per CTA (each
//   item is exactly two of those, the same rows and kv head).
template <int D, int T>
cudaError_t launch_items(const CUtensorMap& qmap, const CUtensorMap& kvmap, const PrefillParams& p, int sms,
                         cudaStream_t stream) {
    const long long n = static_cast<long long>(p.n_row_tiles) * p.batch * (p.g.hq / T);
    constexpr int kFewWaves = 8;
    if (T == 1 || sms <= 0 || n % sms == 0 || n >= static_cast<long long>(kFewWaves) * sms)
        return launch<D, T>(qmap, kvmap, p, 0, n, false, false, stream);
    constexpr int TH = T > 1 ? T / 2 : 1;
    const long long full = n / sms * sms;  // items of the whole waves
    const long long rest = n - full;
    void* ws = nullptr;
    PrefillParams ps = p;
    if (p.prefix && !p.cos_tab) {
        const size_t o_bytes = static_cast<size_t>(rest) * 2 * T * BM * D * sizeof(float);
        const size_t ml_bytes = static_cast<size_t>(rest) * 2 * T * BM * sizeof(float2);
        if (split_scratch(o_bytes + ml_bytes + static_cast<size_t>(rest) * sizeof(int), stream, &ws) == cudaSuccess) {
            ps.ksplit = 1;
            ps.ws_o = static_cast<float*>(ws);
            ps.ws_ml = reinterpret_cast<float2*>(static_cast<uint8_t*>(ws) + o_bytes);
            ps.ws_cnt = reinterpret_cast<int*>(static_cast<uint8_t*>(ws) + o_bytes + ml_bytes);
            cudaError_t e = cudaMemsetAsync(ps.ws_cnt, 0, static_cast<size_t>(rest) * sizeof(int), stream);
            if (e != cudaSuccess) {
                cudaFreeAsync(ws, stream);
                return e;
            }
        } else {
            (void)cudaGetLastError();  // no scratch: the head split needs none
            ws = nullptr;
        }
    }
    cudaError_t e = launch<D, T>(qmap, kvmap, p, 0, full, false, true, stream);
    if (e == cudaSuccess)
        e = ws ? launch<D, T>(qmap, kvmap, ps, full, rest, full > 0, false, stream)
               : launch<D, TH>(qmap, kvmap, p, 2 * full, 2 * rest, full > 0, false, stream);
    if (ws) {
        const cudaError_t f = cudaFreeAsync(ws, stream);
        if (e == cudaSuccess) e = f;
    }
    return e;
}

}  // namespace

cudaError_t launch_prefill(const KGeom& g, const void* q, const void* pool, const int32_t* block_table, int layer,
                           int batch, const int32_t* cu_seqlens, const int32_t* prefix_lens, const int32_t* slots,
                           int max_seqlen, int total_tokens, float scale, void* o, float* lse, int32_t* err,
                           cudaStream_t stream, const float* cos_tab, const float* sin_tab, int max_pos) {
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
    p.prefix = prefix_lens;
    p.slots = slots;
    p.max_seqlen = max_seqlen;
    p.total_tokens = total_tokens;
    p.n_row_tiles = (max_seqlen + BM - 1) / BM;
    // q heads per CTA: as many of one GQA group as tensor memory holds (S and O
    // of every tile: 4 at d 64, 2 at d 128)
    const int tmax = g.d == 64 ? 4 : 2;
    p.heads_per_cta = (g.group % 4 == 0 && tmax >= 4) ? 4 : (g.group % 2 == 0) ? 2 : 1;
    p.scale_log2 = scale * kLog2e;
    p.o = static_cast<__nv_bfloat16*>(o);
    p.o_32b = (reinterpret_cast<uintptr_t>(o) & 31u) == 0;
    p.lse = lse;
    p.err = err;
    p.cos_tab = cos_tab;
    p.sin_tab = sin_tab;
    p.max_pos = max_pos;
    p.hold_first_copy = debug_hold_first_copy();
    p.item_base = 0;
    p.tail = 0;
    p.has_tail = 0;
    p.ksplit = 0;
    p.ws_o = nullptr;
    p.ws_ml = nullptr;
    p.ws_cnt = nullptr;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (g.d == 64) {
        if (p.heads_per_cta == 4) return launch_items<64, 4>(qmap, kvmap, p, sms, stream);
        if (p.heads_per_cta == 2) return launch_items<64, 2>(qmap, kvmap, p, sms, stream);
        return launch_items<64, 1>(qmap, kvmap, p, sms, stream);
    }
    if (p.heads_per_cta == 2) return launch_items<128, 2>(qmap, kvmap, p, sms, stream);
    return launch_items<128, 1>(qmap, kvmap, p, sms, stream);
}

}  // namespace pa

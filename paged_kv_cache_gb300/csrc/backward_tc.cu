// backward_tc.cu -- the column-block kernel of the prefill backward on the
// sm_103a tensor cores (tcgen05.mma, accumulators in tensor memory, operands
// staged by TMA), head dims 64 and 128.
//
// The arithmetic (FlashAttention-2 explainer, "전체
// 흐름": P rebuilt from L; "2. 시퀀스 길이 방향으로도 병렬화" item 4: one
// thread block per key block, dQ added atomically; "4. MQA · GQA 지원": dK, dV
// summed over the group):
//   S^T = K Q^T, dP^T = V dO^T, P^T = e^(scale S^T - L), dS^T = P^T (dP^T - D),
//   dV += P^T dO, dK += dS^T Q, dQ += dS K.
//
// One CTA per (128-key block, sequence, kv head); the key block's K and V stay
// in shared memory and its dK, dV accumulate in tensor memory over every q head
// of the group and every 64-row query block at or after the diagonal.
//  * warp 0 (producer): K, V once (8 pages each, rows through the block table,
//    pages past the end read at an out-of-range row = zeros); then per query
//    block the Q and dO tiles by TMA and -L log2 e, -D (from the prep kernel's
//    workspace) by cp.async, all completing on one mbarrier, into 5 stages
//    (2 at d 128).
//  * warp 1 (MMA issue, elected lane): S^T and dP^T (M 128 keys, N 64 rows,
//    K d dims, both operands K-major) into one of two TMEM buffers; once the
//    elementwise warps hand back P^T and dS^T (bf16, in TMEM over the first
//    8 columns of each 16-column quarter), dV += P^T dO and dK += dS^T Q (A from
//    TMEM, B = the same Q / dO tiles read MN-major, N = d); after every second
//    query block, dQ = dS K for the pair (M 128 rows, N d, K 128 keys; dS from
//    shared memory MN-major, K read MN-major).  At d 64 S^T of the next block
//    is issued before dV / dK of this one, so the tensor core works while the
//    elementwise warps run; at d 128, whose dV, dK and dQ take 384 columns,
//    there is one S^T / dP^T buffer and one dQ buffer, and the next S^T
//    follows dV / dK.  At d 64 a second issuing warp (warp 22) takes dV, dK
//    and dQ, so that S^T / dP^T of the next block need not wait behind them
//    in one warp's issue order; the first issuer refills a buffer once the
//    dV / dK products that read it are done (a barrier per buffer).
//  * warps 2..17 (elementwise): thread = key (TMEM lane), four warps per lane
//    quarter, 16 query rows each.  Mask j <= i < n, P^T, dS^T; P^T and dS^T to
//    TMEM, dS^T also to shared memory (key rows of 64 query rows, 128-byte
//    swizzle) for the dQ product.  Rows of Q / dO past the sequence and K rows
//    past it are zeroed in shared memory first (masked weights are exactly 0,
//    0 x NaN is not).
//  * warps 18..21 (dQ epilogue): thread = query row; dQ of a pair from TMEM,
//    times scale, into a swizzled fp32 staging tile, then one TMA reduce-add
//    per 32 columns into dq (rows past the sequence add zeros; rows past the
//    tensor are clipped).  At the end they write dK * scale and dV.
// TMEM, d 64: S^T 2 x 64 columns, dP^T 2 x 64, dQ 2 x 64, dV 64, dK 64;
// d 128: S^T 64, dP^T 64, dQ 128, dV 128, dK 128 (512 either way).
// Every wait is bounded; on a timeout the CTA records PA_ERR_TIMEOUT, drains
// its copies and products in flight and frees its tensor memory.
#include "pa_internal.cuh"

namespace pa {
namespace {

constexpr int kKeys = 128;        // keys per CTA: TMEM lanes of the key-side products
constexpr int kRowsIt = 64;       // query rows per iteration
constexpr int kProducerWarp = 0;
constexpr int kMmaWarp = 1;
constexpr int kEwWarp0 = 2;       // 16 elementwise warps
constexpr int kEwWarps = 16;
constexpr int kEpiWarp0 = kEwWarp0 + kEwWarps;  // 4 dQ epilogue warps
constexpr int kMmaWarp2 = kEpiWarp0 + 4;         // two issuers: dV, dK and dQ (kMmaWarp: S^T, dP^T)
constexpr int kDsHalf = kKeys * 128;    // dS^T of 64 query rows for 128 keys
constexpr int kDsBuf = 2 * kDsHalf;     // one pair of query blocks
constexpr int kDqBox = 128 * 128;       // 128 rows x 32 fp32
constexpr uint32_t kTmemCols = 512;

template <int D>
struct TcCfg {
    static constexpr int KCH = D / 64;              // 64-dim chunks of a row (128-byte swizzle atoms)
    static constexpr int NBUF = D == 64 ? 2 : 1;    // S^T / dP^T buffers in TMEM
    static constexpr int NDQ = D == 64 ? 2 : 1;     // dQ buffers in TMEM
    static constexpr int NST = D == 64 ? 5 : 2;     // Q / dO / L / D stages
    // Two issuing warps where there are two S^T / dP^T buffers: S^T / dP^T of
    // the next block go out while the other warp issues this block's dV, dK
    // and dQ (d 64: 755 -> 771 TFLOP/s).  With one buffer the next S^T must
    // wait for dV / dK to complete instead of merely following them in one
    // thread's issue order (d 128: 863 -> 791), so d 128 keeps one issuer.
    static constexpr bool TWO_ISSUERS = NBUF == 2;
    static constexpr int THREADS = (kEpiWarp0 + 4 + (TWO_ISSUERS ? 1 : 0)) * 32;
    static constexpr int DQ_BOXES = D == 64 ? 2 : 1;  // 32-column fp32 staging boxes
    static constexpr int KV_CHUNK = kKeys * 128;    // one chunk of the K (or V) tile
    static constexpr int TILE_KV = KCH * KV_CHUNK;
    static constexpr int Q_CHUNK = kRowsIt * 128;   // one chunk of a Q (or dO) tile
    static constexpr int TILE_Q = KCH * Q_CHUNK;
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = TILE_KV;
    static constexpr int OFF_Q = 2 * TILE_KV;                 // [NST]
    static constexpr int OFF_DO = OFF_Q + NST * TILE_Q;       // [NST]
    static constexpr int OFF_DS = OFF_DO + NST * TILE_Q;      // [2] pairs
    static constexpr int OFF_DQ = OFF_DS + 2 * kDsBuf;        // DQ_BOXES boxes
    static constexpr int OFF_LD = OFF_DQ + DQ_BOXES * kDqBox; // [NST] x (64 -L log2e, 64 -D) fp32
    static constexpr int OFF_BAR = OFF_LD + NST * 2 * kRowsIt * 4;
    static constexpr int SMEM = 1024 + OFF_BAR + 512;
    static_assert(SMEM <= 227 * 1024, "shared memory");
    static constexpr uint32_t COL_S = 0;                 // [NBUF] x 64
    static constexpr uint32_t COL_DP = 64 * NBUF;        // [NBUF] x 64
    static constexpr uint32_t COL_DQ = 128 * NBUF;       // [NDQ] x D
    static constexpr uint32_t COL_DV = COL_DQ + NDQ * D;
    static constexpr uint32_t COL_DK = COL_DV + D;
    static_assert(COL_DK + D == kTmemCols, "tensor memory");
};

struct BwdTcParams {
    KGeom g;
    const int32_t* bt;
    int layer;
    const int32_t* cu;
    const int32_t* slots;
    int max_seqlen;
    int total_tokens;
    const float* ws;        // [2][total_tokens][hq]: -L log2 e, -D
    long long ws_half;
    float scale;
    float scale_log2;
    float* dk;
    float* dv;
    bool kv_32b;            // dk and dv 32-byte aligned: rows go out in whole 32-byte sectors
    int32_t* err;
};

// Columns of the bf16 P^T (or dS^T) of query rows 16 ks .. 16 ks + 15 within a
// 64-column buffer: each 16-row quarter keeps its 8 packed columns at its start.
__device__ __forceinline__ uint32_t packed_col(int ks) { return 16u * ks; }

__device__ __forceinline__ void st_shared_v4(uint32_t saddr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(saddr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}
__device__ __forceinline__ void st_shared_v4f(uint32_t saddr, float a, float b, float c, float d) {
    asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(saddr), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}
__device__ __forceinline__ void epi_barrier() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
// Barrier of the four epilogue warps that also ANDs a flag over their threads,
// so that all four leave a loop together.
__device__ __forceinline__ bool epi_all(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, 1, 128, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(v))
        : "memory");
    return r != 0;
}

__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap* map, int x, int y, uint32_t ssrc) {
    asm volatile(
        "cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(x), "r"(y), "r"(ssrc)
        : "memory");
}
// 4 bytes global -> shared, zero-filled when `bytes` is 0 (nothing is read then).
__device__ __forceinline__ void cp_async4_zfill(uint32_t sdst, const float* gsrc, uint32_t bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(sdst), "l"(gsrc), "r"(bytes) : "memory");
}
// Arrives on `bar` once every cp.async this thread issued so far has landed
// (the arrival is counted in the barrier's expected count).
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Zeroes 128-byte rows [r0, r1) of a tile (the swizzle only permutes 16-byte
// chunks within a row), spread over `nthr` threads.
__device__ __forceinline__ void zero_rows(uint32_t tile, int r0, int r1, int t, int nthr) {
    for (int c = t; c < (r1 - r0) * 8; c += nthr) st_shared_v4(tile + (r0 + c / 8) * 128 + (c % 8) * 16, 0, 0, 0, 0);
}

template <int D>
__global__ void __launch_bounds__(TcCfg<D>::THREADS, 1)
bwd_tc_kernel(const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap domap,
              const __grid_constant__ CUtensorMap kvmap, const __grid_constant__ CUtensorMap dqmap,
              const BwdTcParams p) {
    using C = TcCfg<D>;
    constexpr int kNst = C::NST;
    constexpr int OFF_K = C::OFF_K, OFF_V = C::OFF_V, OFF_Q = C::OFF_Q, OFF_DO = C::OFF_DO, OFF_DS = C::OFF_DS,
                  OFF_DQ = C::OFF_DQ, OFF_LD = C::OFF_LD, OFF_BAR = C::OFF_BAR;
    constexpr int kTileQ = C::TILE_Q;
    constexpr uint32_t COL_S = C::COL_S, COL_DP = C::COL_DP, COL_DQ = C::COL_DQ, COL_DV = C::COL_DV,
                       COL_DK = C::COL_DK;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    const uint32_t sb = smem_u32(smem);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    uint64_t* kv_full = bars;              // 1
    uint64_t* q_full = kv_full + 1;        // [kNst]
    uint64_t* q_empty = q_full + kNst;     // [kNst]
    uint64_t* s_full = q_empty + kNst;     // [2]
    uint64_t* p_ready = s_full + 2;        // [2]
    uint64_t* ds_empty = p_ready + 2;      // [2]
    uint64_t* dq_full = ds_empty + 2;      // [2]
    uint64_t* dq_empty = dq_full + 2;      // [2]
    uint64_t* kv_done = dq_empty + 2;      // 1: last dV / dK product done
    uint64_t* mma_done = kv_done + 1;      // 1: every product done
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(mma_done + 2);
    uint64_t* buf_free = mma_done + 3;     // [2] (two issuers): dV / dK of the buffer's block done
    uint64_t* mma_done2 = mma_done + 5;    // 1 (two issuers): every product of the second issuer done
    float* sLD = reinterpret_cast<float*>(smem + OFF_LD);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const KGeom& g = p.g;
    const int b = blockIdx.x / g.hkv, hk = blockIdx.x % g.hkv;
    const int jb = blockIdx.y;
    const int cu0 = p.cu[b], cu1 = p.cu[b + 1];
    const int n = cu1 - cu0;
    const bool bad_len = cu0 < 0 || n < 0 || cu1 > p.total_tokens || n > p.max_seqlen ||
                         n > g.maxb * kBlockTokens;
    if (jb == 0 && hk == 0 && tid == 0 && bad_len) set_error(p.err, PA_ERR_BAD_BLOCK);
    if (bad_len || jb * kKeys >= n) return;
    const int slot = p.slots[b];
    if (slot < 0 || slot >= g.num_slots) {
        if (jb == 0 && hk == 0 && tid == 0) set_error(p.err, PA_ERR_BAD_BLOCK);
        return;
    }
    const int group = g.group;
    const int nph = (n + 2 * kRowsIt - 1) / (2 * kRowsIt) - jb;  // query-block pairs per head
    const int n_it = group * 2 * nph;                            // iterations: (head, pair, half)
    const int n_pairs = group * nph;

    if (tid == 0) {
        mbar_init(kv_full, 1);
        for (int s = 0; s < kNst; ++s) {
            mbar_init(&q_full[s], 1 + 32);  // expect_tx arrival + one cp.async arrival per producer lane
            mbar_init(&q_empty[s], C::TWO_ISSUERS ? 2 : 1);  // (two issuers: S^T / dP^T and dV / dK read it)
        }
        for (int x = 0; x < 2; ++x) {
            mbar_init(&s_full[x], 1);
            mbar_init(&p_ready[x], kEwWarps * 32);
            mbar_init(&ds_empty[x], 1);
            mbar_init(&dq_full[x], 1);
            mbar_init(&dq_empty[x], 4 * 32);
        }
        mbar_init(kv_done, 1);
        mbar_init(mma_done, 1);
        mbar_init(mma_done2, 1);
        for (int x = 0; x < 2; ++x) mbar_init(&buf_free[x], 1);
        *abort_flag = 0;
        mbar_init_fence();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    if (warp == kProducerWarp) {
        // ------------------------------------------------------------ producer
        const long long tbase = (static_cast<long long>(slot) * g.n_layers + p.layer) * g.maxb;
        const int pages_b = (n + kBlockTokens - 1) / kBlockTokens;
        const int oob_row = static_cast<int>(g.nblocks * 32);
        const int lp = jb * (kKeys / kBlockTokens) + lane;
        int row = -1;
        if (lane < kKeys / kBlockTokens && lp < pages_b) {
            const int e = __ldg(p.bt + tbase + lp);
            if (e >= 0 && e < g.nblocks)
                row = e * 32;
            else
                set_error(p.err, PA_ERR_BAD_BLOCK);
        }
        if (lane == 0) {
            prefetch_tensor_map(&qmap);
            prefetch_tensor_map(&domap);
            prefetch_tensor_map(&kvmap);
            mbar_arrive_expect_tx(kv_full, 2 * C::TILE_KV);
        }
#pragma unroll
        for (int k = 0; k < kKeys / kBlockTokens; ++k) {
            const int rr = __shfl_sync(0xffffffffu, row, k);
            if (lane == 0) {
                const int y = rr < 0 ? oob_row : rr;
#pragma unroll
                for (int c = 0; c < C::KCH; ++c) {
                    tma_load_2d(smem + OFF_K + c * C::KV_CHUNK + k * 2048, &kvmap, hk * D + 64 * c, y, kv_full);
                    tma_load_2d(smem + OFF_V + c * C::KV_CHUNK + k * 2048, &kvmap, hk * D + 64 * c, y + 16, kv_full);
                }
            }
        }
        int issued = 0;
        for (int it = 0; it < n_it; ++it) {
            const int s = it % kNst;
            if (it >= kNst &&
                !__all_sync(0xffffffffu, mbar_wait(&q_empty[s], ((it / kNst) - 1) & 1, abort_flag, p.err)))
                break;
            const int pp = it >> 1;
            const int h = hk * group + pp / nph;
            const int ib = 2 * (jb + pp % nph) + (it & 1);
            const uint32_t ld = sb + OFF_LD + s * 2 * kRowsIt * 4;
#pragma unroll
            for (int x = 0; x < 2; ++x) {
                const int r = lane + 32 * x;
                const int i = ib * kRowsIt + r;
                const float* src = p.ws + (i < n ? static_cast<long long>(cu0 + i) * g.hq + h : 0);
                const uint32_t bytes = i < n ? 4u : 0u;
                cp_async4_zfill(ld + r * 4, src, bytes);
                cp_async4_zfill(ld + (kRowsIt + r) * 4, src + p.ws_half, bytes);
            }
            cp_async_arrive_noinc(&q_full[s]);
            if (lane == 0) {
                mbar_arrive_expect_tx(&q_full[s], 2 * kTileQ);
#pragma unroll
                for (int c = 0; c < C::KCH; ++c) {
                    tma_load_2d(smem + OFF_Q + s * kTileQ + c * C::Q_CHUNK, &qmap, h * D + 64 * c, cu0 + ib * kRowsIt,
                                &q_full[s]);
                    tma_load_2d(smem + OFF_DO + s * kTileQ + c * C::Q_CHUNK, &domap, h * D + 64 * c,
                                cu0 + ib * kRowsIt, &q_full[s]);
                }
            }
            ++issued;
        }
        if (lane == 0) {  // every copy issued has landed before the CTA leaves
            mbar_drain(kv_full, 0);
            for (int it = issued > kNst ? issued - kNst : 0; it < issued; ++it)
                mbar_drain(&q_full[it % kNst], (it / kNst) & 1);
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issue
        constexpr uint32_t idesc_t = umma_idesc_bf16(128, 64, false);        // S^T, dP^T
        constexpr uint32_t idesc_kv = umma_idesc_bf16(128, D, true);         // dV, dK (A from TMEM)
        constexpr uint32_t idesc_q = umma_idesc_bf16(128, D, true, true);    // dQ
        auto wait_all = [&](uint64_t* bar, uint32_t parity) {
            return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, p.err));
        };
        const uint32_t sK = sb + OFF_K, sV = sb + OFF_V;
        auto issue_sdp = [&](int it) {
            const int s = it % kNst, x = it % C::NBUF;
            const uint32_t sQ = sb + OFF_Q + s * kTileQ, sO = sb + OFF_DO + s * kTileQ;
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
                umma_ss_elect(tmem + COL_S + 64 * x,
                              umma_sdesc_sw128(sK + (ks >> 2) * C::KV_CHUNK + (ks & 3) * 32, 16, 1024),
                              umma_sdesc_sw128(sQ + (ks >> 2) * C::Q_CHUNK + (ks & 3) * 32, 16, 1024), idesc_t,
                              ks > 0 ? 1u : 0u);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
                umma_ss_elect(tmem + COL_DP + 64 * x,
                              umma_sdesc_sw128(sV + (ks >> 2) * C::KV_CHUNK + (ks & 3) * 32, 16, 1024),
                              umma_sdesc_sw128(sO + (ks >> 2) * C::Q_CHUNK + (ks & 3) * 32, 16, 1024), idesc_t,
                              ks > 0 ? 1u : 0u);
            umma_commit_elect(&s_full[x]);
        };
        if constexpr (C::TWO_ISSUERS) {
            // S^T / dP^T of block it into buffer it % NBUF once the dV / dK
            // products of the block before in that buffer are done
            bool ok = wait_all(kv_full, 0);
            for (int it = 0; ok && it < n_it; ++it) {
                const int s = it % kNst, x = it % C::NBUF;
                if (it >= C::NBUF && !wait_all(&buf_free[x], ((it - C::NBUF) / C::NBUF) & 1)) {
                    ok = false;
                    break;
                }
                if (!wait_all(&q_full[s], (it / kNst) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                issue_sdp(it);
                umma_commit_elect(&q_empty[s]);
            }
        } else {
            bool ok = wait_all(kv_full, 0) && wait_all(&q_full[0], 0);
            if (ok) {
                tc_fence_after_sync();
                issue_sdp(0);
            }
            // the next block's S^T / dP^T: into the other buffer before this block's dV / dK
            // (two buffers), or after them, over the P^T / dS^T they read (one buffer)
            auto next_sdp = [&](int it) {
                if (it + 1 >= n_it) return true;
                if (!wait_all(&q_full[(it + 1) % kNst], ((it + 1) / kNst) & 1)) return false;
                tc_fence_after_sync();
                issue_sdp(it + 1);
                return true;
            };
            for (int it = 0; ok && it < n_it; ++it) {
                const int s = it % kNst, x = it % C::NBUF;
                if (C::NBUF == 2 && !next_sdp(it)) {
                    ok = false;
                    break;
                }
                if (!wait_all(&p_ready[x], (it / C::NBUF) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t sQ = sb + OFF_Q + s * kTileQ, sO = sb + OFF_DO + s * kTileQ;
    #pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    umma_ts_elect(tmem + COL_DV, tmem + COL_S + 64 * x + packed_col(ks),
                                  umma_sdesc_sw128(sO + ks * 2048, C::Q_CHUNK, 1024), idesc_kv,
                                  (it > 0 || ks > 0) ? 1u : 0u);
    #pragma unroll
                for (int ks = 0; ks < 4; ++ks)
                    umma_ts_elect(tmem + COL_DK, tmem + COL_DP + 64 * x + packed_col(ks),
                                  umma_sdesc_sw128(sQ + ks * 2048, C::Q_CHUNK, 1024), idesc_kv,
                                  (it > 0 || ks > 0) ? 1u : 0u);
                umma_commit_elect(&q_empty[s]);
                if (it + 1 == n_it) umma_commit_elect(kv_done);
                if (C::NBUF == 1 && !next_sdp(it)) {
                    ok = false;
                    break;
                }
                if (it & 1) {
                    const int pp = it >> 1, y = pp % C::NDQ, dsb = pp & 1;
                    if (pp >= C::NDQ && !wait_all(&dq_empty[y], ((pp / C::NDQ) - 1) & 1)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint32_t sD = sb + OFF_DS + dsb * kDsBuf;
    #pragma unroll
                    for (int ks = 0; ks < kKeys / 16; ++ks)
                        umma_ss_elect(tmem + COL_DQ + D * y, umma_sdesc_sw128(sD + ks * 2048, kDsHalf, 1024),
                                      umma_sdesc_sw128(sK + ks * 2048, C::KV_CHUNK, 1024), idesc_q, ks > 0 ? 1u : 0u);
                    umma_commit_elect(&dq_full[y]);
                    umma_commit_elect(&ds_empty[dsb]);
                }
            }
        }
        umma_commit_elect(mma_done);
        mbar_drain(mma_done, 0);
        __syncwarp();
    } else if (C::TWO_ISSUERS && warp == kMmaWarp2) {
        // ------------------------------------------------------------ dV, dK, dQ issue (two issuers)
        constexpr uint32_t idesc_kv = umma_idesc_bf16(128, D, true);         // dV, dK (A from TMEM)
        constexpr uint32_t idesc_q = umma_idesc_bf16(128, D, true, true);    // dQ
        auto wait_all = [&](uint64_t* bar, uint32_t parity) {
            return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort_flag, p.err));
        };
        const uint32_t sK = sb + OFF_K;
        bool ok = wait_all(kv_full, 0);
        for (int it = 0; ok && it < n_it; ++it) {
            const int s = it % kNst, x = it % C::NBUF;
            if (!wait_all(&q_full[s], (it / kNst) & 1) || !wait_all(&p_ready[x], (it / C::NBUF) & 1)) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
            const uint32_t sQ = sb + OFF_Q + s * kTileQ, sO = sb + OFF_DO + s * kTileQ;
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                umma_ts_elect(tmem + COL_DV, tmem + COL_S + 64 * x + packed_col(ks),
                              umma_sdesc_sw128(sO + ks * 2048, C::Q_CHUNK, 1024), idesc_kv,
                              (it > 0 || ks > 0) ? 1u : 0u);
#pragma unroll
            for (int ks = 0; ks < 4; ++ks)
                umma_ts_elect(tmem + COL_DK, tmem + COL_DP + 64 * x + packed_col(ks),
                              umma_sdesc_sw128(sQ + ks * 2048, C::Q_CHUNK, 1024), idesc_kv,
                              (it > 0 || ks > 0) ? 1u : 0u);
            umma_commit_elect(&q_empty[s]);
            umma_commit_elect(&buf_free[x]);  // S^T / dP^T of block it + NBUF may overwrite this buffer
            if (it + 1 == n_it) umma_commit_elect(kv_done);
            if (it & 1) {
                const int pp = it >> 1, y = pp % C::NDQ, dsb = pp & 1;
                if (pp >= C::NDQ && !wait_all(&dq_empty[y], ((pp / C::NDQ) - 1) & 1)) {
                    ok = false;
                    break;
                }
                tc_fence_after_sync();
                const uint32_t sD = sb + OFF_DS + dsb * kDsBuf;
#pragma unroll
                for (int ks = 0; ks < kKeys / 16; ++ks)
                    umma_ss_elect(tmem + COL_DQ + D * y, umma_sdesc_sw128(sD + ks * 2048, kDsHalf, 1024),
                                  umma_sdesc_sw128(sK + ks * 2048, C::KV_CHUNK, 1024), idesc_q, ks > 0 ? 1u : 0u);
                umma_commit_elect(&dq_full[y]);
                umma_commit_elect(&ds_empty[dsb]);
            }
        }
        umma_commit_elect(mma_done2);
        mbar_drain(mma_done2, 0);
        __syncwarp();
    } else if (warp < kEpiWarp0) {
        // ------------------------------------------------------------ elementwise
        const int ew = warp - kEwWarp0;          // 0..15
        const int grp = ew >> 2;                 // query rows 16 grp .. 16 grp + 15 of a block
        const int kq = (warp & 3) * 32 + lane;   // key within the block = TMEM lane
        const int key = jb * kKeys + kq;
        const uint32_t lane_addr = tmem + tmem_lane_base(warp);
        const int et = ew * 32 + lane;           // 0 .. 511
        constexpr int kEt = kEwWarps * 32;
        const float sc = p.scale_log2;
        bool ok = __all_sync(0xffffffffu, mbar_wait(kv_full, 0, abort_flag, p.err));
        if (ok && (jb + 1) * kKeys > n) {  // K rows past the sequence: zero (dQ reads them)
#pragma unroll
            for (int c = 0; c < C::KCH; ++c) zero_rows(sb + OFF_K + c * C::KV_CHUNK, n - jb * kKeys, kKeys, et, kEt);
            fence_proxy_async_smem();
        }
        for (int it = 0; ok && it < n_it; ++it) {
            const int s = it % kNst, x = it % C::NBUF, pp = it >> 1;
            const int ib = 2 * (jb + pp % nph) + (it & 1);
            if (!__all_sync(0xffffffffu, mbar_wait(&s_full[x], (it / C::NBUF) & 1, abort_flag, p.err)) ||
                !__all_sync(0xffffffffu, mbar_wait(&q_full[s], (it / kNst) & 1, abort_flag, p.err))) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
            uint32_t sv[16], dv[16];
            tmem_ld_x16_nowait(lane_addr + COL_S + 64 * x + 16 * grp, sv);
            tmem_ld_x16_nowait(lane_addr + COL_DP + 64 * x + 16 * grp, dv);
            if ((ib + 1) * kRowsIt > n) {  // Q / dO rows past the sequence: zero (dK, dV read them)
                const int r0 = max(0, n - ib * kRowsIt);
#pragma unroll
                for (int c = 0; c < C::KCH; ++c) {
                    zero_rows(sb + OFF_Q + s * kTileQ + c * C::Q_CHUNK, r0, kRowsIt, et, kEt);
                    zero_rows(sb + OFF_DO + s * kTileQ + c * C::Q_CHUNK, r0, kRowsIt, et, kEt);
                }
            }
            const float4* nl4 = reinterpret_cast<const float4*>(sLD + s * 2 * kRowsIt + 16 * grp);
            const float4* nd4 = reinterpret_cast<const float4*>(sLD + s * 2 * kRowsIt + kRowsIt + 16 * grp);
            float nl[16], nd[16];
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const float4 a = nl4[v], c = nd4[v];
                nl[4 * v] = a.x; nl[4 * v + 1] = a.y; nl[4 * v + 2] = a.z; nl[4 * v + 3] = a.w;
                nd[4 * v] = c.x; nd[4 * v + 1] = c.y; nd[4 * v + 2] = c.z; nd[4 * v + 3] = c.w;
            }
            const int row0 = ib * kRowsIt + 16 * grp;
            tmem_wait_ld_dep(sv);
            tmem_wait_ld_dep(dv);
            uint32_t pk[8], dk[8];
            const bool full = key <= row0 && row0 + 15 < n;  // no element masked (warp-uniform off the diagonal)
#pragma unroll
            for (int e = 0; e < 16; e += 2) {
                float x0, x1, t0, t1, d0, d1;
                ffma2(x0, x1, __uint_as_float(sv[e]), __uint_as_float(sv[e + 1]), sc, sc, nl[e], nl[e + 1]);
                float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                fadd2(t0, t1, __uint_as_float(dv[e]), __uint_as_float(dv[e + 1]), nd[e], nd[e + 1]);
                fmul2(d0, d1, p0, p1, t0, t1);
                if (!full) {
                    const bool v0 = key <= row0 + e && row0 + e < n;
                    const bool v1 = key <= row0 + e + 1 && row0 + e + 1 < n;
                    p0 = v0 ? p0 : 0.f;
                    d0 = v0 ? d0 : 0.f;
                    p1 = v1 ? p1 : 0.f;
                    d1 = v1 ? d1 : 0.f;
                }
                pk[e >> 1] = pack_bf16x2(p0, p1);
                dk[e >> 1] = pack_bf16x2(d0, d1);
            }
            tmem_st_x8_nowait(lane_addr + COL_S + 64 * x + 16 * grp, pk);
            tmem_st_x8_nowait(lane_addr + COL_DP + 64 * x + 16 * grp, dk);
            // dS^T of this key into the pair's dQ operand: query rows 64 (it & 1) + 16 grp + ..
            if ((it & 1) == 0 && pp >= 2 &&
                !__all_sync(0xffffffffu, mbar_wait(&ds_empty[pp & 1], ((pp >> 1) - 1) & 1, abort_flag, p.err))) {
                tmem_wait_st();
                ok = false;
                break;
            }
            const uint32_t drow = sb + OFF_DS + (pp & 1) * kDsBuf + (it & 1) * kDsHalf + kq * 128;
#pragma unroll
            for (int c = 0; c < 2; ++c)
                st_shared_v4(drow + (((2 * grp + c) ^ (kq & 7)) * 16), dk[4 * c], dk[4 * c + 1], dk[4 * c + 2],
                             dk[4 * c + 3]);
            tmem_wait_st();
            tc_fence_before_sync();
            fence_proxy_async_smem();
            mbar_arrive(&p_ready[x]);
        }
    } else {
        // ------------------------------------------------------------ dQ epilogue, then dK / dV
        const int r = (warp & 3) * 32 + lane;   // query row within a pair = TMEM lane
        const uint32_t lane_addr = tmem + tmem_lane_base(warp);
        const bool leader = warp == kEpiWarp0 && lane == 0;
        bool ok = true;
        for (int pp = 0; ok && pp < n_pairs; ++pp) {
            const int y = pp % C::NDQ;
            if (!epi_all(mbar_wait(&dq_full[y], (pp / C::NDQ) & 1, abort_flag, p.err))) {
                ok = false;
                break;
            }
            tc_fence_after_sync();
            const int h = hk * group + pp / nph;
            const int y0 = cu0 + (jb + pp % nph) * 2 * kRowsIt;
            const uint32_t row_addr = sb + OFF_DQ + r * 128;
            // D / 32 column groups of 32, staged DQ_BOXES at a time and each added by one reduce
#pragma unroll
            for (int part0 = 0; part0 < D / 32; part0 += C::DQ_BOXES) {
                if (leader) bulk_wait_read0();  // the previous reduce has read the staging tile
                epi_barrier();
#pragma unroll
                for (int bx = 0; bx < C::DQ_BOXES; ++bx) {
                    uint32_t v[32];
                    tmem_ld_x32(lane_addr + COL_DQ + D * y + 32 * (part0 + bx), v);
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch)
                        st_shared_v4f(row_addr + bx * kDqBox + ((ch ^ (r & 7)) * 16), p.scale * __uint_as_float(v[4 * ch]),
                                      p.scale * __uint_as_float(v[4 * ch + 1]), p.scale * __uint_as_float(v[4 * ch + 2]),
                                      p.scale * __uint_as_float(v[4 * ch + 3]));
                }
                if (part0 + C::DQ_BOXES >= D / 32) {  // dQ of this pair is out of tensor memory
                    tc_fence_before_sync();
                    mbar_arrive(&dq_empty[y]);
                }
                fence_proxy_async_smem();
                epi_barrier();
                if (leader) {
#pragma unroll
                    for (int bx = 0; bx < C::DQ_BOXES; ++bx)
                        tma_reduce_add_2d(&dqmap, h * D + 32 * (part0 + bx), y0, sb + OFF_DQ + bx * kDqBox);
                    bulk_commit();
                }
            }
        }
        if (leader) bulk_wait0();
        if (ok && __all_sync(0xffffffffu, mbar_wait(kv_done, 0, abort_flag, p.err))) {
            tc_fence_after_sync();
            const int j = jb * kKeys + r;
            uint32_t a[32], c[32];
#pragma unroll
            for (int part = 0; part < D / 32; ++part) {
                tmem_ld_x32_nowait(lane_addr + COL_DK + 32 * part, a);
                tmem_ld_x32_nowait(lane_addr + COL_DV + 32 * part, c);
                tmem_wait_ld_dep(a);
                tmem_wait_ld_dep(c);
                if (j < n && p.kv_32b) {
                    const long long off = (static_cast<long long>(cu0 + j) * g.hkv + hk) * D + 32 * part;
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        uint32_t vk[8], vv[8];
#pragma unroll
                        for (int w = 0; w < 8; ++w) {
                            vk[w] = __float_as_uint(p.scale * __uint_as_float(a[8 * q + w]));
                            vv[w] = c[8 * q + w];
                        }
                        st_global_v8(p.dk + off + 8 * q, vk);
                        st_global_v8(p.dv + off + 8 * q, vv);
                    }
                } else if (j < n) {
                    const long long off = (static_cast<long long>(cu0 + j) * g.hkv + hk) * D + 32 * part;
                    float4* dkr = reinterpret_cast<float4*>(p.dk + off);
                    float4* dvr = reinterpret_cast<float4*>(p.dv + off);
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        dkr[q] = make_float4(p.scale * __uint_as_float(a[4 * q]), p.scale * __uint_as_float(a[4 * q + 1]),
                                             p.scale * __uint_as_float(a[4 * q + 2]),
                                             p.scale * __uint_as_float(a[4 * q + 3]));
                        dvr[q] = make_float4(__uint_as_float(c[4 * q]), __uint_as_float(c[4 * q + 1]),
                                             __uint_as_float(c[4 * q + 2]), __uint_as_float(c[4 * q + 3]));
                    }
                }
            }
        }
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after_sync();
        tmem_dealloc(tmem, kTmemCols);
    }
}

// 2D tensor [rows][cols] (row pitch in bytes), box {box_cols, box_rows},
// 128-byte swizzle, zero fill out of range.
bool encode(CUtensorMap* map, CUtensorMapDataType type, const void* base, unsigned long long cols,
            unsigned long long rows, unsigned long long pitch, unsigned box_cols, unsigned box_rows) {
    EncodeTiledFn fn = tensor_map_encoder();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {pitch};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, type, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int D>
cudaError_t launch_tc(const CUtensorMap& qmap, const CUtensorMap& domap, const CUtensorMap& kvmap,
                      const CUtensorMap& dqmap, const BwdTcParams& p, int batch, int max_seqlen, cudaStream_t stream) {
    using C = TcCfg<D>;
    cudaError_t e = cudaFuncSetAttribute(bwd_tc_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    const dim3 grid(static_cast<unsigned>(batch * p.g.hkv), static_cast<unsigned>((max_seqlen + kKeys - 1) / kKeys));
    bwd_tc_kernel<D><<<grid, C::THREADS, C::SMEM, stream>>>(qmap, domap, kvmap, dqmap, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_backward_tc(const KGeom& g, const void* q, const void* pool, const int32_t* bt, int layer,
                               int batch, const int32_t* cu, const int32_t* slots, int max_seqlen, int total_tokens,
                               float scale, const void* dout, const float* ws, float* dq, float* dk, float* dv,
                               int32_t* err, cudaStream_t stream) {
    CUtensorMap qmap, domap, kvmap, dqmap;
    const unsigned long long qcols = static_cast<unsigned long long>(g.hq) * g.d;
    if (!encode(&qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, q, qcols, total_tokens, qcols * 2, 64, kRowsIt) ||
        !encode(&domap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, dout, qcols, total_tokens, qcols * 2, 64, kRowsIt) ||
        !encode(&kvmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, pool, g.kv_dim, static_cast<unsigned long long>(g.nblocks) * 32,
                static_cast<unsigned long long>(g.kv_dim) * 2, 64, kBlockTokens) ||
        !encode(&dqmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, dq, qcols, total_tokens, qcols * 4, 32, 2 * kRowsIt))
        return cudaErrorInvalidValue;
    BwdTcParams p;
    p.g = g;
    p.bt = bt;
    p.layer = layer;
    p.cu = cu;
    p.slots = slots;
    p.max_seqlen = max_seqlen;
    p.total_tokens = total_tokens;
    p.ws = ws;
    p.ws_half = static_cast<long long>(total_tokens) * g.hq;
    p.scale = scale;
    p.scale_log2 = scale * kLog2e;
    p.dk = dk;
    p.dv = dv;
    p.kv_32b = ((reinterpret_cast<uintptr_t>(dk) | reinterpret_cast<uintptr_t>(dv)) & 31u) == 0;
    p.err = err;
    if (g.d == 64) return launch_tc<64>(qmap, domap, kvmap, dqmap, p, batch, max_seqlen, stream);
    return launch_tc<128>(qmap, domap, kvmap, dqmap, p, batch, max_seqlen, stream);
}

}  // namespace pa

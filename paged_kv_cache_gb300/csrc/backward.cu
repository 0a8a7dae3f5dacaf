// backward.cu -- gradients of the causal prefill with respect to q and to the
// K / V rows it read from the pages (the FlashAttention-2 backward).
//
// FlashAttention-2 explainer, "전체 흐름" (last step) and "2. 시퀀스 길이
// 방향으로도 병렬화" item 4: the backward recomputes the weights P from the
// single stored statistic L = m + ln l, runs one thread block per column block
// (a block of keys), and adds the overlapping dQ contributions with atomics;
// "4. MQA · GQA 지원": the dK / dV of the implicitly repeated kv heads are
// summed.  With s_ij = scale q_i . k_j (j <= i), p_ij = e^(s_ij - L_i),
// do_i the output gradient and o_i the forward output:
//   D_i  = do_i . o_i                       dp_ij = do_i . v_j
//   ds_ij = p_ij (dp_ij - D_i)
//   dv_j = sum_i p_ij do_i    dk_j = scale sum_i ds_ij q_i    dq_i = scale sum_j ds_ij k_j
// (D_i = sum_j p_ij dp_ij = do_i . o_i, since o_i = sum_j p_ij v_j.)
//
// Two kernels.  bwd_prep: D for every (row, q head) from the bf16 o and do,
// and dq set to zero.  Then, for head dim 64, the tensor-core kernel of
// backward_tc.cu; for head dim 128 (whose dK, dV and dQ accumulators do not
// fit tensor memory beside double-buffered S^T and dP^T) bwd_main here: one
// CTA of four warps per (64-key block,
// sequence, kv head).  It stages the block's K and V rows from the pages once,
// keeps dK and dV for its 64 keys in registers, and walks every q head of the
// group and every 64-row query block at or after the diagonal.  Each warp owns
// 16 keys: it forms S^T = K Q^T and dP^T = V dO^T for its keys, P^T and dS^T
// from them, adds P^T dO to dV and dS^T Q to dK, and writes dS^T (bf16) to
// shared memory; then each warp takes 16 query rows of dQ = dS K and adds them
// into dq with fp32 vector atomics.  The products run on mma.sync m16n8k16
// (bf16 in, fp32 accumulate); Q and dO tiles are double-buffered with
// cp.async so the next row block loads while this one computes.
#include "pa_internal.cuh"

namespace pa {
namespace {

constexpr int kBwdRows = 64;       // keys per CTA = query rows per row block
constexpr int kBwdWarps = 4;       // 16 keys per warp
constexpr int kBwdThreads = 32 * kBwdWarps;

template <int D>
struct BwdCfg {
    static constexpr int LD = D + 8;          // bf16 row stride of a staged tile (pad: no ldmatrix bank conflicts)
    static constexpr int TILE_BYTES = kBwdRows * LD * 2;
    static constexpr int DS_LD = kBwdRows + 8;
    static constexpr int K_OFF = 0;
    static constexpr int V_OFF = K_OFF + TILE_BYTES;
    static constexpr int Q_OFF = V_OFF + TILE_BYTES;      // 2 stages
    static constexpr int DO_OFF = Q_OFF + 2 * TILE_BYTES;  // 2 stages
    static constexpr int DS_OFF = DO_OFF + 2 * TILE_BYTES;
    static constexpr int L_OFF = DS_OFF + kBwdRows * DS_LD * 2;  // 2 stages of 64 fp32
    static constexpr int DD_OFF = L_OFF + 2 * kBwdRows * 4;      // 2 stages of 64 fp32
    static constexpr int SMEM = DD_OFF + 2 * kBwdRows * 4;
    static constexpr int CHUNKS = D / 8;  // 16-byte pieces of one head row
};

struct BwdParams {
    KGeom g;
    const uint16_t* q;
    const uint8_t* pool;
    const int32_t* bt;
    int layer;
    int batch;
    const int32_t* cu;
    const int32_t* slots;
    int max_seqlen;
    int total_tokens;
    const uint16_t* o;
    const float* lse;
    const uint16_t* dout;
    float* delta;        // workspace: [2][total_tokens][hq], -L log2 e then -D
    long long ws_half;   // total_tokens * hq
    float scale;
    float scale_log2;
    float* dq;
    float* dk;
    float* dv;
    int32_t* err;
};

__device__ __forceinline__ void cp_async16(uint32_t saddr, const void* gsrc) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(saddr), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t saddr, const void* gsrc) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(saddr), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void st_shared_zero16(uint32_t saddr) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(saddr), "r"(0) : "memory");
}
__device__ __forceinline__ void st_shared_f32(uint32_t saddr, float v) {
    asm volatile("st.shared.f32 [%0], %1;" ::"r"(saddr), "f"(v) : "memory");
}
__device__ __forceinline__ void st_shared_u32(uint32_t saddr, uint32_t v) {
    asm volatile("st.shared.u32 [%0], %1;" ::"r"(saddr), "r"(v) : "memory");
}

// Per (row, q head): D_i = do_i . o_i in fp32 from the bf16 values, stored
// as the two terms the main kernels add, ws[0][row][h] = -L_i log2 e and
// ws[1][row][h] = -D_i; dq = 0.  D / 8 consecutive threads share one (row,
// head): 16 bytes of o and do each.
template <int D>
__global__ void __launch_bounds__(256) bwd_prep_kernel(const uint16_t* __restrict__ o,
                                                       const uint16_t* __restrict__ dout,
                                                       const float* __restrict__ lse,
                                                       float* __restrict__ ws, float* __restrict__ dq,
                                                       long long pairs) {
    constexpr int PER = D / 8;
    const long long t = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const long long pair = t / PER;
    const int part = static_cast<int>(t % PER);
    const bool live = pair < pairs;
    float acc = 0.f;
    if (live) {
        const long long off = pair * D + part * 8;
        const uint4 ov = __ldg(reinterpret_cast<const uint4*>(o + off));
        const uint4 gv = __ldg(reinterpret_cast<const uint4*>(dout + off));
        const uint32_t ow[4] = {ov.x, ov.y, ov.z, ov.w};
        const uint32_t gw[4] = {gv.x, gv.y, gv.z, gv.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            acc = fmaf(bf16lo(ow[k]), bf16lo(gw[k]), acc);
            acc = fmaf(bf16hi(ow[k]), bf16hi(gw[k]), acc);
        }
        float4* z = reinterpret_cast<float4*>(dq + off);
        z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
        z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int s = PER / 2; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
    if (live && part == 0) {
        ws[pair] = -__ldg(lse + pair) * kLog2e;
        ws[pairs + pair] = -acc;
    }
}

template <int D>
__global__ void __launch_bounds__(kBwdThreads) bwd_main_kernel(const BwdParams p) {
    using C = BwdCfg<D>;
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
    const int b = blockIdx.x / p.g.hkv, hk = blockIdx.x % p.g.hkv;
    const int jb = blockIdx.y;

    const int cu0 = p.cu[b], cu1 = p.cu[b + 1];
    const int n = cu1 - cu0;
    const bool bad_len = cu0 < 0 || n < 0 || cu1 > p.total_tokens || n > p.max_seqlen ||
                         n > p.g.maxb * kBlockTokens;
    if (jb == 0 && hk == 0 && tid == 0 && bad_len) set_error(p.err, PA_ERR_BAD_BLOCK);
    if (bad_len || jb * kBwdRows >= n) return;
    const int slot = p.slots[b];
    if (slot < 0 || slot >= p.g.num_slots) {
        if (jb == 0 && hk == 0 && tid == 0) set_error(p.err, PA_ERR_BAD_BLOCK);
        return;
    }
    const int32_t* bt_row = p.bt + (static_cast<long long>(slot) * p.g.n_layers + p.layer) * p.g.maxb;
    const uint32_t sbase = smem_u32(smem);

    // K and V rows of this column block, zero past the sequence's end.
    for (int c = tid; c < kBwdRows * C::CHUNKS; c += kBwdThreads) {
        const int key = c / C::CHUNKS, part = c % C::CHUNKS;
        const int pos = jb * kBwdRows + key;
        const uint32_t so = static_cast<uint32_t>(key * C::LD * 2 + part * 16);
        int blk = -1;
        if (pos < n) {
            blk = bt_row[pos / kBlockTokens];
            if (blk < 0 || blk >= p.g.nblocks) {
                set_error(p.err, PA_ERR_BAD_BLOCK);
                blk = -1;
            }
        }
        if (blk >= 0) {
            const uint8_t* src = p.pool + blk * p.g.page_bytes +
                                 static_cast<long long>(pos % kBlockTokens) * p.g.kv_dim * 2 +
                                 static_cast<long long>(hk) * D * 2 + part * 16;
            cp_async16(sbase + C::K_OFF + so, src);
            cp_async16(sbase + C::V_OFF + so, src + static_cast<long long>(kBlockTokens) * p.g.kv_dim * 2);
        } else {
            st_shared_zero16(sbase + C::K_OFF + so);
            st_shared_zero16(sbase + C::V_OFF + so);
        }
    }

    const int group = p.g.group;
    const int nrb = (n + kBwdRows - 1) / kBwdRows;
    const int per_head = nrb - jb;
    const int iters = group * per_head;

    // Q, dO, L and D of query block (head r, block ib) into stage st.
    auto load_rows = [&](int it, int st) {
        const int r = it / per_head, ib = jb + it % per_head;
        const int h = hk * group + r;
        for (int c = tid; c < kBwdRows * C::CHUNKS; c += kBwdThreads) {
            const int row = c / C::CHUNKS, part = c % C::CHUNKS;
            const int i = ib * kBwdRows + row;
            const uint32_t so = static_cast<uint32_t>(st * C::TILE_BYTES + row * C::LD * 2 + part * 16);
            if (i < n) {
                const long long off = (static_cast<long long>(cu0 + i) * p.g.hq + h) * D + part * 8;
                cp_async16(sbase + C::Q_OFF + so, p.q + off);
                cp_async16(sbase + C::DO_OFF + so, p.dout + off);
            } else {
                st_shared_zero16(sbase + C::Q_OFF + so);
                st_shared_zero16(sbase + C::DO_OFF + so);
            }
        }
        if (tid < kBwdRows) {
            const int i = ib * kBwdRows + tid;
            const uint32_t so = static_cast<uint32_t>((st * kBwdRows + tid) * 4);
            if (i < n) {
                const long long off = static_cast<long long>(cu0 + i) * p.g.hq + h;
                cp_async4(sbase + C::L_OFF + so, p.delta + off);
                cp_async4(sbase + C::DD_OFF + so, p.delta + p.ws_half + off);
            } else {
                st_shared_f32(sbase + C::L_OFF + so, 0.f);
                st_shared_f32(sbase + C::DD_OFF + so, 0.f);
            }
        }
    };
    load_rows(0, 0);
    cp_async_commit();

    float acc_dk[D / 8][4], acc_dv[D / 8][4];
#pragma unroll
    for (int t = 0; t < D / 8; ++t)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc_dk[t][e] = acc_dv[t][e] = 0.f;

    const int key0 = jb * kBwdRows + 16 * w + (lane >> 2);  // key of C-fragment rows 0..7 (+8 for rows 8..15)
    // ldmatrix lane addresses (bytes within a tile), fixed for the kernel.
    const uint32_t a_lane = static_cast<uint32_t>((16 * w + (lane & 15)) * C::LD * 2 + (lane >> 4) * 16);
    const uint32_t bn_lane = static_cast<uint32_t>(((lane & 7) + ((lane >> 4) << 3)) * C::LD * 2 +
                                                   ((lane >> 3) & 1) * 16);
    const uint32_t bt_lane = static_cast<uint32_t>(((lane & 7) + ((lane >> 3) & 1) * 8) * C::LD * 2 +
                                                   (lane >> 4) * 16);
    const uint32_t ds_lane = static_cast<uint32_t>(((lane & 7) + (lane >> 4) * 8) * C::DS_LD * 2 +
                                                   (16 * w + ((lane >> 3) & 1) * 8) * 2);

    for (int it = 0; it < iters; ++it) {
        const int st = it & 1;
        const int r = it / per_head, ib = jb + it % per_head;
        const int h = hk * group + r;
        cp_async_wait_all();
        __syncthreads();
        if (it + 1 < iters) load_rows(it + 1, st ^ 1);
        cp_async_commit();

        const uint32_t q_s = sbase + C::Q_OFF + st * C::TILE_BYTES;
        const uint32_t do_s = sbase + C::DO_OFF + st * C::TILE_BYTES;
        const float* l_s = reinterpret_cast<const float*>(smem + C::L_OFF) + st * kBwdRows;
        const float* d_s = reinterpret_cast<const float*>(smem + C::DD_OFF) + st * kBwdRows;

        // S^T = K_w Q^T and dP^T = V_w dO^T: 16 keys x 64 query rows each.
        float s[8][4], dp[8][4];
#pragma unroll
        for (int t = 0; t < 8; ++t)
#pragma unroll
            for (int e = 0; e < 4; ++e) s[t][e] = dp[t][e] = 0.f;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            uint32_t ak[4], av[4];
            ldmatrix_x4(ak, sbase + C::K_OFF + a_lane + kk * 32);
            ldmatrix_x4(av, sbase + C::V_OFF + a_lane + kk * 32);
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                uint32_t bq[4], bo[4];
                const uint32_t off = bn_lane + np * 16 * C::LD * 2 + kk * 32;
                ldmatrix_x4(bq, q_s + off);
                ldmatrix_x4(bo, do_s + off);
                mma_bf16_16816(s[2 * np], ak, bq[0], bq[1]);
                mma_bf16_16816(s[2 * np + 1], ak, bq[2], bq[3]);
                mma_bf16_16816(dp[2 * np], av, bo[0], bo[1]);
                mma_bf16_16816(dp[2 * np + 1], av, bo[2], bo[3]);
            }
        }

        // P^T = e^(scale s - L) on j <= i < n, else 0; dS^T = P^T (dP^T - D)
        // (shared memory holds -L log2 e and -D).
#pragma unroll
        for (int t = 0; t < 8; ++t) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int col = 8 * t + 2 * (lane & 3) + e;
                const int i = ib * kBwdRows + col;
                const float nl = l_s[col];
                const float nd = d_s[col];
                const bool in_seq = i < n;
                const float p0 = (in_seq && key0 <= i) ? ex2_approx(fmaf(s[t][e], p.scale_log2, nl)) : 0.f;
                const float p1 = (in_seq && key0 + 8 <= i) ? ex2_approx(fmaf(s[t][2 + e], p.scale_log2, nl)) : 0.f;
                s[t][e] = p0;
                s[t][2 + e] = p1;
                dp[t][e] = p0 * (dp[t][e] + nd);
                dp[t][2 + e] = p1 * (dp[t][2 + e] + nd);
            }
        }

        // dS^T to shared memory for the dQ product (rows = keys, columns = query rows).
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            const uint32_t so = sbase + C::DS_OFF +
                                static_cast<uint32_t>(((16 * w + (lane >> 2)) * C::DS_LD + 8 * t + 2 * (lane & 3)) * 2);
            st_shared_u32(so, pack_bf16x2(dp[t][0], dp[t][1]));
            st_shared_u32(so + 8 * C::DS_LD * 2, pack_bf16x2(dp[t][2], dp[t][3]));
        }

        // dV_w += P^T dO and dK_w += dS^T Q (contraction over the 64 query rows).
#pragma unroll
        for (int kt = 0; kt < 4; ++kt) {
            const uint32_t ap[4] = {pack_bf16x2(s[2 * kt][0], s[2 * kt][1]), pack_bf16x2(s[2 * kt][2], s[2 * kt][3]),
                                    pack_bf16x2(s[2 * kt + 1][0], s[2 * kt + 1][1]),
                                    pack_bf16x2(s[2 * kt + 1][2], s[2 * kt + 1][3])};
            const uint32_t as[4] = {pack_bf16x2(dp[2 * kt][0], dp[2 * kt][1]),
                                    pack_bf16x2(dp[2 * kt][2], dp[2 * kt][3]),
                                    pack_bf16x2(dp[2 * kt + 1][0], dp[2 * kt + 1][1]),
                                    pack_bf16x2(dp[2 * kt + 1][2], dp[2 * kt + 1][3])};
#pragma unroll
            for (int dp2 = 0; dp2 < D / 16; ++dp2) {
                uint32_t bo[4], bq[4];
                const uint32_t off = bt_lane + kt * 16 * C::LD * 2 + dp2 * 32;
                ldmatrix_x4_trans(bo, do_s + off);
                ldmatrix_x4_trans(bq, q_s + off);
                mma_bf16_16816(acc_dv[2 * dp2], ap, bo[0], bo[1]);
                mma_bf16_16816(acc_dv[2 * dp2 + 1], ap, bo[2], bo[3]);
                mma_bf16_16816(acc_dk[2 * dp2], as, bq[0], bq[1]);
                mma_bf16_16816(acc_dk[2 * dp2 + 1], as, bq[2], bq[3]);
            }
        }
        __syncthreads();

        // dQ rows 16w .. 16w+15 of this block: dS K over the 64 keys, added to dq.
        float acc_dq[D / 8][4];
#pragma unroll
        for (int t = 0; t < D / 8; ++t)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc_dq[t][e] = 0.f;
#pragma unroll
        for (int kt = 0; kt < 4; ++kt) {
            uint32_t a[4];
            ldmatrix_x4_trans(a, sbase + C::DS_OFF + ds_lane + kt * 16 * C::DS_LD * 2);
#pragma unroll
            for (int dp2 = 0; dp2 < D / 16; ++dp2) {
                uint32_t bk[4];
                ldmatrix_x4_trans(bk, sbase + C::K_OFF + bt_lane + kt * 16 * C::LD * 2 + dp2 * 32);
                mma_bf16_16816(acc_dq[2 * dp2], a, bk[0], bk[1]);
                mma_bf16_16816(acc_dq[2 * dp2 + 1], a, bk[2], bk[3]);
            }
        }
        const int i0 = ib * kBwdRows + 16 * w + (lane >> 2);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int i = i0 + 8 * hh;
            if (i < n) {
                float* dst = p.dq + (static_cast<long long>(cu0 + i) * p.g.hq + h) * D + 2 * (lane & 3);
#pragma unroll
                for (int t = 0; t < D / 8; ++t)
                    atomicAdd(reinterpret_cast<float2*>(dst + 8 * t),
                              make_float2(p.scale * acc_dq[t][2 * hh], p.scale * acc_dq[t][2 * hh + 1]));
            }
        }
    }
    cp_async_wait_all();

    // dK = scale sum ds q and dV for this block's keys (rows past the end are not written).
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        const int j = key0 + 8 * hh;
        if (j < n) {
            const long long off = (static_cast<long long>(cu0 + j) * p.g.hkv + hk) * D + 2 * (lane & 3);
#pragma unroll
            for (int t = 0; t < D / 8; ++t) {
                *reinterpret_cast<float2*>(p.dk + off + 8 * t) =
                    make_float2(p.scale * acc_dk[t][2 * hh], p.scale * acc_dk[t][2 * hh + 1]);
                *reinterpret_cast<float2*>(p.dv + off + 8 * t) =
                    make_float2(acc_dv[t][2 * hh], acc_dv[t][2 * hh + 1]);
            }
        }
    }
}

template <int D>
cudaError_t launch_backward_d(const BwdParams& p, cudaStream_t stream) {
    const long long pairs = static_cast<long long>(p.total_tokens) * p.g.hq;
    const long long threads = pairs * (D / 8);
    const int prep_block = 256;
    bwd_prep_kernel<D><<<static_cast<unsigned>((threads + prep_block - 1) / prep_block), prep_block, 0, stream>>>(
        p.o, p.dout, p.lse, p.delta, p.dq, pairs);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (p.batch == 0 || p.max_seqlen == 0) return cudaSuccess;
    if constexpr (D == 64)
        return launch_backward_tc(p.g, p.q, p.pool, p.bt, p.layer, p.batch, p.cu, p.slots, p.max_seqlen,
                                  p.total_tokens, p.scale, p.dout, p.delta, p.dq, p.dk, p.dv, p.err, stream);
    else {
        using C = BwdCfg<D>;
        e = cudaFuncSetAttribute(bwd_main_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return e;
        const dim3 grid(static_cast<unsigned>(p.batch * p.g.hkv),
                        static_cast<unsigned>((p.max_seqlen + kBwdRows - 1) / kBwdRows));
        bwd_main_kernel<D><<<grid, kBwdThreads, C::SMEM, stream>>>(p);
        return cudaGetLastError();
    }
}

}  // namespace

cudaError_t launch_prefill_backward(const KGeom& g, const void* q, const void* pool, const int32_t* bt,
                                    int layer, int batch, const int32_t* cu, const int32_t* slots,
                                    int max_seqlen, int total_tokens, float scale, const void* o,
                                    const float* lse, const void* dout, float* delta, float* dq, float* dk,
                                    float* dv, int32_t* err, cudaStream_t stream) {
    BwdParams p;
    p.g = g;
    p.q = static_cast<const uint16_t*>(q);
    p.pool = static_cast<const uint8_t*>(pool);
    p.bt = bt;
    p.layer = layer;
    p.batch = batch;
    p.cu = cu;
    p.slots = slots;
    p.max_seqlen = max_seqlen;
    p.total_tokens = total_tokens;
    p.o = static_cast<const uint16_t*>(o);
    p.lse = lse;
    p.dout = static_cast<const uint16_t*>(dout);
    p.delta = delta;
    p.ws_half = static_cast<long long>(total_tokens) * g.hq;
    p.scale = scale;
    p.scale_log2 = scale * kLog2e;
    p.dq = dq;
    p.dk = dk;
    p.dv = dv;
    p.err = err;
    // d 64: the tensor-core kernel (backward_tc.cu); d 128 (its dK, dV and dQ
    // accumulators do not fit tensor memory beside double-buffered S and dP):
    // the mma.sync kernel here
    if (g.d == 64) return launch_backward_d<64>(p, stream);
    return launch_backward_d<128>(p, stream);
}

}  // namespace pa

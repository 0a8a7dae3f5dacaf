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
// Two kernels.  bwd_prep here: D for every (row, q head) from the bf16 o and
// do, and dq set to zero.  Then the column-block kernel on the tensor cores
// (backward_tc.cu), head dims 64 and 128.

#include "pa_internal.cuh"

namespace pa {
namespace {

// Per (row, q head): D_i = do_i . o_i in fp32 from the bf16 values, stored
// as the two terms the column-block kernel adds, ws[0][row][h] = -L_i log2 e and
// ws[1][row][h] = -D_i; dq = 0.  D / 8 consecutive threads share one (row,
// head): 16 bytes of o and do each.
template <int D>
__global__ void __launch_bounds__(256) bwd_prep_kernel(const uint16_t* __restrict__ o,
                                                       const uint16_t* __restrict__ dout,
                                                       const float* __restrict__ lse,
                                                       float* __restrict__ ws, float* __restrict__ dq,
                                                       long long pairs, bool dq_32b) {
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
        if (dq_32b) {  // one whole 32-byte sector
            const uint32_t zero[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
            st_global_v8(dq + off, zero);
        } else {
            float4* z = reinterpret_cast<float4*>(dq + off);
            z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
            z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
#pragma unroll
    for (int s = PER / 2; s > 0; s >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, s);
    if (live && part == 0) {
        ws[pair] = -__ldg(lse + pair) * kLog2e;
        ws[pairs + pair] = -acc;
    }
}

}  // namespace

cudaError_t launch_prefill_backward(const KGeom& g, const void* q, const void* pool, const int32_t* bt,
                                    int layer, int batch, const int32_t* cu, const int32_t* slots,
                                    int max_seqlen, int total_tokens, float scale, const void* o,
                                    const float* lse, const void* dout, float* delta, float* dq, float* dk,
                                    float* dv, int32_t* err, cudaStream_t stream) {
    const long long pairs = static_cast<long long>(total_tokens) * g.hq;
    const long long threads = pairs * (g.d / 8);
    const int prep_block = 256;
    const unsigned prep_grid = static_cast<unsigned>((threads + prep_block - 1) / prep_block);
    const auto* o16 = static_cast<const uint16_t*>(o);
    const auto* do16 = static_cast<const uint16_t*>(dout);
    const bool dq_32b = (reinterpret_cast<uintptr_t>(dq) & 31u) == 0;
    if (g.d == 64)
        bwd_prep_kernel<64><<<prep_grid, prep_block, 0, stream>>>(o16, do16, lse, delta, dq, pairs, dq_32b);
    else
        bwd_prep_kernel<128><<<prep_grid, prep_block, 0, stream>>>(o16, do16, lse, delta, dq, pairs, dq_32b);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (batch == 0 || max_seqlen == 0) return cudaSuccess;
    return launch_backward_tc(g, q, pool, bt, layer, batch, cu, slots, max_seqlen, total_tokens, scale, dout, delta,
                              dq, dk, dv, err, stream);
}

}  // namespace pa

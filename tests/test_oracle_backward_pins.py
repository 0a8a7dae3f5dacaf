"""Pins of the oracle's prefill backward (orc_prefill_backward).

The gradients of the causal prefill with respect to q, k and v for a given
output gradient are fixed by the chain rule; they are pinned against
  * torch fp64 autograd through scaled_dot_product_attention on the
    contiguous K/V (a library routine), the GQA heads repeated so that
    autograd itself adds the repeats' gradients;
  * central finite differences of the forward oracle (a different function of
    this file) at points where x +- h are bf16-exact;
  * identities that hold at any size: the scores are shift-invariant per row,
    so sum_j dk_j = 0 for each (sequence, kv head); the weights of a row add
    up to one, so sum_j dv_j = sum over the group's heads and rows of do.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from paged_kv_cache_gb300 import workloads as W  # noqa: E402


def f64(bits):
    return W.bf16_to_f32(bits).astype(np.float64)


def setup(hq, hkv, d, lens, seed):
    nb = sum((n + 15) // 16 for n in lens) + 4
    geom = W.Geometry(hq, hkv, d, 1, len(lens), 32, nb)
    case = W.make_prefill_case("bwd", geom, lens, seed=seed, pool_fill="nan")
    g = oracle.geom(*geom.as_tuple())
    pool = W.initial_pool(geom, case.pool_fill, case.seed)
    for w in case.writes:
        assert oracle.write_kv(g, pool, case.block_table, w.layer, w.tok_slot, w.tok_pos, w.k, w.v) == 0
    rng = np.random.default_rng(seed + 1)
    dout = W.normal_bf16(rng, case.q.shape)
    return case, g, pool, dout


@pytest.mark.parametrize("hq,hkv,d,lens", [
    (8, 2, 64, [40, 17]),
    (4, 4, 64, [33]),        # MHA
    (6, 1, 64, [29]),        # MQA
    (4, 2, 128, [23, 9]),    # head dim 128
])
def test_matches_torch_autograd(hq, hkv, d, lens):
    case, g, pool, dout = setup(hq, hkv, d, lens, seed=hq * 10 + d)
    st, dq, dk, dv = oracle.prefill_backward(g, case.q, pool, case.block_table, 0, case.cu_seqlens, case.slots,
                                             case.scale, dout)
    assert st == 0
    w = case.writes[0]
    cu = case.cu_seqlens
    sc = float(np.float32(case.scale))
    for b in range(case.batch):
        q = torch.tensor(f64(case.q[cu[b]:cu[b + 1]]).transpose(1, 0, 2), requires_grad=True)
        k = torch.tensor(f64(w.k[cu[b]:cu[b + 1]]).reshape(-1, hkv, d).transpose(1, 0, 2), requires_grad=True)
        v = torch.tensor(f64(w.v[cu[b]:cu[b + 1]]).reshape(-1, hkv, d).transpose(1, 0, 2), requires_grad=True)
        o = torch.nn.functional.scaled_dot_product_attention(
            q, k.repeat_interleave(hq // hkv, dim=0), v.repeat_interleave(hq // hkv, dim=0), is_causal=True, scale=sc)
        o.backward(torch.tensor(f64(dout[cu[b]:cu[b + 1]]).transpose(1, 0, 2)))
        np.testing.assert_allclose(dq[cu[b]:cu[b + 1]], q.grad.numpy().transpose(1, 0, 2), rtol=1e-10, atol=1e-11)
        np.testing.assert_allclose(dk[cu[b]:cu[b + 1]], k.grad.numpy().transpose(1, 0, 2), rtol=1e-10, atol=1e-11)
        np.testing.assert_allclose(dv[cu[b]:cu[b + 1]], v.grad.numpy().transpose(1, 0, 2), rtol=1e-10, atol=1e-11)


def test_central_differences_of_the_forward_oracle():
    """loss = sum do . o; its derivative in one element of q, k and v against
    (loss(x + h) - loss(x - h)) / 2h through the forward oracle."""
    case, g, pool, dout = setup(8, 2, 64, [24], seed=3)
    w = case.writes[0]
    h = 2.0 ** -8  # x = 0.5 or -0.5: x +- h are bf16 numbers

    def loss(q, k, v):
        pl = W.initial_pool(case.geom, case.pool_fill, case.seed)
        assert oracle.write_kv(g, pl, case.block_table, 0, w.tok_slot, w.tok_pos, k, v) == 0
        st2, o, _ = oracle.prefill(g, q, pl, case.block_table, 0, case.cu_seqlens, case.slots, case.scale)
        assert st2 == 0
        return float(np.sum(f64(dout) * o))

    def bumped(a, idx, val):
        x = a.copy()
        x[idx] = W.bf16_bits(np.array([val], np.float32))[0]
        return x

    checks = [("q", (7, 3, 5)), ("k", (2, 70)), ("v", (11, 12))]  # k, v: (row, kv-dim element)
    for which, idx in checks:
        out = []
        for x in (0.5 + h, 0.5 - h):
            q, k, v = case.q, w.k, w.v
            if which == "q":
                q = bumped(q, idx, x)
            elif which == "k":
                k = bumped(k, idx, x)
            else:
                v = bumped(v, idx, x)
            out.append(loss(q, k, v))
        # the gradient at x = 0.5 (the element set to 0.5 on both sides of the difference)
        q0, k0, v0 = case.q, w.k, w.v
        if which == "q":
            q0 = bumped(q0, idx, 0.5)
        elif which == "k":
            k0 = bumped(k0, idx, 0.5)
        else:
            v0 = bumped(v0, idx, 0.5)
        pl = W.initial_pool(case.geom, case.pool_fill, case.seed)
        assert oracle.write_kv(g, pl, case.block_table, 0, w.tok_slot, w.tok_pos, k0, v0) == 0
        _, gq, gk, gv = oracle.prefill_backward(g, q0, pl, case.block_table, 0, case.cu_seqlens, case.slots,
                                                case.scale, dout)
        if which == "q":
            exact = gq[idx]
        elif which == "k":
            exact = gk[idx[0], idx[1] // 64, idx[1] % 64]
        else:
            exact = gv[idx[0], idx[1] // 64, idx[1] % 64]
        fd = (out[0] - out[1]) / (2 * h)
        assert abs(fd - exact) <= 1e-4 * max(1.0, abs(exact)), (which, fd, exact)


def test_identities():
    case, g, pool, dout = setup(8, 2, 64, [300, 41], seed=5)
    st, dq, dk, dv = oracle.prefill_backward(g, case.q, pool, case.block_table, 0, case.cu_seqlens, case.slots,
                                             case.scale, dout)
    assert st == 0
    cu = case.cu_seqlens
    do = f64(dout)
    for b in range(case.batch):
        sk = dk[cu[b]:cu[b + 1]].sum(axis=0)  # [hkv][d]
        assert np.max(np.abs(sk)) < 1e-10 * max(1.0, np.max(np.abs(dk)))
        sv = dv[cu[b]:cu[b + 1]].sum(axis=0)
        want = do[cu[b]:cu[b + 1]].reshape(-1, 2, 4, 64).sum(axis=(0, 2))
        np.testing.assert_allclose(sv, want, rtol=1e-11, atol=1e-10)


@pytest.mark.parametrize("hq,hkv,d,lens", [
    (8, 2, 64, [40, 17, 1]),
    (6, 1, 64, [29, 33]),     # MQA, a group of 6
    (4, 2, 128, [23, 9]),
])
def test_sampled_rows_equal_the_full_backward(hq, hkv, d, lens):
    """prefill_backward_rows (dq of chosen (row, q head), dk / dv of chosen
    (row, kv head)) is the full call's entries, bit for bit: the same
    arithmetic in the same order."""
    case, g, pool, dout = setup(hq, hkv, d, lens, seed=hq * 7 + d)
    args = (g, case.q, pool, case.block_table, 0, case.cu_seqlens, case.slots, case.scale, dout)
    st, dq, dk, dv = oracle.prefill_backward(*args)
    assert st == 0
    T = case.total_tokens
    cu = case.cu_seqlens
    rng = np.random.default_rng(hq + d)
    q_rows = np.concatenate([[0, T - 1, cu[1] - 1, cu[1]], rng.integers(0, T, 12)]).astype(np.int64)
    q_heads = rng.integers(0, hq, q_rows.shape[0]).astype(np.int32)
    k_rows = np.concatenate([[0, T - 1, cu[1] - 1, cu[1]], rng.integers(0, T, 8)]).astype(np.int64)
    k_heads = rng.integers(0, hkv, k_rows.shape[0]).astype(np.int32)
    st2, sq, sk, sv = oracle.prefill_backward_rows(*args, q_rows, q_heads, k_rows, k_heads)
    assert st2 == 0
    np.testing.assert_array_equal(sq, dq[q_rows, q_heads])
    np.testing.assert_array_equal(sk, dk[k_rows, k_heads])
    np.testing.assert_array_equal(sv, dv[k_rows, k_heads])
    # out-of-range samples are refused
    assert oracle.prefill_backward_rows(*args, [T], [0], [], [])[0] != 0
    assert oracle.prefill_backward_rows(*args, [], [], [0], [hkv])[0] != 0

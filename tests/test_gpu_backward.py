"""GPU parity of pa_prefill_backward (the FlashAttention-2 backward over the
paged cache) against the oracle's gradients, through the C ABI.

The GPU forward (pa_prefill) supplies o and lse, as in training; the oracle
recomputes everything in fp64 from the bf16 inputs.  Tolerance, per gradient
tensor: max |gpu - oracle| <= 1e-2 * max |oracle| and a relative Frobenius
error <= 4e-3.  The kernel rounds P and dS to bf16 (relative 2^-9) before
the products that consume them and takes D = do . o from the bf16 output, so
each gradient element carries errors of a few 2^-9 of its terms; the bars are
those of the forward's O check and about twice 2^-9.

Sizes span several 64-key column blocks and 64-row query blocks with ragged
tails, every GQA group size the geometry allows (MHA, GQA 4, MQA with a group
of 6), head dims 64 and 128, a NaN-filled pool and an attended layer that is
not the first.  At the long-prompt size the checks are identities that hold
at any size, with bounds from the same rounding.
"""
import numpy as np
import pytest

import oracle
from paged_kv_cache_gb300 import workloads as W
from tests import helpers as H

pytestmark = pytest.mark.gpu


def gpu_forward_backward(case, pool, bt, dout, offset16=False):
    """GPU pa_prefill then pa_prefill_backward; returns numpy (dq, dk, dv, err).
    offset16: dq, dk and dv start 16 bytes past a 32-byte boundary."""
    torch = H.torch_mod()
    g = H.pa_geom(case)
    T, hq, hkv, d = case.total_tokens, case.geom.num_q_heads, case.geom.num_kv_heads, case.geom.head_dim
    q = H.to_dev(case.q)
    o = torch.empty((T, hq, d), dtype=torch.int16, device="cuda")
    lse = torch.empty((T, hq), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    cu, slots = H.to_dev(case.cu_seqlens), H.to_dev(case.slots)
    H.pa.pa_prefill(g, q, pool, bt, case.layer, cu, slots, case.max_len, case.scale, o, lse, err)
    delta = torch.empty((2, T, hq), dtype=torch.float32, device="cuda")
    def out(shape):
        if not offset16:
            return torch.full(shape, float("nan"), dtype=torch.float32, device="cuda")
        n = int(np.prod(shape))
        flat = torch.full((n + 4,), float("nan"), dtype=torch.float32, device="cuda")
        view = flat[4:].view(shape)
        assert view.data_ptr() % 32 == 16
        return view

    dq, dk, dv = out((T, hq, d)), out((T, hkv, d)), out((T, hkv, d))
    H.pa.pa_prefill_backward(g, q, pool, bt, case.layer, cu, slots, case.max_len, case.scale, o, lse,
                             H.to_dev(dout), delta, dq, dk, dv, err)
    torch.cuda.synchronize()
    return dq.cpu().numpy(), dk.cpu().numpy(), dv.cpu().numpy(), int(err.item())


def assert_grad_close(got, ref, what):
    got = got.astype(np.float64)
    assert np.all(np.isfinite(got)), what + ": non-finite gradient"
    scale = float(np.max(np.abs(ref)))
    err = float(np.max(np.abs(got - ref)))
    fro = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))
    assert err <= 1e-2 * scale, "%s: max err %.3e vs max |ref| %.3e" % (what, err, scale)
    assert fro <= 4e-3, "%s: relative Frobenius error %.3e" % (what, fro)


def backward_case(hq, hkv, d, lens, seed, layers=(0, 1)):
    nb = len(layers) * sum((n + 15) // 16 for n in lens) + 4
    geom = W.Geometry(hq, hkv, d, max(layers) + 1, len(lens), max(1, (max(lens) + 15) // 16), nb)
    case = W.make_prefill_case("bwd", geom, lens, seed=seed, layers=layers, pool_fill="nan")
    rng = np.random.default_rng(seed + 99)
    dout = W.normal_bf16(rng, case.q.shape)
    return case, dout


def oracle_backward(case, dout):
    st, dq, dk, dv = oracle.prefill_backward(
        H.oracle_geom(case), case.q, H.oracle_pool(case), case.block_table, case.layer, case.cu_seqlens,
        case.slots, case.scale, dout)
    assert st == 0
    return dq, dk, dv


@pytest.mark.parametrize("hq,hkv,d,lens", [
    (32, 8, 64, [17, 130, 64, 1]),   # the Llama-3.2-1B head layout, ragged batch
    (8, 2, 64, [200, 3]),
    (4, 4, 64, [65]),                # MHA
    (6, 1, 64, [129, 40]),           # MQA, a group of 6
    (16, 4, 128, [150, 64, 1]),      # head dim 128
    (8, 8, 128, [97]),
    (8, 1, 128, [300, 129]),         # head dim 128, MQA: a group of 8, many query blocks per key block
])
def test_backward_matches_oracle(hq, hkv, d, lens):
    case, dout = backward_case(hq, hkv, d, lens, seed=hq * 13 + d + len(lens))
    pool, bt, werr = H.gpu_setup(case)
    assert werr == 0
    dq, dk, dv, err = gpu_forward_backward(case, pool, bt, dout)
    assert err == 0
    rq, rk, rv = oracle_backward(case, dout)
    tag = "%d/%d d%d %s" % (hq, hkv, d, lens)
    assert_grad_close(dq, rq, "dq " + tag)
    assert_grad_close(dk, rk, "dk " + tag)
    assert_grad_close(dv, rv, "dv " + tag)


def test_rows_outside_the_batch():
    """total_tokens past cu_seqlens[batch]: dq rows there are zero, dk / dv rows
    there are not written."""
    case, dout = backward_case(8, 2, 64, [70, 5], seed=21, layers=(0,))
    torch = H.torch_mod()
    extra = 9
    q_pad = np.concatenate([case.q, W.normal_bf16(np.random.default_rng(1), (extra,) + case.q.shape[1:])])
    dout_pad = np.concatenate([dout, W.normal_bf16(np.random.default_rng(2), (extra,) + dout.shape[1:])])
    pool, bt, werr = H.gpu_setup(case)
    assert werr == 0
    g = H.pa_geom(case)
    T = q_pad.shape[0]
    q = H.to_dev(q_pad)
    o = torch.zeros((T, 8, 64), dtype=torch.int16, device="cuda")
    lse = torch.zeros((T, 8), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    cu, slots = H.to_dev(case.cu_seqlens), H.to_dev(case.slots)
    H.pa.pa_prefill(g, q, pool, bt, 0, cu, slots, case.max_len, case.scale, o, lse, err)
    delta = torch.empty((2, T, 8), dtype=torch.float32, device="cuda")
    dq = torch.full((T, 8, 64), 7.0, dtype=torch.float32, device="cuda")
    dk = torch.full((T, 2, 64), 7.0, dtype=torch.float32, device="cuda")
    dv = torch.full((T, 2, 64), 7.0, dtype=torch.float32, device="cuda")
    H.pa.pa_prefill_backward(g, q, pool, bt, 0, cu, slots, case.max_len, case.scale, o, lse, H.to_dev(dout_pad),
                             delta, dq, dk, dv, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    n = case.total_tokens
    assert np.all(dq.cpu().numpy()[n:] == 0.0)
    assert np.all(dk.cpu().numpy()[n:] == 7.0) and np.all(dv.cpu().numpy()[n:] == 7.0)
    rq, rk, rv = oracle_backward(case, dout)
    assert_grad_close(dq.cpu().numpy()[:n], rq, "dq padded")
    assert_grad_close(dk.cpu().numpy()[:n], rk, "dk padded")
    assert_grad_close(dv.cpu().numpy()[:n], rv, "dv padded")


def test_bad_slot_reports_and_context_recovers():
    case, dout = backward_case(8, 2, 64, [40, 20], seed=23, layers=(0,))
    pool, bt, werr = H.gpu_setup(case)
    assert werr == 0
    good = case.slots
    case.slots = np.array([0, case.geom.num_slots], np.int32)  # second slot out of range
    _, _, _, err = gpu_forward_backward(case, pool, bt, dout)
    assert err == H.pa.PA_ERR_BAD_BLOCK
    case.slots = good
    dq, dk, dv, err = gpu_forward_backward(case, pool, bt, dout)
    assert err == 0
    rq, rk, rv = oracle_backward(case, dout)
    assert_grad_close(dk, rk, "dk after bad slot")


def test_identities_at_long_prompt_size():
    """One 8192-token prompt (Hq 32, Hkv 8, d 64) and a short one.  Per
    (sequence, kv head):
      * sum_j dv_j = sum over the group's heads and rows of do, since every
        row's weights add up to one: the bf16 weights add up to 1 within
        2^-9 + 1e-5, which bounds the difference by that times sum |do|;
      * sum_i <q_i, dq_i> (over the group's heads) = sum_j <k_j, dk_j>: both
        are scale * sum_ij ds_ij <q_i, k_j> over the same bf16 ds, so they
        agree to fp32 rounding (scaling q up and k down leaves the scores)."""
    lens = [8192, 333]
    case, dout = backward_case(32, 8, 64, lens, seed=31, layers=(0,))
    pool, bt, werr = H.gpu_setup(case)
    assert werr == 0
    dq, dk, dv, err = gpu_forward_backward(case, pool, bt, dout)
    assert err == 0
    assert np.all(np.isfinite(dq)) and np.all(np.isfinite(dk)) and np.all(np.isfinite(dv))
    cu = case.cu_seqlens
    do = H.f32(dout)
    q = H.f32(case.q)
    w = case.writes[0]
    k = H.f32(w.k).reshape(-1, 8, 64)
    for b in range(2):
        rows = slice(cu[b], cu[b + 1])
        do_b = do[rows].reshape(-1, 8, 4, 64)                     # [n][hk][group][d]
        want = do_b.sum(axis=(0, 2))
        bound = (2.0 ** -9 + 1e-5) * np.abs(do_b).sum(axis=(0, 2)) + 1e-3
        got = dv[rows].astype(np.float64).sum(axis=0)
        assert np.all(np.abs(got - want) <= bound), float(np.max(np.abs(got - want) / bound))
        lhs = (q[rows].reshape(-1, 8, 4, 64) * dq[rows].astype(np.float64).reshape(-1, 8, 4, 64)).sum(axis=(0, 2, 3))
        rhs = (k[rows] * dk[rows].astype(np.float64)).sum(axis=(0, 2))
        mag = (np.abs(q[rows].reshape(-1, 8, 4, 64) * dq[rows].reshape(-1, 8, 4, 64))).sum(axis=(0, 2, 3))
        assert np.all(np.abs(lhs - rhs) <= 1e-3 * mag + 1e-6), (lhs, rhs, mag)


@pytest.mark.parametrize("hq,hkv,d", [(32, 8, 64), (16, 4, 128)])
def test_bench_size_sampled_rows(hq, hkv, d):
    """The bench's backward workloads in their launch configuration: 4 prompts
    of 8192 tokens, 32 q / 8 kv heads at d 64 and 16 / 4 at d 128, shuffled
    pages.  dq at 48 sampled (row, q head) pairs and dk, dv at 12 sampled (key
    row, kv head) pairs of two (sequence, kv head) units against the oracle's
    sampled backward (the full backward's entries, computed one by one)."""
    B, n = 4, 8192
    pages = n // 16
    geom = W.Geometry(hq, hkv, d, 1, B, pages, B * pages + 64)
    case = W.make_prefill_case("bwd", geom, [n] * B, 1007)
    dout = W.normal_bf16(np.random.default_rng(1008), case.q.shape)
    pool, bt, werr = H.gpu_setup(case)
    assert werr == 0
    dq, dk, dv, err = gpu_forward_backward(case, pool, bt, dout)
    assert err == 0
    rng = np.random.default_rng(5)
    starts = np.arange(B) * n
    q_rows = np.concatenate([starts, starts + n - 1, starts + 127, starts + 128, rng.integers(0, B * n, 32)])
    q_heads = rng.integers(0, hq, q_rows.shape[0]).astype(np.int32)
    units = [(0, 3), (3, hkv - 2)]  # (sequence, kv head)
    k_rows, k_heads = [], []
    for b, hk in units:
        for j in (0, 127, 128, n - 1, int(rng.integers(0, n)), int(rng.integers(0, n))):
            k_rows.append(b * n + j)
            k_heads.append(hk)
    st, rq, rk, rv = oracle.prefill_backward_rows(
        H.oracle_geom(case), case.q, H.oracle_pool(case), case.block_table, 0, case.cu_seqlens, case.slots,
        case.scale, dout, q_rows, q_heads, np.array(k_rows), np.array(k_heads))
    assert st == 0
    assert_grad_close(dq[q_rows, q_heads], rq, "dq sampled, 4 x 8192, d%d" % d)
    assert_grad_close(dk[k_rows, k_heads], rk, "dk sampled, 4 x 8192, d%d" % d)
    assert_grad_close(dv[k_rows, k_heads], rv, "dv sampled, 4 x 8192, d%d" % d)


def test_outputs_16_byte_aligned():
    """dq, dk and dv 16 bytes past a 32-byte boundary (the least alignment the
    call takes): the rows go out in 16-byte stores instead of whole sectors;
    dk and dv equal the aligned run's bit for bit (no atomics in them), dq
    stays within the tolerance."""
    for hq, hkv, d in ((8, 2, 64), (8, 2, 128)):
        case, dout = backward_case(hq, hkv, d, [150, 40], seed=61 + d, layers=(0,))
        pool, bt, werr = H.gpu_setup(case)
        assert werr == 0
        dq0, dk0, dv0, err0 = gpu_forward_backward(case, pool, bt, dout)
        dq1, dk1, dv1, err1 = gpu_forward_backward(case, pool, bt, dout, offset16=True)
        assert err0 == 0 and err1 == 0
        assert np.array_equal(dk0, dk1) and np.array_equal(dv0, dv1)
        rq, rk, rv = oracle_backward(case, dout)
        assert_grad_close(dq1, rq, "dq at a 16-byte offset, d%d" % d)


def test_bad_table_entry_reports_and_context_recovers():
    """A table entry of the attended layer set to -1 where a page is needed:
    the backward (both head dims) reports PA_ERR_BAD_BLOCK without faulting,
    and the next call on the good table is correct."""
    for hq, hkv, d in ((8, 2, 64), (8, 2, 128)):
        case, dout = backward_case(hq, hkv, d, [90, 30], seed=41 + d, layers=(0,))
        pool, bt, werr = H.gpu_setup(case)
        assert werr == 0
        bad = case.block_table.copy()
        bad[case.slots[0], 0, 3] = -1
        dq, dk, dv, err = gpu_forward_backward(case, pool, H.to_dev(bad), dout)
        assert err == H.pa.PA_ERR_BAD_BLOCK
        dq, dk, dv, err = gpu_forward_backward(case, pool, bt, dout)
        assert err == 0
        rq, rk, rv = oracle_backward(case, dout)
        assert_grad_close(dk, rk, "dk after a bad table entry, d%d" % d)

"""GPU parity of pa_prefill_rope (RoPE on the queries in the prefill prologue)
against the oracle, through the C ABI.

Each case turns K on its way into the pages (pa_write_kv_rope on the GPU,
orc_write_kv_rope on the CPU), then runs the RoPE-Q prefill; the oracle turns
the queries with orc_rope_q and attends with orc_prefill_cached.  Covered:
every q-heads-per-CTA variant of the kernel (4, 2, 1 at d 64; 2, 1 at d 128),
prefixes that are and are not multiples of the page and of the tiles, a
NaN-filled pool, the Llama-3.2-1B-shaped prompts, the 4 x 8192 bench
workload on sampled rows, the identity table (the plain prefill of fresh
prompts, bit for bit) and positions past the table.
"""
import numpy as np
import pytest

import oracle
import paged_kv_cache_gb300 as pa
from paged_kv_cache_gb300 import workloads as W
from tests import helpers as H

pytestmark = pytest.mark.gpu


def _write_rope(case, cos_t, sin_t):
    """Device pool and the oracle's pool after the case's writes with K turned."""
    torch = H.torch_mod()
    g = H.oracle_geom(case)
    ref = W.initial_pool(case.geom, case.pool_fill, case.seed)
    pool = H.device_pool(case)
    bt = H.to_dev(case.block_table)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ct, st = H.to_dev(cos_t), H.to_dev(sin_t)
    for w in case.writes:
        assert oracle.write_kv_rope(g, ref, case.block_table, w.layer, w.tok_slot, w.tok_pos, w.k, w.v,
                                    cos_t, sin_t) == 0
        pa.pa_write_kv_rope(H.pa_geom(case), pool, bt, w.layer, H.to_dev(w.tok_slot), H.to_dev(w.tok_pos),
                            H.to_dev(w.k), H.to_dev(w.v), ct, st, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return pool, bt, ref


def _gpu_rope(case, pool, bt, cos_t, sin_t, prefix):
    torch = H.torch_mod()
    T, Hq, D = case.total_tokens, case.geom.num_q_heads, case.geom.head_dim
    o = torch.empty((T, Hq, D), dtype=torch.int16, device="cuda")
    lse = torch.empty((T, Hq), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_prefill_rope(H.pa_geom(case), H.to_dev(case.q), pool, bt, case.layer, H.to_dev(case.cu_seqlens),
                       None if prefix is None else H.to_dev(np.asarray(prefix, np.int32)), H.to_dev(case.slots),
                       case.max_len, case.scale, H.to_dev(cos_t), H.to_dev(sin_t), o, lse, err)
    torch.cuda.synchronize()
    return H.f32(o.cpu().numpy().view(np.uint16)), lse.cpu().numpy().astype(np.float64), int(err.item())


def _check(case, prefix, cos_t, sin_t, what):
    pool, bt, ref = _write_rope(case, cos_t, sin_t)
    o, l, err = _gpu_rope(case, pool, bt, cos_t, sin_t, prefix)
    assert err == 0, what
    st, ro, rl = oracle.prefill_rope(H.oracle_geom(case), case.q, ref, case.block_table, case.layer, case.cu_seqlens,
                                     prefix, case.slots, case.scale, cos_t, sin_t)
    assert st == 0
    H.assert_close(o, l, ro, rl, H.max_abs_v(case), what)


@pytest.mark.parametrize("hq,hkv,d", [(32, 8, 64), (8, 2, 64), (6, 2, 64), (8, 8, 64), (16, 4, 128), (8, 8, 128)])
def test_rope_q_heads_per_cta_variants(hq, hkv, d):
    pre = [0, 17, 128, 300]
    lens = [129, 40, 1, 200]
    nb = sum((p + n + 15) // 16 for p, n in zip(pre, lens)) + 8
    geom = W.Geometry(hq, hkv, d, 1, 4, 64, nb)
    case = W.make_chunked_case("rq", geom, pre, lens, seed=hq * 5 + d, pool_fill="nan")
    cos_t, sin_t = W.rope_tables(600, d, base=10000.0)
    _check(case, case.extra["prefix"], cos_t, sin_t, "rope-q %d/%d d%d" % (hq, hkv, d))


def test_rope_q_tiny_prompt():
    pre, _ = W.tiny_case()
    cos_t, sin_t = W.rope_tables(64, 64, base=10000.0)
    _check(pre, None, cos_t, sin_t, "rope-q tiny prompt")


def test_rope_q_llama_prompts():
    case = W.llama_prefill_case()
    cos_t, sin_t = W.rope_tables(512, 64)
    _check(case, None, cos_t, sin_t, "rope-q Llama prompts")


@pytest.mark.parametrize("hq,hkv,d", [(32, 8, 64), (16, 4, 128)])
def test_identity_table_is_the_plain_prefill(hq, hkv, d):
    """cos 1, sin 0 leaves Q and K as they are: the RoPE-Q prefill of fresh
    prompts equals the plain prefill bit for bit (the same softmax order and
    work split at each head dim)."""
    geom = W.Geometry(hq, hkv, d, 1, 3, 32, 100)
    case = W.make_chunked_case("rq_id", geom, [0, 0, 0], [300, 77, 5], seed=4)
    n = 400
    one, zero = np.ones((n, d // 2), np.float32), np.zeros((n, d // 2), np.float32)
    pool, bt, _ = _write_rope(case, one, zero)
    o1, l1, e1 = _gpu_rope(case, pool, bt, one, zero, None)
    o2, l2, e2 = H.gpu_prefill(case, pool, bt)
    assert e1 == 0 and e2 == 0
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def test_positions_past_the_table_are_reported():
    geom = W.Geometry(8, 2, 64, 1, 2, 16, 40)
    case = W.make_chunked_case("rq_oob", geom, [0, 30], [40, 20], seed=8)
    cos_t, sin_t = W.rope_tables(64, 64)
    pool, bt, ref = _write_rope(case, cos_t, sin_t)
    short_c, short_s = cos_t[:45].copy(), sin_t[:45].copy()  # sequence 1 reaches position 49
    o, l, err = _gpu_rope(case, pool, bt, short_c, short_s, case.extra["prefix"])
    assert err == pa.PA_ERR_BAD_BLOCK
    # sequence 0 (positions 0..39) lies inside the table and is still right
    st, ro, rl = oracle.prefill_rope(H.oracle_geom(case), case.q, ref, case.block_table, 0, case.cu_seqlens,
                                     case.extra["prefix"], case.slots, case.scale, cos_t, sin_t)
    assert st == 0
    n0 = int(case.lens[0])
    H.assert_close(o[:n0], l[:n0], ro[:n0], rl[:n0], H.max_abs_v(case), "rope-q rows inside the table")


@pytest.mark.parametrize("variant", ["d64", "d128"])
def test_rope_q_long_prefill_sampled(variant):
    """The 4 x 8192 bench workload with K and Q turned (32 q / 8 kv heads at
    d 64, 16 / 4 at d 128), on sampled rows of every sequence (both ends of
    each, every head of the last row)."""
    case = W.long_prefill_case(variant)
    cos_t, sin_t = W.rope_tables(8192, case.geom.head_dim)
    pool, bt, ref = _write_rope(case, cos_t, sin_t)
    o, l, err = _gpu_rope(case, pool, bt, cos_t, sin_t, None)
    assert err == 0
    vmax = H.max_abs_v(case)
    assert np.all(np.isfinite(o)) and np.max(np.abs(o)) <= vmax * (1 + 2 ** -7)
    rng = np.random.default_rng(17)
    cu, Hq = case.cu_seqlens, case.geom.num_q_heads
    rows = [cu[b] + r for b in range(case.batch) for r in (0, 1, 127, 128, 4095, 8190, 8191)]
    rows += list(rng.integers(0, case.total_tokens, 160))
    heads = list(rng.integers(0, Hq, len(rows)))
    rows += [case.total_tokens - 1] * Hq
    heads += list(range(Hq))
    rows, heads = np.array(rows, np.int64), np.array(heads, np.int32)
    st, ro, rl = oracle.prefill_rope(H.oracle_geom(case), case.q, ref, case.block_table, 0, cu, None, case.slots,
                                     case.scale, cos_t, sin_t, rows=rows, heads=heads)
    assert st == 0
    H.assert_close(o[rows, heads], l[rows, heads], ro, rl, vmax, "rope-q 4 x 8192")

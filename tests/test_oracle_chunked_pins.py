"""Pins of the oracle's prefill over a cached prefix (chunked prefill).

The definition (tiny-vllm part 6, "논리 블록 → 물리 블록 → 바이트 주소": the
length includes the token just written and nothing past it is read; part 3,
"causalMask and online softmax": a query sees the keys up to its own
position): the i-th query of a chunk that follows `pre` cached tokens sits at
position pre + i and attends keys 0..pre + i.  Pinned against:
  * torch fp64 scaled_dot_product_attention with the bottom-right aligned
    causal mask written out on the contiguous K/V (a library routine);
  * the decode oracle: a chunk of one query at prefix seq_len - 1;
  * the fresh-prompt prefill oracle: prefix 0, and a prompt split into two
    chunks gives the same rows as the whole prompt at once;
  * a closed form: a zero query gives the mean of V over keys 0..pre + i and
    L = ln(pre + i + 1).
"""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from paged_kv_cache_gb300 import workloads as W  # noqa: E402


def oracle_pool(case):
    g = oracle.geom(*case.geom.as_tuple())
    pool = W.initial_pool(case.geom, case.pool_fill, case.seed)
    for w in case.writes:
        assert oracle.write_kv(g, pool, case.block_table, w.layer, w.tok_slot, w.tok_pos, w.k, w.v) == 0
    return pool


def f64(bits):
    return W.bf16_to_f32(bits).astype(np.float64)


def contiguous_kv(case, b):
    """K/V rows of sequence b in position order (prefix write, then chunk write)."""
    pre = int(case.extra["prefix"][b])
    n = int(case.lens[b])
    Hkv, d = case.geom.num_kv_heads, case.geom.head_dim
    parts_k, parts_v = [], []
    for w, count, first in ((case.writes[0], pre, int(np.sum(case.extra["prefix"][:b]))),
                            (case.writes[1], n, int(np.sum(case.lens[:b])))):
        parts_k.append(f64(w.k[first:first + count]))
        parts_v.append(f64(w.v[first:first + count]))
    K = np.concatenate(parts_k).reshape(-1, Hkv, d)
    V = np.concatenate(parts_v).reshape(-1, Hkv, d)
    return K, V


def sdpa_bottom_right(case):
    geom = case.geom
    Hq, Hkv, d = geom.num_q_heads, geom.num_kv_heads, geom.head_dim
    Q = f64(case.q).reshape(-1, Hq, d)
    cu = case.cu_seqlens
    sc = float(np.float32(case.scale))
    outs, lses = [], []
    for b in range(case.batch):
        pre, n = int(case.extra["prefix"][b]), int(case.lens[b])
        K, V = contiguous_kv(case, b)
        q = torch.from_numpy(Q[cu[b]:cu[b + 1]]).transpose(0, 1)
        k = torch.from_numpy(K).transpose(0, 1).repeat_interleave(Hq // Hkv, dim=0)
        v = torch.from_numpy(V).transpose(0, 1).repeat_interleave(Hq // Hkv, dim=0)
        # query i at position pre + i sees keys 0..pre + i
        allowed = torch.arange(pre + n)[None, :] <= (pre + torch.arange(n))[:, None]
        o = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=allowed, scale=sc)
        s = ((q @ k.transpose(1, 2)) * sc).masked_fill(~allowed, float("-inf"))
        outs.append(o.transpose(0, 1))
        lses.append(torch.logsumexp(s, dim=-1).transpose(0, 1))
    return torch.cat(outs).numpy(), torch.cat(lses).numpy()


@pytest.mark.parametrize("hq,hkv,d,pre,lens", [
    (8, 2, 64, [0, 16, 23], [40, 17, 1]),
    (4, 4, 64, [5, 64], [33, 64]),           # MHA
    (6, 1, 64, [100], [29]),                 # MQA
    (4, 2, 128, [31, 1], [47, 16]),          # head dim 128
])
def test_chunked_matches_library_sdpa(hq, hkv, d, pre, lens):
    nb = sum((p + n + 15) // 16 for p, n in zip(pre, lens)) + 5
    geom = W.Geometry(hq, hkv, d, 1, len(lens), 16, nb)
    case = W.make_chunked_case("sdpa", geom, pre, lens, seed=hq * 10 + d + sum(pre), pool_fill="nan")
    g = oracle.geom(*geom.as_tuple())
    st, o, lse = oracle.prefill_cached(g, case.q, oracle_pool(case), case.block_table, 0,
                                       case.cu_seqlens, case.extra["prefix"], case.slots, case.scale)
    assert st == 0
    ro, rl = sdpa_bottom_right(case)
    np.testing.assert_allclose(o, ro, rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(lse, rl, rtol=1e-12, atol=1e-12)


def test_chunk_of_one_is_decode():
    geom = W.Geometry(8, 2, 64, 1, 3, 16, 60)
    pre = np.array([0, 40, 129], np.int32)
    case = W.make_chunked_case("one", geom, pre, [1, 1, 1], seed=3, pool_fill="nan")
    g = oracle.geom(*geom.as_tuple())
    pool = oracle_pool(case)
    st, o, lse = oracle.prefill_cached(g, case.q, pool, case.block_table, 0, case.cu_seqlens, pre,
                                       case.slots, case.scale)
    st2, od, ld = oracle.decode(g, case.q, pool, case.block_table, 0, pre + 1, case.slots, case.scale)
    assert st == st2 == 0
    np.testing.assert_allclose(o, od, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(lse, ld, rtol=1e-13, atol=1e-13)


def test_prefix_zero_is_prefill_and_split_prompt_matches_whole():
    geom = W.Geometry(8, 2, 64, 1, 2, 16, 40)
    whole = W.make_chunked_case("whole", geom, [0, 0], [70, 33], seed=5)
    g = oracle.geom(*geom.as_tuple())
    pool = oracle_pool(whole)
    st, o, lse = oracle.prefill_cached(g, whole.q, pool, whole.block_table, 0, whole.cu_seqlens,
                                       [0, 0], whole.slots, whole.scale)
    st2, o2, l2 = oracle.prefill(g, whole.q, pool, whole.block_table, 0, whole.cu_seqlens, whole.slots,
                                 whole.scale)
    assert st == st2 == 0
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(lse, l2)
    # the same prompts as a first chunk (cached) and a second chunk of queries
    split = np.array([45, 9], np.int32)
    cu = whole.cu_seqlens
    rows = np.concatenate([np.arange(cu[b] + split[b], cu[b + 1]) for b in range(2)])
    q2 = whole.q[rows]
    cu2 = np.array([0, 70 - 45, 70 - 45 + 33 - 9], np.int32)
    st3, o3, l3 = oracle.prefill_cached(g, q2, pool, whole.block_table, 0, cu2, split, whole.slots,
                                        whole.scale)
    assert st3 == 0
    np.testing.assert_allclose(o3, o[rows], rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(l3, lse[rows], rtol=1e-13, atol=1e-13)


def test_zero_query_gives_mean_of_visible_values():
    geom = W.Geometry(4, 2, 64, 1, 1, 16, 20)
    pre, n = 37, 12
    case = W.make_chunked_case("zq", geom, [pre], [n], seed=9)
    case.q[:] = 0
    g = oracle.geom(*geom.as_tuple())
    st, o, lse = oracle.prefill_cached(g, case.q, oracle_pool(case), case.block_table, 0, case.cu_seqlens,
                                       [pre], case.slots, case.scale)
    assert st == 0
    K, V = contiguous_kv(case, 0)
    for i in range(n):
        for h in range(4):
            want = V[:pre + i + 1, h // 2].mean(axis=0)
            np.testing.assert_allclose(o[i, h], want, rtol=1e-12, atol=1e-12)
            assert abs(lse[i, h] - math.log(pre + i + 1)) < 1e-12


def test_rows_match_full_and_bad_prefix_rejected():
    geom = W.Geometry(8, 2, 64, 1, 2, 16, 40)
    pre = np.array([19, 64], np.int32)
    case = W.make_chunked_case("rows", geom, pre, [50, 13], seed=11)
    g = oracle.geom(*geom.as_tuple())
    pool = oracle_pool(case)
    st, o, lse = oracle.prefill_cached(g, case.q, pool, case.block_table, 0, case.cu_seqlens, pre,
                                       case.slots, case.scale)
    rows = np.array([0, 49, 50, 62, 7])
    heads = np.array([1, 7, 0, 4, 2])
    st2, os_, ls = oracle.prefill_cached_rows(g, case.q, pool, case.block_table, 0, case.cu_seqlens, pre,
                                              case.slots, case.scale, rows, heads)
    assert st == st2 == 0
    np.testing.assert_array_equal(os_, o[rows, heads])
    np.testing.assert_array_equal(ls, lse[rows, heads])
    st3, _, _ = oracle.prefill_cached(g, case.q, pool, case.block_table, 0, case.cu_seqlens, [-1, 0],
                                      case.slots, case.scale)
    assert st3 != 0

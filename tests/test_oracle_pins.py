"""Pins for the CPU oracle: it is checked against things other than itself.

* the FlashAttention-2 explainer's worked example (values printed on the page);
* the softmax stress rows quoted from the tiny-vllm softmax test;
* closed forms: q = 0 gives the running mean of V and L = ln(i + 1); causal
  row 0 gives V[0] and L = scale * <q0, k0>;
* the page layout constants and hand-worked byte offsets of the tiny-vllm
  pages, and a second statement of the layout as a numpy array shape;
* invariants: physical-page permutation, decode == prefill row, LSE split/merge;
* a library routine: torch CPU fp64 scaled_dot_product_attention on the
  contiguous K/V, including MHA (Hq == Hkv) and MQA (Hkv == 1).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_gb300 import workloads as W


def load(golden_dir, name):
    with open(os.path.join(golden_dir, name)) as f:
        return json.load(f)


def oracle_pool(case: W.Case) -> np.ndarray:
    g = oracle.geom(*case.geom.as_tuple())
    pool = W.initial_pool(case.geom, case.pool_fill, case.seed)
    for w in case.writes:
        skipped = oracle.write_kv(g, pool, case.block_table, w.layer, w.tok_slot, w.tok_pos, w.k, w.v)
        assert skipped == 0
    return pool


def f32(bits):
    return W.bf16_to_f32(bits).astype(np.float64)


# ----------------------------------------------------------- worked example

def worked_example_case(kind):
    """Encodes the worked example as attention: q = e0, k_j = x_j e0, v_j = value_j e0,
    scale 1, one q head / one kv head, d = 64, keys in 2 pages (block 1 = keys 0-1)."""
    geom = W.Geometry(1, 1, 64, 1, 1, 4, 8)
    x = [1.0, 2.0, 3.0, 0.0]
    vals = [10.0, 20.0, 30.0, 0.0]
    k = np.zeros((4, 64), np.float32)
    v = np.zeros((4, 64), np.float32)
    k[:, 0] = x
    v[:, 0] = vals
    table = W.empty_table(geom)
    table[0, 0, 0] = 6  # any page id; permutation invariance is pinned separately
    write = W.KVWrite(0, np.zeros(4, np.int32), np.arange(4, dtype=np.int32),
                      W.bf16_bits(k), W.bf16_bits(v))
    if kind == "decode":
        q = np.zeros((1, 1, 64), np.float32)
        q[0, 0, 0] = 1.0
        lens = [4]
    else:
        q = np.zeros((4, 1, 64), np.float32)
        q[:, 0, 0] = 1.0
        lens = [4]
    return W.Case("worked_" + kind, geom, 1.0, 0, np.array([0], np.int32),
                  np.array(lens, np.int32), table, [write], W.bf16_bits(q), kind, "nan", 0)


def test_worked_example_decode(golden_dir):
    gold = load(golden_dir, "fa2_worked_example.json")
    case = worked_example_case("decode")
    g = oracle.geom(*case.geom.as_tuple())
    st, o, lse = oracle.decode(g, case.q, oracle_pool(case), case.block_table, 0, case.lens,
                               case.slots, case.scale)
    assert st == 0
    fin = gold["final"]
    assert abs(o[0, 0, 0] - fin["o"]) <= fin["abs_tol"]
    assert np.all(o[0, 0, 1:] == 0.0)
    assert abs(lse[0, 0] - fin["lse"]) <= fin["abs_tol"]
    # the page's backward check: the third weight recovered from L
    bc = gold["backward_check"]
    assert abs(math.exp(3.0 - lse[0, 0]) - bc["third_weight_from_lse"]) <= bc["abs_tol"]


def test_worked_example_prefill_rows(golden_dir):
    """Row 3 sees all four keys; row 1 sees block 1 alone (O = O~/l of block 1);
    row 0 sees key 0 alone (O = 10, L = 1)."""
    gold = load(golden_dir, "fa2_worked_example.json")
    case = worked_example_case("prefill")
    g = oracle.geom(*case.geom.as_tuple())
    st, o, lse = oracle.prefill(g, case.q, oracle_pool(case), case.block_table, 0,
                                case.cu_seqlens, case.slots, case.scale)
    assert st == 0
    fin, b1 = gold["final"], gold["block1"]
    assert abs(o[3, 0, 0] - fin["o"]) <= fin["abs_tol"]
    assert abs(lse[3, 0] - fin["lse"]) <= fin["abs_tol"]
    assert abs(o[1, 0, 0] - b1["o_tilde"] / b1["l"]) <= 0.02
    assert abs(lse[1, 0] - (b1["m"] + math.log(b1["l"]))) <= 0.002
    assert o[0, 0, 0] == 10.0 and lse[0, 0] == 1.0


def test_worked_example_blocks_and_merge(golden_dir):
    gold = load(golden_dir, "fa2_worked_example.json")
    s = np.array(gold["scores"])
    v = np.array(gold["values"]).reshape(4, 1)
    parts = [oracle.partial(s[a:b], v[a:b]) for a, b in gold["blocks"]]
    b1 = gold["block1"]
    m1, l1, acc1 = parts[0]
    assert m1 == b1["m"]
    assert abs(l1 - b1["l"]) <= b1["abs_tol"]
    assert abs(acc1[0] - b1["o_tilde"]) <= b1["abs_tol"]
    b2 = gold["block2"]
    m, l, acc, o, L = oracle.merge([p[0] for p in parts], [p[1] for p in parts],
                                   [p[2] for p in parts])
    assert m == b2["m"]
    assert abs(math.exp(m1 - m) - b2["rescale"]) <= 0.001
    assert abs(acc1[0] * math.exp(m1 - m) - b2["o_tilde_rescaled"]) <= b2["abs_tol"]
    assert abs(acc[0] - b2["o_tilde"]) <= b2["abs_tol"]
    assert abs(l - b2["l"]) <= b2["abs_tol"]
    fin = gold["final"]
    assert abs(o[0] - fin["o"]) <= fin["abs_tol"]
    assert abs(L - fin["lse"]) <= fin["abs_tol"]
    w, _, _ = oracle.softmax_row(s)
    assert np.all(np.abs(w - np.array(fin["weights"])) <= 0.001)


# --------------------------------------------------------- softmax stress

def test_softmax_stress_rows(golden_dir):
    from scipy.special import logsumexp, softmax
    gold = load(golden_dir, "softmax_stress_rows.json")
    for name, row in gold["rows"].items():
        s = np.array(row, np.float64)
        w, m, l = oracle.softmax_row(s)
        assert np.all(np.isfinite(w)), name
        assert abs(w.sum() - 1.0) <= 1e-12, name
        assert abs(w.sum() - 1.0) <= gold["page_sum_tol"]
        np.testing.assert_allclose(w, softmax(s), rtol=1e-13, atol=1e-300)
        assert abs((m + math.log(l)) - logsumexp(s)) <= 1e-13 * max(1.0, abs(logsumexp(s)))
        assert m == s.max()
    w, _, _ = oracle.softmax_row(np.array(gold["rows"]["stability_spike_8"]))
    assert w[3] >= 1 - 1e-15 and np.all(w[np.arange(8) != 3] < 1e-20)
    w, _, _ = oracle.softmax_row(np.array(gold["rows"]["tied_max_8"]))
    assert np.all(w == 0.125)


def test_softmax_masked_entries():
    w, m, l = oracle.softmax_row(np.array([1.0, -np.inf, 2.0]))
    assert w[1] == 0.0 and m == 2.0
    w, m, l = oracle.softmax_row(np.array([-np.inf, -np.inf]))
    assert np.all(w == 0.0) and l == 0.0 and m == -np.inf


# ------------------------------------------------------------ page layout

def test_layout_constants_and_offsets(golden_dir):
    """Writes single distinctive rows and checks where their bytes land, against
    the page's constants and hand-worked offsets."""
    gold = load(golden_dir, "page_layout.json")
    c = gold["constants"]
    geom = W.Geometry(32, c["NUM_KV_HEADS"], c["HEAD_DIM"], c["N_LAYERS"], c["MAX_SEQUENCES"],
                      c["MAX_BLOCKS_PER_SEQ"], c["NUM_BLOCKS"])
    assert geom.kv_dim == c["KV_DIM"] and geom.page_bytes == c["BLOCK_BYTES"]
    assert geom.num_slots * geom.n_layers * geom.max_blocks_per_seq == c["TABLE_ENTRIES"]
    assert geom.pool_bytes == 2 * 1024 ** 3
    g = oracle.geom(*geom.as_tuple())
    for tc in gold["table_index_cases"]:
        # logical pages 0..block_idx of (slot, layer) sit at flat indexes index-block_idx .. index;
        # the last one points at page 7, whose first K row carries a marker
        small = oracle.geom(32, 8, 64, c["N_LAYERS"], c["MAX_SEQUENCES"], c["MAX_BLOCKS_PER_SEQ"], 8)
        table = np.full(c["TABLE_ENTRIES"], -1, np.int32)
        lo = tc["index"] - tc["block_idx"]
        table[lo:tc["index"] + 1] = np.arange(tc["block_idx"] + 1) % 7
        table[tc["index"]] = 7
        pool = np.zeros(8 * 32768, np.uint8)
        pool[7 * 32768:7 * 32768 + 2] = (0x80, 0x3F)  # bf16 1.0 at page 7, token 0, head 0, dim 0
        pos = tc["block_idx"] * 16
        st, K, V = oracle.gather_kv(small, pool, table, tc["layer"], tc["slot"], pos + 1)
        assert st == 0, tc
        assert K[pos, 0, 0] == 1.0 and np.count_nonzero(K) == 1, tc
        st, _, _ = oracle.gather_kv(small, pool, table, tc["layer"], tc["slot"], pos + 17)
        assert st == oracle.BAD_BLOCK or tc["block_idx"] == 127, tc
    for ec in gold["element_cases"]:
        blk, pos = ec["block"], ec["token_pos"]
        # place the block at logical page pos // 16 of slot 1, layer 3
        table = W.empty_table(geom)
        table[1, 3, pos // 16] = blk
        k = np.zeros((1, 512), np.uint16)
        v = np.zeros((1, 512), np.uint16)
        k[0, ec["kv_head"] * 64 + ec["dim"]] = 0x3F80  # bf16 1.0
        v[0, ec["kv_head"] * 64 + ec["dim"]] = 0x4000  # bf16 2.0
        lo = blk * 32768
        pool = np.zeros(geom.pool_bytes, np.uint8)
        pool_view = pool[lo:lo + 32768]
        assert oracle.write_kv(g, pool, table, 3, [1], [pos], k, v) == 0
        nz = np.nonzero(pool_view)[0] + lo
        # bf16 little-endian: 1.0 = 0x3F80 -> bytes (0x80, 0x3F); 2.0 = 0x4000 -> (0x00, 0x40)
        assert sorted(nz.tolist()) == sorted([ec["k_byte"], ec["k_byte"] + 1, ec["v_byte"] + 1]), ec
        assert pool[ec["k_byte"]] == 0x80 and pool[ec["k_byte"] + 1] == 0x3F
        assert pool[ec["v_byte"] + 1] == 0x40
        pool_view[:] = 0


def test_layout_as_array_shape():
    """Second statement of the layout: pool viewed as [block][K|V][token][kv head][dim]."""
    geom = W.Geometry(8, 4, 64, 3, 3, 5, 40)
    case = W.make_prefill_case("shape", geom, [37, 80, 5], seed=5, layers=(0, 2), pool_fill="zero",
                               slots=[2, 0, 1])
    pool = oracle_pool(case)
    ref = W.initial_pool(geom, "zero", 0).view(np.uint16).reshape(
        geom.num_blocks, 2, 16, geom.num_kv_heads, geom.head_dim)
    for w in case.writes:
        for i in range(w.tok_slot.shape[0]):
            blk = case.block_table[w.tok_slot[i], w.layer, w.tok_pos[i] // 16]
            ref[blk, 0, w.tok_pos[i] % 16] = w.k[i].reshape(geom.num_kv_heads, geom.head_dim)
            ref[blk, 1, w.tok_pos[i] % 16] = w.v[i].reshape(geom.num_kv_heads, geom.head_dim)
    assert np.array_equal(pool, ref.reshape(-1).view(np.uint8))


def test_write_kv_rejects_invalid_rows():
    geom = W.Geometry(4, 2, 64, 2, 2, 2, 4)
    g = oracle.geom(*geom.as_tuple())
    table = W.empty_table(geom)
    table[0, 1, 0] = 3
    table[1, 1, 0] = 7  # out of range block id
    pool = np.zeros(geom.pool_bytes, np.uint8)
    k = np.ones((5, 128), np.uint16)
    slots = [0, 1, 0, 2, -1]
    pos = [4, 0, 16, 0, 0]  # ok, bad block, unassigned page, bad slot, bad slot
    assert oracle.write_kv(g, pool, table, 1, slots, pos, k, k) == 4
    assert np.count_nonzero(pool) > 0
    assert oracle.write_kv(g, pool, table, 2, [0], [0], k[:1], k[:1]) == 1  # bad layer
    st, _, _ = oracle.gather_kv(g, pool, table, 1, 0, 17)
    assert st == oracle.BAD_BLOCK


# ---------------------------------------------------------- closed forms

def test_zero_query_gives_running_mean():
    geom = W.Geometry(8, 2, 64, 1, 2, 8, 64)
    case = W.make_prefill_case("mean", geom, [50, 33], seed=11, pool_fill="nan")
    case.q[:] = 0
    g = oracle.geom(*geom.as_tuple())
    st, o, lse = oracle.prefill(g, case.q, oracle_pool(case), case.block_table, 0,
                                case.cu_seqlens, case.slots, case.scale)
    assert st == 0
    w = case.writes[0]
    Vall = f32(w.v).reshape(-1, 2, 64)
    cu = case.cu_seqlens
    for b in range(2):
        V = Vall[cu[b]:cu[b + 1]]
        for i in range(case.lens[b]):
            mean = V[:i + 1].mean(axis=0)  # [kv head][d]
            for h in range(8):
                np.testing.assert_allclose(o[cu[b] + i, h], mean[h // 4], rtol=0, atol=1e-12)
                assert abs(lse[cu[b] + i, h] - math.log(i + 1)) <= 1e-12


def test_causal_row0_is_first_value():
    geom = W.Geometry(12, 3, 128, 1, 1, 4, 16)
    case = W.make_prefill_case("row0", geom, [45], seed=12, scale=0.3)
    g = oracle.geom(*geom.as_tuple())
    st, o, lse = oracle.prefill(g, case.q, oracle_pool(case), case.block_table, 0,
                                case.cu_seqlens, case.slots, case.scale)
    assert st == 0
    K0 = f32(case.writes[0].k[0]).reshape(3, 128)
    V0 = f32(case.writes[0].v[0]).reshape(3, 128)
    q0 = f32(case.q[0])
    for h in range(12):
        np.testing.assert_array_equal(o[0, h], V0[h // 4])
        s00 = float(np.float32(0.3)) * float(q0[h] @ K0[h // 4])
        assert abs(lse[0, h] - s00) <= 1e-12 * max(1.0, abs(s00))


def test_decode_empty_sequence():
    geom = W.Geometry(4, 1, 64, 1, 2, 2, 4)
    g = oracle.geom(*geom.as_tuple())
    st, o, lse = oracle.decode(g, np.ones((2, 4, 64), np.uint16), np.zeros(geom.pool_bytes, np.uint8),
                               W.empty_table(geom), 0, [0, 0], [0, 1], 0.125)
    assert st == 0 and np.all(o == 0) and np.all(lse == -np.inf)


# ------------------------------------------------------------- invariants

def permute_pages(case: W.Case, pool: np.ndarray, seed: int):
    """Moves every page to a new physical id, bytes and table together."""
    geom = case.geom
    perm = np.random.default_rng(seed).permutation(geom.num_blocks)
    pages = pool.reshape(geom.num_blocks, geom.page_bytes)
    new_pool = np.empty_like(pages)
    new_pool[perm] = pages
    table = case.block_table.copy()
    table[table >= 0] = perm[table[table >= 0]]
    return new_pool.reshape(-1), table


def test_page_permutation_invariance():
    geom = W.Geometry(8, 2, 64, 2, 3, 6, 30)
    case = W.make_prefill_case("perm", geom, [70, 16, 3], seed=13, layers=(1,))
    g = oracle.geom(*geom.as_tuple())
    pool = oracle_pool(case)
    st, o1, l1 = oracle.prefill(g, case.q, pool, case.block_table, 1, case.cu_seqlens, case.slots,
                                case.scale)
    pool2, table2 = permute_pages(case, pool, 99)
    assert not np.array_equal(table2, case.block_table)
    st2, o2, l2 = oracle.prefill(g, case.q, pool2, table2, 1, case.cu_seqlens, case.slots,
                                 case.scale)
    assert st == st2 == 0
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_decode_equals_prefill_row():
    pre, dec = W.tiny_case()
    g = oracle.geom(*pre.geom.as_tuple())
    pool = oracle_pool(dec)  # all 41 tokens written
    # prefill over all 41 tokens with the decode query placed at row 40
    q = np.concatenate([pre.q, dec.q], axis=0)
    st, o, lse = oracle.prefill(g, q, pool, dec.block_table, 0, [0, 41], [0], dec.scale)
    st2, od, ld = oracle.decode(g, dec.q, pool, dec.block_table, 0, [41], [0], dec.scale)
    assert st == st2 == 0
    np.testing.assert_array_equal(o[40], od[0])
    np.testing.assert_array_equal(lse[40], ld[0])


def test_lse_split_merge_identity():
    rng = np.random.default_rng(21)
    for n in (1, 5, 64, 300):
        s = rng.standard_normal(n) * 4
        v = rng.standard_normal((n, 7))
        m0, l0, acc0 = oracle.partial(s, v)
        cuts = np.sort(rng.choice(np.arange(1, n), size=min(3, n - 1), replace=False)) if n > 1 else []
        bounds = [0] + list(cuts) + [n]
        parts = [oracle.partial(s[a:b], v[a:b]) for a, b in zip(bounds[:-1], bounds[1:])]
        # an empty part (no keys) must not change the result
        parts.append((-np.inf, 0.0, np.zeros(7)))
        m, l, acc, o, L = oracle.merge([p[0] for p in parts], [p[1] for p in parts],
                                       [p[2] for p in parts])
        assert m == m0
        assert abs(l - l0) <= 1e-12 * l0
        np.testing.assert_allclose(acc, acc0, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(o, acc0 / l0, rtol=1e-12, atol=1e-12)
        assert abs(L - (m0 + math.log(l0))) <= 1e-12 * max(1, abs(L))


# ------------------------------------------------------- library routine

def sdpa_reference(case: W.Case):
    """torch fp64 SDPA (causal) on the contiguous K/V of each sequence, heads
    repeated per GQA group; L from torch.logsumexp of the masked scores."""
    geom = case.geom
    w = [x for x in case.writes if x.layer == case.layer][0]
    Hq, Hkv, d = geom.num_q_heads, geom.num_kv_heads, geom.head_dim
    K = torch.from_numpy(f32(w.k)).reshape(-1, Hkv, d)
    V = torch.from_numpy(f32(w.v)).reshape(-1, Hkv, d)
    Q = torch.from_numpy(f32(case.q)).reshape(-1, Hq, d)
    cu = case.cu_seqlens
    outs, lses = [], []
    for b in range(case.batch):
        q = Q[cu[b]:cu[b + 1]].transpose(0, 1)  # [Hq][n][d]
        k = K[cu[b]:cu[b + 1]].transpose(0, 1).repeat_interleave(Hq // Hkv, dim=0)
        v = V[cu[b]:cu[b + 1]].transpose(0, 1).repeat_interleave(Hq // Hkv, dim=0)
        o = torch.nn.functional.scaled_dot_product_attention(
            q, k, v, is_causal=True, scale=float(np.float32(case.scale)))
        n = q.shape[1]
        s = (q @ k.transpose(1, 2)) * float(np.float32(case.scale))
        s = s.masked_fill(torch.triu(torch.ones(n, n, dtype=torch.bool), 1), float("-inf"))
        outs.append(o.transpose(0, 1))
        lses.append(torch.logsumexp(s, dim=-1).transpose(0, 1))
    return torch.cat(outs).numpy(), torch.cat(lses).numpy()


@pytest.mark.parametrize("hq,hkv,d,lens", [
    (8, 2, 64, [40]),            # the tiny configuration's shape
    (4, 4, 64, [33, 1, 17]),     # MHA
    (6, 1, 64, [29, 64]),        # MQA
    (4, 2, 128, [47, 16]),       # head dim 128
    (32, 8, 64, [17, 48]),       # Llama-3.2-1B head layout
])
def test_prefill_matches_library_sdpa(hq, hkv, d, lens):
    nb = sum((n + 15) // 16 for n in lens) + 5
    geom = W.Geometry(hq, hkv, d, 1, len(lens), 8, nb)
    case = W.make_prefill_case("sdpa", geom, lens, seed=hq * 100 + d + len(lens), pool_fill="nan")
    g = oracle.geom(*geom.as_tuple())
    st, o, lse = oracle.prefill(g, case.q, oracle_pool(case), case.block_table, 0,
                                case.cu_seqlens, case.slots, case.scale)
    assert st == 0
    ro, rl = sdpa_reference(case)
    np.testing.assert_allclose(o, ro, rtol=1e-11, atol=1e-11)
    np.testing.assert_allclose(lse, rl, rtol=1e-12, atol=1e-12)


def test_decode_matches_library_sdpa():
    geom = W.Geometry(8, 2, 64, 1, 3, 8, 40)
    case = W.make_decode_case("dsdpa", geom, [1, 37, 100], seed=31, pool_fill="nan",
                              split_last_write=False)
    g = oracle.geom(*geom.as_tuple())
    st, o, lse = oracle.decode(g, case.q, oracle_pool(case), case.block_table, 0, case.lens,
                               case.slots, case.scale)
    assert st == 0
    w = case.writes[0]
    K = torch.from_numpy(f32(w.k)).reshape(-1, 2, 64)
    V = torch.from_numpy(f32(w.v)).reshape(-1, 2, 64)
    cu = case.cu_seqlens
    for b in range(3):
        q = torch.from_numpy(f32(case.q[b])).reshape(8, 1, 64)
        k = K[cu[b]:cu[b + 1]].transpose(0, 1).repeat_interleave(4, dim=0)
        v = V[cu[b]:cu[b + 1]].transpose(0, 1).repeat_interleave(4, dim=0)
        sc = float(np.float32(case.scale))
        ro = torch.nn.functional.scaled_dot_product_attention(q, k, v, scale=sc)[:, 0]
        rl = torch.logsumexp((q @ k.transpose(1, 2))[:, 0] * sc, dim=-1)
        np.testing.assert_allclose(o[b], ro.numpy(), rtol=1e-11, atol=1e-11)
        np.testing.assert_allclose(lse[b], rl.numpy(), rtol=1e-12, atol=1e-12)


def test_prefill_rows_match_full():
    geom = W.Geometry(8, 2, 64, 1, 2, 8, 20)
    case = W.make_prefill_case("rows", geom, [60, 21], seed=41)
    g = oracle.geom(*geom.as_tuple())
    pool = oracle_pool(case)
    st, o, lse = oracle.prefill(g, case.q, pool, case.block_table, 0, case.cu_seqlens,
                                case.slots, case.scale)
    rows = np.array([0, 59, 60, 80, 33])
    heads = np.array([0, 7, 3, 5, 1])
    st2, os_, ls = oracle.prefill_rows(g, case.q, pool, case.block_table, 0, case.cu_seqlens,
                                       case.slots, case.scale, rows, heads)
    assert st == st2 == 0
    np.testing.assert_array_equal(os_, o[rows, heads])
    np.testing.assert_array_equal(ls, lse[rows, heads])

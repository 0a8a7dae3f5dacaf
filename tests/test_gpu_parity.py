"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle.

Bar: the KV scatter is bit-exact over the whole pool image; bf16 outputs
within max-abs 1e-2 * max|V| (V read by the call); L within 1e-3.  Every
workload of the five configurations runs at full size; where the oracle would
be slow (the 4 x 8192 prefill) it checks sampled rows, and properties that
hold for every row are checked over all of them.
"""
import numpy as np
import pytest

import oracle
import paged_kv_cache_gb300 as pa
from paged_kv_cache_gb300 import workloads as W
from tests import helpers as H

pytestmark = pytest.mark.gpu


def _pool_equal(case, pool_dev, writes=None):
    ref = H.oracle_pool(case, writes)
    got = pool_dev.cpu().numpy()
    if not np.array_equal(got, ref):
        diff = np.nonzero(got != ref)[0]
        raise AssertionError("pool differs at %d bytes, first at %d" % (diff.size, diff[0]))
    return ref


# ------------------------------------------------------------- tiny (40 tokens)

def test_tiny_prefill_write_decode():
    pre, dec = W.tiny_case()
    pool, bt, werr = H.gpu_setup(pre)
    assert werr == 0
    ref_pool = _pool_equal(pre, pool)
    o, l, err = H.gpu_prefill(pre, pool, bt)
    assert err == 0
    ro, rl = H.oracle_prefill(pre, ref_pool)
    H.assert_close(o, l, ro, rl, H.max_abs_v(pre), "c1 prefill")
    # the new token at position 40, then a decode of length 41
    assert H.gpu_write(dec, pool, bt, writes=dec.writes[-1:]) == 0
    ref_pool = _pool_equal(dec, pool)
    od, ld, err = H.gpu_decode(dec, pool, bt)
    assert err == 0
    rod, rld = H.oracle_decode(dec, ref_pool)
    H.assert_close(od, ld, rod, rld, H.max_abs_v(dec), "c1 decode")
    # cross-path: decode at position 40 equals prefill row 40 of the same cache
    both = W.Case("c1_41", dec.geom, dec.scale, 0, dec.slots, np.array([41], np.int32),
                  dec.block_table, dec.writes, np.concatenate([pre.q, dec.q]), "prefill")
    op, lp_, err = H.gpu_prefill(both, pool, bt)
    assert err == 0
    H.assert_close(od[0], ld[0], op[40], lp_[40], H.max_abs_v(dec), "decode vs prefill row 40")


# ------------------------------------------------ Llama-3.2-1B prompts

def test_llama_prefill_layers_0_and_15():
    case = W.llama_prefill_case()
    pool, bt, werr = H.gpu_setup(case)
    assert werr == 0
    ref_pool = _pool_equal(case, pool)
    for layer in (15, 0):
        case.layer = layer
        o, l, err = H.gpu_prefill(case, pool, bt)
        assert err == 0
        ro, rl = H.oracle_prefill(case, ref_pool)
        H.assert_close(o, l, ro, rl, H.max_abs_v(case), "c2 prefill layer %d" % layer)


# ------------------------------------------- 64-sequence decode batch

def test_uniform_decode_batch():
    case = W.uniform_decode_case(pool_fill="nan")
    pool, bt, werr = H.gpu_setup(case)
    assert werr == 0
    ref_pool = _pool_equal(case, pool)
    o, l, err = H.gpu_decode(case, pool, bt)
    assert err == 0
    ro, rl = H.oracle_decode(case, ref_pool)
    H.assert_close(o, l, ro, rl, H.max_abs_v(case), "c3 decode")


# --------------------------------------------- long prefill 4 x 8192

def _sample_rows(case, rng, n_random=160):
    cu = case.cu_seqlens
    rows, heads = [], []
    Hq = case.geom.num_q_heads
    for b in range(case.batch):
        n = int(case.lens[b])
        for r in (0, 1, 127, 128, 129, n // 2, n - 129, n - 128, n - 2, n - 1):
            if 0 <= r < n:
                rows.append(cu[b] + r)
                heads.append(int(rng.integers(Hq)))
    rows += list(rng.integers(0, case.total_tokens, n_random))
    heads += list(rng.integers(0, Hq, n_random))
    # every head of the last row
    rows += [case.total_tokens - 1] * Hq
    heads += list(range(Hq))
    return np.array(rows, np.int64), np.array(heads, np.int32)


@pytest.mark.parametrize("variant", ["d64", "d128"])
def test_long_prefill_sampled_and_one_whole_sequence(variant):
    """The 4 x 8192 bench workload in the bench's launch configuration: every
    output finite and bounded by max|V|; sampled (row, head) outputs of all
    four sequences, and every (row, q head) output of the last sequence (all
    64 row tiles x every head, so each tile position of the heaviest-first
    grid and each head of each CTA's group is compared), against the oracle."""
    case = W.long_prefill_case(variant)
    pool, bt, werr = H.gpu_setup(case)
    assert werr == 0
    o, l, err = H.gpu_prefill(case, pool, bt)
    assert err == 0
    vmax = H.max_abs_v(case)
    # every row: finite, and a convex combination of V is bounded by max|V|
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(l))
    assert np.max(np.abs(o)) <= vmax * (1 + 2 ** -7)
    ref_pool = H.oracle_pool(case)
    rows, heads = _sample_rows(case, np.random.default_rng(7))
    st, ro, rl = oracle.prefill_rows(H.oracle_geom(case), case.q, ref_pool, case.block_table, 0,
                                     case.cu_seqlens, case.slots, case.scale, rows, heads)
    assert st == 0
    H.assert_close(o[rows, heads], l[rows, heads], ro, rl, vmax, "c4 " + variant)
    # every output of the last sequence
    b = case.batch - 1
    Hq = case.geom.num_q_heads
    seq_rows = np.arange(case.cu_seqlens[b], case.cu_seqlens[b + 1], dtype=np.int64)
    rows = np.repeat(seq_rows, Hq)
    heads = np.tile(np.arange(Hq, dtype=np.int32), seq_rows.shape[0])
    st, ro, rl = oracle.prefill_rows(H.oracle_geom(case), case.q, ref_pool, case.block_table, 0,
                                     case.cu_seqlens, case.slots, case.scale, rows, heads)
    assert st == 0
    H.assert_close(o[rows, heads], l[rows, heads], ro, rl, vmax, "c4 %s, sequence %d, every output" % (variant, b))


# ------------------------------------ 256-sequence mixed decode batch

def test_lognormal_decode_step():
    case = W.lognormal_decode_case(pool_fill="nan")
    pool = H.device_pool(case)
    bt = H.to_dev(case.block_table)
    assert H.gpu_write(case, pool, bt, writes=case.writes[:-1]) == 0  # preload c-1 tokens
    assert H.gpu_write(case, pool, bt, writes=case.writes[-1:]) == 0  # the new token
    ref_pool = _pool_equal(case, pool)
    o, l, err = H.gpu_decode(case, pool, bt)
    assert err == 0
    ro, rl = H.oracle_decode(case, ref_pool)
    H.assert_close(o, l, ro, rl, H.max_abs_v(case), "c5 decode")


# ---------------------------------------------------------- edge cases

RAGGED = [1, 15, 16, 17, 127, 128, 129, 255, 256, 300]


@pytest.mark.parametrize("hq,hkv,d", [(8, 2, 64), (8, 2, 128), (4, 4, 64), (6, 1, 64), (16, 2, 128)])
def test_prefill_ragged_lengths(hq, hkv, d):
    lens = RAGGED
    nb = sum((n + 15) // 16 for n in lens) + 9
    geom = W.Geometry(hq, hkv, d, 2, len(lens) + 1, 32, nb)
    case = W.make_prefill_case("ragged", geom, lens, seed=hq * 7 + d, layers=(1,), pool_fill="nan",
                               slots=list(range(1, len(lens) + 1)))
    pool, bt, werr = H.gpu_setup(case)
    assert werr == 0
    ref_pool = _pool_equal(case, pool)
    o, l, err = H.gpu_prefill(case, pool, bt)
    assert err == 0
    ro, rl = H.oracle_prefill(case, ref_pool)
    H.assert_close(o, l, ro, rl, H.max_abs_v(case), "ragged prefill %s" % ((hq, hkv, d),))


@pytest.mark.parametrize("hq,hkv,d", [(8, 2, 64), (32, 8, 64), (8, 8, 64), (16, 8, 64), (32, 4, 64),
                                      (16, 4, 128), (8, 1, 128)])
def test_decode_ragged_lengths(hq, hkv, d):
    lens = [0, 1, 15, 16, 17, 33, 500, 2048, 2049, 7, 0, 1000]
    nb = sum((n + 15) // 16 for n in lens) + 11
    geom = W.Geometry(hq, hkv, d, 1, len(lens), 160, nb)
    case = W.make_decode_case("ragged_dec", geom, lens, seed=hq + d, pool_fill="nan")
    pool, bt, werr = H.gpu_setup(case)
    assert werr == 0
    ref_pool = _pool_equal(case, pool)
    o, l, err = H.gpu_decode(case, pool, bt)
    assert err == 0
    ro, rl = H.oracle_decode(case, ref_pool)
    H.assert_close(o, l, ro, rl, H.max_abs_v(case), "ragged decode %s" % ((hq, hkv, d),))
    assert np.all(o[0] == 0) and np.all(l[0] == -np.inf)  # empty sequence


def test_decode_many_splits_and_tiny_batch():
    """One long sequence split over every CTA, and lengths that leave CTAs empty.
    [16] * 63 + [16384] and [400] * 60 + [2500] * 4: 2048 (sequence, head) rows
    take the warp-per-row merge; the long sequences' pieces (~290 and ~24) take
    its general path, in several rounds and in one."""
    for lens in ([16384], [3], [1, 1], [40] * 3, [16] * 63 + [16384], [400] * 60 + [2500] * 4):
        geom = W.Geometry(32, 8, 64, 1, len(lens), 1024, sum((n + 15) // 16 for n in lens) + 4)
        case = W.make_decode_case("splits", geom, lens, seed=len(lens), pool_fill="nan")
        pool, bt, werr = H.gpu_setup(case)
        assert werr == 0
        o, l, err = H.gpu_decode(case, pool, bt)
        assert err == 0
        ro, rl = H.oracle_decode(case, H.oracle_pool(case))
        H.assert_close(o, l, ro, rl, H.max_abs_v(case), "splits %s" % lens[:2])


def test_worked_example_on_gpu(golden_dir):
    """The FlashAttention-2 explainer's worked example through both GPU kernels."""
    from tests.test_oracle_pins import worked_example_case
    import json
    import os
    gold = json.load(open(os.path.join(golden_dir, "fa2_worked_example.json")))
    for kind in ("decode", "prefill"):
        case = worked_example_case(kind)
        pool, bt, werr = H.gpu_setup(case)
        assert werr == 0
        if kind == "decode":
            o, l, err = H.gpu_decode(case, pool, bt)
            o0, l0 = o[0, 0, 0], l[0, 0]
        else:
            o, l, err = H.gpu_prefill(case, pool, bt)
            o0, l0 = o[3, 0, 0], l[3, 0]
        assert err == 0
        # nearest bf16 of 24.93 is 24.875; the tolerance is 1e-2 * max|V| = 0.3
        assert abs(o0 - gold["final"]["o"]) <= 0.3
        assert abs(l0 - gold["final"]["lse"]) <= gold["final"]["abs_tol"]


# ------------------------------------------------------ invariants / errors

def _permuted(case, seed):
    perm = np.random.default_rng(seed).permutation(case.geom.num_blocks)
    table = case.block_table.copy()
    table[table >= 0] = perm[table[table >= 0]]
    c2 = W.Case(case.name + "_perm", case.geom, case.scale, case.layer, case.slots, case.lens, table,
                case.writes, case.q, case.kind, case.pool_fill, case.seed)
    return c2


def test_page_permutation_bit_identical():
    geom = W.Geometry(16, 4, 64, 1, 5, 64, 400)
    pre = W.make_prefill_case("perm_p", geom, [300, 77, 1, 130, 16], seed=3, pool_fill="nan")
    dec = W.make_decode_case("perm_d", geom, [300, 77, 1, 1000, 16], seed=4, pool_fill="nan")
    for case, run in ((pre, H.gpu_prefill), (dec, H.gpu_decode)):
        pool, bt, _ = H.gpu_setup(case)
        o1, l1, e1 = run(case, pool, bt)
        o1b, l1b, _ = run(case, pool, bt)
        assert np.array_equal(o1, o1b) and np.array_equal(l1, l1b), "run-to-run"
        c2 = _permuted(case, 11)
        pool2, bt2, _ = H.gpu_setup(c2)
        o2, l2, e2 = run(c2, pool2, bt2)
        assert e1 == e2 == 0
        assert np.array_equal(o1, o2) and np.array_equal(l1, l2), case.kind


def test_output_may_alias_query():
    geom = W.Geometry(8, 2, 64, 1, 3, 32, 80)
    pre = W.make_prefill_case("alias_p", geom, [200, 5, 129], seed=5, pool_fill="nan")
    dec = W.make_decode_case("alias_d", geom, [200, 5, 129], seed=6, pool_fill="nan")
    pool, bt, _ = H.gpu_setup(pre)
    o_ref, l_ref, _ = H.gpu_prefill(pre, pool, bt)
    q = H.to_dev(pre.q)
    o_al, l_al, err = H.gpu_prefill(pre, pool, bt, q=q, o=q)
    assert err == 0 and np.array_equal(o_ref, o_al) and np.array_equal(l_ref, l_al)
    pool, bt, _ = H.gpu_setup(dec)
    o_ref, l_ref, _ = H.gpu_decode(dec, pool, bt)
    q = H.to_dev(dec.q)
    o_al, l_al, err = H.gpu_decode(dec, pool, bt, q=q, o=q)
    assert err == 0 and np.array_equal(o_ref, o_al) and np.array_equal(l_ref, l_al)


def test_prefill_output_16_byte_aligned():
    """o 16 bytes past a 32-byte boundary (the least alignment the call takes):
    the rows go out in 16-byte stores instead of whole sectors, with the same
    bytes as an aligned o."""
    import torch
    geom = W.Geometry(8, 2, 64, 1, 3, 32, 80)
    pre = W.make_prefill_case("o16", geom, [200, 5, 129], seed=9, pool_fill="nan")
    pool, bt, _ = H.gpu_setup(pre)
    o_ref, l_ref, _ = H.gpu_prefill(pre, pool, bt)
    T, hq, d = pre.total_tokens, geom.num_q_heads, geom.head_dim
    flat = torch.zeros(T * hq * d + 8, dtype=torch.int16, device="cuda")
    o16 = flat[8:].view(T, hq, d)
    assert o16.data_ptr() % 32 == 16
    o_al, l_al, err = H.gpu_prefill(pre, pool, bt, o=o16)
    assert err == 0 and np.array_equal(o_ref, o_al) and np.array_equal(l_ref, l_al)
    assert np.all(flat[:8].cpu().numpy() == 0)  # nothing written before o


def test_bad_table_entries_report_and_recover():
    import torch
    geom = W.Geometry(8, 2, 64, 1, 2, 16, 40)
    pre = W.make_prefill_case("bad_p", geom, [100, 40], seed=8, pool_fill="nan")
    pool, bt, _ = H.gpu_setup(pre)
    broken = pre.block_table.copy()
    broken[0, 0, 2] = -1
    broken[1, 0, 1] = geom.num_blocks + 5
    bt_bad = H.to_dev(broken)
    _, _, err = H.gpu_prefill(pre, pool, bt_bad)
    assert err == pa.PA_ERR_BAD_BLOCK
    dec = W.Case("bad_d", geom, pre.scale, 0, pre.slots, pre.lens, broken, pre.writes,
                 pre.q[[99, 139]], "decode")
    _, _, err = H.gpu_decode(dec, pool, bt_bad)
    assert err == pa.PA_ERR_BAD_BLOCK
    # write with one bad row: the others land, the flag is set
    k = np.arange(3 * 128, dtype=np.uint16).reshape(3, 128)
    w = W.KVWrite(0, np.array([0, 5, 1], np.int32), np.array([3, 0, 17], np.int32), k, k)
    errt = torch.zeros(1, dtype=torch.int32, device="cuda")
    H.gpu_write(pre, pool, bt, writes=[w], err=errt)
    assert int(errt.item()) == pa.PA_ERR_BAD_BLOCK
    good = W.KVWrite(0, w.tok_slot[[0, 2]], w.tok_pos[[0, 2]], k[[0, 2]], k[[0, 2]])
    _pool_equal(pre, pool, writes=pre.writes + [good])
    # the next correct calls pass
    o, l, err = H.gpu_prefill(pre, pool, bt)
    assert err == 0
    pre_ref_pool = H.oracle_pool(pre, pre.writes + [good])
    ro, rl = H.oracle_prefill(pre, pre_ref_pool)
    H.assert_close(o, l, ro, rl, H.max_abs_v(pre), "after bad table")


def test_host_validation_errors():
    import torch
    geom = W.Geometry(8, 2, 64, 1, 1, 4, 8)
    g = pa.geom(*geom.as_tuple())
    pool = torch.zeros(geom.pool_bytes, dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    bt = torch.zeros((1, 1, 4), dtype=torch.int32, device="cuda")
    ks = torch.zeros(1, dtype=torch.int32, device="cuda")
    rows = torch.zeros((1, 128), dtype=torch.int16, device="cuda")
    with pytest.raises(pa.PaError) as e:
        pa.pa_write_kv(g, pool, bt, 3, ks, ks, rows, rows, err)  # layer out of range
    assert e.value.code == pa.PA_ERR_INVALID_ARG
    with pytest.raises(pa.PaError):
        pa.pa_write_kv(g, pool, bt, 0, ks, ks, pool[16:], rows, err)  # rows inside the pool
    g96 = pa.geom(8, 2, 96, 1, 1, 4, 8)
    q = torch.zeros((4, 8, 96), dtype=torch.int16, device="cuda")
    with pytest.raises(pa.PaError) as e:
        pa.pa_prefill(g96, q, pool, bt, 0, torch.zeros(2, dtype=torch.int32, device="cuda"), ks, 4,
                      0.1, q, None, err)
    assert e.value.code == pa.PA_ERR_UNSUPPORTED
    qd = torch.zeros((1, 8, 64), dtype=torch.int16, device="cuda")
    ws = torch.zeros(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(pa.PaError) as e:
        pa.pa_decode(g, qd, pool, bt, 0, ks, ks, 64, 0.1, qd, None, ws, err)  # workspace too small
    assert e.value.code == pa.PA_ERR_INVALID_ARG
    assert int(err.item()) == 0


# -------------------------------------------- running-max paths of the softmax

def _scale_keys(case, factor_of_pos):
    """Multiplies each token's K row by factor_of_pos(pos) (then rounds to bf16)."""
    out = []
    for w in case.writes:
        f = factor_of_pos(w.tok_pos.astype(np.float32))[:, None]
        k = W.bf16_bits(W.bf16_to_f32(w.k) * f)
        out.append(W.KVWrite(w.layer, w.tok_slot, w.tok_pos, k, w.v))
    case.writes = out
    return case


@pytest.mark.parametrize("kind", ["prefill", "decode"])
def test_growing_scores_move_the_reference_max(kind):
    """Keys whose magnitude grows with position: the running max keeps rising,
    so the reference max moves (and O is rescaled) many times per row."""
    geom = W.Geometry(8, 2, 64, 1, 3, 64, 120)
    lens = [700, 300, 129]
    mk = W.make_prefill_case if kind == "prefill" else W.make_decode_case
    case = mk("ramp", geom, lens, seed=91, pool_fill="nan")
    _scale_keys(case, lambda pos: 0.25 + pos / 60.0)
    pool, bt, werr = H.gpu_setup(case)
    assert werr == 0
    run = H.gpu_prefill if kind == "prefill" else H.gpu_decode
    o, l, err = run(case, pool, bt)
    assert err == 0
    ref = H.oracle_prefill if kind == "prefill" else H.oracle_decode
    ro, rl = ref(case, H.oracle_pool(case))
    H.assert_close(o, l, ro, rl, H.max_abs_v(case), "ramp " + kind)


def _second_half_moves(case):
    """How many (row, q head, key tile) steps of a d-64 prefill move the
    reference max in the tile's second 32-key half, by more than 2^8 past a
    reference the first half may already have moved (host arithmetic on the
    bf16 inputs, independent of the kernel)."""
    g, w, cu = case.geom, case.writes[0], case.cu_seqlens
    grp = g.num_q_heads // g.num_kv_heads
    K = W.bf16_to_f32(w.k).astype(np.float64).reshape(-1, g.num_kv_heads, g.head_dim)
    q = W.bf16_to_f32(case.q).astype(np.float64)
    c = case.scale * np.log2(np.e)
    count = 0
    for b, n in enumerate(case.lens):
        n = int(n)
        sel = np.where(w.tok_slot == case.slots[b])[0]
        sel = sel[np.argsort(w.tok_pos[sel])]
        for h in range(g.num_q_heads):
            s = q[cu[b]:cu[b] + n, h] @ K[sel, h // grp].T * c
            s[np.triu_indices(n, 1)] = -np.inf
            m = np.full(n, -np.inf)
            for j in range((n + 63) // 64):
                live = np.arange(n) >= 64 * j
                halves = [s[:, 64 * j + 32 * k:64 * j + 32 * k + 32] for k in (0, 1)]
                mx = [x.max(axis=1) if x.shape[1] else np.full(n, -np.inf) for x in halves]
                m = np.where(live & (mx[0] > m + 8), mx[0], m)
                moves = live & (mx[1] > m + 8)
                count += int(moves.sum())
                m = np.where(moves, mx[1], m)
    return count


@pytest.mark.parametrize("hq,hkv,d", [(8, 2, 64), (6, 1, 64), (3, 3, 64), (8, 2, 128), (4, 4, 128)])
def test_second_half_moves_the_reference(hq, hkv, d):
    """Key magnitudes that step up every 32 keys: in thousands of key tiles the
    second 32-key half exceeds the reference max by more than 2^8 after the
    first half has formed its P, which must then follow the new reference
    (with the partial sums and l).  At d 128 the same inputs take the
    max-first order.  Every move also rescales O; with two score buffers per
    tile (two or one q heads per CTA: 6 / 1 and 3 / 3 at d 64, every d-128
    case) that waits for the PV product of the key tile before."""
    geom = W.Geometry(hq, hkv, d, 1, 3, 64, 120)
    case = W.make_prefill_case("halfstep", geom, [700, 300, 129], seed=93, pool_fill="nan")
    _scale_keys(case, lambda pos: (0.25 + 0.9 * (pos // 32)).astype(np.float32))
    if d == 64 and hq == 8:
        assert _second_half_moves(case) > 1000
    pool, bt, werr = H.gpu_setup(case)
    assert werr == 0
    o, l, err = H.gpu_prefill(case, pool, bt)
    assert err == 0
    ro, rl = H.oracle_prefill(case, H.oracle_pool(case))
    H.assert_close(o, l, ro, rl, H.max_abs_v(case), "half-step keys d%d" % d)


@pytest.mark.parametrize("kind", ["prefill", "decode"])
def test_large_score_jump(kind):
    """Keys from position 300 on are 40x larger: the tile max jumps by far more
    than 2^64 over the running max: one large move of the reference max, whose
rescale factor for l and O is tiny (it may flush to zero)."""
    geom = W.Geometry(8, 2, 64, 1, 2, 64, 80)
    lens = [520, 310]
    mk = W.make_prefill_case if kind == "prefill" else W.make_decode_case
    case = mk("jump", geom, lens, seed=92, pool_fill="nan")
    _scale_keys(case, lambda pos: np.where(pos >= 300, 40.0, 0.05).astype(np.float32))
    pool, bt, werr = H.gpu_setup(case)
    assert werr == 0
    run = H.gpu_prefill if kind == "prefill" else H.gpu_decode
    o, l, err = run(case, pool, bt)
    assert err == 0
    ref = H.oracle_prefill if kind == "prefill" else H.oracle_decode
    ro, rl = ref(case, H.oracle_pool(case))
    H.assert_close(o, l, ro, rl, H.max_abs_v(case), "jump " + kind)


def test_decode_layer_and_slot_indirection():
    """A three-layer table, the decode reading layer 2 of slots that are not the
    batch index (a permutation of some of six slots), beside a chunked prefill
    reading the same layer: the table index is ((slot L) + layer) MAXB + page."""
    geom = W.Geometry(32, 8, 64, 3, 6, 40, 200)
    lens = [600, 17, 1, 300]
    slots = [5, 0, 3, 1]
    case = W.make_decode_case("layer2", geom, lens, seed=44, layer=2, slots=slots, pool_fill="nan")
    pool, bt, werr = H.gpu_setup(case)
    assert werr == 0
    o, l, err = H.gpu_decode(case, pool, bt)
    assert err == 0
    ro, rl = H.oracle_decode(case, H.oracle_pool(case))
    H.assert_close(o, l, ro, rl, H.max_abs_v(case), "decode at layer 2, slots %s" % slots)
    ccase = W.make_chunked_case("layer2c", geom, [100, 0, 33], [77, 130, 1], seed=45, layer=2, slots=[4, 2, 5],
                                pool_fill="nan")
    pool, bt, werr = H.gpu_setup(ccase)
    assert werr == 0
    o, l, err = H.gpu_prefill_cached(ccase, pool, bt)
    assert err == 0
    ro, rl = H.oracle_prefill_cached(ccase, H.oracle_pool(ccase))
    H.assert_close(o, l, ro, rl, H.max_abs_v(ccase), "chunked prefill at layer 2")

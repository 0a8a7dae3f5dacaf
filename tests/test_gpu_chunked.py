"""GPU parity of pa_prefill_cached (query chunks over a cached prefix) against
the oracle, through the C ABI.

Sizes span several 128-row query tiles and 64-key K/V tiles, prefixes that
are and are not multiples of the 16-token page and of the tiles, chunks of one
query (the decode case), ragged batches, every q-heads-per-CTA variant of the
kernel (4, 2, 1 at d 64; 2, 1 at d 128), a NaN-filled pool (no byte past a
sequence is read into the result) and bad prefixes.
"""
import numpy as np
import pytest

from paged_kv_cache_gb300 import workloads as W
from tests import helpers as H

pytestmark = pytest.mark.gpu


def run_case(case, prefix=None):
    pool, bt, werr = H.gpu_setup(case)
    assert werr == 0
    o, l, err = H.gpu_prefill_cached(case, pool, bt, prefix=prefix)
    return o, l, err


def check_full(case, what):
    o, l, err = run_case(case)
    assert err == 0, what
    ro, rl = H.oracle_prefill_cached(case, H.oracle_pool(case))
    H.assert_close(o, l, ro, rl, H.max_abs_v(case), what)


@pytest.mark.parametrize("hq,hkv,d", [(32, 8, 64), (8, 2, 64), (8, 4, 64), (6, 2, 64), (8, 8, 64),
                                      (16, 4, 128), (8, 8, 128)])
def test_chunked_heads_per_cta_variants(hq, hkv, d):
    pre = [0, 17, 128, 300]
    lens = [129, 40, 1, 200]
    nb = sum((p + n + 15) // 16 for p, n in zip(pre, lens)) + 8
    geom = W.Geometry(hq, hkv, d, 1, 4, 64, nb)
    case = W.make_chunked_case("var", geom, pre, lens, seed=hq * 7 + d, pool_fill="nan")
    check_full(case, "chunked %d/%d d%d" % (hq, hkv, d))


@pytest.mark.parametrize("pre", [1, 15, 16, 63, 64, 65, 127, 191, 1000])
def test_chunked_prefix_offsets(pre):
    lens = [130, 7, 64]
    prefixes = [pre, pre + 3, max(0, pre - 1)]
    nb = sum((p + n + 15) // 16 for p, n in zip(prefixes, lens)) + 8
    geom = W.Geometry(32, 8, 64, 1, 3, 96, nb)
    case = W.make_chunked_case("off", geom, prefixes, lens, seed=pre, pool_fill="nan")
    check_full(case, "prefix %d" % pre)


def test_null_prefix_is_prefill_bit_for_bit():
    """A null prefix array is the plain prefill, bit for bit.  Zero prefixes
    passed as an array give the same attention, but a call with a prefix
    array runs items as key halves when they leave the last wave partial
    (here: fewer items than SMs), so it agrees to rounding, and with the
    oracle."""
    geom = W.Geometry(32, 8, 64, 1, 2, 32, 80)
    case = W.make_chunked_case("null", geom, [0, 0], [300, 77], seed=2)
    pool, bt, werr = H.gpu_setup(case)
    assert werr == 0
    o1, l1, e1 = H.gpu_prefill_cached(case, pool, bt, prefix="null")
    o2, l2, e2 = H.gpu_prefill_cached(case, pool, bt, prefix=[0, 0])
    o3, l3, e3 = H.gpu_prefill(case, pool, bt)
    assert e1 == e2 == e3 == 0
    np.testing.assert_array_equal(o1, o3)
    np.testing.assert_array_equal(l1, l3)
    vmax = H.max_abs_v(case)
    H.assert_close(o2, l2, o1, l1, vmax, "zero prefixes against the null prefix")
    ro, rl = H.oracle_prefill_cached(case, H.oracle_pool(case))
    H.assert_close(o2, l2, ro, rl, vmax, "zero prefixes against the oracle")


def test_chunk_of_one_matches_decode_kernel():
    geom = W.Geometry(32, 8, 64, 1, 3, 64, 200)
    pre = np.array([0, 511, 1000], np.int32)
    case = W.make_chunked_case("one", geom, pre, [1, 1, 1], seed=4, pool_fill="nan")
    pool, bt, werr = H.gpu_setup(case)
    assert werr == 0
    o, l, err = H.gpu_prefill_cached(case, pool, bt)
    assert err == 0
    dec = W.Case("dec", geom, case.scale, 0, case.slots, pre + 1, case.block_table, case.writes, case.q,
                 "decode", case.pool_fill, case.seed)
    od, ld, errd = H.gpu_decode(dec, pool, bt)
    assert errd == 0
    H.assert_close(o, l, od.reshape(o.shape), ld.reshape(l.shape), H.max_abs_v(case), "chunk of one vs decode")
    ro, rl = H.oracle_prefill_cached(case, H.oracle_pool(case))
    H.assert_close(o, l, ro, rl, H.max_abs_v(case), "chunk of one vs oracle")


def test_split_prompt_matches_oracle_whole_prompt():
    geom = W.Geometry(32, 8, 64, 1, 2, 64, 140)
    whole = W.make_chunked_case("whole", geom, [0, 0], [700, 333], seed=6)
    pool, bt, werr = H.gpu_setup(whole)
    assert werr == 0
    split = np.array([450, 200], np.int32)
    cu = whole.cu_seqlens
    rows = np.concatenate([np.arange(cu[b] + split[b], cu[b + 1]) for b in range(2)])
    second = W.Case("second", geom, whole.scale, 0, whole.slots, whole.lens - split, whole.block_table,
                    whole.writes, whole.q[rows], "chunked", whole.pool_fill, whole.seed, extra={"prefix": split})
    o, l, err = H.gpu_prefill_cached(second, pool, bt)
    assert err == 0
    ro, rl = H.oracle_prefill(whole, H.oracle_pool(whole))
    H.assert_close(o, l, ro[rows], rl[rows], H.max_abs_v(whole), "second chunk vs whole prompt")


def test_long_prefix_sampled_rows():
    """A 2048-query chunk after 6144 cached tokens (and a short one): sampled
    (row, head) outputs against the oracle."""
    geom = W.Geometry(32, 8, 64, 1, 2, 520, 1100)
    pre = np.array([6144, 33], np.int32)
    case = W.make_chunked_case("long", geom, pre, [2048, 500], seed=8)
    o, l, err = run_case(case)
    assert err == 0
    rng = np.random.default_rng(3)
    rows = np.concatenate([[0, 127, 128, 2047, 2048, 2547], rng.integers(0, case.total_tokens, 58)])
    heads = rng.integers(0, 32, rows.shape[0]).astype(np.int32)
    ro, rl = H.oracle_prefill_cached(case, H.oracle_pool(case), rows, heads)
    H.assert_close(o[rows, heads], l[rows, heads], ro, rl, H.max_abs_v(case), "long prefix sampled")


def test_bad_prefix_reports_and_recovers():
    geom = W.Geometry(8, 2, 64, 1, 2, 8, 40)
    case = W.make_chunked_case("bad", geom, [3, 0], [20, 30], seed=10)
    pool, bt, werr = H.gpu_setup(case)
    assert werr == 0
    for bad in ([-1, 0], [3, 8 * 16 - 29]):  # negative; prefix + chunk past the table
        _, _, err = H.gpu_prefill_cached(case, pool, bt, prefix=bad)
        assert err == H.pa.PA_ERR_BAD_BLOCK
    o, l, err = H.gpu_prefill_cached(case, pool, bt)  # the context still works
    assert err == 0
    ro, rl = H.oracle_prefill_cached(case, H.oracle_pool(case))
    H.assert_close(o, l, ro, rl, H.max_abs_v(case), "after bad prefixes")


def test_chunked_bench_size_tail_launch():
    """The chunked bench workload (4 x 2048 queries after 6144 cached tokens,
    32 q / 8 kv heads, d 64): 512 four-head work items on the GPU's SMs make
    more than three waves, so the last wave's items (row tiles 0 and 1 of every
    sequence) run in a second, dependent launch as two CTAs each, one per half
    of the item's key tiles, the later of which combines both partials.
    Sampled rows of every sequence, most of them in those row tiles, against
    the oracle."""
    import oracle
    prefix, chunk = 6144, 2048
    pages = (prefix + chunk) // 16
    geom = W.Geometry(32, 8, 64, 1, 4, pages, 4 * pages + 64)
    case = W.make_chunked_case("tail", geom, [prefix] * 4, [chunk] * 4, seed=1006)
    pool, bt, werr = H.gpu_setup(case)
    assert werr == 0
    o, l, err = H.gpu_prefill_cached(case, pool, bt)
    assert err == 0
    vmax = H.max_abs_v(case)
    assert np.all(np.isfinite(o)) and np.max(np.abs(o)) <= vmax * (1 + 2 ** -7)
    rng = np.random.default_rng(23)
    cu, Hq = case.cu_seqlens, geom.num_q_heads
    rows, heads = [], []
    for b in range(case.batch):
        for r in list(rng.integers(0, 256, 24)) + [0, 127, 128, 255, 1024, chunk - 1]:
            rows.append(cu[b] + r)
            heads.append(int(rng.integers(Hq)))
    rows += [cu[1]] * Hq  # every head of one row of the tail
    heads += list(range(Hq))
    rows, heads = np.array(rows, np.int64), np.array(heads, np.int32)
    ro, rl = H.oracle_prefill_cached(case, H.oracle_pool(case), rows=rows, heads=heads)
    H.assert_close(o[rows, heads], l[rows, heads], ro, rl, vmax, "chunked bench size")


def test_key_split_is_deterministic_and_permutation_invariant():
    """Items that run as two key halves (a batch of fewer items than SMs, each
    item split; one-tile items leave the first half empty): whichever half
    finishes second combines the same fp32 partials with the same arithmetic,
    so repeated calls and a permuted page layout give the same bits; and the
    result matches the oracle."""
    pre = [0, 17, 500, 1000, 64]
    lens = [300, 40, 129, 1, 256]
    nb = sum((p + n + 15) // 16 for p, n in zip(pre, lens)) + 16
    geom = W.Geometry(32, 8, 64, 1, 5, 128, nb)
    case = W.make_chunked_case("ksplit", geom, pre, lens, seed=77, pool_fill="nan")
    pool, bt, werr = H.gpu_setup(case)
    assert werr == 0
    runs = [H.gpu_prefill_cached(case, pool, bt) for _ in range(4)]
    for o, l, err in runs:
        assert err == 0
        np.testing.assert_array_equal(o, runs[0][0])
        np.testing.assert_array_equal(l, runs[0][1])
    ro, rl = H.oracle_prefill_cached(case, H.oracle_pool(case))
    H.assert_close(runs[0][0], runs[0][1], ro, rl, H.max_abs_v(case), "key-split chunked")
    # the same logical cache on other physical pages
    rng = np.random.default_rng(5)
    perm = rng.permutation(nb).astype(np.int32)
    moved = W.Case(case.name, case.geom, case.scale, case.layer, case.slots, case.lens,
                   np.where(case.block_table >= 0, perm[np.maximum(case.block_table, 0)], -1).astype(np.int32),
                   case.writes, case.q, case.kind, case.pool_fill, case.seed, dict(case.extra))
    pool2, bt2, werr2 = H.gpu_setup(moved)
    assert werr2 == 0
    o2, l2, err2 = H.gpu_prefill_cached(moved, pool2, bt2)
    assert err2 == 0
    np.testing.assert_array_equal(o2, runs[0][0])
    np.testing.assert_array_equal(l2, runs[0][1])

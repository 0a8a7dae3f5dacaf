"""GPU parity of pa_write_kv_rope (K/V scatter with RoPE on K) against the
oracle: the whole pool must match byte for byte (the rounding to bf16 is the
same decision on both sides: fp32 products and sums, each rounded on its own,
then nearest-even)."""
import numpy as np
import pytest

import oracle
from paged_kv_cache_gb300 import workloads as W
from tests import helpers as H

pytestmark = pytest.mark.gpu


def prompt_case(hq, hkv, d, lens, seed, fill="nan"):
    nb = sum((n + 15) // 16 for n in lens) + 4
    geom = W.Geometry(hq, hkv, d, 2, len(lens), 64, nb)
    return W.make_prefill_case("rope", geom, lens, seed=seed, layers=(1,), pool_fill=fill)


def run_both(case, cos_t, sin_t, positions=None):
    torch = H.torch_mod()
    w = case.writes[0]
    pos = w.tok_pos if positions is None else np.asarray(positions, np.int32)
    g = oracle.geom(*case.geom.as_tuple())
    ref = W.initial_pool(case.geom, case.pool_fill, case.seed)
    skipped = oracle.write_kv_rope(g, ref, case.block_table, w.layer, w.tok_slot, pos, w.k, w.v, cos_t, sin_t)
    pool = H.device_pool(case)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    H.pa.pa_write_kv_rope(H.pa_geom(case), pool, H.to_dev(case.block_table), w.layer, H.to_dev(w.tok_slot),
                          H.to_dev(pos), H.to_dev(w.k), H.to_dev(w.v), H.to_dev(cos_t), H.to_dev(sin_t), err)
    torch.cuda.synchronize()
    return pool.cpu().numpy(), ref, int(err.item()), skipped


@pytest.mark.parametrize("hq,hkv,d,lens", [
    (32, 8, 64, [17, 512]),     # the Llama-3.2-1B layout
    (16, 4, 128, [300, 45]),    # head dim 128
    (8, 1, 64, [1, 77, 16]),    # one kv head
    (12, 6, 64, [33, 100]),     # two heads per K thread
    (6, 3, 32, [50, 9]),        # odd kv head count: one head per K thread
])
def test_rope_scatter_is_byte_exact(hq, hkv, d, lens):
    case = prompt_case(hq, hkv, d, lens, seed=hq + d)
    cos_t, sin_t = W.rope_tables(1024, d)
    got, ref, err, skipped = run_both(case, cos_t, sin_t)
    assert err == 0 and skipped == 0
    np.testing.assert_array_equal(got, ref)


def test_identity_table_is_plain_scatter():
    case = prompt_case(32, 8, 64, [40, 9], seed=2)
    n = 64
    cos_t = np.ones((n, 32), np.float32)
    sin_t = np.zeros((n, 32), np.float32)
    got, _, err, _ = run_both(case, cos_t, sin_t)
    pool, bt, werr = H.gpu_setup(case)
    assert err == 0 and werr == 0
    np.testing.assert_array_equal(got, pool.cpu().numpy())


def test_positions_past_the_table_are_skipped_and_reported():
    case = prompt_case(32, 8, 64, [40], seed=4)
    cos_t, sin_t = W.rope_tables(32, 64)  # rows 32..39 have no angle
    got, ref, err, skipped = run_both(case, cos_t, sin_t)
    assert skipped == 8
    assert err == H.pa.PA_ERR_BAD_BLOCK
    np.testing.assert_array_equal(got, ref)


def test_rope_write_then_prefill_matches_oracle():
    """End to end: K rotated on the way into the pages, then the prefill; the
    oracle takes the same two steps."""
    case = prompt_case(32, 8, 64, [200, 64], seed=6, fill="random")
    cos_t, sin_t = W.rope_tables(256, 64)
    got, ref, err, _ = run_both(case, cos_t, sin_t)
    assert err == 0
    torch = H.torch_mod()
    pool = torch.from_numpy(got).cuda()
    o, l, perr = H.gpu_prefill(case, pool, H.to_dev(case.block_table))
    assert perr == 0
    ro, rl = H.oracle_prefill(case, ref)
    H.assert_close(o, l, ro, rl, H.max_abs_v(case), "rope write + prefill")


@pytest.mark.parametrize("hq,hkv,d", [
    (1, 1, 8),     # one 16-byte chunk per K or V row: one chunk per thread
    (3, 3, 8),     # three chunks per row
    (2, 1, 32),    # four chunks per row: four per thread
    (1, 1, 16),    # RoPE with two V chunks per row
])
def test_narrow_rows_scatter_byte_exact(hq, hkv, d):
    """Rows whose chunk count is not a multiple of four take the one-chunk
    path of both scatters; the whole pool must still match the oracle."""
    lens = [37, 5]
    nb = sum((n + 15) // 16 for n in lens) + 4
    geom = W.Geometry(hq, hkv, d, 2, len(lens), 8, nb)
    case = W.make_prefill_case("narrow", geom, lens, seed=d + hkv, layers=(1,), pool_fill="nan")
    pool, bt, werr = H.gpu_setup(case)
    assert werr == 0
    np.testing.assert_array_equal(pool.cpu().numpy(), H.oracle_pool(case))
    if d % 16 == 0:
        cos_t, sin_t = W.rope_tables(64, d)
        got, ref, err, skipped = run_both(case, cos_t, sin_t)
        assert err == 0 and skipped == 0
        np.testing.assert_array_equal(got, ref)

"""GPU parity at the largest sizes the tests reach: a 12 GiB pool whose used
pages are spread from its start to its last page (byte offsets past 2^31 and
2^32), one 32768-token prompt (256 row tiles, up to 512 key tiles per row
tile) and a decode batch led by one 262144-token sequence (16384 pages, K
turned by RoPE on its way in).

The oracle cannot hold a 12 GiB pool image, so it runs on an equivalent
compact pool: the same writes through a table whose page p is the device's
page p * stride + stride - 1.  The device pages the table names are gathered
and compared with the compact pool byte for byte, then the attention outputs
with the oracle's at the parity bar.  Every other byte of the device pool is
0xFF (bf16 NaN), so a read of a wrong page shows in the outputs.
"""
import dataclasses

import numpy as np
import pytest

import oracle
import paged_kv_cache_gb300 as pa
from paged_kv_cache_gb300 import workloads as W
from tests import helpers as H

pytestmark = pytest.mark.gpu

POOL_BYTES = 12 << 30


def _spread(case):
    """The case on the 12 GiB pool: (device case, stride); compact page p is
    device page p * stride + stride - 1, spread evenly over the whole pool."""
    g = case.geom
    nb = POOL_BYTES // g.page_bytes
    stride = nb // g.num_blocks
    big = dataclasses.replace(g, num_blocks=nb)
    table = np.where(case.block_table >= 0, case.block_table * stride + stride - 1, -1).astype(np.int32)
    return dataclasses.replace(case, geom=big, block_table=table), stride


def _nan_pool(big_case):
    torch = H.torch_mod()
    pool = torch.empty(big_case.geom.pool_bytes, dtype=torch.uint8, device="cuda")
    pool.fill_(0xFF)
    return pool


def _pages_equal(pool, stride, small_geom, ref_pool):
    torch = H.torch_mod()
    pb = small_geom.page_bytes
    idx = torch.arange(small_geom.num_blocks, device="cuda", dtype=torch.int64) * stride + stride - 1
    got = pool.view(-1, pb).index_select(0, idx).cpu().numpy().reshape(-1)
    if not np.array_equal(got, ref_pool):
        diff = np.nonzero(got != ref_pool)[0]
        raise AssertionError("pages differ at %d bytes, first at compact byte %d" % (diff.size, diff[0]))


def test_prefill_32768_tokens_on_a_12_gib_pool():
    geom = W.Geometry(32, 8, 64, 1, 1, 2048 + 8, 2048 + 64)
    case = W.make_prefill_case("far_prefill", geom, [32768], seed=61, pool_fill="nan")
    big, stride = _spread(case)
    used = big.block_table[big.block_table >= 0]
    assert int(used.min()) * geom.page_bytes < (1 << 31) and int(used.max()) * geom.page_bytes > (1 << 33)
    pool = _nan_pool(big)
    bt = H.to_dev(big.block_table)
    assert H.gpu_write(big, pool, bt) == 0
    ref_pool = H.oracle_pool(case)
    _pages_equal(pool, stride, geom, ref_pool)
    o, l, err = H.gpu_prefill(big, pool, bt)
    assert err == 0
    vmax = H.max_abs_v(case)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(l))
    assert np.max(np.abs(o)) <= vmax * (1 + 2 ** -7)
    rng = np.random.default_rng(62)
    n, Hq = case.total_tokens, geom.num_q_heads
    rows = [0, 1, 127, 128, 16383, 16384, 32639, 32640, 32766] + list(rng.integers(0, n, 120))
    heads = list(rng.integers(0, Hq, len(rows)))
    rows += [n - 1] * Hq
    heads += list(range(Hq))
    rows, heads = np.array(rows, np.int64), np.array(heads, np.int32)
    st, ro, rl = oracle.prefill_rows(H.oracle_geom(case), case.q, ref_pool, case.block_table, 0,
                                     case.cu_seqlens, case.slots, case.scale, rows, heads)
    assert st == 0
    H.assert_close(o[rows, heads], l[rows, heads], ro, rl, vmax, "32768-token prefill, 12 GiB pool")
    del pool, bt
    H.torch_mod().cuda.empty_cache()


def test_decode_262144_tokens_rope_written_on_a_12_gib_pool():
    lens = [262144, 1, 4097]
    pages = sum((n + 15) // 16 for n in lens)
    geom = W.Geometry(32, 8, 64, 1, 3, 16384 + 8, pages + 64)
    case = W.make_decode_case("far_decode", geom, lens, seed=63, pool_fill="nan")
    big, stride = _spread(case)
    used = big.block_table[big.block_table >= 0]
    assert int(used.min()) * geom.page_bytes < (1 << 31) and int(used.max()) * geom.page_bytes > (1 << 33)
    cos_t, sin_t = W.rope_tables(262144, 64)
    g_small = H.oracle_geom(case)
    ref_pool = W.initial_pool(geom, "nan", case.seed)
    for w in case.writes:
        assert oracle.write_kv_rope(g_small, ref_pool, case.block_table, w.layer, w.tok_slot, w.tok_pos,
                                    w.k, w.v, cos_t, sin_t) == 0
    torch = H.torch_mod()
    pool = _nan_pool(big)
    bt = H.to_dev(big.block_table)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    ct, st_ = H.to_dev(cos_t), H.to_dev(sin_t)
    for w in case.writes:
        pa.pa_write_kv_rope(H.pa_geom(big), pool, bt, w.layer, H.to_dev(w.tok_slot), H.to_dev(w.tok_pos),
                            H.to_dev(w.k), H.to_dev(w.v), ct, st_, err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    _pages_equal(pool, stride, geom, ref_pool)
    o, l, derr = H.gpu_decode(big, pool, bt)
    assert derr == 0
    ro, rl = H.oracle_decode(case, ref_pool)
    H.assert_close(o, l, ro, rl, H.max_abs_v(case), "262144-token decode, 12 GiB pool")
    del pool, bt, err, ct, st_
    torch.cuda.empty_cache()

"""GPU parity of the device page lifetime (pa_alloc_pages, pa_release_slots)
against the oracle: the same operations on both sides must leave the same
block table and the same free stack, entry for entry (both walk sequences,
then layers, then logical blocks, popping or pushing the stack's top)."""
import numpy as np
import pytest

import oracle
from paged_kv_cache_gb300 import workloads as W
from tests import helpers as H

pytestmark = pytest.mark.gpu


class Pair:
    """The same state on the device and in the oracle."""

    def __init__(self, geom, seed):
        torch = H.torch_mod()
        self.geom, self.g, self.og = geom, H.pa.geom(*geom.as_tuple()), oracle.geom(*geom.as_tuple())
        rng = np.random.default_rng(seed)
        self.table = W.empty_table(geom)
        self.stack = rng.permutation(geom.num_blocks).astype(np.int32)
        self.count = np.array([geom.num_blocks], np.int32)
        self.d_table = torch.from_numpy(self.table.copy()).cuda()
        self.d_stack = torch.from_numpy(self.stack.copy()).cuda()
        self.d_count = torch.from_numpy(self.count.copy()).cuda()
        self.err = torch.zeros(1, dtype=torch.int32, device="cuda")

    def alloc(self, slots, lens, old=None):
        slots = np.asarray(slots, np.int32)
        lens = np.asarray(lens, np.int32)
        r = oracle.alloc_pages(self.og, self.table, slots, lens, self.stack, self.count, old_lens=old)
        self.err.zero_()
        H.pa.pa_alloc_pages(self.g, self.d_table, H.to_dev(slots), H.to_dev(lens), self.d_stack, self.d_count,
                            self.err, old_lens=None if old is None else H.to_dev(np.asarray(old, np.int32)))
        return r, self.check()

    def release(self, slots):
        slots = np.asarray(slots, np.int32)
        r = oracle.release_slots(self.og, self.table, slots, self.stack, self.count)
        self.err.zero_()
        H.pa.pa_release_slots(self.g, self.d_table, H.to_dev(slots), self.d_stack, self.d_count, self.err)
        return r, self.check()

    def check(self):
        H.torch_mod().cuda.synchronize()
        np.testing.assert_array_equal(self.d_table.cpu().numpy(), self.table)
        np.testing.assert_array_equal(self.d_count.cpu().numpy(), self.count)
        n = int(self.count[0])
        np.testing.assert_array_equal(self.d_stack.cpu().numpy()[:n], self.stack[:n])
        return int(self.err.item())


def test_prompt_then_decode_steps_then_release():
    geom = W.Geometry(32, 8, 64, 16, 8, 160, 20000)
    st = Pair(geom, seed=1)
    lens = np.array([17, 512, 1, 2048, 300, 0, 16, 15], np.int32)
    slots = np.arange(8, dtype=np.int32)
    r, err = st.alloc(slots, lens)
    assert err == 0 and r == int(np.sum((lens + 15) // 16)) * 16
    for _ in range(40):  # decode steps: one token each
        r, err = st.alloc(slots, lens + 1, old=lens)
        assert err == 0
        lens = lens + 1
    r, err = st.release([3, 0, 6])
    assert err == 0
    r, err = st.alloc([6, 3], [100, 33])
    assert err == 0


def test_random_operations_match_oracle():
    rng = np.random.default_rng(7)
    geom = W.Geometry(8, 2, 64, 3, 64, 32, 3000)
    st = Pair(geom, seed=7)
    lens = np.zeros(geom.num_slots, np.int32)
    for step in range(60):
        if rng.random() < 0.25:
            s = rng.choice(geom.num_slots, size=rng.integers(1, 10), replace=False).astype(np.int32)
            r, err = st.release(s)
            assert err == 0 and r >= 0
            lens[s] = 0
        else:
            s = rng.choice(geom.num_slots, size=rng.integers(1, 40), replace=False).astype(np.int32)
            new = np.minimum(lens[s] + rng.integers(0, 200, s.shape[0]), 32 * 16).astype(np.int32)
            r, err = st.alloc(s, new, old=lens[s])
            if r < 0:
                assert err == H.pa.PA_ERR_OUT_OF_PAGES
            else:
                assert err == 0
                lens[s] = new


def test_shortage_and_bad_input_change_nothing():
    geom = W.Geometry(8, 2, 64, 2, 4, 64, 30)
    st = Pair(geom, seed=3)
    r, err = st.alloc([0, 1], [160, 160])  # 2 x 2 layers x 10 blocks = 40 > 30 pages
    assert r < 0 and err == H.pa.PA_ERR_OUT_OF_PAGES
    r, err = st.alloc([1, 1], [16, 16])      # a slot named twice
    assert r < 0 and err == H.pa.PA_ERR_BAD_BLOCK
    r, err = st.alloc([2], [64 * 16 + 1])     # longer than the table row
    assert r < 0 and err == H.pa.PA_ERR_BAD_BLOCK
    r, err = st.alloc([2], [40])
    assert err == 0 and r == 6


def test_release_refusals_change_nothing():
    """A slot named twice, and a release whose pages would overflow the stack
    (a page held by two slots: freed twice), change neither the table nor the
    stack, on the device as in the oracle."""
    geom = W.Geometry(8, 2, 64, 2, 4, 64, 30)
    st = Pair(geom, seed=5)
    r, err = st.alloc([0], [160])          # 2 layers x 10 blocks: 20 of the 30 pages
    assert err == 0 and r == 20
    r, err = st.release([0, 0])
    assert r < 0 and err == H.pa.PA_ERR_BAD_BLOCK
    # slot 1's rows name slot 0's pages too: releasing both pushes 40 pages onto 10
    st.table[1] = st.table[0]
    st.d_table[1] = st.d_table[0]
    r, err = st.release([0, 1])
    assert r < 0 and err == H.pa.PA_ERR_OUT_OF_PAGES
    r, err = st.release([0])
    assert err == 0


def test_allocated_table_serves_the_attention_path():
    """Pages from the device allocator, then write + prefill against the oracle."""
    torch = H.torch_mod()
    geom = W.Geometry(32, 8, 64, 1, 3, 64, 400)
    case = W.make_prefill_case("alloc", geom, [300, 17, 129], seed=11, pool_fill="nan")
    st = Pair(geom, seed=11)
    r, err = st.alloc(case.slots, case.lens)
    assert err == 0
    case.block_table = st.table.copy()  # the oracle's (equal) table
    pool = H.device_pool(case)
    bt = st.d_table
    assert H.gpu_write(case, pool, bt) == 0
    o, l, perr = H.gpu_prefill(case, pool, bt)
    assert perr == 0
    ro, rl = H.oracle_prefill(case, H.oracle_pool(case))
    H.assert_close(o, l, ro, rl, H.max_abs_v(case), "prefill on allocated pages")

"""Pins of the oracle's page lifetime (free stack, allocation, release).

tiny-vllm part 6, "물리 블록의 수명: free_blocks 가 관리한다": pages come from
the top of a free stack (pop_back) when a logical block's entry is -1, and go
back (push_back) when a slot ends, its entries becoming -1.  Pinned against a
worked example by hand (tests/golden/page_lifetime.json), the pages' decode
rule (a step takes a page exactly when its token starts a new 16-token block),
and invariants over random operation sequences: every page is either in the
table once or on the stack once, and the lengths' blocks are all assigned.
"""
import json
import os

import numpy as np

import oracle
from paged_kv_cache_gb300 import workloads as W


def geom_of(d):
    return W.Geometry(d["num_q_heads"], d["num_kv_heads"], d["head_dim"], d["n_layers"], d["num_slots"],
                      d["max_blocks_per_seq"], d["num_blocks"])


def test_worked_example(golden_dir):
    gd = json.load(open(os.path.join(golden_dir, "page_lifetime.json")))
    geom = geom_of(gd["geometry"])
    g = oracle.geom(*geom.as_tuple())
    table = W.empty_table(geom)
    stack = np.arange(geom.num_blocks, dtype=np.int32)
    count = np.array([geom.num_blocks], np.int32)
    for st in gd["steps"]:
        if st["op"] == "alloc":
            moved = oracle.alloc_pages(g, table, st["slots"], st["seq_lens"], stack, count, old_lens=st["old_lens"])
        else:
            moved = oracle.release_slots(g, table, st["slots"], stack, count)
        assert moved == st["moved"]
        np.testing.assert_array_equal(table, np.array(st["table"], np.int32))
        np.testing.assert_array_equal(stack[:count[0]], np.array(st["stack"], np.int32))


def test_decode_takes_a_page_only_at_a_new_block():
    geom = W.Geometry(4, 2, 64, 3, 2, 8, 64)
    g = oracle.geom(*geom.as_tuple())
    table = W.empty_table(geom)
    stack = np.arange(geom.num_blocks, dtype=np.int32)
    count = np.array([geom.num_blocks], np.int32)
    assert oracle.alloc_pages(g, table, [1], [5], stack, count) == geom.n_layers
    for n in range(5, 100):  # the token at position n joins: length n -> n + 1
        before = int(count[0])
        moved = oracle.alloc_pages(g, table, [1], [n + 1], stack, count, old_lens=[n])
        want = geom.n_layers if n % 16 == 0 else 0
        assert moved == want and before - int(count[0]) == want, n


def check_conservation(geom, table, stack, count):
    held = table[table >= 0]
    free = stack[:count[0]]
    allp = np.concatenate([held, free])
    assert allp.shape[0] == geom.num_blocks
    np.testing.assert_array_equal(np.sort(allp), np.arange(geom.num_blocks))


def test_random_lifetimes_conserve_pages():
    rng = np.random.default_rng(12)
    geom = W.Geometry(8, 2, 64, 2, 6, 16, 200)
    g = oracle.geom(*geom.as_tuple())
    table = W.empty_table(geom)
    stack = rng.permutation(geom.num_blocks).astype(np.int32)
    count = np.array([geom.num_blocks], np.int32)
    lens = np.zeros(geom.num_slots, np.int32)
    for step in range(300):
        if rng.random() < 0.2:
            s = rng.choice(geom.num_slots, size=rng.integers(1, 3), replace=False).astype(np.int32)
            moved = oracle.release_slots(g, table, s, stack, count)
            assert moved == int(np.sum((lens[s] + 15) // 16)) * geom.n_layers
            lens[s] = 0
        else:
            s = rng.choice(geom.num_slots, size=rng.integers(1, 4), replace=False).astype(np.int32)
            new = np.minimum(lens[s] + rng.integers(0, 40, s.shape[0]), 16 * 16).astype(np.int32)
            snapshot = (table.copy(), stack.copy(), count.copy())
            moved = oracle.alloc_pages(g, table, s, new, stack, count, old_lens=lens[s])
            if moved < 0:  # ran short: all or nothing
                np.testing.assert_array_equal(table, snapshot[0])
                np.testing.assert_array_equal(count, snapshot[2])
                continue
            lens[s] = new
        check_conservation(geom, table, stack, count)
        for sl in range(geom.num_slots):  # exactly the blocks the length needs are assigned
            nb = (lens[sl] + 15) // 16
            assert np.all(table[sl, :, :nb] >= 0) and np.all(table[sl, :, nb:] == -1)

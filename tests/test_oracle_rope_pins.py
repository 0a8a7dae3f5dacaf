"""Pins of the oracle's RoPE scatter (orc_write_kv_rope).

tiny-vllm part 3, "RoPE: a rotation that references a table": in each head,
element i and element i + head_dim/2 form a pair, rotated by the angle of the
token's position read from cos/sin tables; V is not rotated.  Pinned against:
  * a worked example by hand (tests/golden/rope_pairing.json) that fixes the
    pairing, the signs and which table row is read;
  * special angles: no turn is the plain scatter byte for byte, a half turn
    negates K exactly, a quarter turn swaps the halves with one sign;
  * torch: the same fp32 products and sums with torch CPU ops and torch's
    float32 -> bfloat16 rounding, compared byte for byte;
  * the rotation's invariants in fp64: the norm of every pair is kept, and
    the dot product of a query and a key both rotated depends only on their
    distance (checked on the bf16 results, within bf16 rounding).
"""
import json
import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from paged_kv_cache_gb300 import workloads as W  # noqa: E402


def scatter_case(hkv=2, d=64, n=40, seed=0):
    geom = W.Geometry(2 * hkv, hkv, d, 1, 1, 8, 16)
    rng = np.random.default_rng(seed)
    table = W.empty_table(geom)
    free = W.FreeList(geom.num_blocks, rng)
    W.assign_pages(table, free, 0, 0, n)
    k = W.normal_bf16(rng, (n, hkv * d))
    v = W.normal_bf16(rng, (n, hkv * d))
    return geom, table, np.zeros(n, np.int32), np.arange(n, dtype=np.int32), k, v


def rope_pool(geom, table, slot, pos, k, v, cos_t, sin_t):
    g = oracle.geom(*geom.as_tuple())
    pool = np.zeros(geom.pool_bytes, np.uint8)
    assert oracle.write_kv_rope(g, pool, table, 0, slot, pos, k, v, cos_t, sin_t) == 0
    return pool


def gathered(geom, table, pool, n):
    """K/V rows of slot 0 as bf16 bits [n][KV_DIM] (through the page layout)."""
    kv_dim, out_k, out_v = geom.kv_dim, [], []
    for t in range(n):
        blk = table[0, 0, t // 16]
        base = blk * geom.page_bytes + (t % 16) * kv_dim * 2
        out_k.append(pool[base:base + kv_dim * 2].view(np.uint16))
        vb = base + 16 * kv_dim * 2
        out_v.append(pool[vb:vb + kv_dim * 2].view(np.uint16))
    return np.stack(out_k), np.stack(out_v)


def test_worked_example_pairing(golden_dir):
    gd = json.load(open(os.path.join(golden_dir, "rope_pairing.json")))
    d = gd["head_dim"]
    geom = W.Geometry(1, 1, d, 1, 1, 1, 1)
    table = np.zeros((1, 1, 1), np.int32)
    pos = gd["position"]
    k = W.bf16_bits(np.array([gd["k_in"]], np.float32))
    v = W.bf16_bits(np.array([gd["v_in"]], np.float32))
    pool = rope_pool(geom, table, np.zeros(1, np.int32), np.array([pos], np.int32), k, v,
                     np.array(gd["cos_table"], np.float32), np.array(gd["sin_table"], np.float32))
    got_k = W.bf16_to_f32(pool[pos * d * 2:(pos + 1) * d * 2].view(np.uint16))
    vb = 16 * d * 2 + pos * d * 2
    got_v = W.bf16_to_f32(pool[vb:vb + d * 2].view(np.uint16))
    np.testing.assert_array_equal(got_k, np.array(gd["k_out"], np.float32))
    np.testing.assert_array_equal(got_v, np.array(gd["v_out"], np.float32))


def test_special_angles():
    geom, table, slot, pos, k, v = scatter_case()
    n, half = k.shape[0], geom.head_dim // 2
    g = oracle.geom(*geom.as_tuple())
    plain = np.zeros(geom.pool_bytes, np.uint8)
    assert oracle.write_kv(g, plain, table, 0, slot, pos, k, v) == 0
    one, zero = np.ones((n, half), np.float32), np.zeros((n, half), np.float32)
    np.testing.assert_array_equal(rope_pool(geom, table, slot, pos, k, v, one, zero), plain)
    kn, vn = gathered(geom, table, rope_pool(geom, table, slot, pos, k, v, -one, zero), n)
    np.testing.assert_array_equal(kn, k ^ np.uint16(0x8000))  # half turn: every element negated
    np.testing.assert_array_equal(vn, v)
    kq, _ = gathered(geom, table, rope_pool(geom, table, slot, pos, k, v, zero, one), n)
    kk = k.reshape(n, -1, geom.head_dim)
    want = np.concatenate([kk[..., half:] ^ np.uint16(0x8000), kk[..., :half]], axis=-1).reshape(n, -1)
    np.testing.assert_array_equal(kq, want)  # quarter turn: (x1, x2) -> (-x2, x1)


def test_matches_torch_fp32_ops_byte_for_byte():
    geom, table, slot, pos, k, v = scatter_case(hkv=4, d=128, n=48, seed=3)
    cos_t, sin_t = W.rope_tables(64, geom.head_dim)
    pool = rope_pool(geom, table, slot, pos, k, v, cos_t, sin_t)
    got, _ = gathered(geom, table, pool, k.shape[0])
    half = geom.head_dim // 2
    x = torch.from_numpy(W.bf16_to_f32(k)).reshape(k.shape[0], -1, geom.head_dim)
    c = torch.from_numpy(cos_t[pos])[:, None, :]
    s = torch.from_numpy(sin_t[pos])[:, None, :]
    x1, x2 = x[..., :half], x[..., half:]
    y1 = torch.sub(torch.mul(x1, c), torch.mul(x2, s))
    y2 = torch.add(torch.mul(x1, s), torch.mul(x2, c))
    y = torch.cat([y1, y2], dim=-1).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(got, y.reshape(k.shape[0], -1))


def test_rotation_invariants():
    d, n = 64, 40
    geom, table, slot, pos, k, v = scatter_case(hkv=1, d=d, n=n, seed=5)
    cos_t, sin_t = W.rope_tables(64, d, base=10000.0)
    got, _ = gathered(geom, table, rope_pool(geom, table, slot, pos, k, v, cos_t, sin_t), n)
    x = W.bf16_to_f32(k).astype(np.float64)
    y = W.bf16_to_f32(got).astype(np.float64)
    half = d // 2
    # the norm of every (i, i + d/2) pair is kept (within bf16 rounding of the outputs)
    nx = np.hypot(x[:, :half], x[:, half:])
    ny = np.hypot(y[:, :half], y[:, half:])
    assert np.max(np.abs(nx - ny) / np.maximum(nx, 1e-3)) < 2 ** -7
    # rotate one fixed vector to every position with the same call: <r(a, m), r(a, n)> depends on m - n only
    a = np.tile(k[:1], (n, 1))
    ra, _ = gathered(geom, table, rope_pool(geom, table, slot, pos, a, v, cos_t, sin_t), n)
    ra = W.bf16_to_f32(ra).astype(np.float64)
    ref = float(np.dot(x[0], x[0]))
    for delta in (1, 5, 17):
        dots = np.array([np.dot(ra[m], ra[m + delta]) for m in range(n - delta)])
        assert np.max(np.abs(dots - dots[0])) < 0.02 * ref

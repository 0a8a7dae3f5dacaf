"""Pins of the oracle's query rotation (orc_rope_q) and of the RoPE-Q prefill
built on it (rope_q, then the causal prefill over the cached prefix).

tiny-vllm part 3, "RoPE: a rotation that references a table": the program
rotates Q and K with the same kernel and tables before the scores; in each
head, element i and element i + head_dim/2 form a pair turned by the angle of
the token's position.  A query row's position is that of its own token: the
i-th query of a chunk after `pre` cached tokens sits at pre + i (the position
its K row was written at).  Pinned against:
  * the identity table: the rows come back bit for bit, and the RoPE-Q
    prefill is the plain prefill bit for bit;
  * exact special angles chosen per position (no turn, quarter, half and
    three-quarter turns cycling with the position), so every element of the
    answer is a plain copy or negation of an input element -- this fixes the
    pairing, the signs, the heads and the position of every row, prefix
    included;
  * a library routine on real tables: torch turns the pairs as complex
    numbers in fp64 (x1 + i x2) e^(i theta), and its scaled_dot_product_attention
    on the turned queries and keys agrees with the RoPE-Q prefill over keys
    scattered by orc_write_kv_rope, within the bf16 rounding of the turned rows;
  * a position past the table is refused.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from paged_kv_cache_gb300 import workloads as W  # noqa: E402


def _geom(hq=8, hkv=2, d=64, slots=3, pages=8):
    return W.Geometry(hq, hkv, d, 1, slots, pages, slots * pages + 4)


def _cycle_tables(max_pos, half):
    """Row p turns every pair by (p % 4) quarter turns, with exact cos / sin."""
    c = np.array([1.0, 0.0, -1.0, 0.0], np.float32)
    s = np.array([0.0, 1.0, 0.0, -1.0], np.float32)
    p = np.arange(max_pos) % 4
    return np.repeat(c[p][:, None], half, axis=1), np.repeat(s[p][:, None], half, axis=1)


def _turned_by_hand(qf, quarter_turns):
    """(x1, x2) -> (x1, x2), (-x2, x1), (-x1, -x2), (x2, -x1) for 0..3 quarter turns (float32 values)."""
    half = qf.shape[-1] // 2
    x1, x2 = qf[..., :half], qf[..., half:]
    turns = [(x1, x2), (-x2, x1), (-x1, -x2), (x2, -x1)]
    return np.concatenate(turns[quarter_turns], axis=-1)


def test_identity_table_changes_nothing():
    geom = _geom()
    case = W.make_chunked_case("rq_id", geom, [0, 16, 23], [40, 17, 1], seed=3)
    g = oracle.geom(*geom.as_tuple())
    half = geom.head_dim // 2
    one, zero = np.ones((64, half), np.float32), np.zeros((64, half), np.float32)
    st, qr = oracle.rope_q(g, case.q, case.cu_seqlens, case.extra["prefix"], one, zero)
    assert st == 0
    np.testing.assert_array_equal(qr, case.q)
    pool = np.zeros(geom.pool_bytes, np.uint8)
    for w in case.writes:
        assert oracle.write_kv(g, pool, case.block_table, w.layer, w.tok_slot, w.tok_pos, w.k, w.v) == 0
    st, o, lse = oracle.prefill_rope(g, case.q, pool, case.block_table, 0, case.cu_seqlens, case.extra["prefix"],
                                     case.slots, case.scale, one, zero)
    st2, o2, lse2 = oracle.prefill_cached(g, case.q, pool, case.block_table, 0, case.cu_seqlens,
                                          case.extra["prefix"], case.slots, case.scale)
    assert st == 0 and st2 == 0
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(lse, lse2)


@pytest.mark.parametrize("hq,hkv,d", [(8, 2, 64), (4, 4, 128)])
def test_quarter_turns_by_position(hq, hkv, d):
    geom = _geom(hq, hkv, d)
    prefix = [0, 16, 23]
    case = W.make_chunked_case("rq_turns", geom, prefix, [40, 17, 5], seed=7)
    g = oracle.geom(*geom.as_tuple())
    cos_t, sin_t = _cycle_tables(64, d // 2)
    st, qr = oracle.rope_q(g, case.q, case.cu_seqlens, case.extra["prefix"], cos_t, sin_t)
    assert st == 0
    got = W.bf16_to_f32(qr)
    qf = W.bf16_to_f32(case.q)
    cu = case.cu_seqlens
    for b in range(case.batch):
        for i in range(cu[b + 1] - cu[b]):
            t = cu[b] + i
            np.testing.assert_array_equal(got[t], _turned_by_hand(qf[t], (prefix[b] + i) % 4),
                                          err_msg="sequence %d query %d" % (b, i))


def test_prefill_rope_matches_library_sdpa_on_complex_turns():
    hq, hkv, d = 8, 2, 64
    geom = _geom(hq, hkv, d)
    prefix, chunk = [0, 21, 9], [37, 12, 30]
    case = W.make_chunked_case("rq_sdpa", geom, prefix, chunk, seed=11)
    g = oracle.geom(*geom.as_tuple())
    cos_t, sin_t = W.rope_tables(80, d)
    pool = np.zeros(geom.pool_bytes, np.uint8)
    for w in case.writes:
        assert oracle.write_kv_rope(g, pool, case.block_table, w.layer, w.tok_slot, w.tok_pos, w.k, w.v,
                                    cos_t, sin_t) == 0
    st, o, lse = oracle.prefill_rope(g, case.q, pool, case.block_table, 0, case.cu_seqlens, case.extra["prefix"],
                                     case.slots, case.scale, cos_t, sin_t)
    assert st == 0
    half = d // 2
    theta = torch.from_numpy(np.arctan2(sin_t.astype(np.float64), cos_t.astype(np.float64)))
    mag = torch.from_numpy(np.hypot(sin_t.astype(np.float64), cos_t.astype(np.float64)))

    def turn(x, pos):  # x [n][heads][d] fp64, positions [n]
        z = torch.complex(x[..., :half], x[..., half:])
        r = torch.polar(mag[pos], theta[pos])[:, None, :]
        y = z * r
        return torch.cat([y.real, y.imag], dim=-1)

    # every sequence's keys (its prefix, then its chunk) in position order
    kv = {}
    for w in case.writes:
        for t in range(w.tok_slot.shape[0]):
            kv.setdefault(int(w.tok_slot[t]), {})[int(w.tok_pos[t])] = (w.k[t], w.v[t])
    cu = case.cu_seqlens
    vmax = 0.0
    for b in range(case.batch):
        n_keys = prefix[b] + chunk[b]
        rows = [kv[b][p] for p in range(n_keys)]
        kk = torch.from_numpy(W.bf16_to_f32(np.stack([r[0] for r in rows])).astype(np.float64)).reshape(n_keys, hkv, d)
        vv = torch.from_numpy(W.bf16_to_f32(np.stack([r[1] for r in rows])).astype(np.float64)).reshape(n_keys, hkv, d)
        vmax = max(vmax, float(vv.abs().max()))
        qq = torch.from_numpy(W.bf16_to_f32(case.q[cu[b]:cu[b + 1]]).astype(np.float64))
        qpos = torch.arange(prefix[b], prefix[b] + chunk[b])
        kpos = torch.arange(n_keys)
        qt, kt = turn(qq, qpos), turn(kk, kpos)
        rep = hq // hkv
        kt, vr = kt.repeat_interleave(rep, dim=1), vv.repeat_interleave(rep, dim=1)
        mask = kpos[None, :] <= qpos[:, None]
        ref = torch.nn.functional.scaled_dot_product_attention(
            qt.transpose(0, 1), kt.transpose(0, 1), vr.transpose(0, 1), attn_mask=mask, scale=case.scale)
        ref = ref.transpose(0, 1).numpy()
        # the oracle turns bf16 rows and rounds them to bf16 (both Q and K): scores move by a
        # few 2^-9 of their terms, so O by a fraction of a percent of max|V|
        assert np.max(np.abs(o[cu[b]:cu[b + 1]] - ref)) < 1e-2 * vmax, "sequence %d" % b
        s = torch.einsum("qhd,khd->hqk", qt, kt) * case.scale
        s = s.masked_fill(~mask[None], float("-inf"))
        ref_l = torch.logsumexp(s, dim=-1).transpose(0, 1).numpy()
        assert np.max(np.abs(lse[cu[b]:cu[b + 1]] - ref_l)) < 2e-2, "sequence %d" % b


def test_position_past_the_table_is_refused():
    geom = _geom()
    case = W.make_chunked_case("rq_oob", geom, [10], [20], seed=5)
    g = oracle.geom(*geom.as_tuple())
    half = geom.head_dim // 2
    st, _ = oracle.rope_q(g, case.q, case.cu_seqlens, case.extra["prefix"], np.ones((29, half), np.float32),
                          np.zeros((29, half), np.float32))
    assert st != 0  # the last query sits at position 29
    st, _ = oracle.rope_q(g, case.q, case.cu_seqlens, case.extra["prefix"], np.ones((30, half), np.float32),
                          np.zeros((30, half), np.float32))
    assert st == 0

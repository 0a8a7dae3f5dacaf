"""Shared test plumbing: run a workload through the CUDA path (C ABI) and
through the CPU oracle, each from the same seeded inputs."""
import numpy as np

import oracle
import paged_kv_cache_gb300 as pa
from paged_kv_cache_gb300 import workloads as W


def f32(bits):
    return W.bf16_to_f32(bits).astype(np.float64)


# ------------------------------------------------------------------ oracle

def oracle_geom(case):
    return oracle.geom(*case.geom.as_tuple())


def oracle_pool(case, writes=None):
    g = oracle_geom(case)
    pool = W.initial_pool(case.geom, case.pool_fill, case.seed)
    for w in (case.writes if writes is None else writes):
        skipped = oracle.write_kv(g, pool, case.block_table, w.layer, w.tok_slot, w.tok_pos, w.k, w.v)
        assert skipped == 0
    return pool


def oracle_prefill(case, pool):
    st, o, lse = oracle.prefill(oracle_geom(case), case.q, pool, case.block_table, case.layer,
                                case.cu_seqlens, case.slots, case.scale)
    assert st == 0
    return o, lse


def oracle_prefill_cached(case, pool, rows=None, heads=None):
    g = oracle_geom(case)
    if rows is None:
        st, o, lse = oracle.prefill_cached(g, case.q, pool, case.block_table, case.layer, case.cu_seqlens,
                                           case.extra["prefix"], case.slots, case.scale)
    else:
        st, o, lse = oracle.prefill_cached_rows(g, case.q, pool, case.block_table, case.layer, case.cu_seqlens,
                                                case.extra["prefix"], case.slots, case.scale, rows, heads)
    assert st == 0
    return o, lse


def oracle_decode(case, pool):
    st, o, lse = oracle.decode(oracle_geom(case), case.q, pool, case.block_table, case.layer,
                               case.lens, case.slots, case.scale)
    assert st == 0
    return o, lse


def max_abs_v(case):
    """max |V| over the V rows the attention call reads (its layer's writes)."""
    vals = [np.abs(f32(w.v)).max() for w in case.writes if w.layer == case.layer and w.v.size]
    return float(max(vals)) if vals else 0.0


# -------------------------------------------------------------------- GPU

def torch_mod():
    import torch
    if not torch.cuda.is_available():
        raise RuntimeError("CUDA device required for the GPU parity tests")
    return torch


def pa_geom(case):
    return pa.geom(*case.geom.as_tuple())


def to_dev(a, dtype=None):
    torch = torch_mod()
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.cuda()


def device_pool(case):
    torch = torch_mod()
    init = W.initial_pool(case.geom, case.pool_fill, case.seed)
    return torch.from_numpy(init).cuda()


def gpu_write(case, pool, bt, writes=None, err=None):
    torch = torch_mod()
    g = pa_geom(case)
    own_err = err is None
    if own_err:
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
    for w in (case.writes if writes is None else writes):
        pa.pa_write_kv(g, pool, bt, w.layer, to_dev(w.tok_slot), to_dev(w.tok_pos),
                       to_dev(w.k), to_dev(w.v), err)
    torch.cuda.synchronize()
    if own_err:
        return int(err.item())
    return None


def gpu_setup(case):
    """Device pool after all writes, device table; returns (pool, bt, write_err)."""
    pool = device_pool(case)
    bt = to_dev(case.block_table)
    werr = gpu_write(case, pool, bt)
    return pool, bt, werr


def gpu_prefill(case, pool, bt, q=None, o=None, with_lse=True):
    torch = torch_mod()
    g = pa_geom(case)
    q = to_dev(case.q) if q is None else q
    T = case.total_tokens
    o = torch.empty((T, case.geom.num_q_heads, case.geom.head_dim), dtype=torch.int16,
                    device="cuda") if o is None else o
    lse = torch.empty((T, case.geom.num_q_heads), dtype=torch.float32, device="cuda") if with_lse else None
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_prefill(g, q, pool, bt, case.layer, to_dev(case.cu_seqlens), to_dev(case.slots),
                  case.max_len, case.scale, o, lse, err)
    torch.cuda.synchronize()
    o_np = f32(o.cpu().numpy().view(np.uint16))
    l_np = lse.cpu().numpy().astype(np.float64) if with_lse else None
    return o_np, l_np, int(err.item())


def gpu_prefill_cached(case, pool, bt, prefix=None, with_lse=True):
    """pa_prefill_cached of a chunked case; prefix=None passes the case's
    prefix lengths, prefix="null" passes a null pointer."""
    torch = torch_mod()
    g = pa_geom(case)
    q = to_dev(case.q)
    T = case.total_tokens
    o = torch.empty((T, case.geom.num_q_heads, case.geom.head_dim), dtype=torch.int16, device="cuda")
    lse = torch.empty((T, case.geom.num_q_heads), dtype=torch.float32, device="cuda") if with_lse else None
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pre = None if (isinstance(prefix, str) and prefix == "null") else to_dev(
        case.extra["prefix"] if prefix is None else np.asarray(prefix, np.int32))
    pa.pa_prefill_cached(g, q, pool, bt, case.layer, to_dev(case.cu_seqlens), pre, to_dev(case.slots),
                         case.max_len, case.scale, o, lse, err)
    torch.cuda.synchronize()
    o_np = f32(o.cpu().numpy().view(np.uint16))
    l_np = lse.cpu().numpy().astype(np.float64) if with_lse else None
    return o_np, l_np, int(err.item())


def gpu_decode(case, pool, bt, q=None, o=None, max_seq_len=None, with_lse=True, workspace=None):
    torch = torch_mod()
    g = pa_geom(case)
    B = case.batch
    q = to_dev(case.q) if q is None else q
    o = torch.empty((B, case.geom.num_q_heads, case.geom.head_dim), dtype=torch.int16,
                    device="cuda") if o is None else o
    lse = torch.empty((B, case.geom.num_q_heads), dtype=torch.float32, device="cuda") if with_lse else None
    msl = case.max_len if max_seq_len is None else max_seq_len
    if workspace is None:
        nbytes = pa.pa_decode_workspace_size(g, B, msl)
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_decode(g, q, pool, bt, case.layer, to_dev(case.lens), to_dev(case.slots), msl, case.scale,
                 o, lse, workspace, err)
    torch.cuda.synchronize()
    o_np = f32(o.cpu().numpy().view(np.uint16))
    l_np = lse.cpu().numpy().astype(np.float64) if with_lse else None
    return o_np, l_np, int(err.item())


# ------------------------------------------------------------- comparison

def assert_close(o_gpu, l_gpu, o_ref, l_ref, vmax, what=""):
    """The parity bar: |O - O_ref| <= 1e-2 max|V|, |L - L_ref| <= 1e-3."""
    tol_o = 1e-2 * vmax
    assert np.all(np.isfinite(o_gpu)), what + ": non-finite output"
    err_o = float(np.max(np.abs(o_gpu - o_ref))) if o_gpu.size else 0.0
    assert err_o <= tol_o, "%s: max |dO| %.3g > %.3g" % (what, err_o, tol_o)
    if l_gpu is not None:
        same_inf = np.isinf(l_ref) & (l_gpu == l_ref)
        with np.errstate(invalid="ignore"):
            d = np.where(same_inf, 0.0, np.abs(l_gpu - l_ref))
        err_l = float(np.max(d)) if d.size else 0.0
        assert err_l <= 1e-3, "%s: max |dL| %.3g > 1e-3" % (what, err_l)
    return err_o

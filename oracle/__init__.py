"""ctypes wrapper around the C oracle (oracle/oracle.c).

TEST INFRASTRUCTURE ONLY: imported by tests/, ``__graft_entry__.smoke()`` and
the CPU-baseline leg of ``bench.py``.  The product package never imports it.

Arrays are numpy: bf16 data is carried as uint16 bit patterns, the pool as
uint8 bytes, outputs as float64.
"""
import ctypes as C
import os

import numpy as np

from . import build as _build

_lib = None
_lib_path = None  # override used by the mutation tests (a planted-mistake build)


class Geom(C.Structure):
    _fields_ = [
        ("num_q_heads", C.c_int32),
        ("num_kv_heads", C.c_int32),
        ("head_dim", C.c_int32),
        ("n_layers", C.c_int32),
        ("num_slots", C.c_int32),
        ("max_blocks_per_seq", C.c_int32),
        ("num_blocks", C.c_int64),
    ]


OK = 0
BAD_ARG = -1
BAD_BLOCK = -2

_P = C.c_void_p


def lib():
    global _lib
    if _lib is None:
        path = _lib_path or _build.build()
        L = C.CDLL(path)
        L.orc_write_kv.restype = C.c_int64
        L.orc_write_kv.argtypes = [C.POINTER(Geom), _P, _P, C.c_int32, C.c_int64, _P, _P, _P, _P]
        L.orc_write_kv_rope.restype = C.c_int64
        L.orc_write_kv_rope.argtypes = [C.POINTER(Geom), _P, _P, C.c_int32, C.c_int64, _P, _P, _P, _P, _P, _P,
                                        C.c_int32]
        L.orc_rope_q.restype = C.c_int
        L.orc_rope_q.argtypes = [C.POINTER(Geom), _P, C.c_int32, _P, _P, _P, _P, C.c_int32, _P]
        L.orc_alloc_pages.restype = C.c_int64
        L.orc_alloc_pages.argtypes = [C.POINTER(Geom), _P, C.c_int32, _P, _P, _P, _P, _P]
        L.orc_release_slots.restype = C.c_int64
        L.orc_release_slots.argtypes = [C.POINTER(Geom), _P, C.c_int32, _P, _P, _P]
        L.orc_gather_kv.restype = C.c_int
        L.orc_gather_kv.argtypes = [C.POINTER(Geom), _P, _P, C.c_int32, C.c_int32, C.c_int32, _P, _P]
        L.orc_softmax_row.restype = None
        L.orc_softmax_row.argtypes = [_P, C.c_int32, _P, _P, _P]
        L.orc_partial.restype = None
        L.orc_partial.argtypes = [_P, _P, C.c_int32, C.c_int32, _P, _P, _P]
        L.orc_merge.restype = None
        L.orc_merge.argtypes = [C.c_int32, _P, _P, _P, C.c_int32, _P, _P, _P, _P, _P]
        L.orc_prefill.restype = C.c_int
        L.orc_prefill.argtypes = [C.POINTER(Geom), _P, _P, _P, C.c_int32, C.c_int32, _P, _P,
                                  C.c_float, _P, _P, C.c_int32]
        L.orc_prefill_rows.restype = C.c_int
        L.orc_prefill_rows.argtypes = [C.POINTER(Geom), _P, _P, _P, C.c_int32, C.c_int32, _P, _P,
                                       C.c_float, C.c_int64, _P, _P, _P, _P, C.c_int32]
        L.orc_prefill_cached.restype = C.c_int
        L.orc_prefill_cached.argtypes = [C.POINTER(Geom), _P, _P, _P, C.c_int32, C.c_int32, _P, _P, _P,
                                         C.c_float, _P, _P, C.c_int32]
        L.orc_prefill_cached_rows.restype = C.c_int
        L.orc_prefill_cached_rows.argtypes = [C.POINTER(Geom), _P, _P, _P, C.c_int32, C.c_int32, _P, _P, _P,
                                              C.c_float, C.c_int64, _P, _P, _P, _P, C.c_int32]
        L.orc_prefill_backward.restype = C.c_int
        L.orc_prefill_backward.argtypes = [C.POINTER(Geom), _P, _P, _P, C.c_int32, C.c_int32, _P, _P, C.c_float, _P,
                                           _P, _P, _P, C.c_int32]
        L.orc_prefill_backward_rows.restype = C.c_int
        L.orc_prefill_backward_rows.argtypes = [C.POINTER(Geom), _P, _P, _P, C.c_int32, C.c_int32, _P, _P,
                                                C.c_float, _P, C.c_int64, _P, _P, _P, C.c_int64, _P, _P, _P, _P,
                                                C.c_int32]
        L.orc_decode.restype = C.c_int
        L.orc_decode.argtypes = [C.POINTER(Geom), _P, _P, _P, C.c_int32, C.c_int32, _P, _P,
                                 C.c_float, _P, _P, C.c_int32]
        L.orc_default_threads.restype = C.c_int32
        L.orc_default_threads.argtypes = []
        _lib = L
    return _lib


class use_library:
    """Context manager: run the wrapper against another build of oracle.c."""

    def __init__(self, path):
        self.path = path

    def __enter__(self):
        global _lib, _lib_path
        self.saved = (_lib, _lib_path)
        _lib, _lib_path = None, self.path
        return self

    def __exit__(self, *exc):
        global _lib, _lib_path
        _lib, _lib_path = self.saved
        return False


def _ptr(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def geom(num_q_heads, num_kv_heads, head_dim, n_layers, num_slots, max_blocks_per_seq, num_blocks):
    return Geom(num_q_heads, num_kv_heads, head_dim, n_layers, num_slots, max_blocks_per_seq,
                num_blocks)


def default_threads():
    return int(lib().orc_default_threads())


def write_kv(g, pool, block_table, layer, tok_slot, tok_pos, k_new, v_new):
    """Scatter rows into ``pool`` (uint8, modified in place); returns skipped-row count."""
    assert pool.dtype == np.uint8 and pool.flags.c_contiguous
    bt = _c(block_table, np.int32)
    ts, tp = _c(tok_slot, np.int32), _c(tok_pos, np.int32)
    k, v = _c(k_new, np.uint16), _c(v_new, np.uint16)
    n = ts.shape[0]
    r = lib().orc_write_kv(C.byref(g), _ptr(pool), _ptr(bt), layer, n, _ptr(ts), _ptr(tp),
                           _ptr(k), _ptr(v))
    return int(r)


def write_kv_rope(g, pool, block_table, layer, tok_slot, tok_pos, k_new, v_new, cos_tab, sin_tab):
    """Scatter with K rotated by RoPE (tables [max_pos][d/2] fp32); returns skipped-row count."""
    assert pool.dtype == np.uint8 and pool.flags.c_contiguous
    bt = _c(block_table, np.int32)
    ts, tp = _c(tok_slot, np.int32), _c(tok_pos, np.int32)
    k, v = _c(k_new, np.uint16), _c(v_new, np.uint16)
    ct, st = _c(cos_tab, np.float32), _c(sin_tab, np.float32)
    n = ts.shape[0]
    r = lib().orc_write_kv_rope(C.byref(g), _ptr(pool), _ptr(bt), layer, n, _ptr(ts), _ptr(tp),
                                _ptr(k), _ptr(v), _ptr(ct), _ptr(st), int(ct.shape[0]))
    return int(r)


def rope_q(g, q, cu_seqlens, prefix_lens, cos_tab, sin_tab):
    """Query rows rotated by RoPE at position prefix_lens[b] + i (prefix_lens
    None: 0): (status, q_rot[T][Hq][d] bf16 bits)."""
    cu = _c(cu_seqlens, np.int32)
    pre = None if prefix_lens is None else _c(prefix_lens, np.int32)
    q = _c(q, np.uint16)
    ct, stab = _c(cos_tab, np.float32), _c(sin_tab, np.float32)
    out = np.zeros_like(q)
    st = lib().orc_rope_q(C.byref(g), _ptr(q), cu.shape[0] - 1, _ptr(cu), _ptr(pre), _ptr(ct), _ptr(stab),
                          ct.shape[0], _ptr(out))
    return int(st), out


def prefill_rope(g, q, pool, block_table, layer, cu_seqlens, prefix_lens, slots, scale, cos_tab, sin_tab,
                 rows=None, heads=None, nthreads=0):
    """Prefill with RoPE on the queries: the rows rotated at their positions
    (rope_q), then the causal prefill over the cached prefix (prefill_cached;
    prefix_lens None: none) on the rotated rows, at every output or at the
    sampled (row, head) pairs.  (status, O, L)."""
    st, qr = rope_q(g, q, cu_seqlens, prefix_lens, cos_tab, sin_tab)
    if st != OK:
        return st, None, None
    pre = np.zeros(len(cu_seqlens) - 1, np.int32) if prefix_lens is None else prefix_lens
    if rows is None:
        return prefill_cached(g, qr, pool, block_table, layer, cu_seqlens, pre, slots, scale, nthreads)
    return prefill_cached_rows(g, qr, pool, block_table, layer, cu_seqlens, pre, slots, scale, rows, heads,
                               nthreads)


def alloc_pages(g, block_table, slots, seq_lens, free_pages, free_count, old_lens=None):
    """Pops pages for every -1 entry the lengths need (in place on the int32
    arrays block_table, free_pages and the one-element free_count); returns
    the number of pages taken or a negative status."""
    for a in (block_table, free_pages, free_count):
        assert a.dtype == np.int32 and a.flags.c_contiguous
    sl, ln = _c(slots, np.int32), _c(seq_lens, np.int32)
    old = None if old_lens is None else _c(old_lens, np.int32)
    return int(lib().orc_alloc_pages(C.byref(g), _ptr(block_table), int(sl.shape[0]), _ptr(sl),
                                     None if old is None else _ptr(old), _ptr(ln), _ptr(free_pages),
                                     _ptr(free_count)))


def release_slots(g, block_table, slots, free_pages, free_count):
    """Pushes every page of the slots back (in place); returns the count or a negative status."""
    for a in (block_table, free_pages, free_count):
        assert a.dtype == np.int32 and a.flags.c_contiguous
    sl = _c(slots, np.int32)
    return int(lib().orc_release_slots(C.byref(g), _ptr(block_table), int(sl.shape[0]), _ptr(sl),
                                       _ptr(free_pages), _ptr(free_count)))


def gather_kv(g, pool, block_table, layer, slot, n):
    K = np.zeros((n, g.num_kv_heads, g.head_dim), np.float64)
    V = np.zeros_like(K)
    bt = _c(block_table, np.int32)
    st = lib().orc_gather_kv(C.byref(g), _ptr(pool), _ptr(bt), layer, slot, n, _ptr(K), _ptr(V))
    return st, K, V


def softmax_row(s):
    s = _c(s, np.float64)
    w = np.zeros_like(s)
    m, l = C.c_double(), C.c_double()
    lib().orc_softmax_row(_ptr(s), s.shape[0], _ptr(w), C.byref(m), C.byref(l))
    return w, m.value, l.value


def partial(s, v):
    s = _c(s, np.float64)
    v = _c(v, np.float64).reshape(s.shape[0], -1)
    acc = np.zeros(v.shape[1], np.float64)
    m, l = C.c_double(), C.c_double()
    lib().orc_partial(_ptr(s), _ptr(v), s.shape[0], v.shape[1], C.byref(m), C.byref(l), _ptr(acc))
    return m.value, l.value, acc


def merge(ms, ls, accs):
    ms, ls = _c(ms, np.float64), _c(ls, np.float64)
    accs = _c(accs, np.float64).reshape(ms.shape[0], -1)
    dv = accs.shape[1]
    acc_out = np.zeros(dv, np.float64)
    o = np.zeros(dv, np.float64)
    m, l, L = C.c_double(), C.c_double(), C.c_double()
    lib().orc_merge(ms.shape[0], _ptr(ms), _ptr(ls), _ptr(accs), dv, C.byref(m), C.byref(l),
                    _ptr(acc_out), _ptr(o), C.byref(L))
    return m.value, l.value, acc_out, o, L.value


def prefill(g, q, pool, block_table, layer, cu_seqlens, slots, scale, nthreads=0):
    """Returns (status, O[T][Hq][d] float64, L[T][Hq] float64)."""
    cu = _c(cu_seqlens, np.int32)
    sl = _c(slots, np.int32)
    T = int(cu[-1])
    q = _c(q, np.uint16)
    o = np.zeros((T, g.num_q_heads, g.head_dim), np.float64)
    lse = np.zeros((T, g.num_q_heads), np.float64)
    st = lib().orc_prefill(C.byref(g), _ptr(q), _ptr(pool), _ptr(_c(block_table, np.int32)), layer,
                           cu.shape[0] - 1, _ptr(cu), _ptr(sl), C.c_float(scale), _ptr(o), _ptr(lse),
                           nthreads)
    return int(st), o, lse


def prefill_rows(g, q, pool, block_table, layer, cu_seqlens, slots, scale, rows, heads,
                 nthreads=0):
    """Oracle at sampled (packed row, q head) pairs: (status, O[n][d], L[n])."""
    cu = _c(cu_seqlens, np.int32)
    sl = _c(slots, np.int32)
    rows = _c(rows, np.int64)
    heads = _c(heads, np.int32)
    q = _c(q, np.uint16)
    n = rows.shape[0]
    o = np.zeros((n, g.head_dim), np.float64)
    lse = np.zeros(n, np.float64)
    st = lib().orc_prefill_rows(C.byref(g), _ptr(q), _ptr(pool), _ptr(_c(block_table, np.int32)),
                                layer, cu.shape[0] - 1, _ptr(cu), _ptr(sl), C.c_float(scale), n,
                                _ptr(rows), _ptr(heads), _ptr(o), _ptr(lse), nthreads)
    return int(st), o, lse


def prefill_cached(g, q, pool, block_table, layer, cu_seqlens, prefix_lens, slots, scale, nthreads=0):
    """Chunked prefill over a cached prefix: (status, O[T][Hq][d], L[T][Hq])."""
    cu = _c(cu_seqlens, np.int32)
    pre = _c(prefix_lens, np.int32)
    sl = _c(slots, np.int32)
    T = int(cu[-1])
    q = _c(q, np.uint16)
    o = np.zeros((T, g.num_q_heads, g.head_dim), np.float64)
    lse = np.zeros((T, g.num_q_heads), np.float64)
    st = lib().orc_prefill_cached(C.byref(g), _ptr(q), _ptr(pool), _ptr(_c(block_table, np.int32)), layer,
                                  cu.shape[0] - 1, _ptr(cu), _ptr(pre), _ptr(sl), C.c_float(scale), _ptr(o),
                                  _ptr(lse), nthreads)
    return int(st), o, lse


def prefill_cached_rows(g, q, pool, block_table, layer, cu_seqlens, prefix_lens, slots, scale, rows, heads,
                        nthreads=0):
    """prefill_cached at sampled (packed row, q head) pairs: (status, O[n][d], L[n])."""
    cu = _c(cu_seqlens, np.int32)
    pre = _c(prefix_lens, np.int32)
    sl = _c(slots, np.int32)
    rows = _c(rows, np.int64)
    heads = _c(heads, np.int32)
    q = _c(q, np.uint16)
    n = rows.shape[0]
    o = np.zeros((n, g.head_dim), np.float64)
    lse = np.zeros(n, np.float64)
    st = lib().orc_prefill_cached_rows(C.byref(g), _ptr(q), _ptr(pool), _ptr(_c(block_table, np.int32)),
                                       layer, cu.shape[0] - 1, _ptr(cu), _ptr(pre), _ptr(sl), C.c_float(scale),
                                       n, _ptr(rows), _ptr(heads), _ptr(o), _ptr(lse), nthreads)
    return int(st), o, lse


def prefill_backward(g, q, pool, block_table, layer, cu_seqlens, slots, scale, dout, nthreads=0):
    """Gradients of the causal prefill: (status, dQ[T][Hq][d], dK[T][Hkv][d], dV[T][Hkv][d]) float64."""
    cu = _c(cu_seqlens, np.int32)
    sl = _c(slots, np.int32)
    T = int(cu[-1])
    q = _c(q, np.uint16)
    do = _c(dout, np.uint16)
    dq = np.zeros((T, g.num_q_heads, g.head_dim), np.float64)
    dk = np.zeros((T, g.num_kv_heads, g.head_dim), np.float64)
    dv = np.zeros_like(dk)
    st = lib().orc_prefill_backward(C.byref(g), _ptr(q), _ptr(pool), _ptr(_c(block_table, np.int32)), layer,
                                    cu.shape[0] - 1, _ptr(cu), _ptr(sl), C.c_float(scale), _ptr(do), _ptr(dq),
                                    _ptr(dk), _ptr(dv), nthreads)
    return int(st), dq, dk, dv


def prefill_backward_rows(g, q, pool, block_table, layer, cu_seqlens, slots, scale, dout, q_rows, q_heads,
                          k_rows, k_heads, nthreads=0):
    """prefill_backward at sampled outputs: (status, dq[len(q_rows)][d] of (q_rows, q_heads),
    dk, dv [len(k_rows)][d] of (k_rows, kv heads k_heads)), float64, equal to the full call's entries."""
    cu = _c(cu_seqlens, np.int32)
    qr = _c(q_rows, np.int64)
    qh = _c(q_heads, np.int32)
    kr = _c(k_rows, np.int64)
    kh = _c(k_heads, np.int32)
    d = g.head_dim
    dq = np.zeros((qr.shape[0], d), np.float64)
    dk = np.zeros((kr.shape[0], d), np.float64)
    dv = np.zeros_like(dk)
    st = lib().orc_prefill_backward_rows(C.byref(g), _ptr(_c(q, np.uint16)), _ptr(pool),
                                         _ptr(_c(block_table, np.int32)), layer, cu.shape[0] - 1, _ptr(cu),
                                         _ptr(_c(slots, np.int32)), C.c_float(scale), _ptr(_c(dout, np.uint16)),
                                         qr.shape[0], _ptr(qr), _ptr(qh), _ptr(dq), kr.shape[0], _ptr(kr), _ptr(kh),
                                         _ptr(dk), _ptr(dv), nthreads)
    return int(st), dq, dk, dv


def decode(g, q, pool, block_table, layer, seq_lens, slots, scale, nthreads=0):
    """Returns (status, O[B][Hq][d] float64, L[B][Hq] float64)."""
    lens = _c(seq_lens, np.int32)
    sl = _c(slots, np.int32)
    B = lens.shape[0]
    q = _c(q, np.uint16)
    o = np.zeros((B, g.num_q_heads, g.head_dim), np.float64)
    lse = np.zeros((B, g.num_q_heads), np.float64)
    st = lib().orc_decode(C.byref(g), _ptr(q), _ptr(pool), _ptr(_c(block_table, np.int32)), layer, B,
                          _ptr(lens), _ptr(sl), C.c_float(scale), _ptr(o), _ptr(lse), nthreads)
    return int(st), o, lse


LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_build", "liboracle.so")

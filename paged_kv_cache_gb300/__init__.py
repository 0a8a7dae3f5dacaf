"""Paged-KV-cache attention for GB300 (sm_103a): Python binding of libpa.so.

The compute lives entirely in the CUDA kernels behind the C ABI declared in
``include/pa.h``; this module only marshals arguments (tensor pointers,
sizes, the current CUDA stream) into those calls.  There is no CPU or
PyTorch fallback: if ``libpa.so`` is missing the import of the library
raises, and every call that fails returns an error that is raised here.

Calls (same names as the C ABI):

* ``pa_write_kv(geom, pool, block_table, layer, tok_slot, tok_pos, k_new, v_new, err_flag)``
* ``pa_write_kv_rope(geom, pool, block_table, layer, tok_slot, tok_pos, k_new, v_new, cos_table, sin_table, err_flag)``
* ``pa_prefill(geom, q, pool, block_table, layer, cu_seqlens, slots, max_seqlen, scale, o, lse, err_flag)``
* ``pa_prefill_cached(geom, q, pool, block_table, layer, cu_seqlens, prefix_lens, slots, max_seqlen, scale, o, lse, err_flag)``
* ``pa_prefill_rope(geom, q, pool, block_table, layer, cu_seqlens, prefix_lens, slots, max_seqlen, scale, cos_table, sin_table, o, lse, err_flag)``
* ``pa_prefill_backward(geom, q, pool, block_table, layer, cu_seqlens, slots, max_seqlen, scale, o, lse, dout, delta, dq, dk, dv, err_flag)``
* ``pa_decode(geom, q, pool, block_table, layer, seq_lens, slots, max_seq_len, scale, o, lse, workspace, err_flag)``
* ``pa_decode_noalloc(geom, q, pool, block_table, layer, seq_lens, slots, max_seq_len, scale, o, lse, err_flag)``
* ``pa_alloc_pages(geom, block_table, slots, seq_lens, free_pages, free_count, err_flag, old_lens=None)``
* ``pa_release_slots(geom, block_table, slots, free_pages, free_count, err_flag)``
* ``pa_decode_workspace_size(geom, batch, max_seq_len)``, ``pa_page_bytes(geom)``, ``pa_status_string(code)``
* ``pa_debug_hold_first_copy(enable)`` (diagnostic for the tests of the kernels' bounded waits)

Tensors are torch CUDA tensors (bf16 data may be given as bfloat16 or int16
views); ``err_flag`` is a one-element int32 CUDA tensor the caller zeroes.
"""
import ctypes as C
import os

PA_OK = 0
PA_ERR_INVALID_ARG = 1
PA_ERR_UNSUPPORTED = 2
PA_ERR_CUDA = 3
PA_ERR_BAD_BLOCK = 4
PA_ERR_TIMEOUT = 5
PA_ERR_OUT_OF_PAGES = 6
PA_BLOCK_TOKENS = 16

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libpa.so")
EXPORTED = ("pa_page_bytes", "pa_write_kv", "pa_write_kv_rope", "pa_prefill", "pa_prefill_cached", "pa_prefill_rope",
            "pa_prefill_backward", "pa_decode_workspace_size", "pa_decode",
            "pa_decode_noalloc", "pa_alloc_pages", "pa_release_slots", "pa_debug_hold_first_copy",
            "pa_status_string")
PA_DECODE_STATIC_SCRATCH_BYTES = 16 << 20
PA_PAGES_MAX_SLOTS = 65536


class PaGeom(C.Structure):
    """Mirror of ``pa_geom`` in include/pa.h."""
    _fields_ = [
        ("num_q_heads", C.c_int32),
        ("num_kv_heads", C.c_int32),
        ("head_dim", C.c_int32),
        ("n_layers", C.c_int32),
        ("num_slots", C.c_int32),
        ("max_blocks_per_seq", C.c_int32),
        ("num_blocks", C.c_int64),
    ]


class PaError(RuntimeError):
    def __init__(self, call, code):
        self.code = code
        super().__init__("%s failed: %s" % (call, pa_status_string(code)))


_lib = None
_P = C.c_void_p


def load_library(path: str = None):
    """Loads libpa.so (built by ``paged_kv_cache_gb300.build``); raises if absent."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise ImportError("libpa.so not found at %s: build it with "
                          "`python -m paged_kv_cache_gb300.build` (needs nvcc)" % path)
    L = C.CDLL(path)
    L.pa_page_bytes.restype = C.c_size_t
    L.pa_page_bytes.argtypes = [C.POINTER(PaGeom)]
    L.pa_write_kv.restype = C.c_int
    L.pa_write_kv.argtypes = [C.POINTER(PaGeom), _P, _P, C.c_int32, C.c_int32, _P, _P, _P, _P, _P, _P]
    L.pa_write_kv_rope.restype = C.c_int
    L.pa_write_kv_rope.argtypes = [C.POINTER(PaGeom), _P, _P, C.c_int32, C.c_int32, _P, _P, _P, _P, _P, _P,
                                   C.c_int32, _P, _P]
    L.pa_prefill.restype = C.c_int
    L.pa_prefill.argtypes = [C.POINTER(PaGeom), _P, _P, _P, C.c_int32, C.c_int32, _P, _P, C.c_int32,
                             C.c_int32, C.c_float, _P, _P, _P, _P]
    L.pa_prefill_cached.restype = C.c_int
    L.pa_prefill_cached.argtypes = [C.POINTER(PaGeom), _P, _P, _P, C.c_int32, C.c_int32, _P, _P, _P, C.c_int32,
                                    C.c_int32, C.c_float, _P, _P, _P, _P]
    L.pa_prefill_rope.restype = C.c_int
    L.pa_prefill_rope.argtypes = [C.POINTER(PaGeom), _P, _P, _P, C.c_int32, C.c_int32, _P, _P, _P, C.c_int32,
                                  C.c_int32, C.c_float, _P, _P, C.c_int32, _P, _P, _P, _P]
    L.pa_decode_workspace_size.restype = C.c_size_t
    L.pa_prefill_backward.restype = C.c_int
    L.pa_prefill_backward.argtypes = [C.POINTER(PaGeom), _P, _P, _P, C.c_int32, C.c_int32, _P, _P, C.c_int32,
                                      C.c_int32, C.c_float, _P, _P, _P, _P, _P, _P, _P, _P, _P]
    L.pa_decode_workspace_size.argtypes = [C.POINTER(PaGeom), C.c_int32, C.c_int32]
    L.pa_decode.restype = C.c_int
    L.pa_decode.argtypes = [C.POINTER(PaGeom), _P, _P, _P, C.c_int32, C.c_int32, _P, _P, C.c_int32,
                            C.c_float, _P, _P, _P, C.c_size_t, _P, _P]
    L.pa_decode_noalloc.restype = C.c_int
    L.pa_decode_noalloc.argtypes = [C.POINTER(PaGeom), _P, _P, _P, C.c_int32, C.c_int32, _P, _P,
                                    C.c_int32, C.c_float, _P, _P, _P, _P]
    L.pa_alloc_pages.restype = C.c_int
    L.pa_alloc_pages.argtypes = [C.POINTER(PaGeom), _P, C.c_int32, _P, _P, _P, _P, _P, _P, _P]
    L.pa_release_slots.restype = C.c_int
    L.pa_release_slots.argtypes = [C.POINTER(PaGeom), _P, C.c_int32, _P, _P, _P, _P, _P]
    L.pa_debug_hold_first_copy.restype = C.c_int
    L.pa_debug_hold_first_copy.argtypes = [C.c_int32]
    L.pa_status_string.restype = C.c_char_p
    L.pa_status_string.argtypes = [C.c_int]
    if path == LIB_PATH:
        _lib = L
    return L


def lib():
    return load_library()


def geom(num_q_heads, num_kv_heads, head_dim, n_layers, num_slots, max_blocks_per_seq, num_blocks):
    return PaGeom(num_q_heads, num_kv_heads, head_dim, n_layers, num_slots, max_blocks_per_seq,
                  num_blocks)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(call, code):
    if code != PA_OK:
        raise PaError(call, code)


def pa_debug_hold_first_copy(enable: bool) -> None:
    """Diagnostic (tests only): while enabled, the first CTA of each later
    prefill or decode launch arms its first tensor copy without issuing it, so
    its bounded waits run out and the call reports PA_ERR_TIMEOUT."""
    _check("pa_debug_hold_first_copy", lib().pa_debug_hold_first_copy(1 if enable else 0))


def pa_status_string(code: int) -> str:
    return lib().pa_status_string(code).decode()


def pa_page_bytes(g: PaGeom) -> int:
    return int(lib().pa_page_bytes(C.byref(g)))


def pa_decode_workspace_size(g: PaGeom, batch: int, max_seq_len: int) -> int:
    return int(lib().pa_decode_workspace_size(C.byref(g), batch, max_seq_len))


def pa_write_kv(g, pool, block_table, layer, tok_slot, tok_pos, k_new, v_new, err_flag,
                stream=None, n_tokens=None):
    n = int(tok_slot.shape[0]) if n_tokens is None else int(n_tokens)
    _check("pa_write_kv", lib().pa_write_kv(
        C.byref(g), _ptr(pool), _ptr(block_table), layer, n, _ptr(tok_slot), _ptr(tok_pos),
        _ptr(k_new), _ptr(v_new), _ptr(err_flag), _stream(stream)))


def pa_write_kv_rope(g, pool, block_table, layer, tok_slot, tok_pos, k_new, v_new, cos_table, sin_table,
                     err_flag, stream=None, n_tokens=None):
    """pa_write_kv with RoPE on K; cos_table / sin_table: fp32 [max_pos][head_dim/2] CUDA tensors."""
    n = int(tok_slot.shape[0]) if n_tokens is None else int(n_tokens)
    _check("pa_write_kv_rope", lib().pa_write_kv_rope(
        C.byref(g), _ptr(pool), _ptr(block_table), layer, n, _ptr(tok_slot), _ptr(tok_pos),
        _ptr(k_new), _ptr(v_new), _ptr(cos_table), _ptr(sin_table), int(cos_table.shape[0]),
        _ptr(err_flag), _stream(stream)))


def pa_prefill(g, q, pool, block_table, layer, cu_seqlens, slots, max_seqlen, scale, o, lse,
               err_flag, stream=None, batch=None, total_tokens=None):
    batch = int(cu_seqlens.shape[0]) - 1 if batch is None else int(batch)
    total = int(q.shape[0]) if total_tokens is None else int(total_tokens)
    _check("pa_prefill", lib().pa_prefill(
        C.byref(g), _ptr(q), _ptr(pool), _ptr(block_table), layer, batch, _ptr(cu_seqlens),
        _ptr(slots), int(max_seqlen), total, float(scale), _ptr(o), _ptr(lse), _ptr(err_flag),
        _stream(stream)))


def pa_prefill_cached(g, q, pool, block_table, layer, cu_seqlens, prefix_lens, slots, max_seqlen, scale, o, lse,
                      err_flag, stream=None, batch=None, total_tokens=None):
    """Prefill of query chunks after prefix_lens[b] cached tokens (None: no prefix)."""
    batch = int(cu_seqlens.shape[0]) - 1 if batch is None else int(batch)
    total = int(q.shape[0]) if total_tokens is None else int(total_tokens)
    _check("pa_prefill_cached", lib().pa_prefill_cached(
        C.byref(g), _ptr(q), _ptr(pool), _ptr(block_table), layer, batch, _ptr(cu_seqlens),
        _ptr(prefix_lens), _ptr(slots), int(max_seqlen), total, float(scale), _ptr(o), _ptr(lse),
        _ptr(err_flag), _stream(stream)))


def pa_prefill_rope(g, q, pool, block_table, layer, cu_seqlens, prefix_lens, slots, max_seqlen, scale, cos_table,
                    sin_table, o, lse, err_flag, stream=None, batch=None, total_tokens=None):
    """pa_prefill_cached with RoPE on the queries (prefix_lens None: no prefix);
    cos_table / sin_table: fp32 [max_pos][head_dim/2] CUDA tensors."""
    batch = int(cu_seqlens.shape[0]) - 1 if batch is None else int(batch)
    total = int(q.shape[0]) if total_tokens is None else int(total_tokens)
    _check("pa_prefill_rope", lib().pa_prefill_rope(
        C.byref(g), _ptr(q), _ptr(pool), _ptr(block_table), layer, batch, _ptr(cu_seqlens), _ptr(prefix_lens),
        _ptr(slots), int(max_seqlen), total, float(scale), _ptr(cos_table), _ptr(sin_table), int(cos_table.shape[0]),
        _ptr(o), _ptr(lse), _ptr(err_flag), _stream(stream)))


def pa_prefill_backward(g, q, pool, block_table, layer, cu_seqlens, slots, max_seqlen, scale, o, lse, dout,
                        delta, dq, dk, dv, err_flag, stream=None, batch=None, total_tokens=None):
    """Gradients dq [T][Hq][d], dk / dv [T][Hkv][d] (fp32) of the causal prefill
    for the output gradient dout, from the forward's o and lse; delta is an fp32
    workspace of 2 * T * Hq floats."""
    batch = int(cu_seqlens.shape[0]) - 1 if batch is None else int(batch)
    total = int(q.shape[0]) if total_tokens is None else int(total_tokens)
    _check("pa_prefill_backward", lib().pa_prefill_backward(
        C.byref(g), _ptr(q), _ptr(pool), _ptr(block_table), layer, batch, _ptr(cu_seqlens), _ptr(slots),
        int(max_seqlen), total, float(scale), _ptr(o), _ptr(lse), _ptr(dout), _ptr(delta), _ptr(dq), _ptr(dk),
        _ptr(dv), _ptr(err_flag), _stream(stream)))


def pa_decode(g, q, pool, block_table, layer, seq_lens, slots, max_seq_len, scale, o, lse,
              workspace, err_flag, stream=None, batch=None, workspace_bytes=None):
    batch = int(seq_lens.shape[0]) if batch is None else int(batch)
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check("pa_decode", lib().pa_decode(
        C.byref(g), _ptr(q), _ptr(pool), _ptr(block_table), layer, batch, _ptr(seq_lens),
        _ptr(slots), int(max_seq_len), float(scale), _ptr(o), _ptr(lse), _ptr(workspace),
        int(workspace_bytes), _ptr(err_flag), _stream(stream)))


def pa_decode_noalloc(g, q, pool, block_table, layer, seq_lens, slots, max_seq_len, scale, o, lse,
                      err_flag, stream=None, batch=None):
    """pa_decode without a workspace argument, for callers that cannot
    allocate device memory where they decode (see include/pa.h): the split
    partials use a fixed scratch array inside the library's device code."""
    batch = int(seq_lens.shape[0]) if batch is None else int(batch)
    _check("pa_decode_noalloc", lib().pa_decode_noalloc(
        C.byref(g), _ptr(q), _ptr(pool), _ptr(block_table), layer, batch, _ptr(seq_lens),
        _ptr(slots), int(max_seq_len), float(scale), _ptr(o), _ptr(lse), _ptr(err_flag),
        _stream(stream)))


def pa_alloc_pages(g, block_table, slots, seq_lens, free_pages, free_count, err_flag, old_lens=None, stream=None):
    """Pages for every -1 entry the new lengths need, popped from the device free stack."""
    _check("pa_alloc_pages", lib().pa_alloc_pages(
        C.byref(g), _ptr(block_table), int(slots.shape[0]), _ptr(slots), _ptr(old_lens), _ptr(seq_lens),
        _ptr(free_pages), _ptr(free_count), _ptr(err_flag), _stream(stream)))


def pa_release_slots(g, block_table, slots, free_pages, free_count, err_flag, stream=None):
    """Every page of the slots back on the device free stack; their entries become -1."""
    _check("pa_release_slots", lib().pa_release_slots(
        C.byref(g), _ptr(block_table), int(slots.shape[0]), _ptr(slots), _ptr(free_pages), _ptr(free_count),
        _ptr(err_flag), _stream(stream)))

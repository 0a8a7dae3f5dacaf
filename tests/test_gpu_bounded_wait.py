"""The kernels' bounded waits: a wait that cannot complete runs out, the call
reports PA_ERR_TIMEOUT through err_flag, and the GPU stays usable.

pa_debug_hold_first_copy makes the first CTA of a prefill or decode launch
arm the barrier of its first tensor copy without issuing the copy: a phase
that nothing completes.  The roles waiting on it give up after the kernels'
limit (about 2 s), record PA_ERR_TIMEOUT, stop the other roles, let the
copies they did issue land and free the tensor memory.  The test checks the
status, that the other CTAs' outputs are still right, and that the next
normal call matches the oracle.  No kernel traps, faults or hangs here.
"""
import time

import numpy as np
import pytest

import paged_kv_cache_gb300 as pa
from paged_kv_cache_gb300 import workloads as W
from tests import helpers as H

pytestmark = pytest.mark.gpu

WAIT_LIMIT_S = 2.0


def _held(run):
    pa.pa_debug_hold_first_copy(True)
    try:
        t0 = time.perf_counter()
        out = run()
        return out, time.perf_counter() - t0
    finally:
        pa.pa_debug_hold_first_copy(False)


@pytest.mark.parametrize("rope", [False, True])
def test_prefill_wait_runs_out_and_the_next_call_is_right(rope):
    geom = W.Geometry(8, 2, 64, 1, 2, 48, 100)
    case = W.make_prefill_case("held", geom, [700, 300], seed=31, pool_fill="nan")
    pool, bt, werr = H.gpu_setup(case)
    assert werr == 0
    ro, rl = H.oracle_prefill(case, H.oracle_pool(case))
    vmax = H.max_abs_v(case)
    if rope:
        # identity tables: the RoPE-Q kernel then computes the plain prefill
        n = 800
        one, zero = H.to_dev(np.ones((n, 32), np.float32)), H.to_dev(np.zeros((n, 32), np.float32))
        torch = H.torch_mod()

        def run():
            o = torch.zeros((case.total_tokens, 8, 64), dtype=torch.int16, device="cuda")
            lse = torch.empty((case.total_tokens, 8), dtype=torch.float32, device="cuda")
            err = torch.zeros(1, dtype=torch.int32, device="cuda")
            pa.pa_prefill_rope(H.pa_geom(case), H.to_dev(case.q), pool, bt, 0, H.to_dev(case.cu_seqlens), None,
                               H.to_dev(case.slots), case.max_len, case.scale, one, zero, o, lse, err)
            torch.cuda.synchronize()
            return H.f32(o.cpu().numpy().view(np.uint16)), lse.cpu().numpy().astype(np.float64), int(err.item())
    else:
        def run():  # zeroed outputs: the held CTA's rows stay unwritten
            return H.gpu_prefill(case, pool, bt, o=H.torch_mod().zeros((case.total_tokens, 8, 64),
                                                                         dtype=H.torch_mod().int16, device="cuda"))
    (o, l, err), secs = _held(run)
    assert err == pa.PA_ERR_TIMEOUT, pa.pa_status_string(err)
    assert secs >= 0.9 * WAIT_LIMIT_S
    # CTA 0 is the heaviest item: the last 128-row tile of sequence 0, q heads 0..3 (one kv head's group)
    held = np.zeros((case.total_tokens, 8), bool)
    held[640:700, 0:4] = True
    ok = ~held
    H.assert_close(o[ok], l[ok], ro[ok], rl[ok], vmax, "rows of the other CTAs")
    # the next call, with the switch off, is right everywhere
    o2, l2, err2 = run()
    assert err2 == 0
    H.assert_close(o2, l2, ro, rl, vmax, "the call after the timeout")


def test_decode_wait_runs_out_and_the_next_call_is_right():
    geom = W.Geometry(32, 8, 64, 1, 16, 128, 2200)
    case = W.make_decode_case("held_dec", geom, W.uniform_decode_lens(5, 16), seed=32, pool_fill="nan")
    pool, bt, werr = H.gpu_setup(case)
    assert werr == 0
    (o, l, err), secs = _held(lambda: H.gpu_decode(case, pool, bt))
    assert err == pa.PA_ERR_TIMEOUT, pa.pa_status_string(err)
    assert secs >= 0.9 * WAIT_LIMIT_S
    o2, l2, err2 = H.gpu_decode(case, pool, bt)
    assert err2 == 0
    ro, rl = H.oracle_decode(case, H.oracle_pool(case))
    H.assert_close(o2, l2, ro, rl, H.max_abs_v(case), "decode after the timeout")


def test_key_split_wait_runs_out_and_the_next_call_is_right():
    """A chunked call of fewer items than SMs runs every item as two halves of
    its key range, the later half combining both.  CTA 0 (the first half of
    the heaviest item) has its wait run out: its softmax warps still pass the
    split's barriers, its partial is not written, and nothing waits on it;
    the item's rows are then unspecified (the call reports PA_ERR_TIMEOUT),
    the other items are right, and so is the next call."""
    torch = H.torch_mod()
    geom = W.Geometry(8, 2, 64, 1, 2, 72, 160)
    case = W.make_chunked_case("held_split", geom, [300, 200], [700, 300], seed=33, pool_fill="nan")
    pool, bt, werr = H.gpu_setup(case)
    assert werr == 0
    ro, rl = H.oracle_prefill_cached(case, H.oracle_pool(case))
    vmax = H.max_abs_v(case)

    def run():
        o = torch.zeros((case.total_tokens, 8, 64), dtype=torch.int16, device="cuda")
        lse = torch.empty((case.total_tokens, 8), dtype=torch.float32, device="cuda")
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        pa.pa_prefill_cached(H.pa_geom(case), H.to_dev(case.q), pool, bt, 0, H.to_dev(case.cu_seqlens),
                             H.to_dev(case.extra["prefix"]), H.to_dev(case.slots), case.max_len, case.scale,
                             o, lse, err)
        torch.cuda.synchronize()
        return H.f32(o.cpu().numpy().view(np.uint16)), lse.cpu().numpy().astype(np.float64), int(err.item())

    (o, l, err), secs = _held(run)
    assert err == pa.PA_ERR_TIMEOUT, pa.pa_status_string(err)
    assert secs >= 0.9 * WAIT_LIMIT_S
    # item 0: the last 128-row tile of sequence 0 (rows 640..699), q heads 0..3
    held = np.zeros((case.total_tokens, 8), bool)
    held[640:700, 0:4] = True
    ok = ~held
    H.assert_close(o[ok], l[ok], ro[ok], rl[ok], vmax, "rows of the other items")
    o2, l2, err2 = run()
    assert err2 == 0
    H.assert_close(o2, l2, ro, rl, vmax, "the call after the timeout")

"""pa_decode_noalloc: decode for callers that cannot allocate device memory.

Some callers cannot hand pa_decode a workspace: a plugin whose host
application has already reserved the device memory for its own allocator, or
a serving loop that must not call cudaMalloc (it can synchronise the device)
between steps.  pa_decode_noalloc keeps the split partials in a fixed scratch
array inside the library instead.  This test calls it through the C ABI twice
in a row, on two different batches, and checks each result against pa_decode
with a caller workspace on the same inputs -- the same kernels with the same
split, so bit for bit -- and against the CPU oracle at the parity tolerance
of the other GPU tests.  It lives in its own file, collected last, and passes
both in a fresh process (the first call does the per-device set-up) and after
the other tests.
"""
import numpy as np
import pytest

import paged_kv_cache_gb300 as pa
from paged_kv_cache_gb300 import workloads as W
from tests import helpers as H

pytestmark = pytest.mark.gpu


def _noalloc(case, pool, bt):
    torch = H.torch_mod()
    g = H.pa_geom(case)
    B, Hq, D = case.batch, case.geom.num_q_heads, case.geom.head_dim
    o = torch.empty((B, Hq, D), dtype=torch.int16, device="cuda")
    lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.pa_decode_noalloc(g, H.to_dev(case.q), pool, bt, case.layer, H.to_dev(case.lens),
                         H.to_dev(case.slots), case.max_len, case.scale, o, lse, err)
    torch.cuda.synchronize()
    return H.f32(o.cpu().numpy().view(np.uint16)), lse.cpu().numpy().astype(np.float64), int(err.item())


def test_no_alloc_decode_matches_workspace_decode_twice():
    geom = W.Geometry(32, 8, 64, 1, 40, 160, 4000)
    first = W.make_decode_case("noalloc_a", geom, W.uniform_decode_lens(1002, 40), seed=77, pool_fill="nan")
    second = W.make_decode_case("noalloc_b", geom, [0, 1, 17, 2048, 300] * 8, seed=78, pool_fill="nan")
    for case in (first, second):
        pool, bt, werr = H.gpu_setup(case)
        assert werr == 0
        o_ws, l_ws, err_ws = H.gpu_decode(case, pool, bt)  # caller-provided workspace
        o, l, err = _noalloc(case, pool, bt)
        assert err_ws == 0 and err == 0
        # the same kernels and the same split on the same inputs: identical bits
        assert np.array_equal(o, o_ws), "noalloc %s: o differs from pa_decode" % case.name
        assert np.array_equal(l, l_ws), "noalloc %s: lse differs from pa_decode" % case.name
        ro, rl = H.oracle_decode(case, H.oracle_pool(case))
        H.assert_close(o, l, ro, rl, H.max_abs_v(case), "noalloc " + case.name)


def test_no_alloc_rejects_requests_beyond_the_scratch():
    torch = H.torch_mod()
    g = pa.geom(32, 8, 64, 1, 4096, 1024, 1024)
    assert pa.pa_decode_workspace_size(g, 4096, 16384) > pa.PA_DECODE_STATIC_SCRATCH_BYTES
    dummy = torch.zeros(16, dtype=torch.int32, device="cuda")
    with pytest.raises(pa.PaError) as e:
        pa.pa_decode_noalloc(g, dummy, dummy, dummy, 0, dummy, dummy, 16384, 0.125, dummy, None, dummy,
                             batch=4096)
    assert e.value.code == pa.PA_ERR_UNSUPPORTED

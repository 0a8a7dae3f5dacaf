"""Per-phase timeline of the decode kernels (a profiling aid).

Builds the profiling variant of the library (``build.py --trace``:
globaltimer marks in the decode kernels), runs a decode batch the way the
bench times it -- a new token written, then pa_decode, with L2 emptied before
each call (a 256 MiB write, then a 256 MiB read) -- and prints, per call, the
events' duration and the kernels' phases on the GPU's own clock, relative to
the first attend CTA's start:
  last CTA start, median / last first page in shared memory, median / last
  attend CTA end, the merge past its grid dependency, the last merge end;
and for the last call the spread of the attend CTAs' streaming time.

Usage: python -m paged_kv_cache_gb300.decode_trace [--batch 64|256] [--calls N]
  --batch 64:  64 sequences, lengths uniform in [128, 2048], 2 GiB pool;
  --batch 256: 256 sequences, lengths round(LogNormal(ln 1024, 1)) clipped to
               [1, 16384], 4 GiB pool.
32 q / 8 kv heads, d 64, pages shuffled over the pool, seeded as the bench's
decode legs.
"""
import argparse
import ctypes as C

import numpy as np

from . import build as B
from . import workloads as W

ATTEND, MERGE = 1024, 8192  # mark slots of the trace build (decode.cu)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--batch", type=int, choices=[64, 256], default=64)
    ap.add_argument("--calls", type=int, default=6)
    args = ap.parse_args()
    import torch
    import paged_kv_cache_gb300 as pa

    lib = pa.load_library(B.build_trace())
    pa._lib = lib  # every pa_* call of this process goes to the trace build
    lib.pa_trace_decode_read.argtypes = [C.c_void_p, C.c_size_t]
    lib.pa_trace_decode_read.restype = C.c_int
    lib.pa_trace_decode_reset.restype = C.c_int

    if args.batch == 64:
        seed, lens = 1002, W.uniform_decode_lens(1002)
        geom = W.Geometry(32, 8, 64, 1, lens.shape[0], 128, 65536)
    else:
        seed, lens = 1004, W.lognormal_decode_lens(1004)
        geom = W.Geometry(32, 8, 64, 1, lens.shape[0], 1024, 131072)
    B_ = lens.shape[0]
    rng = np.random.default_rng(seed + 1)
    table = W.empty_table(geom)
    free = W.FreeList(geom.num_blocks, rng)
    for b in range(B_):
        W.assign_pages(table, free, b, 0, int(lens[b]))
    g = pa.geom(*geom.as_tuple())
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    gen = torch.Generator(device="cuda")
    gen.manual_seed(seed)
    pre = np.maximum(lens - 1, 0)
    bt = dev(table)
    pool = torch.empty(geom.pool_bytes, dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    k = torch.randn((int(pre.sum()), geom.kv_dim), generator=gen, device="cuda").to(torch.bfloat16)
    v = torch.randn((int(pre.sum()), geom.kv_dim), generator=gen, device="cuda").to(torch.bfloat16)
    pa.pa_write_kv(g, pool, bt, 0, dev(np.repeat(np.arange(B_, dtype=np.int32), pre)),
                   dev(np.concatenate([np.arange(n, dtype=np.int32) for n in pre])), k, v, err)
    del k, v
    new_slot, new_pos = dev(np.arange(B_, dtype=np.int32)), dev((lens - 1).astype(np.int32))
    new_k = torch.randn((B_, geom.kv_dim), generator=gen, device="cuda").to(torch.bfloat16)
    new_v = torch.randn((B_, geom.kv_dim), generator=gen, device="cuda").to(torch.bfloat16)
    q = torch.randn((B_, 32, 64), generator=gen, device="cuda").to(torch.bfloat16)
    lens_d, slots = dev(lens), dev(np.arange(B_, dtype=np.int32))
    o = torch.empty((B_, 32, 64), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B_, 32), dtype=torch.float32, device="cuda")
    max_len = int(lens.max())
    ws = torch.empty(pa.pa_decode_workspace_size(g, B_, max_len), dtype=torch.uint8, device="cuda")
    flush_w = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    flush_r = torch.ones(64 << 20, dtype=torch.float32, device="cuda")
    kv_bytes = float(lens.sum()) * 2 * geom.kv_dim * 2

    def call(ev=None):
        flush_w.zero_()
        flush_r.sum()
        pa.pa_write_kv(g, pool, bt, 0, new_slot, new_pos, new_k, new_v, err)
        if ev:
            ev[0].record()
        pa.pa_decode(g, q, pool, bt, 0, lens_d, slots, max_len, 0.125, o, lse, ws, err)
        if ev:
            ev[1].record()

    for _ in range(3):
        call()
    torch.cuda.synchronize()
    buf = np.zeros(ATTEND * 4 + MERGE * 2, np.uint64)
    print("batch %d: %.1f MB of K/V per call; times in us from the first attend CTA's start" % (B_, kv_bytes / 1e6))
    print("events | last CTA start | first page med / last | CTA end med / last | merge past dependency | "
          "merge end | GB/s by events")
    for _ in range(args.calls):
        assert lib.pa_trace_decode_reset() == 0
        ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
        call(ev)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        assert lib.pa_trace_decode_read(buf.ctypes.data, buf.nbytes) == 0
        a = buf[:ATTEND * 4].reshape(ATTEND, 4).astype(np.int64)
        a = a[a[:, 0] > 0]
        m = buf[ATTEND * 4:].reshape(MERGE, 2).astype(np.int64)
        m = m[m[:, 0] > 0]
        t0 = a[:, 0].min()
        us = lambda x: (x - t0) / 1e3
        e_us = ev[0].elapsed_time(ev[1]) * 1e3
        print("%.2f | %.2f | %.2f / %.2f | %.2f / %.2f | %.2f | %.2f | %.0f" % (
            e_us, us(a[:, 0].max()), us(np.median(a[:, 1])), us(a[:, 1].max()), us(np.median(a[:, 2])),
            us(a[:, 2].max()), us(m[:, 0].min()) if len(m) else -1, us(m[:, 1].max()) if len(m) else -1,
            kv_bytes / e_us / 1e3))
    if len(m):
        pct = lambda x: " ".join("%.1f" % y for y in np.percentile(x, [0, 10, 50, 90, 100]))
        print("last call, %d merge CTAs: past the dependency pct 0/10/50/90/100: %s; its own time (dependency -> "
              "end) %s" % (len(m), pct(us(m[:, 0])), pct((m[:, 1] - m[:, 0]) / 1e3)))
    stream = (a[:, 2] - a[:, 1]) / 1e3
    print("last call, %d attend CTAs: first page -> end, us: min %.2f median %.2f max %.2f; CTA end pct 0/10/50/90/100: %s"
          % (len(a), stream.min(), np.median(stream), stream.max(),
             " ".join("%.1f" % x for x in np.percentile(us(a[:, 2]), [0, 10, 50, 90, 100]))))


if __name__ == "__main__":
    main()

"""Benchmark of the paged-attention hot path on GB300.

One step = one pass of the whole path over one batch, inputs resident in HBM:
  pa_write_kv  (the batch's prompt K/V, 4 x 8192 rows, into shuffled pages)
  pa_prefill   (causal, 4 x 8192 tokens, 32 q / 8 kv heads, d 64)
  pa_write_kv  (one new token per sequence at position 8192)
  pa_decode    (4 sequences of 8193 tokens)
The headline value is the step's algorithmic causal-attention FLOPs per
second (TFLOP/s; exact causal count 4 d Hq sum_b n_b (n_b + 1) / 2 plus the
decode's 4 d Hq n).  The line also carries:
  roofline     -- the prefill kernel (the dominant launch) against the measured
                  dense bf16 peak;
  prefill_d128 -- the same step at head dim 128 (16 q / 4 kv heads, the same
                  FLOPs), its prefill against the same peak (prefill_d64 when
                  --variant d128 is the main step);
  decode       -- decode KV-read GB/s on the large mixed-length batch (256
                  sequences, log-normal lengths, new-token write + decode per
                  step) against the measured HBM copy bandwidth; batch64: the
                  same for 64 sequences of 128..2048 tokens;
  scatter      -- pa_write_kv and pa_write_kv_rope GB/s on the prompt rows
                  against the measured HBM copy bandwidth;
  prefill_rope_q -- the main prefill with RoPE on the queries in the
                  kernel's prologue (pa_prefill_rope), and its cost over the
                  plain prefill;
  llama_prompts -- pa_prefill of the Llama-3.2-1B-shaped prompts (17 and 512
                  tokens, K/V scattered at layers 0 and 15): latency-bound,
                  reported with its own oracle baseline;
  chunked      -- pa_prefill_cached: 4 x 2048-query chunks after 6144 cached
                  tokens, exact-causal TFLOP/s against the same bf16 peak;
  backward     -- pa_prefill_backward on the long prompt (4 x 8192, d 64;
                  d128: 16 q / 4 kv heads): 2.5 x the exact causal count,
                  TFLOP/s against that peak;
  e2e          -- the same metric through the C ABI with host buffers: pinned
                  H2D of every step's inputs and D2H of its outputs inside the
                  timed region, neighbouring steps' copies overlapping the
                  compute (and, as "serial", without that overlap);
  cpu_baseline -- the fp64 CPU oracle timed on a bounded sample of the same
                  workload on this host's cores (and, inside the decode and
                  llama_prompts legs, on samples of those workloads);
  gates        -- last key of the line: each bar's fraction of its measured
                  peak (prefill d 64 / d 128 against 0.55, the two decode
                  batches against 0.75).
N > 1 (torchrun): independent replicas, one per GPU, no collective on the
data path ("weak" scaling); timing is the max over ranks.
``--impl reference`` times the CPU oracle itself as the reference arm.
"""
import argparse
import hashlib
import json
import math
import os
import re
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20  # > the 129 MB L2


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--variant", choices=["d64", "d128"], default="d64")
    ap.add_argument("--decode-steps", type=int, default=None)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="target oracle sample time (10-30 s)")
    ap.add_argument("--only", choices=["all", "prefill", "llama", "decode", "chunked", "scatter", "pages", "backward"],
                    default="all",
                    help="profiling aid: run only the main (prefill) step or only the decode step")
    ap.add_argument("--batch", type=int, default=4, help="prefill sequences (profiling aid)")
    ap.add_argument("--seqlen", type=int, default=8192, help="prefill length (profiling aid)")
    return ap.parse_args()


# ------------------------------------------------------------------ helpers

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash(names=None):
    """Hash of the library's CUDA sources: every .cu / .cuh file, or only the
    files named (a traffic figure taken on other sources is not reported)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_cache_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh")) and (names is None or name in names):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(f.read())
    if names is not None:
        with open(os.path.join(ROOT, "include", "pa.h"), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


# The sources each profiled kernel is built from: its own file(s), the shared
# device header and the C-ABI front end (pa.h is added by kernel_source_hash).
TRAFFIC_SOURCES = {
    "prefill": ("prefill.cu", "pa_internal.cuh", "api.cu"),
    "chunked": ("prefill.cu", "pa_internal.cuh", "api.cu"),
    "decode": ("decode.cu", "pa_internal.cuh", "api.cu"),
    "backward": ("backward.cu", "backward_tc.cu", "pa_internal.cuh", "api.cu"),
    "scatter": ("write_kv.cu", "pa_internal.cuh", "api.cu"),
}


def traffic_key(kernel_tag):
    """Source hash a traffic row must carry: that of the tagged kernel's own sources."""
    return kernel_source_hash(TRAFFIC_SOURCES[kernel_tag.split("_")[0]])


def prefill_heads_per_cta(geom):
    """q heads of one GQA group that one prefill CTA takes (the library's rule:
    as many as tensor memory holds, 4 at d 64 and 2 at d 128)."""
    group = geom.num_q_heads // geom.num_kv_heads
    if geom.head_dim == 64 and group % 4 == 0:
        return 4
    return 2 if group % 2 == 0 else 1


def profiled_traffic(kernel_tag):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current sources of that kernel (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.md")
    if not os.path.exists(path):
        return None
    want = traffic_key(kernel_tag)
    for line in open(path):
        m = re.match(r"\|\s*%s\s*\|\s*([0-9a-f]+)\s*\|\s*([0-9.eE+]+)\s*\|" % re.escape(kernel_tag), line)
        if m and m.group(1) == want:
            return float(m.group(2))
    return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled during the timed region."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", "pa_clocks_%d_%d.csv" % (os.getpid(), gpu_index))

    def start(self):
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.QUERY,
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.out,
                stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons, "samples": len(rows)}


# --------------------------------------------------------------- workloads

def causal_flops(d, hq, lens):
    return float(sum(4.0 * d * hq * n * (n + 1) / 2.0 for n in lens))


class PrefillStep:
    """Device-resident inputs of the main step (write + prefill + write + decode)."""

    def __init__(self, torch, pa, W, variant, seed=1003, batch=4, seqlen=8192):
        self.torch, self.pa = torch, pa
        self.case = W.long_prefill_case(variant, seed=seed, batch=batch, seqlen=seqlen)
        c = self.case
        geom = c.geom
        # one more page per sequence for the decoded token (position 8192)
        self.geom = W.Geometry(geom.num_q_heads, geom.num_kv_heads, geom.head_dim, 1, geom.num_slots,
                               geom.max_blocks_per_seq + 1, geom.num_blocks)
        table = np.full((geom.num_slots, 1, self.geom.max_blocks_per_seq), -1, np.int32)
        table[:, :, :geom.max_blocks_per_seq] = c.block_table
        used = set(c.block_table[c.block_table >= 0].tolist())
        spare = [p for p in range(geom.num_blocks - 1, -1, -1) if p not in used][:c.batch]
        n_prompt = int(c.lens[0])
        for b in range(c.batch):  # page of the decoded token, if the prompt left none
            if table[b, 0, n_prompt // 16] < 0:
                table[b, 0, n_prompt // 16] = spare[b]
        self.table_np = table
        self.g = pa.geom(*self.geom.as_tuple())
        rng = np.random.default_rng(seed + 50)
        n = int(c.lens[0])
        self.new_slot = np.arange(c.batch, dtype=np.int32)
        self.new_pos = np.full(c.batch, n, np.int32)
        self.new_k = W.normal_bf16(rng, (c.batch, geom.kv_dim))
        self.new_v = W.normal_bf16(rng, (c.batch, geom.kv_dim))
        self.dec_q = W.normal_bf16(rng, (c.batch, geom.num_q_heads, geom.head_dim))
        self.dec_lens = np.full(c.batch, n + 1, np.int32)
        dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
        w = c.writes[0]
        self.h = {"q": c.q, "k": w.k, "v": w.v, "tok_slot": w.tok_slot, "tok_pos": w.tok_pos,
                  "cu": c.cu_seqlens, "slots": c.slots, "bt": table, "new_slot": self.new_slot,
                  "new_pos": self.new_pos, "new_k": self.new_k, "new_v": self.new_v, "dec_q": self.dec_q,
                  "dec_lens": self.dec_lens}
        self.d = {k: dev(v) for k, v in self.h.items()}
        self.pool = torch.empty(self.geom.pool_bytes, dtype=torch.uint8, device="cuda")
        T, Hq, D = c.total_tokens, geom.num_q_heads, geom.head_dim
        self.o = torch.empty((T, Hq, D), dtype=torch.int16, device="cuda")
        self.lse = torch.empty((T, Hq), dtype=torch.float32, device="cuda")
        self.dec_o = torch.empty((c.batch, Hq, D), dtype=torch.int16, device="cuda")
        self.dec_lse = torch.empty((c.batch, Hq), dtype=torch.float32, device="cuda")
        self.ws = torch.empty(pa.pa_decode_workspace_size(self.g, c.batch, n + 1), dtype=torch.uint8,
                              device="cuda")
        self.err = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.n = n
        self.flops_prefill = causal_flops(geom.head_dim, Hq, c.lens)
        self.flops_decode = float(4.0 * geom.head_dim * Hq * np.sum(self.dec_lens))
        self.flops = self.flops_prefill + self.flops_decode
        self.launches = 5  # write, prefill, write, attend, merge

    def outputs(self):
        """Fresh device output buffers (o, lse, decode o, decode lse)."""
        return tuple(self.torch.empty_like(t) for t in (self.o, self.lse, self.dec_o, self.dec_lse))

    def run(self, d=None, ev=None, out=None):
        pa, c = self.pa, self.case
        d = self.d if d is None else d
        o, lse, dec_o, dec_lse = (self.o, self.lse, self.dec_o, self.dec_lse) if out is None else out
        pa.pa_write_kv(self.g, self.pool, d["bt"], 0, d["tok_slot"], d["tok_pos"], d["k"], d["v"], self.err)
        if ev is not None:
            ev[0].record()
        pa.pa_prefill(self.g, d["q"], self.pool, d["bt"], 0, d["cu"], d["slots"], self.n, c.scale, o, lse,
                      self.err)
        if ev is not None:
            ev[1].record()
        pa.pa_write_kv(self.g, self.pool, d["bt"], 0, d["new_slot"], d["new_pos"], d["new_k"], d["new_v"],
                       self.err)
        pa.pa_decode(self.g, d["dec_q"], self.pool, d["bt"], 0, d["dec_lens"], d["slots"], self.n + 1,
                     c.scale, dec_o, dec_lse, self.ws, self.err)


class RopePrefillStep:
    """The main step's prompts with RoPE on both sides: the prompt K/V
    scattered with K turned (pa_write_kv_rope), then pa_prefill_rope, which
    turns every query row in the kernel's prologue (same FLOPs as the plain
    prefill: the prologue is what it costs)."""

    def __init__(self, torch, pa, W, step):
        self.torch, self.pa, self.step = torch, pa, step
        geom = step.case.geom
        cos_t, sin_t = W.rope_tables(int(step.case.lens.max()) + 1, geom.head_dim)
        self.cos = torch.from_numpy(cos_t).cuda()
        self.sin = torch.from_numpy(sin_t).cuda()
        self.flops = step.flops_prefill

    def run(self, ev=None):
        pa, st, c, d = self.pa, self.step, self.step.case, self.step.d
        pa.pa_write_kv_rope(st.g, st.pool, d["bt"], 0, d["tok_slot"], d["tok_pos"], d["k"], d["v"], self.cos, self.sin,
                            st.err)
        if ev is not None:
            ev[0].record()
        pa.pa_prefill_rope(st.g, d["q"], st.pool, d["bt"], 0, d["cu"], None, d["slots"], st.n, c.scale, self.cos,
                           self.sin, st.o, st.lse, st.err)
        if ev is not None:
            ev[1].record()


class ScatterStep:
    """The prompt K/V scatter of the main step (4 x 8192 rows of 2 x 512 bf16
    into shuffled pages), plain and with RoPE on K.  Algorithmic bytes per
    call: K and V rows read once and written once, plus (RoPE) one cos and one
    sin table row of head_dim/2 fp32 per token."""

    def __init__(self, torch, pa, W, seed=1003):
        self.torch, self.pa = torch, pa
        c = W.long_prefill_case("d64", seed=seed)
        self.case, self.geom = c, c.geom
        self.g = pa.geom(*c.geom.as_tuple())
        dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
        w = c.writes[0]
        cos_t, sin_t = W.rope_tables(int(c.lens.max()), c.geom.head_dim)
        self.d = {"bt": dev(c.block_table), "tok_slot": dev(w.tok_slot), "tok_pos": dev(w.tok_pos),
                  "k": dev(w.k), "v": dev(w.v), "cos": dev(cos_t), "sin": dev(sin_t)}
        self.pool = torch.empty(c.geom.pool_bytes, dtype=torch.uint8, device="cuda")
        self.err = torch.zeros(1, dtype=torch.int32, device="cuda")
        n = int(w.tok_slot.shape[0])
        self.bytes_plain = float(n * c.geom.kv_dim * 2 * 2 * 2)
        self.bytes_rope = self.bytes_plain + float(n * c.geom.head_dim // 2 * 4 * 2)

    def run(self, rope, ev=None):
        pa, d = self.pa, self.d
        if ev is not None:
            ev[0].record()
        if rope:
            pa.pa_write_kv_rope(self.g, self.pool, d["bt"], 0, d["tok_slot"], d["tok_pos"], d["k"], d["v"],
                                d["cos"], d["sin"], self.err)
        else:
            pa.pa_write_kv(self.g, self.pool, d["bt"], 0, d["tok_slot"], d["tok_pos"], d["k"], d["v"], self.err)
        if ev is not None:
            ev[1].record()


class ChunkedStep:
    """Prefill of query chunks over a cached prefix: 4 sequences, each a
    2048-query chunk after 6144 cached tokens (the last quarter of the long
    prompt of the main step), 32 q / 8 kv heads, d 64.  A step = scatter of
    the chunks' K/V + pa_prefill_cached; the prefix is written once."""

    def __init__(self, torch, pa, W, seed=1006, batch=4, prefix=6144, chunk=2048):
        self.torch, self.pa = torch, pa
        pages = (prefix + chunk) // 16
        geom = W.Geometry(32, 8, 64, 1, batch, pages, batch * pages + 64)
        self.case = W.make_chunked_case("chunk", geom, [prefix] * batch, [chunk] * batch, seed)
        c = self.case
        self.geom, self.g = geom, pa.geom(*geom.as_tuple())
        dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
        w_pre, w_chunk = c.writes
        self.d = {"q": dev(c.q), "bt": dev(c.block_table), "cu": dev(c.cu_seqlens), "pre": dev(c.extra["prefix"]),
                  "slots": dev(c.slots), "tok_slot": dev(w_chunk.tok_slot), "tok_pos": dev(w_chunk.tok_pos),
                  "k": dev(w_chunk.k), "v": dev(w_chunk.v)}
        self.pool = torch.empty(geom.pool_bytes, dtype=torch.uint8, device="cuda")
        self.err = torch.zeros(1, dtype=torch.int32, device="cuda")
        pa.pa_write_kv(self.g, self.pool, self.d["bt"], 0, dev(w_pre.tok_slot), dev(w_pre.tok_pos), dev(w_pre.k),
                       dev(w_pre.v), self.err)
        T, Hq, D = c.total_tokens, geom.num_q_heads, geom.head_dim
        self.o = torch.empty((T, Hq, D), dtype=torch.int16, device="cuda")
        self.lse = torch.empty((T, Hq), dtype=torch.float32, device="cuda")
        self.chunk = chunk
        # exact causal count: query i of a chunk sees prefix + i + 1 keys
        self.flops = float(batch * 4.0 * D * Hq * (chunk * prefix + chunk * (chunk + 1) / 2))

    def run(self, ev=None):
        pa, c, d = self.pa, self.case, self.d
        pa.pa_write_kv(self.g, self.pool, d["bt"], 0, d["tok_slot"], d["tok_pos"], d["k"], d["v"], self.err)
        if ev is not None:
            ev[0].record()
        pa.pa_prefill_cached(self.g, d["q"], self.pool, d["bt"], 0, d["cu"], d["pre"], d["slots"], self.chunk,
                             c.scale, self.o, self.lse, self.err)
        if ev is not None:
            ev[1].record()


class BackwardStep:
    """Gradients of the long-prompt prefill (4 x 8192 tokens; 32 q / 8 kv heads
    at d 64, 16 / 4 at d 128): the forward runs once to give o and lse; a step
    is one pa_prefill_backward (D = do . o, then the column-block kernel)."""

    def __init__(self, torch, pa, W, seed=1007, batch=4, seqlen=8192, heads=(32, 8, 64)):
        self.torch, self.pa = torch, pa
        pages = (seqlen + 15) // 16
        geom = W.Geometry(heads[0], heads[1], heads[2], 1, batch, pages, batch * pages + 64)
        case = W.make_prefill_case("bwd", geom, [seqlen] * batch, seed)
        self.case, self.geom = case, geom
        self.g = pa.geom(*self.geom.as_tuple())
        dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
        w = case.writes[0]
        self.d = {"q": dev(case.q), "bt": dev(case.block_table), "cu": dev(case.cu_seqlens), "slots": dev(case.slots)}
        self.pool = torch.empty(self.geom.pool_bytes, dtype=torch.uint8, device="cuda")
        self.err = torch.zeros(1, dtype=torch.int32, device="cuda")
        pa.pa_write_kv(self.g, self.pool, self.d["bt"], 0, dev(w.tok_slot), dev(w.tok_pos), dev(w.k), dev(w.v),
                       self.err)
        T, Hq, Hkv, D = case.total_tokens, self.geom.num_q_heads, self.geom.num_kv_heads, self.geom.head_dim
        self.o = torch.empty((T, Hq, D), dtype=torch.int16, device="cuda")
        self.lse = torch.empty((T, Hq), dtype=torch.float32, device="cuda")
        pa.pa_prefill(self.g, self.d["q"], self.pool, self.d["bt"], 0, self.d["cu"], self.d["slots"], case.max_len,
                      case.scale, self.o, self.lse, self.err)
        gen = torch.Generator(device="cuda")
        gen.manual_seed(seed)
        self.dout = torch.randn((T, Hq, D), generator=gen, device="cuda").to(torch.bfloat16)
        self.delta = torch.empty((2, T, Hq), dtype=torch.float32, device="cuda")
        self.dq = torch.empty((T, Hq, D), dtype=torch.float32, device="cuda")
        self.dk = torch.empty((T, Hkv, D), dtype=torch.float32, device="cuda")
        self.dv = torch.empty((T, Hkv, D), dtype=torch.float32, device="cuda")
        # 5 products of 2 d flops per (query, key) pair on or below the diagonal: 2.5 x the forward's count
        self.flops = float(10.0 * D * Hq * np.sum(case.lens.astype(np.float64) * (case.lens + 1) / 2))

    def run(self, ev=None):
        pa, c, d = self.pa, self.case, self.d
        if ev is not None:
            ev[0].record()
        pa.pa_prefill_backward(self.g, d["q"], self.pool, d["bt"], 0, d["cu"], d["slots"], c.max_len, c.scale,
                               self.o, self.lse, self.dout, self.delta, self.dq, self.dk, self.dv, self.err)
        if ev is not None:
            ev[1].record()


class LlamaPromptStep:
    """Prefill of the Llama-3.2-1B-shaped prompts (2 slots, 17 and 512 tokens,
    32 q / 8 kv heads, d 64, 2 GiB pool, table [2][16][128]): a step scatters
    both prompts' K/V at layers 0 and 15 and runs pa_prefill at layer 15.
    Exact causal FLOPs 4 d Hq sum n (n + 1) / 2 = 1.077 GFLOP: a
    latency-bound call, reported beside the long prefill, not against its bar."""

    def __init__(self, torch, pa, W):
        self.torch, self.pa = torch, pa
        self.case = c = W.llama_prefill_case()
        self.g = pa.geom(*c.geom.as_tuple())
        dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
        self.d = {"q": dev(c.q), "bt": dev(c.block_table), "cu": dev(c.cu_seqlens), "slots": dev(c.slots)}
        self.w = [(w.layer, dev(w.tok_slot), dev(w.tok_pos), dev(w.k), dev(w.v)) for w in c.writes]
        self.pool = torch.empty(c.geom.pool_bytes, dtype=torch.uint8, device="cuda")
        self.err = torch.zeros(1, dtype=torch.int32, device="cuda")
        T, Hq, D = c.total_tokens, c.geom.num_q_heads, c.geom.head_dim
        self.o = torch.empty((T, Hq, D), dtype=torch.int16, device="cuda")
        self.lse = torch.empty((T, Hq), dtype=torch.float32, device="cuda")
        self.flops = causal_flops(D, Hq, c.lens)
        self.write_bytes = float(sum(w.k.size * 2 * 2 * 2 for w in c.writes))  # K and V, read and written

    def run(self, ev=None):
        pa, c, d = self.pa, self.case, self.d
        for layer, ts, tp, k, v in self.w:
            pa.pa_write_kv(self.g, self.pool, d["bt"], layer, ts, tp, k, v, self.err)
        if ev is not None:
            ev[0].record()
        pa.pa_prefill(self.g, d["q"], self.pool, d["bt"], c.layer, d["cu"], d["slots"], c.max_len, c.scale,
                      self.o, self.lse, self.err)
        if ev is not None:
            ev[1].record()


class DecodeStep:
    """A decode batch: c-1 tokens preloaded, each step writes the token at c-1
    and decodes c.  Default: the large mixed batch (256 sequences, log-normal
    lengths, 4 GiB pool); small=True: 64 sequences, lengths uniform in
    [128, 2048], 2 GiB pool."""

    def __init__(self, torch, pa, W, seed=1004, small=False, layers=1):
        self.torch, self.pa = torch, pa
        self.layers = layers
        if small:
            seed = 1002
            lens = W.uniform_decode_lens(seed)
            self.geom = W.Geometry(32, 8, 64, layers, lens.shape[0], 128, 65536)
        else:
            lens = W.lognormal_decode_lens(seed)
            self.geom = W.Geometry(32, 8, 64, layers, lens.shape[0], 1024, 131072)
        self.lens_np = lens
        B = lens.shape[0]
        rng = np.random.default_rng(seed + 1)
        table = W.empty_table(self.geom)
        free = W.FreeList(self.geom.num_blocks, rng)
        for layer in range(layers):  # every layer has pages of its own
            for b in range(B):
                W.assign_pages(table, free, b, layer, int(lens[b]))
        self.g = pa.geom(*self.geom.as_tuple())
        gen = torch.Generator(device="cuda")
        gen.manual_seed(seed)
        kv_dim = self.geom.kv_dim
        pre = np.maximum(lens - 1, 0)
        tok_slot = np.repeat(np.arange(B, dtype=np.int32), pre)
        tok_pos = np.concatenate([np.arange(n, dtype=np.int32) for n in pre])
        dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
        self.bt = dev(table)
        self.pool = torch.empty(self.geom.pool_bytes, dtype=torch.uint8, device="cuda")
        self.err = torch.zeros(1, dtype=torch.int32, device="cuda")
        for layer in range(layers):
            k = torch.randn((int(pre.sum()), kv_dim), generator=gen, device="cuda").to(torch.bfloat16)
            v = torch.randn((int(pre.sum()), kv_dim), generator=gen, device="cuda").to(torch.bfloat16)
            pa.pa_write_kv(self.g, self.pool, self.bt, layer, dev(tok_slot), dev(tok_pos), k, v, self.err)
            del k, v
        self.new_slot = dev(np.arange(B, dtype=np.int32))
        self.new_pos = dev((lens - 1).astype(np.int32))
        self.new_k = torch.randn((B, kv_dim), generator=gen, device="cuda").to(torch.bfloat16)
        self.new_v = torch.randn((B, kv_dim), generator=gen, device="cuda").to(torch.bfloat16)
        self.q = torch.randn((B, 32, 64), generator=gen, device="cuda").to(torch.bfloat16)
        self.lens = dev(lens)
        self.slots = dev(np.arange(B, dtype=np.int32))
        self.o = torch.empty((B, 32, 64), dtype=torch.bfloat16, device="cuda")
        self.lse = torch.empty((B, 32), dtype=torch.float32, device="cuda")
        self.max_len = int(lens.max())
        self.ws = torch.empty(pa.pa_decode_workspace_size(self.g, B, self.max_len), dtype=torch.uint8,
                              device="cuda")
        self.kv_bytes = float(np.sum(lens)) * 2 * kv_dim * 2  # K and V rows read
        torch.cuda.synchronize()
        assert int(self.err.item()) == 0

    def run(self, ev=None, layer=0):
        pa = self.pa
        pa.pa_write_kv(self.g, self.pool, self.bt, layer, self.new_slot, self.new_pos, self.new_k, self.new_v,
                       self.err)
        if ev is not None:
            ev[0].record()
        pa.pa_decode(self.g, self.q, self.pool, self.bt, layer, self.lens, self.slots, self.max_len, 0.125,
                     self.o, self.lse, self.ws, self.err)
        if ev is not None:
            ev[1].record()


# ----------------------------------------------------------------- timing

class L2Flush:
    """Empties L2 of everything a step touched, between timed steps and outside
    their events: a 256 MiB write (twice the 129 MB L2), then a 256 MiB read.
    The write alone leaves L2 full of its own dirty lines, and the next timed
    kernel then pays for writing them back to DRAM: measured on the decode
    batches, 41.7 against 35.1 us (64 sequences) and 151.4 against 137.8 us
    (256 sequences), and 26.8 against 21.0 us for the prompt scatter.  After
    the read, L2 holds only clean lines of the read buffer, which cost nothing
    to evict, and none of the step's inputs."""

    def __init__(self, torch):
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
        self.r = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
        self.sink = None

    def __call__(self):
        self.w.zero_()
        self.sink = self.r.sum()


def timed(torch, fn, steps, warmup, flush, dist=None, kernel_events=True):
    """Runs fn(ev) warmup + steps times; L2 flushed before every step outside
    the timed events.  Returns (step seconds list, kernel seconds list)."""
    for _ in range(warmup):
        flush()
        fn(None)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    E = torch.cuda.Event
    marks = [(E(enable_timing=True), E(enable_timing=True), E(enable_timing=True), E(enable_timing=True))
             for _ in range(steps)]
    for m in marks:
        flush()
        m[0].record()
        fn((m[2], m[3]) if kernel_events else None)
        m[1].record()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    step_s = [m[0].elapsed_time(m[1]) * 1e-3 for m in marks]
    kern_s = [m[2].elapsed_time(m[3]) * 1e-3 for m in marks] if kernel_events else []
    return step_s, kern_s


def e2e_timing(torch, step, steps, warmup, flush, dist):
    """The step through the C ABI with host buffers: every step copies its
    inputs in from pinned host memory and its outputs (prefill o and lse,
    decode o and lse) back out.  Two figures:
      value  -- pipelined, as a serving loop runs: step s + 1's inputs are
                copied in (copy stream) and step s - 1's outputs copied out
                (another stream) while step s computes; double-buffered
                device inputs and outputs; one timed region over all steps
                (every step's copies inside it; the 201 MB of inputs per step
                exceed L2, so no flush is needed between steps);
      serial -- each step's copy-in, compute and copy-out back to back, L2
                flushed between steps."""
    pin = {k: torch.from_numpy(np.ascontiguousarray(v)).pin_memory() for k, v in step.h.items()}
    h2d = sum(v.numel() * v.element_size() for v in pin.values())
    d_in = [{k: torch.empty_like(v, device="cuda") for k, v in pin.items()} for _ in range(2)]
    d_out = [step.outputs() for _ in range(2)]
    h_out = [tuple(torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in d_out[0]) for _ in range(2)]
    d2h = sum(t.numel() * t.element_size() for t in h_out[0])
    s_c = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    E = torch.cuda.Event
    ev_in = [E(), E()]
    ev_comp = [E(), E()]
    ev_out = [E(), E()]

    def one(s):
        x = s % 2
        with torch.cuda.stream(s_in):
            s_in.wait_event(ev_comp[x])  # the compute of step s - 2 is done with buffer x
            for k, v in pin.items():
                d_in[x][k].copy_(v, non_blocking=True)
            ev_in[x].record(s_in)
        s_c.wait_event(ev_in[x])
        s_c.wait_event(ev_out[x])  # the outputs of step s - 2 have left buffer x
        step.run(d=d_in[x], out=d_out[x])
        ev_comp[x].record(s_c)
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_comp[x])
            for hst, dv in zip(h_out[x], d_out[x]):
                hst.copy_(dv, non_blocking=True)
            ev_out[x].record(s_out)

    for s in range(warmup):
        one(s)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t0, t1 = E(enable_timing=True), E(enable_timing=True)
    t0.record(s_c)
    s_in.wait_stream(s_c)
    s_out.wait_stream(s_c)
    for s in range(steps):
        one(warmup + s)
    s_c.wait_stream(s_out)
    s_c.wait_stream(s_in)
    t1.record(s_c)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    total = t0.elapsed_time(t1) * 1e-3
    rate, total_s, _ = job_rate(torch, dist, step.flops * steps, total)

    def serial_step(ev):
        for k, v in pin.items():
            d_in[0][k].copy_(v, non_blocking=True)
        step.run(d=d_in[0], out=d_out[0])
        for hst, dv in zip(h_out[0], d_out[0]):
            hst.copy_(dv, non_blocking=True)

    es, _ = timed(torch, serial_step, steps, warmup, flush, dist, kernel_events=False)
    s_rate, s_total, _ = job_rate(torch, dist, step.flops * steps, float(np.sum(es)))
    return {"value": rate / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "steps": steps, "ms_per_step": total_s / steps * 1e3,
            "pipelining": "step s+1 copied in and step s-1 copied out while step s computes",
            "serial": {"value": s_rate / 1e12, "unit": "TFLOP/s", "ms_per_step": s_total / steps * 1e3}}


def _rank_device(dist):
    """Tensors for collectives live where the backend wants them: GPU memory
    for NCCL, host memory for gloo."""
    return "cuda" if dist.get_backend() == "nccl" else "cpu"


def max_over_ranks(torch, dist, x):
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=_rank_device(dist))
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(torch, dist, x):
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=_rank_device(dist))
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def job_rate(torch, dist, units, seconds):
    """Whole-job throughput of replicas: the units all ranks processed over
    the slowest rank's time.  Returns (rate, max seconds, total units)."""
    total_s = max_over_ranks(torch, dist, seconds)
    total_u = sum_over_ranks(torch, dist, units)
    return total_u / total_s, total_s, total_u


def page_lifetime_timing(torch, pa, W, warmup, reps=50):
    """Device page allocation for one decode step of 256 sequences x 16 layers
    (lengths log-normal as in the decode batch; every 16th token needs a
    page), and the release of 64 slots; beside them, for context, the copy
    of the whole block table from pinned host memory that the pages' program
    makes after every change.  Latency-bound calls: microseconds per call."""
    lens = W.lognormal_decode_lens()
    B, L = lens.shape[0], 16
    geom = W.Geometry(32, 8, 64, L, B, 1025, B * L * 1100)
    g = pa.geom(*geom.as_tuple())
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    table = dev(W.empty_table(geom))
    stack = dev(np.arange(geom.num_blocks, dtype=np.int32)[::-1].copy())
    count = dev(np.array([geom.num_blocks], np.int32))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    slots = dev(np.arange(B, dtype=np.int32))
    pa.pa_alloc_pages(g, table, slots, dev(lens), stack, count, err)  # the prompts
    old = dev(lens)
    new = dev(lens + 1)
    E = torch.cuda.Event

    def time_call(fn):
        for _ in range(warmup):
            fn()
        torch.cuda.synchronize()
        a, b = E(enable_timing=True), E(enable_timing=True)
        a.record()
        for _ in range(reps):
            fn()
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps * 1e3

    # a step after the first allocates nothing new (old = new - 1 already covered); time the real work:
    # alternate between growing by one token and shrinking the stack back through release/alloc pairs
    alloc_us = time_call(lambda: pa.pa_alloc_pages(g, table, slots, new, stack, count, err, old_lens=old))
    rel = dev(np.arange(64, dtype=np.int32))
    rel_lens = dev(lens[:64])

    def release_then_alloc():
        pa.pa_release_slots(g, table, rel, stack, count, err)
        pa.pa_alloc_pages(g, table, rel, rel_lens, stack, count, err)
    pair_us = time_call(release_then_alloc)
    host_table = torch.from_numpy(W.empty_table(geom)).pin_memory()
    h2d_us = time_call(lambda: table.copy_(host_table, non_blocking=True))
    torch.cuda.synchronize()
    if int(err.item()) != 0:
        raise SystemExit("device error in page lifetime timing: %s" % pa.pa_status_string(int(err.item())))
    return {"metric": "device page lifetime, microseconds per call (256 sequences x 16 layers)",
            "alloc_decode_step_us": alloc_us, "release_64_slots_then_realloc_us": pair_us,
            "table_h2d_copy_us": h2d_us, "table_entries": int(geom.num_slots * L * geom.max_blocks_per_seq),
            "unit": "us"}


# ------------------------------------------------------------ CPU oracle

def oracle_sample(case, seconds, rng_seed=5):
    """Times the oracle on sampled (row, head) outputs of a prefill case,
    growing the sample until it takes about `seconds`.  Returns
    (flops, wall seconds, threads, description)."""
    import oracle
    from paged_kv_cache_gb300 import workloads as W
    g = oracle.geom(*case.geom.as_tuple())
    pool = W.initial_pool(case.geom, "zero", 0)
    for w in case.writes:
        oracle.write_kv(g, pool, case.block_table, w.layer, w.tok_slot, w.tok_pos, w.k, w.v)
    rng = np.random.default_rng(rng_seed)
    cu = case.cu_seqlens
    n_pairs, flops, wall = 16, 0.0, 0.0
    threads = oracle.default_threads()
    while True:
        rows = rng.integers(0, case.total_tokens, n_pairs)
        heads = rng.integers(0, case.geom.num_q_heads, n_pairs).astype(np.int32)
        b = np.searchsorted(cu, rows, side="right") - 1
        pos = rows - cu[b]
        f = float(np.sum(4.0 * case.geom.head_dim * (pos + 1)))
        t0 = time.perf_counter()
        st, _, _ = oracle.prefill_rows(g, case.q, pool, case.block_table, case.layer, cu, case.slots,
                                       case.scale, rows, heads)
        dt = time.perf_counter() - t0
        assert st == 0
        flops, wall = f, dt
        if dt >= seconds * 0.67 or n_pairs >= 1 << 22:
            break
        n_pairs = int(n_pairs * min(64.0, max(1.6, seconds / max(dt, 1e-3))))
    desc = ("%d random (row, q head) outputs of the 4 x 8192 causal prefill (%.3g GFLOP exact-causal), "
            "K/V gathered through the block table, fp64, %d threads" % (n_pairs, flops / 1e9, threads))
    return flops, wall, threads, desc


def oracle_decode_sample(lens, seconds, what, seed, budget_bytes=64 << 20):
    """Times the oracle's decode (fp64, K/V gathered through the block table)
    on the leading sequences of a decode batch -- their lengths, 32 q / 8 kv
    heads, d 64, Q/K/V drawn from N(0, 1) in bf16, pages shuffled -- as many
    as hold about budget_bytes of K/V, the call repeated until it has taken
    about `seconds`.  Returns (KV bytes read, wall seconds, threads,
    description)."""
    import oracle
    from paged_kv_cache_gb300 import workloads as W
    kv_row = 2 * 8 * 64 * 2  # K and V rows of one token, bytes
    k = 1
    while k < lens.shape[0] and float(np.sum(lens[:k + 1].astype(np.float64))) * kv_row <= budget_bytes:
        k += 1
    sub = lens[:k]
    pages = int(np.sum((sub.astype(np.int64) + 15) // 16))
    geom = W.Geometry(32, 8, 64, 1, k, int(max(1, (int(sub.max()) + 15) // 16)), pages + 8)
    case = W.make_decode_case("cpu_" + what, geom, sub, seed, scale=0.125, pool_fill="zero")
    g = oracle.geom(*geom.as_tuple())
    pool = W.initial_pool(geom, "zero", 0)
    for w in case.writes:
        oracle.write_kv(g, pool, case.block_table, w.layer, w.tok_slot, w.tok_pos, w.k, w.v)
    run = lambda: oracle.decode(g, case.q, pool, case.block_table, 0, case.lens, case.slots, case.scale)[0]
    t0 = time.perf_counter()
    assert run() == 0
    dt = time.perf_counter() - t0
    reps = int(min(50, max(1, math.ceil(seconds / max(dt, 1e-3)))))
    t0 = time.perf_counter()
    for _ in range(reps):
        assert run() == 0
    wall = time.perf_counter() - t0
    nbytes = float(np.sum(sub.astype(np.float64))) * kv_row * reps
    desc = ("decode of the first %d of the %d sequences (%.1f MB of K/V), %d calls, fp64 oracle, K/V gathered "
            "through the block table, %d threads" % (k, lens.shape[0], nbytes / reps / 1e6, reps,
                                                     oracle.default_threads()))
    return nbytes, wall, oracle.default_threads(), desc


def oracle_llama_sample(case, seconds):
    """Times the oracle's whole prefill of the Llama-3.2-1B-shaped prompts
    (17 and 512 tokens, every row and head), repeated until it has taken
    about `seconds`.  Returns (FLOPs, wall seconds, threads, description)."""
    import oracle
    from paged_kv_cache_gb300 import workloads as W
    g = oracle.geom(*case.geom.as_tuple())
    pool = W.initial_pool(case.geom, "zero", 0)
    for w in case.writes:
        oracle.write_kv(g, pool, case.block_table, w.layer, w.tok_slot, w.tok_pos, w.k, w.v)
    run = lambda: oracle.prefill(g, case.q, pool, case.block_table, case.layer, case.cu_seqlens, case.slots,
                                 case.scale)[0]
    t0 = time.perf_counter()
    assert run() == 0
    dt = time.perf_counter() - t0
    reps = int(min(50, max(1, math.ceil(seconds / max(dt, 1e-3)))))
    t0 = time.perf_counter()
    for _ in range(reps):
        assert run() == 0
    wall = time.perf_counter() - t0
    flops = causal_flops(case.geom.head_dim, case.geom.num_q_heads, case.lens) * reps
    desc = ("whole prefill of the prompts of 17 and 512 tokens (every row and q head), %d calls, fp64 oracle, "
            "%d threads" % (reps, oracle.default_threads()))
    return flops, wall, oracle.default_threads(), desc


# ------------------------------------------------------------------- arms

METRIC = "causal prefill TFLOP/s (exact causal count, step incl. KV write + decode)"


def step_config(geom, batch, seqlen, world):
    """The workload both arms report: the main step's shape."""
    return {"workload": "long-context causal prefill %d x %d, %d q / %d kv heads, d %d, paged through shuffled "
                        "16-token pages; step = write_kv + prefill + write_kv(new token) + decode(%d)" % (
                            batch, seqlen, geom.num_q_heads, geom.num_kv_heads, geom.head_dim, seqlen + 1),
            "global_batch": batch * world, "seq_len": seqlen, "parallelism": "replicas x%d" % world,
            "l2": "flushed before every timed step, outside the events: a 256 MiB write, then a 256 MiB read "
                  "(so the write's dirty lines are written back before the step, not charged to it)"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    from paged_kv_cache_gb300 import workloads as W
    case = W.long_prefill_case(args.variant)
    per_step = min(5.0, max(0.5, 150.0 / max(1, args.steps + args.warmup)))
    import oracle
    g = oracle.geom(*case.geom.as_tuple())
    pool = W.initial_pool(case.geom, "zero", 0)
    for w in case.writes:
        oracle.write_kv(g, pool, case.block_table, w.layer, w.tok_slot, w.tok_pos, w.k, w.v)
    # calibrate a sample size for ~per_step seconds
    flops1, wall1, threads, _ = oracle_sample(case, per_step)
    rate = flops1 / wall1
    rng = np.random.default_rng(11)
    cu = case.cu_seqlens
    avg_flops_per_pair = 4.0 * case.geom.head_dim * (case.lens.mean() + 1) / 2
    pairs = max(8, int(rate * per_step / avg_flops_per_pair))
    tot_f, tot_t = 0.0, 0.0
    for s in range(args.warmup + args.steps):
        rows = rng.integers(0, case.total_tokens, pairs)
        heads = rng.integers(0, case.geom.num_q_heads, pairs).astype(np.int32)
        b = np.searchsorted(cu, rows, side="right") - 1
        f = float(np.sum(4.0 * case.geom.head_dim * (rows - cu[b] + 1)))
        t0 = time.perf_counter()
        st, _, _ = oracle.prefill_rows(g, case.q, pool, case.block_table, 0, cu, case.slots, case.scale,
                                       rows, heads)
        dt = time.perf_counter() - t0
        assert st == 0
        if s >= args.warmup:
            tot_f += f
            tot_t += dt
    value = tot_f / tot_t / 1e12
    sample = ("per step: %d random (row, q head) outputs of the 4 x 8192 causal prefill, fp64 oracle, "
              "K/V gathered through the block table" % pairs)
    line = {
        "impl": "reference", "metric": METRIC,
        "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": tot_t / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": step_config(case.geom, case.batch, int(case.lens[0]), world),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    args.warmup = max(3, args.warmup)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        run_reference(args, rank, world)
        return

    import torch
    torch.cuda.set_device(local_rank)
    dist = None
    if world > 1:
        import torch.distributed as dist_mod
        dist_mod.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
        dist = dist_mod
    import paged_kv_cache_gb300 as pa
    from paged_kv_cache_gb300 import workloads as W
    pa.load_library()
    peaks, peak_src = load_peaks()
    flush = L2Flush(torch)

    roofline = decode = e2e = other_variant = rope_q = None
    value = total_s = None
    step = None
    clk = {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["not sampled"]}
    clocks = ClockSampler(local_rank)
    clocks.start()
    if args.only in ("all", "prefill"):
        # ------------------------------------------------------ main step
        step = PrefillStep(torch, pa, W, args.variant, batch=args.batch, seqlen=args.seqlen)
        step_s, pre_s = timed(torch, lambda ev: step.run(ev=ev), args.steps, args.warmup, flush, dist)
        torch.cuda.synchronize()
        err = int(step.err.item())
        if err != 0:
            raise SystemExit("device error during the timed steps: %s" % pa.pa_status_string(err))
        rate, total_s, _ = job_rate(torch, dist, step.flops * args.steps, float(np.sum(step_s)))
        value = rate / 1e12
        prefill_avg = float(np.mean(pre_s))
        achieved = step.flops_prefill / prefill_avg / 1e12
        bf16_peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
        roofline = {"bound": "tensor", "achieved": achieved, "peak": bf16_peak, "unit": "TFLOP/s",
                    "frac": achieved / bf16_peak, "traffic": profiled_traffic("prefill_" + args.variant),
                    "kernel": "prefill_kernel<%d, %d>" % (step.geom.head_dim, prefill_heads_per_cta(step.geom)),
                    "peak_source": "%s bf16_tflops (burst)" % peak_src,
                    "algorithmic_flops_per_launch": step.flops_prefill,
                    "avg_launch_ms": prefill_avg * 1e3}
        # the same prefill with RoPE on the queries in the kernel's prologue (K turned by the scatter)
        rstep = RopePrefillStep(torch, pa, W, step)
        rsteps = max(20, args.steps // 4)
        _, rk_s = timed(torch, lambda ev: rstep.run(ev=ev), rsteps, args.warmup, flush, dist)
        torch.cuda.synchronize()
        if int(step.err.item()) != 0:
            raise SystemExit("device error during the RoPE-Q steps: %s" % pa.pa_status_string(int(step.err.item())))
        r_avg = float(np.mean(rk_s))
        r_ach = rstep.flops / r_avg / 1e12
        rope_q = {"metric": "causal prefill TFLOP/s with RoPE on the queries in the prologue (pa_prefill_rope; "
                            "K turned by pa_write_kv_rope), same workload and FLOPs as the main prefill",
                  "value": r_ach, "unit": "TFLOP/s", "steps": rsteps,
                  "prologue_cost": r_avg / prefill_avg - 1.0,
                  "roofline": {"bound": "tensor", "achieved": r_ach, "peak": bf16_peak, "unit": "TFLOP/s",
                               "frac": r_ach / bf16_peak,
                               "kernel": "prefill_kernel<%d, %d, rope>" % (step.geom.head_dim,
                                                                           prefill_heads_per_cta(step.geom)),
                               "peak_source": "%s bf16_tflops (burst)" % peak_src,
                               "algorithmic_flops_per_launch": rstep.flops, "avg_launch_ms": r_avg * 1e3}}
        del rstep
        # the other head-dim variant of the same long prefill (32 q / 8 kv heads at d 64,
        # 16 / 4 at d 128; the same FLOPs), the same step, reported beside the main one
        other = "d128" if args.variant == "d64" else "d64"
        ostep = PrefillStep(torch, pa, W, other, batch=args.batch, seqlen=args.seqlen)
        osteps = max(20, args.steps // 4)
        ostep_s, opre_s = timed(torch, lambda ev: ostep.run(ev=ev), osteps, args.warmup, flush, dist)
        torch.cuda.synchronize()
        if int(ostep.err.item()) != 0:
            raise SystemExit("device error during the %s steps: %s" % (other, pa.pa_status_string(int(ostep.err.item()))))
        o_avg = float(np.mean(opre_s))
        o_ach = ostep.flops_prefill / o_avg / 1e12
        o_rate, o_total, _ = job_rate(torch, dist, ostep.flops * osteps, float(np.sum(ostep_s)))
        other_variant = {
            "metric": "causal prefill TFLOP/s, %s variant (%d q / %d kv heads), same step" % (
                other, ostep.geom.num_q_heads, ostep.geom.num_kv_heads),
            "value": o_rate / 1e12, "unit": "TFLOP/s", "ms_per_step": o_total / osteps * 1e3, "steps": osteps,
            "roofline": {"bound": "tensor", "achieved": o_ach, "peak": bf16_peak, "unit": "TFLOP/s",
                         "frac": o_ach / bf16_peak, "traffic": profiled_traffic("prefill_" + other),
                         "kernel": "prefill_kernel<%d, %d>" % (ostep.geom.head_dim, prefill_heads_per_cta(ostep.geom)),
                         "peak_source": "%s bf16_tflops (burst)" % peak_src,
                         "algorithmic_flops_per_launch": ostep.flops_prefill, "avg_launch_ms": o_avg * 1e3}}
        del ostep

    llama = None
    if args.only in ("all", "llama"):
        # ------------- Llama-3.2-1B-shaped prompts (17 and 512 tokens), layers 0 and 15
        lstep = LlamaPromptStep(torch, pa, W)
        lsteps = max(20, args.steps)
        l_s, lk_s = timed(torch, lambda ev: lstep.run(ev=ev), lsteps, args.warmup, flush, dist)
        torch.cuda.synchronize()
        if int(lstep.err.item()) != 0:
            raise SystemExit("device error in the Llama prompt steps: %s" % pa.pa_status_string(int(lstep.err.item())))
        l_avg = float(np.mean(lk_s))
        bf16_peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
        l_rate, l_total, _ = job_rate(torch, dist, lstep.flops * lsteps, float(np.sum(lk_s)))
        llama = {"metric": "causal prefill TFLOP/s of the Llama-3.2-1B-shaped prompts (17 and 512 tokens, "
                           "32 q / 8 kv heads, d 64; K/V scattered at layers 0 and 15, prefill at 15); "
                           "latency-bound, not the long-prefill bar",
                 "value": l_rate / 1e12, "unit": "TFLOP/s", "steps": lsteps,
                 "step_ms": float(np.mean(l_s)) * 1e3,
                 "roofline": {"bound": "tensor", "achieved": lstep.flops / l_avg / 1e12, "peak": bf16_peak,
                              "unit": "TFLOP/s", "frac": lstep.flops / l_avg / 1e12 / bf16_peak,
                              "kernel": "prefill_kernel<64, 4>", "peak_source": "%s bf16_tflops (burst)" % peak_src,
                              "algorithmic_flops_per_launch": lstep.flops, "avg_launch_ms": l_avg * 1e3}}
        llama_case = lstep.case
        del lstep

    if args.only in ("all", "decode"):
        # ------------------- decode (256 sequences, log-normal lengths)
        dstep = DecodeStep(torch, pa, W)
        dsteps = args.decode_steps or max(20, args.steps)
        dstep_s, dk_s = timed(torch, lambda ev: dstep.run(ev=ev), dsteps, args.warmup, flush, dist)
        torch.cuda.synchronize()
        if int(dstep.err.item()) != 0:
            raise SystemExit("device error in decode steps: %s" % pa.pa_status_string(int(dstep.err.item())))
        dec_avg = float(np.mean(dk_s))
        hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
        dec_gbs = dstep.kv_bytes / dec_avg / 1e9
        d_rate, d_total, _ = job_rate(torch, dist, dstep.kv_bytes * dsteps, float(np.sum(dstep_s)))
        decode = {"metric": "decode KV-read GB/s (256 seqs, log-normal lengths, write + decode per step)",
                  "value": d_rate / 1e9, "unit": "GB/s", "ms_per_step": d_total / dsteps * 1e3,
                  "kv_bytes_per_step": dstep.kv_bytes, "steps": dsteps,
                  "roofline": {"bound": "hbm", "achieved": dec_gbs, "peak": hbm_peak, "unit": "GB/s",
                               "frac": dec_gbs / hbm_peak, "traffic": profiled_traffic("decode_256seq"),
                               "kernel": "decode_attend_kernel<64> + decode_merge_kernel<64>",
                               "peak_source": "%s hbm_gbs" % peak_src,
                               "algorithmic_bytes_per_launch": dstep.kv_bytes,
                               "avg_launch_ms": dec_avg * 1e3}}
        del dstep
        # the 64-sequence batch, lengths uniform in [128, 2048]: 143 MB of K/V per step
        sstep = DecodeStep(torch, pa, W, small=True)
        s_s, sk_s = timed(torch, lambda ev: sstep.run(ev=ev), dsteps, args.warmup, flush, dist)
        torch.cuda.synchronize()
        if int(sstep.err.item()) != 0:
            raise SystemExit("device error in decode steps: %s" % pa.pa_status_string(int(sstep.err.item())))
        s_avg = float(np.mean(sk_s))
        s_gbs = sstep.kv_bytes / s_avg / 1e9
        s_rate, s_total, _ = job_rate(torch, dist, sstep.kv_bytes * dsteps, float(np.sum(s_s)))
        decode["batch64"] = {"metric": "decode KV-read GB/s (64 seqs, lengths uniform in [128, 2048], "
                                       "write + decode per step)",
                             "value": s_rate / 1e9, "unit": "GB/s", "ms_per_step": s_total / dsteps * 1e3,
                             "kv_bytes_per_step": sstep.kv_bytes, "steps": dsteps,
                             "roofline": {"bound": "hbm", "achieved": s_gbs, "peak": hbm_peak, "unit": "GB/s",
                                          "frac": s_gbs / hbm_peak, "traffic": profiled_traffic("decode_64seq"),
                                          "kernel": "decode_attend_kernel<64> + decode_merge_kernel<64>",
                                          "peak_source": "%s hbm_gbs" % peak_src,
                                          "algorithmic_bytes_per_launch": sstep.kv_bytes,
                                          "avg_launch_ms": s_avg * 1e3}}
        del sstep

    chunked = None
    if args.only in ("all", "chunked"):
        # ------------------------------- prefill of chunks over a cached prefix
        cstep = ChunkedStep(torch, pa, W)
        csteps = max(20, args.steps // 2)
        cstep_s, ck_s = timed(torch, lambda ev: cstep.run(ev=ev), csteps, args.warmup, flush, dist)
        torch.cuda.synchronize()
        if int(cstep.err.item()) != 0:
            raise SystemExit("device error in chunked steps: %s" % pa.pa_status_string(int(cstep.err.item())))
        c_avg = float(np.mean(ck_s))
        c_rate, c_total, _ = job_rate(torch, dist, cstep.flops * csteps, float(np.sum(cstep_s)))
        bf16_peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
        c_ach = cstep.flops / c_avg / 1e12
        chunked = {"metric": "chunked prefill TFLOP/s (4 x 2048-query chunks after 6144 cached tokens, "
                             "exact causal count, step incl. the chunks' KV write)",
                   "value": c_rate / 1e12, "unit": "TFLOP/s", "ms_per_step": c_total / csteps * 1e3,
                   "steps": csteps,
                   "roofline": {"bound": "tensor", "achieved": c_ach, "peak": bf16_peak, "unit": "TFLOP/s",
                                "frac": c_ach / bf16_peak, "traffic": profiled_traffic("chunked_d64"),
                                "kernel": "prefill_kernel<64, 4> (prefix)",
                                "peak_source": "%s bf16_tflops (burst)" % peak_src,
                                "algorithmic_flops_per_launch": cstep.flops, "avg_launch_ms": c_avg * 1e3}}
        del cstep

    scatter = None
    if args.only in ("all", "scatter"):
        # ------------------------------------------------- K/V scatter (a1, f2)
        sstep = ScatterStep(torch, pa, W)
        hbm_peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
        scatter = {"metric": "K/V scatter GB/s (4 x 8192 prompt rows of 2 x 512 bf16 into shuffled pages)"}
        for name, rope, nbytes in (("write_kv", False, sstep.bytes_plain), ("write_kv_rope", True, sstep.bytes_rope)):
            ssteps = max(20, args.steps // 2)
            s_s, sk_s = timed(torch, lambda ev: sstep.run(rope, ev=ev), ssteps, args.warmup, flush, dist)
            torch.cuda.synchronize()
            if int(sstep.err.item()) != 0:
                raise SystemExit("device error in scatter steps: %s" % pa.pa_status_string(int(sstep.err.item())))
            s_avg = float(np.mean(sk_s))
            s_rate, _, _ = job_rate(torch, dist, nbytes * ssteps, float(np.sum(sk_s)))
            scatter[name] = {"value": s_rate / 1e9, "unit": "GB/s",
                             "roofline": {"bound": "hbm", "achieved": nbytes / s_avg / 1e9, "peak": hbm_peak,
                                          "unit": "GB/s", "frac": nbytes / s_avg / 1e9 / hbm_peak,
                                          "traffic": profiled_traffic("scatter_" + name),
                                          "kernel": "write_kv_rope_kernel" if rope else "write_kv_kernel",
                                          "peak_source": "%s hbm_gbs" % peak_src,
                                          "algorithmic_bytes_per_launch": nbytes, "avg_launch_ms": s_avg * 1e3}}
        del sstep

    backward = None
    if args.only in ("all", "backward"):
        # ----------------------------------------- FA2 backward over the pages (f4)
        bf16_peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
        for heads in ((32, 8, 64), (16, 4, 128)):
            hq, hkv, hd = heads
            bstep = BackwardStep(torch, pa, W, batch=args.batch, seqlen=args.seqlen, heads=heads)
            bsteps = max(10, args.steps // 4)
            b_s, bk_s = timed(torch, lambda ev: bstep.run(ev=ev), bsteps, args.warmup, flush, dist)
            torch.cuda.synchronize()
            if int(bstep.err.item()) != 0:
                raise SystemExit("device error in backward steps: %s" % pa.pa_status_string(int(bstep.err.item())))
            b_avg = float(np.mean(bk_s))
            b_rate, b_total, _ = job_rate(torch, dist, bstep.flops * bsteps, float(np.sum(b_s)))
            b_ach = bstep.flops / b_avg / 1e12
            leg = {"metric": "prefill backward TFLOP/s (%d x %d tokens, %d q / %d kv heads, d %d; "
                             "exact causal count x 2.5)" % (args.batch, args.seqlen, hq, hkv, hd),
                   "value": b_rate / 1e12, "unit": "TFLOP/s", "ms_per_step": b_total / bsteps * 1e3,
                   "steps": bsteps,
                   "roofline": {"bound": "tensor", "achieved": b_ach, "peak": bf16_peak, "unit": "TFLOP/s",
                                "frac": b_ach / bf16_peak, "traffic": profiled_traffic("backward_d%d" % hd),
                                "kernel": "bwd_prep_kernel<%d> + bwd_tc_kernel<%d>" % (hd, hd),
                                "peak_source": "%s bf16_tflops (burst)" % peak_src,
                                "algorithmic_flops_per_launch": bstep.flops, "avg_launch_ms": b_avg * 1e3}}
            if backward is None:
                backward = leg
            else:
                backward["d%d" % hd] = leg
            del bstep

    pages = None
    if args.only in ("all", "pages"):
        # ----------------------------------- page lifetime on the device (f3)
        pages = page_lifetime_timing(torch, pa, W, args.warmup)
    clk = clocks.stop()

    if step is not None and not args.no_e2e:
        # ------------------------------------------------------------ e2e
        e2e = e2e_timing(torch, step, max(10, args.steps // 4), args.warmup, flush, dist)

    # ------------------------------------------------------- CPU oracle
    cpu = None  # the oracle is timed on rank 0 of a single-GPU run only
    if rank == 0 and world == 1 and step is not None and not args.no_cpu_baseline:
        flops, wall, threads, desc = oracle_sample(step.case, args.cpu_seconds)
        cpu = {"value": flops / wall / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
               "sample": desc, "seconds": wall}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        side = max(2.0, args.cpu_seconds / 4)
        if decode is not None:
            for leg, lens, seed in ((decode, W.lognormal_decode_lens(), 1104),
                                    (decode["batch64"], W.uniform_decode_lens(), 1102)):
                nbytes, wall, threads, desc = oracle_decode_sample(lens, side, "decode", seed)
                leg["cpu_baseline"] = {"value": nbytes / wall / 1e9, "unit": "GB/s", "cores": threads,
                                       "kind": "oracle", "sample": desc, "seconds": wall}
        if llama is not None:
            flops, wall, threads, desc = oracle_llama_sample(llama_case, side)
            llama["cpu_baseline"] = {"value": flops / wall / 1e12, "unit": "TFLOP/s", "cores": threads,
                                     "kind": "oracle", "sample": desc, "seconds": wall}

    if rank == 0 and step is None:
        print(json.dumps({"metric": "%s only (profiling aid)" % args.only, "llama_prompts": llama, "decode": decode,
                          "chunked": chunked,
                          "scatter": scatter, "pages": pages, "backward": backward, "clocks": clk}), flush=True)
    elif rank == 0:
        line = {
            "metric": METRIC,
            "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": total_s / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) bf16, shuffled pages)",
            "config": step_config(step.geom, step.case.batch, step.n, world),
            "gpu_launches": step.launches * args.steps,
            "roofline": roofline,
            "prefill_" + ("d128" if args.variant == "d64" else "d64"): other_variant,
            "prefill_rope_q": rope_q,
            "decode": decode,
            "chunked": chunked,
            "scatter": scatter,
            "pages": pages,
            "backward": backward,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "clocks": clk,
            "kernel_source": kernel_source_hash(),
        }
        # the bars, compactly, at the very end of the line: each row's fraction
        # of its measured peak beside the bar it is held to
        gates = {"prefill_bar": 0.55, "decode_bar": 0.75,
                 "prefill_" + args.variant: round(roofline["frac"], 4)}
        if other_variant is not None:
            gates["prefill_" + ("d128" if args.variant == "d64" else "d64")] = round(
                other_variant["roofline"]["frac"], 4)
        if decode is not None:
            gates["decode_256seq"] = round(decode["roofline"]["frac"], 4)
            gates["decode_64seq"] = round(decode["batch64"]["roofline"]["frac"], 4)
        line["llama_prompts"] = llama
        line["gates"] = gates
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

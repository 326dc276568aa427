"""Benchmark of the paged KV cache hot path on GB300.

A step is one decode iteration of the decode-GQA workload (pool
16384x32x16x8x128 bf16, layer 7, 32 query heads, batch 64, seq_len
U[1024, 8192]): each of the 64 new tokens' K/V rows goes to its slot (the
table lookup of position seq_len - 1) and paged decode attention runs over
every sequence, in one fused pass over the pool (pkv_decode_step), followed
by the split-K combine.  `value` is the KV bytes the attention reads per step
(sum of seq_len x 2 x row bytes) divided by the step time, in GB/s.  The
gather and scatter bandwidths are measured on the gather/scatter workload
(pool 16384x32x16x8x128 bf16, 32 sequences, seq_len U[512, 4096]) and
reported under "legs".

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun each rank runs an independent replica on its own GPU (no
collective on the data path); rank 0 prints one JSON line.  `--impl
reference` times the CPU oracle on a bounded sample of the same workload.
"""

from __future__ import annotations

import os

# The oracle baseline runs single-threaded; set before numpy is imported.
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse
import hashlib
import json
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from workloads import make_workload, fill_pool, new_pool, rand_rows, to_numpy_bits  # noqa: E402

METRIC = "paged decode-attn KV-read GB/s & % of HBM peak; gather/scatter GB/s"
WORKLOAD = "decode_gqa"
LEG_WORKLOAD = "gather_scatter"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 512 << 20


# ---------------------------------------------------------------------------
# small helpers (also exercised by the CPU tests)
# ---------------------------------------------------------------------------

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def reduce_max(x: float) -> float:
    """Max over ranks (identity without torch.distributed)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return x
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def aggregate(units_per_rank: float, world: int, ms_max: float) -> float:
    """Whole-job throughput: the units all ranks processed over the slowest
    rank's time (units per second)."""
    return units_per_rank * world / (ms_max / 1e3)


def decode_bytes(batch, row_bytes: int, hq: int, head_dim: int, elem: int, bs: int) -> dict:
    """Algorithmic bytes of one decode call: K and V rows read once per token,
    the query and output rows, and the block-table entries and per-sequence
    scalars read."""
    lens = batch.seq_lens.astype(np.int64)
    offs = batch.offsets.astype(np.int64)
    nblk = np.where(lens > 0, -(-(offs + lens) // bs), 0)
    kv = int(lens.sum()) * 2 * row_bytes
    qo = 2 * batch.batch * hq * head_dim * elem
    tables = int(nblk.sum()) * 4 + batch.batch * 8
    return {"kv": kv, "total": kv + qo + tables}


def unique_kv_bytes(batch, row_bytes: int, bs: int, num_blocks: int) -> int:
    """K and V bytes of the distinct pool rows a decode call reads: a row that
    several sequences cover (a shared prefix block, or a block id that repeats
    across tables) counts once."""
    covered = np.zeros((num_blocks, bs), dtype=bool)
    for b in range(batch.batch):
        n = int(batch.seq_lens[b])
        if n <= 0:
            continue
        p = int(batch.offsets[b]) + np.arange(n, dtype=np.int64)
        covered[batch.block_tables[b, p // bs], p % bs] = True
    return int(covered.sum()) * 2 * row_bytes


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash() -> str:
    src = os.path.join(ROOT, "paged_kv_cache_blk_gb300", "csrc", "decode.cu")
    with open(src, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def recorded_traffic(name: str = "decode_partial_traffic.txt"):
    """DRAM bytes per launch of a decode partial kernel from a committed ncu
    summary, only if it was taken on the current kernel source."""
    p = os.path.join(ROOT, "profiles", name)
    d = {}
    try:
        with open(p) as f:
            for line in f:
                if line.startswith("#") or ":" not in line:
                    continue
                k, v = line.split(":", 1)
                d[k.strip()] = v.strip()
    except OSError:
        return None
    if d.get("decode_cu_sha256_16") != kernel_source_hash():
        return None
    try:
        return int(d["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi sampled every 200 ms around the timed region.  Samples are
    time-stamped so the summary keeps only those taken while the GPU was
    loaded (from the pre-load steps before the region to its end)."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []  # (time, line)
        self.window = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.t.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, line in self.lines:
            if self.window and not (self.window[0] <= ts <= self.window[1]):
                continue
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def preload(fn, clocks: "ClockSampler", min_s: float = 0.6, max_s: float = 5.0):
    """Untimed steps until the clock sampler has samples under load."""
    t0 = time.time()
    n0 = len(clocks.lines)
    while time.time() - t0 < max_s:
        for _ in range(20):
            fn()
        torch.cuda.synchronize()
        if time.time() - t0 >= min_s and (clocks.proc is None or len(clocks.lines) >= n0 + 2):
            break
    return t0


# ---------------------------------------------------------------------------
# the CUDA path
# ---------------------------------------------------------------------------

class DecodeStep:
    """Device state of one decode-GQA replica and its step.  With ``quant``
    the pool is an int8 pool of the same geometry (token rows of codes plus
    one fp32 scale per kv head) and the scatter quantises the new rows."""

    def __init__(self, dev, seed_shift: int, quant: bool = False):
        import paged_kv_cache_blk_gb300 as pkv
        from workloads import fill_pool_i8
        from workloads.gen import PoolSpec
        self.pkv = pkv
        w = make_workload(WORKLOAD)
        self.w = w
        self.dev = dev
        sp = w.pool
        if quant:
            spec = PoolSpec(sp.num_blocks, sp.num_layers, sp.block_size, sp.num_kv_heads,
                            sp.head_dim, "i8")
            k = torch.empty(spec.shape, dtype=torch.uint8, device=dev)
            v = torch.empty_like(k)
            fill_pool_i8(k, v, spec, w.layer, w.seed + seed_shift)
            self.pool = pkv.Pool(k, v, spec.num_kv_heads, spec.head_dim)
        else:
            spec = sp
            k, v = new_pool(sp, dev)
            fill_pool(k, v, sp, w.layer, w.seed + seed_shift)
            self.pool = pkv.Pool(k, v)
        self.spec = spec
        t = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a)).to(dev, dt)
        b = w.batch
        self.host = {
            "bt": torch.from_numpy(b.block_tables).pin_memory(),
            "lens": torch.from_numpy(b.seq_lens).pin_memory(),
            "offs": torch.from_numpy(b.offsets).pin_memory(),
            "seq": torch.from_numpy(w.tokens.token_seq).pin_memory(),
            "pos": torch.from_numpy(w.tokens.token_pos).pin_memory(),
        }
        self.bt, self.lens, self.offs = (t(b.block_tables, torch.int32),
                                         t(b.seq_lens, torch.int32), t(b.offsets, torch.int32))
        self.seq = t(w.tokens.token_seq, torch.int32)
        self.pos = t(w.tokens.token_pos, torch.int32)
        B, hq, D = b.batch, w.num_q_heads, w.pool.head_dim
        T = w.tokens.num_tokens
        row = (w.pool.num_kv_heads, D)
        self.q = rand_rows((B, hq, D), "bf16", 1000 + seed_shift, dev)
        self.k_new = rand_rows((T,) + row, "bf16", 1001 + seed_shift, dev)
        self.v_new = rand_rows((T,) + row, "bf16", 1002 + seed_shift, dev)
        self.out = torch.empty_like(self.q)
        self.slots = torch.empty(T, dtype=torch.int64, device=dev)
        self.ws = torch.empty(pkv.decode_workspace_size(B, hq, D, dev), dtype=torch.uint8,
                              device=dev)
        for name in ("q", "k_new", "v_new"):
            self.host[name] = getattr(self, name).cpu().pin_memory()
        self.host_out = torch.empty(self.out.shape, dtype=self.out.dtype).pin_memory()
        self.bytes = decode_bytes(b, spec.row_bytes, hq, D, 2, spec.block_size)
        self.quant = quant
        # one fused decode step (new rows stored, quantised for int8, and the
        # attention) + the split-K combine
        self.launches_per_step = 2
        self._INPUTS = ("bt", "lens", "offs", "q", "k_new", "v_new")
        self._pack_inputs()

    def step(self):
        # the new token of sequence b (row b of k_new / v_new) is stored at its
        # slot (position seq_len - 1; quantised for an int8 pool) and attended
        # to, in one pass
        self.pkv.decode_step(self.pool, self.w.layer, self.q, self.w.scale, self.bt, self.lens,
                             self.offs, self.k_new, self.v_new, self.out, self.ws)

    def _pack_inputs(self):
        """Lay every input of the step out in one page-locked host arena and
        one device arena (each input 256-byte aligned), and make the device
        inputs views of the device arena, so that a step's host->device
        traffic is one copy instead of eight small ones."""
        offs, total = {}, 0
        for name in self._INPUTS:
            offs[name] = total
            nb = self.host[name].numel() * self.host[name].element_size()
            total += (nb + 255) // 256 * 256
        self.host_arena = torch.zeros(total, dtype=torch.uint8).pin_memory()
        self.dev_arena = torch.zeros(total, dtype=torch.uint8, device=self.dev)
        for name in self._INPUTS:
            h = self.host[name]
            nb = h.numel() * h.element_size()
            hv = self.host_arena[offs[name]:offs[name] + nb].view(h.dtype).view(h.shape)
            hv.copy_(h)
            self.host[name] = hv
            d = getattr(self, name)
            dv = self.dev_arena[offs[name]:offs[name] + nb].view(d.dtype).view(d.shape)
            dv.copy_(d)
            setattr(self, name, dv)

    def step_e2e(self):
        """The same step from pinned host buffers: every input of the step is
        copied host->device (one copy of the packed input arena) and the
        attention output device->host."""
        self.dev_arena.copy_(self.host_arena, non_blocking=True)
        self.step()
        self.host_out.copy_(self.out, non_blocking=True)

    def e2e_bytes(self):
        return (self.host_arena.numel(),
                self.host_out.numel() * self.host_out.element_size())

    def e2e_pipelined(self, steps: int) -> float:
        """Mean ms per step of `steps` end-to-end steps run as a serving loop
        runs them: step k+1's inputs are copied host->device (into the second
        of two device input arenas) on a copy stream while step k computes,
        and step k's output is read back device->host on a third stream while
        step k+1 computes.  Every step still moves its own inputs and output;
        one pair of events spans the first copy to the last read-back.  The
        K/V a step reads (1.27 GB) is ten times L2, so no flush runs between
        the steps.  Checks that the last output read back equals the device
        result bit for bit."""
        pkv = self.pkv
        comp = torch.cuda.current_stream(self.dev)
        cp, rb = torch.cuda.Stream(self.dev), torch.cuda.Stream(self.dev)
        if not hasattr(self, "_pipe"):
            arena2 = torch.empty_like(self.dev_arena)
            views = []
            for arena in (self.dev_arena, arena2):
                v = {}
                for name in self._INPUTS:
                    d = getattr(self, name)
                    o = d.data_ptr() - self.dev_arena.data_ptr()
                    nb = d.numel() * d.element_size()
                    v[name] = arena[o:o + nb].view(d.dtype).view(d.shape)
                views.append(v)
            outs = [self.out, torch.empty_like(self.out)]
            host_outs = [self.host_out, torch.empty_like(self.host_out).pin_memory()]
            self._pipe = ((self.dev_arena, arena2), views, outs, host_outs)
        arenas, views, outs, host_outs = self._pipe
        ev = lambda: torch.cuda.Event(enable_timing=False)
        h2d = [ev() for _ in range(steps)]
        done = [ev() for _ in range(steps)]
        d2h = [ev() for _ in range(steps)]
        t0, t1 = (torch.cuda.Event(enable_timing=True) for _ in range(2))
        torch.cuda.synchronize(self.dev)
        t0.record(comp)
        cp.wait_event(t0)
        for k in range(steps):
            a = k & 1
            with torch.cuda.stream(cp):
                if k >= 2:
                    cp.wait_event(done[k - 2])  # step k-2 has read arena a
                arenas[a].copy_(self.host_arena, non_blocking=True)
                h2d[k].record(cp)
            comp.wait_event(h2d[k])
            if k >= 2:
                comp.wait_event(d2h[k - 2])  # output a has been read back
            v = views[a]
            pkv.decode_step(self.pool, self.w.layer, v["q"], self.w.scale, v["bt"], v["lens"],
                            v["offs"], v["k_new"], v["v_new"], outs[a], self.ws)
            done[k].record(comp)
            with torch.cuda.stream(rb):
                rb.wait_event(done[k])
                host_outs[a].copy_(outs[a], non_blocking=True)
                d2h[k].record(rb)
        comp.wait_event(d2h[steps - 1])
        t1.record(comp)
        torch.cuda.synchronize(self.dev)
        last = (steps - 1) & 1
        if not torch.equal(host_outs[last], outs[last].cpu()):
            raise RuntimeError("pipelined end-to-end step: read-back output differs")
        return t0.elapsed_time(t1) / steps


class L2Flush:
    """Between timed steps: write a buffer larger than L2 (evicting whatever
    the step left there), then read a second one so that the dirty lines of
    that write are written back before the next step starts instead of
    during it.  Both run outside the step's events."""

    def __init__(self, dev, nbytes: int = L2_FLUSH_BYTES):
        self.w = torch.empty(nbytes // 4, dtype=torch.float32, device=dev)
        self.r = torch.ones(nbytes // 4, dtype=torch.float32, device=dev)
        self.sink = torch.empty(1, dtype=torch.float32, device=dev)

    def zero_(self):
        self.w.zero_()
        torch.sum(self.r, 0, keepdim=True, out=self.sink)


class NoFlush:
    """Stand-in for L2Flush when a figure is taken with L2 left as it is."""

    def zero_(self):
        pass


def timed(fn, steps: int, flush, events_hook=None):
    """Per-step device times (ms) with CUDA events on the current stream and
    an L2 flush between steps outside the events."""
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    inner = []
    for i in range(steps):
        flush.zero_()
        if events_hook is not None:
            inner.append(events_hook())
        starts[i].record()
        fn()
        ends[i].record()
    torch.cuda.synchronize()
    times = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    return times, inner


def step_breakdown(st: "DecodeStep", flush: torch.Tensor, steps: int) -> dict:
    """Eager per-call device times (events between the calls): the fused
    decode step, and for comparison the same work as two calls (append the
    new rows, then decode attention)."""
    pkv = st.pkv
    names = ("decode_step", "append_tokens", "decode_attention")
    acc = {n: 0.0 for n in names}
    for _ in range(steps):
        flush.zero_()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        ev[0].record()
        pkv.decode_step(st.pool, st.w.layer, st.q, st.w.scale, st.bt, st.lens, st.offs,
                        st.k_new, st.v_new, st.out, st.ws)
        ev[1].record()
        flush.zero_()
        ev[2].record()
        pkv.append_tokens(st.pool, st.w.layer, st.bt, st.offs, st.seq, st.pos, st.k_new,
                          st.v_new, st.slots)
        ev3 = torch.cuda.Event(enable_timing=True)
        ev3.record()
        pkv.decode_attention(st.pool, st.w.layer, st.q, st.w.scale, st.bt, st.lens, st.offs,
                             st.out, st.ws)
        ev[3].record()
        torch.cuda.synchronize()
        acc["decode_step"] += ev[0].elapsed_time(ev[1])
        acc["append_tokens"] += ev[2].elapsed_time(ev3)
        acc["decode_attention"] += ev3.elapsed_time(ev[3])
    out = {n: round(v / steps, 4) for n, v in acc.items()}
    return {"decode_step": out["decode_step"],
            "unfused": {"append_tokens": out["append_tokens"],
                        "decode_attention": out["decode_attention"]}}


def run_ours(args, rank, local_rank, world):
    import paged_kv_cache_blk_gb300 as pkv
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    pkv.build()
    pkv.load()
    pkv.set_validate(False)
    pkv.set_decode_ctas(0)
    flush = L2Flush(dev)

    st = DecodeStep(dev, seed_shift=rank)
    for _ in range(args.warmup):
        st.step()
    torch.cuda.synchronize()

    # decode partial-kernel events, recorded by the library on its stream
    def hook():
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(); e1.record()
        pkv.set_decode_events(e0, e1)
        return e0, e1

    clocks = ClockSampler(dev.index).start()
    t_load = preload(st.step, clocks)
    barrier()
    torch.cuda.synchronize()
    times, kev = timed(st.step, args.steps, flush, hook)
    pkv.set_decode_events(None, None)
    torch.cuda.synchronize()
    t_end = time.time()
    time.sleep(0.25)
    clocks.stop()
    clocks.window = (t_load, t_end + 0.25)
    barrier()
    eager_ms = reduce_max(statistics.mean(times))
    part_ms = statistics.mean(a.elapsed_time(b) for a, b in kev)

    # the same step replayed from a CUDA graph (how a serving loop runs its
    # decode step): no host launch gaps between the step's kernels
    graph_ms = None
    timing = None
    if not args.no_graph:
        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.stream(side):
            st.step()
        torch.cuda.current_stream(dev).wait_stream(side)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            st.step()
        for _ in range(args.warmup):
            graph.replay()
        torch.cuda.synchronize()
        barrier()
        gtimes, _ = timed(graph.replay, args.steps, flush)
        barrier()
        graph_ms = reduce_max(statistics.mean(gtimes))
        # the same replays with no L2 flush between them (the inputs exceed L2,
        # so this differs from the flushed figure only by what stays cached)
        htimes, _ = timed(graph.replay, args.steps, NoFlush())
        timing = {"flushed_ms": {"mean": round(statistics.mean(gtimes), 4),
                                 "median": round(statistics.median(gtimes), 4),
                                 "min": round(min(gtimes), 4)},
                  "hot_ms": {"mean": round(statistics.mean(htimes), 4),
                             "median": round(statistics.median(htimes), 4),
                             "min": round(min(htimes), 4)}}
        del graph
    ms_max = graph_ms if graph_ms is not None else eager_ms
    kv = st.bytes["kv"]
    value_gbs = aggregate(kv, world, ms_max) / 1e9
    tokens_s = aggregate(st.w.batch.batch, world, ms_max)

    # end to end from pinned host buffers
    for _ in range(max(1, args.warmup // 2)):
        st.step_e2e()
    torch.cuda.synchronize()
    barrier()
    e2e_times, _ = timed(st.step_e2e, args.steps, flush)
    barrier()
    e2e_serial_ms = reduce_max(statistics.mean(e2e_times))
    # the same steps pipelined as a serving loop runs them (copies overlap compute)
    st.e2e_pipelined(max(3, args.warmup))
    barrier()
    e2e_ms = reduce_max(st.e2e_pipelined(args.steps))
    barrier()
    h2d, d2h = st.e2e_bytes()

    launches = st.launches_per_step * args.steps
    breakdown = step_breakdown(st, flush, max(10, args.steps // 4))

    # gather / scatter legs on their own workload
    legs = run_legs(args, dev, rank, flush, pkv)
    del st
    torch.cuda.empty_cache()

    peak, peak_kind = load_peaks()
    w = make_workload(WORKLOAD)
    db = decode_bytes(w.batch, w.pool.row_bytes, w.num_q_heads, w.pool.head_dim,
                      w.pool.elem_size, w.pool.block_size)
    # the fused step's partial pass also reads each sequence's new K/V row
    # (k_new, v_new) and stores it to the pool: 4 rows per sequence
    step_bytes = db["total"] + 4 * w.batch.batch * w.pool.row_bytes
    achieved = step_bytes / (part_ms / 1e3) / 1e9
    traffic = recorded_traffic()
    # block ids repeat across the decode-GQA tables: the distinct rows read
    uniq = unique_kv_bytes(w.batch, w.pool.row_bytes, w.pool.block_size, w.pool.num_blocks)
    uniq_step = step_bytes - db["kv"] + uniq
    result = {
        "metric": METRIC,
        "value": round(value_gbs, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_max, 4),
        "step_mode": "cuda_graph" if graph_ms is not None else "eager",
        "eager_ms_per_step": round(eager_ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": bench_config(w, kv, world),
        "hbm_pct_of_peak": {"measured": round(100 * value_gbs / world / peak, 1),
                            "nominal_8000": round(100 * value_gbs / world / NOMINAL_HBM_GBS, 1),
                            "peak_kind": peak_kind},
        "tokens_per_s": round(tokens_s, 1),
        "roofline": {
            "kernel": "decode_partial_kernel<bf16,128,4,fused step>",
            "bound": "hbm",
            "achieved": round(achieved, 1),
            "peak": peak,
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": traffic,
            "algorithmic_bytes_per_launch": step_bytes,
            "avg_launch_ms": round(part_ms, 4),
            "peak_source": f"MEASURED_PEAKS.json hbm_gbs ({peak_kind})",
            "unique_bytes_per_launch": uniq_step,
            "frac_unique": round(uniq_step / (part_ms / 1e3) / 1e9 / peak, 4),
            "frac_dram": (None if traffic is None
                          else round(traffic / (part_ms / 1e3) / 1e9 / peak, 4)),
        },
        "step_timing": timing,
        "step_breakdown_ms": breakdown,
        "legs": legs,
        "e2e": {"value": round(aggregate(kv, world, e2e_ms) / 1e9, 1), "unit": "GB/s",
                "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "mode": "pipelined: step k+1's inputs copied host->device (second device "
                        "arena) and step k's output read back on two copy streams while step "
                        "k computes; one event span over all steps; no L2 flush inside it "
                        "(each step reads 1.27 GB of K/V)",
                "serial": {"value": round(aggregate(kv, world, e2e_serial_ms) / 1e9, 1),
                           "ms_per_step": round(e2e_serial_ms, 4),
                           "mode": "copy in, step, copy out in order on one stream, per-step "
                                   "events, L2 flushed between steps"}},
        "gpu_launches": launches,
        "clocks": clocks.summary(),
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(args.cpu_seconds, seed_shift=0, dev=dev)
    result["legs_detail"] = result.pop("legs")
    result["legs"] = compact_legs(result["legs_detail"], peak)
    return result


def decode_events_hook(pkv):
    """Events the library records around the decode partial kernel."""
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(); e1.record()
    pkv.set_decode_events(e0, e1)
    return e0, e1


def graph_step_ms(step, steps: int, warmup: int, flush, dev) -> float:
    """Mean device time of `step` replayed from a CUDA graph."""
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream(dev).wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for _ in range(warmup):
        graph.replay()
    torch.cuda.synchronize()
    times, _ = timed(graph.replay, steps, flush)
    del graph
    return statistics.mean(times)


def int8_leg(args, dev, rank, flush, pkv) -> dict:
    """The decode step of the decode-GQA workload over an int8 pool of the
    same geometry: the 64 new bf16 rows quantised into their slots and decode
    attention, in one fused pass (pkv_decode_step), then the combine.  Step
    time from a CUDA graph, the partial kernel alone from the library's
    events, and its roofline over the int8 bytes."""
    st = DecodeStep(dev, seed_shift=rank, quant=True)
    for _ in range(args.warmup):
        st.step()
    torch.cuda.synchronize()
    times, kev = timed(st.step, args.steps, flush, lambda: decode_events_hook(pkv))
    pkv.set_decode_events(None, None)
    eager_ms = reduce_max(statistics.mean(times))
    part_ms = statistics.mean(a.elapsed_time(b) for a, b in kev)
    graph_ms = None if args.no_graph else reduce_max(
        graph_step_ms(st.step, args.steps, args.warmup, flush, dev))
    ms = graph_ms if graph_ms is not None else eager_ms
    peak, kind = load_peaks()
    db = st.bytes
    # the fused partial pass also reads each sequence's new bf16 K/V rows and
    # stores their int8 rows
    sp = st.spec
    part_bytes = db["total"] + st.w.batch.batch * (2 * sp.num_kv_heads * sp.head_dim * 2
                                                   + 2 * sp.row_bytes)
    out = {
        "what": "decode_gqa step over an int8 pool 16384x32x16x(8x128 codes + 8 fp32 scales) "
                "(1056-byte token rows): the 64 new tokens' bf16 K/V quantised into their "
                "slots and paged decode attention in one fused pass (pkv_decode_step), then "
                "the combine (bf16 q / out)",
        "ms_per_step": round(ms, 4),
        "step_mode": "cuda_graph" if graph_ms is not None else "eager",
        "eager_ms_per_step": round(eager_ms, 4),
        "kv_read_bytes_per_step": db["kv"],
        "GB/s": round(db["kv"] / (ms / 1e3) / 1e9, 1),
        "tokens_per_s": round(st.w.batch.batch / (ms / 1e3), 1),
        "decode_partial": {
            "kernel": "decode_partial_kernel<int8,128,4,fused step>",
            "avg_launch_ms": round(part_ms, 4),
            "algorithmic_bytes_per_launch": part_bytes,
            "achieved_GBps": round(part_bytes / (part_ms / 1e3) / 1e9, 1),
            "frac": round(part_bytes / (part_ms / 1e3) / 1e9 / peak, 4),
            "peak": peak, "peak_kind": kind,
            "traffic": recorded_traffic("decode_partial_i8_traffic.txt"),
        },
    }
    del st
    torch.cuda.empty_cache()
    return out


def run_legs(args, dev, rank, flush, pkv):
    w = make_workload(LEG_WORKLOAD)
    k, v = new_pool(w.pool, dev)
    fill_pool(k, v, w.pool, w.layer, w.seed + rank)
    pool = pkv.Pool(k, v)
    b = w.batch
    t = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a)).to(dev, dt)
    bt, lens, offs, cu = (t(b.block_tables, torch.int32), t(b.seq_lens, torch.int32),
                          t(b.offsets, torch.int32), t(b.cu_seqlens, torch.int64))
    seq, pos = t(w.tokens.token_seq, torch.int32), t(w.tokens.token_pos, torch.int32)
    T = w.tokens.num_tokens
    row = (w.pool.num_kv_heads, w.pool.head_dim)
    k_new = rand_rows((T,) + row, "bf16", 2000 + rank, dev)
    v_new = rand_rows((T,) + row, "bf16", 2001 + rank, dev)
    slots = torch.empty(T, dtype=torch.int64, device=dev)
    pkv.build_slot_mapping(pool, bt, offs, seq, pos, slots)
    ko = torch.empty((b.total_tokens,) + row, dtype=torch.bfloat16, device=dev)
    vo = torch.empty_like(ko)
    scatter = lambda: pkv.write_slots(pool, w.layer, k_new, v_new, slots)
    gather = lambda: pkv.gather(pool, w.layer, bt, lens, offs, cu, ko, vo)
    for _ in range(args.warmup):
        scatter(); gather()
    torch.cuda.synchronize()
    rb = w.pool.row_bytes
    s_bytes = T * 4 * rb + T * 8
    nblk = int((b.block_tables >= 0).sum())
    g_bytes = b.total_tokens * 4 * rb + nblk * 4 + b.batch * 12
    out = {}
    for name, fn, nbytes in (("scatter", scatter, s_bytes), ("gather", gather, g_bytes)):
        times, _ = timed(fn, args.steps, flush)
        ms = reduce_max(statistics.mean(times))
        out[name] = {"GB/s": round(nbytes / (ms / 1e3) / 1e9, 1), "ms": round(ms, 4),
                     "algorithmic_bytes": nbytes, "tokens": T if name == "scatter" else
                     b.total_tokens,
                     "workload": "gather_scatter: pool 16384x32x16x8x128 bf16 layer 0, 32 "
                                 "seqs U[512,4096]"}
    # whole-block moves on the same pool: copy-on-write copies (all layers of
    # 512 block pairs) and swap out / in of 256 blocks to page-locked host memory
    rng = np.random.default_rng(7 + rank)
    perm = rng.permutation(w.pool.num_blocks).astype(np.int32)
    src = torch.from_numpy(perm[:512]).to(dev)
    dst = torch.from_numpy(perm[512:1024]).to(dev)
    blk_bytes = w.pool.num_layers * w.pool.block_size * rb            # one block, all layers
    copy = lambda: pkv.copy_blocks(pool, -1, src, dst)
    sw = torch.from_numpy(perm[1024:1280]).to(dev)
    hk = torch.empty((256,) + tuple(k.shape[1:]), dtype=k.dtype, pin_memory=True)
    hv = torch.empty_like(hk, pin_memory=True)
    swap_out = lambda: pkv.swap_out(pool, -1, sw, hk, hv)
    swap_in = lambda: pkv.swap_in(pool, -1, sw, hk, hv)
    # the same bytes through torch's own page-locked copy, as the link reference
    dk = torch.empty_like(hk, device=dev)
    d2h = lambda: hk.copy_(dk, non_blocking=True)
    h2d = lambda: dk.copy_(hk, non_blocking=True)
    for _ in range(args.warmup):
        copy(); swap_out(); swap_in(); d2h(); h2d()
    torch.cuda.synchronize()
    for name, fn, nbytes, note in (
            ("copy_blocks", copy, 512 * blk_bytes * 2 * 2, "512 block pairs, all 32 layers, K+V "
                                                           "(read + write)"),
            ("swap_out", swap_out, 256 * blk_bytes * 2, "256 blocks, all layers, K+V to "
                                                        "page-locked host"),
            ("swap_in", swap_in, 256 * blk_bytes * 2, "256 blocks, all layers, K+V from "
                                                      "page-locked host"),
            ("torch_d2h_same_bytes", d2h, 256 * blk_bytes, "reference: torch copy of one "
                                                           "256-block buffer to pinned host"),
            ("torch_h2d_same_bytes", h2d, 256 * blk_bytes, "reference: the reverse")):
        times, _ = timed(fn, max(5, args.steps // 10), flush)
        ms = reduce_max(statistics.mean(times))
        out[name] = {"GB/s": round(nbytes / (ms / 1e3) / 1e9, 1), "ms": round(ms, 4),
                     "bytes": nbytes, "what": note}
    del pool, k, v, ko, vo, hk, hv, dk
    torch.cuda.empty_cache()
    out["allocator"] = allocator_leg()
    out["prefill"] = prefill_leg(args, dev, flush, pkv)
    out["int8_decode"] = int8_leg(args, dev, rank, flush, pkv)
    for name in ("long_splitk", "prefix_mix"):
        out["decode_" + name] = decode_leg(name, args, dev, flush, pkv, min(args.steps, 100))
    # the prefix-mix batch through shared-prefix decode: its 64 shared blocks
    # read once (pkv_decode_attention_shared_prefix)
    out["decode_prefix_mix_shared"] = decode_leg("prefix_mix", args, dev, flush, pkv,
                                                 min(args.steps, 100), prefix_blocks=64)
    return out


def compact_legs(legs: dict, peak: float) -> dict:
    """The legs' headline figures in a few short keys: printed last on the
    JSON line so that a tail of the output keeps them."""
    f = lambda x: None if x is None else round(x, 4)
    c = {}
    for name in ("scatter", "gather", "copy_blocks", "swap_out", "swap_in"):
        if name in legs:
            c[name + "_GBps"] = legs[name]["GB/s"]
    for name in ("scatter", "gather", "copy_blocks"):
        if name in legs:
            c[name + "_frac"] = f(legs[name]["GB/s"] / peak)
    for name in ("long_splitk", "prefix_mix", "prefix_mix_shared"):
        d = legs.get("decode_" + name)
        if d:
            c["decode_" + name] = {k: d[k] for k in ("partial_frac", "call_kv_frac",
                                                     "call_unique_frac", "partial_dram_frac",
                                                     "call_kv_GBps", "call_unique_GBps")}
    i8 = legs.get("int8_decode")
    if i8:
        c["int8_step"] = {"ms": i8["ms_per_step"], "tokens_per_s": i8["tokens_per_s"],
                          "partial_frac": i8["decode_partial"]["frac"]}
    pf = legs.get("prefill")
    if pf:
        c["prefill"] = {k: {"TFLOPs": pf[k]["TFLOP/s"], "frac": pf[k]["frac_of_bf16_peak"]}
                        for k in ("prompts", "chunk")}
    al = legs.get("allocator")
    if al:
        c["allocator_ops_per_s"] = al["lib_ops_per_s"]
    return c


def prefill_case(dev, kind: str, seed: int = 0):
    """Prefill workloads on the decode-GQA head geometry (Hkv 8, Hq 32, D 128,
    bf16, block 16) over a 1-layer pool: 'prompts' = 16 prompts of 2048 tokens,
    all of them queries; 'chunk' = 16 sequences of 4096 tokens whose last 512
    are the queries (chunked prefill after a cached prefix)."""
    from workloads.gen import FreeList, PoolSpec, _pack
    B, L, nq = (16, 2048, 2048) if kind == "prompts" else (16, 4096, 512)
    bs, Hkv, G, D = 16, 8, 4, 128
    spec = PoolSpec(B * L // bs + 64, 1, bs, Hkv, D, "bf16")
    rng = np.random.default_rng(seed)
    free = FreeList(rng.permutation(spec.num_blocks))
    batch = _pack([free.pop(L // bs) for _ in range(B)], [L] * B, [0] * B)
    cu = np.arange(B + 1, dtype=np.int64) * nq
    k, v = new_pool(spec, dev)
    fill_pool(k, v, spec, 0, seed)
    q = rand_rows((B * nq, Hkv * G, D), "bf16", seed + 9, dev)
    # algorithmic flops: 2 matmuls x 2 flops per (query, attended key, head, d)
    keys = sum((L - nq + i + 1) for i in range(nq)) * B
    flops = 4 * D * Hkv * G * keys
    return spec, batch, cu, nq, k, v, q, flops


def prefill_leg(args, dev, flush, pkv):
    out = {}
    for kind in ("prompts", "chunk"):
        spec, batch, cu, nq, k, v, q, flops = prefill_case(dev, kind)
        pool = pkv.Pool(k, v)
        t = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a)).to(dev, dt)
        bt, lens, offs, cuq = (t(batch.block_tables, torch.int32), t(batch.seq_lens, torch.int32),
                               t(batch.offsets, torch.int32), t(cu, torch.int64))
        o = torch.empty_like(q)
        fn = lambda: pkv.prefill_attention(pool, 0, q, 128 ** -0.5, bt, lens, offs, cuq, nq, o)
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        times, _ = timed(fn, max(10, args.steps // 10), flush)
        ms = reduce_max(statistics.mean(times))
        out[kind] = {"TFLOP/s": round(flops / (ms / 1e3) / 1e12, 1), "ms": round(ms, 4),
                     "flops": flops, "queries": int(cu[-1]),
                     "what": ("16 prompts x 2048 tokens, causal, Hq 32 / Hkv 8, D 128, bf16"
                              if kind == "prompts" else
                              "16 x (3584 cached + 512 new) tokens, causal, Hq 32 / Hkv 8")}
        del pool, k, v, q, o
        torch.cuda.empty_cache()
    peaks = {}
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        peaks = {"bf16_tflops": d["bf16_tflops"], "kind": "measured"}
    except Exception:
        peaks = {"bf16_tflops": 1900.0, "kind": "fallback"}
    for kind in ("prompts", "chunk"):
        out[kind]["frac_of_bf16_peak"] = round(out[kind]["TFLOP/s"] / peaks["bf16_tflops"], 4)
    out["peak"] = peaks
    return out


def allocator_trace(num_blocks: int, bs: int, seed: int):
    """A serving-shaped operation trace for the block allocator: requests
    arrive with prompts U[16, 2048], some hit the prefix of a live request
    (shared blocks) or fork it, every live request appends one token per
    decode step (copy-on-write where shared), and the oldest leave."""
    rng = np.random.default_rng(seed)
    ops = []
    live, nid = [], 0
    for step in range(400):
        if len(live) < 48 or rng.random() < 0.3:
            sid = nid
            nid += 1
            if live and rng.random() < 0.3:
                ops.append(("fork", int(rng.choice(live)), sid))
            else:
                ops.append(("new", sid, int(rng.integers(0, bs))))
                ops.append(("append", sid, int(rng.integers(16, 2049))))
            live.append(sid)
        for sid in live:
            ops.append(("append", sid, 1))
        if len(live) > 64:
            ops.append(("free", live.pop(0), 0))
    return ops


def _run_trace(ops, m):
    """Replay a trace; the decode appends of a step go in one batched call.
    Returns the number of sequence operations performed."""
    n = 0
    step = []

    def flush_step():
        nonlocal n
        if step:
            try:
                m.seq_append_batch(step)
            except Exception:
                pass
            n += len(step)
            step.clear()

    for op, a, b in ops:
        if op == "append" and b == 1:
            step.append(a)
            continue
        flush_step()
        try:
            if op == "new":
                m.seq_new(a, b)
            elif op == "append":
                m.seq_append(a, b)
            elif op == "fork":
                m.seq_fork(a, b)
            else:
                m.seq_free(a)
        except Exception:
            pass
        n += 1
    flush_step()
    return n


def allocator_leg():
    import paged_kv_cache_blk_gb300 as pkv
    from oracle import allocator as OA
    N, bs = 16384, 16
    ops = allocator_trace(N, bs, 11)
    t0 = time.perf_counter()
    n = _run_trace(ops, pkv.Allocator(N, bs))
    lib_s = time.perf_counter() - t0
    t0 = time.perf_counter()
    _run_trace(ops, OA.KVCacheManager(N, bs))
    ora_s = time.perf_counter() - t0
    return {"ops": n, "lib_ops_per_s": round(n / lib_s, 1), "oracle_ops_per_s": round(n / ora_s, 1),
            "lib_us_per_decode_step": round(lib_s / 400 * 1e6, 2),
            "trace": "16384 blocks of 16; 400 decode steps of <=64 live requests (one batched "
                     "append per step), prompts U[16,2048], 30% forks; through the Python binding"}


# ---------------------------------------------------------------------------
# the CPU oracle (baseline leg and the reference arm)
# ---------------------------------------------------------------------------

def _oracle_inputs(dev=None, seed_shift=0):
    """Layer 7 of the decode-GQA pool and the queries, as oracle arrays."""
    w = make_workload(WORKLOAD)
    spec = w.pool
    d = dev if dev is not None else torch.device("cpu")
    from workloads.gen import PoolSpec
    one = PoolSpec(spec.num_blocks, 1, spec.block_size, spec.num_kv_heads, spec.head_dim,
                   spec.dtype)
    k, v = new_pool(one, d)
    fill_pool(k, v, one, 0, w.seed + seed_shift)
    q = rand_rows((w.batch.batch, w.num_q_heads, spec.head_dim), "bf16", 1000 + seed_shift, d)
    return w, to_numpy_bits(k), to_numpy_bits(v), to_numpy_bits(q)


def _oracle_sample(w, kh, vh, qh, seqs):
    import oracle
    b = w.batch
    t0 = time.perf_counter()
    oracle.decode_attention(kh, vh, 0, qh[seqs], b.block_tables[seqs], b.seq_lens[seqs],
                            b.offsets[seqs], w.scale)
    dt = time.perf_counter() - t0
    kv = int(b.seq_lens[seqs].astype(np.int64).sum()) * 2 * w.pool.row_bytes
    return kv, dt


def _cpu_worker(job):
    """One oracle worker (a spawned process): attach to the shared pool layer
    and queries, then run the oracle over its sequences (every n-th one,
    cycling) for `seconds`.  Returns (K/V bytes, wall start, wall end,
    sequences done)."""
    from multiprocessing import shared_memory
    names, shapes, seconds, first, stride = job
    shms = [shared_memory.SharedMemory(name=n) for n in names]
    try:
        kh, vh, qh = (np.ndarray(sh, dtype=np.uint16, buffer=m.buf) for sh, m in zip(shapes, shms))
        w = make_workload(WORKLOAD)
        B = w.batch.batch
        kv_total, n = 0, 0
        t0 = time.time()
        while time.time() - t0 < seconds:
            kv, _ = _oracle_sample(w, kh, vh, qh, [(first + n * stride) % B])
            kv_total += kv
            n += 1
        t1 = time.time()
        del kh, vh, qh
        return kv_total, t0, t1, n
    finally:
        for m in shms:
            m.close()


def _cpu_all_cores(kh, vh, qh, seconds: float):
    """The oracle on every host core this process may use: one spawned
    worker per core over shared copies of the inputs.  Throughput is all
    workers' K/V bytes over the span from the first start to the last end."""
    import multiprocessing as mp
    from multiprocessing import shared_memory
    cores = len(os.sched_getaffinity(0))
    shms, shapes = [], []
    try:
        for a in (kh, vh, qh):
            m = shared_memory.SharedMemory(create=True, size=a.nbytes)
            np.ndarray(a.shape, dtype=a.dtype, buffer=m.buf)[...] = a
            shms.append(m)
            shapes.append(a.shape)
        jobs = [([m.name for m in shms], shapes, seconds, i, cores) for i in range(cores)]
        # spawned (never forked after CUDA started); a worker that dies raises
        # here instead of leaving the pool waiting
        from concurrent.futures import ProcessPoolExecutor
        with ProcessPoolExecutor(cores, mp_context=mp.get_context("spawn")) as ex:
            futs = [ex.submit(_cpu_worker, j) for j in jobs]
            res = [f.result(timeout=seconds + 300) for f in futs]
    finally:
        for m in shms:
            m.close()
            m.unlink()
    kv = sum(r[0] for r in res)
    span = max(r[2] for r in res) - min(r[1] for r in res)
    return kv / span / 1e9, cores, sum(r[3] for r in res), span, kv


def cpu_baseline(seconds: float, seed_shift=0, dev=None):
    w, kh, vh, qh = _oracle_inputs(dev, seed_shift)
    kv_total, t_total, n = 0, 0.0, 0
    B = w.batch.batch
    while t_total < seconds and n < 16 * B:
        kv, dt = _oracle_sample(w, kh, vh, qh, [n % B])
        kv_total += kv
        t_total += dt
        n += 1
    single = kv_total / t_total / 1e9
    out = {"value": round(single, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
           "sample": f"oracle.decode_attention (numpy, fp64, per-block gather) over {n} "
                     f"decode_gqa sequences taken in order, cycling over the 64 "
                     f"({kv_total / 1e6:.0f} MB of K/V), {t_total:.1f} s, single thread"}
    try:
        value, cores, seqs, span, kv = _cpu_all_cores(kh, vh, qh, seconds)
    except Exception as e:  # no shared memory or no process pool on this host
        out["all_cores_unavailable"] = f"{type(e).__name__}: {e}"
        return out
    out.update({
        "value": round(value, 4), "cores": cores,
        "single_thread": {"value": round(single, 4), "sample": out["sample"]},
        "sample": f"oracle.decode_attention (numpy, fp64) in {cores} spawned processes, one per "
                  f"host core, each cycling over its share of the 64 decode_gqa sequences: "
                  f"{seqs} sequences ({kv / 1e6:.0f} MB of K/V) in {span:.1f} s",
    })
    return out


def bench_config(w, kv: int, world: int) -> dict:
    """The workload description both arms print."""
    return {
        "workload": "decode_gqa: pool 16384x32x16x8x128 bf16 (layer 7), Hq 32 (GQA 4), "
                    "batch 64, seq_len U[1024,8192], random non-contiguous tables; step = "
                    "the 64 new tokens' K/V stored at their slots and paged decode attention "
                    "in one fused pass (pkv_decode_step), then the split-K combine",
        "batch": int(w.batch.batch),
        "kv_read_bytes_per_step": int(kv),
        "l2": "flushed between steps outside the events (512 MiB write, then a 512 MiB read "
              "that retires its dirty lines); inputs (1.27 GB/step) also exceed L2",
        "parallelism": f"replicas x{world}",
    }


def run_reference(args, rank, world):
    if rank != 0:
        return None
    w, kh, vh, qh = _oracle_inputs(None, 0)
    per_step = 2  # sequences per step: a bounded sample (a few seconds of CPU work)
    for i in range(args.warmup):
        _oracle_sample(w, kh, vh, qh, [i % 64])
    kv_total, t_total = 0, 0.0
    times = []
    for i in range(args.steps):
        seqs = [(i * per_step + j) % 64 for j in range(per_step)]
        kv, dt = _oracle_sample(w, kh, vh, qh, seqs)
        kv_total += kv
        t_total += dt
        times.append(dt * 1e3)
    value = kv_total / t_total / 1e9
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 4),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(statistics.mean(times), 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": bench_config(w, w.batch.seq_lens.astype(np.int64).sum() * 2 * w.pool.row_bytes,
                               world),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"the oracle on {per_step} decode_gqa sequences per step "
                                   f"(cycling over the 64), {args.steps} steps, one host "
                                   f"thread"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def decode_leg(name: str, args, dev, flush, pkv, steps: int, prefix_blocks: int = 0) -> dict:
    """Paged decode attention (pkv_decode_attention) on one bf16 decode
    workload: the partial-pass kernel alone (events the library records
    around it) and the whole call (partial + combine), with the L2 flush
    between calls.  Throughput on the algorithmic bytes (every sequence's
    rows counted), on the distinct rows read, and on the DRAM bytes of the
    committed ncu capture of the same kernel source."""
    w = make_workload(name)
    k, v = new_pool(w.pool, dev)
    fill_pool(k, v, w.pool, w.layer, w.seed, w.k_boost_frac, w.k_boost)
    pool = pkv.Pool(k, v)
    b = w.batch
    t = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a)).to(dev, dt)
    bt, lens, offs = (t(b.block_tables, torch.int32), t(b.seq_lens, torch.int32),
                      t(b.offsets, torch.int32))
    q = rand_rows((b.batch, w.num_q_heads, w.pool.head_dim), "bf16", 5, dev)
    out = torch.empty_like(q)
    ws = torch.empty(pkv.decode_workspace_size(b.batch, w.num_q_heads, w.pool.head_dim, dev),
                     dtype=torch.uint8, device=dev)
    call = lambda: pkv.decode_attention(pool, w.layer, q, w.scale, bt, lens, offs, out, ws)
    if prefix_blocks:
        # shared-prefix decode: the library records the events around its
        # suffix pass, which then stands for the "partial" figures
        ws = torch.empty(pkv.decode_shared_prefix_workspace_size(pool, b.batch, w.num_q_heads,
                                                                 prefix_blocks),
                         dtype=torch.uint8, device=dev)
        call = lambda: pkv.decode_attention_shared_prefix(pool, w.layer, q, w.scale, bt, lens,
                                                          offs, prefix_blocks, out, ws)
    for _ in range(args.warmup):
        call()
    torch.cuda.synchronize()
    # the partial pass alone from the library's events; the whole call
    # without them (an event between the launches would end their overlap)
    _, kev = timed(call, steps, flush, lambda: decode_events_hook(pkv))
    pkv.set_decode_events(None, None)
    part_ms = statistics.mean(a.elapsed_time(e) for a, e in kev)
    times, _ = timed(call, steps, flush)
    call_ms = reduce_max(statistics.mean(times))
    peak, kind = load_peaks()
    db = decode_bytes(b, w.pool.row_bytes, w.num_q_heads, w.pool.head_dim, w.pool.elem_size,
                      w.pool.block_size)
    uniq = unique_kv_bytes(b, w.pool.row_bytes, w.pool.block_size, w.pool.num_blocks)
    part_bytes = db["total"]
    if prefix_blocks:
        # the partial pass is the suffix pass: the rows after the shared
        # prefix, the queries, the states and table entries it reads
        tot = b.offsets.astype(np.int64) + b.seq_lens.astype(np.int64)
        suffix_rows = np.maximum(0, tot - prefix_blocks * w.pool.block_size)
        part_bytes = db["total"] - db["kv"] + int(suffix_rows.sum()) * 2 * w.pool.row_bytes
    dram = recorded_traffic(f"decode_partial_{name}{'_shared' if prefix_blocks else ''}"
                            "_traffic.txt")
    gbs = lambda nbytes, ms: nbytes / (ms / 1e3) / 1e9
    entry = {
        "partial_ms": round(part_ms, 4), "call_ms": round(call_ms, 4),
        "kv_bytes": db["kv"], "unique_kv_bytes": uniq, "algorithmic_bytes": db["total"],
        "partial_bytes": part_bytes,
        "partial_GBps": round(gbs(part_bytes, part_ms), 1),
        "partial_frac": round(gbs(part_bytes, part_ms) / peak, 4),
        "call_kv_GBps": round(gbs(db["kv"], call_ms), 1),
        "call_kv_frac": round(gbs(db["kv"], call_ms) / peak, 4),
        "call_unique_GBps": round(gbs(uniq, call_ms), 1),
        "call_unique_frac": round(gbs(uniq, call_ms) / peak, 4),
        "dram_bytes": dram,
        "partial_dram_frac": None if dram is None else round(gbs(dram, part_ms) / peak, 4),
        "tokens_per_s": round(b.batch / (call_ms / 1e3), 1),
        "peak": peak, "peak_kind": kind,
    }
    del pool, k, v, ws
    torch.cuda.empty_cache()
    return entry


def decode_sweep(args) -> int:
    """Decode-attention throughput on every bf16 decode workload (not the
    bench line): partial-pass kernel alone and the whole decode call."""
    import paged_kv_cache_blk_gb300 as pkv
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    pkv.build()
    pkv.load()
    flush = L2Flush(dev)
    res = {name: decode_leg(name, args, dev, flush, pkv, args.steps)
           for name in ("decode_gqa", "long_splitk", "prefix_mix")}
    print(json.dumps({"decode_sweep": res}), flush=True)
    return 0


def ncu_case(kind: str, launches: int = 4) -> int:
    """A small-footprint run of one kernel for ncu: the decode-GQA batch
    (1.27 GB of K/V per launch, larger than L2) over a 1-layer copy of its
    pool (1 GB), the long split-K or prefix-mix decode batches over 1-layer
    copies of theirs (4.3 / 2.1 GB), or the gather/scatter legs over a
    1-layer pool.  Each launch reads the same bytes as on the full pool."""
    import paged_kv_cache_blk_gb300 as pkv
    from workloads.gen import PoolSpec
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    pkv.build()
    pkv.load()
    if kind == "prefill":
        spec, batch, cu, nq, k, v, q, flops = prefill_case(dev, "prompts")
        pool = pkv.Pool(k, v)
        t = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a)).to(dev, dt)
        bt, lens, offs, cuq = (t(batch.block_tables, torch.int32), t(batch.seq_lens, torch.int32),
                               t(batch.offsets, torch.int32), t(cu, torch.int64))
        o = torch.empty_like(q)
        for _ in range(launches):
            pkv.prefill_attention(pool, 0, q, 128 ** -0.5, bt, lens, offs, cuq, nq, o)
        torch.cuda.synchronize()
        print(f"ncu case prefill: {launches} launches done")
        return 0
    name = {"decode_long": "long_splitk", "decode_prefix": "prefix_mix",
            "decode_prefix_shared": "prefix_mix"}.get(
        kind, WORKLOAD if kind.startswith("decode") else LEG_WORKLOAD)
    w = make_workload(name)
    sp = w.pool
    if kind in ("decode_i8", "decode_step_i8"):
        from workloads import fill_pool_i8
        one = PoolSpec(sp.num_blocks, 1, sp.block_size, sp.num_kv_heads, sp.head_dim, "i8")
        k = torch.empty(one.shape, dtype=torch.uint8, device=dev)
        v = torch.empty_like(k)
        fill_pool_i8(k, v, one, 0, w.seed)
        pool = pkv.Pool(k, v, one.num_kv_heads, one.head_dim)
    else:
        one = PoolSpec(sp.num_blocks, 1, sp.block_size, sp.num_kv_heads, sp.head_dim, sp.dtype)
        k, v = new_pool(one, dev)
        fill_pool(k, v, one, 0, w.seed)
        pool = pkv.Pool(k, v)
    b = w.batch
    t = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a)).to(dev, dt)
    bt, lens, offs, cu = (t(b.block_tables, torch.int32), t(b.seq_lens, torch.int32),
                          t(b.offsets, torch.int32), t(b.cu_seqlens, torch.int64))
    row = (sp.num_kv_heads, sp.head_dim)
    if kind.startswith("decode"):
        q = rand_rows((b.batch, w.num_q_heads, sp.head_dim), "bf16", 1, dev)
        out = torch.empty_like(q)
        ws = torch.empty(pkv.decode_workspace_size(b.batch, w.num_q_heads, sp.head_dim, dev),
                         dtype=torch.uint8, device=dev)
        fn = lambda: pkv.decode_attention(pool, 0, q, w.scale, bt, lens, offs, out, ws)
        if kind == "decode_prefix_shared":
            ws = torch.empty(pkv.decode_shared_prefix_workspace_size(pool, b.batch, w.num_q_heads,
                                                                     64),
                             dtype=torch.uint8, device=dev)
            fn = lambda: pkv.decode_attention_shared_prefix(pool, 0, q, w.scale, bt, lens, offs,
                                                            64, out, ws)
        if kind in ("decode_step", "decode_step_i8"):
            kn = rand_rows((b.batch,) + row, "bf16", 2, dev)
            vn = rand_rows((b.batch,) + row, "bf16", 3, dev)
            fn = lambda: pkv.decode_step(pool, 0, q, w.scale, bt, lens, offs, kn, vn, out, ws)
    else:
        T = w.tokens.num_tokens
        slots = torch.empty(T, dtype=torch.int64, device=dev)
        pkv.build_slot_mapping(pool, bt, offs, t(w.tokens.token_seq, torch.int32),
                               t(w.tokens.token_pos, torch.int32), slots)
        kn = rand_rows((T,) + row, "bf16", 2, dev)
        vn = rand_rows((T,) + row, "bf16", 3, dev)
        ko = torch.empty((b.total_tokens,) + row, dtype=torch.bfloat16, device=dev)
        vo = torch.empty_like(ko)
        if kind == "scatter":
            fn = lambda: pkv.write_slots(pool, 0, kn, vn, slots)
        else:
            fn = lambda: pkv.gather(pool, 0, bt, lens, offs, cu, ko, vo)
    for _ in range(launches):
        fn()
    torch.cuda.synchronize()
    print(f"ncu case {kind}: {launches} launches done")
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-graph", action="store_true",
                    help="time the step from eager API calls only (no CUDA graph replay)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ncu-case", choices=["decode", "decode_step", "decode_i8", "decode_step_i8",
                                           "decode_long",
                                           "decode_prefix", "decode_prefix_shared",
                                           "gather", "scatter",
                                           "prefill"],
                    help="run a small-footprint case of one kernel (for ncu) and exit")
    ap.add_argument("--decode-sweep", action="store_true",
                    help="decode throughput on every decode workload (not the bench line)")
    args = ap.parse_args(argv)
    if args.ncu_case:
        return ncu_case(args.ncu_case)
    if args.decode_sweep:
        return decode_sweep(args)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank, local_rank, world = dist_env()
    if world != args.gpus and world > 1:
        ap.error(f"--gpus {args.gpus} but WORLD_SIZE {world}")
    if world > 1:
        import torch.distributed as dist
        if args.impl == "reference" and rank != 0:
            return 0
        if args.impl == "ours":
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            if backend == "nccl":
                torch.cuda.set_device(local_rank)
            dist.init_process_group(backend)
    if args.impl == "reference":
        res = run_reference(args, rank, world)
    else:
        res = run_ours(args, rank, local_rank, world)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())

"""Benchmark: decode-attention microseconds per decode step over the compressed BF16 paged KV cache,
with KV GB/s (compressed and effective-uncompressed), the fraction of the measured HBM peak, and
the same step on the dense-BF16 kernel.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step = one decode step of the workload: for every layer, zf_decode_attn over that layer's
compressed cache (the long-context workload also writes one new token per request into its tail
page through zf_append_tokens each step).  Inputs are resident in HBM; the per-step KV bytes exceed
L2, so the step needs no extra flush.  Prints one JSON line on rank 0: the headline workload's
step, and (default run, one GPU) a `per_config` object with every workload measured the same way
plus, for each, the median of single calls timed alone after an L2 flush, and a `multi_token`
object: several new tokens per request on three shapes, with the kernel the library picks, the
warp-MMA kernel and the dense comparator.  N > 1 runs N
independent replicas (one per GPU, weak scaling); the step time is the maximum over ranks.  Without
torchrun, --gpus N > 1 starts the N ranks itself.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")     # one BLAS thread per oracle worker process

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attn µs/step & KV GB/s (compressed, % of HBM peak) vs dense BF16 path"
DEFAULT_WORKLOAD = "llama7b_mha_8192"
SPEC_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 2 ** 20


def read_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# the sources the attention kernels are compiled from
KERNEL_SOURCES = ("zf_attn.cu", "zf_attn_common.cuh", "zf_device.cuh", "zf_host.h")


def kernel_source_hash() -> str:
    """Hash of the attention kernels' sources with comments and blank space removed: a committed
    ncu capture stays valid across comment-only edits and is dropped when their code changes."""
    import re
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "decode_attention_compressed_gb300", "csrc")
    for f in KERNEL_SOURCES:
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        text = " ".join(text.split())
        h.update(f.encode() + text.encode())
    return h.hexdigest()[:16]


def read_traffic(workload: str):
    """DRAM bytes per launch of the attention kernel from the committed ncu summary, if it was
    taken on the current kernel sources (same source hash); else None."""
    path = os.path.join(ROOT, "profiles", "attn_kernel_dram_traffic_by_workload.txt")
    if not os.path.exists(path):
        return None
    want = kernel_source_hash()
    for line in open(path):
        w = line.split()
        if len(w) >= 4 and not line.startswith("#") and w[0] == workload and w[3] == want:
            return float(w[2])
    return None


class ClockSampler:
    """SM clock and clock-event reasons sampled while the timed region runs: NVML (read-only
    queries through ctypes, about one sample per millisecond from a thread), else nvidia-smi."""

    # NVML clock-event reason bits
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.rows = []            # (sm_mhz, max_mhz, [reason names])
        self.nvml = None
        self.proc = None
        self.path = None

    def _nvml_open(self):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            return None
        h = ctypes.c_void_p()
        if lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.gpu), ctypes.byref(h)) != 0:
            return None
        mx = ctypes.c_uint()
        if lib.nvmlDeviceGetMaxClockInfo(h, ctypes.c_int(1), ctypes.byref(mx)) != 0:
            return None
        return lib, h, mx.value

    def _nvml_loop(self):
        import ctypes
        lib, h, mx = self.nvml
        clk, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self.stop.is_set():
            if lib.nvmlDeviceGetClockInfo(h, ctypes.c_int(1), ctypes.byref(clk)) == 0:
                names = []
                if lib.nvmlDeviceGetCurrentClocksEventReasons(h, ctypes.byref(rs)) == 0:
                    names = [n for bit, n in self.REASONS.items() if rs.value & bit]
                self.rows.append((float(clk.value), float(mx), names))
            time.sleep(0.001)

    def __enter__(self):
        try:
            self.nvml = self._nvml_open()
        except Exception:
            self.nvml = None
        if self.nvml is not None:
            import threading
            self.stop = threading.Event()
            self.thread = threading.Thread(target=self._nvml_loop, daemon=True)
            self.thread.start()
            return self
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.nvml is not None:
            self.stop.set()
            self.thread.join(timeout=5)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        rows = list(self.rows)
        source = "nvml"
        if self.nvml is None:
            source = "nvidia-smi"
            if self.proc is None or not self.path:
                return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}
            names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
            for line in open(self.path):
                w = [x.strip() for x in line.split(",")]
                if len(w) >= 9:
                    try:
                        rows.append((float(w[1]), float(w[2]),
                                     [n for n, v in zip(names, w[5:9]) if v.lower().startswith("active")]))
                    except ValueError:
                        pass
            os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0, "source": source}
        reasons = sorted({n for r in rows for n in r[2]})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows), "source": source}


# ------------------------------------------------------------------------------------ GPU arm
# Every workload the default run measures (one GPU): each is set up, timed and freed in turn.
PER_CONFIG = ("tiny", "llama7b_mha_512", "llama7b_mha_2048", "llama7b_mha_8192", "llama3_8b_batched",
              "qwen2_7b_maxbatch", "long_ctx", "batch64_gqa4_2048", "batch64_gqa4_8192")
# Several new tokens per request (speculative verification) in the default run: workload, tokens.
# Columns per kv head: 14, 28 and 32 (the last two need 4 warp-MMA passes, 1 tensor-memory pass).
MULTI_TOKEN = (("qwen2_7b_maxbatch", 2), ("qwen2_7b_maxbatch", 4), ("batch64_gqa4_8192", 8))
MIN_TIMED_MS = 200.0          # per-config timed regions last at least this long (enough clock samples)
ISOLATED_CALLS = 25           # single calls timed alone, each after an L2 flush
ISOLATED_WARMUP = 3


def tile_bytes(layer, dirs, compressed: bool, tokens: int = 1) -> int:
    """Algorithmic bytes one attention launch reads: per (request, kv head), every 16-token tile
    holding context tokens costs 6272 bytes (compressed page) or 8192 bytes (raw page), plus q,
    page table, seq_lens, out and lse (q, out and lse once per new token)."""
    import torch
    w = layer.workload
    P = w.page_size
    lens = layer.seq_lens.cpu().to(torch.int64)
    table = layer.page_table.cpu().to(torch.int64)
    total = 0
    for b in range(w.batch):
        L = int(lens[b])
        npg = -(-L // P)
        tiles = torch.clamp(L - torch.arange(npg) * P, max=P)
        tiles = (tiles + 15) // 16
        if compressed:
            raw = (dirs[table[b, :npg]] >= 0).to(torch.int64)          # [npg][Hkv]
            per = tiles[:, None] * torch.where(raw.bool(), 8192, 6272)
            total += int(per.sum())
        else:
            total += int(tiles.sum()) * 8192 * w.num_kv_heads
    total += tokens * w.batch * w.num_q_heads * 128 * 2 + table.numel() * 4 + w.batch * 4
    total += tokens * w.batch * w.num_q_heads * (128 * 4 + 4)
    return total


def dense_equiv_bytes(layer) -> int:
    """Bytes the same context occupies as dense BF16 (2 x 128 x 2 per token and kv head)."""
    w = layer.workload
    return int(layer.seq_lens.to("cpu").sum()) * w.num_kv_heads * 512


def setup_layers(zf, I, w, device, extra_pages=0):
    """Every layer of `w`: its inputs, its compressed cache and its dense cache (page i keeps id i
    and may fall back to raw slot i; extra_pages more ids and raw slots for appended pages)."""
    import torch
    layers = []
    for l in range(w.layers):
        layer = I.make_layer(w, layer=l, device=device)
        npg = layer.num_pages
        cache = zf.Cache(npg + extra_pages, w.num_kv_heads, w.page_size, npg + extra_pages, device=device)
        zf.encode_pages(cache, layer.k_pages, layer.v_pages, list(range(npg)), layer.n_valid, list(range(npg)))
        dense = zf.Cache(npg + extra_pages, w.num_kv_heads, w.page_size, npg + extra_pages, device=device,
                         compressed=False)
        zf.encode_pages(dense, layer.k_pages, layer.v_pages, list(range(npg)), layer.n_valid, list(range(npg)),
                        force_raw=True)
        torch.cuda.synchronize()
        if cache.status_word() or dense.status_word():
            raise RuntimeError("encode reported a device error")
        dirs = cache.dir.cpu()
        layer.k_pages = layer.v_pages = None          # the caches hold the data now
        layers.append(dict(layer=layer, cache=cache, dense=dense, dirs=dirs, num_pages=npg))
    return layers


def prefill_encode(zf, I, device, peak):
    """A full-prefill encode: 8192 tokens x 32 layers, 8 kv heads, 64-token pages (one
    zf_encode_pages call per layer, the 32 calls replayed as one CUDA graph), timed with CUDA
    events; bytes read (BF16 source) and written (compressed records and directory entries)."""
    import torch
    w = I.scaled(I.WORKLOADS["long_ctx"], batch=1, ctx=8192)
    layer = I.make_layer(w, device=device)
    npg = layer.num_pages
    caches = [zf.Cache(npg, w.num_kv_heads, w.page_size, 8, device=device) for _ in range(32)]
    ids = torch.arange(npg, dtype=torch.int32, device=device)
    nv = layer.n_valid.to(device)
    rs = torch.full((npg,), -1, dtype=torch.int32, device=device)

    def prefill():
        for c in caches:
            zf.encode_pages(c, layer.k_pages, layer.v_pages, ids, nv, rs)

    def time_ms(run, reps):
        for _ in range(3):
            run()
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for _ in range(reps):
            run()
        e.record()
        torch.cuda.synchronize()
        return s.elapsed_time(e) / reps

    # the 32 calls replayed as one CUDA graph (device time); eager calls from Python beside it
    g = capture(prefill)
    ms = time_ms(g.replay, 20)
    eager_ms = time_ms(prefill, 5)
    del g
    if any(c.status_word() for c in caches):
        raise RuntimeError("prefill encode reported a device error")
    read = 2 * layer.k_pages.numel() * 2 * 32
    written = sum(c.stored_bytes() for c in caches)
    gbs = (read + written) / (ms * 1e-3) / 1e9
    return {"ms": round(ms, 4), "eager_ms": round(eager_ms, 4), "launch_mode": "cuda_graph (32 zf_encode_pages calls)",
            "tokens": 8192, "layers": 32, "kv_heads": w.num_kv_heads, "page_size": w.page_size,
            "bytes_read": read, "bytes_written": written, "read_write_gbs": round(gbs, 1),
            "pct_of_hbm_peak": round(100 * gbs / peak, 1), "src_gbs": round(read / (ms * 1e-3) / 1e9, 1)}


def max_over_ranks(value: float, device) -> float:
    """The largest `value` over all ranks of the default process group."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_requests(batch: int, rank: int, world: int):
    """Requests a replica owns when a batch is sharded over ranks (contiguous, balanced)."""
    per, extra = divmod(batch, world)
    start = rank * per + min(rank, extra)
    return list(range(start, start + per + (1 if rank < extra else 0)))


def arm_config(w, tokens: int, kernel: str, world: int) -> dict:
    """The `config` object of a bench line, the same for this library's arm and the reference arm.
    The L2 note uses a lower bound on the KV bytes a step reads: every request's shortest possible
    context, all of it in compressed pages."""
    from decode_attention_compressed_gb300 import accounting as A
    min_bytes = w.batch * w.num_kv_heads * (w.ctx_min or w.ctx) * A.compressed_bytes_per_token_head() * w.layers
    if min_bytes > L2_BYTES:
        l2 = (f"no flush: every step reads at least {min_bytes / 1e9:.2f} GB of compressed KV "
              f"(> {L2_BYTES / 2**20:.0f} MiB L2)")
    else:
        l2 = f"no flush: a step reads from {min_bytes / 1e6:.1f} MB of KV, which may stay in the {L2_BYTES / 2**20:.0f} MiB L2"
    return {"workload": w.name, "note": w.note, "batch": w.batch, "q_heads": w.num_q_heads,
            "kv_heads": w.num_kv_heads, "head_dim": 128, "page_size": w.page_size, "ctx": w.ctx,
            "layers_per_step": w.layers, "new_tokens_per_request": tokens, "kernel": kernel,
            "parallelism": "replicas" if world > 1 else "single", "l2": l2}


def workload_of(args):
    from decode_attention_compressed_gb300 import inputs as I
    w = I.WORKLOADS[args.workload]
    kw = {}
    if args.layers is not None:
        kw["layers"] = min(args.layers, w.layers)
    if args.batch is not None:
        kw["batch"] = min(args.batch, w.batch)
    return I.scaled(w, **kw) if kw else w


def capture(fn):
    """fn() captured once into a CUDA graph (after one eager warm-up on a side stream)."""
    import torch
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


class Workbench:
    """One workload on one GPU: every layer's compressed and dense cache, queries, outputs and one
    workspace, and the decode step over them (CUDA graph, or eager for the long-context step whose
    appends change pointers every step)."""

    def __init__(self, zf, I, w, device, tokens=1, world=1, local_rank=0, max_steps=0, kernel="auto"):
        import torch
        self.zf, self.I, self.w, self.device, self.T = zf, I, w, device, tokens
        self.kernel = kernel            # compressed attention kernel: auto, warp_mma or tcgen05
        self.world, self.local_rank = world, local_rank
        if tokens > 1 and w.name == "long_ctx":
            raise SystemExit("--tokens > 1 is not combined with the long-context append step")
        extra = LongContextAppend.extra_pages(w, max_steps) if w.name == "long_ctx" else 0
        self.layers = setup_layers(zf, I, w, device, extra)
        T = tokens
        self.qs = [I.make_multi_queries(w, T, layer=i, device=device) if T > 1 else ent["layer"].q
                   for i, ent in enumerate(self.layers)]
        self.oshape = (w.batch, T, w.num_q_heads) if T > 1 else (w.batch, w.num_q_heads)
        self.outs = [(torch.empty(*self.oshape, 128, device=device), torch.empty(*self.oshape, device=device))
                     for _ in self.layers]
        self.append = None
        max_pages = int(self.layers[0]["layer"].page_table.shape[1])
        if w.name == "long_ctx":
            self.append = LongContextAppend(zf, I, w, self.layers[0], device, max_steps)
            max_pages = int(self.append.table.shape[1])
        ws_bytes = zf.workspace_size_multi(w.batch, T, w.num_q_heads, w.num_kv_heads, w.page_size, max_pages)
        self.workspace = zf.new_workspace(ws_bytes, device)
        self.graphs = {}

    # ---- the step
    def attn(self, cache, q, table, lens, scale, out, lse, dense=False):
        kernel = "auto" if dense else self.kernel
        if self.T > 1:
            self.zf.decode_attn_multi(cache, q, table, lens, scale, out=out, lse=lse, workspace=self.workspace,
                                      dense=dense, kernel=kernel)
        else:
            self.zf.decode_attn(cache, q, table, lens, scale, out=out, lse=lse, workspace=self.workspace,
                                dense=dense, kernel=kernel)

    def step(self, dense=False, events=None, reencode=False):
        if self.append is not None:
            self.append.step(dense, reencode)
        for i, ent in enumerate(self.layers):
            lay = ent["layer"]
            lens = self.append.lens if self.append is not None else lay.seq_lens
            table = self.append.table if self.append is not None else lay.page_table
            if events is not None:
                events[i][0].record()
            self.attn(ent["dense"] if dense else ent["cache"], self.qs[i], table, lens, lay.scale, self.outs[i][0],
                      self.outs[i][1], dense)
            if events is not None:
                events[i][1].record()

    def graph(self, key, fn):
        if key not in self.graphs:
            self.graphs[key] = capture(fn)
        return self.graphs[key].replay

    # ---- timing
    def timed(self, run, steps, warmup, per_call=False, min_ms=0.0, dense=False, reencode=False):
        """Device time per step of `run` over `steps` steps (CUDA events on the launching stream,
        max over ranks); with min_ms, more steps so the timed region lasts at least that long.
        Returns (ms per step, mean attention-call ms when per_call, clocks, steps timed)."""
        import torch
        import torch.distributed as dist
        if self.append is not None:
            self.append.reset()
        for _ in range(warmup):
            run()
        torch.cuda.synchronize()
        if min_ms > 0:
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record()
            for _ in range(3):
                run()
            e.record()
            torch.cuda.synchronize()
            steps = max(steps, math.ceil(min_ms / max(s.elapsed_time(e) / 3, 1e-3)))
            if self.append is not None:
                steps = min(steps, self.append.max_steps - warmup - 3)
        if self.append is not None:
            self.append.reset()
            for _ in range(warmup):
                run()
        torch.cuda.synchronize()
        if self.world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        events = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in self.layers] for _ in range(steps)] if per_call else None
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with ClockSampler(self.local_rank) as clk:
            s.record()
            for k in range(steps):
                if per_call:
                    self.step(dense, events[k], reencode)
                else:
                    run()
            e.record()
            torch.cuda.synchronize()
        if self.world > 1:
            dist.barrier()
        ms = s.elapsed_time(e)
        calls = [x.elapsed_time(y) for row in events for (x, y) in row] if per_call else None
        if self.world > 1:
            ms = max_over_ranks(ms, self.device)
        return ms / steps, (statistics.mean(calls) if calls else None), clk.summary(), steps

    def isolated_call_ms(self, dense=False, calls=ISOLATED_CALLS):
        """Median device time of one attention call (layer 0, static inputs) timed alone: before
        each call a plain fill kernel writes a buffer of twice the L2 size, so the call starts with
        none of its inputs in L2 and with no attention grid ahead of it to overlap with."""
        import torch
        ent = self.layers[0]
        lay = ent["layer"]
        flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=self.device)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(calls + ISOLATED_WARMUP)]
        for s, e in ev:
            flush.zero_()
            s.record()
            self.attn(ent["dense"] if dense else ent["cache"], self.qs[0], lay.page_table, lay.seq_lens, lay.scale,
                      self.outs[0][0], self.outs[0][1], dense)
            e.record()
        torch.cuda.synchronize()
        del flush
        return statistics.median(s.elapsed_time(e) for s, e in ev[ISOLATED_WARMUP:])

    def restore_ms(self, steps, warmup, min_ms=0.0):
        """Restore-then-attend (ZipFusion §II.B): each layer decompressed into one shared dense
        buffer (zf_decompress_to_raw), then the dense kernel; static inputs, one CUDA graph."""
        import torch
        zf, w = self.zf, self.w
        max_np = max(ent["num_pages"] for ent in self.layers)
        shared = zf.Cache(max_np, w.num_kv_heads, w.page_size, max_np, device=self.device, compressed=False)
        ids = [torch.arange(ent["num_pages"], dtype=torch.int32, device=self.device) for ent in self.layers]

        def restore_step():
            for i, ent in enumerate(self.layers):
                lay = ent["layer"]
                zf.decompress_to_raw(ent["cache"], ids[i], shared)
                self.attn(shared, self.qs[i], lay.page_table, lay.seq_lens, lay.scale, self.outs[i][0],
                          self.outs[i][1], dense=True)

        g = capture(restore_step)
        append, self.append = self.append, None
        try:
            ms, _, _, _ = self.timed(g.replay, steps, warmup, min_ms=min_ms)
        finally:
            self.append = append
        del g, shared
        return ms

    # ---- bytes
    def bytes(self):
        T = self.T
        layers = self.layers
        comp = sum(tile_bytes(ent["layer"], ent["dirs"], True, T) for ent in layers)
        dense = sum(tile_bytes(ent["layer"], ent["dirs"], False, T) for ent in layers)
        uncompressed = sum(dense_equiv_bytes(ent["layer"]) for ent in layers)
        stored = sum(ent["cache"].stored_bytes(ent["num_pages"]) for ent in layers)
        w = self.w
        dense_stored = sum(ent["num_pages"] * w.num_kv_heads * 2 * w.page_size * 128 * 2 for ent in layers)
        raw = sum(float((ent["dirs"][: ent["num_pages"]] >= 0).float().mean()) for ent in layers) / len(layers)
        return comp, dense, uncompressed, dense_stored / stored, raw

    def status(self):
        return [ent["cache"].status_word() | ent["dense"].status_word() for ent in self.layers]

    # ---- one entry of multi_token
    def multi_token_summary(self, steps, warmup, peak):
        """T new tokens per request: the step with the kernel ZF_KERNEL_AUTO picks, with the warp-MMA
        kernel named, and with the dense comparator (CUDA-graph replays, each timed region at least
        MIN_TIMED_MS long)."""
        w, L, T = self.w, len(self.layers), self.T
        cols = w.num_q_heads // w.num_kv_heads * T
        self.kernel = "auto"
        ms, _, clocks, n = self.timed(self.graph("comp", lambda: self.step(False)), steps, warmup, min_ms=MIN_TIMED_MS)
        self.kernel = "warp_mma"
        mms, _, mclocks, _ = self.timed(self.graph("comp_mma", lambda: self.step(False)), steps, warmup,
                                        min_ms=MIN_TIMED_MS)
        self.kernel = "auto"
        dms, _, dclocks, _ = self.timed(self.graph("dense", lambda: self.step(True)), steps, warmup,
                                        min_ms=MIN_TIMED_MS)
        comp_b, dense_b, _, ratio, _ = self.bytes()
        if any(self.status()):
            raise RuntimeError(f"device status word set: {self.status()}")
        return {"workload": w.name, "tokens": T, "columns_per_kv_head": cols, "layers_per_step": L,
                "auto_kernel": "tcgen05" if cols > 8 else "warp_mma",
                "us_per_step": round(ms * 1e3, 3), "steps_timed": n,
                "pct_of_hbm_peak_one_pass": round(100 * comp_b / (ms * 1e-3) / 1e9 / peak, 1),
                "warp_mma_us_per_step": round(mms * 1e3, 3), "dense_us_per_step": round(dms * 1e3, 3),
                "speedup_vs_warp_mma": round(mms / ms, 4), "speedup_vs_dense": round(dms / ms, 4),
                "compression_ratio": round(ratio, 4), "clocks": clocks, "warp_mma_clocks": mclocks,
                "dense_clocks": dclocks}

    # ---- one entry of per_config
    def summary(self, steps, warmup, peak):
        """The workload measured the same way as the headline (graph replays or eager appending
        steps), each timed region at least MIN_TIMED_MS long, plus single calls timed alone."""
        w, L = self.w, len(self.layers)
        eager = self.append is not None
        if eager:
            ms, call_ms, clocks, n = self.timed(lambda: self.step(False), steps, warmup, per_call=True,
                                                min_ms=MIN_TIMED_MS)
            dms, dcall_ms, dclocks, dn = self.timed(lambda: self.step(True), steps, warmup, per_call=True,
                                                    min_ms=MIN_TIMED_MS, dense=True)
            rms, _, _, _ = self.timed(lambda: self.step(False, reencode=True), steps, warmup,
                                      min_ms=MIN_TIMED_MS, reencode=True)
        else:
            ms, _, clocks, n = self.timed(self.graph("comp", lambda: self.step(False)), steps, warmup,
                                          min_ms=MIN_TIMED_MS)
            dms, _, dclocks, dn = self.timed(self.graph("dense", lambda: self.step(True)), steps, warmup,
                                             min_ms=MIN_TIMED_MS)
            call_ms, dcall_ms = ms / L, dms / L
        iso = self.isolated_call_ms(False)
        iso_d = self.isolated_call_ms(True)
        restore = self.restore_ms(steps, warmup, min_ms=MIN_TIMED_MS)
        comp_b, dense_b, unc_b, ratio, raw = self.bytes()
        call_b, dcall_b = comp_b / L, dense_b / L
        speed = dms / ms
        out = {
            "workload": w.name, "note": w.note, "layers_per_step": L, "launch_mode": "eager" if eager else "cuda_graph",
            "us_per_step": round(ms * 1e3, 3), "call_us": round(call_ms * 1e3, 3), "steps_timed": n,
            "timed_ms": round(ms * n, 1),
            "kv_gbs_compressed": round(comp_b / (ms * 1e-3) / 1e9, 1),
            "kv_gbs_effective_uncompressed": round(unc_b / (ms * 1e-3) / 1e9, 1),
            "pct_of_hbm_peak": round(100 * comp_b / (ms * 1e-3) / 1e9 / peak, 1),
            "pct_of_8tbs_spec": round(100 * comp_b / (ms * 1e-3) / 1e9 / SPEC_HBM_GBS, 1),
            "call_pct_of_hbm_peak": round(100 * call_b / (call_ms * 1e-3) / 1e9 / peak, 1),
            "compression_ratio": round(ratio, 4), "raw_page_heads": round(raw, 6),
            "dense_us_per_step": round(dms * 1e3, 3), "dense_call_us": round(dcall_ms * 1e3, 3),
            "dense_pct_of_hbm_peak": round(100 * dense_b / (dms * 1e-3) / 1e9 / peak, 1),
            "speedup_vs_dense": round(speed, 4),
            "speedup_bars": {"ratio_x_0.9": round(ratio * 0.9, 4), "ratio_minus_0.1": round(ratio - 0.1, 4),
                             "meets_both": speed >= max(ratio * 0.9, ratio - 0.1)},
            "isolated_call": {"compressed_us": round(iso * 1e3, 3), "dense_us": round(iso_d * 1e3, 3),
                              "speedup_vs_dense": round(iso_d / iso, 4),
                              "pct_of_hbm_peak": round(100 * call_b / (iso * 1e-3) / 1e9 / peak, 1),
                              "calls": ISOLATED_CALLS, "stat": "median",
                              "method": f"layer 0, one call after a {2 * L2_BYTES >> 20} MiB fill kernel "
                                        "(L2 flushed, no attention grid ahead to overlap)"},
            "restore_then_attend_us_per_step": round(restore * 1e3, 3),
            "fused_speedup_vs_restore": round(restore / ms, 4),
            "traffic_bytes_per_call": read_traffic(w.name) if self.T == 1 else None,
            "clocks": clocks, "dense_clocks": dclocks,
        }
        if eager:
            out["reencode_us_per_step"] = round(rms * 1e3, 3)
            out["step_note"] = ("each step writes one token per request into its tail page with zf_append_tokens "
                                "(a page the token fills is compressed), then attends; reencode_us_per_step: the "
                                "same step re-encoding the whole tail page with zf_encode_pages instead")
        if any(self.status()):
            raise RuntimeError(f"{w.name}: device status word set: {self.status()}")
        return out


class LongContextAppend:
    """Long-context step: every request writes one new token into its tail page, then attends.
    The compressed cache takes the token through zf_append_tokens (into the page's raw slot; the
    token that fills a page compresses it), or, in the re-encode variant, re-encodes the whole
    tail page through zf_encode_pages (raw while partial, compressed once it is full).  The dense
    comparator's step writes the same tail page raw into the dense cache (the slot of a page id is
    the id itself there).

    All requests have the same length, so the tail page index is shared.  Tail pages (natural
    layout) come from a seeded staging buffer [new page][request][Hkv][P][128] and each step's
    tokens from the same values; per-step lengths, fill counts, positions, page ids and raw slots
    are precomputed device arrays, so a step launches only the write and the attention kernels."""

    @staticmethod
    def count_new_pages(w, max_steps):
        return (max_steps + w.page_size - 1) // w.page_size + 1

    @staticmethod
    def extra_pages(w, max_steps):
        return LongContextAppend.count_new_pages(w, max_steps) * w.batch

    def __init__(self, zf, I, w, ent, device, max_steps):
        import torch
        self.zf, self.w, self.ent = zf, w, ent
        lay = ent["layer"]
        P, B = w.page_size, w.batch
        L0 = [int(x) for x in lay.seq_lens.cpu()]
        assert len(set(L0)) == 1, "append path expects equal request lengths"
        L0 = L0[0]
        assert L0 % P == 0, "append path starts from full pages"
        self.new_pages = self.count_new_pages(w, max_steps)
        spare0 = ent["num_pages"]
        ids = torch.arange(self.new_pages * B, dtype=torch.int32).reshape(self.new_pages, B) + spare0
        self.table = torch.cat([lay.page_table.cpu(), ids.t()], dim=1).contiguous().to(device)
        steps = torch.arange(1, max_steps + 1)
        lens = L0 + steps
        self.page_of_step = ((lens - 1) // P - L0 // P).tolist()
        self.lens_all = lens[:, None].expand(max_steps, B).to(torch.int32).contiguous().to(device)
        self.fill_all = ((lens - 1) % P + 1)[:, None].expand(max_steps, B).to(torch.int32).contiguous().to(device)
        self.pos_all = self.fill_all - 1
        self.ids_all = ids.to(device)
        self.raw_reencode = torch.arange(B, dtype=torch.int32, device=device)
        # appends: a fresh raw slot per new page (raw slot = page id: the cache has a raw slot for
        # every id), so a page left raw keeps its slot
        self.raw_append = self.ids_all
        gen = torch.Generator(device=device)
        gen.manual_seed(w.seed * 1000 + 999)
        shape = (self.new_pages, B, w.num_kv_heads, P, 128)
        self.src_k = torch.randn(shape, generator=gen, device=device).to(torch.bfloat16).view(torch.int16)
        self.src_v = torch.randn(shape, generator=gen, device=device).to(torch.bfloat16).view(torch.int16)
        # the token step n writes: position (L0 + n) % P of new page page_of_step[n], [step][B][Hkv][128]
        j = torch.tensor(self.page_of_step, device=device)
        pos = ((lens - 1) % P).to(device)
        self.tok_k = self.src_k[j, :, :, pos].contiguous()
        self.tok_v = self.src_v[j, :, :, pos].contiguous()
        self.max_steps = max_steps
        self.base_lens = lay.seq_lens
        self.reset()

    def reset(self):
        self.n = 0
        self.lens = self.base_lens

    def step(self, dense=False, reencode=False):
        import ctypes
        import torch
        if self.n >= self.max_steps:
            raise RuntimeError("more append steps than planned")
        j = self.page_of_step[self.n]
        d = self.ent["dense" if dense else "cache"].desc()
        P = ctypes.c_void_p
        stream = torch.cuda.current_stream().cuda_stream
        if dense or reencode:
            slots = self.ids_all[j] if dense else self.raw_reencode
            code = self.zf.lib().zf_encode_pages(
                ctypes.byref(d), P(self.src_k[j].data_ptr()), P(self.src_v[j].data_ptr()),
                P(self.ids_all[j].data_ptr()), P(self.fill_all[self.n].data_ptr()), P(slots.data_ptr()), self.w.batch,
                self.zf.ENCODE_FORCE_RAW if dense else 0, stream)
            name = "zf_encode_pages"
        else:
            code = self.zf.lib().zf_append_tokens(
                ctypes.byref(d), P(self.tok_k[self.n].data_ptr()), P(self.tok_v[self.n].data_ptr()),
                P(self.ids_all[j].data_ptr()), P(self.pos_all[self.n].data_ptr()),
                P(self.raw_append[j].data_ptr()), self.w.batch, stream)
            name = "zf_append_tokens"
        if code != 0:
            raise RuntimeError(f"{name} failed: {code}")
        self.lens = self.lens_all[self.n]
        self.n += 1


def run_gpu(args, rank, world, local_rank):
    import torch

    from decode_attention_compressed_gb300 import build as B
    from decode_attention_compressed_gb300 import inputs as I

    B.build()
    from decode_attention_compressed_gb300 import zf

    device = torch.device(f"cuda:{local_rank}")
    torch.cuda.set_device(device)
    w = workload_of(args)
    T = args.tokens
    peak, peak_kind = read_peaks()
    max_steps = 4 * (args.steps + args.warmup) + 64
    if w.name == "long_ctx":
        max_steps = max(max_steps, 2 * math.ceil(MIN_TIMED_MS / 0.2) + 64)
    wb = Workbench(zf, I, w, device, T, world, local_rank, max_steps, kernel=args.kernel)
    layers = wb.layers
    L = len(layers)
    use_graph = wb.append is None           # the append step changes pointers every step: eager
    if use_graph:
        ms_step, _, clocks, _ = wb.timed(wb.graph("comp", lambda: wb.step(False)), args.steps, args.warmup)
        call_ms = ms_step / L
        dense_ms_step, _, dense_clocks, _ = wb.timed(wb.graph("dense", lambda: wb.step(True)), args.steps,
                                                     args.warmup)
        dense_call_ms = dense_ms_step / L
        eager_ms, _, _, _ = wb.timed(lambda: wb.step(False), args.steps, args.warmup)
        eager_dense_ms, _, _, _ = wb.timed(lambda: wb.step(True), args.steps, args.warmup)
    else:
        ms_step, call_ms, clocks, _ = wb.timed(lambda: wb.step(False), args.steps, args.warmup, per_call=True)
        dense_ms_step, dense_call_ms, dense_clocks, _ = wb.timed(lambda: wb.step(True), args.steps, args.warmup,
                                                                 per_call=True, dense=True)
        eager_ms, eager_dense_ms = ms_step, dense_ms_step
    restore_ms = wb.restore_ms(args.steps, args.warmup)

    # end to end through the public API: every layer's q and seq_lens from pinned host memory (one
    # copy of the stacked step inputs), the calls, every layer's out + lse back (one copy each)
    qs, oshape = wb.qs, wb.oshape
    q_host = torch.stack([q.cpu() for q in qs]).pin_memory()
    lens_host = torch.stack([ent["layer"].seq_lens.cpu() for ent in layers]).pin_memory()
    q_dev, lens_dev = torch.empty_like(q_host, device=device), torch.empty_like(lens_host, device=device)
    out_dev = torch.empty((L, *oshape, 128), device=device)
    lse_dev = torch.empty((L, *oshape), device=device)
    out_host = torch.empty(out_dev.shape, pin_memory=True)
    lse_host = torch.empty(lse_dev.shape, pin_memory=True)

    def e2e_step():
        q_dev.copy_(q_host, non_blocking=True)
        lens_dev.copy_(lens_host, non_blocking=True)
        for i, ent in enumerate(layers):
            lay = ent["layer"]
            wb.attn(ent["cache"], q_dev[i], lay.page_table, lens_dev[i], lay.scale, out_dev[i], lse_dev[i])
        out_host.copy_(out_dev, non_blocking=True)
        lse_host.copy_(lse_dev, non_blocking=True)

    if use_graph:
        append, wb.append = wb.append, None
        e2e_ms, _, _, _ = wb.timed(wb.graph("e2e", e2e_step), args.steps, args.warmup)
        e2e_eager_ms, _, _, _ = wb.timed(e2e_step, args.steps, args.warmup)
        wb.append = append
        h2d = q_host.numel() * q_host.element_size() + lens_host.numel() * lens_host.element_size()
        d2h = out_host.numel() * 4 + lse_host.numel() * 4
    else:
        e2e_ms = e2e_eager_ms = None
        h2d = d2h = 0

    comp_bytes, dense_bytes, uncompressed, ratio, raw = wb.bytes()
    per_launch = comp_bytes / L
    achieved = per_launch / (call_ms * 1e-3) / 1e9
    if any(wb.status()):
        raise RuntimeError(f"device status word set: {wb.status()}")
    result = dict(
        metric=METRIC, value=round(ms_step * 1e3, 3), unit="us/step", n_gpus=world, steps=args.steps,
        warmup=args.warmup, ms_per_step=round(ms_step, 5), higher_is_better=False, scaling="weak",
        vs_baseline=None, dtype="bf16", data="synthetic (seeded, distributions of the workload)",
        config=arm_config(w, T, args.kernel, world),
        kv_gbs_compressed=round(comp_bytes / (ms_step * 1e-3) / 1e9, 1),
        kv_gbs_effective_uncompressed=round(uncompressed / (ms_step * 1e-3) / 1e9, 1),
        pct_of_hbm_peak=round(100 * comp_bytes / (ms_step * 1e-3) / 1e9 / peak, 1),
        pct_of_8tbs_spec=round(100 * comp_bytes / (ms_step * 1e-3) / 1e9 / SPEC_HBM_GBS, 1),
        compression_ratio=round(ratio, 4), raw_page_heads=round(raw, 6),
        bytes_read_ratio=round(dense_bytes / comp_bytes, 4),
        dense={"us_per_step": round(dense_ms_step * 1e3, 3), "kv_gbs": round(dense_bytes / (dense_ms_step * 1e-3) / 1e9, 1),
               "pct_of_hbm_peak": round(100 * dense_bytes / (dense_ms_step * 1e-3) / 1e9 / peak, 1),
               "call_us": round(dense_call_ms * 1e3, 3), "clocks": dense_clocks},
        speedup_vs_dense=round(dense_ms_step / ms_step, 4),
        restore_then_attend={"us_per_step": round(restore_ms * 1e3, 3),
                             "speedup_of_fused": round(restore_ms / ms_step, 4),
                             "note": "per layer: zf_decompress_to_raw of all its pages into one shared dense "
                                     "buffer, then zf_dense_decode_attn (static inputs; CUDA graph)"},
        launch_mode="cuda_graph (one graph per decode step)" if use_graph else "eager",
        eager={"us_per_step": round(eager_ms * 1e3, 3), "dense_us_per_step": round(eager_dense_ms * 1e3, 3),
               "e2e_us_per_step": round(e2e_eager_ms * 1e3, 3) if e2e_eager_ms else None},
        roofline={"kernel": "attn_kernel<compressed> + merge_kernel (one "
                            + ("zf_decode_attn_multi" if T > 1 else "zf_decode_attn") + " call; "
                            + ("step time / layers" if use_graph else "events around each call") + ")",
                  "bound": "hbm",
                  "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
                  "peak_source": peak_kind, "bytes_per_launch": int(per_launch), "call_us": round(call_ms * 1e3, 3),
                  # the committed capture is of the warp-MMA kernel, single token, full batch
                  "traffic": read_traffic(w.name) if T == 1 and args.kernel != "tcgen05"
                  and args.batch is None else None},
        e2e={"value": round(e2e_ms * 1e3, 3) if e2e_ms else None, "unit": "us/step", "h2d_bytes_per_step": h2d,
             "d2h_bytes_per_step": d2h},
        gpu_launches=args.steps * L * 2 + (args.steps if wb.append is not None else 0),
        gpu_launches_note="per timed region of the compressed path: attention + merge per layer (+1 token write "
                          "per step when appending)",
        clocks=clocks,
    )
    per_config = rank == 0 and world == 1 and not args.no_per_config and T == 1 and args.layers is None \
        and args.batch is None
    if per_config:
        per = {}
        for name in PER_CONFIG:
            if name == w.name:
                per[name] = wb.summary(args.steps, args.warmup, peak)
                continue
            other = Workbench(zf, I, I.WORKLOADS[name], device, 1, world, local_rank,
                              max(max_steps, 2 * math.ceil(MIN_TIMED_MS / 0.2) + 64))
            per[name] = other.summary(args.steps, args.warmup, peak)
            del other
            torch.cuda.empty_cache()
        per["long_ctx"]["prefill_encode"] = prefill_encode(zf, I, device, peak)
        result["per_config"] = per
        multi = {}
        for name, T in MULTI_TOKEN:
            mt = Workbench(zf, I, I.WORKLOADS[name], device, T, world, local_rank, max_steps)
            multi[f"{name}_t{T}"] = mt.multi_token_summary(args.steps, args.warmup, peak)
            del mt
            torch.cuda.empty_cache()
        result["multi_token"] = multi
        result["prefill_encode"] = per["long_ctx"]["prefill_encode"]
    return result


# ------------------------------------------------------------------------------ CPU oracle arm
def usable_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def _oracle_head_inputs(w, heads, out_dir, tokens=1):
    """Request 0 of layer 0: for each of `heads` kv heads, its BF16 keys, values, query rows (of
    `tokens` new tokens) and length, saved under out_dir (one .npz per head) for the oracle worker
    processes."""
    import numpy as np
    import torch
    from decode_attention_compressed_gb300 import inputs as I
    layer = I.make_layer(w, layer=0, device="cpu")
    qm = I.make_multi_queries(w, tokens, layer=0) if tokens > 1 else None
    P = w.page_size
    L = int(layer.seq_lens[0])
    pages = layer.page_table[0, : -(-L // P)].to(torch.long)
    paths = []
    for h in heads:
        g = h % w.num_kv_heads
        path = os.path.join(out_dir, f"head{h}.npz")
        np.savez(path, k=layer.k_pages[pages][:, g:g + 1].numpy().view(np.uint16),
                 v=layer.v_pages[pages][:, g:g + 1].numpy().view(np.uint16),
                 n_valid=layer.n_valid[pages].numpy(),
                 q=(qm[:1, :, g * w.group:(g + 1) * w.group] if tokens > 1
                    else layer.q[:1, g * w.group:(g + 1) * w.group]).numpy().view(np.uint16),
                 L=np.array([L]), P=np.array([P]), scale=np.array([layer.scale]))
        paths.append(path)
    return paths


def _oracle_worker(path, barrier, queue, target_s, reps):
    """One oracle process: encode its kv head's pages (untimed), wait for the others, then run the
    oracle's decode attention for that head `reps` times (or for target_s seconds)."""
    import numpy as np
    from oracle import zf_oracle as O
    d = np.load(path)
    P, L = int(d["P"][0]), int(d["L"][0])
    npg = d["k"].shape[0]
    oc = O.Cache(num_pages=npg, num_kv_heads=1, page_size=P, num_raw=npg)
    O.encode_pages(oc, d["k"], d["v"], list(range(npg)), d["n_valid"], list(range(npg)))
    table = np.arange(npg, dtype=np.int32)[None]
    lens, q, scale = np.array([L]), d["q"], float(d["scale"][0])
    attend = O.decode_attention_multi if q.ndim == 4 else O.decode_attention   # [1][T][heads][128]: T tokens
    attend(q, oc, table, lens, scale)                      # untimed warm-up
    barrier.wait(timeout=900)
    t0 = time.perf_counter()
    n = 0
    while (reps and n < reps) or (not reps and (n == 0 or time.perf_counter() - t0 < target_s)):
        attend(q, oc, table, lens, scale)
        n += 1
    queue.put((n, time.perf_counter() - t0))


def oracle_pool(w, workers, target_s=0.0, reps=0, warm_reps=0, tokens=1):
    """Run the oracle on `workers` host cores at once (one process per core, one kv head of request
    0 each, spawn start method).  Returns (head-calls per second, calls per worker, wall seconds)."""
    import multiprocessing as mp
    import shutil
    ctx = mp.get_context("spawn")
    tmp = tempfile.mkdtemp(prefix="zf_oracle_")
    try:
        paths = _oracle_head_inputs(w, range(workers), tmp, tokens)
        barrier, queue = ctx.Barrier(workers), ctx.Queue()
        procs = [ctx.Process(target=_oracle_worker, args=(p, barrier, queue, target_s, reps)) for p in paths]
        for p in procs:
            p.start()
        res = []
        deadline = time.time() + 1800
        while len(res) < len(procs):
            try:
                res.append(queue.get(timeout=1.0))
            except Exception:                       # queue.Empty: check that every worker is alive
                dead = [p.exitcode for p in procs if p.exitcode not in (None, 0)]
                if dead or time.time() > deadline:
                    for p in procs:
                        if p.is_alive():
                            p.terminate()
                    raise RuntimeError(f"oracle worker failed (exit codes {dead})")
        for p in procs:
            p.join(timeout=60)
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
    calls = sum(n for n, _ in res)
    wall = max(t for _, t in res)
    return calls / wall, [n for n, _ in res], wall


def cpu_baseline(w, target_s=12.0, tokens=1):
    """Time the oracle (as it stands) on the host cores on a bounded sample — one kv head of
    request 0, layer 0, per core, for about target_s seconds — and scale to microseconds per full
    decode step (all requests, kv heads and layers)."""
    cores = usable_cores()
    rate, calls, wall = oracle_pool(w, cores, target_s=target_s, tokens=tokens)
    head_calls = w.batch * w.num_kv_heads * w.layers
    lens_note = "request 0" if w.ctx_min is None else "request 0 (lengths vary; scaled by batch)"
    return {"value": round(head_calls / rate * 1e6, 1), "unit": "us/step", "cores": cores, "kind": "oracle",
            "extrapolated": True,
            "sample": f"{cores} processes (one per core), each the oracle's decode attention of one kv head "
                      f"({w.group} query heads, {tokens} new token{'s' if tokens > 1 else ''}) of {lens_note}, "
                      f"layer 0 of {w.name}, {sum(calls)} calls in "
                      f"{wall:.1f} s; scaled x{head_calls} head-calls to the full step"}


def run_reference(args, rank):
    if rank != 0:
        return None
    w = workload_of(args)
    cores = usable_cores()
    # each step: every core runs the oracle for one kv head (request 0, layer 0); the full step's
    # time is that sample's time scaled by the head-calls of the step over the cores' heads
    rate, calls, wall = oracle_pool(w, cores, reps=args.steps + args.warmup, tokens=args.tokens)
    head_calls = w.batch * w.num_kv_heads * w.layers
    per = head_calls / rate
    v = round(per * 1e6, 1)
    return dict(metric=METRIC, value=v, unit="us/step", n_gpus=0, steps=args.steps, warmup=args.warmup,
                ms_per_step=round(per * 1e3, 3), higher_is_better=False, scaling="weak", vs_baseline=None,
                dtype="f64", data="synthetic (seeded, distributions of the workload)",
                config=arm_config(w, args.tokens, args.kernel, int(os.environ.get("WORLD_SIZE", "1"))),
                impl="reference", extrapolated=True,
                sample_wall_s=round(wall, 2),
                cpu_baseline={"value": v, "unit": "us/step", "cores": cores, "kind": "oracle",
                              "sample": f"each step: {cores} processes, each the oracle's decode attention of one "
                                        f"kv head ({w.group} query heads, {args.tokens} new token"
                                        f"{'s' if args.tokens > 1 else ''}) of request 0, layer 0 ({sum(calls)} calls "
                                        f"incl. warm-up in {wall:.1f} s); scaled x{head_calls} head-calls over "
                                        f"{cores} cores to the full step: an extrapolation, not a full step run"},
                e2e={"value": v, "unit": "us/step", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0})


def _free_port() -> int:
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def launch_ranks(n: int, argv, script=None, capture_output=False):
    """Start `script` (this file by default) under torch.distributed.run with n ranks on this node
    (one per GPU), rendezvous on 127.0.0.1; returns the finished process."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", f"--nproc-per-node={n}",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), script or os.path.abspath(__file__),
           *argv]
    return subprocess.run(cmd, capture_output=capture_output, text=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=240)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="measure only the headline workload (no per_config object)")
    ap.add_argument("--kernel", default="auto", choices=["auto", "warp_mma", "tcgen05"],
                    help="compressed attention kernel (zf_decode_attn_multi_kernel)")
    ap.add_argument("--tokens", type=int, default=1,
                    help="new tokens per request per call (speculative verification; zf_decode_attn_multi)")
    ap.add_argument("--layers", type=int, default=None,
                    help="use only the first N layers of a multi-layer workload (profiling captures)")
    ap.add_argument("--batch", type=int, default=None,
                    help="use only the first B requests (profiling captures on a smaller device footprint)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # started without torchrun: start the N ranks (one replica per GPU) and pass their output on
        raise SystemExit(launch_ranks(args.gpus, sys.argv[1:]).returncode)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        res = run_reference(args, rank)
        if res is not None:
            print(json.dumps(res), flush=True)
        return

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    res = run_gpu(args, rank, world, local_rank)
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline(workload_of(args), tokens=args.tokens)
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

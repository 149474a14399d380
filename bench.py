"""Benchmark: decode-attention microseconds per decode step over the compressed BF16 paged KV cache,
with KV GB/s (compressed and effective-uncompressed), the fraction of the measured HBM peak, and
the same step on the dense-BF16 kernel.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step = one decode step of the workload: for every layer, zf_decode_attn over that layer's
compressed cache (the long-context workload also appends one token per request through
zf_encode_pages each step).  Inputs are resident in HBM; the per-step KV bytes exceed L2, so no
extra flush is needed.  Prints one JSON line on rank 0.  N > 1 runs N independent replicas (one
per GPU, weak scaling); the step time is the maximum over ranks.
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

os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")     # the CPU baseline runs the oracle on one core

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
KERNEL_SOURCES = ("zf_attn.cu", "zf_device.cuh", "zf_host.h")


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
    path = os.path.join(ROOT, "profiles", "traffic.txt")
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


def setup_layers(zf, I, w, device):
    import torch
    layers = []
    for l in range(w.layers):
        layer = I.make_layer(w, layer=l, device=device)
        npg = layer.num_pages
        extra = 0
        if w.name == "long_ctx":
            extra = 8 * w.batch       # spare page ids for the appended tokens
        # page i keeps id i; raw slot i is its fallback (partial tails, blocks with > 6 escapes)
        cache = zf.Cache(npg + extra, w.num_kv_heads, w.page_size, npg + extra, device=device)
        zf.encode_pages(cache, layer.k_pages, layer.v_pages, list(range(npg)), layer.n_valid, list(range(npg)))
        dense = zf.Cache(npg + extra, w.num_kv_heads, w.page_size, npg + extra, device=device, compressed=False)
        zf.encode_pages(dense, layer.k_pages, layer.v_pages, list(range(npg)), layer.n_valid, list(range(npg)),
                        force_raw=True)
        torch.cuda.synchronize()
        if cache.status_word() or dense.status_word():
            raise RuntimeError("encode reported a device error")
        dirs = cache.dir.cpu()
        entry = dict(layer=layer, cache=cache, dense=dense, dirs=dirs, num_pages=npg)
        if w.name != "long_ctx":
            layer.k_pages = layer.v_pages = None          # the caches hold the data now
        layers.append(entry)
    return layers


def prefill_encode_ms(zf, I, device):
    """Time a full-prefill encode: 8192 tokens x 32 layers, 8 kv heads, 64-token pages."""
    import torch
    w = I.scaled(I.WORKLOADS["long_ctx"], batch=1, ctx=8192)
    layer = I.make_layer(w, device=device)
    npg = layer.num_pages
    caches = [zf.Cache(npg, w.num_kv_heads, w.page_size, 8, device=device) for _ in range(32)]
    ids = torch.arange(npg, dtype=torch.int32, device=device)
    nv = layer.n_valid.to(device)
    rs = torch.full((npg,), -1, dtype=torch.int32, device=device)
    for c in caches[:2]:
        zf.encode_pages(c, layer.k_pages, layer.v_pages, ids, nv, rs)
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for c in caches:
        zf.encode_pages(c, layer.k_pages, layer.v_pages, ids, nv, rs)
    e.record()
    torch.cuda.synchronize()
    ms = s.elapsed_time(e)
    src_bytes = 2 * layer.k_pages.numel() * 2 * 32
    return ms, src_bytes / (ms * 1e-3) / 1e9


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


def workload_of(args):
    from decode_attention_compressed_gb300 import inputs as I
    w = I.WORKLOADS[args.workload]
    kw = {}
    if args.layers is not None:
        kw["layers"] = min(args.layers, w.layers)
    if args.batch is not None:
        kw["batch"] = min(args.batch, w.batch)
    return I.scaled(w, **kw) if kw else w


def run_gpu(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    from decode_attention_compressed_gb300 import build as B
    from decode_attention_compressed_gb300 import inputs as I

    B.build()
    from decode_attention_compressed_gb300 import zf

    device = torch.device(f"cuda:{local_rank}")
    torch.cuda.set_device(device)
    w = workload_of(args)
    layers = setup_layers(zf, I, w, device)
    stream = torch.cuda.current_stream()
    T = args.tokens
    if T > 1 and w.name == "long_ctx":
        raise SystemExit("--tokens > 1 is not combined with the long-context append step")
    # several new tokens per request: each layer's queries [batch][T][heads][128] (zf_decode_attn_multi)
    qs = [I.make_multi_queries(w, T, layer=i, device=device) if T > 1 else ent["layer"].q
          for i, ent in enumerate(layers)]
    oshape = (w.batch, T, w.num_q_heads) if T > 1 else (w.batch, w.num_q_heads)
    outs = [(torch.empty(*oshape, 128, device=device), torch.empty(*oshape, device=device)) for _ in layers]

    def attn(cache, q, table, lens, scale, out, lse, dense=False):
        if T > 1:
            zf.decode_attn_multi(cache, q, table, lens, scale, out=out, lse=lse, workspace=workspace, dense=dense)
        else:
            zf.decode_attn(cache, q, table, lens, scale, out=out, lse=lse, workspace=workspace, dense=dense)

    append = None
    max_pages = int(layers[0]["layer"].page_table.shape[1])
    if w.name == "long_ctx":
        append = LongContextAppend(zf, I, w, layers[0], device, 2 * (args.steps + args.warmup))
        max_pages = int(append.table.shape[1])
    ws_bytes = zf.workspace_size_multi(w.batch, T, w.num_q_heads, w.num_kv_heads, w.page_size, max_pages)
    workspace = zf.new_workspace(ws_bytes, device)

    def step(dense=False, events=None):
        if append is not None:
            append.step(dense)
        for i, ent in enumerate(layers):
            lay = ent["layer"]
            lens = append.lens if append is not None else lay.seq_lens
            table = append.table if append is not None else lay.page_table
            if events is not None:
                events[i][0].record()
            attn(ent["dense"] if dense else ent["cache"], qs[i], table, lens, lay.scale, outs[i][0], outs[i][1], dense)
            if events is not None:
                events[i][1].record()

    def capture(fn):
        """fn() captured once into a CUDA graph (after one eager warm-up on a side stream)."""
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

    def timed(run, steps=args.steps, warmup=args.warmup, per_call=False, dense=False):
        """Device time per step of `run` (CUDA events on the launching stream; max over ranks),
        the mean per-call duration when per_call is set (eager only), and the clocks seen."""
        for _ in range(warmup):
            run()
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        events = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in layers] for _ in range(steps)] if per_call else None
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with ClockSampler(local_rank) as clk:
            s.record()
            for k in range(steps):
                if per_call:
                    step(dense, events[k])
                else:
                    run()
            e.record()
            torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        ms = s.elapsed_time(e)
        calls = [x.elapsed_time(y) for row in events for (x, y) in row] if per_call else None
        if world > 1:
            ms = max_over_ranks(ms, device)
        return ms / steps, (statistics.mean(calls) if calls else None), clk.summary()

    use_graph = append is None           # the append step changes pointers every step: eager
    if use_graph:
        g_comp = capture(lambda: step(False))
        g_dense = capture(lambda: step(True))
        ms_step, _, clocks = timed(g_comp.replay)
        call_ms = ms_step / len(layers)
        dense_ms_step, _, dense_clocks = timed(g_dense.replay)
        dense_call_ms = dense_ms_step / len(layers)
        eager_ms, _, _ = timed(lambda: step(False))
        eager_dense_ms, _, _ = timed(lambda: step(True))
    else:
        append.reset()
        ms_step, call_ms, clocks = timed(lambda: step(False), per_call=True)
        append.reset()
        dense_ms_step, dense_call_ms, dense_clocks = timed(lambda: step(True), per_call=True, dense=True)
        eager_ms, eager_dense_ms = ms_step, dense_ms_step

    # Restore-then-attend baseline (ZipFusion §II.B): each layer is decompressed into one shared
    # dense buffer (zf_decompress_to_raw) and the dense kernel attends over it.  Static inputs (the
    # long-context workload without its per-step append).
    max_np = max(ent["num_pages"] for ent in layers)
    shared = zf.Cache(max_np, w.num_kv_heads, w.page_size, max_np, device=device, compressed=False)
    all_ids = [torch.arange(ent["num_pages"], dtype=torch.int32, device=device) for ent in layers]

    def restore_step():
        for i, ent in enumerate(layers):
            lay = ent["layer"]
            zf.decompress_to_raw(ent["cache"], all_ids[i], shared)
            attn(shared, qs[i], lay.page_table, lay.seq_lens, lay.scale, outs[i][0], outs[i][1], dense=True)

    g_restore = capture(restore_step)
    restore_ms, _, _ = timed(g_restore.replay)
    del g_restore, shared

    # end to end through the public API: every layer's q and seq_lens from pinned host memory (one
    # copy of the stacked step inputs), the 32 calls, every layer's out + lse back (one copy each)
    L = len(layers)
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
            attn(ent["cache"], q_dev[i], lay.page_table, lens_dev[i], lay.scale, out_dev[i], lse_dev[i])
        out_host.copy_(out_dev, non_blocking=True)
        lse_host.copy_(lse_dev, non_blocking=True)

    if append is None:
        g_e2e = capture(e2e_step)
        e2e_ms, _, _ = timed(g_e2e.replay)
        e2e_eager_ms, _, _ = timed(e2e_step)
        h2d = q_host.numel() * q_host.element_size() + lens_host.numel() * lens_host.element_size()
        d2h = out_host.numel() * 4 + lse_host.numel() * 4
    else:
        e2e_ms = e2e_eager_ms = None
        h2d = d2h = 0

    comp_bytes = sum(tile_bytes(ent["layer"], ent["dirs"], True, T) for ent in layers)
    dense_bytes = sum(tile_bytes(ent["layer"], ent["dirs"], False, T) for ent in layers)
    uncompressed = sum(dense_equiv_bytes(ent["layer"]) for ent in layers)
    stored = sum(ent["cache"].stored_bytes(ent["num_pages"]) for ent in layers)
    dense_stored = sum(ent["num_pages"] * w.num_kv_heads * 2 * w.page_size * 128 * 2 for ent in layers)
    per_launch = comp_bytes / len(layers)
    peak, peak_kind = read_peaks()
    achieved = per_launch / (call_ms * 1e-3) / 1e9
    status = [ent["cache"].status_word() | ent["dense"].status_word() for ent in layers]
    if any(status):
        raise RuntimeError(f"device status word set: {status}")
    extra = {}
    if append is not None:
        extra["append_encode_per_step"] = {"requests": w.batch, "calls": 1}
        extra["prefill_encode_ms"], extra["prefill_encode_src_gbs"] = prefill_encode_ms(zf, I, device)
    result = dict(
        metric=METRIC, value=round(ms_step * 1e3, 3), unit="us/step", n_gpus=world, steps=args.steps,
        warmup=args.warmup, ms_per_step=round(ms_step, 5), higher_is_better=False, scaling="weak",
        vs_baseline=None, dtype="bf16", data="synthetic (seeded, distributions of the workload)",
        config={"workload": w.name, "note": w.note, "batch": w.batch, "q_heads": w.num_q_heads,
                "kv_heads": w.num_kv_heads, "head_dim": 128, "page_size": w.page_size, "ctx": w.ctx,
                "layers_per_step": w.layers, "new_tokens_per_request": T,
                "parallelism": "replicas" if world > 1 else "single",
                "l2": f"no flush: {comp_bytes / 1e9:.2f} GB of compressed KV read per step "
                      f"(> {L2_BYTES / 2**20:.0f} MiB L2)"},
        kv_gbs_compressed=round(comp_bytes / (ms_step * 1e-3) / 1e9, 1),
        kv_gbs_effective_uncompressed=round(uncompressed / (ms_step * 1e-3) / 1e9, 1),
        pct_of_hbm_peak=round(100 * comp_bytes / (ms_step * 1e-3) / 1e9 / peak, 1),
        pct_of_8tbs_spec=round(100 * comp_bytes / (ms_step * 1e-3) / 1e9 / SPEC_HBM_GBS, 1),
        compression_ratio=round(dense_stored / stored, 4),
        raw_page_heads=round(sum(float((ent["dirs"][: ent["num_pages"]] >= 0).float().mean()) for ent in layers)
                             / len(layers), 6),
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
                  "traffic": read_traffic(w.name) if T == 1 else None},
        e2e={"value": round(e2e_ms * 1e3, 3) if e2e_ms else None, "unit": "us/step", "h2d_bytes_per_step": h2d,
             "d2h_bytes_per_step": d2h},
        gpu_launches=args.steps * len(layers) * 2 + (args.steps if append is not None else 0),
        gpu_launches_note="per timed region of the compressed path: attention + merge per layer (+1 encode per step when appending)",
        clocks=clocks, **extra,
    )
    return result


class LongContextAppend:
    """Long-context step: every request appends one token to its tail page and that page is
    re-encoded through zf_encode_pages (raw while partial, compressed once it is full).  The dense
    comparator's step appends too: the same tail pages written raw into the dense cache (the slot
    of a page id is the id itself there).

    All requests have the same length, so the tail page index is shared.  Tail pages (natural
    layout) come from a seeded staging buffer [new page][request][Hkv][P][128]; per-step lengths,
    fill counts and page ids are precomputed device arrays, so a step launches only the encode
    and the attention kernels."""

    def __init__(self, zf, I, w, ent, device, max_steps):
        import torch
        self.zf, self.w, self.ent = zf, w, ent
        lay = ent["layer"]
        P, B = w.page_size, w.batch
        L0 = [int(x) for x in lay.seq_lens.cpu()]
        assert len(set(L0)) == 1, "append path expects equal request lengths"
        L0 = L0[0]
        base_pages = lay.page_table.shape[1]
        self.new_pages = (L0 % P + max_steps) // P + 1
        spare0 = ent["num_pages"]
        ids = torch.arange(self.new_pages * B, dtype=torch.int32).reshape(self.new_pages, B) + spare0
        self.table = torch.cat([lay.page_table.cpu(), ids.t()], dim=1).contiguous().to(device)
        steps = torch.arange(1, max_steps + 1)
        lens = L0 + steps
        self.page_of_step = ((lens - 1) // P - (L0 + P - 1) // P).tolist()
        self.lens_all = lens[:, None].expand(max_steps, B).to(torch.int32).contiguous().to(device)
        self.fill_all = ((lens - 1) % P + 1)[:, None].expand(max_steps, B).to(torch.int32).contiguous().to(device)
        self.ids_all = ids.to(device)
        self.raw_slots = torch.arange(B, dtype=torch.int32, device=device)
        gen = torch.Generator(device=device)
        gen.manual_seed(w.seed * 1000 + 999)
        shape = (self.new_pages, B, w.num_kv_heads, P, 128)
        self.src_k = torch.randn(shape, generator=gen, device=device).to(torch.bfloat16).view(torch.int16)
        self.src_v = torch.randn(shape, generator=gen, device=device).to(torch.bfloat16).view(torch.int16)
        self.max_steps = max_steps
        self.base_lens = lay.seq_lens
        self.reset()

    def reset(self):
        self.n = 0
        self.lens = self.base_lens

    def step(self, dense=False):
        import ctypes
        import torch
        if self.n >= self.max_steps:
            raise RuntimeError("more append steps than planned")
        j = self.page_of_step[self.n]
        d = self.ent["dense" if dense else "cache"].desc()
        P = ctypes.c_void_p
        slots = self.ids_all[j] if dense else self.raw_slots
        code = self.zf.lib().zf_encode_pages(
            ctypes.byref(d), P(self.src_k[j].data_ptr()), P(self.src_v[j].data_ptr()), P(self.ids_all[j].data_ptr()),
            P(self.fill_all[self.n].data_ptr()), P(slots.data_ptr()), self.w.batch,
            self.zf.ENCODE_FORCE_RAW if dense else 0, torch.cuda.current_stream().cuda_stream)
        if code != 0:
            raise RuntimeError(f"zf_encode_pages failed: {code}")
        self.lens = self.lens_all[self.n]
        self.n += 1


# ------------------------------------------------------------------------------ CPU oracle arm
def oracle_sample(I, O, w, heads, seed_layer=0):
    """Oracle cache for request 0 of layer 0 restricted to `heads` kv heads (built untimed), and a
    callable that runs the oracle's decode attention for the query heads of those kv heads."""
    import numpy as np
    import torch
    layer = I.make_layer(w, layer=seed_layer, device="cpu")
    P = w.page_size
    L = int(layer.seq_lens[0])
    pages = layer.page_table[0, : -(-L // P)].to(torch.long)
    kb = layer.k_pages[pages][:, :heads].numpy().view(np.uint16)
    vb = layer.v_pages[pages][:, :heads].numpy().view(np.uint16)
    npg = len(pages)
    oc = O.Cache(num_pages=npg, num_kv_heads=heads, page_size=P, num_raw=npg)
    O.encode_pages(oc, kb, vb, list(range(npg)), layer.n_valid[pages].numpy(), list(range(npg)))
    q = layer.q[:1, : heads * w.group].numpy().view(np.uint16)
    table = np.arange(npg, dtype=np.int32)[None]
    lens = np.array([L])

    def run():
        return O.decode_attention(q, oc, table, lens, layer.scale)
    return run


def cpu_baseline(w, target_s=12.0):
    """Time the oracle (as it stands) on a bounded sample: some kv heads of request 0, layer 0;
    scale to microseconds per full decode step (all requests, heads and layers)."""
    from decode_attention_compressed_gb300 import inputs as I
    from oracle import zf_oracle as O
    heads = 1
    run = oracle_sample(I, O, w, heads)
    t0 = time.perf_counter()
    run()
    one = time.perf_counter() - t0
    reps = max(1, int(target_s / max(one, 1e-3)))
    t0 = time.perf_counter()
    for _ in range(reps):
        run()
    per = (time.perf_counter() - t0) / reps
    scale = w.batch * w.num_kv_heads * w.layers / heads
    lens_note = "request 0" if w.ctx_min is None else "request 0 (lengths vary; scaled by batch)"
    return {"value": round(per * scale * 1e6, 1), "unit": "us/step", "cores": 1, "kind": "oracle",
            "sample": f"{reps}x oracle decode attention of 1 kv head ({w.group} query heads), {lens_note}, "
                      f"layer 0 of {w.name}; scaled x{scale:.0f} to the full step"}


def run_reference(args, rank):
    from decode_attention_compressed_gb300 import inputs as I
    from oracle import zf_oracle as O
    if rank != 0:
        return None
    w = workload_of(args)
    run = oracle_sample(I, O, w, 1)
    scale = w.batch * w.num_kv_heads * w.layers
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    per = (time.perf_counter() - t0) / args.steps * scale
    v = round(per * 1e6, 1)
    return dict(metric=METRIC, value=v, unit="us/step", n_gpus=0, steps=args.steps, warmup=args.warmup,
                ms_per_step=round(per * 1e3, 3), higher_is_better=False, scaling="weak", vs_baseline=None,
                dtype="f64", data="synthetic (seeded, distributions of the workload)",
                config={"workload": w.name, "batch": w.batch, "q_heads": w.num_q_heads, "kv_heads": w.num_kv_heads,
                        "page_size": w.page_size, "ctx": w.ctx, "layers_per_step": w.layers},
                impl="reference",
                cpu_baseline={"value": v, "unit": "us/step", "cores": 1, "kind": "oracle",
                              "sample": f"each step: oracle decode attention of 1 kv head ({w.group} query heads) "
                                        f"of request 0, layer 0, scaled x{scale} to the full step"},
                e2e={"value": v, "unit": "us/step", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0})


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--tokens", type=int, default=1,
                    help="new tokens per request per call (speculative verification; zf_decode_attn_multi)")
    ap.add_argument("--layers", type=int, default=None,
                    help="use only the first N layers of a multi-layer workload (profiling captures)")
    ap.add_argument("--batch", type=int, default=None,
                    help="use only the first B requests (profiling captures on a smaller device footprint)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", str(args.gpus if args.gpus == 1 else 1)))
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
        from decode_attention_compressed_gb300 import inputs as I
        if world == 1 and not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline(workload_of(args))
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

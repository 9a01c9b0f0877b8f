"""Benchmark of segment-relocated MLA attention (RedKnot-MLA online step).

One step = one forward of the whole path (plan built once, outside the timed
region) over the 128K long-context workload: 48 shuffled 2048-row document
latents + a 32768-row recomputed tail, H = 128 (112 Local / 16 Global),
d_nope = 512, d_rope = 64, sink 4, window 256, 25 % protected budget.

Prints ONE JSON line.  `value` is algorithmic attention TFLOP/s (2 d_k +
2 d_v FLOP per attended query-key pair); the decode-shaped batch (64
requests, split over segments) is reported alongside in HBM GB/s.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("seg-relocated MLA attention TFLOP/s & % bf16 peak (1×GB300); "
          "decode HBM GB/s")
WORKLOAD = "ctx128k"


def workload_desc(name: str) -> str:
    """One-line description of a named synthetic workload."""
    from position_independent_kv_gb300.workloads import SPECS
    sp = SPECS[name]
    hg = sp.H // 8
    if sp.decode_requests:
        lo, hi = sp.decode_len_range
        s0, s1 = sp.decode_seg_range
        seg = (f"{sp.decode_requests} requests x 1 row, {s0}-{s1} segments, {lo}-{hi} keys")
    elif sp.seg_lengths:
        seg = (f"{len(sp.seg_lengths)} x {sp.seg_lengths[0]}-row latents"
               f"{' (shuffled)' if sp.shuffle else ''} + {sp.n_new} new rows")
    else:
        lo, hi = sp.seg_len_range
        seg = f"{sp.n_segments} latents of {lo}-{hi} rows (shuffled) + {sp.n_new} new rows"
    r = sp.rule
    if r.none:
        prot = "no protected rows"
    elif r.budget:
        prot = f"protected budget {int(round(100 * r.budget))}% (boundary {r.boundary} first)"
    elif r.p_random:
        prot = f"protected: boundary {r.boundary} + {int(round(100 * r.p_random))}% random"
    else:
        prot = f"protected: query rows + boundary {r.boundary}"
    out = f", {int(round(100 * sp.outlier_frac))}% outlier rows x8" if sp.outlier_frac else ""
    vr = ", V = the whole latent row (output phase restored)" if sp.v_rope else ""
    if sp.q_tail:
        vr += f", only the last {sp.q_tail} rows computed"
    return (f"{name}: {seg}, H={sp.H} ({sp.H - hg} Local/{hg} Global), d_nope={sp.d_nope}, "
            f"d_rope={sp.d_rope}{vr}, sink={sp.sink}, w={sp.window}, {prot}, "
            f"bf16 N(0,1)/sqrt({sp.d_nope + sp.d_rope}){out}, seed 0")


FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(FALLBACK), "fallback"


PLAN_FLAGS = {"auto": 0, "pair": 8, "single": 4, "legacy": 2, "noside": 64}
KERNEL_SOURCES = {"mma_sync": ["dense_mma.cu", "common.cuh"],
                  "tcgen05_small": ["dense_tcs.cu", "tc_tile.cuh", "tc_ptx.cuh", "common.cuh"],
                  "tcgen05": ["dense_tc.cu", "tc_ptx.cuh", "common.cuh"],
                  "tcgen05_pair": ["dense_tc2.cu", "tc_tile.cuh", "tc_ptx.cuh", "common.cuh"],
                  "tcgen05_quad": ["dense_tc4.cu", "dense_side.cu", "tc_tile.cuh", "tc_ptx.cuh",
                                   "common.cuh"]}


def kernel_source_hash(kernel: str) -> str:
    """Hash of the source files of one kernel (traffic records go stale when
    these change)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "position_independent_kv_gb300", "csrc")
    for f in KERNEL_SOURCES[kernel]:
        fp = os.path.join(csrc, f)
        if os.path.exists(fp):
            h.update(open(fp, "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p))
        e = d.get(f"{kernel}:{workload}")
        if e and e.get("source_hash") == kernel_source_hash(kernel):
            return e.get("dram_bytes_per_launch")
    except Exception:
        return None
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.f = None

    def _bus_id(self):
        import torch
        try:
            pr = torch.cuda.get_device_properties(self.dev)
            return "%08x:%02x:%02x.0" % (pr.pci_domain_id, pr.pci_bus_id, pr.pci_device_id)
        except Exception:
            return None

    def start(self):
        try:
            self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            cmd = ["nvidia-smi", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                   "-lms", "200"]
            bus = self._bus_id()
            if bus:
                cmd += ["-i", bus]
            self.proc = subprocess.Popen(cmd, stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.flush()
        self.f.seek(0)
        rows = [l.strip().split(",") for l in self.f.read().splitlines() if l.strip()]
        os.unlink(self.f.name)
        sm, smax, pw, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            r = [x.strip() for x in r]
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
                pw.append(float(r[3]))
            except ValueError:
                continue
            for n, v in zip(names, r[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "power_w_max": max(pw), "samples": len(sm), "reasons": sorted(reasons)}


# --------------------------------------------------------------------------


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def setup(args):
    import torch
    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def _reduce(x: float, ws: int, op: str) -> float:
    """All-reduce one scalar over the ranks (host tensor for gloo, device
    tensor for nccl)."""
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


def max_over_ranks(x: float, ws: int) -> float:
    return _reduce(x, ws, "max")


def sum_over_ranks(x: float, ws: int) -> float:
    return _reduce(x, ws, "sum")


def prefill_flops(info, d_k, d_v):
    """Algorithmic and performed FLOPs: 2 d_k (scores) + 2 d_v (P V) per
    attended, resp. issued, (row, head, key) pair."""
    per_pair = 2 * d_k + 2 * d_v
    return per_pair * (info["pairs_global"] + info["pairs_local"]), per_pair * info["performed_pairs"]


def decode_bytes(wl):
    tot = 0
    for r in wl.requests:
        tot += r.T * wl.d_k * 2
        tot += wl.H * (wl.d_k * 2 + wl.d_v * 2 + 4)
    return tot


def bench_prefill(args, ws, local, pk):
    import torch
    from position_independent_kv_gb300 import binding as B
    from position_independent_kv_gb300.protected import build_bitmap
    from position_independent_kv_gb300.workloads import make_workload

    dev = torch.device("cuda", local)
    wl = make_workload(args.workload, seed=0, device=dev)
    bm, _ = build_bitmap(wl)
    stream = torch.cuda.current_stream(dev)
    plan = B.SegAttnPlan.from_workload(wl, bitmap=bm, stream=stream,
                                       flags=PLAN_FLAGS[args.kernel])
    info = plan.info
    ws_buf = None
    if plan.workspace_bytes:
        ws_buf = torch.empty(plan.workspace_bytes, dtype=torch.uint8, device=dev)
    out, lse = wl.out_init, wl.lse_init          # forward overwrites in place
    alg_flops, perf_flops = prefill_flops(info, wl.d_k, wl.d_v)

    for _ in range(args.warmup):
        plan.forward(wl.q, out, lse, ws_buf, stream=stream)
    torch.cuda.synchronize(dev)
    if plan.device_status(stream=stream) != 0:
        raise RuntimeError("device status error during warm-up")

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    barrier(ws)
    torch.cuda.synchronize(dev)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for i in range(args.steps):
        ev[i][0].record(stream)
        plan.forward(wl.q, out, lse, ws_buf, stream=stream)
        ev[i][1].record(stream)
    t1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(ws)
    clk = clocks.stop()
    total_ms = t0.elapsed_time(t1)
    launch_ms = [a.elapsed_time(b) for a, b in ev]
    if plan.device_status(stream=stream) != 0:
        raise RuntimeError("device status error in the timed region")

    # the side kernel beside the 4-CTA clusters: a prefill-only plan keeps its
    # work queue at the start of the workspace, whose counter's high half
    # counts the side kernel's claims in the last forward
    side_claims = 0
    if info["kernel"] == 3 and info["side_pairs"] and not info["split_chunks"] and ws_buf is not None:
        side_claims = (int(ws_buf[:8].cpu().view(torch.int64).item()) & ((1 << 64) - 1)) >> 32
    res = dict(total_ms=total_ms, launch_ms=launch_ms, info=info, alg_flops=alg_flops,
               perf_flops=perf_flops, clocks=clk, side_claims=side_claims,
               launches_per_step=(1 if info["dense_tiles"] else 0) + (1 if side_claims else 0) +
               (1 if info["split_chunks"] else 0))

    # end to end through the C ABI with host buffers (pinned), copies inside
    if not args.no_e2e:
        h_q = torch.empty(wl.q.shape, dtype=wl.q.dtype, pin_memory=True)
        h_q.copy_(wl.q)
        h_out = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
        h_out.copy_(out)
        h_lse = torch.empty(lse.shape, dtype=lse.dtype, pin_memory=True)
        h_lse.copy_(lse)
        h_lat = torch.empty(wl.latent_pool.shape, dtype=wl.latent_pool.dtype, pin_memory=True)
        h_lat.copy_(wl.latent_pool)
        torch.cuda.synchronize(dev)
        # in: q, lse and the latents (out is not uploaded: no kernel reads
        # it).  Out: lse and the written elements of out: the Global heads of
        # every row (one strided copy per row range) and the whole protected
        # rows, so the Global heads of protected rows travel twice and are
        # counted twice
        h2d = sum(t.numel() * t.element_size() for t in (h_q, h_lse, h_lat))
        o_head = wl.d_v * out.element_size()
        if info["num_local_heads"]:
            heads = info["protected_local_rows"] * wl.H + info["rows"] * info["num_global_heads"]
        else:
            heads = info["rows"] * wl.H
        d2h = heads * o_head + lse.numel() * lse.element_size()
        steps = max(1, min(args.steps, 3))
        # one untimed pass: the first device reads of freshly written host
        # pages are slower than the steady state
        wl.latent_pool.copy_(h_lat, non_blocking=True)
        plan.forward_host(h_q, h_out, h_lse, wl.q, out, lse, ws_buf, stream=stream)
        barrier(ws)
        torch.cuda.synchronize(dev)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            # latents to the device, then the forward from host q/out/lse
            # (its copies overlap its kernels; it returns the results to
            # h_out/h_lse before the stream continues)
            wl.latent_pool.copy_(h_lat, non_blocking=True)
            plan.forward_host(h_q, h_out, h_lse, wl.q, out, lse, ws_buf, stream=stream)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        barrier(ws)
        res["e2e_ms"] = e0.elapsed_time(e1) / steps
        res["h2d"] = h2d
        res["d2h"] = d2h
        del h_q, h_out, h_lse, h_lat
    plan.close()
    res["wl"] = wl
    res["q_bytes"] = wl.q.numel() * wl.q.element_size()
    res["o_bytes"] = wl.out_init.numel() * wl.out_init.element_size()
    return res


def bench_decode(args, local):
    import torch
    from position_independent_kv_gb300 import binding as B
    from position_independent_kv_gb300.protected import build_bitmap
    from position_independent_kv_gb300.workloads import make_workload

    dev = torch.device("cuda", local)
    wl = make_workload("decode", seed=0, device=dev)
    bm, _ = build_bitmap(wl)
    stream = torch.cuda.current_stream(dev)
    plan = B.SegAttnPlan.from_workload(wl, bitmap=bm, stream=stream)
    ws_buf = torch.empty(max(16, plan.workspace_bytes), dtype=torch.uint8, device=dev)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    out, lse = wl.out_init, wl.lse_init
    for _ in range(5):
        plan.forward(wl.q, out, lse, ws_buf, stream=stream)
    torch.cuda.synchronize(dev)
    times = []
    for _ in range(20):
        flush.zero_()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        plan.forward(wl.q, out, lse, ws_buf, stream=stream)
        b.record(stream)
        torch.cuda.synchronize(dev)
        times.append(a.elapsed_time(b))
    ok = plan.device_status(stream=stream) == 0
    byt = decode_bytes(wl)
    ms = statistics.median(times)
    info = plan.info
    plan.close()
    del flush
    return dict(ms=ms, bytes=byt, gbs=byt / (ms * 1e-3) / 1e9, ok=ok, info=info)


def bench_other_prefill(local: int, pk: dict, names=("flash", "varlen", "tiny")) -> dict:
    """The other prefill-shaped workloads on the default plan: device time per
    forward (CUDA events on the launching stream, 3 warm-ups, median of 20);
    algorithmic and performed TFLOP/s, attended pairs/s and the fraction of
    the bf16 peak.  Tiny fits in L2, so L2 is flushed (256 MB write) before
    each of its iterations; the others read more than L2 per forward."""
    import torch
    from position_independent_kv_gb300 import binding as B
    from position_independent_kv_gb300.protected import build_bitmap
    from position_independent_kv_gb300.workloads import make_workload
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    res = {}
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    for name in names:
        wl = make_workload(name, seed=0, device=dev)
        bm, _ = build_bitmap(wl)
        plan = B.SegAttnPlan.from_workload(wl, bitmap=bm, stream=stream)
        ws_buf = torch.empty(max(16, plan.workspace_bytes), dtype=torch.uint8, device=dev)
        out, lse = wl.out_init, wl.lse_init
        in_bytes = (wl.q.numel() * wl.q.element_size() + out.numel() * out.element_size())
        do_flush = in_bytes < 2 * 129 * 1024 * 1024
        for _ in range(3):
            plan.forward(wl.q, out, lse, ws_buf, stream=stream)
        torch.cuda.synchronize(dev)
        times = []
        for _ in range(20):
            if do_flush:
                flush.zero_()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            plan.forward(wl.q, out, lse, ws_buf, stream=stream)
            b.record(stream)
            torch.cuda.synchronize(dev)
            times.append(a.elapsed_time(b))
        ok = plan.device_status(stream=stream) == 0
        info = plan.info
        ms = statistics.median(times)
        alg, perf = prefill_flops(info, wl.d_k, wl.d_v)
        pairs = info["pairs_global"] + info["pairs_local"]
        kernel = {0: "mma_sync", 1: "tcgen05", 2: "tcgen05_pair", 3: "tcgen05_quad",
                  4: "tcgen05_small"}.get(info["kernel"], str(info["kernel"]))
        res[name] = {"workload": workload_desc(name), "ms": round(ms, 4),
                     "tflops": round(alg / (ms * 1e-3) / 1e12, 2),
                     "performed_tflops": round(perf / (ms * 1e-3) / 1e12, 2),
                     "pairs_per_s": pairs / (ms * 1e-3),
                     "frac_of_peak": round(alg / (ms * 1e-3) / 1e12 / pk["bf16_tflops"], 4),
                     "performed_frac_of_peak": round(perf / (ms * 1e-3) / 1e12 / pk["bf16_tflops"], 4),
                     "flop_per_pair": 2 * wl.d_k + 2 * wl.d_v, "attended_pairs": pairs,
                     "performed_pairs": info["performed_pairs"], "kernel": kernel,
                     "dense_tile_pairs": info.get("tc_pairs", info["dense_tiles"]),
                     "l2": "256 MB flush between iterations" if do_flush else
                           f"inputs larger than L2 ({in_bytes / 1e9:.2f} GB of Q + O), no flush",
                     "status_ok": ok}
        plan.close()
        del wl, out, lse, ws_buf
        torch.cuda.empty_cache()
    del flush
    return res


def bench_vrope(local: int, pk: dict) -> dict:
    """The rotary-value path (V = the whole latent row, output phase
    restored; d = 448 + 64): the long-context prefill (CUDA events, 3 warm-ups,
    median of 3 launches) and the decode batch (L2 flushed, median of 20)."""
    import torch
    from position_independent_kv_gb300 import binding as B
    from position_independent_kv_gb300.protected import build_bitmap
    from position_independent_kv_gb300.workloads import make_workload
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    res = {}
    ok = True
    for name in ("ctx128k_vrope", "decode_vrope"):
        wl = make_workload(name, seed=0, device=dev)
        bm, _ = build_bitmap(wl)
        plan = B.SegAttnPlan.from_workload(wl, bitmap=bm, stream=stream)
        ws_buf = torch.empty(max(16, plan.workspace_bytes), dtype=torch.uint8, device=dev)
        flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev) \
            if name.startswith("decode") else None
        out, lse = wl.out_init, wl.lse_init
        for _ in range(3):
            plan.forward(wl.q, out, lse, ws_buf, stream=stream)
        torch.cuda.synchronize(dev)
        times = []
        for _ in range(20 if flush is not None else 3):
            if flush is not None:
                flush.zero_()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            plan.forward(wl.q, out, lse, ws_buf, stream=stream)
            b.record(stream)
            torch.cuda.synchronize(dev)
            times.append(a.elapsed_time(b))
        ok = ok and plan.device_status(stream=stream) == 0
        ms = statistics.median(times)
        info = plan.info
        if flush is None:
            alg, perf = prefill_flops(info, wl.d_k, wl.d_v)
            res["prefill"] = {"workload": workload_desc(name), "ms": round(ms, 3),
                              "tflops": round(alg / (ms * 1e-3) / 1e12, 1),
                              "performed_tflops": round(perf / (ms * 1e-3) / 1e12, 1),
                              "frac_of_peak": round(alg / (ms * 1e-3) / 1e12 / pk["bf16_tflops"], 4),
                              "kernel": info["kernel"]}
        else:
            byt = decode_bytes(wl)
            gbs = byt / (ms * 1e-3) / 1e9
            res["decode"] = {"workload": workload_desc(name), "ms": round(ms, 4),
                             "GB/s": round(gbs, 1), "bytes": byt,
                             "frac_of_hbm": round(gbs / pk["hbm_gbs"], 4),
                             "l2": "256 MB flush between iterations"}
        plan.close()
        del wl, out, lse, ws_buf, flush
        torch.cuda.empty_cache()
    res["status_ok"] = ok
    res["flop_per_pair"] = 2 * 512 + 2 * 512
    return res


def bench_seg_paged(local: int, pk: dict, prefill: str = "qwen32b_128k") -> dict:
    """SegPagedAttention on GQA pages (Qwen3-32B shape, 1 Global KV head in
    8): the 128K-token prefill on the paged walk and on the dense + mask arm
    (CUDA events, 3 warm-ups, median of 3), and 64 decode steps whose Local
    heads keep only sink and window pages (L2 flushed, median of 20)."""
    import torch
    from position_independent_kv_gb300 import binding as B
    from position_independent_kv_gb300.paged_workloads import make_paged_workload
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    res = {}
    ok = True

    def timed(plan, pw, out, lse, n, flush=None):
        ws = torch.empty(max(16, plan.workspace_bytes), dtype=torch.uint8, device=dev)
        for _ in range(3):
            plan.forward(pw.q, pw.k_pages, pw.v_pages, out, lse, ws, stream=stream)
        torch.cuda.synchronize(dev)
        ts = []
        for _ in range(n):
            if flush is not None:
                flush.zero_()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            plan.forward(pw.q, pw.k_pages, pw.v_pages, out, lse, ws, stream=stream)
            b.record(stream)
            torch.cuda.synchronize(dev)
            ts.append(a.elapsed_time(b))
        return statistics.median(ts), plan.device_status(stream=stream) == 0

    pw = make_paged_workload(prefill, seed=0, device=dev)
    out = torch.empty((pw.rows, pw.Hq, 128), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((pw.rows, pw.Hq), dtype=torch.float32, device=dev)
    for flags, key in ((0, "prefill"), (B.RK_SEGPAGED_DENSE_MASK, "prefill_dense_mask")):
        plan = B.SegPagedPlan.from_workload(pw, flags=flags, stream=stream)
        info = plan.info
        ms, good = timed(plan, pw, out, lse, 3)
        ok = ok and good
        alg = 512.0 * info["pairs"]
        res[key] = {"ms": round(ms, 3), "tflops": round(alg / (ms * 1e-3) / 1e12, 1),
                    "performed_tflops": round(512.0 * info["performed_pairs"] / (ms * 1e-3) / 1e12, 1),
                    "frac_of_peak": round(alg / (ms * 1e-3) / 1e12 / pk["bf16_tflops"], 4),
                    "kv_blocks": info["kv_blocks"], "tiles": info["tiles"]}
        plan.close()
    res["prefill"]["workload"] = (f"{prefill}: 1 x {int(pw.seq_len[0])} tokens, 64 query heads over "
                                  "8 KV heads (d 128, 1 Global), per-head pages of 128 tokens, "
                                  "sink 4, w 256, bf16 N(0,1)/sqrt(128), seed 0")
    res["dense_mask_over_paged"] = round(res["prefill_dense_mask"]["ms"] / res["prefill"]["ms"], 2)
    del pw, out, lse
    torch.cuda.empty_cache()
    # relocated documents: the first 96K tokens are 48 documents of 2048
    # tokens cached alone (keys with RoPE at 0..2047), the query turns by
    # -delta; every tile on the one-sub-tile kernel
    pw = make_paged_workload("qwen32b_reloc_128k", seed=0, device=dev)
    out = torch.empty((pw.rows, pw.Hq, 128), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((pw.rows, pw.Hq), dtype=torch.float32, device=dev)
    plan = B.SegPagedPlan.from_workload(pw, stream=stream)
    info = plan.info
    ms, good = timed(plan, pw, out, lse, 3)
    ok = ok and good
    alg = 512.0 * info["pairs"]
    res["prefill_relocated"] = {
        "workload": "qwen32b_reloc_128k: the 128K prefill with 48 relocated documents of 2048 "
                    "tokens (keys cached at positions 0..2047, query turned by -delta) and a "
                    "32K tail", "ms": round(ms, 3),
        "tflops": round(alg / (ms * 1e-3) / 1e12, 1),
        "performed_tflops": round(512.0 * info["performed_pairs"] / (ms * 1e-3) / 1e12, 1),
        "frac_of_peak": round(alg / (ms * 1e-3) / 1e12 / pk["bf16_tflops"], 4),
        "tiles": info["tiles"]}
    plan.close()
    del pw, out, lse
    torch.cuda.empty_cache()
    pw = make_paged_workload("qwen32b_decode", seed=0, device=dev)
    out = torch.empty((pw.rows, pw.Hq, 128), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((pw.rows, pw.Hq), dtype=torch.float32, device=dev)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    plan = B.SegPagedPlan.from_workload(pw, stream=stream)
    ms, good = timed(plan, pw, out, lse, 20, flush)
    ok = ok and good
    # algorithmic bytes: the K and V rows each KV head's decode row sees, plus q, out, lse
    byt = 0
    for T in pw.seq_len:
        T = int(T)
        p = T - 1
        for g in range(pw.Hkv):
            n = p + 1 if pw.kv_role[g] else (p + 1 if max(0, p - pw.window) <= pw.sink
                                            else min(pw.sink, p + 1) + pw.window + 1)
            byt += n * 128 * 2 * 2
        byt += pw.Hq * (256 + 256 + 4)
    gbs = byt / (ms * 1e-3) / 1e9
    res["decode"] = {"workload": "qwen32b_decode: 64 requests x 1 row over 8K-64K tokens, Local "
                                 "heads keep sink + window pages only", "ms": round(ms, 4),
                     "GB/s": round(gbs, 1), "bytes": byt, "frac_of_hbm": round(gbs / pk["hbm_gbs"], 4),
                     "pages": pw.num_pages, "split_parts": plan.info["split_parts"],
                     "l2": "256 MB flush between iterations"}
    plan.close()
    del pw, out, lse, flush
    torch.cuda.empty_cache()
    res["status_ok"] = ok
    res["flop_per_pair"] = 512
    return res


def bench_protected_builder(name: str, local: int) -> dict:
    """rk_protected_build on a workload's geometry (device time per build,
    CUDA events, median of 20 after 3 warm-ups)."""
    import torch
    from position_independent_kv_gb300 import binding as B
    from position_independent_kv_gb300.workloads import make_geometry
    dev = torch.device("cuda", local)
    wl = make_geometry(name, 0)
    segs, begins = [], [0]
    for r in wl.requests:
        segs += [(s.n, s.delta, s.is_new) for s in r.segments]
        begins.append(len(segs))
    rows = sum(r.T for r in wl.requests)
    u = torch.from_numpy(np.concatenate([r.u for r in wl.requests]).astype(np.float64)).to(dev)
    sc = torch.empty(rows, dtype=torch.float32, device=dev).uniform_()
    bitmap = torch.empty(sum((r.T + 31) // 32 for r in wl.requests), dtype=torch.int32, device=dev)
    ws = torch.empty(B.protected_workspace_bytes(len(wl.requests), len(segs)), dtype=torch.uint8,
                     device=dev)
    ru = wl.rule
    args = (segs, begins, ru.boundary, ru.p_random, int(round(100 * ru.budget)), ru.none, u, sc,
            None, bitmap, ws)
    for _ in range(3):
        B.protected_build(*args)
    torch.cuda.synchronize(dev)
    times = []
    for _ in range(20):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        B.protected_build(*args)
        b.record()
        torch.cuda.synchronize(dev)
        times.append(a.elapsed_time(b))
    ms = statistics.median(times)
    return {"workload": name, "rows": rows, "requests": len(wl.requests), "ms": round(ms, 4),
            "rows_per_s": rows / (ms * 1e-3)}


def bench_projection(local: int, name: str = "ctx128k", dg: int = 1024, dm: int = 4096) -> dict:
    """rk_project_forward on the workload's rows and protected rows (random
    bf16 operands of those shapes): device time per call (CUDA events, median
    of 5 after 3 warm-ups), algorithmic and performed TFLOP/s."""
    import torch
    from position_independent_kv_gb300 import binding as B
    from position_independent_kv_gb300.protected import build_bitmap
    from position_independent_kv_gb300.workloads import make_geometry
    dev = torch.device("cuda", local)
    wl = make_geometry(name, 0)
    words, rows_prot = build_bitmap(wl)
    rows = sum(r.T - r.q_row_begin for r in wl.requests)
    prot = np.concatenate([p[r.q_row_begin:] for r, p in zip(wl.requests, rows_prot)])
    bits = np.zeros((rows + 31) // 32, np.uint32)
    idx = np.nonzero(prot)[0]
    np.bitwise_or.at(bits, idx // 32, (np.uint32(1) << (idx % 32).astype(np.uint32)))
    H, G = wl.H, wl.H // 8
    g = torch.Generator(device=dev).manual_seed(0)
    o = torch.randn(rows, H, 512, device=dev, generator=g).to(torch.bfloat16)
    z_off = torch.randn(rows, G, dg, device=dev, generator=g).to(torch.bfloat16)
    w_a = (torch.randn(G, dg, 4096, device=dev, generator=g) / 64.0).to(torch.bfloat16)
    w_b = (torch.randn(dm, G * dg, device=dev, generator=g) / (G * dg) ** 0.5).to(torch.bfloat16)
    z = torch.empty(rows, G * dg, dtype=torch.bfloat16, device=dev)
    y = torch.empty(rows, dm, dtype=torch.bfloat16, device=dev)
    pw = torch.from_numpy(bits.view(np.int32)).to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    role = wl.head_role
    for _ in range(3):
        B.project_forward(o, z_off, pw, w_a, w_b, z, y, role, status)
    torch.cuda.synchronize(dev)
    times = []
    for _ in range(5):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        B.project_forward(o, z_off, pw, w_a, w_b, z, y, role, status)
        b.record()
        torch.cuda.synchronize(dev)
        times.append(a.elapsed_time(b))
    ms = statistics.median(times)
    ngl = int(role.sum())  # Global heads
    nloc = H - ngl
    P = int(prot.sum())
    alg = 2.0 * dg * 512 * (rows * ngl + P * nloc) + 2.0 * rows * G * dg * dm
    # tiles holding a protected row run the Local part for all their 128 rows
    tiles_l = len(set((idx // 128).tolist()))
    perf = 2.0 * dg * 512 * (((rows + 127) // 128) * 128 * ngl + tiles_l * 128 * nloc) + \
        2.0 * ((rows + 127) // 128) * 128 * G * dg * dm
    ok = int(status.item()) == 0
    del o, z_off, w_a, w_b, z, y
    torch.cuda.empty_cache()
    return {"workload": f"{name} rows and protected rows, H={H}, d_v=512, d_g={dg}, "
                        f"d_model={dm}, random bf16 weights",
            "ms": round(ms, 3), "tflops": round(alg / (ms * 1e-3) / 1e12, 1),
            "performed_tflops": round(perf / (ms * 1e-3) / 1e12, 1), "status_ok": ok,
            "protected_rows": P, "rows": rows}


def cpu_baseline(wl, budget_s: float = 20.0):
    """The fp64 oracle on a bounded, stratified sample of the workload's rows
    (host cores; relocation of all keys included in the time)."""
    import torch
    import oracle as O
    from position_independent_kv_gb300.protected import build_bitmap
    bm, prot_rows = build_bitmap(wl)
    req = wl.requests[0]
    rng = np.random.default_rng(0)
    t_start = time.perf_counter()
    segs = [(s.latent.double().cpu().numpy(), s.delta, s.is_new) for s in req.segments]
    allp = np.arange(req.q_row_begin, req.T)
    order = rng.permutation(allp)
    rows_done, pairs, i = 0, 0, 0
    K, V = O.relocate([(l, d) for l, d, _ in segs], req.T, wl.d_nope, wl.rope_base)
    t_reloc = time.perf_counter() - t_start
    glob = np.nonzero(wl.head_role)[0]
    loc = np.nonzero(wl.head_role == 0)[0]
    new = np.zeros(req.T, bool)
    for s in req.segments:
        if s.is_new:
            new[s.delta:s.delta + s.n] = True
    prot = prot_rows[0] | new
    while time.perf_counter() - t_start < budget_s and i < len(order):
        p = int(order[i])
        i += 1
        q = wl.q[p - req.q_row_begin].double().cpu().numpy()
        O.attend(q[glob], K[:p + 1], V[:p + 1], wl.scale)
        pairs += len(glob) * (p + 1)
        if prot[p] and len(loc):
            keys = O.visible_keys(p, False, wl.sink, wl.window)
            O.attend(q[loc], K[keys], V[keys], wl.scale)
            pairs += len(loc) * len(keys)
        rows_done += 1
    el = time.perf_counter() - t_start
    per_pair = 2 * wl.d_k + 2 * wl.d_v
    return {"value": pairs * per_pair / el / 1e12, "unit": "TFLOP/s",
            "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{rows_done} random rows of the {wl.name} workload (all heads each), "
                      f"fp64 NumPy, key relocation ({t_reloc:.1f}s) included, {el:.1f}s"}


def run_ours(args):
    import torch
    ws, rank, local = setup(args)
    pk, pk_kind = peaks()
    if rank == 0:
        from position_independent_kv_gb300 import build as BUILD
        BUILD.build()
    barrier(ws)
    res = bench_prefill(args, ws, local, pk)
    ms_step = max_over_ranks(res["total_ms"] / args.steps, ws)
    flops_all = sum_over_ranks(res["alg_flops"], ws)
    value = flops_all / (ms_step * 1e-3) / 1e12
    perf_value = sum_over_ranks(res["perf_flops"], ws) / (ms_step * 1e-3) / 1e12
    launch_ms = statistics.mean(res["launch_ms"])
    achieved = res["alg_flops"] / (launch_ms * 1e-3) / 1e12
    e2e = None
    if "e2e_ms" in res:
        e2e_ms = max_over_ranks(res["e2e_ms"], ws)
        e2e = {"value": flops_all / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": int(res["h2d"]), "d2h_bytes_per_step": int(res["d2h"]),
               "ms_per_step": e2e_ms}
    wl = res.pop("wl")
    dec = None
    if not args.no_decode:
        dec = bench_decode(args, local)
    prot = None
    if not args.no_builder and rank == 0:
        prot = [bench_protected_builder(n, local) for n in ("ctx128k", "decode")]
    proj = None
    if not args.no_projection and rank == 0:
        proj = bench_projection(local, args.projection_workload)
    others = None
    if not args.no_others and rank == 0:
        others = bench_other_prefill(local, pk)
    vrope = None
    if not args.no_vrope and rank == 0:
        vrope = bench_vrope(local, pk)
    paged = None
    if not args.no_paged and rank == 0:
        paged = bench_seg_paged(local, pk, args.paged_prefill)
    line = None
    if rank == 0:
        info = res["info"]
        kernel = {0: "mma_sync", 1: "tcgen05", 2: "tcgen05_pair", 3: "tcgen05_quad",
                  4: "tcgen05_small"}[info["kernel"]]
        peak = pk["bf16_tflops"]
        line = {
            "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": workload_desc(args.workload), "name": args.workload,
                       "parallelism": f"replicas{ws}",
                       "l2": (f"inputs larger than L2 (Q {res['q_bytes'] / 1e9:.1f} GB + "
                              f"O {res['o_bytes'] / 1e9:.1f} GB per step), no flush"),
                       "kernel": kernel, "dense_tiles": info["dense_tiles"],
                       "side_pairs": info["side_pairs"], "side_claims": res["side_claims"],
                       "pairs_global": info["pairs_global"], "pairs_local": info["pairs_local"],
                       "performed_pairs": info["performed_pairs"]},
            "performed_tflops": round(perf_value, 3),
            "performed_frac_of_peak": round(perf_value / ws / peak, 4),
            "pairs_per_s": (info["pairs_global"] + info["pairs_local"]) * ws / (ms_step * 1e-3),
            "roofline": {"bound": "tensor", "achieved": round(achieved, 3), "peak": peak,
                         "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                         "peak_kind": f"{pk_kind} bf16 burst",
                         "frac_of_sustained": round(achieved / pk.get("bf16_tflops_sustained", peak), 4),
                         "traffic": recorded_traffic(kernel, args.workload),
                         "kernel": f"{kernel} dense tiles" +
                                   (" + side CTA pairs" if res["side_claims"] else "")},
            "gpu_launches": res["launches_per_step"] * args.steps,
            "clocks": res["clocks"],
        }
        if e2e:
            line["e2e"] = e2e
        if prot:
            line["protected_builder"] = prot
        if proj:
            proj["frac_of_peak"] = round(proj["tflops"] / peak, 4)
            line["projection"] = proj
        if others:
            line["configs"] = others
        if vrope:
            line["v_rope"] = vrope
        if paged:
            line["seg_paged_gqa"] = paged
        if dec:
            line["decode"] = {"workload": "64 requests x 1 row, 4-32 segments, 8K-64K keys, "
                                          "H=64 (56/8), split over segments + fused LSE merge",
                              "GB/s": round(dec["gbs"], 1), "ms": round(dec["ms"], 4),
                              "bytes": dec["bytes"], "frac_of_hbm": round(dec["gbs"] / pk["hbm_gbs"], 4),
                              "hbm_peak": pk["hbm_gbs"], "split_chunks": dec["info"]["split_chunks"],
                              "l2": "256 MB flush between iterations"}
        if not args.no_cpu:
            line["cpu_baseline"] = cpu_baseline(wl, budget_s=args.cpu_seconds)
        print(json.dumps(line), flush=True)
    barrier(ws)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_reference(args):
    """The oracle, as it stands, on the host cores: each step is a bounded
    sample of the same workload (rows of the 128K request)."""
    ws, rank, local = dist_env()
    if rank != 0:
        return
    import torch
    from position_independent_kv_gb300.workloads import make_workload
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    if dev == "cuda":
        torch.cuda.set_device(local)
    wl = make_workload(args.workload, seed=0, device=dev, with_out=False)
    per = max(2.0, args.cpu_seconds / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        cpu_baseline(wl, budget_s=per)
    vals = []
    t0 = time.perf_counter()
    last = None
    for _ in range(args.steps):
        last = cpu_baseline(wl, budget_s=per)
        vals.append(last["value"])
    el = time.perf_counter() - t0
    v = statistics.mean(vals)
    line = {"metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference",
            "config": {"workload": workload_desc(args.workload), "name": args.workload},
            "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": last["cores"],
                             "kind": "oracle", "sample": last["sample"]},
            "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--kernel", default="auto", choices=list(PLAN_FLAGS),
                    help="prefill tile kernel: auto (4-CTA clusters where eligible, with the "
                         "side kernel on the SMs they leave free), noside (4-CTA clusters "
                         "alone), pair (tile pairs per half of d_v), single (one tile per two "
                         "CTAs), legacy (mma.sync)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-projection", action="store_true",
                    help="skip the timing of the projected-state / W_b step")
    ap.add_argument("--no-paged", action="store_true",
                    help="skip the timing of SegPagedAttention on GQA pages")
    ap.add_argument("--paged-prefill", default="qwen32b_128k",
                    help="paged workload of the SegPagedAttention prefill timing")
    ap.add_argument("--no-others", action="store_true",
                    help="skip the timing of the flash-like, variable-length and tiny workloads")
    ap.add_argument("--no-vrope", action="store_true",
                    help="skip the timing of the rotary-value (output-phase restore) path")
    ap.add_argument("--projection-workload", default="ctx128k",
                    help="rows and protected rows of this workload feed the projection step")
    ap.add_argument("--no-builder", action="store_true",
                    help="skip the timing of the on-device protected-row builder")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=20.0)
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()

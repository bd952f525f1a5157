#!/usr/bin/env python
"""CSA2 sparse-attention decode benchmark.

One step = one pass of the whole hot path over one batch: the Full-mode CSA2
layer of the 32-query, 64K-token-context decode workload (indexer scores over
16384 FP4/FP8 entries per query, top-2048, gather + dequantise + 64-head MQA
attention, split combine), replayed as one CUDA graph of csa2_layer_group.
Inputs are resident in HBM; L2 is flushed (512 MiB write) before every timed
step and each step is timed with its own CUDA events.

Prints one JSON line (rank 0).  `--impl reference` times the CPU oracle on a
bounded sample of the same workload instead.  Under torchrun every rank runs
an independent replica (the path has no data exchange); the reported value is
the queries of all ranks over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "CSA2 query-tokens/s per layer at 64K ctx; % of GB300 HBM roofline"
UNIT = "query-tokens/s"
DEFAULT_WORKLOAD = "decode_b32_ctx64k"
FLUSH_BYTES = 512 << 20


class L2Flush:
    """Writes a 512 MiB buffer (evicts everything), then reads a 256 MiB one so
    that L2 is left holding clean lines: the timed kernel then pays no
    write-back of the flush's dirty lines."""

    def __init__(self, device):
        import torch
        self.w = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=device)
        self.r = torch.ones(FLUSH_BYTES // 2 // 4, dtype=torch.int32, device=device)

    def __call__(self):
        self.w.zero_()
        self.r.max()


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="csa2", choices=["csa2", "reference"])
    p.add_argument("--workload", default=DEFAULT_WORKLOAD)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--kernel-loop", default="",
                   help="run only this many launches of the layer group (for profilers)")
    return p.parse_args()


def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def allreduce_max(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if dist.get_backend() == "nccl" else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def step_throughput(B: int, steps: int, world: int, total_s: float, n_layers: int) -> float:
    """Whole-job query-tokens/s per layer: every rank runs `steps` steps of B queries
    through n_layers layers; total_s is the slowest rank's time (max over ranks)."""
    return B * steps * world * n_layers / total_s


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d.get("bf16_tflops", 1900.0)), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle samples every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.dev = device_index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.dev)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        busy = [x for x in sm if smax and x > 0.5 * smax] or sm
        return {"sm_mhz": statistics.median(busy) if busy else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def algorithmic_bytes(w):
    """Per step: indexer K of every scored entry, indexer q, selected FP4 rows,
    SWA window rows, main queries (bf16) and outputs (fp32), as the workload's
    layers read them."""
    from sparse_attention_decode_csa2_gb300.synthetic import FULL, REINDEX, REUSE
    B, N, k = w.B, w.N, w.k
    total = 0
    per_layer = []
    for l, m in enumerate(w.modes):
        b = B * k * w.row_bytes + B * w.H * w.D * 2 + B * w.H * w.D * 4
        if m == FULL or (m == REINDEX and not w.pool):
            n_scored = sum(min(N, (int(p) + 1) // w.ratio) for p in w.q_pos())
            b += n_scored * w.idx_row_bytes + B * w.H_I * w.idx_row_bytes
            if w.q_per_seq > 1:   # one shared context: its K is read once
                b -= n_scored * w.idx_row_bytes
                b += w.n_seq * N * w.idx_row_bytes
        elif m == REINDEX:
            b += B * w.pool * (w.idx_row_bytes + 4) + B * w.H_I * w.idx_row_bytes
        if w.n_win:   # each query's SWA window (E4M3 rows of D bytes)
            b += sum(min(w.n_win, int(p) + 1) for p in w.q_pos() if p >= 0) * w.D
        per_layer.append(b)
        total += b
    return total, per_layer


QUANT_D_MX = 128   # indexer-key width the MXFP4 packer is timed on


def kernel_bytes(w):
    """Algorithmic bytes of each timed component op (one launch over the batch;
    the packers over the whole cache of the workload: fp32 read + packed write)."""
    B, N, k = w.B, w.N, w.k
    n_scored = sum(min(N, (int(p) + 1) // w.ratio) for p in w.q_pos())
    n_win = sum(min(w.n_win, int(p) + 1) for p in w.q_pos() if p >= 0) if w.n_win else 0
    rows = w.n_seq * N
    # queries sharing one context read its indexer K once
    k_bytes = (w.n_seq * N if w.q_per_seq > 1 else n_scored) * w.idx_row_bytes
    return {
        "quantize_kv_fp4": rows * (w.D * 4 + w.row_bytes),
        "quantize_mxfp4": rows * (QUANT_D_MX * 4 + QUANT_D_MX // 2 + QUANT_D_MX // 32),
        "index_scores": k_bytes + B * w.H_I * w.idx_row_bytes + B * N * 4,
        "topk": n_scored * 4 + B * k * 4,
        "sparse_attn_fp4": B * k * (w.row_bytes + 4) + n_win * w.D + B * w.H * w.D * (2 + 4) +
                           B * w.H * 4,
    }


def attn_flops(w):
    return 4.0 * w.B * w.H * (w.k + w.n_win) * w.D


def kernel_flops(w):
    """Tensor-core work of the contractions (2 flops per multiply-add): the
    indexer's FP8 products of every visible entry, the attention's QK^T and PV."""
    n_scored = sum(min(w.N, (int(p) + 1) // w.ratio) for p in w.q_pos())
    return {"index_scores": 2.0 * n_scored * w.H_I * w.D_I, "sparse_attn_fp4": attn_flops(w)}


def run_gpu(args, rank, world, local):
    import numpy as np
    import torch
    from sparse_attention_decode_csa2_gb300 import build
    if rank == 0 or not os.path.exists(build.LIB_PATH):
        build.build()
    barrier(world)
    from sparse_attention_decode_csa2_gb300 import csa2, workload
    from sparse_attention_decode_csa2_gb300.synthetic import FULL, REINDEX, REUSE, WORKLOADS

    w = WORKLOADS[args.workload]
    dev = torch.device("cuda", torch.cuda.current_device())
    inp = workload.prepare(w, device=dev)
    lg = inp.layer_group(reuse_idx_copy=False)
    flush = L2Flush(dev)

    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        for _ in range(2):
            lg()
    stream.synchronize()
    code, bits = csa2.read_status(lg.ws)
    if code != 0:
        raise RuntimeError(f"device status {bits} after warm-up")
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        lg()
    torch.cuda.synchronize()

    if args.kernel_loop:
        for _ in range(int(args.kernel_loop)):
            flush()
            graph.replay()
        torch.cuda.synchronize()
        return None

    K, W = args.steps, args.warmup
    for _ in range(W):
        flush()
        graph.replay()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(K)]
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    cur = torch.cuda.current_stream()
    for i in range(K):
        flush()
        ev[i][0].record(cur)
        graph.replay()
        ev[i][1].record(cur)
    torch.cuda.synchronize()
    barrier(world)
    t_wall = time.perf_counter() - t_wall
    step_ms = [a.elapsed_time(b) for a, b in ev]

    # component ops, each timed alone over the same batch (L2 flushed before each)
    comp = {}
    scores = torch.empty((w.B, w.N), dtype=torch.float32, device=dev)
    idx = torch.empty((w.B, w.k), dtype=torch.int32, device=dev)
    out = torch.empty((w.B, w.H, w.D), dtype=torch.float32, device=dev)
    lse = torch.empty((w.B, w.H), dtype=torch.float32, device=dev)
    ws = csa2.make_workspace(w.B, w.N, w.k, w.H, w.pool, dev)
    ops = {
        "index_scores": (lambda: csa2.index_scores_mxfp4(
            inp.qi[0], inp.ki_fp8, w.N, w.kv_seq_stride, w.q_per_seq, inp.q_pos, w.ratio,
            out=scores)) if w.indexer_fmt else
        (lambda: csa2.index_scores(inp.qi[0], inp.ki_fp8, w.N, w.kv_seq_stride, w.q_per_seq,
                                   inp.q_pos, w.ratio, out=scores)),
        "topk": lambda: csa2.topk(scores, w.k, inp.q_pos, w.ratio, ws, out=idx),
        "sparse_attn_fp4": (lambda: csa2.sparse_attn_fp4_swa(
            inp.q[0], inp.kv_fp4, w.N, w.kv_seq_stride, w.q_per_seq, idx, inp.swa[0], w.n_win,
            inp.q_pos, inp.scale, out=out, lse=lse, ws=ws)) if w.n_win else
        (lambda: csa2.sparse_attn_fp4(inp.q[0], inp.kv_fp4, w.N, w.kv_seq_stride, w.q_per_seq,
                                      idx, inp.scale, out=out, lse=lse, ws=ws)),
    }
    # the packers, over the workload's whole cache (timed alone, not in the step)
    qrows = w.n_seq * w.N
    qx = torch.randn((qrows, w.D), dtype=torch.float32, device=dev)
    qo = torch.empty((qrows, w.row_bytes), dtype=torch.uint8, device=dev)
    mx = torch.randn((qrows, QUANT_D_MX), dtype=torch.float32, device=dev)
    mo = torch.empty((qrows, QUANT_D_MX // 2 + QUANT_D_MX // 32), dtype=torch.uint8, device=dev)
    ops["quantize_kv_fp4"] = lambda: csa2.quantize_kv_fp4(qx, out=qo)
    ops["quantize_mxfp4"] = lambda: csa2.quantize_mxfp4(mx, out=mo)
    for name, fn in ops.items():
        fn()
        torch.cuda.synchronize()
        e = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(K)]
        for i in range(K):
            flush()
            e[i][0].record(cur)
            fn()
            e[i][1].record(cur)
        torch.cuda.synchronize()
        comp[name] = statistics.mean(a.elapsed_time(b) for a, b in e)
    clocks = sampler.stop()
    del qx, qo, mx, mo

    # end to end through the public API with host buffers.  The FP4 cache, the
    # indexer K and the SWA rings are state that stays resident across decode
    # steps; what a step brings in from the host is its queries (main and
    # indexer, every layer), their positions and the cache entries its tokens
    # append: the new main-KV entries as fp32 latent rows (packed into FP4 on
    # the device), their indexer keys and each layer's SWA ring row of the
    # newest token.  All of it sits in one pinned buffer that csa2_upload moves
    # with one copy and places with one kernel; then the layer group runs and
    # every layer's output is copied back.  The step is timed twice: issued
    # call by call, and as one CUDA graph per step (the graph's copy nodes read
    # and write the pinned host buffers on every replay).
    e2e = None
    if not args.no_e2e:
        from sparse_attention_decode_csa2_gb300 import csa2 as _c
        S, N = w.n_seq, w.N
        pos = w.q_pos()
        ents = np.clip(pos.astype(np.int64) // w.ratio, 0, N - 1)
        e_lo, e_hi = int(ents.min()), int(ents.max())
        kv3 = inp.kv_fp4.view(S, N, w.row_bytes)
        ki3 = inp.ki_fp8.view(S, N, w.idx_row_bytes)
        segs, fills = [], []
        rows = np.arange(e_lo, e_hi + 1)
        if e_lo == e_hi:   # one appended entry per sequence, at the same index
            segs.append((_c.UPLOAD_KV_FP4, kv3[:, e_lo]))
            fills.append(np.concatenate([w.kv_latent_rows(s_, rows) for s_ in range(S)]))
            segs.append((_c.UPLOAD_RAW, ki3[:, e_lo]))
            fills.append(ki3[:, e_lo].cpu().numpy())
        else:
            for s_ in range(S):
                segs.append((_c.UPLOAD_KV_FP4, kv3[s_, e_lo:e_hi + 1]))
                fills.append(w.kv_latent_rows(s_, rows))
                segs.append((_c.UPLOAD_RAW, ki3[s_, e_lo:e_hi + 1]))
                fills.append(ki3[s_, e_lo:e_hi + 1].cpu().numpy())
        if w.n_win:
            r_lo, r_hi = int(pos.min()) % w.swa_ring, int(pos.max()) % w.swa_ring
            if r_hi - r_lo == int(pos.max() - pos.min()):
                for t in inp.swa:   # the ring rows of the step's tokens
                    for s_ in range(S):
                        segs.append((_c.UPLOAD_RAW, t[s_, r_lo:r_hi + 1]))
                        fills.append(t[s_, r_lo:r_hi + 1].cpu().numpy())
        cache_segs, cache_fills = list(segs), list(fills)
        # the main queries (most of the bytes; first read by the attention)
        # travel on a side stream, beside the indexer and the top-k
        q_segs = [(_c.UPLOAD_RAW, t.view(-1, 512)) for t in inp.q]
        q_fills = [t.view(-1, 512).cpu().numpy() for t in inp.q]
        for t in inp.qi:
            if t is not None:
                v = t.view(t.shape[0], -1)
                segs.append((_c.UPLOAD_RAW, v))
                fills.append(v.cpu().numpy())
        segs.append((_c.UPLOAD_RAW, inp.q_pos.view(1, -1)))
        fills.append(inp.q_pos.view(1, -1).cpu().numpy())
        up = _c.StepUpload(segs, device=dev)
        up_q = _c.StepUpload(q_segs, device=dev)
        for u, fl in ((up, fills), (up_q, q_fills)):
            for pay, f in zip(u.payloads, fl):
                pay.copy_(torch.from_numpy(np.ascontiguousarray(f)).view(pay.dtype).view(pay.shape))
        side = torch.cuda.Stream(device=dev)
        ev_q = torch.cuda.Event()
        ev_q.record(side)                       # the event exists before the group names it
        lg2 = inp.layer_group(reuse_idx_copy=False, q_ready=ev_q)
        host_out = [torch.empty_like(o, device="cpu").pin_memory() for o in lg2.out]
        ref_out = [o.clone() for o in lg.out]
        h2d = up.bytes + up_q.bytes
        d2h = sum(o.numel() * 4 for o in host_out)

        def e2e_step():
            main = torch.cuda.current_stream()
            side.wait_stream(main)              # the last step's attention has read the queries
            with torch.cuda.stream(side):
                up_q()
                ev_q.record(side)
            up()
            outs, _, _, _ = lg2()               # its attention waits for ev_q
            for h, o in zip(host_out, outs):
                h.copy_(o, non_blocking=True)

        for _ in range(max(1, min(W, 3))):
            e2e_step()
        torch.cuda.synchronize()
        # the uploaded step reproduces the resident one (appended rows packed
        # on the device are the cache's own bytes)
        same = all(torch.equal(h, r.cpu()) for h, r in zip(host_out, ref_out))
        Ke = max(3, min(K, 10))

        def timed(step):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            barrier(world)
            e0.record(cur)
            for _ in range(Ke):
                step()
            e1.record(cur)
            torch.cuda.synchronize()
            return allreduce_max(e0.elapsed_time(e1) / 1e3, world)

        # the transfers alone (same buffers, same stream): where the e2e time goes
        def d2h_only():
            for h, o in zip(host_out, lg2.out):
                h.copy_(o, non_blocking=True)

        parts = {"upload_ms": timed(up) / Ke * 1e3, "upload_q_ms": timed(up_q) / Ke * 1e3,
                 "d2h_ms": timed(d2h_only) / Ke * 1e3}
        eager_s = timed(e2e_step)
        eager_v = step_throughput(w.B, Ke, world, eager_s, len(w.modes))
        e2e = {"value": eager_v, "unit": UNIT, "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "eager_value": eager_v,
               "inputs": ("queries, positions and the appended entries (main KV as fp32 latent, "
                          "packed to FP4 on the device; indexer keys; SWA rows) in two pinned "
                          "buffers, each one copy + one placing kernel: the main queries on a "
                          "side stream the attention waits for, the rest before the indexer; "
                          "cache resident"),
               "outputs_match_resident_run": bool(same),
               "parts_ms": parts,
               "h2d_gbs": h2d / ((parts["upload_ms"] + parts["upload_q_ms"]) / 1e3) / 1e9,
               "d2h_gbs": d2h / (parts["d2h_ms"] / 1e3) / 1e9,
               "issue": "call by call"}
        try:
            g_e2e = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g_e2e, stream=stream):
                e2e_step()
            torch.cuda.synchronize()
            for _ in range(max(1, min(W, 3))):
                g_e2e.replay()
            torch.cuda.synchronize()
            graph_s = timed(g_e2e.replay)
            graph_v = step_throughput(w.B, Ke, world, graph_s, len(w.modes))
            e2e["graph_value"] = graph_v
            # the value is the faster of the two ways a caller can issue the
            # step (both go through the same calls and buffers); the
            # host-link copies of the large prompt-shaped steps have run
            # slower inside the graph on some boxes
            if graph_v >= eager_v:
                e2e["value"] = graph_v
                e2e["issue"] = ("one CUDA graph per step: packed uploads, layer group, copies "
                                "out (eager_value: the same step issued call by call)")
            else:
                e2e["issue"] = ("call by call, faster here than the same step as one CUDA "
                                "graph (graph_value)")
        except RuntimeError as ex:  # keep the call-by-call number, say why
            torch.cuda.synchronize()
            e2e["issue"] = f"call by call (graph capture failed: {str(ex).splitlines()[0]})"

        # Steps in flight together, as a serving loop runs them: two sets of
        # the per-step buffers (queries, positions, outputs).  On an upload
        # stream step i brings in its main queries while step i - 1 computes,
        # then (once step i - 1 has read the cache) its packed appended rows,
        # indexer queries and positions; its layer group runs on the compute
        # stream; a download stream copies its outputs out while step i + 1
        # computes.  Thirty-two such steps are one CUDA graph (launching them one
        # call at a time keeps the host busier than the GPU); the graph's
        # replays follow one another, so one step boundary in thirty-two does not
        # overlap.  Every step still moves all its bytes in and out.
        try:
            sets = []
            for b_ in range(2):
                if b_ == 0:
                    qb, qib, pb = inp.q, inp.qi, inp.q_pos
                else:
                    qb = [t.clone() for t in inp.q]
                    qib = [None if t is None else t.clone() for t in inp.qi]
                    pb = inp.q_pos.clone()
                lgb = _c.LayerGroup(w.modes, qb, qib, inp.kv_fp4, inp.ki_fp8, w.N,
                                    w.kv_seq_stride, w.q_per_seq, pb, w.ratio, w.k, w.pool,
                                    inp.scale, reuse_idx_copy=False, pool_block=w.pool_block,
                                    swa_kv=inp.swa, n_win=w.n_win, indexer_fmt=w.indexer_fmt)
                sg, fl = list(cache_segs), list(cache_fills)
                for t in qib:
                    if t is not None:
                        v = t.view(t.shape[0], -1)
                        sg.append((_c.UPLOAD_RAW, v))
                        fl.append(v.cpu().numpy())
                sg.append((_c.UPLOAD_RAW, pb.view(1, -1)))
                fl.append(pb.view(1, -1).cpu().numpy())
                upb = _c.StepUpload(sg, device=dev)
                upqb = _c.StepUpload([(_c.UPLOAD_RAW, t.view(-1, 512)) for t in qb], device=dev)
                for u, fl_ in ((upb, fl), (upqb, q_fills)):
                    for pay, f in zip(u.payloads, fl_):
                        pay.copy_(torch.from_numpy(np.ascontiguousarray(f)).view(pay.dtype)
                                  .view(pay.shape))
                hob = [torch.empty_like(o, device="cpu").pin_memory() for o in lgb.out]
                sets.append(dict(up_q=upqb, up=upb, lg=lgb, out=lgb.out, host=hob))
            s_up, s_dn = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
            n_cap = 32
            evs = [{k_: torch.cuda.Event() for k_ in ("up", "c", "d")} for _ in range(n_cap)]
            for st_ in sets:   # first launches (library set-up) outside the capture
                st_["lg"]()
            torch.cuda.synchronize()
            g_p = torch.cuda.CUDAGraph()
            def copy_out(i):
                st_ = sets[i & 1]
                with torch.cuda.stream(s_dn):
                    s_dn.wait_event(evs[i]["c"])
                    if i + 1 < n_cap:   # the next step's small upload goes first on the link
                        s_dn.wait_event(evs[i + 1]["up"])
                    for h, o in zip(st_["host"], st_["out"]):
                        h.copy_(o, non_blocking=True)
                    evs[i]["d"].record(s_dn)

            with torch.cuda.graph(g_p, stream=stream):
                s_up.wait_stream(stream)
                s_dn.wait_stream(stream)
                for i in range(n_cap):
                    st_ = sets[i & 1]
                    with torch.cuda.stream(s_up):
                        if i >= 2:
                            s_up.wait_event(evs[i - 2]["c"])   # step i - 2 has read the queries
                        st_["up_q"]()
                        if i >= 1:
                            s_up.wait_event(evs[i - 1]["c"])   # step i - 1 has read the cache
                        st_["up"]()
                        evs[i]["up"].record(s_up)
                    stream.wait_event(evs[i]["up"])
                    if i >= 2:
                        stream.wait_event(evs[i - 2]["d"])     # step i - 2's outputs are out
                    st_["lg"]()
                    evs[i]["c"].record(stream)
                    if i >= 1:
                        copy_out(i - 1)
                copy_out(n_cap - 1)
                stream.wait_stream(s_up)
                stream.wait_stream(s_dn)
            torch.cuda.synchronize()
            for _ in range(max(1, min(W, 3))):
                g_p.replay()
            torch.cuda.synchronize()
            same_p = all(torch.equal(h, r.cpu()) for st_ in sets
                         for h, r in zip(st_["host"], ref_out))
            reps = max(2, (Ke + n_cap - 1) // n_cap)
            e0p, e1p = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            barrier(world)
            e0p.record(cur)
            for _ in range(reps):
                g_p.replay()
            e1p.record(cur)
            torch.cuda.synchronize()
            piped_s = allreduce_max(e0p.elapsed_time(e1p) / 1e3, world)
            piped_v = step_throughput(w.B, reps * n_cap, world, piped_s, len(w.modes))
            e2e["pipelined_value"] = piped_v
            e2e["pipelined_outputs_match_resident_run"] = bool(same_p)
            if same_p and piped_v > e2e["value"]:
                e2e["value"] = piped_v
                e2e["issue"] = ("steps in flight together: per step the queries' upload, then the "
                                "packed rest, on an upload stream, the layer group on the compute "
                                "stream, the outputs' copy on a download stream; thirty-two "
                                "steps per CUDA graph (graph_value / eager_value: one step at a "
                                "time)")
            del g_p, sets
        except RuntimeError as ex:
            torch.cuda.synchronize()
            e2e["pipelined_value"] = None
            e2e["pipelined_error"] = str(ex).splitlines()[0]

    total_s = allreduce_max(sum(step_ms) / 1e3, world)
    ms_per_step = total_s * 1e3 / K
    value = step_throughput(w.B, K, world, total_s, len(w.modes))

    hbm_peak, bf16_peak, peak_src = measured_peaks()
    step_bytes, _ = algorithmic_bytes(w)
    kb = kernel_bytes(w)
    step_ops = ("index_scores", "topk", "sparse_attn_fp4")
    dom = max(step_ops, key=comp.get)   # the step's dominant kernel
    kernels_frac = {n: kb[n] / (comp[n] / 1e3) / 1e9 / hbm_peak for n in comp}
    # queries sharing one context (prefill-shaped): the rows are L2-resident
    # and the contractions bind (fp8 indexer products at twice the bf16 rate)
    kf = kernel_flops(w)
    if w.q_per_seq > 1 and dom in kf:
        t_peak = bf16_peak * (2.0 if dom == "index_scores" else 1.0)
        achieved = kf[dom] / (comp[dom] / 1e3) / 1e12
        roof = {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": t_peak,
                "unit": "TFLOP/s", "frac": achieved / t_peak, "traffic": None,
                "peak_source": peak_src + (" (fp8: bf16 x 2, the nominal ratio)"
                                           if dom == "index_scores" else " (bf16 burst)")}
    else:
        achieved = kb[dom] / (comp[dom] / 1e3) / 1e9
        roof = {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": hbm_peak,
                "unit": "GB/s", "frac": achieved / hbm_peak, "traffic": None,
                "peak_source": peak_src}
    traffic = None
    tpath = os.path.join(ROOT, "profiles", "traffic.json")
    if os.path.exists(tpath):
        try:
            with open(tpath) as f:
                t = json.load(f)
            rec = t.get(args.workload, {}).get(dom)
            if rec and rec.get("kernel_rev") == kernel_revision():
                traffic = rec.get("bytes_per_launch")
                roof["traffic"] = traffic
        except Exception:
            traffic = None
    n_launch = csa2.group_launches(lg)
    res = {
        "metric": METRIC,
        "value": value,
        "unit": UNIT,
        "n_gpus": world,
        "steps": K,
        "warmup": W,
        "ms_per_step": ms_per_step,
        "step_ms_quantiles": step_quantiles(step_ms),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": ("fp16-mma/fp32-acc (fp4 KV, mxfp4 indexer)" if w.indexer_fmt else
                  "fp16-mma/fp32-acc (fp4 KV, e4m3 indexer)"),
        "data": ("synthetic (seeded SplitMix64: N(0,1) latent -> FP4, MXFP4 indexer rows drawn "
                 "in format, bf16 N(0,1) queries)" if w.indexer_fmt else
                 "synthetic (seeded SplitMix64: N(0,1) latent -> FP4, "
                 + ("bf16 N(0,1)" if w.float_indexer else "integer") + " E4M3 indexer, "
                 "bf16 N(0,1) queries)"),
        "config": {"workload": w.name, "queries": w.B, "entries_per_seq": w.N,
                   "ctx_tokens": w.N * w.ratio, "heads": w.H, "indexer_heads": w.H_I,
                   "top_k": w.k, "modes": [["FULL", "REINDEX", "REUSE"][m] for m in w.modes],
                   "indexer": "mxfp4" if w.indexer_fmt else "e4m3",
                   "l2": "flushed before every timed step (512 MiB write, then 256 MiB read)",
                   "cuda_graph": True, "parallelism": f"replicas x{world}"},
        "step_bytes": step_bytes,
        "hbm_frac_step": (step_bytes / (ms_per_step / 1e3) / 1e9) / hbm_peak,
        "roofline": roof,
        "kernels_ms": comp,
        "kernels_hbm_frac": kernels_frac,
        "kernels_bytes": {n: int(kb[n]) for n in comp},
        "attn_tflops": attn_flops(w) / (comp["sparse_attn_fp4"] / 1e3) / 1e12,
        "gpu_launches": n_launch * K,
        "clocks": clocks,
        "e2e": e2e,
        "wall_s": t_wall,
    }
    return res


def step_quantiles(step_ms) -> dict:
    """p10 / median / p90 of this rank's timed steps (ms), nearest-rank."""
    xs = sorted(float(x) for x in step_ms)
    if not xs:
        return {}
    pick = lambda q: xs[min(len(xs) - 1, max(0, math.ceil(q * len(xs)) - 1))]
    return {"p10": pick(0.10), "p50": pick(0.50), "p90": pick(0.90)}


def kernel_revision() -> str:
    import hashlib
    h = hashlib.sha1()
    d = os.path.join(ROOT, "sparse_attention_decode_csa2_gb300", "csrc")
    for n in sorted(os.listdir(d)):
        with open(os.path.join(d, n), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:12]


# ---------------------------------------------------------------------------
# CPU oracle (baseline and reference arm)
# ---------------------------------------------------------------------------

class OracleSample:
    """The oracle's inputs for queries of a workload, prepared outside any timing."""

    def __init__(self, w, queries):
        import oracle
        self.oracle = oracle
        self.w = w
        self.items = []
        cache = {}
        for q in queries:
            s = q // w.q_per_seq
            if s not in cache:
                cache[s] = (oracle.quantize_kv_fp4(w.kv_latent(s)), w.ki_rows(s))
            kv, ki = cache[s]
            L = len(w.modes)
            self.items.append(dict(q=q, kv=kv, ki=ki, qpos=w.q_pos()[q:q + 1],
                                   qb=[w.q_bf16(l, [q]) for l in range(L)],
                                   qi=[w.qi_rows(l, [q]) if w.modes[l] != 2 else None
                                       for l in range(L)],
                                   swa=[w.swa_kv(l, s)[None] for l in range(L)]
                                   if w.n_win else None))

    def run(self, item):
        w, o = self.w, self.oracle
        o.layer_group(w.modes, item["qb"], item["qi"], item["kv"], item["ki"], w.N, 0, 1,
                      item["qpos"], w.ratio, w.k, w.pool, 1.0 / math.sqrt(w.D),
                      pool_block=w.pool_block, swa_kv=item["swa"], swa_ring=w.swa_ring,
                      n_win=w.n_win, indexer_fmt=w.indexer_fmt, D_I=w.D_I)


def cpu_baseline(w, budget_s=12.0):
    n_setup = 2
    smp = OracleSample(w, list(range(min(n_setup, w.B))))
    done, t0 = 0, time.perf_counter()
    while True:
        smp.run(smp.items[done % len(smp.items)])
        done += 1
        el = time.perf_counter() - t0
        if el >= budget_s or done >= 64:
            break
    value = done * len(w.modes) / el if len(w.modes) > 1 else done / el
    return {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{done} query passes of {w.name} (queries 0..{len(smp.items) - 1} of "
                      f"sequence 0..), single-threaded fp64 C oracle, cache quantised by the "
                      f"oracle before timing", "seconds": el}


def run_reference(args, rank, world):
    from sparse_attention_decode_csa2_gb300.synthetic import WORKLOADS
    import oracle
    oracle.build()
    w = WORKLOADS[args.workload]
    smp = OracleSample(w, [0])
    for _ in range(args.warmup):
        smp.run(smp.items[0])
    t = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        smp.run(smp.items[0])
        t.append(time.perf_counter() - t0)
    total = sum(t)
    L = len(w.modes)
    value = args.steps * L / total if L > 1 else args.steps / total
    base = {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"1 query of {w.name} per step (the full layer path for that query), "
                      f"single-threaded fp64 C oracle"}
    return {
        "metric": METRIC, "value": value, "unit": UNIT, "impl": "reference", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": total * 1e3 / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded SplitMix64)",
        "config": {"workload": w.name, "queries_per_step": 1, "entries_per_seq": w.N,
                   "top_k": w.k, "heads": w.H},
        "cpu_baseline": base,
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    args = parse_args()
    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        world = int(os.environ.get("WORLD_SIZE", "1"))
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args, rank, world)), flush=True)
        return 0
    rank, world, local = dist_setup(args)
    res = run_gpu(args, rank, world, local)
    if res is None:
        return 0
    if rank == 0:
        if world == 1 and not args.no_cpu_baseline:
            from sparse_attention_decode_csa2_gb300.synthetic import WORKLOADS
            res["cpu_baseline"] = cpu_baseline(WORKLOADS[args.workload])
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())

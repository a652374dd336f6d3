"""Benchmark of the paged KV hot path on GB300: one step = for every layer,
append the step's token(s) per row with fused quantization, then paged GQA
decode attention (split-K + LSE merge) through the block tables.

Default workload (N = 1): K8V4 long-context decode batch, C = 8 rows of
131072 tokens (K FP8-E4M3FN-row, V NVFP4-G16), 32 q / 4 kv heads, head_dim
128, 16 layers, pool of M = 16384 shuffled pages (13.56 GB per step); the
same JSON line carries the K8V4 4-token verify, the INT8-G64 C = 8 decode,
the FP8-row shared-prefix decode and the BF16 chunked-prefill workloads under
"workloads".  Other headline workloads: --workload.

Prints ONE JSON line (rank 0).  `value` is KV GB/s of the whole step:
algorithmic bytes (each valid KV token-head read once, shared pages once,
plus q / out / lse / appended K,V and codes) over the device time of the
step, inputs resident in HBM, L2 flushed before every timed step.  `e2e` is
the same metric through the C ABI with the step's inputs copied from pinned
host memory and the outputs copied back inside the timed region.

--impl reference times the oracle (plain NumPy float64, test
infrastructure) on the host cores on a bounded sample of the same workload:
(layer, row, KV head) units over each row's last 4096 keys.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "paged decode-attn KV GB/s (% of GB300 HBM peak) and decode rows/s at C=1..8"


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def peaks_tensor():
    """Dense bf16 tensor peak (burst: the prefill kernel is timed alone)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["bf16_tflops"]), "measured"
    return 1900.0, "fallback"


def traffic(workload, kernel, algorithmic_now):
    """DRAM bytes per launch of the roofline kernel from the committed ncu
    capture (profiles/traffic.json), scaled by algorithmic work to this
    launch (all but its fixed part); None when the kernel's sources changed
    since the capture."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        ent = json.load(open(p))["workloads"][workload]
    except (OSError, KeyError, ValueError):
        return None
    if ent.get("kernel") != kernel:
        return None
    h = hashlib.sha256()
    for f in ent["files"]:
        h.update(f.encode())
        h.update(b"\0")
        try:
            h.update(open(os.path.join(ROOT, f), "rb").read())
        except OSError:
            return None
    if h.hexdigest() != ent["sha256"]:
        return None
    fixed = ent.get("fixed_bytes_per_launch", 0)  # bytes that do not grow with the work (split partials)
    return int(round((ent["dram_bytes_per_launch"] - fixed) * algorithmic_now
                     / ent["algorithmic_per_launch_at_capture"] + fixed))


def make_workload(name, layers=None, context=None):
    """The named workload; `layers` / `context` shrink it (profiling runs)."""
    from paged_kv_cache_append_gb300 import workloads as W
    kw = {}
    if layers:
        kw["num_layers"] = layers
    if context:
        kw["S"] = context
    if name == "k8v4_verify":
        return W.k8v4_long(T=4, **kw)
    if name == "tiny_bf16":
        return W.tiny_bf16()
    if name in ("int8_prefill", "fp8_prefill", "k8v4_prefill", "nvfp4_prefill"):
        return W.bf16_prefill(profile={"int8_prefill": "int8_g64", "fp8_prefill": "fp8_row", "k8v4_prefill": "k8v4",
                                       "nvfp4_prefill": "nvfp4_g16"}[name], **kw)
    return W.WORKLOADS[name](**kw)


def workload_desc(w):
    return (f"{w.name}: {w.profile}, C={w.C} rows, T={w.T}, {w.Hq}q/{w.Hkv}kv heads, D={w.D}, "
            f"{w.num_layers} layers, S={w.S}, M={w.M}, contexts {int(w.context.min()) + w.T}.."
            f"{int(w.context.max()) + w.T}")


# ------------------------------------------------------------ ranks

def init_ranks(world):
    """One process per GPU (replicas): NCCL where CUDA is present, gloo
    otherwise; the rendezvous comes from the torchrun environment."""
    if world <= 1:
        return
    import torch
    import torch.distributed as dist
    if not dist.is_initialized():
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device="cpu"):
    """The largest of every rank's value (the slowest replica sets the
    step time)."""
    if world <= 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(units_per_rank, ms, world):
    """Whole-job throughput: every rank's units over the slowest rank's time
    (weak scaling: the per-rank work is fixed)."""
    return world * units_per_rank / (ms * 1e-3)


# ------------------------------------------------------------ clock sampler

class Clocks:
    """Samples nvidia-smi every 200 ms while the measured region runs.
    mark() brackets the timed steps inside it; summary() reports the median
    SM clock and any throttle reason over the whole sampled window (untimed
    replays of the same step right before the timed ones, then the timed
    steps), and how many samples fell inside the timed steps."""

    def __init__(self, index=0):
        self.index = index
        self.proc = None
        self.path = None
        self.marks = []

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        q = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.3)
        return self

    def mark(self):
        self.marks.append(time.time())

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        import datetime
        sm, mx, pw, reasons, in_timed = [], [], [], set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        lo = self.marks[0] if self.marks else None
        hi = self.marks[-1] if len(self.marks) > 1 else None
        try:
            for line in open(self.path):
                f = [x.strip() for x in line.split(",")]
                if len(f) < 10:
                    continue
                try:
                    sm.append(float(f[2]))
                    mx.append(float(f[3]))
                except ValueError:
                    continue
                try:
                    pw.append(float(f[4]))
                except ValueError:
                    pass
                for n, v in zip(names, f[6:10]):
                    if v.lower() == "active":
                        reasons.add(n)
                try:
                    t = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    if lo is not None and hi is not None and lo - 0.2 <= t <= hi + 0.2:
                        in_timed += 1
                except ValueError:
                    pass
        except OSError:
            pass
        finally:
            try:
                os.unlink(self.path)
            except OSError:
                pass
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        out = {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
               "samples": len(sm), "samples_in_timed_steps": in_timed,
               "window": "untimed replays of the same step graph right before the timed steps, "
                         "then the timed steps"}
        if pw:
            out["power_w_max"] = max(pw)
        return out


# ------------------------------------------------------------ GPU arm

def _arena(tensors, device):
    """One contiguous device buffer holding copies of `tensors` (256-byte
    aligned), and views of it in the same order: a step's inputs (or outputs)
    then move between host and device in one copy."""
    import torch
    offs, total = [], 0
    for t in tensors:
        offs.append(total)
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    buf = torch.empty(max(total, 256), dtype=torch.uint8, device=device)
    views = []
    for t, off in zip(tensors, offs):
        n = t.numel() * t.element_size()
        v = buf[off:off + n].view(t.dtype).view(t.shape)
        v.copy_(t)
        views.append(v)
    return buf, views


class Bench:
    """Device state of one workload; `share` reuses another Bench's filled
    pool (a sub-batch of its first B rows)."""

    def __init__(self, w, device, B=None, share=None, fused=True, host_values=False):
        import torch
        from paged_kv_cache_append_gb300 import nk
        self.torch, self.nk, self.w, self.dev = torch, nk, w, device
        self.fused = fused
        self.host_values = host_values   # context values drawn on the host (the oracle's stream)
        B = w.B if B is None else B
        self.B = B
        self.tables = torch.from_numpy(w.tables).to(device)
        self.rows = torch.from_numpy(w.table_rows[:B].copy()).to(device)
        self.ctx = torch.from_numpy(w.context[:B].copy()).to(device)
        self.front = torch.from_numpy((w.context[:B] + w.T).astype(np.int32)).to(device)
        if share is not None:
            self.pool = share.pool
        else:
            self.pool = nk.Pool(w.profile, w.num_layers, w.Hkv, w.D, w.S, w.C, w.M, device=device)
            self._fill()
        # per-layer step inputs, resident on the device
        # every layer's q, k, v in one device buffer (one host -> device copy
        # per step), every layer's out and lse in another
        ins = []
        for layer in range(w.num_layers):
            k, v = w.step_kv(layer)
            ins += [w.step_q(layer)[:B].contiguous(), k[:B].contiguous(), v[:B].contiguous()]
        self.in_buf, views = _arena(ins, device)
        self.q, self.k, self.v = views[0::3], views[1::3], views[2::3]
        outs = []
        for layer in range(w.num_layers):
            outs += [torch.zeros(self.q[layer].shape, dtype=torch.bfloat16),
                     torch.zeros((B, w.T, w.Hq), dtype=torch.float32)]
        self.out_buf, views = _arena(outs, device)
        self.out, self.lse = views[0::2], views[1::2]
        n = nk.nk_decode_workspace_bytes(self.pool.handle, B, w.T, w.Hq)
        self.ws = torch.zeros(max(n, 16), dtype=torch.uint8, device=device)
        # per layer: the fused append + decode launch and the split merge, or
        # the append, the decode and the merge
        self.launches_per_step = (2 if fused else 3) * w.num_layers
        # chunked prefill rows (bf16_prefill): append the chunk, then attend
        self.Bp = len(w.prefill_rows) if share is None else 0
        if self.Bp:
            self.prow = torch.from_numpy(w.prefill_rows).to(device)
            self.pre = torch.from_numpy(w.prefix_len).to(device)
            self.chk = torch.from_numpy(w.chunk_len).to(device)
            cins = []
            for layer in range(w.num_layers):
                k, v = w.chunk_kv(layer, device=device)
                cins += [w.chunk_q(layer, device=device).contiguous(), k.contiguous(), v.contiguous()]
            self.cin_buf, views = _arena(cins, device)
            self.cq, self.ck, self.cv = views[0::3], views[1::3], views[2::3]
            self.cout_buf = torch.zeros(w.num_layers * self.cq[0].numel() * 2, dtype=torch.uint8,
                                        device=device)
            self.cout = [self.cout_buf[i * self.cq[0].numel() * 2:(i + 1) * self.cq[0].numel() * 2]
                         .view(torch.bfloat16).view(self.cq[0].shape) for i in range(w.num_layers)]
            self.side = torch.cuda.Stream(device=device)
            # chunk append + prefill per layer (quantized pages are dequantized
            # inside the prefill kernel)
            self.launches_per_step += 2 * w.num_layers

    def _fill(self):
        """Context of every table row (device-side seeded values), written
        with the library's append; shared-prefix rows reuse row 0's pages."""
        torch, w = self.torch, self.w
        P = 64
        sh, full, tail = w.shared_len, w.shared_len // P, w.shared_len % P
        ctx = np.zeros(w.C, np.int64)
        ctx[w.table_rows] = w.context
        if len(w.prefill_rows):
            ctx[w.prefill_rows] = w.prefix_len
        gen_dev = self.dev if (w.S * w.C * w.Hkv * w.D > (1 << 26) and not self.host_values) else "cpu"
        for layer in range(w.num_layers):
            for r in range(w.C):
                start = sh if (sh and r > 0) else 0
                n = int(ctx[r]) - start
                if n <= 0:
                    continue
                k, v = w.context_kv(layer, r, int(ctx[r]), device=gen_dev)
                for t0 in range(start, int(ctx[r]), 32768):
                    t1 = min(int(ctx[r]), t0 + 32768)
                    kk = k[t0:t1].unsqueeze(0).contiguous().to(self.dev)
                    vv = v[t0:t1].unsqueeze(0).contiguous().to(self.dev)
                    self.pool.append(layer, self.tables,
                                     torch.tensor([r], dtype=torch.int32, device=self.dev),
                                     torch.tensor([t0], dtype=torch.int32, device=self.dev), kk, vv)
                del k, v
            if sh and tail and layer == w.num_layers - 1:
                for r in range(1, w.C):
                    self.pool.copy_columns(int(w.tables[0, full]), int(w.tables[r, full]), tail)
        torch.cuda.synchronize()

    def step(self, stream=None):
        w = self.w
        torch = self.torch
        if self.Bp:   # prefill rows on a second stream, joined at the end of the step
            cur = torch.cuda.current_stream()
            self.side.wait_stream(cur)
            with torch.cuda.stream(self.side):
                for layer in range(w.num_layers):
                    self.prefill_only(layer, append=True)
        for layer in range(w.num_layers):
            self.attend(layer, stream)

        if self.Bp:
            torch.cuda.current_stream().wait_stream(self.side)

    def prefill_only(self, layer, append=False):
        w = self.w
        if append:
            self.pool.append(layer, self.tables, self.prow, self.pre, self.ck[layer], self.cv[layer],
                             counts=self.chk)
        self.pool.prefill(layer, self.cq[layer], self.tables, self.prow, self.pre, self.chk, w.scale,
                          out=self.cout[layer], lse=None)

    def flops_prefill_layer(self):
        """Algorithmic flops of one prefill launch: 4 * D * Hq * (prefix * S +
        S (S + 1) / 2) per row (QK^T and PV over the visible query-key pairs)."""
        w = self.w
        tot = 0
        for P0, S in zip(w.prefix_len.astype(np.int64), w.chunk_len.astype(np.int64)):
            tot += 4 * w.D * w.Hq * (P0 * S + S * (S + 1) // 2)
        return int(tot)

    def attend(self, layer, stream=None):
        """The decode step of one layer: append the new tokens, then attend
        (one fused launch, or the two separate calls)."""
        w = self.w
        if self.fused:
            self.pool.append_decode(layer, self.q[layer], self.k[layer], self.v[layer], self.tables,
                                    self.rows, self.front, w.scale, out=self.out[layer],
                                    lse=self.lse[layer], workspace=self.ws, stream=stream)
        else:
            self.pool.append(layer, self.tables, self.rows, self.ctx, self.k[layer], self.v[layer],
                             stream=stream)
            self.pool.decode(layer, self.q[layer], self.tables, self.rows, self.front, w.scale,
                             out=self.out[layer], lse=self.lse[layer], workspace=self.ws, stream=stream)

    def roofline_launch(self, layer):
        """The dominant kernel of a decode layer: the fused append + decode
        launch (or the plain decode launch when not fused)."""
        w = self.w
        if self.fused:
            self.attend(layer)
        else:
            self.pool.decode(layer, self.q[layer], self.tables, self.rows, self.front, w.scale,
                             out=self.out[layer], lse=self.lse[layer], workspace=self.ws)

    def bytes_roofline_launch(self):
        return self.bytes_decode_layer() + (self.bytes_append_layer() if self.fused else 0)

    # -- accounting --------------------------------------------------------
    def bytes_decode_layer(self):
        """Algorithmic bytes of one decode launch (one layer): every valid KV
        token-head once (pages shared by several rows once), plus q, out, lse."""
        w = self.w
        bpt = self.pool.kv_bytes_per_token_head()
        F = (w.context[:self.B] + w.T).astype(np.int64)
        tokens = int(F.sum())
        if w.shared_len:
            tokens -= (self.B - 1) * min(w.shared_len, int(F.min()))
        kv = tokens * w.Hkv * bpt
        qo = self.B * w.T * w.Hq * (2 * w.D * 2 + 4)
        return kv + qo

    def bytes_append_layer(self):
        w = self.w
        return self.B * w.T * w.Hkv * (2 * w.D * 2 + self.pool.kv_bytes_per_token_head())

    def bytes_step(self):
        """Decode-side algorithmic bytes of a step (the prefill rows are
        reported in flops)."""
        return self.w.num_layers * (self.bytes_decode_layer() + self.bytes_append_layer())


def _flush_fn(torch, device):
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    buf = torch.empty(max(2 * l2, 1 << 28) // 4, dtype=torch.float32, device=device)
    return lambda: buf.fill_(1.0), 2 * l2


def _timed_graph(torch, graph, steps, flush, stream):
    """Mean and per-step ms of `steps` replays of `graph`, L2 flushed before
    each, CUDA events on the launching stream."""
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for e0, e1 in evs:
        flush()
        e0.record(stream)
        graph.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    ms = [e0.elapsed_time(e1) for e0, e1 in evs]
    return statistics.mean(ms), ms


def _capture(torch, fn):
    """fn() once eagerly, then captured into a CUDA graph (replayed twice)."""
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    return g


def measure(bench, args, flush, stream, world, device, soak_s=0.0):
    """Step throughput of one workload plus the in-step time of its dominant
    kernel.  The step is one CUDA graph over all layers; the roofline kernel
    is timed as a graph of that kernel's launches for all layers, back to
    back (so launch gaps and the L2 state match the step), divided by the
    layer count.  `soak_s` seconds of untimed replays run right before the
    timed steps while the clock sampler runs, so its record covers the
    steady state the timed steps ran in."""
    import torch
    w = bench.w
    for _ in range(max(args.warmup, 3)):
        bench.step()
    torch.cuda.synchronize()
    graph = _capture(torch, bench.step)
    barrier(world)
    torch.cuda.synchronize()
    with Clocks(torch.cuda.current_device()) as clk:
        if soak_s > 0:
            t_end = time.perf_counter() + soak_s
            while time.perf_counter() < t_end:
                for _ in range(8):
                    flush()
                    graph.replay()
                torch.cuda.synchronize()
        clk.mark()
        t_wall = time.perf_counter()
        mean_ms, step_ms = _timed_graph(torch, graph, args.steps, flush, stream)
        t_wall = time.perf_counter() - t_wall
        clk.mark()
    barrier(world)
    ms = max_over_ranks(mean_ms, world, device)
    res = {"graph": graph, "ms": ms, "step_ms": step_ms, "clocks": clk.summary(), "t_wall": t_wall}

    # dominant kernel, in step: the fused decode call (decode + merge launches)
    # of every layer; for the fused decode step that graph is the step itself
    if bench.fused and not bench.Bp:
        kms, how = ms / w.num_layers, "the timed step graph / layers (the step is these launches)"
    else:
        rg = _capture(torch, lambda: [bench.roofline_launch(l) for l in range(w.num_layers)])
        kms = _timed_graph(torch, rg, max(3, args.steps // 2), flush, stream)[0] / w.num_layers
        how = "a graph of this kernel's launches for all layers / layers"
        del rg
    res["kms"], res["kms_how"] = kms, how
    res["achieved"] = bench.bytes_roofline_launch() / (kms * 1e-3) / 1e9

    if bench.Bp:   # the prefill kernel of every layer, back to back, in one graph
        pg = _capture(torch, lambda: [bench.prefill_only(l) for l in range(w.num_layers)])
        pms = _timed_graph(torch, pg, max(3, args.steps // 4), flush, stream)[0] / w.num_layers
        del pg
        res["pms"] = pms
        res["tflops"] = bench.flops_prefill_layer() / (pms * 1e-3) / 1e12
    return res


def extra_workloads(names, args, flush, stream, world, device, shared):
    """Step value and in-step roofline of further workloads (no e2e, sweep or
    CPU baseline); `shared` maps a workload name to a Bench whose pool the
    workload reuses (the verify reads the long-context pool)."""
    import torch
    hbm_peak, _ = peaks()
    tf_peak, _ = peaks_tensor()
    out = {}
    for name in names:
        w = make_workload(name)
        base = shared.get(name)
        b = Bench(w, device, share=base) if base is not None else Bench(w, device)
        r = measure(b, args, flush, stream, world, device)
        value = job_value(b.bytes_step(), r["ms"], world) / 1e9
        ent = {"workload": workload_desc(w), "value": round(value, 2), "unit": "GB/s",
               "ms_per_step": round(r["ms"], 5),
               "pct_of_hbm_peak": round(100 * value / world / hbm_peak, 2),
               "pct_of_nominal_8tbs": round(100 * value / world / 8000.0, 2),
               "rows_per_s": round(world * b.B * w.T / (r["ms"] * 1e-3), 1),
               "roofline": {"bound": "hbm", "kernel": "decode call (decode + merge), one layer",
                            "achieved": round(r["achieved"], 1), "unit": "GB/s",
                            "frac": round(r["achieved"] / hbm_peak, 4),
                            "traffic": traffic(name, "nk_paged_append_decode_attention", b.bytes_roofline_launch()),
                            "algorithmic_bytes_per_launch": b.bytes_roofline_launch(),
                            "avg_launch_ms": round(r["kms"], 5), "timed_as": r["kms_how"]},
               "clocks": r["clocks"]}
        if w.name == "tiny_bf16":  # latency-bound: one row, one layer, 200 tokens
            ent["us_per_step"] = round(1e3 * r["ms"], 2)
        if not b.Bp and w.B > 1 and not args.no_sweep:
            ent["sweep_rows_per_s"] = sweep_rows(b, args, flush, stream, device)
        if b.Bp:
            ent["value_note"] = "decode-side GB/s of the whole step (prefill rows on a second stream)"
            ent["roofline"] = {"bound": "tensor", "kernel": "nk_paged_prefill_attention (tcgen05), one layer",
                               "achieved": round(r["tflops"], 1), "unit": "TFLOP/s",
                               "frac": round(r["tflops"] / tf_peak, 4),
                               "traffic": traffic(name, "nk_paged_prefill_attention", b.flops_prefill_layer()),
                               "algorithmic_flops_per_launch": b.flops_prefill_layer(),
                               "avg_launch_ms": round(r["pms"], 4),
                               "timed_as": "a graph of the prefill launches for all layers / layers"}
        out[name] = ent
        del r, b
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    return out


def sweep_rows(bench, args, flush, stream, device):
    """Rows/s (and KV GB/s) of the step over the first c rows, c = 1..B, each
    step replayed as its own graph (the rows share the filled pool)."""
    import torch
    w = bench.w
    sweep = {}
    for c in range(1, w.B + 1):
        bc = Bench(w, device, B=c, share=bench, fused=bench.fused) if c != w.B else bench
        g = _capture(torch, bc.step)
        sm = _timed_graph(torch, g, max(5, args.steps // 4), flush, stream)[0]
        sweep[str(c)] = {"rows_per_s": round(c * w.T / (sm * 1e-3), 1),
                         "kv_gbs": round(bc.bytes_step() / (sm * 1e-3) / 1e9, 1),
                         "ms_per_step": round(sm, 4)}
        del g, bc
    return sweep


EXTRAS = {"k8v4_long": ["k8v4_verify", "int8_decode", "fp8_shared", "bf16_prefill", "tiny_bf16"]}


def run_gpu(args, rank, world):
    import torch
    device = f"cuda:{int(os.environ.get('LOCAL_RANK', 0))}"
    torch.cuda.set_device(device)
    w = make_workload(args.workload, args.layers, args.context)
    hbm_peak, peak_kind = peaks()
    bench = Bench(w, device, fused=not args.unfused)
    flush, flush_bytes = _flush_fn(torch, device)
    stream = torch.cuda.current_stream()

    r = measure(bench, args, flush, stream, world, device, soak_s=args.soak)
    graph, ms, clocks, t_wall = r["graph"], r["ms"], r["clocks"], r["t_wall"]
    kms, achieved = r["kms"], r["achieved"]

    # ---- prefill kernel (prefill workloads): tensor roofline ---------------------
    prefill_line = None
    if bench.Bp:
        tf_peak, tf_kind = peaks_tensor()
        pms, tflops = r["pms"], r["tflops"]
        prefill_line = {"bound": "tensor", "achieved": round(tflops, 1), "peak": tf_peak,
                        "peak_kind": tf_kind, "unit": "TFLOP/s", "frac": round(tflops / tf_peak, 4),
                        "traffic": traffic(args.workload, "nk_paged_prefill_attention",
                                           bench.flops_prefill_layer()),
                        "traffic_unit": "bytes per launch",
                        "kernel": "nk_paged_prefill_attention (tcgen05), one layer",
                        "algorithmic_flops_per_launch": bench.flops_prefill_layer(),
                        "avg_launch_ms": round(pms, 4),
                        "timed_as": "a graph of the prefill launches for all layers / layers"}

    # ---- end to end through the C ABI with host buffers ----------------------
    # the step's inputs (q, k, v of every layer; the prefill chunks) come from
    # pinned host memory and its outputs (out, lse; prefill out) go back, one
    # copy per buffer, inside the timed region
    h_in = [bench.in_buf.cpu().pin_memory()]
    d_in = [bench.in_buf]
    h_out = [torch.empty(bench.out_buf.shape, dtype=torch.uint8, pin_memory=True)]
    d_out = [bench.out_buf]
    if bench.Bp:
        h_in.append(bench.cin_buf.cpu().pin_memory())
        d_in.append(bench.cin_buf)
        h_out.append(torch.empty(bench.cout_buf.shape, dtype=torch.uint8, pin_memory=True))
        d_out.append(bench.cout_buf)
    h2d = sum(x.numel() for x in h_in)
    d2h = sum(x.numel() for x in h_out)

    def e2e_step():
        for d, h in zip(d_in, h_in):
            d.copy_(h, non_blocking=True)
        graph.replay()
        for h, d in zip(h_out, d_out):
            h.copy_(d, non_blocking=True)

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    eev = []
    for _ in range(args.steps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        flush()
        e0.record(stream)
        e2e_step()
        e1.record(stream)
        eev.append((e0, e1))
    torch.cuda.synchronize()
    e2e_ms = statistics.mean(e0.elapsed_time(e1) for e0, e1 in eev)

    # ---- rows/s at C = 1..8 ------------------------------------------------------
    sweep = {}
    if not args.no_sweep and w.B > 1:
        sweep = sweep_rows(bench, args, flush, stream, device)

    roof_kernel = "nk_paged_append_decode_attention" if bench.fused else "nk_paged_decode_attention"
    value = job_value(bench.bytes_step(), ms, world) / 1e9
    e2e_ms = max_over_ranks(e2e_ms, world, device)
    e2e_val = job_value(bench.bytes_step(), e2e_ms, world) / 1e9
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": (f"{w.profile} KV codes; " + ("bf16" if w.profile == "bf16" else "f16")
                  + " mma, fp32 accumulate"),
        "data": "synthetic (seeded N(0,1) bf16; tables are seeded permutations)",
        "config": {"workload": workload_desc(w), "rows": bench.B, "layers": w.num_layers,
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "l2": (f"flushed ({flush_bytes >> 20} MiB write) before every timed step"
                          + ("; the step also reads far more than L2"
                             if bench.bytes_step() > 4 * flush_bytes else "")),
                   "graph": "one CUDA graph per step",
                   "step": ("fused append + decode launch per layer" if bench.fused
                            else "append launch + decode launch per layer")},
        "rows_per_s": round(world * bench.B * w.T / (ms * 1e-3), 1),
        "pct_of_hbm_peak": round(100 * value / world / hbm_peak, 2),
        "pct_of_nominal_8tbs": round(100 * value / world / 8000.0, 2),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm_peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": round(achieved / hbm_peak, 4),
                     "traffic": (traffic(args.workload, roof_kernel, bench.bytes_roofline_launch())
                                 if not bench.Bp else None),
                     "traffic_unit": "bytes per launch",
                     "kernel": roof_kernel + (" (append + decode + merge)" if bench.fused
                                              else " (decode + merge)") + ", one layer",
                     "algorithmic_bytes_per_launch": bench.bytes_roofline_launch(),
                     "avg_launch_ms": round(kms, 5), "timed_as": r["kms_how"]},
        "e2e": {"value": round(e2e_val, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 5)},
        "gpu_launches": bench.launches_per_step * args.steps,
        "clocks": clocks,
        "wall_s_timed": round(t_wall, 4),
    }
    if sweep:
        line["sweep_rows_per_s"] = sweep
    if prefill_line:
        # the prefill kernel dominates this workload's step: it is the roofline
        line["decode_roofline"] = line["roofline"]
        line["roofline"] = prefill_line
        line["prefill_tflops"] = prefill_line["achieved"]
    extras = [] if args.no_extra or args.layers or args.context else EXTRAS.get(args.workload, [])
    if extras:
        del graph, r
        line["workloads"] = extra_workloads(extras, args, flush, stream, world, device,
                                            shared={"k8v4_verify": bench} if w.name == "k8v4_long" else {})
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
        one = cpu_baseline_one_thread(args.workload, args.layers, args.context, args.cpu_seconds / 3)
        if one is not None:
            line["cpu_baseline"]["value_1_thread"] = one
    return line


# ------------------------------------------------------------ oracle arm

WINDOW = 4096   # keys per oracle sample unit


class OracleUnits:
    """Bounded sample units of a decode workload for the oracle: one (layer,
    row, KV head) over the row's last min(F, 4096) keys, which hold the step's
    T new tokens.  That is the row's last split-K range: the oracle encodes
    those tokens, decodes them and attends the head's G query heads over them
    with the exact visibility of the full row (query t sees keys up to
    F - T + t), giving that range's normalised partial (out, lse), which the
    exact log-sum-exp merge combines with the other ranges.  Drawing the
    inputs is not timed; the oracle's arithmetic is."""

    def __init__(self, w):
        self.w = w
        self._cache = (None, None)
        self.ks = {}

    def _inputs(self, layer, b):
        from paged_kv_cache_append_gb300.workloads import bf16_to_bits
        w = self.w
        key = (layer, b)
        if self._cache[0] != key:
            r = int(w.table_rows[b])
            n = int(w.context[b])
            lo = max(0, n + w.T - WINDOW)
            kc, vc = w.context_kv(layer, r, n)
            if w.shared_len and r != 0 and lo < w.shared_len:
                k0, v0 = w.context_kv(layer, 0, int(w.context[0]))
                kc = torch_cat(k0[:w.shared_len], kc[w.shared_len:])
                vc = torch_cat(v0[:w.shared_len], vc[w.shared_len:])
            if layer not in self.ks:
                self.ks[layer] = (w.step_kv(layer), w.step_q(layer))
            (ks, vs), q = self.ks[layer]
            kb = np.concatenate([bf16_to_bits(kc[lo:]), bf16_to_bits(ks[b])], axis=0)
            vb = np.concatenate([bf16_to_bits(vc[lo:]), bf16_to_bits(vs[b])], axis=0)
            self._cache = (key, (kb, vb, bf16_to_bits(q[b]), n + w.T - lo))
        return self._cache[1]

    def run(self, layer, b, h):
        """Returns (algorithmic bytes of the unit, oracle seconds)."""
        from oracle import attention as OA, codec as OC, formats as OF
        w = self.w
        kb, vb, qb, n_win = self._inputs(layer, b)
        G = w.Hq // w.Hkv
        t0 = time.perf_counter()
        planes = OC.encode_kv(w.profile, kb[:, h:h + 1], vb[:, h:h + 1])
        K, V = OC.decode_kv(w.profile, planes)
        q = OF.bf16_bits_to_f64(qb[:, h * G:(h + 1) * G])
        OA.decode(q, K, V, n_win, w.scale)
        dt = time.perf_counter() - t0
        bpt = sum(p.shape[-1] for p in planes.values())
        return n_win * bpt + w.T * G * (2 * w.D * 2 + 4), dt


def torch_cat(a, b):
    import torch
    return torch.cat([a, b])


def cpu_baseline(w, seconds=15.0):
    """The oracle on sample units of the workload (KV heads, then rows, then
    layers) until `seconds` of oracle time have passed."""
    cores = len(os.sched_getaffinity(0))
    units = OracleUnits(w)
    done, n, spent = 0, 0, 0.0
    i = 0
    while spent < seconds:
        h = i % w.Hkv                     # the KV heads of one row share its drawn inputs
        b = (i // w.Hkv) % w.B
        layer = (i // (w.B * w.Hkv)) % w.num_layers
        by, dt = units.run(layer, b, h)
        done += by
        spent += dt
        n += 1
        i += 1
    return {"value": round(done / spent / 1e9, 6), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} units of {w.name}, each one (layer, row, KV head) over the row's last "
                      f"min(F, {WINDOW}) keys (its last split-K range, holding the new tokens): "
                      f"encode, decode, float64 attention; {spent:.1f} s of oracle time"}


def cpu_baseline_one_thread(name, layers, context, seconds):
    """The same oracle sample on one host thread: a fresh interpreter whose
    BLAS and OpenMP pools have one thread (set before NumPy loads); its GB/s,
    or None when it cannot run."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    code = ("import json, bench; "
            f"w = bench.make_workload({name!r}, {layers!r}, {context!r}); "
            f"print(json.dumps(bench.cpu_baseline(w, {seconds!r})))")
    try:
        res = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True,
                             timeout=300)
        return json.loads(res.stdout.strip().splitlines()[-1])["value"] if res.returncode == 0 else None
    except (subprocess.SubprocessError, ValueError, IndexError, KeyError):
        return None


def run_reference(args, rank, world):
    w = make_workload(args.workload, args.layers, args.context)
    cores = len(os.sched_getaffinity(0))
    units = OracleUnits(w)
    for i in range(args.warmup):
        units.run(0, 0, i % w.Hkv)
    times, done = [], 0
    for s in range(args.steps):
        by, dt = units.run(0, (s // w.Hkv) % w.B, s % w.Hkv)
        done += by
        times.append(dt)
    tot = sum(times)
    value = done / tot / 1e9
    sample = (f"each step: one (layer 0, row, KV head) unit over the row's last min(F, {WINDOW}) keys "
              "(encode, decode, float64 attention)")
    line = {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 6), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * tot / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) bf16; tables are seeded permutations)",
        "config": {"workload": workload_desc(w), "rows": w.B, "layers": w.num_layers,
                   "parallelism": "single process (host cores)", "sample": sample},
        "cpu_baseline": {"value": round(value, 6), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 6), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    return line


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="nk", choices=["nk", "reference"])
    ap.add_argument("--workload", default="k8v4_long",
                    choices=["tiny_bf16", "int8_decode", "fp8_shared", "k8v4_long", "k8v4_verify",
                             "bf16_prefill", "int8_prefill", "fp8_prefill", "k8v4_prefill", "nvfp4_prefill"])
    ap.add_argument("--layers", type=int, default=None, help="fewer layers (profiling)")
    ap.add_argument("--context", type=int, default=None, help="smaller max context S (profiling)")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--unfused", action="store_true",
                    help="separate append and decode launches instead of the fused call")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="only the chosen workload (no further workloads in the line)")
    ap.add_argument("--soak", type=float, default=2.0,
                    help="seconds of untimed step replays under the clock sampler before the timed steps")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args, rank, world)), flush=True)
        return
    init_ranks(world)
    line = run_gpu(args, rank, world)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

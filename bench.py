"""Benchmark of sliding-window split-KV verify attention on GB300.

Metric: verify-attention microseconds per call and KV-cache GB/s (as a
fraction of HBM bandwidth) at window 188, q_len 8.  `value` is KV GB/s
(higher is better); `us_per_call` is reported beside it.

One step = one swa_verify_attn call over one batch of the workload.  The
default workload is the single-stream Gemma-style verify (1 sequence, 8/2
heads, head_dim 256, context 4096, W 188, q_len 8); `--workload` selects
another (batched, stress_w{188,512,1024}_q{1,8,64}, window_vs_full_w{188,4096},
tiny_q{1,8}).  Inputs are seeded synthetic bf16 (no dataset exists for this
path).

Timing: the K timed steps are replays of a CUDA graph of calls, bracketed by
a barrier and torch.cuda.synchronize() on both sides and timed with CUDA
events on the launching stream.  L2 is defeated by rotating input replicas
whose combined footprint is at least twice the L2 size (or, when one call
already reads more than L2, by the size of the inputs).

Algorithmic bytes per call = sum over sequences of
  Hkv * S_b * 2 * D * 2   (K and V rows of the window span, S_b keys)
+ 2 * q_len * Hq * D * 2  (q in, out)
+ 4 * q_len * Hq          (lse)
with S_b = min(q_pos + q_len, seq_len) - max(0, q_pos - W + 1).

Beside the timed value, rank 0 of a one-GPU run reports:
  e2e        the same metric per step of a caller with host buffers: one
             packed input copy from pinned memory, the fused append + verify
             call, one packed output copy back (copies inside the timed region);
  roofline   the dominant kernel's achieved GB/s against the measured copy
             bandwidth and the nominal 7.9 TB/s, its ncu DRAM traffic per
             launch while the kernel sources match the capture, and the launch
             floors;
  also, prefill, paged, append, accept
             the other workloads and entry points, measured the same way;
  cpu_baseline
             the fp64 oracle on the host cores (all threads, and one thread).

--impl reference times the fp64 CPU oracle (the only reference this path
has) on the host cores, same workload, metric and unit.
"""
import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

KERNEL_NAMES = {1: "swa_simt_kernel", 2: "swa_tc_kernel", 3: "swa_rows_kernel", 4: "swa_pair_kernel"}
METRIC = "verify-attn µs/call and KV GB/s (% of GB300 HBM peak) at W=188, q_len=8"
UNIT = "GB/s"


# ----------------------------------------------------------------- workloads

def make_workload(name, device, seed=0):
    from sliding_window_speculative_gb300 import inputs
    if name == "single_stream":
        return inputs.single_stream(device=device, seed=seed)
    if name == "batched":
        return inputs.batched(device=device, seed=seed)
    if name.startswith("window_vs_full_w"):
        return inputs.window_vs_full(int(name.rsplit("w", 1)[1]), device=device, seed=seed)
    if name.startswith("tiny_q"):
        return inputs.tiny(int(name[6:]), device=device, seed=seed)
    if name.startswith("prefill_q"):
        # prefill_q{Q}[_b{B}]: sliding-window prefill chunks of Q tokens
        parts = name.split("_")
        Q = int(parts[1][1:])
        B = int(parts[2][1:]) if len(parts) > 2 else 1
        return inputs.prefill(Q, batch=B, device=device, seed=seed)
    if name.startswith("stress_w"):
        # stress_w{W}_q{Q}[_l{L}]: the bandwidth-stress batch; _l shortens the
        # cache (and the context range) for profiler captures.
        parts = name.split("_")
        W, Q = int(parts[1][1:]), int(parts[2][1:])
        L = int(parts[3][1:]) if len(parts) > 3 else 32768
        return inputs.stress(W, Q, device=device, max_len=L, seed=seed)
    raise ValueError(f"unknown workload {name}")


def workload_bytes(case):
    d = case.dims
    kv = 0
    for sl, qp in zip(case.seq_lens_host, case.q_pos_host):
        lo = max(0, qp - case.window + 1)
        hi = min(qp + d["q_len"], sl)
        kv += d["num_kv_heads"] * max(0, hi - lo) * 2 * d["head_dim"] * 2
    qo = 2 * d["batch"] * d["q_len"] * d["num_q_heads"] * d["head_dim"] * 2
    lse = 4 * d["batch"] * d["q_len"] * d["num_q_heads"]
    return kv, kv + qo + lse


def workload_flops(case):
    d = case.dims
    G = d["num_q_heads"] // d["num_kv_heads"]
    f = 0
    for sl, qp in zip(case.seq_lens_host, case.q_pos_host):
        for i in range(d["q_len"]):
            p = qp + i
            n = max(0, min(p, sl - 1) - max(0, p - case.window + 1) + 1)
            f += n * 4 * d["head_dim"] * G * d["num_kv_heads"]
    return f


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""
    FIELDS = ["clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.active",
              "clocks_event_reasons.hw_slowdown", "clocks_event_reasons.hw_thermal_slowdown",
              "clocks_event_reasons.sw_thermal_slowdown", "clocks_event_reasons.sw_power_cap"]

    def __init__(self, device_index):
        self.proc = None
        sel = None
        try:
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            sel = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            vis = os.environ.get("CUDA_VISIBLE_DEVICES")
            sel = vis.split(",")[device_index] if vis else str(device_index)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + ",".join(self.FIELDS),
                 "--format=csv,noheader,nounits", "-lms", "100", "-i", sel],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        self.lines = []
        self.t = None
        if self.proc is not None:
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self):
        return time.time()

    def stop(self, t0, t1):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=2)
        except Exception:
            self.proc.kill()
        if self.t is not None:
            self.t.join(timeout=2)
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) != len(self.FIELDS):
                continue
            rows.append((ts, parts))
        window = [p for ts, p in rows if t0 - 0.15 <= ts <= t1 + 0.15] or [p for _, p in rows]
        mhz = [float(p[0]) for p in window if p[0].replace(".", "").isdigit()]
        mx = [float(p[1]) for p in window if p[1].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for p in window:
            for n, val in zip(names, p[4:]):
                if val.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(mhz) if mhz else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(window)}


# ------------------------------------------------------------- GPU timing

class Replicas:
    """Copies of a workload's tensors at distinct addresses, so consecutive
    calls read cold data."""

    def __init__(self, case, n, append=None):
        self.n = n
        self.case = case
        self.append = append  # None, "fused" (swa_append_verify_attn) or "torch" (copies + verify)
        B = case.q.shape[0]
        self.q = case.q.unsqueeze(0).repeat(n, 1, 1, 1, 1) if n > 1 else case.q.unsqueeze(0)
        if n > 1:
            self.k = torch.empty((n,) + tuple(case.k_cache.shape), dtype=torch.bfloat16,
                                 device=case.q.device)
            self.v = torch.empty_like(self.k)
            self.k[:] = case.k_cache
            self.v[:] = case.v_cache
        else:
            self.k = case.k_cache.unsqueeze(0)
            self.v = case.v_cache.unsqueeze(0)
        self.out = torch.empty_like(self.q)
        self.lse = torch.empty((n, B, case.q.shape[1], case.q.shape[2]), dtype=torch.float32,
                               device=case.q.device)
        if append is not None:
            # the verify block's rows as the projection would hand them over,
            # [B, q_len, Hkv, D]; appending them rewrites the same values
            q_len = case.q.shape[1]
            Hkv, L, D = case.k_cache.shape[1:]
            kn = torch.zeros((B, q_len, Hkv, D), dtype=torch.bfloat16, device=case.q.device)
            vn = torch.zeros_like(kn)
            for b, qp in enumerate(case.q_pos_host):
                kn[b] = case.k_cache[b, :, qp:qp + q_len].transpose(0, 1)
                vn[b] = case.v_cache[b, :, qp:qp + q_len].transpose(0, 1)
            self.kn = kn.unsqueeze(0).repeat(n, 1, 1, 1, 1)
            self.vn = vn.unsqueeze(0).repeat(n, 1, 1, 1, 1)

    def call(self, i, num_splits=0):
        from sliding_window_speculative_gb300 import swa_append_verify_attn, swa_verify_attn
        r = i % self.n
        c = self.case
        if self.append == "fused":
            swa_append_verify_attn(self.q[r], self.kn[r], self.vn[r], self.k[r], self.v[r],
                                   c.seq_lens, c.q_pos, c.window, c.scale, out=self.out[r],
                                   lse=self.lse[r], num_splits=num_splits)
            return
        if self.append == "torch":
            q_len = c.q.shape[1]
            for b, qp in enumerate(c.q_pos_host):
                self.k[r][b, :, qp:qp + q_len].copy_(self.kn[r][b].transpose(0, 1))
                self.v[r][b, :, qp:qp + q_len].copy_(self.vn[r][b].transpose(0, 1))
        swa_verify_attn(self.q[r], self.k[r], self.v[r], c.seq_lens, c.q_pos, c.window, c.scale,
                        out=self.out[r], lse=self.lse[r], num_splits=num_splits)


def hold_stream(stream, us=500.0):
    """Queue a sleep kernel of about `us` microseconds on `stream` ahead of
    a timed region, so that the host has submitted the region's work before
    the device reaches the start event: the events then bracket device
    execution only, not the host's launch latency (the end-to-end timing
    keeps its host costs on purpose and does not use this)."""
    with torch.cuda.stream(stream):
        torch.cuda._sleep(int(us * 2.1e3))  # cycles at up to 2.1 GHz


def replica_count(case, bytes_per_call, steps, l2=None):
    """Input replicas that keep every timed call's reads out of L2.

    Returns (n, l2, distinct).  distinct: the timed calls each read their
    own replica (n >= steps) and L2 is flushed before the timed replay.
    Otherwise the calls cycle through n replicas that together hold at least
    twice the L2 size.  n = 1 when one call alone reads more than L2."""
    if l2 is None:
        l2 = (getattr(torch.cuda.get_device_properties(case.q.device), "L2_cache_size", 0) or
              (126 << 20))
    if bytes_per_call >= l2:
        return 1, l2, False
    slab = case.k_cache.numel() * 2 * 2 + case.q.numel() * 2 * 2
    cap = max(2, int((16 << 30) // max(slab, 1)))   # replicas fit in 16 GiB
    cycle = math.ceil(2 * l2 / bytes_per_call)
    if steps < cycle and steps <= cap:
        return max(2, steps), l2, True
    return min(cycle, cap), l2, False


def time_device(case, steps, warmup, num_splits=0, graph_len=1000, dist=None, append=None):
    """Device time of `steps` calls (graph replays), L2 defeated by replicas.

    With fewer timed calls than one cycle of replicas needs, every timed
    call reads its own replica and a read of twice the L2 size runs between
    the graph's warm-up replay and the timed replay, so no timed call finds
    its inputs in L2.  Otherwise the graph cycles through replicas holding at
    least twice the L2 size, so between two uses of one replica the other
    calls read that much.  Returns dict with total seconds and per-call
    microseconds."""
    kv, total = workload_bytes(case)
    nrep, l2, distinct = replica_count(case, total, steps)
    rep = Replicas(case, nrep, append)
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for i in range(max(warmup, 3)):
            rep.call(i, num_splits)
    stream.synchronize()

    def capture(idx):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in idx:
                rep.call(i, num_splits)
        return g

    flush = None
    if distinct:
        timed = [capture(range(steps))]
        flush = torch.empty(2 * l2 // 8, dtype=torch.int64, device=case.q.device)
        scheme = (f"each timed call reads its own replica ({steps} of {nrep}); {2 * l2 >> 20} MiB "
                  f"read between the warm-up and the timed replay (a read leaves no dirty lines "
                  f"to write back during the timed calls)")
    else:
        g_len = nrep * max(1, min(graph_len, steps) // nrep) if nrep <= steps else steps
        full, rest = divmod(steps, g_len)
        timed = [capture(range(g_len))] * full + ([capture(range(rest))] if rest else [])
        scheme = (f"calls cycle through {nrep} replicas ({nrep * total >> 20} MiB per cycle)"
                  if nrep > 1 else "every call reads more than L2")
    # warm the graphs themselves (first replays upload them), then push every
    # replica out of L2 by reading a buffer twice its size
    with torch.cuda.stream(stream):
        for g in dict.fromkeys(timed):
            g.replay()
        if flush is not None:
            flush.sum()
    stream.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    hold_stream(stream)
    with torch.cuda.stream(stream):
        start.record(stream)
        for g in timed:
            g.replay()
        end.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    if dist is not None:
        dist.barrier()
    ms = start.elapsed_time(end)
    del timed, flush, rep
    return {"seconds": ms / 1e3, "us_per_call": ms * 1e3 / steps, "replicas": nrep,
            "l2_bytes": l2, "l2_scheme": scheme, "wall": (t0, t1), "kv_bytes": kv,
            "bytes": total}


def _packed(parts, device=None, pin=False, align=256):
    """One byte buffer holding tensors of the given (shape, dtype) at
    `align`-byte offsets; returns (buffer, views)."""
    offs, n = [], 0
    for shape, dtype in parts:
        offs.append(n)
        nbytes = math.prod(shape) * torch.empty((), dtype=dtype).element_size()
        n = (n + nbytes + align - 1) // align * align
    buf = torch.empty(n, dtype=torch.uint8, device=device)
    if pin:
        buf = buf.pin_memory()
    views = []
    for (shape, dtype), o in zip(parts, offs):
        nbytes = math.prod(shape) * torch.empty((), dtype=dtype).element_size()
        views.append(buf[o:o + nbytes].view(dtype).view(shape))
    return buf, views


def time_e2e(case, steps, warmup, graph=False):
    """Through the public call with host buffers: each step copies the
    step's inputs (q, the q_len new K/V rows of every sequence and KV head,
    seq_lens, q_pos), packed in one pinned host buffer, to the device in one
    copy; issues swa_append_verify_attn (prepared once: validated and
    marshalled outside the loop), which writes the new rows into the cache
    and attends over it; and copies out and lse, packed in one device
    buffer, back to pinned host memory in one copy.  With graph=True the
    three operations of a step are captured once as one CUDA graph and each
    step is one replay (the single-graph decode step of the pages,
    ONEGRAPH): the copies still run every step.  Timed with CUDA events
    around all steps, three times over; the median of the three is kept (a
    host stall inside one short run moves its mean by tens of percent)."""
    from sliding_window_speculative_gb300 import prepare, swa_append_verify_attn
    B, q_len, Hq, D = case.q.shape
    Hkv = case.k_cache.shape[1]
    dev = case.q.device
    rows = (B, q_len, Hkv, D)
    parts_in = [(tuple(case.q.shape), torch.bfloat16), (rows, torch.bfloat16),
                (rows, torch.bfloat16), ((B,), torch.int32), ((B,), torch.int32)]
    h_in, (h_q, h_kn, h_vn, h_sl, h_qp) = _packed(parts_in, pin=True)
    d_in, (d_q, d_kn, d_vn, d_sl, d_qp) = _packed(parts_in, device=dev)
    h_q.copy_(case.q.cpu())
    h_sl.copy_(case.seq_lens.cpu())
    h_qp.copy_(case.q_pos.cpu())
    for b, p in enumerate(case.q_pos_host):
        # the block's rows as the cache holds them: [q_len, Hkv, D]
        h_kn[b].copy_(case.k_cache[b, :, p:p + q_len].transpose(0, 1).cpu())
        h_vn[b].copy_(case.v_cache[b, :, p:p + q_len].transpose(0, 1).cpu())
    parts_out = [(tuple(case.q.shape), torch.bfloat16), ((B, q_len, Hq), torch.float32)]
    d_out, (out, lse) = _packed(parts_out, device=dev)
    h_out, (h_o, h_l) = _packed(parts_out, pin=True)
    stream = torch.cuda.Stream()
    h2d = h_in.numel()
    d2h = h_out.numel()
    call = prepare(swa_append_verify_attn, d_q, d_kn, d_vn, case.k_cache, case.v_cache, d_sl,
                   d_qp, case.window, case.scale, out=out, lse=lse, stream=stream)

    def step():
        d_in.copy_(h_in, non_blocking=True)
        call()
        h_out.copy_(d_out, non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(max(warmup, 3)):
            step()
    stream.synchronize()
    run = step
    if graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step()
        with torch.cuda.stream(stream):
            g.replay()
        stream.synchronize()
        run = g.replay
    runs = []
    for _ in range(3):
        h_o.zero_()
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            start.record(stream)
            for _ in range(steps):
                run()
            end.record(stream)
        torch.cuda.synchronize()
        runs.append(start.elapsed_time(end))
    ms = sorted(runs)[1]
    return {"us_per_call": ms * 1e3 / steps, "h2d": h2d, "d2h": d2h, "steps": steps,
            "runs_us": [round(r * 1e3 / steps, 3) for r in runs],
            "out": h_o.clone(), "lse": h_l.clone()}


def e2e_entry(case, steps, warmup, graph):
    kv, _ = workload_bytes(case)
    e = time_e2e(case, steps, warmup, graph=graph)
    return {"value": round(kv / (e["us_per_call"] * 1e-6) / 1e9, 3), "unit": UNIT,
            "us_per_call": round(e["us_per_call"], 3), "runs_us": e["runs_us"],
            "h2d_bytes_per_step": e["h2d"], "d2h_bytes_per_step": e["d2h"]}


# ------------------------------------------------------------ CPU oracle

def time_paged(name, page_size, steps=50, warmup=5, seed=0):
    """Device time of swa_verify_attn_paged on workload `name` whose cache is
    scattered over a shuffled page pool (pages of `page_size` rows)."""
    from sliding_window_speculative_gb300 import swa_verify_attn_paged
    case = make_workload(name, torch.device("cuda"), seed=seed)
    B, Hkv, L, D = case.k_cache.shape
    nb = L // page_size
    g = torch.Generator().manual_seed(seed)
    table = torch.randperm(B * nb, generator=g).view(B, nb).to(torch.int32)
    inv = torch.empty_like(table.view(-1))
    inv[table.view(-1).long()] = torch.arange(B * nb, dtype=torch.int32)
    # page table[b, k] holds rows [k*page_size, (k+1)*page_size) of sequence b
    src_k = case.k_cache.view(B, Hkv, nb, page_size, D).permute(0, 2, 1, 3, 4).reshape(B * nb, Hkv, page_size, D)
    src_v = case.v_cache.view(B, Hkv, nb, page_size, D).permute(0, 2, 1, 3, 4).reshape(B * nb, Hkv, page_size, D)
    kp = src_k[inv.long().cuda()].contiguous()
    vp = src_v[inv.long().cuda()].contiguous()
    table = table.cuda()
    kv, total = workload_bytes(case)
    out = torch.empty_like(case.q)
    lse = torch.empty(case.q.shape[:3], dtype=torch.float32, device="cuda")
    del src_k, src_v
    case.k_cache = case.v_cache = None
    torch.cuda.empty_cache()
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for _ in range(max(warmup, 3)):
            swa_verify_attn_paged(case.q, kp, vp, table, case.seq_lens, case.q_pos, case.window,
                                  case.scale, out=out, lse=lse)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for _ in range(steps):
            swa_verify_attn_paged(case.q, kp, vp, table, case.seq_lens, case.q_pos, case.window,
                                  case.scale, out=out, lse=lse)
    with torch.cuda.stream(stream):
        graph.replay()
    stream.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    hold_stream(stream)
    with torch.cuda.stream(stream):
        start.record(stream)
        graph.replay()
        end.record(stream)
    torch.cuda.synchronize()
    us = start.elapsed_time(end) * 1e3 / steps
    del kp, vp, graph
    torch.cuda.empty_cache()
    return {"workload": name, "page_size": page_size, "us_per_call": round(us, 3),
            "achieved_gbs": round(total / (us * 1e-6) / 1e9, 2)}


def time_append(name, steps=2000, warmup=5, seed=0):
    """Fused KV append + verify (swa_append_verify_attn) against the plain
    verify call on workload `name`; for one sequence also the unfused way
    (two strided copies into the cache, then the verify call)."""
    case = make_workload(name, torch.device("cuda"), seed=seed)
    kv, total = workload_bytes(case)
    B, q_len, Hq, D = case.q.shape
    new_bytes = 2 * 2 * B * q_len * case.k_cache.shape[1] * D * 2  # K+V rows read and written
    plain = time_device(case, steps, warmup)["us_per_call"]
    fused = time_device(case, steps, warmup, append="fused")["us_per_call"]
    res = {"workload": name, "verify_us": round(plain, 3), "fused_append_verify_us": round(fused, 3),
           "fused_achieved_gbs": round((total + new_bytes) / (fused * 1e-6) / 1e9, 2)}
    if B == 1:
        unf = time_device(case, steps, warmup, append="torch")["us_per_call"]
        res["torch_copies_then_verify_us"] = round(unf, 3)
    del case
    torch.cuda.empty_cache()
    return res


def time_accept(B, q_len, V, steps=2000, warmup=5, seed=0, graph_len=1000):
    """Device time of swa_greedy_accept on bf16 N(0,1) logits [B, q_len, V]
    (graph replays, L2 defeated by logit replicas)."""
    from sliding_window_speculative_gb300 import swa_greedy_accept
    g = torch.Generator(device="cuda").manual_seed(seed)
    nbytes = B * q_len * V * 2
    l2 = getattr(torch.cuda.get_device_properties(0), "L2_cache_size", 0) or (126 << 20)
    nrep = 1 if nbytes >= l2 else max(2, min(512, math.ceil(2 * l2 / nbytes)))
    logits = torch.randn((nrep, B, q_len, V), generator=g, device="cuda").to(torch.bfloat16)
    draft = torch.randint(0, V, (B, max(q_len - 1, 1)), generator=g, device="cuda",
                          dtype=torch.int32)[:, :q_len - 1].contiguous()
    am = torch.empty((B, q_len), dtype=torch.int32, device="cuda")
    acc = torch.empty((B,), dtype=torch.int32, device="cuda")
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for i in range(max(warmup, 3)):
            swa_greedy_accept(logits[i % nrep], draft, None, am, acc)
    stream.synchronize()
    n = max(1, min(graph_len, steps))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(n):
            swa_greedy_accept(logits[i % nrep], draft, None, am, acc)
    with torch.cuda.stream(stream):
        graph.replay()
    stream.synchronize()
    reps = max(1, steps // n)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    hold_stream(stream)
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(reps):
            graph.replay()
        end.record(stream)
    torch.cuda.synchronize()
    us = start.elapsed_time(end) * 1e3 / (reps * n)
    return {"batch": B, "q_len": q_len, "vocab": V, "us_per_call": round(us, 3),
            "logit_gbs": round(nbytes / (us * 1e-6) / 1e9, 1), "replicas": nrep}


def oracle_window(case, seqs):
    """Host copies of the windows of sequences `seqs` (the oracle's input)
    and their KV bytes."""
    from oracle.slices import host_slices
    d = case.dims
    kv = 0
    for b in seqs:
        lo = max(0, case.q_pos_host[b] - case.window + 1)
        hi = min(case.q_pos_host[b] + d["q_len"], case.seq_lens_host[b])
        kv += d["num_kv_heads"] * max(0, hi - lo) * 2 * d["head_dim"] * 2
    return host_slices(case, seqs, margin=0), kv


def time_oracle(case, budget_s, threads=None, steps=None, warmup=0):
    """The fp64 oracle (``oracle.attention``, as it stands) timed on the host
    cores over a bounded sample of the workload: the first n sequences (all
    heads and draft rows of each), n sized from one sequence's cost so a call
    takes about a quarter of the budget.  Runs `steps` calls after `warmup`
    untimed ones, or calls until the budget is spent.  Both the CPU-baseline
    leg and the reference arm use this routine.  Returns seconds per call,
    the KV GB/s of the sample, and how it was sampled."""
    import oracle
    B = case.q.shape[0]
    threads = threads or oracle.default_threads()
    (q, k, v, base, sl, qp), _ = oracle_window(case, [0])
    t0 = time.perf_counter()
    oracle.attention(q, k, v, sl, qp, case.window, case.scale, base=base, threads=threads)
    per_seq = max(time.perf_counter() - t0, 1e-6)
    per_call_budget = budget_s / 4 if steps is None else budget_s / max(steps + warmup, 1)
    n_seq = max(1, min(B, int(per_call_budget / per_seq)))
    (q, k, v, base, sl, qp), kv = oracle_window(case, list(range(n_seq)))
    for _ in range(warmup):
        oracle.attention(q, k, v, sl, qp, case.window, case.scale, base=base, threads=threads)
    calls = 0
    t0 = time.perf_counter()
    while True:
        oracle.attention(q, k, v, sl, qp, case.window, case.scale, base=base, threads=threads)
        calls += 1
        el = time.perf_counter() - t0
        if (steps is not None and calls >= steps) or (steps is None and el >= budget_s):
            break
    per_call = el / calls
    used = min(threads, n_seq * case.q.shape[2])
    sample = (f"{calls} fp64 oracle calls over {n_seq} of {B} sequences (all heads and draft rows "
              f"of each), {el:.2f} s, {used} threads busy of {threads} started")
    return {"seconds_per_call": per_call, "kv_gbs": kv / per_call / 1e9, "sample": sample,
            "threads_used": used, "sequences": n_seq}


def cpu_baseline(case, budget_s):
    """The oracle at all host threads and at one thread (a third of the
    budget), reported in the metric's unit (KV GB/s of the sampled
    sequences)."""
    host = os.cpu_count() or 1
    a = time_oracle(case, budget_s)
    one = time_oracle(case, max(0.2, budget_s / 3), threads=1)
    return {"value": round(a["kv_gbs"], 6), "unit": UNIT, "cores": a["threads_used"],
            "threads_used": a["threads_used"], "host_cores": host, "kind": "oracle",
            "sample": a["sample"],
            "single_thread": {"value": round(one["kv_gbs"], 6), "unit": UNIT, "cores": 1,
                              "sample": one["sample"]}}


# ------------------------------------------------------------------- main

def aggregate(seconds, bytes_per_step, steps, dist=None, device="cpu"):
    """Whole-job throughput: the slowest rank's time, every rank's bytes.
    Returns (max seconds over ranks, aggregate GB/s)."""
    world = 1
    secs = torch.tensor([float(seconds)], dtype=torch.float64, device=device)
    if dist is not None:
        world = dist.get_world_size()
        dist.all_reduce(secs, op=dist.ReduceOp.MAX)
    slowest = float(secs.item())
    return slowest, bytes_per_step * steps * world / slowest / 1e9


def source_digest():
    """sha256 (first 16 hex digits) of the CUDA library's sources: a traffic
    figure taken by ncu applies only while it matches."""
    import hashlib
    csrc = os.path.join(ROOT, "sliding_window_speculative_gb300", "csrc")
    h = hashlib.sha256()
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload):
    """DRAM bytes (read + write) per launch of the dominant kernel, from the
    committed ncu summary profiles/traffic.json, or None when that capture
    predates the current kernel sources."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
    except Exception:
        return None, None
    if d.get("source_sha") != source_digest():
        return None, "stale"
    w = d.get("workloads", {}).get(workload)
    if not w:
        return None, None
    return int(w["dram_bytes_per_launch"]), w.get("kernel")


def launch_floor(steps, graph_len=1000):
    """Per-launch time of a one-element kernel replayed from a CUDA graph the
    way the calls are: the floor any single-kernel call sits on."""
    x = torch.zeros(1, device="cuda")
    stream = torch.cuda.Stream()
    n = max(1, min(graph_len, steps))
    with torch.cuda.stream(stream):
        for _ in range(3):
            x.add_(1.0)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(n):
            x.add_(1.0)
    with torch.cuda.stream(stream):
        g.replay()
    stream.synchronize()
    reps = max(1, steps // n)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    hold_stream(stream)
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(reps):
            g.replay()
        end.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(end) * 1e3 / (reps * n)


def launch_floor_stream(steps):
    """Per-launch time of the same one-element kernel launched from the host
    one call at a time (no graph): the floor of an eager caller."""
    x = torch.zeros(1, device="cuda")
    stream = torch.cuda.Stream()
    n = max(1, min(steps, 2000))
    with torch.cuda.stream(stream):
        for _ in range(3):
            x.add_(1.0)
    stream.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        start.record(stream)
        for _ in range(n):
            x.add_(1.0)
        end.record(stream)
    torch.cuda.synchronize()
    return start.elapsed_time(end) * 1e3 / n


NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e nominal bandwidth

# every configuration of the workload table beside the headline one: tiny
# (q_len 1 and 8), window-vs-full (W 188 and the whole context), the batched
# verify, and the nine bandwidth-stress combinations
ALSO_DEFAULT = (["tiny_q1", "tiny_q8", "window_vs_full_w188", "window_vs_full_w4096", "batched"] +
                [f"stress_w{w}_q{q}" for w in (188, 512, 1024) for q in (1, 8, 64)])


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def tensor_peak():
    """Dense bf16 TFLOP/s for a kernel timed alone (burst), and its source."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def extra_entry(name, dev, peak, tpeak, sms, steps=None, cpu_budget=0.0):
    """One more workload measured like the main one (device time, graph
    replay, L2 defeated): time per call, HBM and tensor-pipe fractions of
    the peaks, the plan the library picks for it and, with a CPU budget, the
    oracle on a sample of it at all host threads and at one."""
    import sliding_window_speculative_gb300 as swa
    case = make_workload(name, dev)
    kv, total = workload_bytes(case)
    steps = steps or max(50, min(2000, int(0.3e9 / max(total, 1))))
    r = time_device(case, steps, 5)
    plan = swa.swa_plan(swa.dims_of(case.q, case.k_cache), case.window, sms)
    sec = r["us_per_call"] * 1e-6
    ach = total / sec / 1e9
    tf = workload_flops(case) / sec / 1e12
    entry = {"kernel": KERNEL_NAMES.get(plan["kernel"], "?"),
             "us_per_call": round(r["us_per_call"], 3),
             "kv_gbs": round(kv / sec / 1e9, 2),
             "achieved_gbs": round(ach, 2), "frac": round(ach / peak, 4),
             "frac_nominal": round(ach / NOMINAL_HBM_GBS, 4),
             "useful_tflops": round(tf, 3), "tensor_frac": round(tf / tpeak, 5),
             "tokens_per_s": round(case.q.shape[0] * case.q.shape[1] / sec),
             "steps": steps, "replicas": r["replicas"], "l2": r["l2_scheme"],
             "splits": plan["num_splits"], "traffic": ncu_traffic(name)[0]}
    if cpu_budget > 0:
        entry["cpu_baseline"] = cpu_baseline(case, cpu_budget)
    del case
    torch.cuda.empty_cache()
    return entry


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="single_stream")
    ap.add_argument("--splits", type=int, default=0, help="force a split count (0 = heuristic)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--also", default=",".join(ALSO_DEFAULT),
                    help="extra workloads measured the same way (rank 0, device time)")
    ap.add_argument("--cpu-budget", type=float, default=10.0,
                    help="seconds of oracle time for the headline workload's CPU baseline")
    ap.add_argument("--also-cpu-budget", type=float, default=1.2,
                    help="seconds of oracle time for each extra workload's CPU baseline")
    args = ap.parse_args()

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        return main_reference(args, world, rank)

    from sliding_window_speculative_gb300 import build as libbuild
    if rank == 0:
        libbuild.build()
    dist = None
    if world > 1:
        import torch.distributed as tdist
        torch.cuda.set_device(local)
        tdist.init_process_group("nccl")
        dist = tdist
        dist.barrier()
        libbuild.build()
    else:
        torch.cuda.set_device(local)
    import sliding_window_speculative_gb300 as swa
    dev = torch.device("cuda", local)
    case = make_workload(args.workload, dev, seed=rank)
    kv, total = workload_bytes(case)
    plan = swa.swa_plan(swa.dims_of(case.q, case.k_cache, args.splits), case.window,
                        torch.cuda.get_device_properties(dev).multi_processor_count)

    sampler = ClockSampler(local)
    r = time_device(case, args.steps, args.warmup, args.splits, dist=dist)
    clocks = sampler.stop(*r["wall"])
    seconds, value = aggregate(r["seconds"], kv, args.steps, dist, dev)
    us = seconds * 1e6 / args.steps

    peak, peak_src = peaks()
    tpeak, _ = tensor_peak()
    launches_per_call = 1 + plan["merge"]
    achieved = total / (us * 1e-6) / 1e9
    traffic, traffic_kernel = ncu_traffic(args.workload)
    floor_us = launch_floor(args.steps) if rank == 0 else None
    floor_stream_us = launch_floor_stream(args.steps) if rank == 0 else None
    line = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": us / 1e3,
        "us_per_call": round(us, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": args.workload, **case.dims, "window": case.window,
                   "kv_bytes_per_call": kv, "bytes_per_call": total,
                   "l2": (f"defeated by {r['replicas']} input replicas: {r['l2_scheme']}"
                          if r["replicas"] > 1 else "inputs larger than L2"),
                   "timing": ("CUDA graph of calls, CUDA events on the launching stream; a "
                              "sleep kernel ahead of the start event lets the host queue the "
                              "replays first, so the events bracket device execution"),
                   "plan": plan, "parallelism": f"replicas x{world}" if world > 1 else "1 GPU"},
        "roofline": {"bound": "hbm", "kernel": KERNEL_NAMES.get(plan["kernel"], "?") +
                     (" + swa_merge_kernel" if plan["merge"] else ""),
                     "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_source": peak_src,
                     "nominal_peak": NOMINAL_HBM_GBS,
                     "frac_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
                     "traffic": traffic,
                     "traffic_source": ("profiles/traffic.json (ncu dram__bytes_read.sum + "
                                        "dram__bytes_write.sum per launch)" if traffic else
                                        ("stale: kernel sources changed since the capture"
                                         if traffic_kernel == "stale" else None)),
                     "launch_floor_us": round(floor_us, 3) if floor_us else None,
                     "launch_floor_stream_us": (round(floor_stream_us, 3)
                                                if floor_stream_us else None),
                     "floor_frac": round(floor_us * launches_per_call / us, 4) if floor_us else None,
                     "note": "achieved = algorithmic bytes per call / device time per call "
                             "(one attention kernel per call when the plan does not split); "
                             "floor_frac = launch floor x kernels per call / time per call; "
                             "launch floors: a one-element kernel replayed from a CUDA graph, "
                             "and launched from the host one call at a time"},
        "clocks": clocks,
        "gpu_launches": launches_per_call * args.steps,
    }
    if rank == 0 and not args.no_e2e:
        # host loop: per step one input copy, the prepared call, one output copy
        n_e2e = min(args.steps, 2000)
        line["e2e"] = e2e_entry(case, n_e2e, args.warmup, graph=False)
        line["e2e"]["how"] = ("host loop per step: H2D copy of the packed inputs from pinned "
                              "memory, the prepared swa_append_verify_attn call, D2H copy of "
                              "out and lse into pinned memory; the K steps timed three times, "
                              "the median kept")
        # the same step captured once as one CUDA graph, replayed per step
        line["e2e"]["graph"] = e2e_entry(case, n_e2e, args.warmup, graph=True)
        if world == 1 and args.workload != "batched":
            bcase = make_workload("batched", dev)
            line["e2e"]["batched"] = e2e_entry(bcase, min(n_e2e, 500), args.warmup, graph=False)
            line["e2e"]["batched"]["graph"] = e2e_entry(bcase, min(n_e2e, 500), args.warmup,
                                                        graph=True)
            del bcase
    if rank == 0 and world == 1 and args.also:
        sms = torch.cuda.get_device_properties(dev).multi_processor_count
        budget = 0.0 if args.no_cpu_baseline else args.also_cpu_budget
        line["also"] = {name: extra_entry(name, dev, peak, tpeak, sms, cpu_budget=budget)
                        for name in args.also.split(",") if name and name != args.workload}
        # greedy verification of the draft block over a Gemma-size vocabulary
        # (one sequence, and a 64-sequence batch)
        line["accept"] = [time_accept(1, 8, 262144), time_accept(64, 8, 262144, steps=500)]
        # the bandwidth-stress batch (inputs larger than L2) on a paged cache
        line["paged"] = [time_paged("stress_w188_q8", 16), time_paged("stress_w188_q8", 64)]
        # sliding-window prefill chunks of 512 tokens (one sequence, and 64)
        line["prefill"] = {name: extra_entry(name, dev, peak, tpeak, sms, steps=200)
                           for name in ("prefill_q512", "prefill_q512_b64")}
        # the cache write of the verify block fused into the attention call
        line["append"] = [time_append("single_stream"), time_append("batched"),
                          time_append("stress_w188_q8", steps=200)]
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(case, args.cpu_budget)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


def main_reference(args, world, rank):
    """The oracle as the reference arm: each step is one oracle call over a
    bounded sample of the workload's sequences (all heads and rows of each),
    sized so that warm-up plus K steps stay within about three minutes; timed
    by the same routine as the CPU-baseline leg of the GPU arm."""
    if rank != 0:
        return
    from oracle import build as oraclebuild
    oraclebuild.build()
    case = make_workload(args.workload, "cpu")
    r = time_oracle(case, 150.0, steps=args.steps, warmup=args.warmup)
    per_step = r["seconds_per_call"]
    value = r["kv_gbs"]
    line = {
        "metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": per_step * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "impl": "reference",
        "config": {"workload": args.workload, **case.dims, "window": case.window,
                   "sampled_sequences": r["sequences"]},
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": r["threads_used"],
                         "threads_used": r["threads_used"], "host_cores": os.cpu_count() or 1,
                         "kind": "oracle", "sample": r["sample"]},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()

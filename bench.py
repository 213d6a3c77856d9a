#!/usr/bin/env python3
"""Benchmark of the paged-KV attention hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One bench step is one continuous-batching step of the mixed workload (a
Llama-3.1-8B-like layer, GQA 32/8, head_dim 128, 16-token pages): one
26,926-token prompt prefilled in 2,048-row chunks against its own cached
prefix, plus 32 decode rows with contexts ~ U[128, 16384]; step c appends
chunk c and one token per decode row (kv_append), then prefills chunk c
(paged_attn_prefill) and decodes the 32 rows (paged_attn_decode: split
kernel + combine).  Both need only the append, so they run side by side:
the prefill, bound by the tensor cores, on part of the SMs
(pkv_overlap_prefill_ctas) and the decode, bound by HBM, on a second stream
over the rest (--sequential runs them one after the other on one stream).
Steps cycle through the 14 chunks; with K a multiple of
14 every chunk is timed equally often.  All inputs (1.2 GB pool, every
step's rows) are resident in HBM before the timed region; the pool is larger
than L2, so no separate flush is needed there.

The JSON line reports the step time (value, us per step) and, from CUDA
events around every call (on the stream that runs it), decode HBM GB/s and
prefill TFLOP/s; the roofline object is for the prefill kernel, which
dominates the step, with the share of the SMs it held.  "configs" holds
the other workloads (single-sequence decode, 1,024-token prefill, batched
decode, INT8 32k decode, 16-token verify steps through the multi-token
decode, the fused attention-input step on a 2,048-token chunk) timed with an
L2 flush before each run that leaves L2 clean and cold (a 512 MB write, then
a 512 MB read; the decode lines also give the time after the write alone,
whose dirty lines the timed launch then writes back).
`--impl reference` times the fp64 CPU oracle on the host cores instead.
"""
import argparse
import json
import os
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_flash_gb300 import workloads as W  # noqa: E402

# Per-launch DRAM traffic and tensor-pipe share of the prefill kernel come from
# the committed ncu summary below; each figure carries the SHA-256 of the
# kernel's sources when it was captured, and is reported only while the
# sources still match (otherwise null: the counters describe another kernel).
PREFILL_PROFILE = os.path.join(ROOT, "profiles", "prefill_kernel_mixed_step.md")
PREFILL_SOURCES = [os.path.join(ROOT, "paged_kv_flash_gb300", "csrc", f)
                   for f in ("prefill.cu", "common.cuh", "internal.h")]
# Dense bf16 tensor-core peak of one GB300 from NVIDIA's HGX B300 figures:
# 36 PFLOP/s FP16/BF16 per 8 GPUs, quoted with 2:4 sparsity, so 2.25 PFLOP/s
# dense per GPU.
SPEC_BF16_TFLOPS = 2250.0

METRIC = ("decode attn µs & HBM GB/s (% of 8 TB/s); prefill attn TFLOP/s (% of peak)")
NOMINAL_HBM_GBS = 8000.0
D = W.HEAD_DIM
SCALE = 1.0 / np.sqrt(D)


def peaks():
    """(HBM GB/s, bf16 burst TFLOP/s, bf16 sustained TFLOP/s, source, median SM
    MHz under load while they were measured or None)."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        mhz = (p.get("clocks_under_load") or {}).get("sm_mhz_median")
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p["bf16_tflops_sustained"]), \
            "measured", (float(mhz) if mhz else None)
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback", None


def sources_sha256(paths):
    import hashlib
    h = hashlib.sha256()
    for path in paths:
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def prefill_profile():
    """Figures of the committed prefill ncu summary whose recorded source hash
    matches the current prefill sources: {key: float}.  The summary holds
    lines `key = value  (sha256 <hex>)`."""
    out = {}
    try:
        cur = sources_sha256(PREFILL_SOURCES)
        with open(PREFILL_PROFILE) as f:
            for line in f:
                line = line.strip().strip("`")
                if " = " not in line or "(sha256 " not in line:
                    continue
                key, rest = line.split(" = ", 1)
                val, sha = rest.split("(sha256 ", 1)
                if sha.rstrip(")").strip() == cur:
                    out[key.strip()] = float(val.strip())
    except (OSError, ValueError):
        pass
    return out


# ------------------------------------------------------------------ clocks

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.path = tempfile.mktemp(prefix="pkv_clocks_", suffix=".csv")
        self.proc = None
        self.dev = device_index

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 8:
                    continue
                try:
                    sm.append(float(parts[0]))
                    smax.append(float(parts[1]))
                    power.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[4:8]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(smax)),
                "power_w_max": float(max(power)), "samples": len(sm),
                "reasons": sorted(reasons)}


# ------------------------------------------------------------- helpers

def to_dev_bf16(torch, bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def to_dev(torch, a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def pinned_bf16(torch, bits):
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.pin_memory()


def prefill_flops(chunk_len, L, Hq):
    """4 * D * (keys seen) per query row and head: QK^T and PV, causal part only."""
    first = L - chunk_len + 1                    # keys seen by the chunk's first row
    keys = chunk_len * first + chunk_len * (chunk_len - 1) // 2
    return 4.0 * D * Hq * keys


def decode_bytes(lens, Hkv, per_pos=2 * D * 2):
    return float(np.asarray(lens, np.int64).sum()) * Hkv * per_pos


# ------------------------------------------------------- mixed workload

class Mixed:
    """Device-resident mixed workload and its step function.  overlap: the
    prefill runs on part of the SMs (pkv_overlap_prefill_ctas) while the
    decode runs beside it on a second stream; else one after the other."""

    def __init__(self, torch, pk, overlap=True):
        self.torch, self.pk = torch, pk
        self.overlap = overlap
        # the prefill's stream goes first when both wait for the append, so
        # that it takes its SMs and the decode's CTAs fill the others
        self.s_pre = torch.cuda.Stream(priority=-1)
        self.s_dec = torch.cuda.Stream()
        wl = W.mixed_step()
        self.wl = wl
        self.R = len(wl.decode_lens0)
        self.pool = pk.Pool(to_dev_bf16(torch, wl.k_pool), to_dev_bf16(torch, wl.v_pool))
        bt = wl.layout.block_table
        self.bt_all = to_dev(torch, bt)
        self.bt_prompt = to_dev(torch, bt[:1])
        self.bt_dec = to_dev(torch, np.ascontiguousarray(bt[1:]))
        self.steps = []
        for s in wl.steps:
            cu_app, lens_app = wl.step_append(s)
            st = dict(
                cu_app=to_dev(torch, cu_app), lens_app=to_dev(torch, lens_app),
                k_new=to_dev_bf16(torch, s.k_new), v_new=to_dev_bf16(torch, s.v_new),
                q_chunk=to_dev_bf16(torch, s.q_chunk), q_dec=to_dev_bf16(torch, s.q_decode),
                cu_q=to_dev(torch, W.cu_from_counts([s.chunk_len])),
                lens_p=to_dev(torch, np.array([s.prefill_len], np.int32)),
                lens_d=to_dev(torch, s.decode_lens), chunk_len=s.chunk_len, context=s.prefill_len,
                max_dec=int(s.decode_lens.max()),
                flops=prefill_flops(s.chunk_len, s.prefill_len, wl.Hq),
                dbytes=decode_bytes(s.decode_lens, wl.Hkv),
                host=s)
            S, C, ws, _ = pk.decode_plan(self.R, wl.Hq, wl.Hkv, st["max_dec"])
            st["splits"] = S
            st["ctas"] = pk.overlap_prefill_ctas(st["flops"], st["dbytes"])
            st["launches"] = 3 + (1 if S > 1 else 0)
            self.steps.append(st)
        plans = [pk.decode_plan(self.R, wl.Hq, wl.Hkv, s["max_dec"]) for s in self.steps]
        self.ws = pk.decode_workspace(max(p[2] for p in plans), max(p[3] for p in plans))
        self.ws_p = pk.prefill_workspace()
        T = max(s["chunk_len"] for s in self.steps)
        self.out_p = torch.empty((T, wl.Hq, D), dtype=torch.bfloat16, device="cuda")
        self.lse_p = torch.empty((T, wl.Hq), dtype=torch.float32, device="cuda")
        self.out_d = torch.empty((self.R, wl.Hq, D), dtype=torch.bfloat16, device="cuda")
        self.lse_d = torch.empty((self.R, wl.Hq), dtype=torch.float32, device="cuda")

    def step(self, i, ev=None, inputs=None, outs=None):
        """Step i (chunk i mod 14) on the current stream's timeline: it starts
        after the work queued there and the work queued there after it waits
        for it.  ev: 5 events to record (step start, append end, prefill end,
        decode start, decode end) or None.  inputs: per-step device tensors
        that replace the resident ones (end-to-end path); outs: (out_p,
        lse_p, out_d, lse_d) to write instead of the resident outputs."""
        torch, pk, wl = self.torch, self.pk, self.wl
        st = self.steps[i % len(self.steps)]
        x = inputs or st
        out_p, lse_p, out_d, lse_d = outs or (self.out_p, self.lse_p, self.out_d, self.lse_d)
        n = st["chunk_len"]
        cur = torch.cuda.current_stream()
        sp = self.s_pre if self.overlap else cur
        sd = self.s_dec if self.overlap else cur
        sp.wait_stream(cur)
        if ev: ev[0].record(sp)
        pk.kv_append(self.pool, x["k_new"], x["v_new"], st["cu_app"], self.bt_all, st["lens_app"],
                     stream=sp)
        if ev: ev[1].record(sp)
        if self.overlap:
            sd.wait_stream(sp)                    # the decode needs the append only
        pk.paged_attn_prefill(self.pool, x["q_chunk"], st["cu_q"], self.bt_prompt, st["lens_p"],
                              n, SCALE, workspace=self.ws_p, out=out_p[:n], lse=lse_p[:n],
                              stream=sp, num_ctas=st["ctas"] if self.overlap else 0)
        if ev: ev[2].record(sp)
        if ev: ev[3].record(sd)
        pk.paged_attn_decode(self.pool, x["q_dec"], self.bt_dec, st["lens_d"], st["max_dec"],
                             SCALE, workspace=self.ws, out=out_d, lse=lse_d, stream=sd)
        if ev: ev[4].record(sd)
        if self.overlap:
            cur.wait_stream(sp)
            cur.wait_stream(sd)


def max_over_ranks(torch, x):
    """The largest x over the ranks of the default process group (x itself
    without one): the job's time is its slowest replica's."""
    dist = torch.distributed
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def time_mixed(torch, pk, mixed, K, Wu, world, rank):
    dist = torch.distributed if world > 1 else None
    for i in range(Wu):
        mixed.step(i)
    torch.cuda.synchronize()
    assert pk.poll_device_error() == pk.OK, "device-side error during warm-up"
    nsteps = len(mixed.steps)
    # per-step events (step start, append end, prefill end, decode start and end)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)] for _ in range(K)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    t0.record()
    for i in range(K):
        mixed.step(Wu + i, ev=evs[i])
    t1.record()
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    clk = clocks.stop()
    assert pk.poll_device_error() == pk.OK, "device-side error in the timed region"
    total_ms = t0.elapsed_time(t1)
    app_ms = pre_ms = dec_ms = 0.0
    flops = dbytes = 0.0
    launches = 0
    # per chunk of the prompt (step i runs chunk i mod 14): summed phase
    # times, summed step times (from this step's first event to the next
    # step's), count
    per = [[0.0, 0.0, 0.0, 0.0, 0] for _ in range(nsteps)]
    cta_ms = 0.0                                  # prefill time x its CTA count
    all_ctas = pk.prefill_plan()[0]
    ctas_of = lambda st: st["ctas"] if mixed.overlap else all_ctas
    for i in range(K):
        e = evs[i]
        c = (Wu + i) % nsteps
        st = mixed.steps[c]
        a, p, d = e[0].elapsed_time(e[1]), e[1].elapsed_time(e[2]), e[3].elapsed_time(e[4])
        whole = e[0].elapsed_time(evs[i + 1][0] if i + 1 < K else t1)
        app_ms += a
        pre_ms += p
        dec_ms += d
        cta_ms += p * ctas_of(st)
        for j, v in enumerate((a, p, d, whole)):
            per[c][j] += v
        per[c][4] += 1
        flops += st["flops"]
        dbytes += st["dbytes"]
        launches += st["launches"]
    chunks = []
    for c, (a, p, d, w, n) in enumerate(per):
        if not n:
            continue
        st = mixed.steps[c]
        chunks.append({"chunk": c, "rows": st["chunk_len"], "context": st["context"],
                       "prefill_ctas": ctas_of(st),
                       "step_us": round(w * 1e3 / n, 2),
                       "append_us": round(a * 1e3 / n, 2), "prefill_us": round(p * 1e3 / n, 2),
                       "prefill_TFLOPs": round(st["flops"] / (p * 1e-3 / n) / 1e12, 1),
                       "decode_us": round(d * 1e3 / n, 2),
                       "decode_GBps": round(st["dbytes"] / (d * 1e-3 / n) / 1e9, 1)})
    # The step time weighs the 14 chunks equally (the mean over chunks of the
    # chunk's mean step time), so that it does not depend on which chunks
    # K steps happen to cover; with K < 14 it is the plain mean.
    if len(chunks) == nsteps:
        step_ms = float(np.mean([per[c][3] / per[c][4] for c in range(nsteps)]))
        balanced = True
    else:
        step_ms, balanced = total_ms / K, False
    step_ms = max_over_ranks(torch, step_ms)
    total_ms = max_over_ranks(torch, total_ms)
    return dict(total_ms=total_ms, step_ms=step_ms, balanced=balanced, app_ms=app_ms,
                pre_ms=pre_ms, dec_ms=dec_ms, flops=flops, dbytes=dbytes, launches=launches,
                clocks=clk, chunks=chunks, overlap=mixed.overlap, steps=K,
                sm_share=cta_ms / pre_ms / all_ctas if pre_ms > 0 else 1.0)


def time_e2e(torch, pk, mixed, K, first):
    """The steps first .. first + K - 1 (the device-timed steps when K is a
    whole number of passes over the 14 chunks) through the public API from
    pinned host buffers: every step copies its inputs host->device and reads
    its outputs back.  The copies overlap the kernels, as a serving loop
    would run them: step i+1's inputs go up on one copy stream while step i
    computes, and step i's outputs come back on another from one of two
    output buffers (the compute stream waits for a buffer's read-back before
    reusing it)."""
    host = []
    for st in mixed.steps:
        s = st["host"]
        host.append(dict(k_new=pinned_bf16(torch, s.k_new), v_new=pinned_bf16(torch, s.v_new),
                         q_chunk=pinned_bf16(torch, s.q_chunk),
                         q_dec=pinned_bf16(torch, s.q_decode)))
    nsteps = len(mixed.steps)
    dev = [dict((k, torch.empty_like(v, device="cuda")) for k, v in h.items()) for h in host]
    outs = [(mixed.out_p, mixed.lse_p, mixed.out_d, mixed.lse_d),
            tuple(torch.empty_like(t) for t in (mixed.out_p, mixed.lse_p, mixed.out_d,
                                                 mixed.lse_d))]
    host_out = tuple(torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in outs[0])
    compute = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(nsteps)]       # inputs of chunk j are on the device
    ev_used = [torch.cuda.Event() for _ in range(nsteps)]     # step using chunk j's inputs is done
    ev_done = [torch.cuda.Event() for _ in range(2)]          # step writing output buffer b is done
    ev_back = [torch.cuda.Event() for _ in range(2)]          # output buffer b has been read back
    counts = {"h2d": 0, "d2h": 0}
    used = [False] * nsteps
    back = [False, False]

    def upload(i):
        j = i % nsteps
        with torch.cuda.stream(up):
            if used[j]:
                up.wait_event(ev_used[j])
            for k, v in host[j].items():
                dev[j][k].copy_(v, non_blocking=True)
                counts["h2d"] += v.numel() * v.element_size()
            ev_in[j].record(up)

    def run(i):
        j, b = i % nsteps, i % 2
        compute.wait_event(ev_in[j])
        if back[b]:
            compute.wait_event(ev_back[b])
        mixed.step(i, inputs=dev[j], outs=outs[b])
        ev_used[j].record(compute)
        used[j] = True
        ev_done[b].record(compute)
        n = mixed.steps[j]["chunk_len"]
        with torch.cuda.stream(down):
            down.wait_event(ev_done[b])
            op, lp, od, ld = outs[b]
            host_out[0][:n].copy_(op[:n], non_blocking=True)
            host_out[1][:n].copy_(lp[:n], non_blocking=True)
            host_out[2].copy_(od, non_blocking=True)
            host_out[3].copy_(ld, non_blocking=True)
            ev_back[b].record(down)
        back[b] = True
        counts["d2h"] += (n * op.shape[1] * D * 2 + n * lp.shape[1] * 4 + od.numel() * 2 +
                          ld.numel() * 4)

    def loop(start, n_iter):
        upload(start)
        for i in range(start, start + n_iter):
            if i + 1 < start + n_iter:
                upload(i + 1)
            run(i)
        t_enq = time.perf_counter()                # everything queued; the GPU still runs
        torch.cuda.synchronize()
        return t_enq

    loop(first, nsteps)                            # warm-up pass over every chunk
    counts["h2d"] = counts["d2h"] = 0
    t0 = time.perf_counter()
    t_enq = loop(first, K)
    dt = time.perf_counter() - t0
    return dt * 1e6 / K, counts["h2d"] // K, counts["d2h"] // K, (t_enq - t0) * 1e6 / K


# ------------------------------------------------------ other workloads

class L2Flush:
    """Evicts a timed launch's inputs from L2 between timed runs: writes a
    512 MB buffer (four times the 129 MB L2), then reads another 512 MB, so
    the dirty lines of that write go back to HBM before the timed region
    instead of inside it (the launch starts on a clean, cold L2, as under
    ncu's cache control).  flush(clean=False) does the write alone."""

    def __init__(self, torch):
        self.w = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
        self.r = torch.ones(128 << 20, dtype=torch.float32, device="cuda")

    def __call__(self, clean=True):
        self.w.zero_()
        if clean:
            self.r.sum()


def time_events(torch, fn, iters=20, warm=5, flush=None, clean=True):
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ts = []
    for i in range(iters + warm):
        if flush is not None:
            flush(clean)
        s.record()
        fn()
        e.record()
        torch.cuda.synchronize()
        if i >= warm:
            ts.append(s.elapsed_time(e) * 1e3)
    return float(np.median(ts)), float(np.min(ts))


def time_graph(torch, fn, reps=20):
    """Back-to-back launches captured in one CUDA graph (per-launch us)."""
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(st):
        fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            for _ in range(reps):
                fn()
    torch.cuda.current_stream().wait_stream(st)
    g.replay()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(5):
        g.replay()
    e.record()
    torch.cuda.synchronize()
    return s.elapsed_time(e) * 1e3 / (5 * reps)


def other_configs(torch, pk, hbm, bf16):
    flush = L2Flush(torch)
    res = {}

    def decode_entry(name, case, pool, per_pos, smooth=None, graph=False, fused=False):
        q = to_dev_bf16(torch, case.q)
        bt, sl = to_dev(torch, case.layout.block_table), to_dev(torch, case.seq_lens)
        ms = int(case.seq_lens.max())
        S, C, wsb, zb = pk.decode_plan(case.B, case.Hq, case.Hkv, ms, dtype=pool.dtype)
        ws = pk.decode_workspace(wsb, zb)
        out = torch.empty_like(q)
        lse = torch.empty((case.B, case.Hq), dtype=torch.float32, device="cuda")
        w = to_dev(torch, smooth) if smooth is not None else None
        fn = lambda: pk.paged_attn_decode(pool, q, bt, sl, ms, SCALE, k_smooth=w, workspace=ws,
                                          out=out, lse=lse, fused=fused)
        med, mn = time_events(torch, fn, flush=flush)
        med_w, _ = time_events(torch, fn, flush=flush, clean=False)
        byts = decode_bytes(case.seq_lens, case.Hkv, per_pos)
        r = {"us": round(med, 2), "us_min": round(mn, 2), "GBps": round(byts / med / 1e3, 1),
             "frac_of_8TBps": round(byts / med / 1e3 / NOMINAL_HBM_GBS, 4),
             "frac_of_measured": round(byts / med / 1e3 / hbm, 4), "bytes": int(byts),
             "splits": S, "cold_l2": "clean",
             "us_write_only_flush": round(med_w, 2),
             "frac_of_measured_write_only_flush": round(byts / med_w / 1e3 / hbm, 4)}
        if fused:
            r["note"] = "combine fused into the split kernel (pkv_paged_attn_decode_fused)"
        if graph:
            g = time_graph(torch, fn)
            r["graph_us_per_launch"] = round(g, 2)
            r["graph_note"] = "back-to-back launches in one CUDA graph, warm L2"
        res[name] = r
        assert pk.poll_device_error() == pk.OK
        return out

    c1 = W.decode_1k()
    p1 = pk.Pool(to_dev_bf16(torch, c1.k_pool), to_dev_bf16(torch, c1.v_pool))
    decode_entry("decode_1k_b1_gqa16x8", c1, p1, 512, graph=True)
    decode_entry("decode_1k_b1_gqa16x8_fused", c1, p1, 512, graph=True, fused=True)
    c3 = W.batched_decode()
    p3 = pk.Pool(to_dev_bf16(torch, c3.k_pool), to_dev_bf16(torch, c3.v_pool))
    decode_entry("batched_decode_b64_gqa32x8", c3, p3, 512)
    decode_entry("batched_decode_b64_gqa32x8_fused", c3, p3, 512, fused=True)
    del c3, p3
    for B in (1, 8):
        # The same keys and values in a bf16 pool and in INT8 pools with and
        # without key smoothing; the bf16 decode's output is the reference
        # the quantisation error is measured against.
        app, q = W.int8_long_decode(B=B)
        case = W.DecodeCase(32, app.Hkv, app.seq_lens, app.layout, q, None, None)
        kn, vn = to_dev_bf16(torch, app.k_new), to_dev_bf16(torch, app.v_new)
        cu, btd, sld = (to_dev(torch, app.cu_new), to_dev(torch, app.layout.block_table),
                        to_dev(torch, app.seq_lens))
        pb = pk.Pool.empty(app.layout.num_pages, app.Hkv)
        pk.kv_append(pb, kn, vn, cu, btd, sld)
        ref = decode_entry(f"bf16_decode_32k_b{B}", case, pb, 512).float()
        del pb
        for smooth in (True, False):
            pool = pk.Pool.empty(app.layout.num_pages, app.Hkv, dtype=torch.int8)
            w = app.k_smooth if smooth else None
            pk.kv_append(pool, kn, vn, cu, btd, sld,
                         k_smooth=to_dev(torch, w) if w is not None else None)
            name = f"int8_decode_32k_b{B}" + ("" if smooth else "_no_smoothing")
            o = decode_entry(name, case, pool, 264, smooth=w).float()
            res[name]["rel_l2_err_vs_bf16_decode"] = float(
                f"{((o - ref).norm() / ref.norm()).item():.3g}")
            res[name]["max_abs_err_vs_bf16_decode"] = float(f"{(o - ref).abs().max().item():.3g}")
            res[name]["key_smoothing"] = smooth
            del pool
        del kn, vn
    # 1,024-token prompt: append + prefill
    app, q = W.prefill_prompt()
    pool = pk.Pool.empty(app.layout.num_pages, app.Hkv)
    bt, sl, cu = (to_dev(torch, app.layout.block_table), to_dev(torch, app.seq_lens),
                  to_dev(torch, app.cu_new))
    kn, vn, qd = to_dev_bf16(torch, app.k_new), to_dev_bf16(torch, app.v_new), to_dev_bf16(torch, q)
    out = torch.empty_like(qd)
    lse = torch.empty((1024, 32), dtype=torch.float32, device="cuda")
    ap = lambda: pk.kv_append(pool, kn, vn, cu, bt, sl)
    ap()
    ws_p = pk.prefill_workspace()
    pf = lambda: pk.paged_attn_prefill(pool, qd, cu, bt, sl, 1024, SCALE, workspace=ws_p, out=out,
                                       lse=lse)
    a_med, _ = time_events(torch, ap, flush=flush)
    p_med, p_min = time_events(torch, pf, flush=flush)
    fl = prefill_flops(1024, 1024, 32)
    g = time_graph(torch, pf)
    res["prefill_1k_gqa32x8"] = {
        "us": round(p_med, 2), "us_min": round(p_min, 2), "TFLOPs": round(fl / p_med / 1e6, 1),
        "frac_of_measured_burst": round(fl / p_med / 1e6 / bf16, 4), "flops": fl,
        "graph_us_per_launch": round(g, 2), "graph_TFLOPs": round(fl / g / 1e6, 1),
        "graph_note": "back-to-back launches in one CUDA graph, warm L2",
        "append_us": round(a_med, 2), "append_GBps": round(2 * 2 * 1024 * 8 * 256 / a_med / 1e3, 1)}
    assert pk.poll_device_error() == pk.OK
    del pool
    # short chunks against a long cached context (chunked prefill of a long
    # prompt in 512-row chunks): few long units, cut between CTAs
    for qn, L in ((512, 8192), (128, 32768)):
        c = W.decode_bf16(np.random.default_rng(1007), [L], 32, 8)
        pool = pk.Pool(to_dev_bf16(torch, c.k_pool), to_dev_bf16(torch, c.v_pool))
        qc = to_dev_bf16(torch, W.normal_bf16(np.random.default_rng(1008), (qn, 32, D)))
        cuc, btc, slc = (to_dev(torch, W.cu_from_counts([qn])),
                         to_dev(torch, c.layout.block_table), to_dev(torch, c.seq_lens))
        oc = torch.empty_like(qc)
        lc = torch.empty((qn, 32), dtype=torch.float32, device="cuda")
        pc = lambda: pk.paged_attn_prefill(pool, qc, cuc, btc, slc, qn, SCALE, workspace=ws_p,
                                           out=oc, lse=lc)
        med, mn = time_events(torch, pc, flush=flush)
        fl = prefill_flops(qn, L, 32)
        res[f"prefill_chunk{qn}_ctx{L}_gqa32x8"] = {
            "us": round(med, 2), "us_min": round(mn, 2), "TFLOPs": round(fl / med / 1e6, 1),
            "frac_of_measured_burst": round(fl / med / 1e6 / bf16, 4), "flops": fl}
        assert pk.poll_device_error() == pk.OK
        del pool, c
    # verify steps (multi-token decode), with the prefill kernel on the same step
    rng = np.random.default_rng(1006)
    for name, lens, qlens in (("verify_16tok_1k_b1_gqa32x8", [1024], [16]),
                              ("verify_16tok_b8_ctx4k_8k_gqa32x8",
                               rng.integers(4096, 8193, 8), [16] * 8)):
        res[name] = verify_entry(torch, pk, rng, lens, qlens, flush, hbm, bf16)
    # fused attention inputs for one 2,048-token chunk at positions 14,336..16,383
    fn, byts = qkv_prep_fn(torch, pk, 95)
    med, mn = time_events(torch, fn, flush=flush)
    res["qkv_norm_rope_append_chunk2048"] = {
        "us": round(med, 2), "us_min": round(mn, 2), "GBps": round(byts / med / 1e3, 1),
        "frac_of_measured": round(byts / med / 1e3 / hbm, 4), "bytes": int(byts),
        "note": ("q/k RMSNorm + RoPE + KV write from the q/k/v projection output, "
                 "GQA 32/8; bytes = projection read + q_out, K, V writes + RoPE rows")}
    assert pk.poll_device_error() == pk.OK
    return res


def verify_entry(torch, pk, rng, lens, qlens, flush, hbm, bf16, Hq=32, Hkv=8):
    """A step of qlens[b] tokens per sequence through the multi-token decode
    (split kernel + combine), and the same step through the prefill kernel."""
    case = W.multi_token_decode(rng, lens, qlens, Hq, Hkv)
    pool = pk.Pool(to_dev_bf16(torch, case.k_pool), to_dev_bf16(torch, case.v_pool))
    q, cu = to_dev_bf16(torch, case.q), to_dev(torch, case.cu_q)
    bt, sl = to_dev(torch, case.layout.block_table), to_dev(torch, case.seq_lens)
    mq, ms = int(max(qlens)), int(max(lens))
    S, C, wsb = pk.decode_multi_plan(len(lens), len(case.q), Hq, Hkv, mq, ms)
    ws = torch.empty(max(wsb, 256), dtype=torch.uint8, device="cuda")
    out = torch.empty_like(q)
    lse = torch.empty((len(case.q), Hq), dtype=torch.float32, device="cuda")
    fm = lambda: pk.paged_attn_decode_multi(pool, q, cu, bt, sl, mq, ms, SCALE, workspace=ws,
                                            out=out, lse=lse)
    wsp = pk.prefill_workspace()
    fp = lambda: pk.paged_attn_prefill(pool, q, cu, bt, sl, mq, SCALE, workspace=wsp, out=out,
                                       lse=lse)
    m_med, m_min = time_events(torch, fm, flush=flush)
    p_med, _ = time_events(torch, fp, flush=flush)
    assert pk.poll_device_error() == pk.OK
    byts = decode_bytes(lens, Hkv)
    fl = sum(prefill_flops(qn, L, Hq) for qn, L in zip(qlens, lens))
    r = {"us": round(m_med, 2), "us_min": round(m_min, 2), "GBps": round(byts / m_med / 1e3, 1),
         "frac_of_measured": round(byts / m_med / 1e3 / hbm, 4), "bytes": int(byts),
         "TFLOPs": round(fl / m_med / 1e6, 1), "splits": S,
         "prefill_kernel_us": round(p_med, 2),
         "note": ("multi-token decode (pkv_paged_attn_decode_multi): split kernel + combine; "
                  "prefill_kernel_us = the same step through pkv_paged_attn_prefill")}
    if byts < 64 * 2**20:                         # small steps are launch- and latency-bound
        r["graph_us_per_launch"] = round(time_graph(torch, fm), 2)
        r["graph_prefill_kernel_us_per_launch"] = round(time_graph(torch, fp), 2)
        r["graph_note"] = "back-to-back launches in one CUDA graph, warm L2"
    return r


def qkv_prep_fn(torch, pk, seed, T=2048, L=16384, Hq=32, Hkv=8):
    """The fused attention-input call for T new tokens ending at position L,
    and its algorithmic bytes (every input and output element once)."""
    case = W.qkv_prep_case(seed, [T], [L], Hq=Hq, Hkv=Hkv)
    pool = pk.Pool.empty(case.layout.num_pages, Hkv)
    qkv = to_dev_bf16(torch, case.qkv)
    tf = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    qw, kw, cs, sn = tf(case.q_w), tf(case.k_w), tf(case.cos), tf(case.sin)
    cu, bt, sl = (to_dev(torch, case.cu_new), to_dev(torch, case.layout.block_table),
                  to_dev(torch, case.seq_lens))
    q_out = torch.empty((T, Hq, D), dtype=torch.bfloat16, device="cuda")
    fn = lambda: pk.qkv_norm_rope_append(pool, qkv, Hq, cu, bt, sl, q_norm_w=qw, k_norm_w=kw,
                                         rope_cos=cs, rope_sin=sn, q_out=q_out)
    byts = T * (Hq + 2 * Hkv) * D * 2 * 2 + T * D * 4
    return fn, byts


# ----------------------------------------------------- CPU baseline (oracle)

def oracle_step_sample(mixed_wl, c, n_prefill_rows, n_dec_rows, rng, nthreads):
    """Time the oracle on a sample of step c and extrapolate to the whole step
    by the number of (row, head, key) triples, which its cost is linear in."""
    import oracle
    s = mixed_wl.steps[c]
    bt = mixed_wl.layout.block_table
    # pool state at step c: prompt positions < chunk end, decode rows as of this step
    kp, vp = mixed_wl.k_pool, mixed_wl.v_pool
    # only the rows sampled are evaluated; K/V they read must be present:
    # the prompt's prefix up to this chunk and the decode rows' new tokens.
    t0 = time.perf_counter()
    rows = np.sort(rng.choice(s.chunk_len, min(n_prefill_rows, s.chunk_len),
                              replace=False)).astype(np.int32)
    cu = W.cu_from_counts([s.chunk_len])
    lens = np.array([s.prefill_len], np.int32)
    oracle.paged_attention(kp, vp, s.q_chunk, cu, bt[:1], lens, SCALE, rows=rows,
                           nthreads=nthreads)
    drows = np.sort(rng.choice(len(s.decode_lens), n_dec_rows, replace=False)).astype(np.int32)
    oracle.paged_attention(kp, vp, s.q_decode, np.arange(len(s.decode_lens) + 1, dtype=np.int32),
                           bt[1:], s.decode_lens, SCALE, rows=drows, nthreads=nthreads)
    dt = time.perf_counter() - t0
    first = s.prefill_len - s.chunk_len
    keys_sampled = float(np.sum(first + rows + 1)) + float(np.sum(s.decode_lens[drows]))
    keys_total = (s.chunk_len * (first + 1) + s.chunk_len * (s.chunk_len - 1) / 2 +
                  float(np.sum(s.decode_lens)))
    return dt * keys_total / keys_sampled, dt


def fill_prompt_for_oracle(wl):
    """The oracle reads the pool as it stands after every step's append:
    write all of them with one oracle append (rows regrouped per sequence:
    the prompt's chunks in order, then each decode row's 14 new tokens)."""
    import oracle
    R = len(wl.decode_lens0)
    n = [s.chunk_len for s in wl.steps]
    k_rows = [np.concatenate([s.k_new[:c] for s, c in zip(wl.steps, n)])]
    v_rows = [np.concatenate([s.v_new[:c] for s, c in zip(wl.steps, n)])]
    for r in range(R):
        k_rows.append(np.stack([s.k_new[c + r] for s, c in zip(wl.steps, n)]))
        v_rows.append(np.stack([s.v_new[c + r] for s, c in zip(wl.steps, n)]))
    cu = W.cu_from_counts([sum(n)] + [len(wl.steps)] * R)
    lens = np.concatenate([[wl.steps[-1].prefill_len],
                           wl.decode_lens0 + len(wl.steps)]).astype(np.int32)
    wl.k_pool, wl.v_pool = oracle.kv_append_bf16(wl.k_pool, wl.v_pool, np.concatenate(k_rows),
                                                 np.concatenate(v_rows), cu,
                                                 wl.layout.block_table, lens)


def cpu_baseline(mixed_wl, budget_s=20.0):
    nthreads = os.cpu_count() or 1
    rng = np.random.default_rng(99)
    nsteps = len(mixed_wl.steps)
    est, spent, n = [], 0.0, 0
    # one pass over the 14 steps with a small sample each, enlarged while the
    # budget allows
    rows = 32
    while spent < budget_s and n < 3 * nsteps:
        c = n % nsteps
        e, dt = oracle_step_sample(mixed_wl, c, rows, 4, rng, nthreads)
        est.append((c, e))
        spent += dt
        n += 1
    per_step = {}
    for c, e in est:
        per_step.setdefault(c, []).append(e)
    mean_s = float(np.mean([np.mean(v) for v in per_step.values()]))
    return {"value": round(mean_s * 1e6, 1), "unit": "us", "cores": nthreads, "kind": "oracle",
            "sample": (f"fp64 oracle on {rows} seeded prefill rows and 4 decode rows (all 32 "
                       f"heads) of each of {len(per_step)} mixed steps, {n} samples, "
                       f"{spent:.1f} s of CPU work; scaled to the full step by the number of "
                       f"(row, head, key) triples")}


# ------------------------------------------------------- profiling cases

def _decode_fn(torch, pk, case, pool, smooth=None):
    q = to_dev_bf16(torch, case.q)
    bt, sl = to_dev(torch, case.layout.block_table), to_dev(torch, case.seq_lens)
    ms = int(case.seq_lens.max())
    _, _, wsb, zb = pk.decode_plan(case.B, case.Hq, case.Hkv, ms, dtype=pool.dtype)
    ws = pk.decode_workspace(wsb, zb)
    out = torch.empty_like(q)
    lse = torch.empty((case.B, case.Hq), dtype=torch.float32, device="cuda")
    w = to_dev(torch, smooth) if smooth is not None else None
    return lambda: pk.paged_attn_decode(pool, q, bt, sl, ms, SCALE, k_smooth=w, workspace=ws,
                                        out=out, lse=lse)


def profile_config_case(torch, pk, name):
    """The benchmarked workloads, one kernel each, exactly as `configs` times
    them: (launch function, algorithmic work, unit) or None for other names."""
    if name == "decode_1k":                        # single sequence, 1,024 positions, 16/8
        c = W.decode_1k()
        pool = pk.Pool(to_dev_bf16(torch, c.k_pool), to_dev_bf16(torch, c.v_pool))
        return _decode_fn(torch, pk, c, pool), decode_bytes(c.seq_lens, c.Hkv), "GB/s"
    if name == "decode_b64":                       # 64 sequences, 512..8,192 positions, 32/8
        c = W.batched_decode()
        pool = pk.Pool(to_dev_bf16(torch, c.k_pool), to_dev_bf16(torch, c.v_pool))
        return _decode_fn(torch, pk, c, pool), decode_bytes(c.seq_lens, c.Hkv), "GB/s"
    if name in ("decode_int8_b1", "decode_int8_b8", "append_int8_32k"):
        B = 8 if name == "decode_int8_b8" else 1
        app, qh = W.int8_long_decode(B=B)
        pool = pk.Pool.empty(app.layout.num_pages, app.Hkv, dtype=torch.int8)
        w = to_dev(torch, app.k_smooth)
        kn, vn = to_dev_bf16(torch, app.k_new), to_dev_bf16(torch, app.v_new)
        cu, bt, sl = (to_dev(torch, app.cu_new), to_dev(torch, app.layout.block_table),
                      to_dev(torch, app.seq_lens))
        ap = lambda: pk.kv_append(pool, kn, vn, cu, bt, sl, k_smooth=w)
        ap()
        if name == "append_int8_32k":
            T = int(app.seq_lens.sum())
            # bf16 K and V read, int8 codes and fp32 scales written
            return ap, float(T * app.Hkv * (2 * 256 + 2 * (128 + 4))), "GB/s"
        case = W.DecodeCase(32, app.Hkv, app.seq_lens, app.layout, qh, None, None)
        return (_decode_fn(torch, pk, case, pool, app.k_smooth),
                decode_bytes(case.seq_lens, case.Hkv, 264), "GB/s")
    if name in ("prefill_1k", "append_bf16_1k"):   # the 1,024-token prompt, 32/8
        app, q = W.prefill_prompt()
        pool = pk.Pool.empty(app.layout.num_pages, app.Hkv)
        bt, sl, cu = (to_dev(torch, app.layout.block_table), to_dev(torch, app.seq_lens),
                      to_dev(torch, app.cu_new))
        kn, vn = to_dev_bf16(torch, app.k_new), to_dev_bf16(torch, app.v_new)
        ap = lambda: pk.kv_append(pool, kn, vn, cu, bt, sl)
        ap()
        if name == "append_bf16_1k":
            return ap, float(2 * 2 * 1024 * 8 * 256), "GB/s"
        qd = to_dev_bf16(torch, q)
        out = torch.empty_like(qd)
        lse = torch.empty((1024, 32), dtype=torch.float32, device="cuda")
        ws_p = pk.prefill_workspace()
        return (lambda: pk.paged_attn_prefill(pool, qd, cu, bt, sl, 1024, SCALE, workspace=ws_p,
                                              out=out, lse=lse),
                prefill_flops(1024, 1024, 32), "TFLOP/s")
    return None


PROFILE_CASES = ["prefill_chunk", "decode_bf16", "decode_int8", "qkv_prep", "verify_step",
                 "decode_1k", "decode_b64", "decode_int8_b1", "decode_int8_b8",
                 "append_int8_32k", "prefill_1k", "append_bf16_1k"]


def profile_case(torch, pk, name, reps=3):
    """One kernel on a fixed, seeded workload, launched `reps` times (for ncu
    captures of a single launch: -k <kernel> -s 2 -c 1).  Prints the median
    CUDA-event time of 10 more launches, each after an L2 flush."""
    rng = np.random.default_rng(5)
    cfg = profile_config_case(torch, pk, name)
    if cfg is not None:
        fn, work, unit = cfg
    elif name == "prefill_chunk":
        qlen, L = 2048, 16384
        case = W.decode_bf16(rng, [L], 32, 8)
        q = to_dev_bf16(torch, W.normal_bf16(rng, (qlen, 32, D)))
        pool = pk.Pool(to_dev_bf16(torch, case.k_pool), to_dev_bf16(torch, case.v_pool))
        cu, bt, sl = (to_dev(torch, W.cu_from_counts([qlen])), to_dev(torch, case.layout.block_table),
                      to_dev(torch, case.seq_lens))
        out = torch.empty_like(q)
        lse = torch.empty((qlen, 32), dtype=torch.float32, device="cuda")
        ws_p = pk.prefill_workspace()
        fn = lambda: pk.paged_attn_prefill(pool, q, cu, bt, sl, qlen, SCALE, workspace=ws_p,
                                           out=out, lse=lse)
        work = prefill_flops(qlen, L, 32)
        unit = "TFLOP/s"
    elif name in ("decode_bf16", "decode_int8"):
        if name == "decode_bf16":
            case = W.batched_decode(B=16)
            pool = pk.Pool(to_dev_bf16(torch, case.k_pool), to_dev_bf16(torch, case.v_pool))
            w, per = None, 512
        else:
            app, qh = W.int8_long_decode(B=2)
            pool = pk.Pool.empty(app.layout.num_pages, app.Hkv, dtype=torch.int8)
            w = to_dev(torch, app.k_smooth)
            pk.kv_append(pool, to_dev_bf16(torch, app.k_new), to_dev_bf16(torch, app.v_new),
                         to_dev(torch, app.cu_new), to_dev(torch, app.layout.block_table),
                         to_dev(torch, app.seq_lens), k_smooth=w)
            case = W.DecodeCase(32, app.Hkv, app.seq_lens, app.layout, qh, None, None)
            per = 264
        q = to_dev_bf16(torch, case.q)
        bt, sl = to_dev(torch, case.layout.block_table), to_dev(torch, case.seq_lens)
        ms = int(case.seq_lens.max())
        _, _, wsb, zb = pk.decode_plan(case.B, case.Hq, case.Hkv, ms, dtype=pool.dtype)
        ws = pk.decode_workspace(wsb, zb)
        out = torch.empty_like(q)
        lse = torch.empty((case.B, case.Hq), dtype=torch.float32, device="cuda")
        fn = lambda: pk.paged_attn_decode(pool, q, bt, sl, ms, SCALE, k_smooth=w, workspace=ws,
                                          out=out, lse=lse)
        work = decode_bytes(case.seq_lens, case.Hkv, per)
        unit = "GB/s"
    elif name == "qkv_prep":
        fn, work = qkv_prep_fn(torch, pk, 95)
        unit = "GB/s"
    elif name == "verify_step":
        # 8 sequences with 16-token steps at contexts 4k-8k, GQA 32/8
        lens = rng.integers(4096, 8193, 8)
        case = W.multi_token_decode(rng, lens, [16] * 8, 32, 8)
        pool = pk.Pool(to_dev_bf16(torch, case.k_pool), to_dev_bf16(torch, case.v_pool))
        q, cu = to_dev_bf16(torch, case.q), to_dev(torch, case.cu_q)
        bt, sl = to_dev(torch, case.layout.block_table), to_dev(torch, case.seq_lens)
        ms = int(lens.max())
        _, _, wsb = pk.decode_multi_plan(8, len(case.q), 32, 8, 16, ms)
        ws = torch.empty(max(wsb, 256), dtype=torch.uint8, device="cuda")
        out = torch.empty_like(q)
        lse = torch.empty((len(case.q), 32), dtype=torch.float32, device="cuda")
        fn = lambda: pk.paged_attn_decode_multi(pool, q, cu, bt, sl, 16, ms, SCALE, workspace=ws,
                                                out=out, lse=lse)
        work = decode_bytes(lens, 8)
        unit = "GB/s"
    else:
        raise SystemExit(f"unknown profile case {name}")
    for _ in range(reps):
        fn()
    torch.cuda.synchronize()
    # per-launch time with an L2 flush before each launch (back-to-back
    # launches of a short kernel would time the Python call, not the kernel)
    flush = L2Flush(torch)
    us, _ = time_events(torch, fn, iters=10, warm=0, flush=flush)
    rate = work / us / (1e6 if unit == "TFLOP/s" else 1e3)
    assert pk.poll_device_error() == pk.OK
    print(json.dumps({"profile_case": name, "us": round(us, 2), unit: round(rate, 1)}))


def make_line(K, Wu, world, r, e2e, peaks_, prof, config, nsteps=14):
    """The JSON line of the mixed-step run from the timings r (time_mixed),
    the end-to-end result e2e = (us, h2d bytes, d2h bytes, steps), the peaks
    (peaks()) and the prefill profile figures (prefill_profile())."""
    hbm, bf16, bf16_sus, peak_src, peak_mhz = peaks_
    e2e_us, h2d, d2h, K_e2e = e2e[:4]
    host_us = e2e[4] if len(e2e) > 4 else None
    us_per_step = r["step_ms"] * 1e3
    pre_tflops = r["flops"] / (r["pre_ms"] * 1e-3) / 1e12
    dec_gbs = r["dbytes"] / (r["dec_ms"] * 1e-3) / 1e9
    # the timed region is short (well under a second at the default steps),
    # so the kernel runs at burst clocks: the burst peak is the denominator
    region_s = r["total_ms"] * 1e-3
    peak, peak_kind = (bf16, "burst") if region_s < 1.0 else (bf16_sus, "sustained")
    frac = pre_tflops / peak
    n_pre = K                                        # one prefill launch per step
    traffic = prof.get("dram_bytes_per_launch_mixed_step")
    sm_mhz = r["clocks"].get("sm_mhz")
    roofline = {
        "kernel": "prefill_kernel (tcgen05)", "bound": "tensor",
        "achieved": round(pre_tflops, 1), "peak": peak, "unit": "TFLOP/s",
        "frac": round(frac, 4), "traffic": traffic,
        "peak_source": (f"{peak_src} bf16 {peak_kind} (MEASURED_PEAKS.json; timed region "
                        f"{region_s:.3f} s)"),
        "achieved_note": (f"causal flops 4*D*Hq*keys over the {n_pre} prefill launches / their "
                          "summed CUDA-event durations in the timed region"),
        "traffic_note": ("mean dram read+write bytes per prefill launch of the mixed step's 14 "
                         "chunks, from the committed ncu summary of this kernel's sources"
                         if traffic is not None else
                         "null: no ncu capture of the current prefill sources"),
        "frac_of_spec_dense_bf16": round(pre_tflops / SPEC_BF16_TFLOPS, 4),
        "spec_peak_note": ("2,250 TFLOP/s dense bf16 per GPU: NVIDIA HGX B300 36 PFLOP/s "
                           "FP16/BF16 per 8 GPUs with 2:4 sparsity, halved"),
    }
    if peak_mhz and sm_mhz:
        roofline["frac_clock_normalized"] = round(pre_tflops / (peak * sm_mhz / peak_mhz), 4)
        roofline["clock_note"] = (f"peak scaled by bench SM clock {sm_mhz:.0f} MHz / "
                                  f"{peak_mhz:.0f} MHz median under load when the peaks were "
                                  "measured")
    share = r.get("sm_share", 1.0)
    alone = r.get("alone")
    if alone:
        a_tf = alone["flops"] / (alone["pre_ms"] * 1e-3) / 1e12
        roofline["achieved_alone"] = round(a_tf, 1)
        roofline["frac_alone"] = round(a_tf / peak, 4)
        roofline["alone_note"] = ("the same steps run one after the other right after the timed "
                                  f"region ({alone['steps']} steps): the prefill alone on every SM")
    if r.get("overlap"):
        # the prefill held part of the SMs (the decode ran beside it on the
        # others): its attainable peak is that share of the GPU's
        roofline["sm_share"] = round(share, 4)
        roofline["frac_of_sm_share"] = round(frac / share, 4)
        roofline["sm_share_note"] = ("prefill launches ran on part of the SMs (time-weighted "
                                     "mean CTAs / all) beside the decode on a second stream; "
                                     "frac_of_sm_share = achieved / (peak x sm_share)")
    if "tensor_pipe_active_pct_2048x16384" in prof:
        roofline["ncu_tensor_pipe_active_pct"] = prof["tensor_pipe_active_pct_2048x16384"]
        roofline["ncu_note"] = ("sm__pipe_tensor_cycles_active of one 2,048-row x 16,384-"
                                "position launch (same sources)")

    line = {
        "metric": METRIC, "value": round(us_per_step, 2), "unit": "us", "n_gpus": world,
        "steps": K, "warmup": Wu, "ms_per_step": round(us_per_step / 1e3, 4),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded; shapes of the pages' workloads)", "config": config,
        "value_note": ("us per step, the 14 prompt chunks weighted equally (mean over chunks of "
                       "each chunk's mean step time)" if r["balanced"] else
                       "us per step, plain mean (fewer than 14 steps timed)"),
        "plain_mean_us": round(r["total_ms"] * 1e3 / K, 2),
        "schedule": ("overlapped: append, then the prefill on part of the SMs "
                     "(pkv_overlap_prefill_ctas) beside the decode on a second stream"
                     if r.get("overlap") else "sequential: append, prefill, decode on one stream"),
        "decode": {"us_per_step": round(r["dec_ms"] * 1e3 / K, 2), "GBps": round(dec_gbs, 1),
                   "frac_of_8TBps": round(dec_gbs / NOMINAL_HBM_GBS, 4),
                   "frac_of_measured": round(dec_gbs / hbm, 4),
                   "bytes_per_step": round(r["dbytes"] / K)},
        "prefill": {"us_per_step": round(r["pre_ms"] * 1e3 / K, 2),
                    "TFLOPs": round(pre_tflops, 1),
                    "frac_of_measured_burst": round(pre_tflops / bf16, 4),
                    "frac_of_measured_sustained": round(pre_tflops / bf16_sus, 4),
                    "frac_of_spec_dense": round(pre_tflops / SPEC_BF16_TFLOPS, 4),
                    "flops_per_step": round(r["flops"] / K)},
        "append": {"us_per_step": round(r["app_ms"] * 1e3 / K, 2)},
        # the 14 steps of one pass over the prompt (each the mean over the
        # timed steps that ran that chunk), and their sum
        "chunk_steps": r["chunks"],
        "prompt_pass": {"step_us": round(sum(c["step_us"] for c in r["chunks"]), 1),
                        "prefill_us": round(sum(c["prefill_us"] for c in r["chunks"]), 1),
                        "decode_us": round(sum(c["decode_us"] for c in r["chunks"]), 1),
                        "append_us": round(sum(c["append_us"] for c in r["chunks"]), 1),
                        "chunks": len(r["chunks"])},
        "roofline": roofline,
        "e2e": {"value": round(e2e_us, 2), "unit": "us", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h), "steps": K_e2e,
                "note": (f"steps {Wu}..{Wu + K_e2e - 1} (whole passes over the 14 chunks) through "
                         "the public API, inputs from pinned host memory each step, outputs read "
                         "back each step; wall clock"),
                "host_enqueue_us_per_step": round(host_us, 2) if host_us is not None else None},
        "gpu_launches": r["launches"],
        "clocks": r["clocks"],
    }
    if alone:
        a_dec = alone["dbytes"] / (alone["dec_ms"] * 1e-3) / 1e9
        a_pre = alone["flops"] / (alone["pre_ms"] * 1e-3) / 1e12
        n_a = alone["steps"]
        line["sequential"] = {
            "note": ("the same steps one after the other on one stream (each kernel alone on "
                     "the GPU), timed right after the overlapped region"),
            "steps": n_a, "value": round(alone["step_ms"] * 1e3, 2),
            "decode": {"us_per_step": round(alone["dec_ms"] * 1e3 / n_a, 2),
                       "GBps": round(a_dec, 1), "frac_of_measured": round(a_dec / hbm, 4),
                       "frac_of_8TBps": round(a_dec / NOMINAL_HBM_GBS, 4)},
            "prefill": {"us_per_step": round(alone["pre_ms"] * 1e3 / n_a, 2),
                        "TFLOPs": round(a_pre, 1),
                        "frac_of_measured_burst": round(a_pre / bf16, 4),
                        "frac_of_spec_dense": round(a_pre / SPEC_BF16_TFLOPS, 4)},
            "append": {"us_per_step": round(alone["app_ms"] * 1e3 / n_a, 2)}}
        line["decode"]["note"] = ("overlapped with the prefill: time from the decode's start to "
                                  "its end while the prefill holds most SMs (alone: see "
                                  "'sequential')")
        line["prefill"]["note"] = ("overlapped with the decode, on part of the SMs (see "
                                   "roofline.sm_share; alone: see 'sequential')")
    return line


# ---------------------------------------------------------------- main

def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1400)
    ap.add_argument("--warmup", type=int, default=28)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-configs", action="store_true", help="skip the other workloads")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sequential", action="store_true",
                    help="mixed step on one stream (no prefill/decode overlap)")
    ap.add_argument("--profile-case", choices=PROFILE_CASES,
                    help="run one kernel on a fixed workload (for ncu) and exit")
    args = ap.parse_args(argv)
    K, Wu = args.steps, max(3, args.warmup)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    config = {"workload": ("mixed continuous-batching step: one 26,926-token causal prompt "
                           "prefilled in 2,048-row chunks against its cached prefix + 32 decode "
                           "rows (contexts U[128,16384]); per step the append, then the prefill "
                           "and the decode (both after the append; overlapped on two streams "
                           "unless --sequential)"),
              "heads_q": 32, "heads_kv": 8, "head_dim": 128, "page_size": 16,
              "prompt_len": 26926, "chunk": 2048, "decode_rows": 32,
              "l2": "working set 1.2 GB > 129 MB L2 (no flush between steps)",
              "parallelism": f"replicas x{args.gpus}"}

    if args.impl == "reference":
        if rank != 0:
            return 0
        wl = W.mixed_step()
        fill_prompt_for_oracle(wl)
        nthreads = os.cpu_count() or 1
        rng = np.random.default_rng(98)
        nsteps = len(wl.steps)
        for i in range(Wu):
            if i >= 1:
                break                         # one untimed sample warms the oracle
            oracle_step_sample(wl, i % nsteps, 4, 2, rng, nthreads)
        ests, spent = [], 0.0
        for i in range(K):
            c = (Wu + i) % nsteps
            e, dt = oracle_step_sample(wl, c, 4, 2, rng, nthreads)
            ests.append((c, e))
            spent += dt
            if spent > 150.0:
                break
        per = {}
        for c, e in ests:
            per.setdefault(c, []).append(e)
        # the 14 chunks weighted equally when every chunk was sampled, as in
        # the GPU arm's value; otherwise the plain mean
        v = (float(np.mean([np.mean(x) for x in per.values()])) if len(per) == nsteps
             else float(np.mean([e for _, e in ests]))) * 1e6
        line = {"impl": "reference", "metric": METRIC, "value": round(v, 1), "unit": "us",
                "n_gpus": args.gpus, "steps": len(ests), "warmup": Wu,
                "ms_per_step": round(v / 1e3, 3), "higher_is_better": False, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": config,
                "cpu_baseline": {"value": round(v, 1), "unit": "us", "cores": nthreads,
                                 "kind": "oracle",
                                 "sample": (f"fp64 oracle, 4 prefill rows + 2 decode rows (32 "
                                            f"heads) per step, {len(ests)} steps, "
                                            f"{spent:.1f} s; scaled by (row, head, key) "
                                            f"triples to the full step")},
                "e2e": {"value": round(v, 1), "unit": "us", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0},
                "sampled_cpu_seconds": round(spent, 2),
                "value_note": ("per-step time of the whole step extrapolated from the sampled "
                               "rows; the run itself spent sampled_cpu_seconds")}
        print(json.dumps(line), flush=True)
        return 0

    import torch
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    from paged_kv_flash_gb300 import pagedkv as pk

    if args.profile_case:
        profile_case(torch, pk, args.profile_case)
        return 0
    hbm, bf16, bf16_sus, peak_src, peak_mhz = peaks()
    mixed = Mixed(torch, pk, overlap=not args.sequential)
    r = time_mixed(torch, pk, mixed, K, Wu, world, rank)
    nsteps = len(mixed.steps)
    if mixed.overlap:
        # the same steps one after the other, briefly: each kernel alone on
        # the whole GPU, for the per-kernel figures beside the overlapped step
        mixed.overlap = False
        r["alone"] = time_mixed(torch, pk, mixed, 20 * nsteps, nsteps, world, rank)
        mixed.overlap = True
    K_e2e = -(-K // nsteps) * nsteps               # whole passes over the 14 chunks
    e2e_us, h2d, d2h, host_us = time_e2e(torch, pk, mixed, K_e2e, Wu)

    e2e = (e2e_us, h2d, d2h, K_e2e, host_us)
    line = make_line(K, Wu, world, r, e2e, (hbm, bf16, bf16_sus, peak_src, peak_mhz),
                     prefill_profile(), config, nsteps)
    if rank == 0 and world == 1 and not args.no_configs:
        line["configs"] = other_configs(torch, pk, hbm, bf16)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        wl = mixed.wl
        fill_prompt_for_oracle(wl)
        line["cpu_baseline"] = cpu_baseline(wl)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())

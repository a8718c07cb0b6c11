"""Benchmark of the quantized-KV hot path on one GB300 (or N, one process per GPU).

One run measures every workload shape of the pages (synthetic, seeded):

  * mistral7b_hotcold (the headline line): Mistral-7B shape, 32 layers, 32
    query / 8 kv heads, D = 128, batch 64, T = 32768; keys stored pre-RoPE
    (split-half RoPE applied in the decode kernel), the newest 128 tokens in a
    16-bit window, the 4096 before them 4-bit (KIVI: K per channel over
    32-token groups, V per token over 32-channel groups), older tokens 2-bit;
    a 48 GB cache.
  * q8_0_mha_1k, q4_0_mha_1k: one layer, 4 heads, D = 128, T = 1024 (fits in
    L2: launch-bound, a parity shape, not a bandwidth figure).
  * llama2_7b_kivi4: Llama-2-7B shape, 32 layers x 32 heads, T = 32768, KIVI
    4-bit with a 128-token window.
  * gqa8b_hadamard4_paged: 32 layers, 32 / 8 heads, batch 16 of ragged
    2K-8K tokens in 16-token pages, Hadamard-128 + 4-bit 66 B/128 blocks.
  * ctx262k_hadamard4 / ctx262k_hadamard3: 16 layers, 24 / 4 heads, D = 256,
    T = 262144, Hadamard-128 + 66 B/128 or 50 B/128 blocks.

One step of a workload is one decode step of the whole hot path for every
layer: quantize-on-append of the new token of every sequence and decode
attention over the grown cache (kvq_decode_step: one fused launch where the
formats allow), then the length commit.  value = (cache bytes the step reads
+ the new tokens' source bytes) / step time, in GB/s.  Every cache except the
1K-token ones is larger than L2, so no flush is needed between steps.

Also reported per workload: bulk append GB/s (one layer per call, L2 flushed
before each call), the decode launch's roofline fraction, the same decode
issued as one call per layer (how a model calls it), an end-to-end number
through the C ABI with host buffers, and the score distortion max |ds| of the
quantized keys on a sampled sequence.  The headline line adds the CPU oracle
timed on a bounded sample, on all host cores and on one.

`--impl reference` times the CPU oracle (the reference arm of this build) on
the headline workload, a bounded sample per step on all host cores.
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
sys.path.insert(0, ROOT)

METRIC = "quantized-KV decode attention: effective HBM GB/s and % of peak; append GB/s"
HEADLINE = "mistral7b_hotcold"
# every workload shape of the pages, the headline first
WORKLOADS = (HEADLINE, "q8_0_mha_1k", "q4_0_mha_1k", "llama2_7b_kivi4", "gqa8b_hadamard4_paged",
             "ctx262k_hadamard4", "ctx262k_hadamard3")
SIDE_STEPS = 10  # timed steps of the non-headline workloads


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.file, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self.proc is not None

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.file.name)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


class NvmlClockSampler:
    """SM clock and clock-event (throttle) reasons read through NVML every
    `period` seconds on a background thread (read-only queries)."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown",
               0x80: "hw_power_brake_slowdown"}

    def __init__(self, cuda_index: int, period: float = 0.002):
        import ctypes
        import threading

        self.ok = False
        self.samples = []
        self.period = period
        self._stop = threading.Event()
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                return
            count = ctypes.c_uint()
            lib.nvmlDeviceGetCount_v2(ctypes.byref(count))
            handle = ctypes.c_void_p()
            idx = 0 if count.value == 1 else cuda_index
            if lib.nvmlDeviceGetHandleByIndex_v2(idx, ctypes.byref(handle)) != 0:
                return
            mx = ctypes.c_uint()
            lib.nvmlDeviceGetMaxClockInfo(handle, 1, ctypes.byref(mx))
            self.max_mhz = mx.value
            self.lib, self.handle, self.ctypes = lib, handle, ctypes
            fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
            self.reasons_fn = fn
            self.ok = True
        except Exception:
            self.ok = False
        if self.ok:
            self.thread = threading.Thread(target=self._run, daemon=True)

    def _run(self):
        c = self.ctypes
        clk, rs = c.c_uint(), c.c_ulonglong()
        while not self._stop.is_set():
            if self.lib.nvmlDeviceGetClockInfo(self.handle, 1, c.byref(clk)) == 0 and \
                    self.reasons_fn(self.handle, c.byref(rs)) == 0:
                self.samples.append((clk.value, rs.value))
            time.sleep(self.period)

    def start(self):
        if self.ok:
            self.thread.start()
        return self.ok

    def stop(self):
        if not self.ok:
            return None
        self._stop.set()
        self.thread.join()
        if not self.samples:
            return None
        reasons = sorted({name for _, r in self.samples for bit, name in self.REASONS.items() if r & bit})
        return {"sm_mhz": statistics.median([c for c, _ in self.samples]), "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(self.samples), "source": "nvml, 2 ms period"}


def _clock_sampler(local):
    s = NvmlClockSampler(local)
    if s.start():
        return s
    s = ClockSampler(local)
    s.start()
    return s


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def aggregate(values_bytes, times_s):
    """Whole-job throughput: bytes of all ranks / the slowest rank's time."""
    return sum(values_bytes) / max(times_s)


def _job_seconds(local_s: float, device) -> float:
    """The slowest rank's timed seconds, returned on every rank (the local
    time when there is one rank)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return local_s
    t = torch.tensor([local_s], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _job_gbs(bytes_per_rank: float, world: int, seconds: float) -> float:
    """Whole-job GB/s: every rank processes its own sequences (weak scaling),
    so the job moves world x the bytes of one rank in the slowest rank's time."""
    return bytes_per_rank * world / seconds / 1e9


def _barrier(ws):
    if ws > 1:
        import torch.distributed as dist

        dist.barrier()


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------


def score_distortion(w, cache, seq_lens, dev, seed):
    """Score distortion of the quantized keys (nalar.dev, "Error pada key
    mengubah input softmax": a key error moves the softmax input by
    q.e_i / sqrt(D), so keys are judged by that, not by their MSE): on layer
    0, sequence 0, every query head, ds_t = q.(k_hat_t - k_t) / sqrt(D) over
    the packed tokens [0, q_end), keys turned by RoPE at t where they are
    stored pre-RoPE.  k_hat comes from kvq_dequantize; k is the source the
    cache was filled from.  A quality diagnostic, computed in fp64 with torch
    after the timed regions."""
    import torch

    from bit_kv_cache_04_gb300 import kvq as K
    from bit_kv_cache_04_gb300 import workloads as W

    cfg = w.cfg
    T = w.lengths[0]
    gam = 32 if K.AXIS_CHANNEL in (cfg.k_fmt.axis, cfg.v_fmt.axis) else 1
    qe = 0 if T <= cfg.residual_window else (T - cfg.residual_window) // gam * gam
    if qe == 0:
        return None
    kh = torch.empty((T, cfg.H_kv, cfg.D), dtype=torch.float32, device=dev)
    vh = torch.empty_like(kh)
    lens0 = torch.full_like(seq_lens, T)
    cache.dequantize(0, 0, 0, T, lens0, kh, vh)
    k, _ = W.kv_tokens(w, 0, 0, 0, T, dev, seed)
    e = (kh[:qe].double() - k[:qe].double())  # [qe, H_kv, D]
    if cfg.flags & K.K_PRE_ROPE:
        h = cfg.D // 2
        inv = cfg.rope_theta ** (-2.0 * torch.arange(h, dtype=torch.float64, device=dev) / cfg.D)
        ang = torch.arange(qe, dtype=torch.float64, device=dev)[:, None] * inv[None, :]
        c, s = torch.cos(ang)[:, None, :], torch.sin(ang)[:, None, :]
        a, b = e[..., :h], e[..., h:]
        e = torch.cat([a * c - b * s, a * s + b * c], dim=-1)
    q = W.queries(w, 1, dev, seed=seed + 99)[0, 0].double()  # [H_q, D]
    g = cfg.H_q // cfg.H_kv
    ds = torch.einsum("thd,hgd->thg", e, q.view(cfg.H_kv, g, cfg.D)) / math.sqrt(cfg.D)
    torch.cuda.synchronize()
    return {"max_abs": float(ds.abs().max()), "rms": float(ds.pow(2).mean().sqrt()),
            "tokens": qe, "heads": cfg.H_q,
            "what": "layer 0, sequence 0: max |q.(k_hat - k)| / sqrt(D) over the packed tokens, every query head"}


def measure(wname, steps, warm, dev, rank, ws, headline=False, ablation=False, layers=0, batch=0):
    """Fills a workload's cache and times its decode steps.  Returns a dict
    of figures (the headline also keeps the raw pieces of the JSON line)."""
    import torch

    from bit_kv_cache_04_gb300 import kvq as K
    from bit_kv_cache_04_gb300 import workloads as W

    extra = 3 * (steps + warm) + 16  # fused steps, unfused steps, end-to-end steps
    w = W.make(wname, extra_tokens=extra)
    if layers or batch:
        w = w.scaled(L=layers or None, lengths=w.lengths[: batch or len(w.lengths)], extra=extra)
    cfg = w.cfg
    L, B, H, Hq, D = cfg.L, cfg.batch, cfg.H_kv, cfg.H_q, cfg.D
    stream = torch.cuda.current_stream(dev)
    cache = K.KVCache(cfg, dev, block_table=W.page_table(w, rank))
    seq_lens = torch.zeros(B, dtype=torch.int32, device=dev)
    dt = torch.float16 if cfg.in_dtype == K.DT_F16 else torch.bfloat16
    peak, peak_kind = _peaks()

    # ---- bulk append, one layer per call (timed per call) ----------------
    # Calls are enqueued back to back (no host synchronization between them)
    # so that each call's events bracket GPU work, not host latency.
    app_ev, app_bytes = [], []
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)  # 256 MB > L2
    for l in range(L):
        ks, vs, cu = W.layer_batch(w, l, [0] * B, w.lengths, dev, seed=rank)
        cu_d = torch.tensor(cu, dtype=torch.int32, device=dev)
        if l == 0:
            # untimed first call (kernel loading); lengths are committed only
            # after all layers, so repeating a layer's append rewrites the
            # same rows with the same bytes
            cache.append(l, 1, ks[None], vs[None], cu_d, seq_lens, cu[-1], max(w.lengths))
            torch.cuda.synchronize()
        flush.zero_()  # evict the freshly generated inputs from L2
        e0, e1 = torch.cuda.Event(True), torch.cuda.Event(True)
        e0.record(stream)
        cache.append(l, 1, ks[None], vs[None], cu_d, seq_lens, cu[-1], max(w.lengths))
        e1.record(stream)
        app_ev.append((e0, e1))
        src = ks.numel() * 2 * 2
        packed = sum(K.kvq_cache_bytes(cfg, t) for t in w.lengths) // L
        app_bytes.append(src + packed)
        del ks, vs
    torch.cuda.synchronize()
    app_ms = [e0.elapsed_time(e1) for e0, e1 in app_ev]
    del flush
    cu_all = torch.tensor([0] + w.lengths, dtype=torch.int32, device=dev).cumsum(0, dtype=torch.int32)
    cache.commit_lengths(cu_all, seq_lens)
    torch.cuda.synchronize()
    distortion = score_distortion(w, cache, seq_lens, dev, rank) if rank == 0 else None
    lengths = list(w.lengths)
    cache_gb = sum(K.kvq_cache_bytes(cfg, t) for t in lengths) / 1e9

    # ---- decode steps ----------------------------------------------------
    n_steps = warm + steps
    g = torch.Generator(device=dev).manual_seed(1234 + rank)
    new_k = torch.randn((n_steps, L, B, H, D), generator=g, device=dev).to(dt)
    new_v = torch.randn((n_steps, L, B, H, D), generator=g, device=dev).to(dt)
    qs = torch.randn((n_steps, L, B, Hq, D), generator=g, device=dev).to(dt)
    out = torch.empty((L, B, Hq, D), dtype=torch.float32, device=dev)
    cu1 = torch.arange(0, B + 1, dtype=torch.int32, device=dev)

    dec0 = [torch.cuda.Event(True) for _ in range(n_steps)]
    dec1 = [torch.cuda.Event(True) for _ in range(n_steps)]

    def step(i):
        # one decode step: the new token of every (layer, sequence) appended and
        # attention over the grown cache (one fused launch where the formats
        # allow), then the length commit
        dec0[i].record(stream)
        cache.decode_step(0, L, new_k[i], new_v[i], qs[i], seq_lens, out, 0, stream)
        dec1[i].record(stream)
        cache.commit_lengths(cu1, seq_lens, stream)

    step_bytes = []
    for i in range(n_steps):
        # step i reads the cache grown by its token: lengths + 1, plus the
        # token's source bytes
        lengths = [t + 1 for t in lengths]
        step_bytes.append(sum(K.kvq_cache_bytes(cfg, t) for t in lengths) + L * B * H * D * 2 * 2)
    for i in range(warm):
        step(i)
    torch.cuda.synchronize()
    _barrier(ws)
    clocks = _clock_sampler(dev.index or 0) if headline else None
    t0, t1 = torch.cuda.Event(True), torch.cuda.Event(True)
    t0.record(stream)
    for i in range(warm, n_steps):
        step(i)
    t1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop() if clocks else None
    elapsed = _job_seconds(t0.elapsed_time(t1) / 1e3, dev)
    value = _job_gbs(sum(step_bytes[warm:]), ws, elapsed)
    dec_ms = [dec0[i].elapsed_time(dec1[i]) for i in range(warm, n_steps)]
    achieved = sum(step_bytes[warm:]) / (sum(dec_ms) / 1e3) / 1e9
    status = cache.device_status()
    step_launches = K.kvq_step_launches(cfg)

    # ---- the same steps unfused: kvq_append, decode attention, commit -----
    def step_unfused(i):
        cache.append(0, L, new_k[i], new_v[i], cu1, seq_lens, B, 1, stream)
        cache.decode(0, L, qs[i], seq_lens, out, 0, stream)
        cache.commit_lengths(cu1, seq_lens, stream)

    for i in range(warm):
        step_unfused(i)
        lengths = [t + 1 for t in lengths]
    torch.cuda.synchronize()
    u0, u1 = torch.cuda.Event(True), torch.cuda.Event(True)
    u0.record(stream)
    for i in range(warm, n_steps):
        step_unfused(i)
        lengths = [t + 1 for t in lengths]
    u1.record(stream)
    torch.cuda.synchronize()
    unfused_ms = u0.elapsed_time(u1) / steps

    # ---- end to end through the C ABI with host buffers -------------------
    hk = new_k.cpu().pin_memory()
    hv = new_v.cpu().pin_memory()
    hq = qs.cpu().pin_memory()
    hout = torch.empty(out.shape, dtype=torch.float32).pin_memory()
    dk = torch.empty_like(new_k[0])
    dv = torch.empty_like(new_v[0])
    dq = torch.empty_like(qs[0])
    e2e_bytes = 0

    def e2e_step(i):
        dk.copy_(hk[i], non_blocking=True)
        dv.copy_(hv[i], non_blocking=True)
        dq.copy_(hq[i], non_blocking=True)
        cache.decode_step(0, L, dk, dv, dq, seq_lens, out, 0, stream)
        cache.commit_lengths(cu1, seq_lens, stream)
        hout.copy_(out, non_blocking=True)

    for i in range(min(warm, 3)):
        e2e_step(i)
        lengths = [t + 1 for t in lengths]
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(True), torch.cuda.Event(True)
    e0.record(stream)
    for i in range(warm, n_steps):
        lengths = [t + 1 for t in lengths]
        e2e_bytes += sum(K.kvq_cache_bytes(cfg, t) for t in lengths) + L * B * H * D * 4
        e2e_step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_s = _job_seconds(e0.elapsed_time(e1) / 1e3, dev)
    h2d = (dk.numel() + dv.numel() + dq.numel()) * 2
    d2h = hout.numel() * 4

    # ---- the same decode as L single-layer calls (how a model calls it) ----
    per_layer = None
    if L > 1:
        reps = 3
        for rnd in range(2):  # the second round timed
            p0, p1 = torch.cuda.Event(True), torch.cuda.Event(True)
            p0.record(stream)
            for r in range(reps):
                for l in range(L):
                    cache.decode(l, 1, qs[r % n_steps][l:l + 1], seq_lens, out[l:l + 1], 0, stream)
            p1.record(stream)
            torch.cuda.synchronize()
        pl_ms = p0.elapsed_time(p1) / reps
        pl_bytes = sum(K.kvq_cache_bytes(cfg, t) for t in lengths)
        pl_gbs = pl_bytes / (pl_ms / 1e3) / 1e9
        per_layer = {"ms": round(pl_ms, 4), "GBps": round(pl_gbs, 2), "pct_of_peak": round(100 * pl_gbs / peak, 2),
                     "splits": K.kvq_decode_splits(cfg, 1)}

    append_gbs = sum(app_bytes) / (sum(app_ms) / 1e3) / 1e9
    res = {
        "workload": wname,
        "value": value, "elapsed": elapsed, "steps": steps, "step_bytes": sum(step_bytes[warm:]),
        "decode": {"GBps": round(achieved, 2), "pct_of_peak": round(100 * achieved / peak, 2),
                   "ms_per_launch": round(statistics.mean(dec_ms), 4),
                   "tokens_per_s": round(B / statistics.mean(dec_ms) * 1e3, 2),
                   "launches": step_launches, "splits": K.kvq_decode_splits(cfg, L)},
        "per_layer_decode": per_layer,
        "step": {"fused_ms": round(statistics.mean(dec_ms), 4), "unfused_ms": round(unfused_ms, 4),
                 "unfused": "kvq_append + kvq_decode_attention + commit per step", "launches": step_launches},
        "append": {"GBps": round(append_gbs, 2), "pct_of_peak": round(100 * append_gbs / peak, 2),
                   "ms_per_layer": round(statistics.median(app_ms), 4)},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": _traffic(wname, L),
                     "kernel": ("fused decode step: append + decode attention, one multi-layer launch"
                                if step_launches == 1 else "decode step: append and decode launches"),
                     "peak_source": peak_kind},
        "e2e": {"value": round(_job_gbs(e2e_bytes, ws, e2e_s), 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "score_distortion": distortion,
        "device_status": status,
        "gpu_launches": steps * (step_launches + 1),  # decode step + length commit
        "clocks": clk,
        "cache_gb": round(cache_gb, 3),
        "l2": ("inputs larger than L2 (cache %.2f GB)" % cache_gb) if cache_gb > 0.26
        else "cache %.4f GB fits in L2: launch-bound parity shape, not a bandwidth figure" % cache_gb,
        "cfg": cfg, "lengths": w.lengths,
    }
    if ablation:
        res["ablation_unfused"] = unfused_ablation(cache, cfg, w, seq_lens, stream)
    del cache, new_k, new_v, qs, out, hk, hv, hq, hout, dk, dv, dq
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return res


def _per_config_row(r):
    """The per-workload summary that goes into the JSON line."""
    return {"step_GBps": round(r["value"], 2), "ms_per_step": round(r["elapsed"] / r["steps"] * 1e3, 4),
            "decode_GBps": r["decode"]["GBps"], "decode_pct": r["decode"]["pct_of_peak"],
            "tokens_per_s": r["decode"]["tokens_per_s"], "roofline_frac": r["roofline"]["frac"],
            "per_layer_GBps": None if r["per_layer_decode"] is None else r["per_layer_decode"]["GBps"],
            "per_layer_pct": None if r["per_layer_decode"] is None else r["per_layer_decode"]["pct_of_peak"],
            "append_GBps": r["append"]["GBps"], "append_pct": r["append"]["pct_of_peak"],
            "e2e_GBps": r["e2e"]["value"], "launches_per_step": r["decode"]["launches"],
            "score_max_abs_ds": None if r["score_distortion"] is None
            else round(r["score_distortion"]["max_abs"], 6),
            "cache_GB": r["cache_gb"], "device_status": r["device_status"], "timed_steps": r["steps"]}


def run_ours(args):
    import torch

    from bit_kv_cache_04_gb300 import kvq as K

    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    head = args.workload or HEADLINE
    side = [] if (args.workload or args.only_headline) else [x for x in WORKLOADS if x != head]
    main = measure(head, args.steps, args.warmup, dev, rank, ws, headline=True, ablation=args.ablation,
                   layers=args.layers, batch=args.batch)
    rows = {head: _per_config_row(main)}
    for wname in side:
        r = measure(wname, min(args.steps, SIDE_STEPS), 3, dev, rank, ws)
        rows[wname] = _per_config_row(r)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(head, args.cpu_heads)

    cfg = main["cfg"]
    fmt_text, bits_text = _format_text(cfg)
    in_text = "f16" if cfg.in_dtype == K.DT_F16 else "bf16"
    B = cfg.batch
    result = {
        "metric": METRIC,
        "value": round(main["value"], 2),
        "unit": "GB/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(main["elapsed"] / args.steps * 1e3, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": f"{in_text} in, packed {bits_text} codes + fp16 scales, fp32 math",
        "data": "synthetic (seeded)",
        "config": {"workload": head, "layers": cfg.L, "heads_q": cfg.H_q, "heads_kv": cfg.H_kv,
                   "head_dim": cfg.D, "batch": B,
                   "context_tokens": main["lengths"][0] if len(set(main["lengths"])) == 1 else main["lengths"],
                   "format": fmt_text,
                   "step": "kvq_decode_step over all layers (1 new token per sequence appended, attention over the "
                           "grown cache) + length commit",
                   "decode_launch": "one fused multi-layer launch" if main["decode"]["launches"] == 1
                   else f"{main['decode']['launches']} launches (append, then decode)",
                   "l2": main["l2"],
                   "parallelism": f"replicas x{ws}"},
        "step": main["step"],
        "decode": main["decode"],
        "per_layer_decode": main["per_layer_decode"],
        "append": dict(main["append"], what=f"bulk quantize-on-append of one layer ({sum(main['lengths'])} tokens "
                                            f"x {cfg.H_kv} kv heads) per call; bytes = {in_text} source read + "
                                            f"packed blocks and window written"),
        "roofline": main["roofline"],
        "e2e": main["e2e"],
        "score_distortion": main["score_distortion"],
        "gpu_launches": main["gpu_launches"],
        "clocks": main["clocks"],
        "device_status": main["device_status"],
        "per_config": rows,
    }
    if cpu:
        result["cpu_baseline"] = cpu
    if "ablation_unfused" in main:
        result["ablation_unfused"] = main["ablation_unfused"]
    if rank == 0:
        print(json.dumps(result))
    if ws > 1:
        torch.distributed.destroy_process_group()


# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one decode-step
# launch per layer it covers, from an ncu capture of the multi-layer launch,
# with the SHA-256 of the kernel sources it was taken on; the roofline reports
# them scaled to the timed launch while those sources are unchanged, else null.
DECODE_TRAFFIC = {
    "llama2_7b_kivi4": {"sha256": "83ae845cef27e59b91f0de995e58fe7892e40b85583ec76d462aa6229551f076",
                        "bytes_per_layer": (610.612736e6 + 8.897536e6) / 4},
    # a 2-layer step (64 sequences x 32768 tokens) captured whole, halved
    "mistral7b_hotcold": {"sha256": "f2ef69394305ff6186fda78b363a1bd0bdd77670f6bf220ab59c59cba18c2fd9",
                          "bytes_per_layer": (3022.001664e6 + 17.611264e6) / 2},
}
# the sources each workload's decode-step kernel is built from
_COMMON_SOURCES = ("decode_mma.cuh", "append_generic.cuh", "append_common.cuh", "block_codec.cuh")
_TRAFFIC_SOURCES = {
    "llama2_7b_kivi4": _COMMON_SOURCES[:1] + ("decode_step_kivi.cu",) + _COMMON_SOURCES[1:],
    "mistral7b_hotcold": _COMMON_SOURCES + ("decode_step_d128.cu", "split_combine.cuh", "kvq_internal.cuh"),
}


def _kernel_sha(workload: str) -> str:
    import hashlib

    h = hashlib.sha256()
    for f in _TRAFFIC_SOURCES.get(workload, ()):
        with open(os.path.join(ROOT, "bit_kv_cache_04_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def _traffic(workload: str, layers: int):
    rec = DECODE_TRAFFIC.get(workload)
    if rec is None or rec["sha256"] != _kernel_sha(workload):
        return None
    return round(rec["bytes_per_layer"] * layers)


def _format_text(cfg):
    """Human-readable cache format of a config and the code widths it holds."""
    from bit_kv_cache_04_gb300 import kvq as K

    def one(f, zp, tb):
        if f is None or f.bits == 0:
            return None
        axis = "per-channel (32 tokens)" if f.axis == K.AXIS_CHANNEL else f"per-token ({f.group} values)"
        bb = K.kvq_block_bytes(f.bits, f.group) + (2 if zp else 0)
        kind = "TBQ4 norm + Lloyd-Max indices" if tb else ("scale + zero" if zp else "scale")
        return f"{f.bits}-bit {axis}, {bb} B/{f.group if f.axis == K.AXIS_TOKEN else 32} ({kind})"
    fl = cfg.flags
    parts = [f"K {one(cfg.k_fmt, fl & K.ZP_K, fl & K.TBQ4_K)}", f"V {one(cfg.v_fmt, fl & K.ZP_V, fl & K.TBQ4_V)}"]
    if cfg.hot_window:
        parts.append(f"hot {cfg.hot_window} tokens, cold K {one(cfg.k_cold, fl & K.ZP_K, 0)}, "
                     f"cold V {one(cfg.v_cold, fl & K.ZP_V, 0)}")
    if fl & (K.ROTATE_K | K.ROTATE_V):
        parts.append("randomized Hadamard-128 on " + "+".join(n for n, b in (("K", K.ROTATE_K), ("V", K.ROTATE_V))
                                                          if fl & b))
    if fl & K.K_PRE_ROPE:
        parts.append("keys pre-RoPE (turned in the kernel)")
    if cfg.residual_window:
        parts.append(f"{cfg.residual_window}-token 16-bit window")
    if cfg.page_tokens:
        parts.append(f"{cfg.page_tokens}-token pages")
    bits = sorted({f.bits for f in (cfg.k_fmt, cfg.v_fmt, cfg.k_cold, cfg.v_cold) if f is not None and f.bits})
    return "; ".join(parts), "/".join(f"int{b}" for b in bits)


def unfused_ablation(cache, cfg, w, seq_lens, stream, layers=4):
    """What fusion buys: per layer, the fused decode of one step against
    kvq_dequantize of the whole cache to fp32 followed by dense attention
    (torch scaled_dot_product_attention over the dequantized, rotation-undone
    K and V; keys stored pre-RoPE are not turned, so that case times the
    memory traffic only).  Averages over the first `layers` layers."""
    import torch

    from bit_kv_cache_04_gb300 import kvq as K

    L, B, H, Hq, D = cfg.L, cfg.batch, cfg.H_kv, cfg.H_q, cfg.D
    g = Hq // H
    layers = min(layers, L)
    dt = torch.float16 if cfg.in_dtype == K.DT_F16 else torch.bfloat16
    q = torch.randn((1, B, Hq, D), device=stream.device).to(dt)
    out = torch.empty((1, B, Hq, D), dtype=torch.float32, device=stream.device)
    lens = seq_lens.cpu().tolist()
    Tmax = max(lens)
    kf = torch.empty((Tmax, H, D), dtype=torch.float32, device=stream.device)
    vf = torch.empty_like(kf)
    fused, deq, att = [], [], []
    for l in range(layers):
        for rep in range(2):  # second round timed
            ev = [torch.cuda.Event(True) for _ in range(2 + 2 * B)]
            ev[0].record(stream)
            cache.decode(l, 1, q, seq_lens, out, 0, stream)
            ev[1].record(stream)
            with torch.cuda.stream(stream):
                for b in range(B):
                    T = lens[b]
                    cache.dequantize(l, b, 0, T, seq_lens, kf[:T], vf[:T], stream)
                    ev[2 + 2 * b].record(stream)
                    kk = kf[:T].permute(1, 0, 2).repeat_interleave(g, 0)[None]
                    vv = vf[:T].permute(1, 0, 2).repeat_interleave(g, 0)[None]
                    qq = q[0, b].float()[None, :, None, :]
                    torch.nn.functional.scaled_dot_product_attention(qq, kk, vv)
                    ev[3 + 2 * b].record(stream)
            torch.cuda.synchronize()
        fused.append(ev[0].elapsed_time(ev[1]))
        deq.append(sum(ev[(1 if b == 0 else 1 + 2 * b)].elapsed_time(ev[2 + 2 * b]) for b in range(B)))
        att.append(sum(ev[2 + 2 * b].elapsed_time(ev[3 + 2 * b]) for b in range(B)))
    f, d, a_ = statistics.mean(fused), statistics.mean(deq), statistics.mean(att)
    u = d + a_
    return {"fused_ms_per_layer": round(f, 4), "unfused_ms_per_layer": round(u, 4), "speedup": round(u / f, 2),
            "unfused_dequantize_ms": round(d, 4), "unfused_attention_ms": round(a_, 4),
            "what": "per layer: one fused decode launch vs kvq_dequantize (fp32) of every sequence + torch "
                    "scaled_dot_product_attention in fp32 (GQA by repeating kv heads)", "layers": layers}


# ---------------------------------------------------------------------------
# the CPU oracle, timed: worker interpreters with one BLAS thread each
# ---------------------------------------------------------------------------


# Arm implementer / part codes of /proc/cpuinfo (it has no model name on Arm)
_ARM_PARTS = {(0x41, 0xD4F): "Arm Neoverse-V2", (0x41, 0xD40): "Arm Neoverse-V1", (0x41, 0xD0C): "Arm Neoverse-N1",
              (0x41, 0xD49): "Arm Neoverse-N2", (0x41, 0xD8E): "Arm Neoverse-N3", (0x41, 0xD84): "Arm Neoverse-V3"}


def _cpu_model() -> str:
    impl = part = None
    try:
        with open("/proc/cpuinfo") as fh:
            for line in fh:
                key = line.split(":", 1)[0].strip().lower()
                if key in ("model name", "cpu model"):
                    return line.split(":", 1)[1].strip()
                if key == "cpu implementer" and impl is None:
                    impl = int(line.split(":", 1)[1].strip(), 0)
                if key == "cpu part" and part is None:
                    part = int(line.split(":", 1)[1].strip(), 0)
    except (OSError, ValueError):
        pass
    if impl is not None and part is not None:
        return _ARM_PARTS.get((impl, part), f"aarch64 (implementer {impl:#x}, part {part:#x})")
    import platform

    return platform.processor() or platform.machine()


_ONE_THREAD = {"OMP_NUM_THREADS": "1", "OPENBLAS_NUM_THREADS": "1", "MKL_NUM_THREADS": "1"}


def _oracle_cfg(c):
    from oracle import kvq_oracle as O

    zk, zv = bool(c.flags & 32), bool(c.flags & 64)  # the library's asymmetric-block flags
    f = lambda x, zp: None if x is None else O.Fmt(x.bits, x.group, x.axis, zp)  # noqa: E731
    return O.Config(L=c.L, H_kv=c.H_kv, H_q=c.H_q, D=c.D, batch=c.batch, max_T=c.max_T, in_dtype=c.in_dtype,
                    k_fmt=f(c.k_fmt, zk), v_fmt=f(c.v_fmt, zv), k_cold=f(c.k_cold, zk), v_cold=f(c.v_cold, zv),
                    hot_window=c.hot_window, residual_window=c.residual_window, flags=c.flags,
                    rope_theta=c.rope_theta, sign_seed=c.sign_seed, page_tokens=c.page_tokens,
                    n_pages=c.n_pages, max_pages_per_seq=c.max_pages_per_seq)


def _oracle_prep(workload, heads, T, seed):
    """Inputs of one oracle sample: layer 0 of one sequence (drawn with
    `seed`), `heads` kv heads over T tokens, and one query per query head.
    Imports the seeded generators and the oracle only (no CUDA library)."""
    import numpy as np
    import torch

    from bit_kv_cache_04_gb300 import workloads as W

    w = W.make(workload, extra_tokens=0)
    c = w.cfg
    sub = w.scaled(L=1, lengths=[T], extra=0)
    oc = _oracle_cfg(sub.cfg)
    oc.H_kv = heads
    oc.H_q = heads * (c.H_q // c.H_kv)
    table = None
    if oc.page_tokens:
        n = -(-T // oc.page_tokens)
        oc.n_pages, oc.max_pages_per_seq = n, n
        table = np.arange(n, dtype=np.int32)[None]
    k, v = W.kv_tokens(sub, 0, 0, 0, T, "cpu", seed)
    raw = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)  # noqa: E731
    q = W.queries(sub, 1, "cpu", seed)[:, :, : oc.H_q]
    return oc, raw(k[:, :heads]), raw(v[:, :heads]), raw(q), T, table


def _oracle_run(state):
    """One oracle step on prepared inputs: quantize-on-append (fp32), then fp64
    decode attention of every query head.  Returns the packed bytes decoded."""
    from oracle import kvq_oracle as O

    oc, k, v, q, T, table = state
    bufs = O.new_buffers(oc)
    O.append(oc, bufs, 0, k, v, [T], [0], block_table=table)
    O.decode_attention(oc, bufs, 0, 1, q, [T], block_table=table)
    return O.cache_bytes(oc, T)


def _oracle_worker():
    """Worker loop: JSON commands on stdin ("prep", "run", "quit"), one JSON
    reply per command on stdout."""
    state = None
    for line in sys.stdin:
        msg = json.loads(line)
        if msg["cmd"] == "prep":
            state = _oracle_prep(msg["workload"], msg["heads"], msg["T"], msg["seed"])
            reply = {"ready": True}
        elif msg["cmd"] == "run":
            t0 = time.perf_counter()
            nbytes = _oracle_run(state)
            reply = {"dt": time.perf_counter() - t0, "bytes": nbytes}
        else:
            break
        sys.stdout.write(json.dumps(reply) + "\n")
        sys.stdout.flush()


class OraclePool:
    """`n` oracle worker interpreters, one BLAS thread each, started fresh
    (never forked from a process that touched the GPU)."""

    def __init__(self, n: int):
        env = dict(os.environ, **_ONE_THREAD)
        self.procs = [subprocess.Popen([sys.executable, "-c", "import bench; bench._oracle_worker()"],
                                       stdin=subprocess.PIPE, stdout=subprocess.PIPE, text=True, env=env, cwd=ROOT)
                      for _ in range(n)]

    def _ask(self, msgs):
        for p, m in zip(self.procs, msgs):
            p.stdin.write(json.dumps(m) + "\n")
            p.stdin.flush()
        out = []
        for p in self.procs[: len(msgs)]:
            line = p.stdout.readline()
            if not line:
                raise RuntimeError("oracle worker exited")
            out.append(json.loads(line))
        return out

    def prep(self, specs):
        self._ask([dict(cmd="prep", **s) for s in specs])

    def run(self, n=None):
        """Every prepared worker (the first n) runs its sample at once.
        Returns (wall seconds, packed bytes, [per-worker seconds])."""
        n = len(self.procs) if n is None else n
        t0 = time.perf_counter()
        res = self._ask([{"cmd": "run"}] * n)
        wall = time.perf_counter() - t0
        return wall, sum(r["bytes"] for r in res), [r["dt"] for r in res]

    def close(self):
        for p in self.procs:
            try:
                p.stdin.write(json.dumps({"cmd": "quit"}) + "\n")
                p.stdin.close()
            except (BrokenPipeError, OSError):
                pass
        for p in self.procs:
            p.wait(timeout=60)


def _host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _sample_heads(workload: str, heads: int) -> int:
    from bit_kv_cache_04_gb300 import workloads as W

    return max(1, min(heads, W.make(workload, extra_tokens=0).cfg.H_kv))


def cpu_baseline(workload: str, heads: int = 8):
    """The oracle timed on the host: every core at once (one worker per core,
    each on its own sequence) and one core alone, on the same per-worker
    sample (layer 0, `heads` kv heads over the workload's full context)."""
    from bit_kv_cache_04_gb300 import workloads as W

    w = W.make(workload, extra_tokens=0)
    T = w.lengths[0]
    heads = _sample_heads(workload, heads)
    cores = _host_cores()
    pool = OraclePool(cores)
    try:
        pool.prep([{"workload": workload, "heads": heads, "T": T, "seed": i} for i in range(cores)])
        wall_all, bytes_all, _ = pool.run()
        wall_one, bytes_one, _ = pool.run(1)
    finally:
        pool.close()
    sample = (f"per worker: layer 0 of one sequence, {heads} of {w.cfg.H_kv} kv heads x T={T}: oracle "
              f"quantize-on-append (fp32) + fp64 decode attention of their query heads (numpy, one BLAS thread)")
    return {"value": round(bytes_all / wall_all / 1e9, 5), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{cores} workers at once ({bytes_all} packed bytes in {wall_all:.2f} s); " + sample,
            "one_core": {"value": round(bytes_one / wall_one / 1e9, 5), "unit": "GB/s", "cores": 1,
                         "sample": f"1 worker ({bytes_one} packed bytes in {wall_one:.2f} s); " + sample},
            "cpu_model": _cpu_model(), "host_cores": cores}


# ---------------------------------------------------------------------------
# reference arm: the CPU oracle
# ---------------------------------------------------------------------------


def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return
    from bit_kv_cache_04_gb300 import workloads as W

    workload = args.workload or HEADLINE
    w = W.make(workload, extra_tokens=0)
    T = w.lengths[0]
    heads = _sample_heads(workload, 4)
    cores = _host_cores()
    pool = OraclePool(cores)
    try:
        pool.prep([{"workload": workload, "heads": heads, "T": T, "seed": i} for i in range(cores)])
        for _ in range(args.warmup):
            pool.run()
        walls, nbytes = [], 0
        for _ in range(args.steps):
            wall, b, _ = pool.run()
            walls.append(wall)
            nbytes += b
    finally:
        pool.close()
    total_t = sum(walls)
    value = nbytes / total_t / 1e9
    sample = (f"per step: {cores} workers at once, each layer 0 of its own sequence, {heads} of {w.cfg.H_kv} kv "
              f"heads x T={T}: oracle quantize-on-append (fp32) + fp64 decode attention (numpy, one BLAS thread "
              f"per worker)")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 5), "unit": "GB/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(total_t / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32 quantize, f64 attention",
            "data": "synthetic (seeded)",
            "config": {"workload": workload, "sample": f"{cores} x (layer 0, one sequence, {heads} kv heads, T={T})"},
            "cpu_baseline": {"value": round(value, 5), "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": sample, "cpu_model": _cpu_model(), "host_cores": cores},
            "e2e": {"value": round(value, 5), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="",
                    help="measure only this workload (as the headline); default: every workload, "
                         f"{HEADLINE} as the headline")
    ap.add_argument("--only-headline", action="store_true", help="skip the other workloads")
    ap.add_argument("--cpu-heads", type=int, default=8, help="kv heads per oracle worker in the CPU baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ablation", action="store_true",
                    help="also time the unfused path: kvq_dequantize to fp32, then dense attention (torch)")
    ap.add_argument("--layers", type=int, default=0,
                    help="use only this many layers of the headline workload (small cases for profiler captures)")
    ap.add_argument("--batch", type=int, default=0,
                    help="use only the first this many sequences of the headline workload (profiler captures)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()

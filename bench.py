"""Benchmark of the KV-cached Talker forward on GB300 (one JSON line on stdout).

Headline: decode steps/s at batch 1 on the Talker geometry (28 layers, bf16
weights and cache), prefill T=96 then 512 decode steps (cache lengths 97..608),
seeded synthetic weights and embeddings. One timed step = one decode step: the
whole hot path (28 x [norm, QKV, QK-norm, RoPE, KV append, attention, o_proj,
norm, SwiGLU, down] + final norm, codec_head, argmax) for one new row.
Extra fields: prefill tokens/s (T=96) and batched decode steps/s (16 streams).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

--impl reference times the fp64 CPU oracle (this method has no runnable
reference implementation) on a bounded sample of the same workload.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from kv_cached_qwen3_gb300 import inputs  # noqa: E402

METRIC = "decode steps/s (B=1, B=16) + prefill tok/s; % of HBM / bf16 TC roofline"
# DRAM read + write of one decode step (all kernels of the graph) from one ncu capture of the current
# decode kernels (the launch-list summary under profiles/); None whenever a decode kernel changes.
STEP_TRAFFIC = {"bytes": 906790400,
                "note": "ncu dram__bytes_read.sum + dram__bytes_write.sum over the 113 kernels of one decode "
                        "step at cache length about 100, where the algorithmic bytes are 898.8 MB"}
UNIT = "steps/s"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=512)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-extra", action="store_true", help="skip the prefill and batched side measurements")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--prefill-only", type=int, default=0, metavar="T",
                    help="profiling aid: run `--steps` prefills of T rows on the Talker geometry and print their time")
    ap.add_argument("--decode-only", type=int, default=0, metavar="L",
                    help="profiling aid: run `--steps` single-stream decode steps against L imported cache rows "
                         "(Talker widths, --layers layers, --kv storage) and print their time")
    ap.add_argument("--layers", type=int, default=0, help="with --decode-only: layers (default: the Talker's 28)")
    ap.add_argument("--kv", default="bf16", choices=["bf16", "q8_0"], help="with --decode-only: KV storage")
    ap.add_argument("--batched-only", action="store_true",
                    help="profiling aid: run `--steps` 16-stream decode steps (start lengths U{128..2048}) and "
                         "print their time")
    return ap.parse_args()


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def max_over_ranks(values, world, device):
    """Element-wise maximum of a list of floats over the ranks of the default process group
    (one all-reduce; device "cuda" under NCCL, "cpu" under gloo). world == 1: unchanged."""
    if world <= 1:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.p = None

    def __enter__(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                                       "--format=csv,noheader,nounits", "-lms", "100"],
                                      stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.p = None
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.p is not None:
            self.p.terminate()
            try:
                self.out, _ = self.p.communicate(timeout=5)
            except Exception:
                self.p.kill()

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (getattr(self, "out", "") or "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def step_bytes(g, attended_rows):
    """Algorithmic HBM bytes of one decode step for one stream: weights + KV read + KV write."""
    wbytes = g.n_linear_params() * (2 if g.weight_dtype == "bf16" else 4)
    norm_bytes = 4 * (g.n_layers * (2 * g.hidden + 2 * g.head_dim) + g.hidden)
    kv_row = 2 * g.n_layers * g.kv_dim * (2 if g.kv_dtype == "bf16" else 4)
    return wbytes + norm_bytes, kv_row * attended_rows + kv_row


# ----------------------------------------------------------------------------- our arm

def run_ours(args, rank, world, local_rank):
    import torch
    from kv_cached_qwen3_gb300.talker import Talker

    torch.cuda.set_device(local_rank)
    wl = inputs.WORKLOADS["talker_b1"]
    g = wl.geometry
    w = inputs.make_weights(g, wl.seed + 17 * rank)
    T0 = wl.prefill_T
    K, W = args.steps, max(3, args.warmup)
    emb_np = inputs.make_embeddings(g, wl.seed, 0, T0 + max(K, W))
    tk = Talker(g, w)
    tk.kv_init_batched(1, T0 + max(K, W) + 1)
    st = tk.stream
    emb_all = torch.from_numpy(emb_np).cuda()
    e1 = torch.empty(1, g.hidden, device="cuda")
    lg = torch.empty(1, g.vocab, device="cuda")
    am = torch.empty(1, device="cuda", dtype=torch.int32)
    pre = emb_all[:T0].contiguous()

    def one_pass(n, timed):
        tk.prefill(0, pre)
        torch.cuda.synchronize()
        if timed and world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        ev0.record(st)
        for t in range(n):
            e1.copy_(emb_all[T0 + t:T0 + t + 1])
            tk.decode(e1, lg, None, am)
        ev1.record(st)
        torch.cuda.synchronize()
        return ev0.elapsed_time(ev1) / 1e3

    one_pass(W, False)                       # warm-up: W decode steps (graph capture happens here)
    with ClockSampler(local_rank) as cs:
        secs = one_pass(K, True)
    status = tk.sync_status()
    launches_before = tk.kernel_launches()
    # per-kernel count inside one timed step: the graph of one decode step
    tk.prefill(0, pre)
    l0 = tk.kernel_launches()
    e1.copy_(emb_all[T0:T0 + 1])
    tk.decode(e1, lg, None, am)
    per_step_kernels = tk.kernel_launches() - l0
    del launches_before

    # end to end: pinned host embeddings -> device, decode, logits + argmax -> pinned host
    host_emb = torch.from_numpy(emb_np).pin_memory()
    host_lg = torch.empty(K, g.vocab).pin_memory()
    host_am = torch.empty(K, dtype=torch.int32).pin_memory()
    tk.prefill(0, pre)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(st):
        ev0.record(st)
        for t in range(K):
            e1.copy_(host_emb[T0 + t:T0 + t + 1], non_blocking=True)
            tk.decode(e1, lg, None, am)
            host_lg[t].copy_(lg[0], non_blocking=True)
            host_am[t:t + 1].copy_(am, non_blocking=True)
        ev1.record(st)
    torch.cuda.synchronize()
    e2e_secs = ev0.elapsed_time(ev1) / 1e3

    secs, e2e_secs = max_over_ranks([secs, e2e_secs], world, "cuda")

    wbytes, _ = step_bytes(g, 0)
    kv_total = sum(step_bytes(g, T0 + t + 1)[1] for t in range(K))
    total_bytes = wbytes * K + kv_total
    hbm, tc, peak_kind = peaks()
    achieved = total_bytes / secs / 1e9

    extra = {}
    if not args.no_extra:
        extra = side_measurements(tk, g, wl, torch, st, emb_all, pre, hbm, tc)
    tk.close()
    result = {
        "metric": METRIC, "value": world * K / secs, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": secs / K * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (seeded N(0,0.02) weights, N(0,1) embeddings)",
        "config": {"workload": "talker_b1: Talker geometry bf16, prefill T=96 then %d decode steps at batch 1 "
                               "(cache lengths %d..%d)" % (K, T0 + 1, T0 + K),
                   "global_batch": world, "seq_len": T0 + K, "parallelism": "replicas (dp%d)" % world,
                   "l2": "inputs larger than L2 (887 MB of weights streamed per step)"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                     "traffic": STEP_TRAFFIC["bytes"], "traffic_note": STEP_TRAFFIC["note"], "peak_kind": peak_kind,
                     "kernel": "decode step (one CUDA graph of %d kernels)" % per_step_kernels,
                     "algorithmic_bytes_per_step": total_bytes / K},
        "e2e": {"value": world * K / e2e_secs, "unit": UNIT, "h2d_bytes_per_step": g.hidden * 4,
                "d2h_bytes_per_step": g.vocab * 4 + 4},
        "gpu_launches": per_step_kernels * K,
        "clocks": cs.summary(),
        "device_status": status,
    }
    result.update(extra)
    return result


def side_measurements(tk, g, wl, torch, st, emb_all, pre, hbm, tc):
    """Prefill tokens/s at T=96 and batched 16-stream decode steps/s."""
    out = {}
    T0 = wl.prefill_T
    for _ in range(3):
        tk.prefill(0, pre)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    reps = 10
    ev0.record(st)
    for _ in range(reps):
        tk.prefill(0, pre)
    ev1.record(st)
    torch.cuda.synchronize()
    s = ev0.elapsed_time(ev1) / 1e3 / reps
    flops = 2.0 * g.n_linear_params() * T0
    out["prefill"] = {"T": T0, "tokens_per_s": T0 / s, "ms": s * 1e3, "tflops": flops / s / 1e12,
                      "frac_bf16_peak": flops / s / 1e12 / tc}
    # batched: 16 streams, start lengths U{128..2048} (imported N(0,1) K/V), 32 timed steps
    from kv_cached_qwen3_gb300.talker import Talker  # noqa: F401
    b = inputs.WORKLOADS["batched16"]
    lens = inputs.make_start_lengths(b.seed, b.n_streams, *b.start_len_range)
    steps = 32
    tk.kv_init_batched(b.n_streams, int(lens.max()) + steps + 8)
    kvd = torch.bfloat16 if g.kv_dtype == "bf16" else torch.float32
    for s_ in range(b.n_streams):
        L = int(lens[s_])
        kk = torch.randn(g.n_layers, g.n_kv_heads, L, g.head_dim, device="cuda").to(kvd)
        vv = torch.randn(g.n_layers, g.n_kv_heads, L, g.head_dim, device="cuda").to(kvd)
        tk.kv_import(s_, kk, vv, L)
        del kk, vv
    eb = torch.randn(b.n_streams, g.hidden, device="cuda")
    lg = torch.empty(b.n_streams, g.vocab, device="cuda")
    for _ in range(3):
        tk.decode(eb, lg)
    torch.cuda.synchronize()
    ev0.record(st)
    for _ in range(steps):
        tk.decode(eb, lg)
    ev1.record(st)
    torch.cuda.synchronize()
    s = ev0.elapsed_time(ev1) / 1e3 / steps
    wbytes, _ = step_bytes(g, 0)
    kvb = sum(step_bytes(g, int(L) + 3 + steps // 2)[1] for L in lens)
    out["batched16"] = {"streams": int(b.n_streams), "steps_per_s": 1.0 / s, "tokens_per_s": b.n_streams / s,
                        "ms_per_step": s * 1e3, "hbm_frac": (wbytes + kvb) / s / 1e9 / hbm,
                        "start_lengths": [int(x) for x in lens]}
    out["long_context"] = long_context(tk, g, torch, st, hbm, tc)
    out["predictor_loop"] = predictor_loop(torch, hbm)
    return out


def predictor_loop(torch, hbm):
    """Frames/s of the predictor loop: per frame a T=2 prefill (rewinds to 0) and 15 decode steps."""
    from kv_cached_qwen3_gb300.talker import Talker
    pl = inputs.WORKLOADS["predictor_loop"]
    g = pl.geometry
    tk = Talker(g, inputs.make_weights(g, pl.seed))
    T0, n = pl.prefill_T, pl.decode_steps
    tk.kv_init_batched(1, T0 + n + 1)
    emb = torch.from_numpy(inputs.make_embeddings(g, pl.seed, 0, T0 + n)).cuda()
    rows = [emb[T0 + t:T0 + t + 1].contiguous() for t in range(n)]
    lg = torch.empty(1, g.vocab, device="cuda")
    am = torch.empty(1, device="cuda", dtype=torch.int32)
    e1 = torch.empty(1, g.hidden, device="cuda")
    pre = emb[:T0].contiguous()

    def frame():
        tk.prefill(0, pre)
        for t in range(n):
            e1.copy_(rows[t])
            tk.decode(e1, lg, None, am)
    for _ in range(3):
        frame()
    torch.cuda.synchronize()
    frames = 32
    s = timed(torch, tk.stream, frame, frames)
    wbytes, _ = step_bytes(g, 0)
    kv = sum(step_bytes(g, L)[1] for L in range(T0, T0 + n))
    per_frame = (n + 1) * wbytes + kv
    # the same frame as one CUDA graph, each step's input gathered on the device from the previous
    # step's code (15 random bf16 code tables [V, H]) and each code taken through its own output
    # head (15 random bf16 heads [V, H], code j through head j mod 15)
    tables = [torch.randn(g.vocab, g.hidden, device="cuda").to(torch.bfloat16) for _ in range(n)]
    heads = [(0.02 * torch.randn(g.vocab, g.hidden, device="cuda")).to(torch.bfloat16) for _ in range(15)]
    step_heads = [heads[j % 15] for j in range(n + 1)]
    tk.set_code_tables(tables, True)
    codes = torch.empty(n + 1, device="cuda", dtype=torch.int32)
    steps = list(range(n))
    for _ in range(3):
        tk.frame(pre, steps, codes, heads=step_heads)
    torch.cuda.synchronize()
    sg = timed(torch, tk.stream, lambda: tk.frame(pre, steps, codes, heads=step_heads), frames)
    tk.close()
    return {"frames_per_s": 1.0 / s, "ms_per_frame": s * 1e3, "passes_per_frame": n + 1,
            "hbm_frac": per_frame / s / 1e9 / hbm,
            "frame_graph": {"frames_per_s": 1.0 / sg, "ms_per_frame": sg * 1e3,
                            "hbm_frac": per_frame / sg / 1e9 / hbm}}


def timed(torch, st, fn, reps):
    """Average seconds of fn() over reps runs, CUDA events on the library's stream."""
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(st)
    for _ in range(reps):
        fn()
    ev1.record(st)
    torch.cuda.synchronize()
    return ev0.elapsed_time(ev1) / 1e3 / reps


def long_context(tk, g, torch, st, hbm, tc):
    """Prefill T=4096 (tokens/s, tensor-core FLOP rate) and single-stream decode at 8K/16K/32K cached rows."""
    lc = inputs.WORKLOADS["long_context"]
    T = lc.prefill_T
    res = {}
    tk.kv_init_batched(1, max(lc.long_lengths) + 8)
    emb = torch.randn(T, g.hidden, device="cuda")
    for _ in range(2):
        tk.prefill(0, emb)
    torch.cuda.synchronize()
    s = timed(torch, st, lambda: tk.prefill(0, emb), 3)
    layer_params = g.n_linear_params() - g.vocab * g.hidden
    gemm = 2.0 * layer_params * T
    attn = 4.0 * g.n_layers * g.n_q_heads * g.head_dim * T * (T + 1) / 2
    res["prefill"] = {"T": T, "ms": s * 1e3, "tokens_per_s": T / s, "gemm_tflop": gemm / 1e12,
                      "attention_tflop": attn / 1e12, "tflops": (gemm + attn) / s / 1e12,
                      "frac_bf16_peak": (gemm + attn) / s / 1e12 / tc}
    kvd = torch.bfloat16 if g.kv_dtype == "bf16" else torch.float32
    e1 = torch.randn(1, g.hidden, device="cuda")
    lg = torch.empty(1, g.vocab, device="cuda")
    wbytes, _ = step_bytes(g, 0)
    res["decode"] = []
    for L in lc.long_lengths:
        kk = torch.randn(g.n_layers, g.n_kv_heads, L, g.head_dim, device="cuda").to(kvd)
        vv = torch.randn(g.n_layers, g.n_kv_heads, L, g.head_dim, device="cuda").to(kvd)
        tk.kv_import(0, kk, vv, L)
        del kk, vv
        steps = 5

        def run():
            tk.rewind(0, L)
            for _ in range(steps):
                tk.decode(e1, lg)
        run()
        torch.cuda.synchronize()
        s = timed(torch, st, run, 2) / steps
        kvb = step_bytes(g, L + steps // 2)[1]
        res["decode"].append({"L": L, "ms_per_step": s * 1e3, "steps_per_s": 1.0 / s,
                              "hbm_frac": (wbytes + kvb) / s / 1e9 / hbm})
    res["decode_q8_0_kv"] = long_context_q8(torch, lc, hbm)
    return res


def long_context_q8(torch, lc, hbm):
    """Single-stream decode at 8K/16K/32K cached rows with the Q8_0 KV storage (136 of 256 bytes per head row)."""
    from dataclasses import replace
    from kv_cached_qwen3_gb300.talker import Talker
    g = replace(lc.geometry, kv_dtype="q8_0")
    tk = Talker(g, inputs.make_weights(g, lc.seed))
    tk.kv_init_batched(1, max(lc.long_lengths) + 8)
    e1 = torch.randn(1, g.hidden, device="cuda")
    lg = torch.empty(1, g.vocab, device="cuda")
    wbytes = g.n_linear_params() * 2 + 4 * (g.n_layers * (2 * g.hidden + 2 * g.head_dim) + g.hidden)
    row = 2 * g.n_layers * g.n_kv_heads * (g.head_dim + g.head_dim // 32 * 2)   # K and V, codes + scales
    out = []
    for L in lc.long_lengths:
        kk = torch.randn(g.n_layers, g.n_kv_heads, L, g.head_dim, device="cuda")
        vv = torch.randn(g.n_layers, g.n_kv_heads, L, g.head_dim, device="cuda")
        tk.kv_import(0, kk, vv, L)
        del kk, vv
        steps = 5

        def run():
            tk.rewind(0, L)
            for _ in range(steps):
                tk.decode(e1, lg)
        run()
        torch.cuda.synchronize()
        s = timed(torch, tk.stream, run, 2) / steps
        out.append({"L": L, "ms_per_step": s * 1e3, "steps_per_s": 1.0 / s,
                    "hbm_frac": (wbytes + row * (L + steps // 2 + 1)) / s / 1e9 / hbm})
    tk.close()
    return out


# ----------------------------------------------------------------------------- oracle arms

def oracle_decode_rate(budget_s, max_steps):
    """Time the fp64 oracle's incremental decode on the talker_b1 workload: steps/s, sample description."""
    from oracle import Oracle, OracleCache
    wl = inputs.WORKLOADS["talker_b1"]
    g = wl.geometry
    w = inputs.make_weights(g, wl.seed)
    o = Oracle(g, w)
    T0 = wl.prefill_T
    emb = inputs.make_embeddings(g, wl.seed, 0, T0 + max_steps)
    c = OracleCache(o, 1, T0 + max_steps + 1)
    c.prefill(0, emb[:T0])
    t0 = time.perf_counter()
    n = 0
    while n < max_steps and (n == 0 or time.perf_counter() - t0 < budget_s):
        c.decode(emb[T0 + n:T0 + n + 1])
        n += 1
    secs = time.perf_counter() - t0
    return n / secs, "fp64 numpy oracle, talker_b1 decode steps %d..%d after a T=96 prefill (%d steps, %.1f s)" % (
        T0 + 1, T0 + n, n, secs)


def run_reference(args, rank, world):
    if rank != 0:
        return None
    K = max(1, args.steps)
    rate, sample = oracle_decode_rate(budget_s=60.0, max_steps=K)
    cores = os.cpu_count()
    return {"metric": METRIC, "value": rate, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
            "ms_per_step": 1e3 / rate, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": {"workload": "talker_b1: Talker geometry, prefill T=96 then decode at batch 1"},
            "cpu_baseline": {"value": rate, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": rate, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def prefill_only(T, steps, warmup):
    """Prefill of T rows (Talker geometry, long-context weights), `steps` timed runs after `warmup`."""
    import torch
    from kv_cached_qwen3_gb300.talker import Talker
    lc = inputs.WORKLOADS["long_context"]
    g = lc.geometry
    tk = Talker(g, inputs.make_weights(g, lc.seed))
    tk.kv_init_batched(1, T + 8)
    emb = torch.from_numpy(inputs.make_embeddings(g, lc.seed, 0, T)).cuda()
    for _ in range(warmup):
        tk.prefill(0, emb)
    torch.cuda.synchronize()
    s = timed(torch, tk.stream, lambda: tk.prefill(0, emb), steps)
    out = {"prefill_only": {"T": T, "ms": s * 1e3, "tokens_per_s": T / s, "status": tk.sync_status()}}
    tk.close()
    return out


def decode_only(L, layers, kv, steps, warmup):
    """Single-stream decode steps at cache length L (rewound before every timed pass)."""
    import torch
    from dataclasses import replace
    from kv_cached_qwen3_gb300.talker import Talker
    lc = inputs.WORKLOADS["long_context"]
    g = replace(lc.geometry, kv_dtype=kv, n_layers=layers or lc.geometry.n_layers)
    tk = Talker(g, inputs.make_weights(g, lc.seed))
    tk.kv_init_batched(1, L + steps + warmup + 1)
    kvd = torch.bfloat16 if kv == "bf16" else torch.float32
    kk = torch.randn(g.n_layers, g.n_kv_heads, L, g.head_dim, device="cuda").to(kvd)
    tk.kv_import(0, kk, kk, L)
    del kk
    e1 = torch.randn(1, g.hidden, device="cuda")
    lg = torch.empty(1, g.vocab, device="cuda")
    for _ in range(warmup):
        tk.decode(e1, lg)
    tk.rewind(0, L)
    torch.cuda.synchronize()
    s = timed(torch, tk.stream, lambda: tk.decode(e1, lg), steps)
    out = {"decode_only": {"L": L, "layers": g.n_layers, "kv": kv, "ms_per_step": s * 1e3, "status": tk.sync_status()}}
    tk.close()
    return out


def batched_only(steps, warmup):
    """16-stream decode steps on the Talker geometry (the batched workload's start lengths)."""
    import torch
    from kv_cached_qwen3_gb300.talker import Talker
    b = inputs.WORKLOADS["batched16"]
    g = b.geometry
    lens = inputs.make_start_lengths(b.seed, b.n_streams, *b.start_len_range)
    tk = Talker(g, inputs.make_weights(g, b.seed))
    tk.kv_init_batched(b.n_streams, int(lens.max()) + steps + warmup + 1)
    for s_ in range(b.n_streams):
        kk = torch.randn(g.n_layers, g.n_kv_heads, int(lens[s_]), g.head_dim, device="cuda").to(torch.bfloat16)
        tk.kv_import(s_, kk, kk, int(lens[s_]))
        del kk
    eb = torch.randn(b.n_streams, g.hidden, device="cuda")
    lg = torch.empty(b.n_streams, g.vocab, device="cuda")
    for _ in range(warmup):
        tk.decode(eb, lg)
    torch.cuda.synchronize()
    s = timed(torch, tk.stream, lambda: tk.decode(eb, lg), steps)
    out = {"batched_only": {"streams": int(b.n_streams), "ms_per_step": s * 1e3, "status": tk.sync_status()}}
    tk.close()
    return out


def main():
    args = parse()
    rank, world, local_rank = dist_env()
    if world > 1:
        import torch
        backend = "nccl" if args.impl == "ours" else "gloo"
        if args.impl == "ours":
            torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group(backend)
    if args.impl == "reference":
        res = run_reference(args, rank, world)
        if res is not None:
            print(json.dumps(res))
        return
    if args.prefill_only:
        print(json.dumps(prefill_only(args.prefill_only, max(1, args.steps), max(1, args.warmup))))
        return
    if args.decode_only:
        print(json.dumps(decode_only(args.decode_only, args.layers, args.kv, max(1, args.steps), max(1, args.warmup))))
        return
    if args.batched_only:
        print(json.dumps(batched_only(max(1, args.steps), max(1, args.warmup))))
        return
    res = run_ours(args, rank, world, local_rank)
    if rank == 0:
        if not args.no_cpu_baseline:
            rate, sample = oracle_decode_rate(budget_s=15.0, max_steps=64)
            res["cpu_baseline"] = {"value": rate, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
                                   "sample": sample}
        print(json.dumps(res))
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()

#!/usr/bin/env python
"""Decode benchmark: Qwen2.5-7B-shaped W4A16 model, batch 1, context 512.

One step = one greedy decode token through the whole path (embedding, 28
decoder layers of RMSNorm / q|k|v W4A16 GEMV / RoPE + paged KV append / paged
GQA attention with split-K combine / o GEMV / gate|up GEMV + SiLU-mul / down
GEMV, final RMSNorm, fp16 lm_head, argmax), replayed from a CUDA graph.
Inputs are seeded synthetic random-init weights of the model's shapes, with
the prompt's 512 tokens of KV already in the paged cache.

Prints one JSON line (rank 0).  `--impl reference` times the CPU oracle on
the host cores instead (bounded sample, same metric and unit).
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "Qwen2.5-7B-shape W4A16 decode tok/s @b=1,ctx512; kernel HBM GB/s vs peak"
UNIT = "tok/s"
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=128)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--layers", type=int, default=28, help="decoder layers (28 = the workload)")
    ap.add_argument("--context", type=int, default=512)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-kernel-timing", action="store_true")
    ap.add_argument("--seed", type=int, default=1002)
    ap.add_argument("--kernel", default=None,
                    choices=["gateup", "down", "qkv", "o", "attention", "lm_head", "attention_long",
                             "attention_fp8", "prefill", "batching"],
                    help="time one kernel of the workload alone (per-launch JSON line)")
    ap.add_argument("--batch", type=int, default=1, help="sequences (kernel mode)")
    ap.add_argument("--clock-log", default=None,
                    help="write the raw nvidia-smi clock samples of the timed region to this CSV file")
    ap.add_argument("--decode-path", default="auto", choices=["auto", "kernels", "persistent"],
                    help="how decode_step runs a b=1 step (auto: the library's default)")
    ap.add_argument("--workload", default="b1", choices=["b1", "b32"],
                    help="b1: 28-layer b=1 ctx-512 decode; b32: 28-layer batched decode, 32 sequences of "
                         "U[1,4096] tokens in a 16384-page pool")
    return ap.parse_args()


def model_cfg(layers):
    from w4a16_decode_paged_gb300 import synth
    return dict(synth.QWEN_MODEL, n_layers=layers)


def make_inputs(cfg, seed, lens, gen_tokens, pool_pages):
    """numpy weights, pools and paging state for the whole model: B = len(lens)
    sequences with lens[b] tokens already cached and pages assigned for
    gen_tokens more."""
    from w4a16_decode_paged_gb300 import synth
    return synth.model_case(cfg, lens=lens, gen_tokens=gen_tokens, pool_pages=pool_pages, seed=seed)


def workload(args):
    """(cfg, cached lengths per sequence, pool pages, label) of the timed workload."""
    from w4a16_decode_paged_gb300 import synth
    if args.workload == "b32":
        cfg = dict(synth.QWEN_BATCHED, n_layers=args.layers)
        post = synth.batched_lens(synth.rng(cfg["seed"]), cfg["batch"], cfg["max_context"], cfg["forced_lens"])
        label = (f"qwen2.5-7b-{cfg['n_layers']}L-b32-ctxU[1,4096] (15/16/17 forced) batched greedy decode "
                 f"(CUDA graph, tcgen05 projections)")
        return cfg, post - 1, cfg["pool_pages"], label
    cfg = model_cfg(args.layers)
    label = f"qwen2.5-7b-{cfg['n_layers']}L-b1-ctx{args.context} greedy decode (CUDA graph of decode_step)"
    return cfg, np.array([args.context], np.int32), 256, label


# ---------------------------------------------------------------------------- bytes (roofline)

def gemv_bytes(N, K, M=1, bias=False, residual=False):
    b = N * K // 2 + N * (K // 128) * 2 + M * K * 2 + M * N * 2
    if bias:
        b += N * 2
    if residual:
        b += M * N * 2
    return b


def layer_bytes(cfg, lens):
    """(projection bytes, attention bytes) of one layer for sequences whose
    attention covers lens[b] tokens."""
    lens = np.atleast_1d(np.asarray(lens, np.int64))
    B = len(lens)
    H, Hq, Hkv, D, I = cfg["hidden"], cfg["n_q_heads"], cfg["n_kv_heads"], cfg["head_dim"], cfg["inter"]
    nqkv = (Hq + 2 * Hkv) * D
    g = gemv_bytes(nqkv, H, B, bias=True) + gemv_bytes(H, Hq * D, B, residual=True) + \
        (gemv_bytes(2 * I, H, B) - B * I * 2) + gemv_bytes(H, I, B, residual=True)
    att = int(sum(2 * Hkv * int(L) * D * 2 + 4 * math.ceil(int(L) / 16) for L in lens)) + B * 2 * Hq * D * 2
    return g, att


def step_bytes(cfg, lens):
    lens = np.atleast_1d(lens)
    g, att = layer_bytes(cfg, lens)
    lm = cfg["vocab"] * cfg["hidden"] * 2
    return cfg["n_layers"] * (g + att) + lm + len(lens) * cfg["hidden"] * 2


# ---------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples (every 200 ms) of SM clock, power and throttle
    reasons while the timed region runs, read from its stdout; `path`, if
    given, receives a copy of the raw CSV lines."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id, path=None, command=None):
        self.gpu_id = gpu_id
        self.path = path
        self.proc = None
        self.lines = []
        cmd = command or ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
        if command is None and gpu_id is not None:
            cmd += ["-i", str(gpu_id)]
        self.cmd = cmd

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is None:
            return
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = (out or "").splitlines()
        if self.path:
            try:
                with open(self.path, "w") as f:
                    f.write("\n".join(self.lines) + "\n")
            except OSError:
                pass

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        sm, mx, reasons = [], [], set()
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(self.REASONS, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def gpu_uuid(torch, dev):
    try:
        u = torch.cuda.get_device_properties(dev).uuid
        s = str(u)
        return s if s.startswith("GPU-") else "GPU-" + s
    except Exception:
        return None


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            v = d.get("hbm_gbs")
            if isinstance(v, dict):
                v = v.get("value")
            if v:
                return float(v), "measured (MEASURED_PEAKS.json hbm_gbs)"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback (no MEASURED_PEAKS.json on this box)"


def traffic_record(kernel):
    """Per-launch DRAM bytes of `kernel` from the committed ncu summary, or
    None when that summary was taken on different kernel source."""
    import hashlib
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p)).get(kernel)
        if not d:
            return None
        src = os.path.join(ROOT, d["source"])
        h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        return d["dram_bytes_per_launch"] if h == d["source_sha256_16"] else None
    except Exception:
        return None


# ---------------------------------------------------------------------------- oracle timing

def oracle_token_time(cfg, inp, budget_s=15.0):
    """Seconds the CPU oracle needs for one decode step of the workload's
    batch, from a bounded sample: as many whole layers (all sequences) as
    fit in ~budget_s (>= 1), scaled to the model's layer count, plus the
    lm_head rows of one sequence scaled to the batch, and the argmax."""
    import oracle as orc
    from w4a16_decode_paged_gb300 import synth
    orc.build()
    nthreads = orc.num_threads()
    lens = inp["lens"] + 1
    B = len(lens)
    x = inp["embed"][inp["tok"]].copy()
    t_layers, n_done = 0.0, 0
    for l in range(cfg["n_layers"]):
        kp, vp = synth.host_pool(inp, l, "k"), synth.host_pool(inp, l, "v")
        t0 = time.perf_counter()
        x = orc.decoder_layer(cfg, inp["layers"][l], x, kp, vp, inp["bt"], lens)
        t_layers += time.perf_counter() - t0
        n_done += 1
        if t_layers > budget_s * 0.7:
            break
    t0 = time.perf_counter()
    xn = orc.rmsnorm(x[:1], inp["fnorm"], cfg["eps"])
    logits = orc.fp16_gemv(xn[0], inp["lm"])
    orc.argmax(logits)
    t_lm = (time.perf_counter() - t0) * B
    per_step = t_layers / n_done * cfg["n_layers"] + t_lm
    sample = (f"{n_done} of {cfg['n_layers']} decoder layers timed at batch {B} (x{cfg['n_layers'] / n_done:.2f}) "
              f"+ lm_head GEMV and argmax of one sequence (x{B}); contexts {int(lens.min())}..{int(lens.max())}")
    return per_step, nthreads, sample, t_layers + t_lm / B


def run_reference(args):
    """CPU oracle arm: each step is one decoder layer (cycling over the 28)
    plus 1/28 of the lm_head rows, for every sequence of the workload, i.e.
    1/28 of a decode step."""
    import oracle as orc
    from w4a16_decode_paged_gb300 import synth
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    orc.build()
    cfg, lens0, pool_pages, label = workload(args)
    inp = make_inputs(cfg, args.seed if args.workload == "b1" else cfg["seed"], lens0, 16, pool_pages)
    L = cfg["n_layers"]
    lens = inp["lens"] + 1
    B = len(lens)
    x = inp["embed"][inp["tok"]].copy()
    rows = math.ceil(cfg["vocab"] / L)

    def one(i):
        nonlocal x
        l = i % L
        kp, vp = synth.host_pool(inp, l, "k"), synth.host_pool(inp, l, "v")
        x = orc.decoder_layer(cfg, inp["layers"][l], x, kp, vp, inp["bt"], lens)
        lo = (i % L) * rows
        xn = orc.rmsnorm(x, inp["fnorm"], cfg["eps"])
        for b in range(B):
            orc.fp16_gemv(xn[b], inp["lm"][lo:lo + rows])

    for i in range(args.warmup):
        one(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        one(i)
    dt = time.perf_counter() - t0
    tokens = B * args.steps / L
    value = tokens / dt
    out = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic (seeded random-init weights, N(0,1) KV)",
           "config": {"workload": label, "batch": B, "context": int(lens.max()), "layers": L},
           "cpu_baseline": {"value": value, "unit": UNIT, "cores": orc.num_threads(), "kind": "oracle",
                            "sample": f"each step = 1 of {L} decoder layers + 1/{L} of the lm_head rows "
                                      f"(= 1/{L} decode step of {B} sequence(s)), {args.steps} steps"},
           "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out))
    return 0


# ---------------------------------------------------------------------------- native arm

def run_kernel(args):
    """One kernel of the Qwen-shaped layer, launched K times from a CUDA graph
    (weights rotated over enough copies to exceed L2), timed with events."""
    import torch
    from w4a16_decode_paged_gb300 import api, build, synth
    build.build()
    dev = torch.device("cuda", 0)
    cfg = dict(synth.QWEN_LAYER, codes="symmetric")
    H, Hq, Hkv, D, I = cfg["hidden"], cfg["n_q_heads"], cfg["n_kv_heads"], cfg["head_dim"], cfg["inter"]
    B, L = args.batch, args.context
    r = synth.rng(args.seed)
    tdev = lambda a: torch.from_numpy(np.ascontiguousarray(a.view(np.int32) if a.dtype == np.uint32 else a)).to(dev)
    name = args.kernel
    if name == "prefill":
        # the 28-layer model (the b=1 workload's weights), a 512-token prompt
        # prefilled args.steps times from an empty cache
        from w4a16_decode_paged_gb300 import synth as _s  # noqa: F401
        cfg, lens0, pool_pages, _ = workload(args)
        inp = make_inputs(cfg, args.seed, lens0, 64, pool_pages)
        dls = [api.device_layer(w, api.device_pool(inp, l, "k", dev), api.device_pool(inp, l, "v", dev), device=dev)
               for l, w in enumerate(inp["layers"])]
        model = api.Model(cfg, dls, embed=tdev(inp["embed"]), final_norm=tdev(inp["fnorm"]), lm_head=tdev(inp["lm"]),
                          max_batch=1, max_context=600, num_pages=inp["pool_pages"])
        stream = torch.cuda.Stream(device=dev)
        res = time_prefill(torch, api, model, cfg, tdev(inp["bt"]), dev, stream, T=512, reps=max(1, args.steps))
        res.update({"kernel": "prefill", "workload": "28 layers, 512-token prompt, empty cache"})
        print(json.dumps(res))
        model.close()
        return 0
    if name == "batching":
        # the 28-layer model (the b=1 workload's weights) under continuous
        # batching: 64 sequences through 32 batch slots
        cfg, lens0, pool_pages, _ = workload(args)
        inp = make_inputs(cfg, args.seed, lens0, 64, pool_pages)
        Hkv, D = cfg["n_kv_heads"], cfg["head_dim"]
        zeros = lambda n: (torch.zeros((n, Hkv, 16, D), dtype=torch.float16, device=dev),
                           torch.zeros((n, Hkv, 16, D), dtype=torch.float16, device=dev))
        res = time_batching(api, cfg, inp["layers"], tdev(inp["embed"]), tdev(inp["fnorm"]), tdev(inp["lm"]),
                            zeros, lambda: torch.cuda.synchronize(dev), time.perf_counter)
        res.update({"kernel": "batching", "workload": "28 layers, 64 sequences, prompts U[16,128], 64 new tokens "
                                                      "each, 32 batch slots"})
        print(json.dumps(res))
        return 0
    if name in ("attention_long", "attention_fp8"):
        stream = torch.cuda.Stream(device=dev)
        with torch.cuda.stream(stream):
            res = time_attention_long(torch, api, dev, stream, reps=max(1, args.steps), fp8=name == "attention_fp8")
        peak, src = measured_peak()
        res.update({"kernel": name, "frac_of_peak": res["gbs"] / peak, "peak_gbs": peak, "peak_source": src})
        print(json.dumps(res))
        return 0
    if name == "attention":
        lens = np.full(B, L, np.int32)
        pages = B * ((L + 15) // 16) + 8
        kp = torch.randn((pages, Hkv, 16, D), device=dev).half()
        vp = torch.randn((pages, Hkv, 16, D), device=dev).half()
        bt = tdev(synth.block_table(r, lens, pages))
        ld = tdev(lens)
        q = torch.randn((B, Hq, D), device=dev).half()
        out = torch.empty_like(q)
        part = api.paged_gqa_decode_default_partition(B, Hkv, L) if args.context < 8192 else 512
        ws = torch.zeros(api.paged_gqa_decode_workspace_size(B, Hq, Hkv, L, part), dtype=torch.uint8, device=dev)
        nbytes = B * (2 * Hkv * L * D * 2 + 4 * ((L + 15) // 16) + 2 * Hq * D * 2)
        copies = 1
        fns = [lambda: api.paged_gqa_decode(q, kp, vp, bt, ld, max_context=L, partition_tokens=part, workspace=ws,
                                            out=out)]
        extra = {"partition_tokens": part, "context": L, "batch": B}
    elif name == "lm_head":
        lm = torch.randn((cfg.get("vocab", 152064) or 152064, H), device=dev).half() * 0.02
        x = torch.randn((B, H), device=dev).half()
        ws = torch.zeros(api.load().lm_head_argmax_workspace_size(B, lm.shape[0]), dtype=torch.uint8, device=dev)
        toks = torch.empty(B, dtype=torch.int32, device=dev)
        nbytes = lm.numel() * 2 + B * H * 2 + B * 4
        copies = 1
        fns = [lambda: api.lm_head_argmax(x, lm, tokens_out=toks, workspace=ws)]
        extra = {"vocab": lm.shape[0], "batch": B}
    else:
        shapes = {"gateup": (I, H), "down": (H, I), "qkv": ((Hq + 2 * Hkv) * D, H), "o": (H, Hq * D)}
        N, K = shapes[name]
        one = (2 * N if name == "gateup" else N) * (K // 2 + K // 128 * 2)
        copies = max(1, math.ceil(3 * 128e6 / one))
        x = torch.randn((B, K), device=dev).half()
        g = torch.ones(K, device=dev).half()
        res = torch.randn((B, N), device=dev).half()
        y = torch.empty((B, N), dtype=torch.float16, device=dev)
        fns = []
        tc = B > 4   # decode batches above 4 take the tensor-core GEMM (RMSNorm not fused)
        if tc:
            ws = torch.zeros(api.load().w4a16_gemm_workspace_size(B, K, N, int(name == "gateup")),
                             dtype=torch.uint8, device=dev)
        for _ in range(copies):
            qw, sc = synth.int4_weight(r, N, K, "symmetric")
            qw, sc = tdev(qw), tdev(sc)
            if tc and name == "gateup":
                qu, su = synth.int4_weight(r, N, K, "symmetric")
                qu, su = tdev(qu), tdev(su)
                fns.append(lambda qw=qw, sc=sc, qu=qu, su=su: api.w4a16_gemm_silu_mul(x, qw, sc, qu, su, out=y,
                                                                                      workspace=ws))
            elif tc:
                fns.append(lambda qw=qw, sc=sc: api.w4a16_gemm(x, qw, sc, residual=res if name in ("down", "o")
                                                               else None, out=y, workspace=ws))
            elif name == "gateup":
                qu, su = synth.int4_weight(r, N, K, "symmetric")
                qu, su = tdev(qu), tdev(su)
                fns.append(lambda qw=qw, sc=sc, qu=qu, su=su: api.w4a16_gemv_silu_mul(x, g, 1e-6, qw, sc, qu, su, out=y))
            elif name == "qkv":
                fns.append(lambda qw=qw, sc=sc: api.w4a16_gemv_rmsnorm(x, g, 1e-6, qw, sc, out=y))
            else:
                fns.append(lambda qw=qw, sc=sc: api.w4a16_gemv(x, qw, sc, residual=res, out=y))
        nbytes = one + B * K * 2 + B * N * 2 + (B * N * 2 if name in ("down", "o") else 0)
        extra = {"N": N, "K": K, "batch": B, "weight_copies": copies}
    stream = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(stream):
        for f in fns:
            f()
        stream.synchronize()
        g_ = torch.cuda.CUDAGraph()
        per_graph = max(len(fns), 8)
        with torch.cuda.graph(g_, stream=stream, capture_error_mode="relaxed"):
            for i in range(per_graph):
                fns[i % len(fns)]()
        for _ in range(args.warmup):
            g_.replay()
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            g_.replay()
        e1.record(stream)
        stream.synchronize()
    per = e0.elapsed_time(e1) / 1e3 / (args.steps * per_graph)
    peak, src = measured_peak()
    out = {"kernel": name, "us_per_launch": per * 1e6, "bytes_per_launch": nbytes, "gbs": nbytes / per / 1e9,
           "frac_of_peak": nbytes / per / 1e9 / peak, "peak_gbs": peak, "peak_source": src,
           "launches_timed": args.steps * per_graph, **extra}
    print(json.dumps(out))
    return 0


def time_attention_long(torch, api, dev, stream, reps=6, fp8=False):
    """paged_gqa_decode on the long-context workload: 4 sequences of 32768
    tokens (2048 pages each, scattered over a 16384-page pool), 28 query /
    4 kv heads, 512-token partitions merged by the last partition.  Two pool
    copies alternate so the 268 MB a launch reads does not stay in L2; a
    CUDA graph of 8 launches, CUDA events on the launching stream.  fp8:
    the same over FP8 (E4M3) pools with fp32 row scales (134 MB of codes +
    4 MB of scales per launch)."""
    from w4a16_decode_paged_gb300 import synth
    c = synth.QWEN_LONG
    B, Hq, Hkv, D, L, pool, part = (c["batch"], c["n_q_heads"], c["n_kv_heads"], c["head_dim"], c["context"],
                                    c["pool_pages"], c["partition_tokens"])
    r = synth.rng(c["seed"] + 11)
    lens = np.full(B, L, np.int32)
    bt = torch.from_numpy(synth.block_table(r, lens, pool)).to(dev)
    ld = torch.from_numpy(lens).to(dev)
    q = torch.randn((B, Hq, D), device=dev, dtype=torch.float16)
    out = torch.empty_like(q)
    ws = torch.zeros(api.paged_gqa_decode_workspace_size(B, Hq, Hkv, L, part), dtype=torch.uint8, device=dev)
    if fp8:
        codes = lambda: torch.randint(0, 0x7E, (pool, Hkv, 16, D), device=dev, dtype=torch.uint8)
        scales = lambda: torch.rand((pool, Hkv, 16), device=dev, dtype=torch.float32) * 0.01 + 0.001
        pools = [(codes(), codes(), scales(), scales()) for _ in range(2)]
        fn = lambda i: api.paged_gqa_decode_fp8(q, *pools[i % 2], bt, ld, max_context=L, partition_tokens=part,
                                                workspace=ws, out=out)
        nbytes = B * (2 * Hkv * L * (D + 4) + 4 * ((L + 15) // 16) + 2 * Hq * D * 2)
    else:
        pools = [(torch.randn((pool, Hkv, 16, D), device=dev, dtype=torch.float16),
                  torch.randn((pool, Hkv, 16, D), device=dev, dtype=torch.float16)) for _ in range(2)]
        fn = lambda i: api.paged_gqa_decode(q, pools[i % 2][0], pools[i % 2][1], bt, ld, max_context=L,
                                            partition_tokens=part, workspace=ws, out=out)
        nbytes = B * (2 * Hkv * L * D * 2 + 4 * ((L + 15) // 16) + 2 * Hq * D * 2)
    per = _graph_time(torch, stream, fn, 8, reps)
    del pools
    return {"us_per_launch": per * 1e6, "bytes_per_launch": nbytes, "gbs": nbytes / per / 1e9,
            "launches_timed": 8 * reps, "workload": f"b={B} x ctx {L}, {Hq}/{Hkv} heads, partitions of {part}"
                                                    + (", FP8 E4M3 pages" if fp8 else "")}


def time_layer_long(torch, api, dls, dev, stream, reps=6):
    """One whole decoder layer (RMSNorm, q|k|v, RoPE + append + attention,
    o + residual, RMSNorm, gate|up + SiLU-mul, down + residual) on the
    long-context workload: 4 sequences of 32768 tokens in a 16384-page pool,
    512-token partitions, the b=1 workload's layer-0 weights (CUDA-core
    GEMVs at M = 4).  The 268 MB of KV a call reads pushes the layer's
    120 MB of weights out of L2 between calls; a CUDA graph of 4 calls, CUDA
    events on the launching stream.  The appended token's slot is the same
    every call (the lengths are not advanced)."""
    from w4a16_decode_paged_gb300 import synth
    c = synth.QWEN_LONG
    B, Hkv, D, L, pool, part = (c["batch"], c["n_kv_heads"], c["head_dim"], c["context"], c["pool_pages"],
                                c["partition_tokens"])
    r = synth.rng(c["seed"] + 13)
    lens = np.full(B, L, np.int32)
    bt = torch.from_numpy(synth.block_table(r, lens, pool)).to(dev)
    ld = torch.from_numpy(lens).to(dev)
    layer = {**dls[0], "k_pool": torch.randn((pool, Hkv, 16, D), device=dev, dtype=torch.float16),
             "v_pool": torch.randn((pool, Hkv, 16, D), device=dev, dtype=torch.float16)}
    model = api.Model(dict(c, vocab=0), [layer], max_batch=B, max_context=L, num_pages=pool, partition_tokens=part)
    x = (torch.randn((B, c["hidden"]), device=dev) * 0.5).half()
    fn = lambda i: model.layer(0, x, bt, ld, stream=stream)
    per = _graph_time(torch, stream, fn, 4, reps)
    assert model.check_errors(stream) == 0
    g, att = layer_bytes(c, lens)
    model.close()
    del layer
    return {"us_per_launch": per * 1e6, "bytes_per_launch": g + att, "gbs": (g + att) / per / 1e9,
            "launches_timed": 4 * reps,
            "workload": f"one decoder layer, b={B} x ctx {L}, partitions of {part} (weights {g / 1e6:.1f} MB, "
                        f"KV {att / 1e6:.1f} MB)"}


def _graph_time(torch, stream, fn, per_graph, reps):
    """Seconds per call of fn(i), i = 0..per_graph-1 captured in one CUDA
    graph and replayed `reps` times (CUDA events on the launching stream)."""
    for i in range(min(2, per_graph)):
        fn(i)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
        for i in range(per_graph):
            fn(i)
    g.replay()
    stream.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        g.replay()
    e1.record(stream)
    stream.synchronize()
    return e0.elapsed_time(e1) / 1e3 / (reps * per_graph)


def time_b32_step(torch, api, cfg, dls, embed, fnorm, lm, dev, stream, steps=20, warmup=3):
    """The batched decode workload on the same 28 layers' weights: 32
    sequences whose lengths are uniform on [1, 4096] with 15/16/17 forced
    into three slots, each layer with its own 16384-page K and V pools
    (N(0,1)), random disjoint block tables; decode_step (tensor-core
    projections, CUDA graph) timed over `steps` steps."""
    from w4a16_decode_paged_gb300 import synth
    c = synth.QWEN_BATCHED
    B, pool = c["batch"], c["pool_pages"]
    r = synth.rng(c["seed"])
    post = synth.batched_lens(r, B, c["max_context"], c["forced_lens"])
    lens0 = post - 1
    gen = steps + warmup + 4
    bt_np = synth.block_table(r, lens0 + gen, pool)
    Hkv, D = cfg["n_kv_heads"], cfg["head_dim"]
    layers = []
    for w in dls:
        layers.append({**w, "k_pool": torch.randn((pool, Hkv, 16, D), device=dev, dtype=torch.float16),
                       "v_pool": torch.randn((pool, Hkv, 16, D), device=dev, dtype=torch.float16)})
    model = api.Model(cfg, layers, embed=embed, final_norm=fnorm, lm_head=lm, max_batch=B,
                      max_context=int(lens0.max()) + gen, num_pages=pool)
    bt = torch.from_numpy(bt_np).to(dev)
    lens = torch.from_numpy(lens0.astype(np.int32)).to(dev)
    tok = torch.from_numpy(r.integers(0, cfg["vocab"], size=B).astype(np.int32)).to(dev)
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            model.decode_step(tok, tok, bt, lens, use_graph=True)
        stream.synchronize()
        assert model.check_errors(stream) == 0
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            model.decode_step(tok, tok, bt, lens, use_graph=True)
        e1.record(stream)
        stream.synchronize()
        assert model.check_errors(stream) == 0
    ms = e0.elapsed_time(e1) / steps
    mid = lens0 + 1 + warmup + steps // 2
    sb = step_bytes(cfg, mid)
    model.close()
    del layers
    return {"ms_per_step": ms, "tok_per_s": B / (ms / 1e3), "bytes_per_step": sb, "gbs": sb / (ms / 1e3) / 1e9,
            "steps_timed": steps, "kernels_per_step": None,
            "workload": "28 layers, batch 32, lengths U[1,4096] (15/16/17 forced), 16384-page pools, CUDA graph"}


def time_prefill(torch, api, model, cfg, bt, dev, stream, T=512, reps=3):
    """Time to first token of a T-token prompt on the model: w4a16_prefill
    (every layer over the T rows, the prompt's KV pages written, the last
    token's lm_head and argmax), CUDA events on the launching stream, each
    rep from an empty cache; the prompt is seeded random tokens."""
    r = np.random.default_rng(4242)
    tokens = torch.from_numpy(r.integers(0, cfg["vocab"], size=T).astype(np.int32)).to(dev)
    lens0 = torch.zeros(1, dtype=torch.int32, device=dev)
    out_tok = torch.empty(1, dtype=torch.int32, device=dev)
    ws = torch.empty(int(api.load().w4a16_prefill_workspace_size(model._h, T, bt.shape[1])), dtype=torch.uint8,
                     device=dev)
    times = []
    with torch.cuda.stream(stream):
        for i in range(reps + 1):
            lens0.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            model.prefill(tokens, bt[:1].contiguous(), lens0, token_out=out_tok, workspace=ws, stream=stream)
            e1.record(stream)
            stream.synchronize()
            if i > 0:
                times.append(e0.elapsed_time(e1))
        assert model.check_errors(stream) == 0
    ms = statistics.median(times)
    return {"ms": ms, "prompt_tokens": T, "tok_per_s": T / (ms / 1e3), "reps": reps,
            "how": "w4a16_prefill: tensor-core GEMMs over row blocks of 128 (gate|up 64), causal paged attention, "
                   "lm_head"}


def batching_prompts(seed, n_seq, lo=16, hi=128):
    """Seeded prompt lengths of the continuous-batching run: uniform on [lo, hi]."""
    r = np.random.default_rng(seed)
    return [int(n) for n in r.integers(lo, hi + 1, size=n_seq)]


def time_batching(api, cfg, dls, embed, fnorm, lm, new_pools, sync, clock, n_seq=64, max_batch=32,
                  new_tokens=64, seed=4343):
    """Continuous batching through the library's scheduler and page allocator
    (w4a16_batcher_*): n_seq sequences with prompts of 16..128 seeded random
    tokens and new_tokens generated tokens each, through max_batch slots.  A
    prompt is fed one token per step, so a sequence with a p-token prompt
    occupies its slot for p + new_tokens - 1 steps.  The pool gives every
    slot room for its longest sequence (no preemption).  The same submissions
    run twice; the first pass captures the step's graph for every batch size
    it meets and is not timed.  Time is host wall clock around the step loop
    (scheduling, uploads and the decode steps), the device synchronised on
    both sides."""
    plens = batching_prompts(seed, n_seq)
    max_context = max(plens) + new_tokens
    max_blocks = (max_context + 15) // 16
    num_pages = max_batch * max_blocks
    layers = [api.device_layer(w, *new_pools(num_pages)) for w in dls]
    model = api.Model(cfg, layers, embed=embed, final_norm=fnorm, lm_head=lm, max_batch=max_batch,
                      max_context=max_context, num_pages=num_pages)
    bat = api.Batcher(model, num_pages=num_pages, max_batch=max_batch, max_blocks=max_blocks,
                      max_context=max_context)
    r = np.random.default_rng(seed + 1)
    prompts = [r.integers(0, cfg["vocab"], size=p).astype(np.int32) for p in plens]
    res = None
    for timed in (False, True):
        ids = [bat.submit(p, new_tokens) for p in prompts]
        steps = token_steps = 0
        sync()
        t0 = clock()
        while True:
            n = bat.step()
            if n == 0:
                break
            steps += 1
            token_steps += n
        sync()
        sec = clock() - t0
        gen = sum(len(bat.poll(i)[0]) for i in ids)
        if timed:
            st = bat.stats()
            res = {"sequences": n_seq, "max_batch": max_batch, "new_tokens_each": new_tokens,
                   "prompt_tokens": int(sum(plens)), "generated_tokens": gen, "steps": steps,
                   "token_steps": token_steps, "mean_batch": token_steps / max(steps, 1), "seconds": sec,
                   "generated_tok_per_s": gen / sec, "token_steps_per_s": token_steps / sec,
                   "ms_per_step": sec / max(steps, 1) * 1e3, "preemptions": st["preemptions"],
                   "free_pages_after": st["free_pages"], "num_pages": num_pages,
                   "how": "w4a16_batcher_step loop, host wall clock, prompts fed one token per step"}
    bat.close()
    model.close()
    return res


def max_over_ranks(values, dev, world):
    """Each timing, maximised over the ranks of the job (the slowest replica
    sets the job's time).  dev: the device of the collective's tensor (cuda
    for NCCL, cpu for gloo)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=dev)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def job_throughput(world, batch, steps, seconds):
    """Tokens per second of the whole job: every rank decodes `batch`
    sequences for `steps` steps (weak scaling), in `seconds` (max over ranks)."""
    return world * batch * steps / seconds


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    if args.kernel:
        return run_kernel(args)

    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)

    from w4a16_decode_paged_gb300 import api, build
    build.build()

    cfg, lens0, pool_pages, label = workload(args)
    B = len(lens0)
    K, W = args.steps, args.warmup
    gen = K + W + 16
    max_ctx = int(lens0.max()) + gen
    seed = (args.seed if args.workload == "b1" else cfg["seed"]) + rank
    t_gen = time.perf_counter()
    inp = make_inputs(cfg, seed, lens0, gen, pool_pages)
    t_gen = time.perf_counter() - t_gen

    tdev = lambda a: torch.from_numpy(np.ascontiguousarray(a.view(np.int32) if a.dtype == np.uint32 else a)).to(dev)
    dls = [api.device_layer(w, api.device_pool(inp, l, "k", dev), api.device_pool(inp, l, "v", dev), device=dev)
           for l, w in enumerate(inp["layers"])]
    embed, fnorm, lm = tdev(inp["embed"]), tdev(inp["fnorm"]), tdev(inp["lm"])
    model = api.Model(cfg, dls, embed=embed, final_norm=fnorm, lm_head=lm, max_batch=B, max_context=max_ctx,
                      num_pages=inp["pool_pages"])
    bt = tdev(inp["bt"])
    tok = tdev(inp["tok"])
    lens_init = tdev(inp["lens"])
    lens = lens_init.clone()
    stream = torch.cuda.Stream(device=dev)
    model.set_decode_path(args.decode_path)
    kernels_per_step = model.kernel_count(B)
    path = model.decode_path(B)

    def barrier():
        if world > 1:
            dist.barrier()

    with torch.cuda.stream(stream):
        # ---- device-resident timing: K graph replays --------------------
        lens.copy_(lens_init)
        for _ in range(W):
            model.decode_step(tok, tok, bt, lens, use_graph=True)
        stream.synchronize()
        assert model.check_errors(stream) == 0
        lens.copy_(lens_init)
        stream.synchronize()
        barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with ClockSampler(gpu_uuid(torch, dev), args.clock_log) as clk:
            e0.record(stream)
            for _ in range(K):
                model.decode_step(tok, tok, bt, lens, use_graph=True)
            e1.record(stream)
            stream.synchronize()
        torch.cuda.synchronize()
        barrier()
        ms = e0.elapsed_time(e1)
        assert torch.equal(lens, lens_init + K)
        assert model.check_errors(stream) == 0

        # ---- end to end through the C ABI with host buffers --------------
        h_in = torch.empty(B, dtype=torch.int32, pin_memory=True)
        h_out = torch.empty(B, dtype=torch.int32, pin_memory=True)
        h_in.copy_(torch.from_numpy(inp["tok"]))
        lens.copy_(lens_init)
        for _ in range(2):
            tok.copy_(h_in, non_blocking=True)
            model.decode_step(tok, tok, bt, lens, use_graph=True)
            h_out.copy_(tok, non_blocking=True)
            stream.synchronize()
        lens.copy_(lens_init)
        stream.synchronize()
        barrier()
        t0 = time.perf_counter()
        for _ in range(K):
            tok.copy_(h_in, non_blocking=True)
            model.decode_step(tok, tok, bt, lens, use_graph=True)
            h_out.copy_(tok, non_blocking=True)
            stream.synchronize()
            h_in.copy_(h_out)
        e2e_s = time.perf_counter() - t0
        barrier()

        # ---- the same steps without the CUDA graph (direct launches) ------
        eager = None
        if not args.no_kernel_timing:
            ke = min(K, 20)
            lens.copy_(lens_init)
            for _ in range(2):
                model.decode_step(tok, tok, bt, lens, use_graph=False)
            stream.synchronize()
            lens.copy_(lens_init)
            g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            g0.record(stream)
            for _ in range(ke):
                model.decode_step(tok, tok, bt, lens, use_graph=False)
            g1.record(stream)
            stream.synchronize()
            assert model.check_errors(stream) == 0
            eager = {"ms_per_step": g0.elapsed_time(g1) / ke, "steps": ke,
                     "how": "decode_step with use_graph=0: the same kernels launched from the host each step"}
            lens.copy_(lens_init)

        # ---- the other decode path on the same model (b=1): its step time --
        other = None
        if args.workload == "b1" and not args.no_kernel_timing:
            alt = "persistent" if path == "kernels" else "kernels"
            model.set_decode_path(alt)
            if model.decode_path(B) == alt:
                lens.copy_(lens_init)
                for _ in range(3):
                    model.decode_step(tok, tok, bt, lens, use_graph=True)
                stream.synchronize()
                assert model.check_errors(stream) == 0
                lens.copy_(lens_init)
                a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a0.record(stream)
                for _ in range(K):
                    model.decode_step(tok, tok, bt, lens, use_graph=True)
                a1.record(stream)
                stream.synchronize()
                assert model.check_errors(stream) == 0
                other = {"decode_path": alt, "ms_per_step": a0.elapsed_time(a1) / K,
                         "tok_per_s": B * K / (a0.elapsed_time(a1) / 1e3), "kernels_per_step": model.kernel_count(B)}
            model.set_decode_path(args.decode_path)
            lens.copy_(lens_init)

        # ---- time to first token: a 512-token prompt in one prefill -------
        ttft = None
        if args.workload == "b1" and not args.no_kernel_timing:
            ttft = time_prefill(torch, api, model, cfg, bt, dev, stream, T=512)
            lens.copy_(lens_init)

        # ---- the projections alone, and the other workloads' kernels -------
        kern = None
        if not args.no_kernel_timing:
            kern = time_gemv_kernels(torch, api, cfg, dls, dev, stream, B)
            if args.workload == "b1":
                kern["attention_b4_ctx32768"] = time_attention_long(torch, api, dev, stream)
                kern["attention_fp8_b4_ctx32768"] = time_attention_long(torch, api, dev, stream, fp8=True)
                kern["layer_b4_ctx32768"] = time_layer_long(torch, api, dls, dev, stream)
                kern["gateup_tc_m32"] = time_gemv_kernels(torch, api, cfg, dls, dev, stream, 32,
                                                          only=("gateup",))["gateup"]
                kern["b32_step"] = time_b32_step(torch, api, cfg, dls, embed, fnorm, lm, dev, stream)
                torch.cuda.empty_cache()

    # max over ranks
    ms, e2e_s = max_over_ranks([ms, e2e_s], dev, world)
    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    peak, peak_src = measured_peak()
    value = job_throughput(world, B, K, ms / 1e3)
    mid_lens = inp["lens"] + 1 + K // 2
    sb = step_bytes(cfg, mid_lens)
    out = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": W,
           "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
           "dtype": "int4 weights x fp16 activations, fp32 accumulate",
           "data": "synthetic (seeded random-init weights of the model's shapes; N(0,1) KV prefill)",
           "config": {"workload": label, "batch": B,
                      "context": args.context if B == 1 else f"{int(inp['lens'].min()) + 1}..{int(inp['lens'].max()) + 1}",
                      "layers": cfg["n_layers"],
                      "l2": f"inputs larger than L2: {sb / 1e9:.2f} GB read per step",
                      "parallelism": f"replicas x{world}"},
           "gpu_launches": kernels_per_step * K,
           "decode_path": path,
           "e2e": {"value": world * B * K / e2e_s, "unit": UNIT, "h2d_bytes_per_step": 4 * B,
                   "d2h_bytes_per_step": 4 * B},
           "clocks": clk.summary()}
    out["step_roofline"] = {"bytes_per_step": sb, "achieved_gbs": sb / (ms / K / 1e3) / 1e9, "peak_gbs": peak,
                            "frac": sb / (ms / K / 1e3) / 1e9 / peak, "roofline_ms": sb / (peak * 1e9) * 1e3}
    if path == "persistent":
        # one kernel is the whole step: its bytes are the step's bytes
        ach = sb / (ms / K / 1e3) / 1e9
        out["roofline"] = {"bound": "hbm", "kernel": "w4pg_decode_persistent (the whole b=1 step, one launch)",
                           "achieved": ach, "peak": peak, "unit": "GB/s", "frac": ach / peak,
                           "peak_source": peak_src, "traffic": traffic_record("decode_persistent_b1")}
    elif kern is not None:
        kname = ("w4a16_gemv_silu_mul (gate|up, 3584->2x18944)" if B <= 4 else
                 f"w4a16_gemm_silu_mul (tcgen05, M={B}, gate|up, 3584->2x18944)")
        out["roofline"] = {"bound": "hbm", "kernel": kname,
                           "achieved": kern["gateup"]["gbs"], "peak": peak, "unit": "GB/s",
                           "frac": kern["gateup"]["gbs"] / peak, "peak_source": peak_src,
                           "traffic": traffic_record("gemv_gateup" if B <= 4 else "gemm_tc_gateup_b32")}
    if eager is not None:
        eager["graph_speedup"] = eager["ms_per_step"] / (ms / K)
        out["eager"] = eager
    if ttft is not None:
        out["ttft"] = ttft
    if other is not None:
        other["bytes_roofline_frac"] = sb / (other["ms_per_step"] / 1e3) / 1e9 / peak
        out["other_decode_path"] = other
    if kern is not None:
        for k, v in kern.items():
            if isinstance(v, dict) and "gbs" in v:
                v["frac_of_peak"] = v["gbs"] / peak
        out["kernels"] = kern
    if not args.no_cpu_baseline:
        import oracle as orc
        per_step, cores, sample, spent = oracle_token_time(cfg, inp)
        out["cpu_baseline"] = {"value": B / per_step, "unit": UNIT, "cores": cores, "kind": "oracle",
                               "sample": sample, "seconds_spent": round(spent, 2)}
        orc.set_num_threads(1)
        try:
            per1, _, sample1, spent1 = oracle_token_time(cfg, inp, budget_s=12.0)
        finally:
            orc.set_num_threads(cores)
        out["cpu_baseline"]["single_core"] = {"value": B / per1, "unit": UNIT, "cores": 1, "kind": "oracle",
                                              "sample": sample1, "seconds_spent": round(spent1, 2)}
    out["setup_s"] = {"generate_inputs": round(t_gen, 1)}
    print(json.dumps(out))
    if world > 1:
        dist.destroy_process_group()
    return 0


def fused_qkv(torch, dls):
    """Per layer, the q|k|v weights, scales and biases as one matrix (rows of
    q, then k, then v): the single launch the decode step makes."""
    out = []
    for w in dls:
        out.append({"w": torch.cat([w["wq"], w["wk"], w["wv"]], 0).contiguous(),
                    "s": torch.cat([w["sq"], w["sk"], w["sv"]], 0).contiguous(),
                    "b": torch.cat([w["bq"], w["bk"], w["bv"]], 0).contiguous() if w["bq"] is not None else None,
                    "ln1": w["ln1"]})
    return out


def time_gemv_kernels(torch, api, cfg, dls, dev, stream, B=1, reps=3, only=None):
    """Average device time per launch of each projection kind as used in the
    step at batch B (CUDA-core GEMVs for B <= 4, tensor-core GEMMs with split
    K above), over all layers' weights (rotating, so nothing stays in L2),
    captured in a CUDA graph and timed with CUDA events on the launching
    stream.  The q|k|v projection is timed as the one fused launch of
    (Hq + 2 Hkv) * D rows the step makes."""
    H, Hq, Hkv, D, I = cfg["hidden"], cfg["n_q_heads"], cfg["n_kv_heads"], cfg["head_dim"], cfg["inter"]
    NQKV = (Hq + 2 * Hkv) * D
    x = torch.randn((B, H), device=dev).half()
    xi = torch.randn((B, I), device=dev).half()
    xa = torch.randn((B, Hq * D), device=dev).half()
    y_i = torch.empty((B, I), dtype=torch.float16, device=dev)
    y_h = torch.empty((B, H), dtype=torch.float16, device=dev)
    y_q = torch.empty((B, NQKV), dtype=torch.float16, device=dev)
    qkv = fused_qkv(torch, dls) if (only is None or "qkv" in only) else None
    if B <= 4:
        kinds = {
            "gateup": (lambda i: api.w4a16_gemv_silu_mul(x, dls[i]["ln2"], 1e-6, dls[i]["wg"], dls[i]["sg"],
                                                         dls[i]["wu"], dls[i]["su"], out=y_i),
                       gemv_bytes(2 * I, H, B) - B * I * 2),
            "down": (lambda i: api.w4a16_gemv(xi, dls[i]["wd"], dls[i]["sd"], residual=x, out=y_h),
                     gemv_bytes(H, I, B, residual=True)),
            "qkv": (lambda i: api.w4a16_gemv_rmsnorm(x, qkv[i]["ln1"], 1e-6, qkv[i]["w"], qkv[i]["s"],
                                                     bias=qkv[i]["b"], out=y_q),
                    gemv_bytes(NQKV, H, B, bias=True)),
            "o": (lambda i: api.w4a16_gemv(xa, dls[i]["wo"], dls[i]["so"], residual=x, out=y_h),
                  gemv_bytes(H, Hq * D, B, residual=True)),
        }
    else:
        ws = torch.zeros(max(api.load().w4a16_gemm_workspace_size(B, K_, N_, s_) for N_, K_, s_ in
                             ((I, H, 1), (H, I, 0), (NQKV, H, 0), (H, Hq * D, 0))),
                         dtype=torch.uint8, device=dev)
        kinds = {
            "gateup": (lambda i: api.w4a16_gemm_silu_mul(x, dls[i]["wg"], dls[i]["sg"], dls[i]["wu"], dls[i]["su"],
                                                         out=y_i, workspace=ws),
                       gemv_bytes(2 * I, H, B) - B * I * 2),
            "down": (lambda i: api.w4a16_gemm(xi, dls[i]["wd"], dls[i]["sd"], residual=x, out=y_h, workspace=ws),
                     gemv_bytes(H, I, B, residual=True)),
            "qkv": (lambda i: api.w4a16_gemm(x, qkv[i]["w"], qkv[i]["s"], bias=qkv[i]["b"], out=y_q, workspace=ws),
                    gemv_bytes(NQKV, H, B, bias=True)),
            "o": (lambda i: api.w4a16_gemm(xa, dls[i]["wo"], dls[i]["so"], residual=x, out=y_h, workspace=ws),
                  gemv_bytes(H, Hq * D, B, residual=True)),
        }
    if only is not None:
        kinds = {k: v for k, v in kinds.items() if k in only}
    res = {}
    n = len(dls)
    for name, (fn, nbytes) in kinds.items():
        for i in range(min(2, n)):
            fn(i)  # eager warm-up outside capture
        stream.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
            for i in range(n):
                fn(i)
        g.replay()
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
        stream.synchronize()
        per = e0.elapsed_time(e1) / (reps * len(dls)) / 1e3
        res[name] = {"us_per_launch": per * 1e6, "bytes_per_launch": nbytes, "gbs": nbytes / per / 1e9,
                     "launches_timed": reps * len(dls)}
        del g
    return res


if __name__ == "__main__":
    sys.exit(main())

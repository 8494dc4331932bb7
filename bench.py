#!/usr/bin/env python
"""Benchmark of the GB300 decoder layer through its C ABI.

Headline: prefill tokens/s of one MHA layer shaped like a 7B model (B=1, S=2048, d=4096,
H=G=32, D=128, d_inter=11008, bf16 with fp32 accumulation).  Also measured: the decode
step of the GQA 8B-shaped layer (B=64, cache [64, 8, 4096, 128]) in us/step and the GQA
8B-shaped prefill (B=4, S=4096).  A step is one full pass of the layer.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One JSON line on rank 0.  Under torchrun each rank runs an independent replica on its own
GPU (the layer has no exchange step); `value` sums the tokens of all ranks over the slowest
rank's time.  `--impl reference` times the fp64 CPU oracle on the host cores instead.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decoder-layer prefill tokens/s + decode µs/step on 1 GB300; % of TC/HBM roofline"
MAIN = "mha7b_bf16_b1_s2048"
# the layer's kernels in launch order: both RMSNorms run in the prologue of the GEMM after them
PREFILL_KERNELS = ["qkv_rope_gemm", "attention_prefill", "o_proj_residual_gemm", "gate_up_swiglu_gemm",
                   "down_residual_gemm"]
DECODE_KERNELS = ["rmsnorm_attn", "qkv_gemm_stream", "qkv_rope_fixup", "attention_decode_split",
                  "attention_decode_combine", "o_proj_gemm_stream", "o_proj_residual_rmsnorm_fixup",
                  "gate_up_gemm_stream", "swiglu_fixup", "down_gemm_stream", "down_residual_fixup"]
L2_FLUSH_BYTES = 256 << 20


class L2Flush:
    """Run between timed steps: write a 256 MiB buffer (evicts everything from the 129 MB L2),
    then read another 256 MiB, so that the write's dirty lines go back to HBM here and not
    inside the next timed region (where they would cost an HBM-bound kernel ~19 us)."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        # fp32, so that the sum reads the buffer as it is (an integer sum would first widen it
        # to int64 in a temporary copy: new dirty lines)
        self.r = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def __call__(self):
        self.w.zero_()
        self.r.sum()

# DRAM bytes (read + write) per launch of the dominant kernel, dram__bytes_read.sum +
# dram__bytes_write.sum from one ncu capture of that kernel alone at the headline shapes
# (`bench.py --case NAME`), keyed by kernel and the sha1 of the source file it was measured
# on; a changed source makes the figure stale (reported as null).
NCU_TRAFFIC = {("gate_up_swiglu_gemm", "004dd89b26bf"): 232772608}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extra", action="store_true", help="only the headline workload")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--case", choices=["attention", "gate_up", "down", "o_proj", "qkv", "decode_attention",
                                       "decode_layer", "rmsnorm", "layernorm"],
                    help="time one step alone (W + K launches, CUDA events) instead of the layer")
    ap.add_argument("--workload", default=MAIN, help="workload whose shapes --case uses")
    return ap.parse_args()


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": d["hbm_gbs"], "bf16": d["bf16_tflops"], "bf16_sustained": d["bf16_tflops_sustained"],
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16": 1900.0, "bf16_sustained": 1700.0, "source": "fallback"}


def src_sha(name):
    import hashlib
    with open(os.path.join(ROOT, "llama_decoder_block_gb300", "csrc", name), "rb") as f:
        return hashlib.sha1(f.read()).hexdigest()[:12]


# ------------------------------------------------------------------ clocks

class Clocks:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]
        return False

    def summary(self):
        import statistics
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = max(mx, float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ workloads on the GPU

def dev_weights_from_synth(wl, dev):
    import numpy as np
    import torch
    from llama_decoder_block_gb300 import synth
    st = synth.layer_weights(wl)
    return {k: torch.from_numpy(np.ascontiguousarray(v.data).view(np.int16)).to(dev).view(torch.bfloat16)
            for k, v in st.items()}


def dev_weights_random(wl, dev, seed):
    """Same recipe drawn on the device (seeded torch generator): for the extra workloads."""
    import torch
    L = wl.layer
    g = torch.Generator(device=dev).manual_seed(seed)
    d, H, G, D, I = L.d_model, L.n_heads, L.n_kv_heads, L.head_dim, L.d_inter
    shapes = {"wq": (H * D, d), "wk": (G * D, d), "wv": (G * D, d), "wo": (d, H * D), "w_gate": (I, d),
              "w_up": (I, d), "w_down": (d, I)}
    w = {k: (torch.randn(s, generator=g, device=dev) * 0.02).to(torch.bfloat16) for k, s in shapes.items()}
    for k in ("attn_norm", "ffn_norm"):
        if L.gamma == "ones":
            w[k] = torch.ones(d, dtype=torch.bfloat16, device=dev)
        else:
            w[k] = (1 + 0.1 * torch.randn(d, generator=g, device=dev)).to(torch.bfloat16)
    return w


def bench_stack(api, wl, steps, warmup, dev, pk):
    """The full stack: embedding, n_layers layers, final RMSNorm, fp32 LM head, one step = one forward."""
    import numpy as np
    import torch
    L = wl.layer
    B, S, V = wl.B, wl.S, wl.vocab
    layers = [dev_weights_random(wl, dev, wl.seed * 1000 + l) for l in range(wl.n_layers)]
    g = torch.Generator(device=dev).manual_seed(wl.seed)
    embed = (torch.randn(V, L.d_model, generator=g, device=dev) * 0.02).to(torch.bfloat16)
    lm_head = (torch.randn(V, L.d_model, generator=g, device=dev) * 0.02).to(torch.bfloat16)
    final_norm = torch.ones(L.d_model, dtype=torch.bfloat16, device=dev)
    tokens = torch.randint(0, V, (B, S), generator=g, device=dev, dtype=torch.int32)
    dims = api.Dims(L.d_model, L.n_heads, L.n_kv_heads, L.head_dim, L.d_inter, L.rms_eps, torch.bfloat16)
    st = api.StackArgs(dims, layers, final_norm, embed, lm_head)
    logits = torch.empty(B, S, V, dtype=torch.float32, device=dev)
    c, s = api.rope_tables(L.rope_base, L.head_dim, S)
    cos, sin = torch.from_numpy(c).to(dev), torch.from_numpy(s).to(dev)
    ws = api.workspace(st.workspace_bytes(B, S), dev)
    flush = L2Flush(dev)
    ts = []
    for i in range(warmup + steps):
        flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        api.stack_forward(st, tokens, logits, cos, sin, ws)
        e1.record()
        e1.synchronize()
        if i >= warmup:
            ts.append(e0.elapsed_time(e1))
    assert api.device_status() == 0
    ms = float(np.mean(ts))
    flops = wl.n_layers * sum(prefill_flops(L, B, S).values()) + 2.0 * B * S * L.d_model * V
    res = {"workload": wl.name, "ms_per_forward": round(ms, 2), "tokens_per_s": round(B * S / (ms * 1e-3), 1),
           "tflops": round(flops / (ms * 1e-3) / 1e12, 1),
           "frac_of_burst_peak": round(flops / (ms * 1e-3) / 1e12 / pk["bf16"], 4),
           "frac_of_sustained_peak": round(flops / (ms * 1e-3) / 1e12 / pk["bf16_sustained"], 4),
           "weights_GB": round(sum(t.numel() for w in layers for t in w.values()) * 2 / 1e9, 2)}
    del layers, st, logits, ws, flush
    torch.cuda.empty_cache()
    return res


def bench_stack_decode(api, wl, steps, warmup, dev, pk):
    """One decode step of the whole model (embedding, n_layers layers, final RMSNorm, fp32 LM
    head) for B sequences, replayed as one CUDA graph; direct calls timed beside it."""
    import numpy as np
    import torch
    from llama_decoder_block_gb300 import synth
    L = wl.layer
    B, T, V, d, G, D = wl.B, wl.T_max, wl.vocab, L.d_model, L.n_kv_heads, L.head_dim
    layers = [dev_weights_random(wl, dev, wl.seed * 1000 + l) for l in range(wl.n_layers)]
    g = torch.Generator(device=dev).manual_seed(wl.seed)
    embed = (torch.randn(V, d, generator=g, device=dev) * 0.02).to(torch.bfloat16)
    lm_head = (torch.randn(V, d, generator=g, device=dev) * 0.02).to(torch.bfloat16)
    final_norm = torch.ones(d, dtype=torch.bfloat16, device=dev)
    caches = []
    for _ in range(wl.n_layers):
        k = torch.empty(B, G, T, D, dtype=torch.bfloat16, device=dev).normal_(generator=g)
        v = torch.empty(B, G, T, D, dtype=torch.bfloat16, device=dev).normal_(generator=g)
        caches.append((k, v))
    pos_h = synth.decode_positions(wl)
    pos = torch.from_numpy(pos_h).to(dev)
    tokens = torch.randint(0, V, (B,), generator=g, device=dev, dtype=torch.int32)
    dims = api.Dims(d, L.n_heads, G, D, L.d_inter, L.rms_eps, torch.bfloat16)
    st = api.StackArgs(dims, layers, final_norm, embed, lm_head)
    logits = torch.empty(B, V, dtype=torch.float32, device=dev)
    c, s = api.rope_tables(L.rope_base, D, T)
    cos, sin = torch.from_numpy(c).to(dev), torch.from_numpy(s).to(dev)
    ws = api.workspace(api.stack_decode_workspace_bytes(st, B), dev)
    graph = api.StackDecodeGraph(st, tokens, pos, logits, cos, sin, caches, ws)

    def timed(fn):
        ts = []
        for i in range(warmup + steps):   # the step streams ~36 GB, far more than L2
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            e1.synchronize()
            if i >= warmup:
                ts.append(e0.elapsed_time(e1))
        return float(np.median(ts))

    ms_graph = timed(graph.launch)
    rc = api.device_status()
    assert rc == 0, f"stack decode graph replays: status {rc} {api.timeout_record()}"
    ms_direct = timed(lambda: api.stack_decode(st, tokens, pos, logits, cos, sin, caches, ws))
    rc = api.device_status()
    assert rc == 0, f"stack decode direct calls: status {rc} {api.timeout_record()}"
    w_bytes = sum(t.numel() for w in layers for t in w.values()) * 2
    kv_bytes = wl.n_layers * (int(np.sum(pos_h + 1)) * G * D * 2 * 2)
    total = w_bytes + kv_bytes + V * d * 2
    res = {"workload": wl.name, "us_per_step": round(ms_graph * 1e3, 1),
           "us_per_step_direct_calls": round(ms_direct * 1e3, 1),
           "tokens_per_s": round(B / (ms_graph * 1e-3), 1), "GB_per_step": round(total / 1e9, 2),
           "GBps": round(total / (ms_graph * 1e-3) / 1e9, 1),
           "frac_of_hbm": round(total / (ms_graph * 1e-3) / 1e9 / pk["hbm_gbs"], 4),
           "kernels_per_step": graph.kernel_count}
    graph.close()
    del layers, caches, st, logits, ws, graph
    torch.cuda.empty_cache()
    return res


def prefill_flops(L, B, S):
    M = B * S
    d, H, G, D, I = L.d_model, L.n_heads, L.n_kv_heads, L.head_dim, L.d_inter
    return {
        "qkv_rope_gemm": 2.0 * M * d * (H + 2 * G) * D,
        "attention_prefill": 4.0 * D * H * B * S * (S + 1) / 2,
        "o_proj_residual_gemm": 2.0 * M * H * D * d,
        "gate_up_swiglu_gemm": 2.0 * M * d * 2 * I,
        "down_residual_gemm": 2.0 * M * I * d,
    }


def bench_variants(api, steps, warmup, dev, pk):
    """The layer's variants timed at benchmark sizes (random weights, L2 flushed before each
    step, one event pair per step): a 512-token chunk on top of 3584 cached tokens for 4
    sequences (GQA-8B layer), and the MHA-7B layer with half-split RoPE and with one KV head
    for all 32 query heads."""
    import numpy as np
    import torch
    from llama_decoder_block_gb300 import synth
    g8, m7 = synth.WORKLOADS["gqa8b_bf16_b4_s4096"], synth.WORKLOADS["mha7b_bf16_b1_s2048"]
    cases = [("chunk_gqa8b_b4_s512_after_3584", synth.scaled(g8, S=512, name="chunk"), 3584, 4096),
             ("mha7b_half_split_rope", synth.scaled(m7, rope_style="half", name="half"), None, None),
             ("mqa7b_g1_half_split_rope", synth.scaled(m7, n_kv_heads=1, rope_style="half", name="mqa"), None, None)]
    res = {}
    for name, wl, start, T in cases:
        L = wl.layer
        B, S = wl.B, wl.S
        T = T or S
        g = torch.Generator(device=dev).manual_seed(wl.seed + 7)
        w = dev_weights_random(wl, dev, wl.seed)
        x = torch.randn(B, S, L.d_model, generator=g, device=dev).to(torch.bfloat16)
        out = torch.empty_like(x)
        c, s_ = api.rope_tables(L.rope_base, L.head_dim, T)
        cos, sin = torch.from_numpy(c).to(dev), torch.from_numpy(s_).to(dev)
        kc = torch.randn(B, L.n_kv_heads, T, L.head_dim, generator=g, device=dev).to(torch.bfloat16)
        vc = torch.randn(B, L.n_kv_heads, T, L.head_dim, generator=g, device=dev).to(torch.bfloat16)
        dims = api.Dims(L.d_model, L.n_heads, L.n_kv_heads, L.head_dim, L.d_inter, L.rms_eps, torch.bfloat16,
                        rope_style=1 if L.rope_style == "half" else 0)
        ws = api.workspace(api.prefill_workspace_bytes(dims, B, S), dev)
        st = torch.full((B,), start or 0, dtype=torch.int32, device=dev)
        if start is None:
            fn = lambda: api.layer_prefill(dims, w, x, out, cos, sin, kc, vc, ws)
        else:
            fn = lambda: api.layer_prefill_chunk(dims, w, x, out, cos, sin, st, kc, vc, ws)
        flush = L2Flush(dev)
        for _ in range(warmup):
            flush()
            fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(max(3, steps // 2)):
            flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            e1.synchronize()
            ts.append(e0.elapsed_time(e1))
        assert api.device_status() == 0
        ms = float(np.mean(ts))
        f = prefill_flops(L, B, S)
        p0 = start or 0
        # the chunk's queries see the cache before them: sum over s of (p0 + s + 1) keys
        f["attention_prefill"] = 4.0 * L.head_dim * L.n_heads * B * (S * p0 + S * (S + 1) / 2)
        tf = sum(f.values()) / (ms * 1e-3) / 1e12
        res[name] = {"B": B, "S": S, "cached_before": p0, "H": L.n_heads, "G": L.n_kv_heads,
                     "rope": L.rope_style, "ms_per_step": round(ms, 4),
                     "tokens_per_s": round(B * S / (ms * 1e-3), 1), "tflops": round(tf, 1),
                     "frac_of_burst_peak": round(tf / pk["bf16"], 4),
                     "frac_of_sustained_peak": round(tf / pk["bf16_sustained"], 4)}
        del w, x, out, kc, vc, ws, flush
        torch.cuda.empty_cache()
    return res


def bench_prefill(api, wl, steps, warmup, dev, pk, from_synth):
    import numpy as np
    import torch
    L = wl.layer
    B, S = wl.B, wl.S
    w = dev_weights_from_synth(wl, dev) if from_synth else dev_weights_random(wl, dev, wl.seed)
    if from_synth:
        from llama_decoder_block_gb300 import synth
        x = torch.from_numpy(synth.activations(wl).data.view(np.int16)).to(dev).view(torch.bfloat16)
    else:
        x = torch.randn(B, S, L.d_model, generator=torch.Generator(device=dev).manual_seed(wl.seed + 1),
                        device=dev).to(torch.bfloat16)
    out = torch.empty_like(x)
    c, s = api.rope_tables(L.rope_base, L.head_dim, S)
    cos, sin = torch.from_numpy(c).to(dev), torch.from_numpy(s).to(dev)
    kc = torch.empty(B, L.n_kv_heads, S, L.head_dim, dtype=torch.bfloat16, device=dev)
    vc = torch.empty_like(kc)
    dims = api.Dims(L.d_model, L.n_heads, L.n_kv_heads, L.head_dim, L.d_inter, L.rms_eps, torch.bfloat16)
    ws = api.workspace(api.prefill_workspace_bytes(dims, B, S), dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream()

    def step():
        api.layer_prefill(dims, w, x, out, cos, sin, kc, vc, ws, stream)

    for _ in range(warmup):
        flush()
        step()
    torch.cuda.synchronize()
    assert api.device_status(stream) == 0
    # the timed region: one event pair per step, nothing between the layer's kernels (an event
    # between two kernels would stop the next one from starting under the previous one's tail)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    barrier()
    torch.cuda.synchronize()
    n0 = api.launch_count()
    t0 = time.perf_counter()
    for e0, e1 in evs:
        flush()
        e0.record(stream)
        step()
        e1.record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    launches = api.launch_count() - n0
    barrier()
    assert api.device_status(stream) == 0
    step_ms = np.array([e0.elapsed_time(e1) for e0, e1 in evs])
    # kernel by kernel: the same steps again with the library's per-kernel events
    traces = [api.KernelTrace(len(PREFILL_KERNELS), stream) for _ in range(steps)]
    for tr in traces:
        flush()
        with tr:
            step()
    torch.cuda.synchronize()
    assert api.device_status(stream) == 0
    per_kernel = np.array([tr.kernel_ms() for tr in traces])           # [steps, kernels]
    res = {"ms_per_step": float(step_ms.mean()), "tokens_per_step": B * S, "wall_s": wall, "launches": launches,
           "traced_ms_per_step": float(per_kernel.sum(axis=1).mean()),
           "kernel_ms": {n: float(per_kernel[:, i].mean()) for i, n in enumerate(PREFILL_KERNELS)}}
    flops = prefill_flops(L, B, S)
    res["tflops_total"] = sum(flops.values()) / (res["ms_per_step"] * 1e-3) / 1e12
    dom = max(flops, key=lambda k: res["kernel_ms"][k])
    t = res["kernel_ms"][dom] * 1e-3
    achieved = flops[dom] / t / 1e12
    # the kernel runs inside a sub-millisecond step and the whole timed region lasts well under
    # a second: the burst bf16 peak is its denominator (the sustained one is for seconds-long loops)
    res["roofline"] = {"kernel": dom, "bound": "tensor", "achieved": round(achieved, 1),
                       "peak": pk["bf16"], "unit": "TFLOP/s",
                       "frac": round(achieved / pk["bf16"], 4),
                       "frac_of_sustained_peak": round(achieved / pk["bf16_sustained"], 4),
                       "peak_kind": f"{pk['source']} burst bf16", "flop_per_launch": flops[dom],
                       "traffic": NCU_TRAFFIC.get((dom, src_sha("gemm_tc.cu"))),
                       "traffic_unit": "bytes per launch (ncu dram read+write)"}
    res["kernel_tflops"] = {k: round(v / (res["kernel_ms"][k] * 1e-3) / 1e12, 1) for k, v in flops.items()}

    # end to end through the C ABI, run as a serving loop runs it: every step's input goes up
    # from pinned host memory and its output comes back, each direction on its own copy
    # stream, while the layer of the neighbouring step computes (device input and output
    # double-buffered, ordered by events).  The timed region spans all K steps' uploads, layers and downloads; the
    # weights (404 MB) exceed L2, so no flush runs between these steps.
    xh = torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
    xh.copy_(x.cpu())
    ohs = [torch.empty(out.shape, dtype=out.dtype, pin_memory=True) for _ in range(2)]
    xds = [torch.empty_like(x) for _ in range(2)]
    ods = [torch.empty_like(out) for _ in range(2)]
    up, down = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev = lambda: torch.cuda.Event()
    up_done, layer_done, down_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]

    def pipeline(n):
        for i in range(n):
            k = i % 2
            if i >= 2:
                up.wait_event(layer_done[k])        # the layer two steps back has read xds[k]
            with torch.cuda.stream(up):
                xds[k].copy_(xh, non_blocking=True)
                up_done[k].record(up)
            stream.wait_event(up_done[k])
            if i >= 2:
                stream.wait_event(down_done[k])     # ods[k] went back to the host
            api.layer_prefill(dims, w, xds[k], ods[k], cos, sin, kc, vc, ws, stream)
            layer_done[k].record(stream)
            down.wait_event(layer_done[k])
            with torch.cuda.stream(down):
                ohs[k].copy_(ods[k], non_blocking=True)
                down_done[k].record(down)

    pipeline(warmup)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(up)
    pipeline(steps)
    down.wait_event(down_done[(steps - 1) % 2])
    e1.record(down)
    torch.cuda.synchronize()
    e2e = [e0.elapsed_time(e1) / steps]
    assert torch.equal(ohs[(steps - 1) % 2], out.cpu()), "end-to-end output differs from the device-timed run"
    res["e2e_ms"] = float(np.mean(e2e))
    res["h2d_bytes"] = x.numel() * 2
    res["d2h_bytes"] = out.numel() * 2
    del w, ws, flush, kc, vc
    torch.cuda.empty_cache()
    return res


def bench_decode(api, wl, steps, warmup, dev, pk):
    import numpy as np
    import torch
    from llama_decoder_block_gb300 import synth
    L = wl.layer
    B, T = wl.B, wl.T_max
    w = dev_weights_random(wl, dev, wl.seed)
    g = torch.Generator(device=dev).manual_seed(wl.seed + 2)
    kc = torch.randn(B, L.n_kv_heads, T, L.head_dim, generator=g, device=dev).to(torch.bfloat16)
    vc = torch.randn(B, L.n_kv_heads, T, L.head_dim, generator=g, device=dev).to(torch.bfloat16)
    pos_h = synth.decode_positions(wl)
    pos = torch.from_numpy(pos_h.astype(np.int32)).to(dev)
    x = torch.randn(B, L.d_model, generator=g, device=dev).to(torch.bfloat16)
    out = torch.empty_like(x)
    c, s = api.rope_tables(L.rope_base, L.head_dim, T)
    cos, sin = torch.from_numpy(c).to(dev), torch.from_numpy(s).to(dev)
    dims = api.Dims(L.d_model, L.n_heads, L.n_kv_heads, L.head_dim, L.d_inter, L.rms_eps, torch.bfloat16)
    ws = api.workspace(api.decode_workspace_bytes(dims, B, T), dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream()

    def step():
        api.layer_decode(dims, w, x, out, cos, sin, pos, kc, vc, ws, stream)

    for _ in range(warmup):
        flush()
        step()
    torch.cuda.synchronize()
    assert api.device_status(stream) == 0
    # one event pair per step (kernels overlap their predecessors' tails), then a traced pass
    # for the per-kernel times
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for e0, e1 in evs:
        flush()
        e0.record(stream)
        step()
        e1.record(stream)
    torch.cuda.synchronize()
    assert api.device_status(stream) == 0
    step_ms = np.array([e0.elapsed_time(e1) for e0, e1 in evs])
    traces = [api.KernelTrace(len(DECODE_KERNELS), stream) for _ in range(steps)]
    for tr in traces:
        flush()
        with tr:
            step()
    torch.cuda.synchronize()
    assert api.device_status(stream) == 0
    per_kernel = np.array([tr.kernel_ms() for tr in traces])
    d, H, G, D, I = L.d_model, L.n_heads, L.n_kv_heads, L.head_dim, L.d_inter
    w_bytes = 2 * (d * (H + 2 * G) * D + H * D * d + 3 * d * I + 2 * d)
    kv_read = int(np.sum(pos_h + 1)) * G * D * 2 * 2
    step_bytes = w_bytes + kv_read + B * (H + 2 * G) * D * 2
    us = float(step_ms.mean() * 1e3)
    km = {n: float(per_kernel[:, i].mean()) for i, n in enumerate(DECODE_KERNELS)}
    attn_ms = km["attention_decode_split"]
    attn_gbs = kv_read / (attn_ms * 1e-3) / 1e9
    res = {"workload": wl.name, "us_per_step": round(us, 1), "bytes_per_step": step_bytes,
           "traced_us_per_step": round(float(per_kernel.sum(axis=1).mean() * 1e3), 1),
           "hbm_GBps": round(step_bytes / (us * 1e-6) / 1e9, 1),
           "frac_of_hbm": round(step_bytes / (us * 1e-6) / 1e9 / pk["hbm_gbs"], 4),
           "kernel_us": {k: round(v * 1e3, 1) for k, v in km.items()},
           "attention_roofline": {"bound": "hbm", "achieved": round(attn_gbs, 1), "peak": pk["hbm_gbs"],
                                  "unit": "GB/s", "frac": round(attn_gbs / pk["hbm_gbs"], 4),
                                  "bytes_per_launch": kv_read}}
    del w, kc, vc, ws, flush
    torch.cuda.empty_cache()
    return res


def bench_norm(api, dev, pk, kind, rows=16384, d=4096, reps=20):
    """RMSNorm or LayerNorm alone on [rows, d] bf16, L2 flushed before each run."""
    import torch
    xs = [torch.randn(rows, d, device=dev).to(torch.bfloat16) for _ in range(2)]
    g = torch.ones(d, dtype=torch.bfloat16, device=dev)
    bt = torch.zeros(d, dtype=torch.bfloat16, device=dev)
    y = torch.empty_like(xs[0])
    flush = L2Flush(dev)
    if kind == "rmsnorm":
        fn = lambda x: api.rmsnorm(x, g, y, 1e-5)
    else:
        fn = lambda x: api.layernorm(x, g, bt, y, 1e-5)
    ts = []
    for i in range(reps + 3):
        flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn(xs[i % 2])
        e1.record()
        e1.synchronize()
        if i >= 3:
            ts.append(e0.elapsed_time(e1))
    ms = sorted(ts)[len(ts) // 2]
    gbs = 2 * rows * d * 2 / (ms * 1e-3) / 1e9
    return {"rows": rows, "d": d, "us": round(ms * 1e3, 1), "GBps": round(gbs, 1),
            "frac_of_hbm": round(gbs / pk["hbm_gbs"], 4)}


def bench_case(api, case, wl, steps, warmup, dev, pk):
    """One step alone at the workload's shapes: mean launch time over `steps` launches."""
    import numpy as np
    import torch
    from llama_decoder_block_gb300 import synth
    if case.startswith("decode") and wl.kind != "decode":
        wl = synth.WORKLOADS["decode_gqa8b_bf16_b64_t4096"]
    L = wl.layer
    d, H, G, D, I = L.d_model, L.n_heads, L.n_kv_heads, L.head_dim, L.d_inter
    dims = api.Dims(d, H, G, D, I, L.rms_eps, torch.bfloat16)
    g = torch.Generator(device=dev).manual_seed(7)

    def rnd(*shape, std=1.0):
        return (torch.randn(*shape, generator=g, device=dev) * std).to(torch.bfloat16)

    B, S = wl.B, max(wl.S, 1)
    M = B * S
    if case == "attention":
        q, k, v = rnd(B, H, S, D), rnd(B, G, S, D), rnd(B, G, S, D)
        o = torch.empty(B, S, H * D, dtype=torch.bfloat16, device=dev)
        fn = lambda: api.attention_prefill(dims, q, k, v, o)
        work, unit = 4.0 * D * H * B * S * (S + 1) / 2, "flop"
    elif case == "gate_up":
        # as in the layer: the FFN RMSNorm in the gate/up GEMM's prologue
        x, gm, wg, wu = rnd(M, d), 1 + rnd(d, std=0.1), rnd(I, d, std=0.02), rnd(I, d, std=0.02)
        a = torch.empty(M, I, dtype=torch.bfloat16, device=dev)
        xn, sync = torch.empty_like(x), torch.empty(4, dtype=torch.int32, device=dev)
        fn = lambda: api.norm_linear_swiglu(x, gm, L.rms_eps, wg, wu, a, xn, sync)
        work, unit = 2.0 * M * d * 2 * I, "flop"
    elif case in ("down", "o_proj"):
        K = I if case == "down" else H * D
        a, wd, r = rnd(M, K), rnd(d, K, std=0.02), rnd(M, d)
        out = torch.empty(M, d, dtype=torch.bfloat16, device=dev)
        fn = lambda: api.linear_residual(a, wd, r, out)
        work, unit = 2.0 * M * K * d, "flop"
    elif case == "qkv":
        # as in the layer: the attention RMSNorm in the QKV GEMM's prologue
        x, gm = rnd(B, S, d), 1 + rnd(d, std=0.1)
        wq, wk, wv = rnd(H * D, d, std=0.02), rnd(G * D, d, std=0.02), rnd(G * D, d, std=0.02)
        q = torch.empty(B, H, S, D, dtype=torch.bfloat16, device=dev)
        kc = torch.empty(B, G, S, D, dtype=torch.bfloat16, device=dev)
        vc = torch.empty_like(kc)
        xn, sync = torch.empty_like(x), torch.empty(4, dtype=torch.int32, device=dev)
        c, s = api.rope_tables(L.rope_base, D, S)
        cos, sin = torch.from_numpy(c).to(dev), torch.from_numpy(s).to(dev)
        fn = lambda: api.norm_qkv_rope(dims, x, gm, wq, wk, wv, cos, sin, kc, vc, q, xn, sync)
        work, unit = 2.0 * M * d * (H + 2 * G) * D, "flop"
    elif case in ("decode_attention", "decode_layer"):
        dw = wl
        B, T = dw.B, dw.T_max
        pos_h = synth.decode_positions(dw)
        pos = torch.from_numpy(pos_h).to(dev)
        kc, vc = rnd(B, G, T, D), rnd(B, G, T, D)
        kv = int(np.sum(pos_h + 1)) * G * D * 2 * 2
        if case == "decode_attention":
            q = rnd(B, H, D)
            o = torch.empty(B, H * D, dtype=torch.bfloat16, device=dev)
            ws = api.workspace(api.attention_decode_workspace_bytes(dims, B, T), dev)
            fn = lambda: api.attention_decode(dims, q, kc, vc, pos, o, ws)
            work, unit = kv, "byte"
        else:
            w = dev_weights_random(dw, dev, 3)
            x = rnd(B, d)
            y = torch.empty_like(x)
            c, s = api.rope_tables(L.rope_base, D, T)
            cos, sin = torch.from_numpy(c).to(dev), torch.from_numpy(s).to(dev)
            ws = api.workspace(api.decode_workspace_bytes(dims, B, T), dev)
            fn = lambda: api.layer_decode(dims, w, x, y, cos, sin, pos, kc, vc, ws)
            work, unit = kv + 2 * (d * (H + 2 * G) * D + H * D * d + 3 * d * I), "byte"
    elif case == "layernorm":
        x, gm, bt = rnd(M, d), rnd(d), rnd(d)
        y = torch.empty_like(x)
        fn = lambda: api.layernorm(x, gm, bt, y, L.rms_eps)
        work, unit = 2.0 * M * d * 2, "byte"
    else:   # rmsnorm
        x, gm = rnd(M, d), rnd(d)
        y = torch.empty_like(x)
        fn = lambda: api.rmsnorm(x, gm, y, L.rms_eps)
        work, unit = 2.0 * M * d * 2, "byte"
    flush = L2Flush(dev)
    ts = []
    for i in range(warmup + steps):
        flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        fn()
        e1.record()
        e1.synchronize()
        if i >= warmup:
            ts.append(e0.elapsed_time(e1))
    assert api.device_status() == 0
    ms = float(np.mean(ts))
    rate = work / (ms * 1e-3)
    if unit == "flop":
        return {"case": case, "workload": wl.name, "ms": round(ms, 4), "TFLOPs": round(rate / 1e12, 1),
                "frac_of_burst_bf16": round(rate / 1e12 / pk["bf16"], 4)}
    return {"case": case, "workload": wl.name, "ms": round(ms, 4), "GBps": round(rate / 1e9, 1),
            "frac_of_hbm": round(rate / 1e9 / pk["hbm_gbs"], 4)}


# ------------------------------------------------------------------ the oracle on the host cores

class OracleSample:
    """The fp64 oracle (as it stands) on a causal prefix of a prefill workload, on the host cores."""

    def __init__(self, wl):
        import numpy as np
        import oracle
        from llama_decoder_block_gb300 import synth
        L = wl.layer
        self.wl, self.oracle = wl, oracle
        self.w64 = {k: v.f64() for k, v in synth.layer_weights(wl).items()}
        self.x64 = synth.activations(wl).f64()
        c, s = oracle.rope_tables(L.rope_base, L.head_dim, wl.S)
        self.c, self.s = c.astype(np.float32).astype(np.float64), s.astype(np.float32).astype(np.float64)
        self.kw = dict(n_heads=L.n_heads, n_kv_heads=L.n_kv_heads, head_dim=L.head_dim, rms_eps=L.rms_eps,
                       store_bf16=True)

    def run(self, n):
        t = time.perf_counter()
        self.oracle.decoder_layer(self.x64[:, :n], self.w64, self.c, self.s, **self.kw)
        return time.perf_counter() - t

    def calibrate(self, seconds):
        """Largest power-of-two prefix (128 .. S tokens) whose run takes about `seconds`."""
        n = 128
        dt = self.run(n)
        while dt < seconds / 2 and n < self.wl.S:
            n = min(self.wl.S, n * 2)
            dt = self.run(n)
        return n


def oracle_prefill_sample(wl, target_s=15.0):
    """Times the oracle for about `target_s` seconds; returns (tokens/s, tokens per run, seconds per run)."""
    o = OracleSample(wl)
    n = o.calibrate(target_s / 3)
    total, reps = 0.0, 0
    while total < target_s and reps < 8:
        total += o.run(n)
        reps += 1
    per = total / reps
    return wl.B * n / per, n, per


def oracle_decode_sample(wl, n_seq=8, target_s=10.0):
    """Times the oracle's decode step (one new token per sequence on top of its cache) for the
    first `n_seq` sequences of the decode workload, on the host cores, for about `target_s`
    seconds; returns (seconds per step, the sample's description)."""
    import numpy as np
    import oracle
    from llama_decoder_block_gb300 import synth
    L = wl.layer
    w64 = {k: v.f64() for k, v in synth.layer_weights(wl).items()}
    x = synth.activations(wl).f64()[:n_seq, None, :]
    pos = synth.decode_positions(wl)[:n_seq].astype(np.int64)
    T = int(pos.max()) + 1
    rng = np.random.default_rng(wl.seed)
    pk = rng.standard_normal((n_seq, L.n_kv_heads, T, L.head_dim))
    pv = rng.standard_normal((n_seq, L.n_kv_heads, T, L.head_dim))
    c, s = oracle.rope_tables(L.rope_base, L.head_dim, wl.T_max)
    kw = dict(n_heads=L.n_heads, n_kv_heads=L.n_kv_heads, head_dim=L.head_dim, rms_eps=L.rms_eps, store_bf16=True)
    total, reps = 0.0, 0
    while total < target_s and reps < 8:
        t = time.perf_counter()
        oracle.decoder_layer(x, w64, c, s, past_k=pk, past_v=pv, past_len=pos, **kw)
        total += time.perf_counter() - t
        reps += 1
    per = total / reps
    return per, (f"fp64 numpy oracle, one decode step of the first {n_seq} of the {wl.B} sequences "
                 f"(positions {int(pos.min())}..{int(pos.max())}, caches N(0,1)), {reps} runs of {per:.2f} s")


def cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


# ------------------------------------------------------------------ distributed plumbing

_DIST = {"on": False}


def barrier():
    if _DIST["on"]:
        import torch.distributed as dist
        dist.barrier()


def reduce_max(v: float) -> float:
    """The largest of the ranks' values (every rank gets it); v itself on one process."""
    if not _DIST["on"]:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_value(world: int, tokens_per_step: int, ms_max: float) -> float:
    """Whole-job tokens/s of `world` replicas that each process tokens_per_step per step, timed
    by the slowest rank (ms_max per step)."""
    return world * tokens_per_step / (ms_max * 1e-3)


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    from llama_decoder_block_gb300 import synth
    wl = synth.WORKLOADS[MAIN]
    L = wl.layer
    cfg = {"workload": MAIN, "B": wl.B, "S": wl.S, "d": L.d_model, "H": L.n_heads, "G": L.n_kv_heads,
           "D": L.head_dim, "d_inter": L.d_inter, "layers": 1, "global_batch": wl.B * max(world, 1),
           "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
           "l2": "flushed between timed steps (256 MiB write, then 256 MiB read); weights 404 MB > L2"}

    if args.impl == "reference":
        if rank != 0:
            return
        # each step: the oracle on a causal prefix sized so that W + K steps take a few minutes
        o = OracleSample(wl)
        n = o.calibrate(max(1.0, min(10.0, 150.0 / max(1, args.steps + args.warmup))))
        for _ in range(args.warmup):
            o.run(n)
        total = sum(o.run(n) for _ in range(args.steps))
        per = total / max(1, args.steps)
        tps = wl.B * n / per
        line = {"impl": "reference", "metric": METRIC, "value": round(tps, 2), "unit": "tokens/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(per * 1e3, 1),
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": cfg,
                "cpu_baseline": {"value": round(tps, 2), "unit": "tokens/s", "cores": cores(), "kind": "oracle",
                                 "sample": f"fp64 numpy oracle, one layer, first {n} tokens of the B=1 S=2048 "
                                           "prefill (exact causal prefix), bf16 storage points"},
                "e2e": {"value": round(tps, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    import torch
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        _DIST["on"] = True
    else:
        torch.cuda.set_device(0)
    dev = torch.device("cuda", local if world > 1 else 0)
    import __graft_entry__
    __graft_entry__.build()
    from llama_decoder_block_gb300 import api
    pk = peaks()
    if args.case:
        print(json.dumps(bench_case(api, args.case, synth.WORKLOADS[args.workload], args.steps, args.warmup, dev, pk)))
        return

    with Clocks(dev.index) as clk:
        main_res = bench_prefill(api, wl, args.steps, args.warmup, dev, pk, from_synth=True)
    ms = reduce_max(main_res["ms_per_step"])
    e2e_ms = reduce_max(main_res["e2e_ms"])
    value = replica_value(world, main_res["tokens_per_step"], ms)
    line = {"metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded PCG64: x ~ N(0,1), W ~ N(0,0.02), gamma ~ 1+N(0,0.1))",
            "config": cfg, "roofline": main_res["roofline"],
            "e2e": {"value": round(replica_value(world, main_res["tokens_per_step"], e2e_ms), 1), "unit": "tokens/s",
                    "h2d_bytes_per_step": main_res["h2d_bytes"], "d2h_bytes_per_step": main_res["d2h_bytes"]},
            "gpu_launches": main_res["launches"], "clocks": clk.summary(),
            "prefill_tflops": round(main_res["tflops_total"], 1),
            "prefill_frac_of_burst_peak": round(main_res["tflops_total"] / pk["bf16"], 4),
            "kernel_ms": {k: round(v, 4) for k, v in main_res["kernel_ms"].items()},
            "kernel_tflops": main_res["kernel_tflops"]}
    if not args.no_extra:
        torch.cuda.empty_cache()
        line["decode"] = bench_decode(api, synth.WORKLOADS["decode_gqa8b_bf16_b64_t4096"], max(10, args.steps // 2),
                                      args.warmup, dev, pk)
        g8 = synth.WORKLOADS["gqa8b_bf16_b4_s4096"]
        r8 = bench_prefill(api, g8, max(5, args.steps // 4), args.warmup, dev, pk, from_synth=False)
        line["gqa8b_prefill"] = {"workload": g8.name, "tokens_per_s": round(g8.B * g8.S / (r8["ms_per_step"] * 1e-3), 1),
                                 "ms_per_step": round(r8["ms_per_step"], 3), "tflops": round(r8["tflops_total"], 1),
                                 "frac_of_burst_peak": round(r8["tflops_total"] / pk["bf16"], 4),
                                 "frac_of_sustained_peak": round(r8["tflops_total"] / pk["bf16_sustained"], 4),
                                 "kernel_ms": {k: round(v, 3) for k, v in r8["kernel_ms"].items()},
                                 "kernel_tflops": r8["kernel_tflops"]}
        line["variants"] = bench_variants(api, args.steps, args.warmup, dev, pk)
        line["rmsnorm"] = bench_norm(api, dev, pk, "rmsnorm")
        line["layernorm"] = bench_norm(api, dev, pk, "layernorm")
        line["layernorm"]["time_vs_rmsnorm"] = round(line["layernorm"]["us"] / line["rmsnorm"]["us"], 3)
        line["stack32_forward"] = bench_stack(api, synth.WORKLOADS["stack32_gqa8b_bf16_s8192_v32000"], 3, 2, dev, pk)
        line["stack32_decode"] = bench_stack_decode(api, synth.WORKLOADS["stack32_decode_gqa8b_bf16_b64_t4096_v32000"],
                                                    max(10, args.steps // 2), args.warmup, dev, pk)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tps, n, per = oracle_prefill_sample(wl)
        line["cpu_baseline"] = {"value": round(tps, 2), "unit": "tokens/s", "cores": cores(), "kind": "oracle",
                                "sample": f"fp64 numpy oracle, one layer, first {n} tokens of the B=1 S=2048 prefill "
                                          f"(exact causal prefix), {per:.1f} s per run"}
        if "decode" in line:
            dwl = synth.WORKLOADS["decode_gqa8b_bf16_b64_t4096"]
            per_d, sample = oracle_decode_sample(dwl)
            n = int(sample.split("first ")[1].split(" ")[0])
            line["decode"]["cpu_baseline"] = {"value": round(per_d * 1e6, 1), "unit": "us per step of the sample",
                                              "us_per_sequence": round(per_d * 1e6 / n, 1), "cores": cores(),
                                              "kind": "oracle", "sample": sample}
    if rank == 0:
        print(json.dumps(line))
    if _DIST["on"]:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

#!/usr/bin/env python
"""Throughput of the Compass-style decoder path on GB300, one JSON line on stdout.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

A step is one whole pass of the path over one batch of synthetic input: the layer stack
and the tied head. `value` is prefill tokens/s on the 28-layer stack (3:1 sliding:full,
bf16, T = 8192 with three 32x32 images, deepstack adds after layers 0-2, head on the last
token over a 256000 vocabulary); `--prefill-workload pair|varlen` selects the two-layer
pair (T = 2048) or the varlen packed prefill (T = 32768) instead. Extra keys carry the
two-layer pair, the single fp32 layer (T = 128, a latency in microseconds) and the batched
decode step (64 sequences x 4096 cached tokens, paged KV, head on all 64 rows), each with
its kernels against their rooflines. Inputs are resident in HBM when the timed region
starts; every step reads several GB of weights (more than the 129 MB L2), so no flush is
needed. `e2e` repeats the prefill measurement with host buffers: the step's inputs are
copied from pinned host memory and its logits copied back inside the timed region.

Under torchrun (N > 1) every rank runs an independent replica on its own GPU (the path
does not shard within a step); value = tokens of all ranks / max time over ranks.
`--impl reference` times the CPU oracle (fp64 NumPy) on a stated sample of the same
workload as the reference arm.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "prefill tokens/s and decode tokens/s (1 GB300) + % of bf16 tensor / HBM roofline"
PREFILL_WORKLOADS = {"stack28": "stack28_T8192", "pair": "pair_T2048", "varlen": "varlen_T32768"}
_SHAPES = ("hidden 2048, 16/4 heads, head_dim 128, SwiGLU 8192, interleaved MRoPE [24,20,20], "
           "theta 50000")
PREFILL_DESC = {
    "stack28": ("28-layer prefill stack (3:1 sliding:full, full NoPE at every 4th layer), bf16, "
                "batch 1, seq 8192, " + _SHAPES + ", window 4096, three 32x32 images, deepstack "
                "[3072,2048] after layers 0-2, tied head on the last token, vocab 256000, "
                "logit_scale 0.0625"),
    "pair": ("two-layer pair (sliding+interleaved MRoPE, full NoPE), bf16, batch 1, seq 2048, "
             + _SHAPES + ", window 512, one 16x16 image at token 300, deepstack [256,2048] "
             "after layer 0, tied head on the last token, vocab 256000"),
    "varlen": ("two-layer pair, varlen packed prefill of 4096/8192/12288/8192 tokens (T = 32768), "
               + _SHAPES + ", window 4096, 1-4 images per sequence, deepstack after layers "
               "0-1, head on the last token of each sequence"),
}
DECODE_DESC = ("decode step on the two-layer pair: 64 sequences x 4096 cached bf16 tokens in "
               "16-token pages (permuted page table), window 4096, head on all 64 rows")
# tokens of the oracle's sample (the first tokens of the workload's sequence, every layer and
# the head): sized for roughly 5-15 s of fp64 work per pass on the GPU machine's host cores
CPU_SAMPLE_TOKENS = {"stack28": 512, "pair": 2048, "varlen": 2048}


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--no-decode", action="store_true")
    p.add_argument("--no-prefill", action="store_true", help="decode leg only (profiling)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-q4", action="store_true", help="skip the 4-bit weight decode timing")
    p.add_argument("--cpu-tokens", type=int, default=0,
                   help="oracle sample: first N tokens of the prefill workload (0: the default "
                        "sample of the workload)")
    p.add_argument("--prefill-workload", choices=["stack28", "pair", "varlen"], default="stack28",
                   help="prefill workload: stack28 = 28-layer stack T=8192 (the headline), "
                        "pair = two-layer pair T=2048, varlen = varlen packed T=32768")
    p.add_argument("--layers", type=int, default=0,
                   help="profiling only: keep the first N layers of the workload (0: all)")
    p.add_argument("--no-context", action="store_true",
                   help="skip the extra workloads (two-layer pair, fp32 layer)")
    return p.parse_args()


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sus=d["bf16_tflops_sustained"],
                    src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sus=1700.0, src="fallback")


# ------------------------------------------------------------------------------ traffic
# DRAM bytes per launch of a kernel on a workload, from an ncu capture, kept in
# profiles/traffic.json under "<kernel>@<workload>" with a hash of the sources the kernel is
# built from; reported only while those sources are unchanged since the capture.
KERNEL_SOURCES = {
    "gemm_qkv_mlp": ["gemm.cu", "ptx.cuh", "kernels.h", "common.h"],
    "attn_decode": ["decode.cu", "ptx.cuh", "kernels.h", "common.h"],
}


def sources_sha256(kernel):
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "cohere_compass_decoder_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def measured_traffic(kernel, workload):
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path) or kernel not in KERNEL_SOURCES:
        return None
    with open(path) as f:
        rec = json.load(f).get(f"{kernel}@{workload}")
    if not rec or rec.get("sources_sha256") != sources_sha256(kernel):
        return None
    return rec["dram_bytes_per_launch"]


# ------------------------------------------------------------------------------ dist
class Dist:
    def __init__(self, n):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            backend = "nccl" if _cuda() else "gloo"
            dist.init_process_group(backend)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x):
        if not self.pg:
            return x
        import torch
        t = torch.tensor([x], dtype=torch.float64, device="cuda" if _cuda() else "cpu")
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


def _cuda():
    import torch
    return torch.cuda.is_available()


# ------------------------------------------------------------------------------ clocks
class Clocks:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.gpu = gpu_index
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [r.split(", ") for r in out.strip().splitlines() if r.count(",") >= 8]
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].strip() == "Active"})
        busy = [s for s in sm if s > 0.5 * (max(mx) if mx else 1)] or sm
        return {"sm_mhz": statistics.median(busy) if busy else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------------------ timing
def time_steps(fn, steps, warmup, dist, stream):
    """W untimed steps, then exactly K steps bracketed by barrier + synchronize; CUDA
    events on the launching stream; returns the max over ranks in ms."""
    import torch
    for i in range(warmup):
        fn(i)
    torch.cuda.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for k in range(steps):
        fn(warmup + k)
    t1.record(stream)
    torch.cuda.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    return dist.max(t0.elapsed_time(t1))


def kernel_profile(gw, fn, steps, base):
    """Per kernel class: launches and mean device time per launch, from the library's
    CUDA-event records over `steps` further steps."""
    import torch
    import cohere_compass_decoder_gb300._lib as L
    L.cc_profile_read(gw.stack.plan)
    L.cc_profile_enable(gw.stack.plan, True)
    for k in range(steps):
        fn(base + k)
    torch.cuda.synchronize()
    prof = L.cc_profile_read(gw.stack.plan)
    L.cc_profile_enable(gw.stack.plan, False)
    total = sum(ms for _, ms in prof.values()) or 1.0
    out = {}
    for name, (n, ms) in prof.items():
        if n:
            out[name] = {"launches_per_step": n / steps, "avg_us": 1000.0 * ms / n,
                         "share": ms / total}
    return out


# ------------------------------------------------------------------------------ legs
def make_workload(key, layers=0):
    """The named prefill workload, optionally cut to its first `layers` layers (profiling)."""
    import dataclasses
    from synth.configs import WORKLOADS
    wl = WORKLOADS[PREFILL_WORKLOADS[key]]()
    if layers and layers < wl.shape.num_layers:
        shape = dataclasses.replace(wl.shape, num_layers=layers,
                                    layer_types=wl.shape.layer_types[:layers])
        wl = dataclasses.replace(wl, shape=shape, n_deepstack=min(wl.n_deepstack, layers))
    return wl


def weight_bytes(shape):
    """Bytes of the layer weights and of the tied head that one prefill step reads."""
    H, d, I = shape.hidden_size, shape.head_dim, shape.intermediate_size
    N1 = (shape.num_attention_heads + 2 * shape.num_key_value_heads) * d + 2 * I
    K2 = shape.num_attention_heads * d + I
    return shape.num_layers * (N1 * H + H * K2) * 2, shape.vocab_size * H * 2


def prefill_leg(args, dist, pk, key, context=False):
    """The prefill + head of workload `key`: K timed steps, then the per-kernel profile.
    context=True: a shorter run for the extra keys (no e2e, no next rows)."""
    import torch
    from synth import Inputs
    from cohere_compass_decoder_gb300.workload import GpuWorkload

    wl = make_workload(key, 0 if context else args.layers)
    inp = Inputs(wl)
    gw = GpuWorkload(inp)
    stream = torch.cuda.current_stream()
    K, W = args.steps, args.warmup
    n_prof = max(3, min(K, 10))
    pool = [gw.fresh_hidden() for _ in range(K + W + n_prof)]
    logits = torch.empty(len(inp.head_rows), inp.shape.vocab_size, device="cuda")

    def step(i):
        gw.step(pool[i], logits)

    ms = time_steps(step, K, W, dist, stream)
    gw.sync()
    kern = kernel_profile(gw, step, n_prof, K + W)
    T = inp.wl.total_tokens
    s = inp.shape
    N1 = (s.num_attention_heads + 2 * s.num_key_value_heads) * s.head_dim + 2 * s.intermediate_size
    g1 = kern.get("gemm_qkv_mlp", {})
    flops = 2.0 * T * N1 * s.hidden_size
    ach = flops / (g1["avg_us"] * 1e-6) / 1e12 if g1 else None
    roof = {"kernel": "gemm_qkv_mlp", "bound": "tensor", "achieved": ach, "peak": pk["bf16"],
            "unit": "TFLOP/s", "frac": (ach / pk["bf16"]) if ach else None,
            "frac_of_sustained": (ach / pk["bf16_sus"]) if ach else None,
            "traffic": None if args.layers else measured_traffic("gemm_qkv_mlp", wl.name),
            "peak_source": f"bf16 burst (of {pk['src']}); frac_of_sustained: against the "
                           f"sustained {pk['bf16_sus']} TFLOP/s (of {pk['src']})",
            "algorithmic_per_launch": f"2*T*N1*H = {flops:.4g} FLOP"}
    if g1:
        g1["tflops"] = ach
        g1["frac_of_bf16_peak"] = ach / pk["bf16"]
        g1["frac_of_sustained"] = ach / pk["bf16_sus"]
    # other classes against their own roofs
    g2 = kern.get("gemm_out_resid")
    if g2:
        K2 = s.num_attention_heads * s.head_dim + s.intermediate_size
        f2 = 2.0 * T * s.hidden_size * K2
        g2["tflops"] = f2 / (g2["avg_us"] * 1e-6) / 1e12
        g2["frac_of_bf16_peak"] = g2["tflops"] / pk["bf16"]
        g2["frac_of_sustained"] = g2["tflops"] / pk["bf16_sus"]
    at = kern.get("attn_prefill")
    if at:
        fa = attn_flops(inp) / at["launches_per_step"]
        at["tflops"] = fa / (at["avg_us"] * 1e-6) / 1e12
        at["frac_of_bf16_peak"] = at["tflops"] / pk["bf16"]
        at["frac_of_sustained"] = at["tflops"] / pk["bf16_sus"]
    gh = kern.get("gemm_head")
    if gh:
        hb = s.vocab_size * s.hidden_size * 2 + len(inp.head_rows) * s.vocab_size * 4
        gh["gbs"] = hb / (gh["avg_us"] * 1e-6) / 1e9
        gh["frac_of_hbm"] = gh["gbs"] / pk["hbm"]
    value = T * K * dist.world / (ms / 1e3)
    launches = sum(v["launches_per_step"] for v in kern.values())
    extra = kern.get("row_maps", {}).get("launches_per_step", 0) and 1  # ds map: fill + scatter
    res = dict(ms=ms, value=value, kernels=kern, roofline=roof,
               launches=int(round((launches + extra) * K)), tokens=T,
               batch=len(inp.wl.seq_lens), workload=wl.name, shape=s)
    if s.dtype == "bf16" and context:
        res["next_rows"] = {"embed_merge_ln": embed_merge_timing(inp, gw, pk)}
        if key == "pair":
            res["next_rows"]["chunked_prefill"] = chunked_prefill_timing(inp, gw, pk)
    # e2e through host buffers
    if not args.no_e2e and not context:
        res["e2e"] = prefill_e2e(gw, inp, K, W, dist, stream)
    gw.close()
    return res


def fp32_layer_latency(args):
    """The single fp32 layer (T = 128) and its head, a latency: microseconds per step with
    CUDA events over the timed steps (inputs resident)."""
    import torch
    from synth import Inputs
    from synth.configs import layer_fp32_T128
    from cohere_compass_decoder_gb300.workload import GpuWorkload
    inp = Inputs(layer_fp32_T128())
    gw = GpuWorkload(inp)
    steps, warm = max(args.steps, 20), max(args.warmup, 3)
    pool = [gw.fresh_hidden() for _ in range(steps + warm)]
    logits = torch.empty(len(inp.head_rows), inp.shape.vocab_size, device="cuda")
    for i in range(warm):
        gw.step(pool[i], logits)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(steps):
        gw.step(pool[warm + i], logits)
    e1.record()
    torch.cuda.synchronize()
    gw.sync()
    gw.close()
    us = 1000.0 * e0.elapsed_time(e1) / steps
    return {"workload": "single sliding layer, fp32, batch 1, seq 128, hidden 256, 4/1 heads, "
                        "head_dim 64, SwiGLU 512, window 32, MRoPE [12,10,10], head over 1024 "
                        "rows x 128 tokens",
            "us_per_step": us, "tokens_per_s": 128 / (us * 1e-6), "steps": steps,
            "note": "a latency: the layer stack and head launched back to back, CUDA events"}


def embed_merge_timing(inp, gw, pk, iters=20):
    """The step before the path (embedding lookup + image-row merge fused with layer 0's
    LayerNorm) through its C-ABI op on the workload's token ids, timed with CUDA events."""
    import numpy as np
    import torch
    import cohere_compass_decoder_gb300._lib as L
    s = inp.shape
    T, H, V = inp.wl.total_tokens, s.hidden_size, s.vocab_size
    tok = torch.from_numpy(inp.token_ids).cuda()
    rows = torch.from_numpy(inp.mm_rows.astype(np.int32)).cuda()
    from cohere_compass_decoder_gb300.model import to_device
    feats = to_device(inp.mm_embeds)
    R = int(rows.numel())
    h = torch.empty(T, H, dtype=torch.float32, device="cuda")
    a = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    st = gw.stack

    def run():
        L.cc_op_embed_merge(tok, T, st.embed, V, H, rows if R else None, feats if R else None, R,
                            h, st.ln[0], s.layer_norm_eps, a)
    for _ in range(3):
        run()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(iters):
        run()
    e1.record()
    torch.cuda.synchronize()
    L.cc_op_sync()
    op_us = e0.elapsed_time(e1) * 1000.0 / iters
    # the fused kernel alone, as the token-input prefill launches it (library CUDA events)
    L.cc_profile_read(st.plan)
    L.cc_profile_enable(st.plan, True)
    for _ in range(3):
        st.prefill_tokens(tok, rows if R else None, feats if R else None, h, gw.pos, gw.cu,
                          gw.n_seqs, gw.ds_rows, gw.ds_feats)
    torch.cuda.synchronize()
    prof = L.cc_profile_read(st.plan)
    L.cc_profile_enable(st.plan, False)
    n, ms = prof["embed_merge"]
    us = 1000.0 * ms / max(n, 1)
    nbytes = T * H * 2 + T * 4 + R * 4 + H * 2 + T * H * 4 + T * H * 2
    gbs = nbytes / (us * 1e-6) / 1e9
    return {"avg_us": us, "bytes": nbytes, "gbs": gbs, "frac_of_hbm": gbs / pk["hbm"],
            "op_us": op_us,
            "note": "embedding lookup + image-row merge fused with layer 0's LayerNorm; avg_us: "
                    "the kernel in cc_prefill_forward_tokens; op_us: cc_op_embed_merge (row map "
                    "and scratch allocation included)"}


def chunked_prefill_timing(inp, gw, pk, steps=10):
    """Chunked prefill (the handoff step): the workload's tokens as a second chunk that
    continues a cached prefix of the same length, attention over the paged cache."""
    import numpy as np
    import torch
    import cohere_compass_decoder_gb300._lib as L
    s = inp.shape
    T = inp.wl.total_tokens
    if len(inp.wl.seq_lens) != 1:
        return None
    spans = [(i.seq, i.start, i.grid_t, i.grid_h, i.grid_w) for i in inp.images]
    pos2, _ = L.cc_build_mrope_positions(spans, [2 * T])
    pos_a = torch.tensor(np.ascontiguousarray(np.asarray(pos2)[:, :T]), dtype=torch.int32,
                         device="cuda")
    pos_b = torch.tensor(np.ascontiguousarray(np.asarray(pos2)[:, T:]), dtype=torch.int32,
                         device="cuda")
    ps = 16
    max_pages = (2 * T + ps - 1) // ps
    table = torch.arange(max_pages, dtype=torch.int32, device="cuda").view(1, -1)
    kp = [torch.zeros(max_pages, s.num_key_value_heads, ps, s.head_dim, dtype=torch.bfloat16,
                      device="cuda") for _ in range(s.num_layers)]
    vp = [torch.zeros_like(t) for t in kp]
    kv = L.make_kv_pool(kp, vp, max_pages)
    st = gw.stack
    cu = gw.cu
    h = gw.fresh_hidden()
    L.cc_prefill_forward(st.plan, h, pos_a, cu, 1, T, gw.ds_rows,
                         0 if gw.ds_rows is None else int(gw.ds_rows.numel()), gw.ds_feats, kv,
                         table, max_pages)
    prefix = torch.tensor([T], dtype=torch.int32, device="cuda")
    pool = [gw.fresh_hidden() for _ in range(steps + 3)]

    def run(i):
        L.cc_prefill_forward_chunk(st.plan, pool[i], pos_b, cu, 1, T, prefix, kv, table,
                                   max_pages)
    for i in range(3):
        run(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(steps):
        run(3 + i)
    e1.record()
    torch.cuda.synchronize()
    L.cc_sync(st.plan)
    ms = e0.elapsed_time(e1) / steps
    # attention of the chunk: query T + i sees T + i + 1 keys (full) or min(., window)
    i = np.arange(T, 2 * T)
    vis = 0
    for lt in s.layer_types:
        vis += int((i + 1).sum() if lt != "sliding_attention" else np.minimum(i + 1, s.sliding_window).sum())
    flops = 4.0 * s.head_dim * s.num_attention_heads * vis
    return {"chunk_tokens": T, "prefix_tokens": T, "ms_per_chunk": ms,
            "tokens_per_s": T / (ms / 1e3), "attn_gflop_per_chunk": flops / 1e9,
            "note": "cc_prefill_forward_chunk: the layer stack over a 2048-token chunk that "
                    "continues a 2048-token prefix in the paged cache (no head)"}


def attn_flops(inp):
    """4 * d * n_q * (visible keys summed over queries) over all layers of the workload."""
    s = inp.shape
    total = 0
    for lt in s.layer_types:
        W = s.sliding_window if lt == "sliding_attention" else None
        for L in inp.wl.seq_lens:
            i = __import__("numpy").arange(L)
            vis = i + 1 if W is None else __import__("numpy").minimum(i + 1, W)
            total += int(vis.sum())
    return 4.0 * s.head_dim * s.num_attention_heads * total


def prefill_e2e(gw, inp, K, W, dist, stream):
    """The prefill through host buffers, as a serving loop runs it: every step copies its
    inputs from pinned host memory and reads its logits back, inside the timed region. The
    copies run on a second stream into two alternating input sets, so step i + 1's upload and
    step i's read-back overlap step i's compute; the timed region ends when the last logits
    are on the host."""
    import torch
    host_h = torch.from_numpy(inp.hidden).pin_memory()
    host_pos = gw.pos.cpu().pin_memory()
    host_cu = gw.cu.cpu().pin_memory()
    host_rows = gw.ds_rows.cpu().pin_memory() if gw.ds_rows is not None else None
    host_ds = [f.cpu().pin_memory() for f in gw.ds_feats]
    n_rows = len(inp.head_rows)
    n_out = n_rows * inp.shape.vocab_size
    host_out = [torch.empty(n_out, dtype=torch.float32).pin_memory() for _ in range(2)]
    sets = [dict(h=torch.empty_like(gw.hidden0), pos=torch.empty_like(gw.pos),
                 cu=torch.empty_like(gw.cu),
                 rows=torch.empty_like(gw.ds_rows) if gw.ds_rows is not None else None,
                 ds=[torch.empty_like(f) for f in gw.ds_feats],
                 logits=torch.empty(n_rows, inp.shape.vocab_size, device="cuda"))
            for _ in range(2)]
    copy = torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]     # set b's inputs are on the device
    ev_done = [torch.cuda.Event() for _ in range(2)]   # the step that used set b has finished
    ev_out = [torch.cuda.Event() for _ in range(2)]    # set b's logits are on the host
    bi = (host_h.numel() * 4 + host_pos.numel() * 4 + host_cu.numel() * 4
          + (host_rows.numel() * 4 if host_rows is not None else 0)
          + sum(f.numel() * f.element_size() for f in host_ds))
    bo = n_out * 4

    def upload(b):
        st = sets[b]
        with torch.cuda.stream(copy):
            copy.wait_event(ev_done[b])
            st["h"].copy_(host_h, non_blocking=True)
            st["pos"].copy_(host_pos, non_blocking=True)
            st["cu"].copy_(host_cu, non_blocking=True)
            if host_rows is not None:
                st["rows"].copy_(host_rows, non_blocking=True)
            for d, h in zip(st["ds"], host_ds):
                d.copy_(h, non_blocking=True)
            ev_in[b].record(copy)

    def run(n, start_event=None):
        if start_event is not None:
            copy.wait_event(start_event)
        upload(0)
        for i in range(n):
            b = i & 1
            if i + 1 < n:
                upload(1 - b)
            st = sets[b]
            stream.wait_event(ev_in[b])
            stream.wait_event(ev_out[b])             # the previous read-back of this set
            gw.stack.prefill(st["h"], st["pos"], st["cu"], gw.n_seqs, st["rows"], st["ds"])
            gw.logits(st["h"], st["logits"])
            ev_done[b].record(stream)
            with torch.cuda.stream(copy):
                copy.wait_event(ev_done[b])
                host_out[b].copy_(st["logits"].view(-1), non_blocking=True)
                ev_out[b].record(copy)
        stream.wait_event(ev_out[(n - 1) & 1])

    for b in range(2):                              # all events recorded once
        ev_done[b].record(stream)
        ev_out[b].record(stream)
    run(W)
    torch.cuda.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    run(K, t0)
    t1.record(stream)
    torch.cuda.synchronize()
    dist.barrier()
    torch.cuda.synchronize()
    ms = dist.max(t0.elapsed_time(t1))
    T = inp.wl.total_tokens
    return {"value": T * K * dist.world / (ms / 1e3), "unit": "tokens/s", "ms_per_step": ms / K,
            "h2d_bytes_per_step": int(bi), "d2h_bytes_per_step": int(bo),
            "overlap": "uploads and read-backs on a second stream, two alternating input sets"}


def decode_leg(args, dist, pk):
    import torch
    from synth import Inputs
    from synth.configs import decode_B64_cache4096
    from cohere_compass_decoder_gb300.workload import GpuWorkload

    inp = Inputs(decode_B64_cache4096())
    gw = GpuWorkload(inp)
    stream = torch.cuda.current_stream()
    K, W = args.steps, args.warmup
    n_prof = max(3, min(K, 10))
    pool = [gw.fresh_hidden() for _ in range(K + W + n_prof)]
    logits = torch.empty(len(inp.head_rows), inp.shape.vocab_size, device="cuda")

    def step(i):
        gw.step(pool[i], logits)

    ms = time_steps(step, K, W, dist, stream)
    gw.sync()
    kern = kernel_profile(gw, step, n_prof, K + W)
    s = inp.shape
    B = inp.wl.decode_batch
    n = inp.wl.cache_len + 1
    kv_bytes = 0
    for lt in s.layer_types:
        keys = min(n, s.sliding_window) if lt == "sliding_attention" else n
        kv_bytes += B * keys * s.num_key_value_heads * s.head_dim * 2 * 2
    ad = kern.get("attn_decode")
    per_launch = kv_bytes / len(s.layer_types)
    ach = per_launch / (ad["avg_us"] * 1e-6) / 1e9 if ad else None
    roof = {"kernel": "attn_decode", "bound": "hbm", "achieved": ach, "peak": pk["hbm"],
            "unit": "GB/s", "frac": (ach / pk["hbm"]) if ach else None,
            "traffic": measured_traffic("attn_decode", inp.wl.name),
            "peak_source": f"HBM copy (of {pk['src']})",
            "algorithmic_per_launch": f"K+V of the visible keys, {per_launch:.4g} B"}
    gh = kern.get("gemm_head")
    if gh:
        hb = s.vocab_size * s.hidden_size * 2 + B * s.vocab_size * 4
        gh["gbs"] = hb / (gh["avg_us"] * 1e-6) / 1e9
        gh["frac_of_hbm"] = gh["gbs"] / pk["hbm"]
    value = B * K * dist.world / (ms / 1e3)
    launches = sum(v["launches_per_step"] for v in kern.values())
    launches += kern.get("attn_decode", {}).get("launches_per_step", 0)  # + split combine
    res = dict(ms=ms, value=value, kernels=kern, roofline=roof, launches=int(round(launches * K)))
    res["next_rows"] = {"decode_graph": decode_graph_timing(gw, inp, steps=max(K, 10))}
    if not args.no_q4:
        res["next_rows"]["decode_q4"] = decode_q4_timing(inp, gw, pk)
    gw.close()
    return res


def decode_graph_timing(gw, inp, steps=20):
    """The decode step + head captured once into a CUDA graph (the hidden-state reset
    included) and replayed, against the same work launched eagerly: what a serving loop that
    replays one graph per step saves in launch overhead."""
    import torch
    n = int(gw.head_rows.numel())
    h = gw.fresh_hidden()
    lg = torch.empty(n, inp.shape.vocab_size, dtype=torch.float32, device="cuda")

    def once():
        h.copy_(gw.hidden0)
        gw.step(h, lg)
    once()                                   # sizes the plan's scratch before capture
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        once()
    torch.cuda.current_stream().wait_stream(side)

    def timed(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(steps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / steps
    eager = timed(once)
    graph = timed(g.replay)
    gw.sync()
    B = inp.wl.decode_batch
    return {"ms_per_step_graph": graph, "ms_per_step_eager": eager,
            "tokens_per_s_graph": B / (graph / 1e3),
            "note": "cc_decode_step + cc_logits (and the hidden-state reset) captured in one CUDA "
                    "graph and replayed, against the same calls launched eagerly"}


def decode_q4_timing(inp, gw, pk, steps=10):
    """The decode step + head on 4-bit affine weights (group 64): the same workload and
    cache, weights streamed at a quarter of their bf16 bytes; per GEMM class the weight
    stream's bandwidth against the HBM roof."""
    import torch
    import cohere_compass_decoder_gb300._lib as L
    s = inp.shape
    st = gw.stack
    st.attach_q4(inp.layer_q4, inp.embed_q4)
    B = inp.wl.decode_batch
    n = int(gw.head_rows.numel())
    lg = torch.empty(n, s.vocab_size, dtype=torch.float32, device="cuda")
    pool = [gw.fresh_hidden() for _ in range(steps + 3)]

    def run(i):
        st.decode_q4(pool[i], gw.pos, gw.seq_lens, gw.page_table, gw.max_pages, gw.kv)
        st.logits_q4(pool[i], gw.head_rows, n, lg)
    for i in range(3):
        run(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(steps):
        run(3 + i)
    e1.record()
    torch.cuda.synchronize()
    st.sync()
    ms = e0.elapsed_time(e1) / steps
    for i in range(steps):
        pool[3 + i].copy_(gw.hidden0)
    L.cc_profile_read(st.plan)
    L.cc_profile_enable(st.plan, True)
    for i in range(steps):
        run(3 + i)
    torch.cuda.synchronize()
    prof = L.cc_profile_read(st.plan)
    L.cc_profile_enable(st.plan, False)
    H, V = s.hidden_size, s.vocab_size
    N1 = (s.num_attention_heads + 2 * s.num_key_value_heads) * s.head_dim + 2 * s.intermediate_size
    K2 = s.num_attention_heads * s.head_dim + s.intermediate_size

    def wbytes(N, K):       # packed words + (scale, bias) words
        return N * K // 2 + N * (K // 64) * 4
    per = {"gemm_qkv_mlp": wbytes(N1, H), "gemm_out_resid": wbytes(H, K2),
           "gemm_head": wbytes(V, H)}
    out = {}
    for name, nb in per.items():
        cnt, tot = prof.get(name, (0, 0.0))
        if cnt:
            us = 1000.0 * tot / cnt
            out[name] = {"avg_us": us, "weight_bytes": nb, "gbs": nb / (us * 1e-6) / 1e9,
                         "frac_of_hbm": nb / (us * 1e-6) / 1e9 / pk["hbm"]}
    return {"ms_per_step": ms, "tokens_per_s": B / (ms / 1e3), "kernels": out,
            "note": "cc_decode_step_q4 + cc_logits_q4 on the decode workload (64 sequences, "
                    "4096 cached tokens each); gbs counts the 4-bit weight stream only"}


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def cpu_sample(key, tokens=0):
    """The oracle's sample of prefill workload `key`: its first `tokens` tokens (0: the
    default sample size) through every layer and the head. Causal attention makes these rows
    of the stack identical to the same rows of the whole prefill; images are kept when they
    lie wholly inside the sample."""
    import dataclasses
    wl = make_workload(key)
    tokens = tokens or CPU_SAMPLE_TOKENS[key]
    if len(wl.seq_lens) > 1 or tokens >= wl.total_tokens:
        return wl, f"the whole workload ({wl.total_tokens} tokens)"
    imgs = [i for i in wl.images if i.start + i.n_tokens <= tokens]
    wl = dataclasses.replace(wl, name=wl.name + f"_first{tokens}", seq_lens=[tokens],
                             images=imgs, n_deepstack=wl.n_deepstack if imgs else 0)
    return wl, (f"the first {tokens} of the {sum(make_workload(key).seq_lens)} tokens "
                f"({len(imgs)} image(s) inside), every layer and the head")


def cpu_baseline(args, key):
    """The oracle (fp64 NumPy, as it stands) on a sample of prefill workload `key`; returns
    the line's cpu_baseline object and the pass's seconds."""
    from synth import Inputs
    from oracle import runs
    wl, what = cpu_sample(key, args.cpu_tokens)
    inp = Inputs(wl)
    for i in range(wl.shape.num_layers):
        inp.layer(i)
    _ = inp.embed
    _ = inp.hidden
    t0 = time.perf_counter()
    runs.run_prefill(inp)
    dt = time.perf_counter() - t0
    return {"value": wl.total_tokens / dt, "unit": "tokens/s", "cores": host_cores(),
            "kind": "oracle",
            "sample": f"one oracle prefill + head over {what} (fp64 NumPy, BLAS on all host "
                      f"cores, inputs drawn before the clock starts)"}, dt


def cpu_baseline_decode():
    """The oracle's decode step + head on the whole decode workload (64 sequences)."""
    from synth import Inputs
    from synth.configs import decode_B64_cache4096
    from oracle import runs
    inp = Inputs(decode_B64_cache4096())
    for i in range(inp.shape.num_layers):
        inp.layer(i)
        inp.kv(i)
    _ = inp.embed
    _ = inp.hidden
    t0 = time.perf_counter()
    runs.run_decode(inp)
    dt = time.perf_counter() - t0
    B = inp.wl.decode_batch
    return {"value": B / dt, "unit": "tokens/s", "cores": host_cores(), "kind": "oracle",
            "sample": f"one oracle decode step + head over all {B} sequences (4096 cached "
                      f"tokens each, both layers; fp64 NumPy, BLAS on all host cores)"}


def line_config(args, world):
    """The `config` of the JSON line, the same for both arms."""
    wl = make_workload(args.prefill_workload, args.layers)
    wb, hb = weight_bytes(wl.shape)
    cfg = {"workload": wl.name + ": " + PREFILL_DESC[args.prefill_workload],
           "global_batch": len(wl.seq_lens) * world, "seq_len": wl.total_tokens,
           "parallelism": "replicas" if world > 1 else "single",
           "l2": f"inputs larger than L2: {wb / 1e9:.2f} GB of layer weights and a "
                 f"{hb / 1e9:.2f} GB head read per step"}
    if args.layers:
        cfg["layers"] = wl.shape.num_layers
    return cfg


def run_reference(args):
    """The reference arm: the oracle on the host cores, each step one pass over the sample of
    the prefill workload (rank 0 only; other ranks exit without work)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if int(os.environ.get("RANK", "0")) != 0:
        return 0
    secs, cpu = [], None
    for i in range(args.warmup + args.steps):
        cpu, dt = cpu_baseline(args, args.prefill_workload)
        if i >= args.warmup:
            secs.append(dt)
    tokens = cpu_sample(args.prefill_workload, args.cpu_tokens)[0].total_tokens
    value = tokens * len(secs) / sum(secs)
    cpu["value"] = value
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 * sum(secs) / len(secs), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": line_config(args, world), "cpu_baseline": cpu,
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    import torch
    dist = Dist(args.gpus)
    torch.cuda.set_device(dist.local)
    import cohere_compass_decoder_gb300 as pkg
    if not os.path.exists(pkg._lib.LIB_PATH):
        from cohere_compass_decoder_gb300.build import build
        build()
    pk = peaks()
    clocks = Clocks(dist.local) if dist.rank == 0 else None
    t_start = time.time()
    pre = None if args.no_prefill else prefill_leg(args, dist, pk, args.prefill_workload)
    ctx = {}
    if not args.no_prefill and not args.no_context:
        if args.prefill_workload != "pair":
            ctx["pair"] = prefill_leg(args, dist, pk, "pair", context=True)
        ctx["fp32"] = fp32_layer_latency(args)
    dec = None if args.no_decode else decode_leg(args, dist, pk)
    # keep the clock sampler running for at least ~1 s of GPU work
    if clocks and time.time() - t_start < 1.5:
        time.sleep(0.1)
    clk = clocks.stop() if clocks else None
    cpu = cpu_dec = None
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
        if pre is not None:
            cpu, _ = cpu_baseline(args, args.prefill_workload)
        if dec is not None:
            cpu_dec = cpu_baseline_decode()
    if dist.rank == 0 and pre is None:
        print(json.dumps({"decode": dec, "cpu_baseline_decode": cpu_dec}, default=str))
    elif dist.rank == 0:
        line = {
            "metric": METRIC, "value": pre["value"], "unit": "tokens/s", "n_gpus": dist.world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": pre["ms"] / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded; random-init weights of the workload's shapes)",
            "config": line_config(args, dist.world),
            "roofline": pre["roofline"], "cpu_baseline": cpu,
            "e2e": pre.get("e2e"), "gpu_launches": pre["launches"], "clocks": clk,
            "kernels": pre["kernels"],
        }
        if "pair" in ctx:
            c = ctx["pair"]
            line["pair_T2048"] = {"workload": PREFILL_DESC["pair"], "value": c["value"],
                                  "unit": "tokens/s", "ms_per_step": c["ms"] / args.steps,
                                  "roofline": c["roofline"], "gpu_launches": c["launches"],
                                  "kernels": c["kernels"]}
        for c in (pre, ctx.get("pair")):
            if c and c.get("next_rows"):
                line.setdefault("next_rows", {}).update(c["next_rows"])
        if "fp32" in ctx:
            line["layer_fp32_T128"] = ctx["fp32"]
        if dec:
            line["decode"] = {"workload": DECODE_DESC, "value": dec["value"], "unit": "tokens/s",
                              "ms_per_step": dec["ms"] / args.steps, "roofline": dec["roofline"],
                              "gpu_launches": dec["launches"], "kernels": dec["kernels"],
                              "cpu_baseline": cpu_dec}
            if dec.get("next_rows"):
                line.setdefault("next_rows", {}).update(dec["next_rows"])
        print(json.dumps(line))
    dist.close()
    return 0


if __name__ == "__main__":
    sys.exit(main())

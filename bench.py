"""Benchmark of the greedy decode step (one JSON line on stdout).

Workload (default ``dense4b``): a 36-layer 4B-class dense GQA decoder
(H=2560, Hq=32, Hkv=8, D=128, I=9728, V=151936, tied embeddings, bf16
weights N(0, 0.02), norm gains 1 + N(0, 0.02), seeded synthetic data), batch
1, a 512-token uniform-random prompt through the batched prompt pass
(tensor-core GEMMs; untimed), then greedy decode steps through the native loop (CUDA-graph
replays, EOS id 0 checked every 16 steps).  A "step" is one decode step of
the whole model; the timed steps cycle over the workload's 256 decode
positions 511..766 (the cache slots are rewritten on each pass).

``--impl reference`` times the fp64 CPU oracle on the host cores instead
(bounded sample, rank 0 only).  With N > 1 (torchrun) every rank decodes its
own replica (no collective on the data path) and rank 0 reports the total.
"""
from __future__ import annotations

import argparse
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "greedy decode tok/s at b=1 (36-layer 4B-class); HBM GB/s vs 8 TB/s peak"
POSITIONS_PER_PASS = 256
WORKLOAD_DESC = ("dense4b: 36 layers, H=2560, Hq=32, Hkv=8, D=128, I=9728, V=151936 tied; b=1; 512-token prompt "
                 "(batched prompt pass on tensor-core GEMMs, untimed); 256 greedy decode positions (511..766) per "
                 "pass through the CUDA-graph decode loop, EOS id 0 checked every 16 steps")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=256)
    ap.add_argument("--warmup", type=int, default=16)
    ap.add_argument("--impl", default="gemv", choices=["gemv", "reference"])
    ap.add_argument("--workload", default="dense4b",
                    choices=["dense4b", "layer4b", "dense4b_b8", "gqa12x3_b16", "select_b16", "attn_gqa12x3_b16",
                             "attn_dense4b_b8"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--prompt", type=int, default=None, help="prompt length (default: the workload's 512)")
    return ap.parse_args()


def max_over_ranks(ms: float, world: int, device) -> float:
    """The slowest rank's time (the whole job's time) of the timed region."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.barrier()
    return float(t.item())


def job_rate(units_per_rank: int, world: int, ms: float) -> float:
    """Whole-job throughput: the units all ranks processed over the slowest rank's time."""
    return units_per_rank * world / (ms / 1e3)


def dist_setup(n):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# ----------------------------------------------------------------------------- measured peaks

def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def committed_traffic(kernel_tag: str):
    """DRAM bytes per launch of a kernel from a committed ncu summary, if present."""
    p = os.path.join(ROOT, "profiles", f"{kernel_tag}.md")
    if not os.path.exists(p):
        return None
    m = re.search(r"dram bytes per launch[^0-9]*([0-9][0-9_,.]*)", open(p).read())
    if not m:
        return None
    return float(m.group(1).replace(",", "").replace("_", ""))


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- workload

def host_model(name, seed=0):
    import synth
    w = synth.workload(name)
    m = w.model
    layers = [synth.make_layer(seed, m, l) for l in range(m.n_layers)]
    head = w.extra.get("lm_head", True)
    E = synth.make_embedding(seed, m) if head else None
    fn = synth.make_final_norm(seed, m) if head else None
    return w, m, layers, E, fn


def bytes_per_step(m, positions, B=1, head=True):
    """Algorithmic HBM bytes of one step: every weight once, plus the KV rows read."""
    H, Hq, Hkv, D, I, V = m.hidden, m.n_heads, m.n_kv_heads, m.head_dim, m.intermediate, m.vocab
    per_layer = 2 * (Hq * D * H + 2 * Hkv * D * H + H * Hq * D + 3 * I * H) + 2 * 2 * H
    w = m.n_layers * per_layer + (2 * V * H + 2 * H if head else 0)
    kv = sum(2 * m.n_layers * Hkv * D * 2 * (p + 1) for p in positions)
    return w, kv


def run_layer(args, world, rank, local):
    """One 4B-class layer (no embedding, no LM head) stepped K times at the
    4096-token cache length: per-layer timing and profiling."""
    import torch
    import greedy_decode_step_gb300 as gd
    import synth

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w, m, layers_h, _, _ = host_model("layer4b")
    B, L0 = 1, w.kv_len[0]

    def to_dev(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)

    model = gd.Model(m.n_layers, m.hidden, m.n_heads, m.n_kv_heads, m.head_dim, m.intermediate, m.vocab,
                     m.rms_eps, m.rope_theta, [{k: to_dev(v) for k, v in l.items()} for l in layers_h])
    S_max = L0 + args.steps + args.warmup + 8
    kc = np.zeros((B, m.n_kv_heads, S_max, m.head_dim), np.uint16)
    vc = np.zeros_like(kc)
    synth.make_kv_prefix(w.seed, m, 0, 0, L0, "k", kc[0])
    synth.make_kv_prefix(w.seed, m, 0, 0, L0, "v", vc[0])
    st = gd.State(model, B, S_max, device=dev, k_cache=[to_dev(kc)], v_cache=[to_dev(vc)]).init()
    st.pos.fill_(L0)
    st.residual.copy_(torch.from_numpy(synth.make_residual(w.seed, B, m.hidden)).to(dev))
    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        gd.dec_step(model, st)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        e0.record(stream)
        for _ in range(args.steps):
            gd.dec_step(model, st)
        e1.record(stream)
        torch.cuda.synchronize(dev)
    assert gd.device_error(clear=True) == 0
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, dev)
    # positions L0 + W .. L0 + W + K - 1 (the warm-up steps advanced the cache)
    positions = list(range(L0 + args.warmup, L0 + args.warmup + args.steps))
    w_bytes, kv_bytes = bytes_per_step(m, positions, B, head=False)
    step_bytes = w_bytes + kv_bytes / len(positions)
    gbs = step_bytes / (ms / 1e3) / 1e9
    peak, src = peaks()
    launches = gd.dec_step_launches(model, st)
    roof = {"kernel": "step_kernel<1,128> (the whole layer step: norm, QKV+RoPE, attention, o_proj, norm, "
                      "gate/up, down)" if launches == 1 else "per-op layer step",
            "bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s", "frac": round(gbs / peak, 4),
            "peak_source": f"{src} copy bandwidth", "traffic": committed_traffic("step_kernel_layer4b"),
            "algorithmic_bytes_per_launch": int(step_bytes), "avg_launch_us": round(ms * 1e3, 2),
            "launches_timed": args.steps}
    e2e = None
    if not args.no_e2e:
        # from host buffers: pinned residual in, one step, residual out
        hr = torch.from_numpy(synth.make_residual(w.seed, B, m.hidden)).pin_memory()
        hout = torch.empty_like(hr).pin_memory()
        st.pos.fill_(L0)
        torch.cuda.synchronize(dev)
        e2 = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        e2[0].record(stream)
        for _ in range(args.steps):
            st.residual.copy_(hr, non_blocking=True)
            gd.dec_step(model, st)
            hout.copy_(st.residual, non_blocking=True)
        e2[1].record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = e2[0].elapsed_time(e2[1]) / args.steps
        e2e = {"value": round(e2e_ms * 1e3, 2), "unit": "us/step", "h2d_bytes_per_step": 4 * B * m.hidden,
               "d2h_bytes_per_step": 4 * B * m.hidden,
               "what": "pinned host residual -> H2D -> dec_step (one layer) -> D2H residual, per step"}
    res = {"metric": "one 4B-class layer step (b=1, 4096-token cache)", "value": round(ms * 1e3, 2),
           "unit": "us/step", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
           "ms_per_step": round(ms, 5), "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
           "dtype": "bf16", "data": "synthetic (seeded Philox weights, N(0,1) cache prefix)",
           "config": {"workload": "layer4b: H=2560, Hq=32, Hkv=8, D=128, I=9728, b=1, 4096-token cache, dec_step",
                      "l2": "inputs larger than L2 are not used: the layer's 202 MB of weights exceed L2 (129 MB)",
                      "step_bytes": int(step_bytes), "step_hbm_gbs": round(gbs, 1),
                      "step_hbm_frac_of_measured": round(gbs / peak, 4)},
           "roofline": roof,
           "glu_alone": glu_roofline(gd, torch, model, m, dev, stream, reps=20),
           "gpu_launches": launches * args.steps, "clocks": clk.summary()}
    if e2e:
        res["e2e"] = e2e

    def cpu_baseline():
        import oracle
        S = L0 + 64
        kch = np.zeros((1, m.n_kv_heads, S, m.head_dim), np.uint16)
        vch = np.zeros_like(kch)
        synth.make_kv_prefix(w.seed, m, 0, 0, L0, "k", kch[0])
        synth.make_kv_prefix(w.seed, m, 0, 0, L0, "v", vch[0])
        om = oracle.Model(m, layers_h, None, None, None, [kch], [vch])
        x = synth.make_residual(w.seed, B, m.hidden)[0].astype(np.float64)
        done, t0 = 0, time.time()
        while done < 60 and time.time() - t0 < 20.0:
            om.step(0, L0 + done, x_in=x)
            done += 1
        el = time.time() - t0
        return {"value": round(el / done * 1e6, 1), "unit": "us/step", "cores": 1, "kind": "oracle",
                "sample": f"{done} one-layer steps of the fp64 oracle at positions {L0}.. over the same "
                          f"{L0}-token cache prefix, single thread, {cpu_model()}"}

    return res, cpu_baseline


def run_batched(args, world, rank, local):
    """The batched configurations (not the headline): b=8 on the 36-layer
    4B-class model with the workload's seeded cache lengths U{1024..32768}, or
    b=16 on the 24-layer H=1536 12/3-head model with 8192-token caches; decode
    steps through dec_decode.  Weights and gains are the seeded synthetic
    recipe of the parity tests (bf16 N(0, 0.02), 1 + N(0, 0.02)); the caches
    are bf16 N(0, 1) drawn on the device from a seeded torch generator (same
    distribution, not the same numbers as the host recipe)."""
    import torch
    import greedy_decode_step_gb300 as gd

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    gd.lib()
    name = "dense4b_b8" if args.workload == "dense4b_b8" else "gqa12x3"
    w, m, layers_h, E_h, fn_h = host_model(name)
    L, H, Hq, Hkv, D, I, V, B = (m.n_layers, m.hidden, m.n_heads, m.n_kv_heads, m.head_dim, m.intermediate,
                                 m.vocab, w.batch)
    kv = [int(x) for x in w.kv_len]
    steps = min(args.steps, w.steps)

    def to_dev(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)

    layers = [{k: to_dev(v) for k, v in l.items()} for l in layers_h]
    E, fn = to_dev(E_h), to_dev(fn_h)
    model = gd.Model(L, H, Hq, Hkv, D, I, V, m.rms_eps, m.rope_theta, layers, embed=E, final_norm=fn, lm_head=E)
    S_max = max(kv) + steps + 16 + args.warmup + 8
    st = gd.State(model, B, S_max, device=dev).init()
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed)
    for l in range(L):
        st.k_cache[l].normal_(generator=g)
        st.v_cache[l].normal_(generator=g)
    p0 = torch.tensor(kv, dtype=torch.int32, device=dev)
    t0 = torch.randint(0, V, (B,), dtype=torch.int32, device=dev, generator=g)
    out = torch.empty((B, steps), dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def restart():
        st.pos.copy_(p0)
        st.token.copy_(t0)

    # the first 16-step call captures the decode graph (set-up), then W warm-up steps
    restart()
    gd.dec_decode(model, st, 16, -1, torch.empty((B, 16), dtype=torch.int32, device=dev))
    if args.warmup > 0:
        restart()
        gd.dec_decode(model, st, args.warmup, -1, torch.empty((B, args.warmup), dtype=torch.int32, device=dev))
    torch.cuda.synchronize(dev)
    restart()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        e0.record(stream)
        n = gd.dec_decode(model, st, steps, -1, out)
        e1.record(stream)
        torch.cuda.synchronize(dev)
    assert gd.device_error(clear=True) == 0
    ms = max_over_ranks(e0.elapsed_time(e1) / n, world, dev)
    w_bytes = L * 2 * (2 * Hq * D * H + 2 * Hkv * D * H + 3 * I * H) + 2 * V * H + L * 2 * 2 * H + 2 * H
    kv_bytes = sum(2 * L * Hkv * D * 2 * (p + (n - 1) / 2 + 1) for p in kv)
    gbs = (w_bytes + kv_bytes) / (ms / 1e3) / 1e9
    peak, src = peaks()
    first_tok = int(out[0, 0])
    roof = attn_roofline(gd, torch, model, st, m, dev, stream, f"attn_kernel_{args.workload}")
    e2e = None if args.no_e2e else batched_end_to_end(gd, torch, model, st, p0, t0, steps, dev, stream, B)
    res = {"metric": f"greedy decode tok/s at b={B} ({args.workload}); HBM GB/s", "value": round(B * world / (ms / 1e3), 2),
           "unit": "tok/s", "n_gpus": world, "steps": n, "warmup": args.warmup, "ms_per_step": round(ms, 5),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
           "data": "synthetic (seeded Philox N(0,0.02) weights; seeded torch N(0,1) caches)",
           "config": {"workload": f"{args.workload}: {w.description}", "batch": B, "layers": L, "kv_lens": kv,
                      "l2": "inputs larger than L2: every step streams the weights and all caches",
                      "step_bytes": int(w_bytes + kv_bytes), "step_hbm_gbs": round(gbs, 1),
                      "step_hbm_frac_of_measured": round(gbs / peak, 4),
                      "path": "weight GEMMs on this library's tcgen05 tensor-core GEMM (hi/lo bf16 activations "
                              "into one fp32 accumulator), split-K tensor-core attention"},
           "roofline": roof,
           "gpu_launches": gd.dec_step_launches(model, st) * n + 2, "clocks": clk.summary()}
    if e2e:
        res["e2e"] = e2e

    def cpu_baseline():
        return batched_oracle_rate(torch, m, layers_h, E_h, fn_h, st, kv[0], int(t0[0]), first_tok)

    return res, cpu_baseline


def run_attn_op(args, world, rank, local):
    """The split-K attention alone (dec_gqa_decode_attn) on one layer of a
    batched configuration: b=16, Hq=12, Hkv=3 with 8192-token caches, or b=8,
    Hq=32, Hkv=8 with the dense4b_b8 cache lengths.  bf16 N(0,1) caches and
    fp32 N(0,1) queries from a seeded torch generator; inputs larger than L2
    (201 MB / 1.1 GB of K/V per launch)."""
    import torch
    import greedy_decode_step_gb300 as gd

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    gd.lib()
    w = synth_workload("dense4b_b8" if args.workload == "attn_dense4b_b8" else "gqa12x3")
    m, B = w.model, w.batch
    Hq, Hkv, D = m.n_heads, m.n_kv_heads, m.head_dim
    kv = [int(x) for x in w.kv_len]
    S_max = max(kv) + 8
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed)
    K = torch.randn((B, Hkv, S_max, D), device=dev, generator=g).to(torch.bfloat16)
    V = torch.randn((B, Hkv, S_max, D), device=dev, generator=g).to(torch.bfloat16)
    q = torch.randn((B, Hq, D), device=dev, generator=g)
    pos = torch.tensor(kv, dtype=torch.int32, device=dev)
    o = torch.empty_like(q)
    ws = gd.dec_gqa_decode_attn(q, K, V, pos, o)
    for _ in range(max(3, args.warmup)):
        gd.dec_gqa_decode_attn(q, K, V, pos, o, ws=ws)
    torch.cuda.synchronize(dev)
    stream = torch.cuda.current_stream(dev)
    n = max(1, min(args.steps, 200))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        e0.record(stream)
        for _ in range(n):
            gd.dec_gqa_decode_attn(q, K, V, pos, o, ws=ws)
        e1.record(stream)
        torch.cuda.synchronize(dev)
    assert gd.device_error(clear=True) == 0
    avg_s = max_over_ranks(e0.elapsed_time(e1) / n, world, dev) / 1e3
    alg = sum(Hkv * (p + 1) * D * 2 * 2 for p in kv) + 2 * B * Hq * D * 4
    peak, src = peaks()
    gbs = alg / avg_s / 1e9
    res = {"metric": f"GQA decode attention GB/s ({args.workload})", "value": round(gbs * world, 1), "unit": "GB/s",
           "n_gpus": world, "steps": n, "warmup": max(3, args.warmup), "ms_per_step": round(avg_s * 1e3, 5),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
           "data": "synthetic (seeded torch N(0,1) caches and queries)",
           "config": {"workload": f"{args.workload}: one layer of {w.description}", "batch": B, "Hq": Hq,
                      "Hkv": Hkv, "head_dim": D, "kv_lens": kv,
                      "l2": "inputs larger than L2 (K/V bytes per launch above 129 MB)"},
           "roofline": {"kernel": "attn_kernel / attn_lean_kernel (balanced schedule beyond one wave)", "bound": "hbm",
                        "achieved": round(gbs, 1), "peak": peak,
                        "unit": "GB/s", "frac": round(gbs / peak, 4), "peak_source": f"{src} (burst copy)",
                        "traffic": committed_traffic(f"attn_kernel_{args.workload[5:]}"),
                        "algorithmic_bytes_per_launch": int(alg), "avg_launch_us": round(avg_s * 1e6, 2),
                        "launches_timed": n,
                        "note": "each call also carries its ticket reset (a memset node), inside the timing"},
           "gpu_launches": n, "clocks": clk.summary()}
    return res, None


def synth_workload(name):
    import synth
    return synth.workload(name)


def attn_roofline(gd, torch, model, st, m, dev, stream, tag, reps=4):
    """The dominant kernel of the batched step, the split-K attention, timed
    alone through its C-ABI entry point on every layer's cache at the
    positions the decode reached (CUDA events around reps x layers launches;
    each call also carries its 4-byte-per-group ticket reset, a memset node,
    so the achieved rate is a floor)."""
    B, Hq, D = st.batch, m.n_heads, m.head_dim
    q = torch.randn((B, Hq, D), device=dev, dtype=torch.float32)
    o = torch.empty_like(q)
    pos = st.pos.clone()
    ws = gd.dec_gqa_decode_attn(q, st.k_cache[0], st.v_cache[0], pos, o)
    for l in range(min(4, m.n_layers)):
        gd.dec_gqa_decode_attn(q, st.k_cache[l], st.v_cache[l], pos, o, ws=ws)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    n = 0
    for _ in range(reps):
        for l in range(m.n_layers):
            gd.dec_gqa_decode_attn(q, st.k_cache[l], st.v_cache[l], pos, o, ws=ws)
            n += 1
    e1.record(stream)
    torch.cuda.synchronize(dev)
    assert gd.device_error(clear=True) == 0
    avg_s = e0.elapsed_time(e1) / 1e3 / n
    lens = [int(p) + 1 for p in pos.cpu().tolist()]
    alg = sum(m.n_kv_heads * k * D * 2 * 2 for k in lens) + 2 * B * Hq * D * 4
    peak, src = peaks()
    achieved = alg / avg_s / 1e9
    return {"kernel": "split-K GQA decode attention on the tensor cores (attn_kernel; attn_lean_kernel, the "
                      "balanced schedule, when the split grid exceeds one wave)", "bound": "hbm",
            "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
            "peak_source": f"{src} (burst copy; kernel timed alone)", "traffic": committed_traffic(tag),
            "algorithmic_bytes_per_launch": int(alg), "avg_launch_us": round(avg_s * 1e6, 2), "launches_timed": n,
            "kv_lens": lens}


def batched_end_to_end(gd, torch, model, st, p0, t0, steps, dev, stream, B):
    """The user call from host buffers: pinned positions and tokens -> H2D,
    dec_decode over the steps, D2H of the generated tokens."""
    hp, ht = p0.cpu().pin_memory(), t0.cpu().pin_memory()
    hout = torch.empty((B, steps), dtype=torch.int32).pin_memory()
    dout = torch.empty((B, steps), dtype=torch.int32, device=dev)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    st.pos.copy_(hp, non_blocking=True)
    st.token.copy_(ht, non_blocking=True)
    n = gd.dec_decode(model, st, steps, -1, dout)
    hout.copy_(dout, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1)
    return {"value": round(n * B / (ms / 1e3), 2), "unit": "tok/s", "h2d_bytes_per_step": round(8 * B / n, 3),
            "d2h_bytes_per_step": 4 * B,
            "what": "pinned host positions and tokens -> H2D -> dec_decode -> D2H tokens; tokens / wall time"}


def batched_oracle_rate(torch, m, layers_h, E_h, fn_h, st, p, token, gpu_first, max_seconds=25.0):
    """The fp64 oracle's decode steps of sequence 0 from the same position,
    token and cache prefix (copied from the device), single thread, for up to
    max_seconds; its first token is compared with the GPU's."""
    import oracle
    S = p + 16  # the oracle's steps stay below this slot

    def host(t):
        return t[:1, :, :S].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)

    kc = [host(st.k_cache[l]) for l in range(m.n_layers)]
    vc = [host(st.v_cache[l]) for l in range(m.n_layers)]
    om = oracle.Model(m, layers_h, E_h, fn_h, E_h, kc, vc)
    done, t0 = 0, time.time()
    first = None
    while True:
        token, logits, _ = om.step(0, p + done, token=token)
        if first is None:
            first = (token, float(np.sort(logits)[-1] - np.sort(logits)[-2]))
        done += 1
        if time.time() - t0 > max_seconds or done >= 8:
            break
    el = time.time() - t0
    return {"value": round(done / el, 5), "unit": "tok/s", "cores": 1, "kind": "oracle",
            "sample": f"{done} decode steps of sequence 0 (all {m.n_layers} layers + LM head, cache of {p} "
                      f"tokens copied from the device) by the fp64 oracle, single thread, {cpu_model()}",
            "first_token_oracle": first[0], "first_token_gpu": gpu_first, "oracle_top2_margin": round(first[1], 5)}


def run_select(args, world, rank, local):
    """Token selection (not the headline): dec_select_tokens on b=16 rows of
    V=151936 float32 logits (synth draws, std 4) with a repetition penalty
    over 512 listed ids per row, temperature 0.7, top-k 50 and top-p 0.9, so
    that every phase of the kernel runs.  L2 is flushed (a 256 MB write)
    before every timed call; each call is timed by its own CUDA events."""
    import torch
    import greedy_decode_step_gb300 as gd
    import oracle
    import synth

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    B, V, n_prev = 16, 151936, 512
    kw = dict(repetition_penalty=1.1, temperature=0.7, top_k=50, top_p=0.9)
    z = synth.make_logits(0, "bench.select", B, V, 4.0, True)
    u = synth.make_uniforms(0, "bench.select.u", B)
    prev = synth.uniform_int(0, "bench.select.prev", (B, n_prev), 0, V - 1)
    zd, ud, pd = (torch.from_numpy(x).to(dev) for x in (z, u, prev))
    out = torch.empty(B, dtype=torch.int32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(max(3, args.warmup)):
        gd.dec_select_tokens(zd, out, u=ud, prev_tokens=pd, **kw)
    torch.cuda.synchronize(dev)
    steps = max(1, min(args.steps, 200))
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    with ClockSampler(local) as clk:
        for e0, e1 in ev:
            flush.zero_()
            e0.record(stream)
            gd.dec_select_tokens(zd, out, u=ud, prev_tokens=pd, **kw)
            e1.record(stream)
        torch.cuda.synchronize(dev)
    assert gd.device_error(clear=True) == 0
    ms = statistics.mean(e0.elapsed_time(e1) for e0, e1 in ev)
    # one row alone (one cluster): the latency of a row, without other clusters beside it
    out1 = torch.empty(1, dtype=torch.int32, device=dev)
    ev1 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(20)]
    for e0, e1 in ev1:
        flush.zero_()
        e0.record(stream)
        gd.dec_select_tokens(zd[:1], out1, u=ud[:1], prev_tokens=pd[:1], **kw)
        e1.record(stream)
    torch.cuda.synchronize(dev)
    ms1 = statistics.mean(e0.elapsed_time(e1) for e0, e1 in ev1)
    # the same row with top-p alone (no top-k cut): the sampling of the pages' rollout
    kw_p = dict(kw, top_k=0)
    for e0, e1 in ev1:
        flush.zero_()
        e0.record(stream)
        gd.dec_select_tokens(zd[:1], out1, u=ud[:1], prev_tokens=pd[:1], **kw_p)
        e1.record(stream)
    torch.cuda.synchronize(dev)
    ms1p = statistics.mean(e0.elapsed_time(e1) for e0, e1 in ev1)
    # end to end from pinned host buffers: logits, draws and ids in, tokens out
    zh, uh, ph = (torch.from_numpy(x).pin_memory() for x in (z, u, prev))
    oh = torch.empty(B, dtype=torch.int32).pin_memory()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        zd.copy_(zh, non_blocking=True)
        ud.copy_(uh, non_blocking=True)
        pd.copy_(ph, non_blocking=True)
        gd.dec_select_tokens(zd, out, u=ud, prev_tokens=pd, **kw)
        oh.copy_(out, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = e0.elapsed_time(e1) / steps
    algo = B * V * 4 + B * n_prev * 4 + B * 4 + B * 4
    peak, src = peaks()
    gbs = algo / (ms / 1e3) / 1e9
    t0 = time.perf_counter()
    ref = [oracle.select_token(z[b], prev=prev[b], penalty=float(np.float32(1.1)), temperature=float(np.float32(0.7)),
                               top_k=50, top_p=float(np.float32(0.9)), u=float(u[b]))[0] for b in range(B)]
    cpu_ms = (time.perf_counter() - t0) * 1e3
    agree = int(sum(int(a == b) for a, b in zip(out.cpu().tolist(), ref)))
    res = {"metric": "token selection us per call (b=16, V=151936; penalty, temperature, top-k 50, top-p 0.9)",
           "value": round(ms * 1e3, 2), "unit": "us/call", "n_gpus": 1, "steps": steps,
           "warmup": max(3, args.warmup), "ms_per_step": round(ms, 5), "higher_is_better": False,
           "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic (synth logits, std 4)",
           "config": {"workload": "select_b16: 16 rows x 151936 fp32 logits, 512 penalised ids per row, T=0.7, "
                                  "top_k=50, top_p=0.9; L2 flushed before each call",
                      "tokens_equal_to_oracle": f"{agree}/{B}", "one_row_us": round(ms1 * 1e3, 2),
                      "one_row_top_p_only_us": round(ms1p * 1e3, 2)},
           "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peak, "unit": "GB/s",
                        "frac": round(gbs / peak, 4), "traffic": committed_traffic("select_kernel_b16"),
                        "peak_source": src,
                        "note": "one cluster of 8 CTAs per row; top-k 50 takes the candidate path (one "
                                "cluster barrier); latency of the dependent steps, not DRAM, bounds the call"},
           "e2e": {"value": round(e2e_ms * 1e3, 2), "unit": "us/call", "h2d_bytes_per_step": int(algo - B * 4),
                   "d2h_bytes_per_step": B * 4},
           "cpu_baseline": {"value": round(cpu_ms * 1e3, 1), "unit": "us/call", "cores": 1, "kind": "oracle",
                            "sample": f"the fp64 oracle's selection of the same {B} rows, single thread, "
                                      f"{cpu_model()}"},
           "gpu_launches": steps, "clocks": clk.summary()}
    return res, None


def run_gpu(args, world, rank, local):
    import torch
    import greedy_decode_step_gb300 as gd
    import synth

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    gd.lib()
    w, m, layers_h, E_h, fn_h = host_model(args.workload)
    B = 1

    def to_dev(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(dev).view(torch.bfloat16)

    t0 = time.time()
    layers = [{k: to_dev(v) for k, v in l.items()} for l in layers_h]
    E = to_dev(E_h) if E_h is not None else None
    fn = to_dev(fn_h) if fn_h is not None else None
    model = gd.Model(m.n_layers, m.hidden, m.n_heads, m.n_kv_heads, m.head_dim, m.intermediate, m.vocab,
                     m.rms_eps, m.rope_theta, layers, embed=E, final_norm=fn, lm_head=E)
    P = args.prompt or w.prompt_len
    S_max = P + POSITIONS_PER_PASS + 8
    st = gd.State(model, B, S_max, device=dev).init()
    prompt_h = synth.make_tokens(w.seed, "prompt", (B, w.prompt_len), m.vocab)[:, :P].copy()
    prompt = torch.from_numpy(prompt_h).to(dev)
    setup_s = time.time() - t0
    stream = torch.cuda.current_stream(dev)

    # prompt pass (untimed for the metric; reported)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    gd.dec_prefill(model, st, prompt)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    prefill_ms = e0.elapsed_time(e1)
    pos0 = st.pos.clone()
    tok0 = st.token.clone()

    def restart():
        st.pos.copy_(pos0)
        st.token.copy_(tok0)

    # set-up: the first 16-step call captures the decode graph (not counted
    # as warm-up); then exactly W untimed warm-up steps
    t_cap = time.time()
    restart()
    cap_out = torch.empty((B, 16), dtype=torch.int32, device=dev)
    gd.dec_decode(model, st, 16, w.eos_id, cap_out)
    torch.cuda.synchronize(dev)
    capture_s = time.time() - t_cap
    if args.warmup > 0:
        restart()
        gd.dec_decode(model, st, args.warmup, w.eos_id, torch.empty((B, args.warmup), dtype=torch.int32, device=dev))
        torch.cuda.synchronize(dev)

    # timed: exactly K steps, in passes over the workload's decode positions
    passes = []
    left = args.steps
    while left > 0:
        passes.append(min(POSITIONS_PER_PASS, left))
        left -= passes[-1]
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize(dev)
    executed = 0
    positions = []
    outs = [torch.empty((B, n), dtype=torch.int32, device=dev) for n in passes]
    done_per_pass = []
    with ClockSampler(local) as clk:
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * len(passes))]
        for i, n in enumerate(passes):
            restart()
            ev[2 * i].record(stream)
            d = gd.dec_decode(model, st, n, w.eos_id, outs[i])
            ev[2 * i + 1].record(stream)
            executed += d
            done_per_pass.append(d)
            positions += list(range(int(pos0[0]), int(pos0[0]) + n))
        torch.cuda.synchronize(dev)
    ms = sum(ev[2 * i].elapsed_time(ev[2 * i + 1]) for i in range(len(passes)))
    ms = max_over_ranks(ms, world, dev)
    # end-of-sequence tokens actually emitted in the executed columns (the
    # columns after a row's first EOS are padding and not counted)
    eos_emitted = 0
    for o, d in zip(outs, done_per_pass):
        t = o.cpu().numpy()[:, :d]
        for row in t:
            hit = np.nonzero(row == w.eos_id)[0]
            eos_emitted += 1 if hit.size else 0
    assert gd.device_error(clear=True) == 0

    w_bytes, kv_bytes = bytes_per_step(m, positions, B)
    step_bytes = w_bytes + kv_bytes / max(1, len(positions))
    ms_per_step = ms / executed
    tok_s = job_rate(executed * B, world, ms)

    # dominant kernel: the persistent step kernel (one launch is one whole
    # step); its average launch time is the timed region over the steps run,
    # which also holds the two tiny control kernels per pass and the host's
    # end-of-sequence check every 16 steps, so the achieved rate is a floor
    launches_per_step = gd.dec_step_launches(model, st)
    peak, src = peaks()
    achieved = step_bytes / (ms_per_step / 1e3) / 1e9
    roof = {"kernel": "step_kernel<1,128> (the whole decode step: 36 layers + LM head + argmax)" if launches_per_step == 1
            else "per-op step (GEMV + attention kernels)",
            "bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "peak_source": f"{src} copy bandwidth (the only HBM figure; no sustained copy figure is given)",
            "traffic": committed_traffic("step_kernel_dense4b"),
            "algorithmic_bytes_per_launch": int(step_bytes), "avg_launch_us": round(ms_per_step * 1e3, 2),
            "launches_timed": executed}
    # the gate/up GEMV alone through its C-ABI entry point (36 launches over
    # the layers' weights), for reference
    glu_alone = glu_roofline(gd, torch, model, m, dev, stream)

    e2e = None
    if not args.no_e2e:
        e2e = end_to_end(gd, torch, model, st, m, w, prompt_h, dev, stream, B)

    res = {
        "metric": METRIC,
        "value": round(tok_s, 2),
        "unit": "tok/s",
        "n_gpus": world,
        "steps": executed,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded Philox N(0,0.02) weights, uniform prompt tokens)",
        "config": {
            "workload": WORKLOAD_DESC,
            "batch": B, "prompt_len": P, "decode_positions": [positions[0], positions[-1]] if positions else None,
            "accumulate": "fp32", "weights": "bf16", "kv_cache": "bf16", "activations": "fp32",
            "l2": "inputs larger than L2: every step streams 8.0 GB of weights (L2 129 MB)",
            "parallelism": f"replicas x{world} (no collective)",
            "prefill_ms": round(prefill_ms, 2), "graph_capture_s": round(capture_s, 3),
            "graph_capture_steps": 16,
            "setup_s": round(setup_s, 2),
            "step_bytes": int(step_bytes), "step_weight_bytes": int(w_bytes),
            "step_hbm_gbs": round(step_bytes / (ms_per_step / 1e3) / 1e9, 1),
            "step_hbm_frac_of_measured": round(step_bytes / (ms_per_step / 1e3) / 1e9 / peaks()[0], 4),
            "step_hbm_frac_of_8tbs": round(step_bytes / (ms_per_step / 1e3) / 8e12, 4),
            "rows_that_emitted_eos": eos_emitted,
        },
        "roofline": roof,
        "glu_alone": glu_alone,
        "gpu_launches": executed * launches_per_step + 2 * len(passes),
        "clocks": clk.summary(),
    }
    if e2e:
        res["e2e"] = e2e

    def cpu_baseline():
        done, el = oracle_rate(m, layers_h, E_h, fn_h, 3, max_seconds=25.0)
        return {"value": round(done / el, 5), "unit": "tok/s", "cores": 1, "kind": "oracle",
                "sample": f"{done} full decode steps (36 layers + LM head) of the fp64 oracle at positions 511.. "
                          f"over a 511-token N(0,1) cache, single thread, {cpu_model()}"}

    return res, cpu_baseline


def glu_roofline(gd, torch, model, m, dev, stream, reps=3):
    B = 1
    y = torch.randn((B, m.hidden), device=dev, dtype=torch.float32)
    h = torch.empty((B, m.intermediate), device=dev, dtype=torch.float32)
    layers = model.layers
    for l in layers[:4]:
        gd.dec_glu_gemv(y, l["wg"], l["wu"], h)
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    n = 0
    for _ in range(reps):
        for l in layers:
            gd.dec_glu_gemv(y, l["wg"], l["wu"], h)
            n += 1
    e1.record(stream)
    torch.cuda.synchronize(dev)
    avg_s = e0.elapsed_time(e1) / 1e3 / n
    alg = 2 * 2 * m.intermediate * m.hidden + 4 * B * m.hidden + 4 * B * m.intermediate
    peak, src = peaks()
    achieved = alg / avg_s / 1e9
    traffic = committed_traffic("gemv_glu_dense4b")
    return {"kernel": "gemv_kernel<GLU,1> (gate/up GEMV + SiLU*mul)", "bound": "hbm",
            "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
            "peak_source": f"{src} (burst copy; kernel timed alone)", "traffic": traffic,
            "algorithmic_bytes_per_launch": alg, "avg_launch_us": round(avg_s * 1e6, 2), "launches_timed": n}


def end_to_end(gd, torch, model, st, m, w, prompt_h, dev, stream, B):
    """The user call from host buffers: pinned prompt -> H2D, dec_generate
    (prompt pass + 256 decode steps), D2H of the tokens."""
    P = prompt_h.shape[1]
    n = POSITIONS_PER_PASS
    host_prompt = torch.from_numpy(prompt_h).pin_memory()
    host_out = torch.empty((B, n), dtype=torch.int32).pin_memory()
    dprompt = torch.empty((B, P), dtype=torch.int32, device=dev)
    dout = torch.empty((B, n), dtype=torch.int32, device=dev)
    st.pos.zero_()
    torch.cuda.synchronize(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    dprompt.copy_(host_prompt, non_blocking=True)
    done = gd.dec_generate(model, st, dprompt, n, w.eos_id, dout)
    host_out.copy_(dout, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = e0.elapsed_time(e1)
    return {"value": round(done * B / (ms / 1e3), 2), "unit": "tok/s",
            "h2d_bytes_per_step": round(B * P * 4 / done, 2), "d2h_bytes_per_step": B * 4,
            "what": "pinned host prompt -> H2D -> dec_generate (512-token prompt pass + 256 decode steps) -> "
                    "D2H tokens; tokens generated / wall time of the whole call"}


# ----------------------------------------------------------------------------- CPU oracle

def oracle_rate(m, layers_h, E_h, fn_h, max_steps, max_seconds=25.0, seed=0):
    """Decode steps of the fp64 oracle on one host core at positions 511.. with a
    511-token N(0,1) cache prefix (the oracle cannot afford the 511-step prompt pass)."""
    import oracle
    import synth
    P = 511
    S_max = P + max_steps + 2
    kc, vc = [], []
    for l in range(m.n_layers):
        k = np.zeros((1, m.n_kv_heads, S_max, m.head_dim), np.uint16)
        v = np.zeros_like(k)
        synth.make_kv_prefix(seed, m, l, 0, P, "k", k[0])
        synth.make_kv_prefix(seed, m, l, 0, P, "v", v[0])
        kc.append(k)
        vc.append(v)
    om = oracle.Model(m, layers_h, E_h, fn_h, E_h, kc, vc)
    t = int(synth.make_tokens(seed, "prompt", (1, 512), m.vocab)[0, -1])
    done, t0 = 0, time.time()
    while done < max_steps:
        t, _, _ = om.step(0, P + done, token=t)
        done += 1
        if time.time() - t0 > max_seconds:
            break
    el = time.time() - t0
    return done, el


def cpu_model():
    try:
        for line in open("/proc/cpuinfo"):
            if "model name" in line or "CPU part" in line:
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def main():
    args = parse()
    world, rank, local = dist_setup(args.gpus)
    if args.impl == "reference":
        if rank != 0:
            return 0
        _, m, layers_h, E_h, fn_h = host_model(args.workload)
        n = max(1, min(args.steps, 4))
        done, el = oracle_rate(m, layers_h, E_h, fn_h, n, max_seconds=60.0)
        v = done / el
        line = {"metric": METRIC, "value": round(v, 5), "unit": "tok/s", "n_gpus": args.gpus, "steps": done,
                "warmup": 0, "ms_per_step": round(el / done * 1e3, 1), "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
                "config": {"workload": WORKLOAD_DESC,
                           "reference_sample": "the fp64 oracle's decode steps at positions 511.. over a 511-token "
                                               "N(0,1) cache prefix (bounded sample of the same workload)"},
                "cpu_baseline": {"value": round(v, 5), "unit": "tok/s", "cores": 1, "kind": "oracle",
                                 "sample": f"{done} full decode steps (36 layers + LM head) of the fp64 oracle, "
                                           f"single thread, {cpu_model()}"},
                "e2e": {"value": round(v, 5), "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return 0

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    if args.workload == "layer4b":
        res, host = run_layer(args, world, rank, local)
    elif args.workload in ("dense4b_b8", "gqa12x3_b16"):
        res, host = run_batched(args, world, rank, local)
    elif args.workload == "select_b16":
        res, host = run_select(args, world, rank, local)
    elif args.workload.startswith("attn_"):
        res, host = run_attn_op(args, world, rank, local)
    else:
        res, host = run_gpu(args, world, rank, local)
    if rank == 0 and host is not None and not args.no_cpu_baseline:
        res["cpu_baseline"] = host()
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(res))
    return 0


if __name__ == "__main__":
    sys.exit(main())

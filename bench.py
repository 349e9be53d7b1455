"""Benchmark of the INT8-QK attention path on GB300.

One step = the whole path once on the banded cross-window workload
(B1 H56 Q4096 K33600 D128, bf16, per-key raised-cosine skirt bias):
  1. K mean + INT8 quantisation of Q and K          (2 launches)
  2. core keys [6720, 26880) without bias, with LSE (1 launch)
  3. left and right skirt keys with the bias, LSE   (2 launches, key sub-range views)
  4. two exact LSE merges                           (2 launches)
value = 4*B*H*Q*K*D / step time (TOPS). The single unmasked call and the
single bias call over all keys are timed too (their ratio is the bias cost).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Under torchrun each rank runs its own copy of the workload on its GPU (the
heads are independent; no collective on the data path), rank 0 prints one
JSON line. ``--impl reference`` times the CPU oracle on the host cores on a
bounded sample of the same workload.
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

METRIC = "attention TOPS and ms per call at 4096x33600x56x128 (unmasked/bias); % of roofline"
UNIT = "TOPS"
# comfy-kitchen issue #177, RTX 5090: core 20160 keys unmasked 5.19 ms + skirt
# 13440 keys masked 5.86 ms = 11.05 ms for the same 4096x33600x56x128 problem.
PAGE_SPLIT_MS = 11.05

# DRAM traffic of attn_fwd_kernel from one ncu capture (dram__bytes_read.sum +
# dram__bytes_write.sum) of the 16-head banded case (Sq 4096, Sk 33600,
# unmasked), recorded with the SHA-256 of the kernel sources it was taken on. A launch's traffic is scaled
# from it per head, with the key-proportional part scaled by the keys of the
# launch. When the kernel sources change, the figure no longer applies.
ATTN_TRAFFIC = {"source_sha256": "955c2c8ac1c2a758f6f496fa873c80ed14e2036a0a7a925829e0902873be4bd5",
                "heads": 16, "sq": 4096, "sk": 33600, "d": 128, "bytes": 245499648.0}


def attn_source_sha():
    """SHA-256 of the attention kernel's code: attention.cu and ptx.cuh with their
    comments and whitespace removed, so that a comment edit keeps the figure."""
    import hashlib
    import re
    h = hashlib.sha256()
    for f in ("attention.cu", "ptx.cuh"):
        with open(os.path.join(ROOT, "int8_qk_quantized_gb300", "csrc", f), encoding="utf-8") as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()


def attn_traffic_per_launch(H, Sq, sk_list, D):
    """Average DRAM bytes per attention launch, or None if not measured on this source."""
    t = ATTN_TRAFFIC
    if t["bytes"] is None or t["source_sha256"] != attn_source_sha():
        return None
    fixed = t["sq"] * t["d"] * 3 + t["sq"] * 8          # q8 + out + lse + q_scale per head
    per_key = (t["bytes"] / t["heads"] - fixed) / t["sk"]
    per_launch = [H * (Sq * D * 3 + Sq * 8 + per_key * sk) for sk in sk_list]
    return sum(per_launch) / len(per_launch)


def dist_info():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def dist_max(value, dist, device):
    """The largest `value` over all ranks (the slowest rank times the job)."""
    import torch
    t = torch.tensor([float(value)], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.item()


def weak_value(world_size, ops_per_rank, ms_per_step):
    """Whole-job throughput in TOPS when every rank runs its own copy of the workload."""
    return world_size * ops_per_rank / (ms_per_step * 1e-3) / 1e12


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return d["hbm_gbs"], d["bf16_tflops"], d.get("bf16_tflops_sustained"), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


def start_clock_sampler():
    try:
        return subprocess.Popen(
            ["nvidia-smi", "--query-gpu=index,clocks.sm,clocks.max.sm,power.draw,"
             "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap", "--format=csv,noheader,nounits", "-lms", "200"],
            stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
    except Exception:
        return None


def stop_clock_sampler(proc, gpu_index):
    if proc is None:
        return None
    proc.terminate()
    try:
        out, _ = proc.communicate(timeout=5)
    except Exception:
        proc.kill()
        out = ""
    sm, mx, reasons = [], None, set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    for line in out.strip().splitlines():
        f = [x.strip() for x in line.split(",")]
        if len(f) < 9 or f[0] != str(gpu_index):
            continue
        try:
            sm.append(float(f[1]))
            mx = float(f[2])
        except ValueError:
            continue
        for n, v in zip(names, f[5:9]):
            if v.lower() == "active":
                reasons.add(n)
    if not sm:
        return None
    loaded = [s for s in sm if mx is None or s > 0.5 * mx] or sm
    return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": mx, "reasons": sorted(reasons),
            "samples": len(sm)}


def run_reference(args):
    """The CPU oracle, timed on the host cores on a bounded sample per step."""
    ws, rank, _ = dist_info()
    if rank != 0:
        return
    import numpy as np
    import torch

    import oracle
    from workloads import WORKLOADS, make_inputs

    wl = WORKLOADS["banded"]
    sample_heads, sample_rows = 1, 256
    small = wl.with_(H=sample_heads)
    inp = make_inputs(small, "cpu")
    qn = inp.q.float().numpy()[:, :, :sample_rows]
    kn = inp.k.float().numpy()
    vn = inp.v.float().numpy()
    bias = inp.bias.numpy()

    def step():
        oracle.quantize_and_attend(qn, kn, vn, bias=bias)

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = (time.perf_counter() - t0) / args.steps
    ops = 4.0 * sample_heads * sample_rows * wl.Sk * wl.D
    val = ops / dt / 1e12
    cores = os.cpu_count()
    sample = (f"{sample_heads} head x {sample_rows} query rows x {wl.Sk} keys per step: K mean "
              f"+ quantise + same-quantisation fp64 attention with the skirt bias")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": val, "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": "banded cross-window attention B1 H56 Q4096 K33600 D128 bf16, "
                              "per-key skirt bias", "sample": sample},
        "cpu_baseline": {"value": val, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": val, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def cpu_baseline(seconds_target=12.0):
    """The oracle as it stands on a bounded sample of the workload (host cores)."""
    import numpy as np

    import oracle
    from workloads import WORKLOADS, make_inputs

    wl = WORKLOADS["banded"].with_(H=1)
    inp = make_inputs(wl, "cpu")
    qn = inp.q.float().numpy()
    kn = inp.k.float().numpy()
    vn = inp.v.float().numpy()
    bias = inp.bias.numpy()
    rows = 512
    t0 = time.perf_counter()
    n = 0
    total_rows = 0
    while time.perf_counter() - t0 < seconds_target and n < 64:
        oracle.quantize_and_attend(qn[:, :, :rows], kn, vn, bias=bias)
        total_rows += rows
        n += 1
    dt = time.perf_counter() - t0
    ops = 4.0 * total_rows * wl.Sk * wl.D
    return {"value": ops / dt / 1e12, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle",
            "sample": f"{n} runs of 1 head x {rows} query rows x {wl.Sk} keys (K mean + "
                      f"quantise + fp64 attention with bias) in {dt:.1f} s"}


def graph_ms(torch, fn, n=20, reps=3):
    """ms per call of fn() captured n times in one CUDA graph and replayed reps
    times (CUDA events around the replays, after one untimed replay)."""
    fn()
    torch.cuda.synchronize()
    gs = torch.cuda.Stream()
    gs.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=gs):
        for _ in range(n):
            fn()
    graph.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        graph.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / (n * reps)


def time_workloads(ia, torch, names=("tiny", "sdxl", "anima4k", "anima9k", "sparse"), n=10):
    """Quantise and attention times of the other workloads (CUDA events,
    after 3 warm-up calls). TOPS use algorithmic ops (kept tiles for sparse)."""
    from workloads import WORKLOADS, algorithmic_ops, make_inputs
    res = {}
    for name in names:
        wl = WORKLOADS[name]
        inp = make_inputs(wl, "cuda")
        kept = None
        if wl.sparse:
            kept = inp.block_mask.float().sum(-1).mean().item()
        q8, qs, k8, ks = ia.quantize_qk(inp.q, inp.k, granularity=wl.granularity,
                                        kv_valid=inp.kv_valid)
        out, lse = ia.attention(q8, k8, qs, ks, inp.v, bias=inp.bias, block_mask=inp.block_mask,
                                v_scale=inp.v_scale, kv_valid=inp.kv_valid,
                                granularity=wl.granularity, return_lse=True)

        def tq():
            ia.quantize_qk(inp.q, inp.k, granularity=wl.granularity, kv_valid=inp.kv_valid)

        def tk():
            ia.quantize_qk(None, inp.k, granularity=wl.granularity, kv_valid=inp.kv_valid)

        def ta():
            ia.attention(q8, k8, qs, ks, inp.v, bias=inp.bias, block_mask=inp.block_mask,
                         v_scale=inp.v_scale, kv_valid=inp.kv_valid, granularity=wl.granularity,
                         out=out, lse=lse, return_lse=True)

        def tf():
            ia.attention_quant_q(inp.q, k8, ks, inp.v, bias=inp.bias, block_mask=inp.block_mask,
                                 v_scale=inp.v_scale, kv_valid=inp.kv_valid,
                                 granularity=wl.granularity, out=out, lse=lse, return_lse=True)

        ms = {}
        # device time alone: the same calls replayed from a CUDA graph, so that the
        # host's per-call work (argument checks, output allocation) is not in it
        ms["quantize_graph_ms"] = graph_ms(torch, tq)
        ms["attention_graph_ms"] = graph_ms(torch, ta)
        for key, fn in (("quantize_ms", tq), ("attention_ms", ta), ("quantize_k_ms", tk),
                        ("fused_q_attention_ms", tf)):
            for _ in range(3):
                fn()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(n):
                fn()
            e1.record()
            torch.cuda.synchronize()
            ms[key] = e0.elapsed_time(e1) / n
        ia.device_status()
        ops = algorithmic_ops(wl, kept)
        ms["attention_tops"] = ops / (ms["attention_ms"] * 1e-3) / 1e12
        ms["two_pass_path_ms"] = ms["quantize_ms"] + ms["attention_ms"]
        ms["fused_q_path_ms"] = ms["quantize_k_ms"] + ms["fused_q_attention_ms"]
        ms["shape"] = f"B{wl.B} H{wl.H} Sq{wl.Sq} Sk{wl.Sk} D{wl.D} {wl.dtype}"
        if kept is not None:
            ms["kept_tiles_per_row"] = kept
        res[name] = ms
        del inp, q8, k8, out
        torch.cuda.empty_cache()
    return res


def run_profile(args):
    """One kernel alone on a (possibly smaller) copy of its workload, for ncu."""
    import torch

    import __graft_entry__
    __graft_entry__.build()
    import int8_qk_quantized_gb300 as ia
    from workloads import WORKLOADS, make_inputs

    name = args.profile
    wl = WORKLOADS[{"sparse": "sparse", "sparse_fused_q": "sparse", "sdxl": "sdxl"}.get(name, "banded")]
    if args.heads:
        wl = wl.with_(H=args.heads)
    inp = make_inputs(wl, "cuda")
    g = wl.granularity
    q8, qs, k8, ks = ia.quantize_qk(inp.q, inp.k, kv_valid=inp.kv_valid, granularity=g)
    out, lse = ia.attention(q8, k8, qs, ks, inp.v, block_mask=inp.block_mask,
                            kv_valid=inp.kv_valid, return_lse=True, granularity=g)
    o2, l2 = out.clone(), lse.clone()
    fns = {
        # the head-dim-64 workload as the benchmark times it (default key split)
        "sdxl": lambda: ia.attention(q8, k8, qs, ks, inp.v, out=out, lse=lse, return_lse=True,
                                     granularity=g),
        "attention": lambda: ia.attention(q8, k8, qs, ks, inp.v, out=out, lse=lse, return_lse=True),
        "attention_bias": lambda: ia.attention(q8, k8, qs, ks, inp.v, bias=inp.bias, out=out,
                                               lse=lse, return_lse=True),
        "quantize": lambda: ia.quantize_qk(inp.q, inp.k),
        "merge": lambda: ia.merge_lse(out, lse, o2, l2, out=o2, lse_out=l2),
        "sparse": lambda: ia.attention(q8, k8, qs, ks, inp.v, block_mask=inp.block_mask,
                                       kv_valid=inp.kv_valid, out=out, lse=lse, return_lse=True),
    }
    # the block-sparse call with Q quantized in the kernel (16-bit Q rows in)
    fns["sparse_fused_q"] = lambda: ia.attention_quant_q(inp.q, k8, ks, inp.v, block_mask=inp.block_mask,
                                                         kv_valid=inp.kv_valid, out=out, lse=lse,
                                                         return_lse=True)
    if name == "rowmask":  # the materialised bf16 [1,1,Q,K] mask of the skirt bias (per-row path)
        m = inp.bias.to(torch.bfloat16).view(1, 1, 1, -1).expand(1, 1, wl.Sq, wl.Sk).contiguous()
        fns["rowmask"] = lambda: ia.attention(q8, k8, qs, ks, inp.v, mask=m, out=out, kv_splits=1)
    fn = fns[name]
    for _ in range(args.warmup):
        fn()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    ia.device_status()
    print(json.dumps({"profile": name, "workload": wl.name, "H": wl.H,
                      "ms_per_call": e0.elapsed_time(e1) / args.steps}), flush=True)


def time_prologue(ia, torch, names=("anima4k", "anima9k"), n=10):
    """RMSNorm + RoPE (split-half pairs, both weights) fused before the
    quantization, on the RoPE-model workloads: the quantize pass with and
    without it, and the fused-Q attention with and without it."""
    from workloads import WORKLOADS, make_inputs, norm_weight, rope_tables
    res = {}
    for name in names:
        wl = WORKLOADS[name]
        inp = make_inputs(wl, "cuda")
        cos, sin = (torch.from_numpy(t).cuda() for t in rope_tables(max(wl.Sq, wl.Sk), wl.D))
        wq, wk = (torch.from_numpy(norm_weight(wl.D, s)).cuda() for s in (1, 2))
        pro = ia.make_prologue(q_norm_weight=wq, k_norm_weight=wk, rope="split_half", cos=cos,
                               sin=sin)
        q8, qs, k8, ks = ia.quantize_qk(inp.q, inp.k, prologue=pro)
        out = torch.empty_like(inp.q)
        fns = {
            "quantize_qk_ms": lambda: ia.quantize_qk(inp.q, inp.k),
            "quantize_qk_prologue_ms": lambda: ia.quantize_qk(inp.q, inp.k, prologue=pro),
            "quantize_k_prologue_ms": lambda: ia.quantize_qk(None, inp.k, prologue=pro),
            "attention_ms": lambda: ia.attention(q8, k8, qs, ks, inp.v, v_scale=inp.v_scale,
                                                 out=out),
            "fused_q_attention_ms": lambda: ia.attention_quant_q(inp.q, k8, ks, inp.v,
                                                                 v_scale=inp.v_scale, out=out),
            "fused_q_prologue_attention_ms": lambda: ia.attention_quant_q(
                inp.q, k8, ks, inp.v, v_scale=inp.v_scale, out=out, prologue=pro),
        }
        ms = {}
        for key, fn in fns.items():
            for _ in range(3):
                fn()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(n):
                fn()
            e1.record()
            torch.cuda.synchronize()
            ms[key] = e0.elapsed_time(e1) / n
        ia.device_status()
        ms["two_pass_path_ms"] = ms["quantize_qk_prologue_ms"] + ms["attention_ms"]
        ms["fused_q_path_ms"] = ms["quantize_k_prologue_ms"] + ms["fused_q_prologue_attention_ms"]
        res[name] = ms
        del inp, q8, k8, out
        torch.cuda.empty_cache()
    return res


def time_mask_forms(ia, torch, q8, k8, qs, ks, v, bias, out, n=10):
    """The attn_mask forms of the comfy-kitchen int8_attention issue's table
    (The measurement) on the same 4096 x 33600 x 56 x 128 problem: ms per
    call and the ratio to the unmasked call."""
    import math
    Sq, Sk = q8.shape[2], k8.shape[2]
    b16 = bias.to(torch.bfloat16).view(1, 1, 1, -1)
    forms = {
        "none": {},
        "fp32 bias [K]": dict(bias=bias),
        "bf16 [1,1,1,K]": dict(mask=b16),
        "fp32 [1,1,1,K]": dict(mask=bias.view(1, 1, 1, -1)),
        "fp16 [1,1,1,K]": dict(mask=bias.to(torch.float16).view(1, 1, 1, -1)),
        "bf16 [1,1,Q,K] expanded": dict(mask=b16.expand(1, 1, Sq, Sk)),
        "bool [1,1,1,K]": dict(mask=(bias > math.log(1e-3)).view(1, 1, 1, -1)),
        "bf16 [1,1,Q,K] materialised (per-row path)": dict(mask=b16.expand(1, 1, Sq, Sk).contiguous()),
    }
    res = {}
    for name, kw in forms.items():
        def fn(kw=kw):
            ia.attention(q8, k8, qs, ks, v, out=out, kv_splits=1, **kw)
        for _ in range(3):
            fn()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(n):
            fn()
        e1.record()
        torch.cuda.synchronize()
        res[name] = {"ms": e0.elapsed_time(e1) / n}
    ia.device_status()
    for name in res:
        res[name]["vs_unmasked"] = res[name]["ms"] / res["none"]["ms"]
    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip timing the other four workloads")
    ap.add_argument("--profile", default=None,
                    choices=["attention", "attention_bias", "quantize", "merge", "sparse", "sparse_fused_q", "sdxl",
                             "rowmask"],
                    help="run one kernel alone, --steps times after --warmup (for ncu)")
    ap.add_argument("--heads", type=int, default=None, help="heads of the --profile case")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.impl == "reference":
        run_reference(args)
        return
    if args.profile:
        run_profile(args)
        return

    import torch

    ws, rank, local = dist_info()
    torch.cuda.set_device(local)
    pg = None
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        pg = dist

    import __graft_entry__
    __graft_entry__.build()
    import int8_qk_quantized_gb300 as ia
    from workloads import WORKLOADS, algorithmic_ops, make_inputs

    wl = WORKLOADS["banded"]
    B, H, Sq, Sk, D = wl.B, wl.H, wl.Sq, wl.Sk, wl.D
    lo, hi = wl.skirt_width, Sk - wl.skirt_width
    dev = torch.device("cuda", local)
    inp = make_inputs(wl, dev)
    q, k, v, bias = inp.q, inp.k, inp.v, inp.bias
    stream = torch.cuda.current_stream()

    # preallocated outputs: the step allocates nothing
    q8 = torch.empty(B, H, Sq, D, dtype=torch.int8, device=dev)
    k8 = torch.empty(B, H, Sk, D, dtype=torch.int8, device=dev)
    qs = torch.empty(B, H, Sq, device=dev)
    ks = torch.empty(B, H, Sk, device=dev)
    o_core = torch.empty(B, H, Sq, D, dtype=q.dtype, device=dev)
    o_l = torch.empty_like(o_core)
    o_r = torch.empty_like(o_core)
    l_core = torch.empty(B, H, Sq, device=dev)
    l_l = torch.empty_like(l_core)
    l_r = torch.empty_like(l_core)
    o_full = torch.empty_like(o_core)
    l_full = torch.empty_like(l_core)

    L = ia.load_library()
    import ctypes
    # a buffer for the K mean: with it the library runs its mean and code
    # kernels instead of the fused kernel (faster on this K)
    k_mu = torch.empty(B, H, D, dtype=torch.float32, device=dev)

    def quantize(qq, kk):
        st = (ctypes.c_int64 * 3)(*qq.stride()[:3])
        sk = (ctypes.c_int64 * 3)(*kk.stride()[:3])
        ia._check(L.ia_quantize_qk(ia._ptr(qq), ia._ptr(kk), ia.BF16, B, H, Sq, Sk, D, st, sk,
                                   ia.PER_TOKEN, 1, None, None, ia._ptr(q8), ia._ptr(k8),
                                   ia._ptr(qs), ia._ptr(ks), ia._ptr(k_mu), ia._stream(stream)))

    def attn(a, b_, bias_t, out, lse, vv):
        ia.attention(q8, k8[:, :, a:b_], qs, ks[:, :, a:b_], vv[:, :, a:b_], bias=bias_t,
                     out=out, lse=lse, return_lse=True, stream=stream)

    att_events = []

    def step(record=False, ins=None, outs=None):
        """One pass of the path on the compute stream: inputs (q, k, v, bias),
        outputs (o, lse); the quantized codes and partials are shared scratch."""
        qq, kk, vv, bb = ins if ins is not None else (q, k, v, bias)
        oc, lc = outs if outs is not None else (o_core, l_core)
        quantize(qq, kk)
        for (a, b_, bt, o_, l_) in ((lo, hi, None, oc, lc),
                                    (0, lo, bb[:lo], o_l, l_l),
                                    (hi, Sk, bb[hi:], o_r, l_r)):
            if record:
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(stream)
            attn(a, b_, bt, o_, l_, vv)
            if record:
                e1.record(stream)
                att_events.append((e0, e1, 4.0 * B * H * Sq * (b_ - a) * D))
        ia.merge_lse(oc, lc, o_l, l_l, out=oc, lse_out=lc, stream=stream)
        ia.merge_lse(oc, lc, o_r, l_r, out=oc, lse_out=lc, stream=stream)

    launches_per_step = 2 + 3 + 2

    for _ in range(args.warmup):
        step()
    ia.device_status()

    sampler = start_clock_sampler() if rank == 0 else None
    torch.cuda.synchronize()
    if pg:
        pg.barrier()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for _ in range(args.steps):
        step(record=True)
    t_end.record(stream)
    torch.cuda.synchronize()
    if pg:
        pg.barrier()
    clocks = stop_clock_sampler(sampler, local)
    ia.device_status()
    elapsed_ms = t_start.elapsed_time(t_end)
    att_ms = sum(e0.elapsed_time(e1) for e0, e1, _ in att_events)
    att_ops = sum(o for _, _, o in att_events)
    if pg:
        elapsed_ms = dist_max(elapsed_ms, pg, dev)
    ms_per_step = elapsed_ms / args.steps
    ops = algorithmic_ops(wl)
    value = weak_value(ws, ops, ms_per_step)

    # single calls over all keys: unmasked and with the bias
    def time_call(fn, n=20):
        for _ in range(3):
            fn()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / n

    unmasked_ms = time_call(lambda: ia.attention(q8, k8, qs, ks, v, out=o_full, lse=l_full,
                                                 return_lse=True, stream=stream))
    bias_ms = time_call(lambda: ia.attention(q8, k8, qs, ks, v, bias=bias, out=o_full,
                                             lse=l_full, return_lse=True, stream=stream))
    quant_ms = time_call(lambda: quantize(q, k))

    def step_fused_q():  # K quantized alone; each attention call quantizes Q itself
        sk_ = (ctypes.c_int64 * 3)(*k.stride()[:3])
        ia._check(L.ia_quantize_qk(None, ia._ptr(k), ia.BF16, B, H, Sq, Sk, D, None, sk_,
                                   ia.PER_TOKEN, 1, None, None, None, ia._ptr(k8), None,
                                   ia._ptr(ks), ia._ptr(k_mu), ia._stream(stream)))
        for (a, b_, bt, o_, l_) in ((lo, hi, None, o_core, l_core),
                                    (0, lo, bias[:lo], o_l, l_l),
                                    (hi, Sk, bias[hi:], o_r, l_r)):
            ia.attention_quant_q(q, k8[:, :, a:b_], ks[:, :, a:b_], v[:, :, a:b_], bias=bt,
                                 out=o_, lse=l_, return_lse=True, stream=stream)
        ia.merge_lse(o_core, l_core, o_l, l_l, out=o_core, lse_out=l_core, stream=stream)
        ia.merge_lse(o_core, l_core, o_r, l_r, out=o_core, lse_out=l_core, stream=stream)

    step_ms = time_call(step, n=10)
    step_fused_ms = time_call(step_fused_q, n=10)
    # the merge is short enough that Python launch overhead would dominate: time
    # 50 calls captured in a CUDA graph
    def time_graph(fn, n=50, reps=4):
        fn()
        torch.cuda.synchronize()
        gs = torch.cuda.Stream(device=dev)
        gs.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=gs):
            for _ in range(n):
                fn(gs)
        graph.replay()
        torch.cuda.synchronize()
        g0 = torch.cuda.Event(enable_timing=True)
        g1 = torch.cuda.Event(enable_timing=True)
        cur = torch.cuda.current_stream()  # replay() launches on the current stream
        g0.record(cur)
        for _ in range(reps):
            graph.replay()
        g1.record(cur)
        torch.cuda.synchronize()
        return g0.elapsed_time(g1) / (n * reps)

    merge_ms = time_graph(lambda st=stream: ia.merge_lse(o_l, l_l, o_r, l_r, out=o_full,
                                                         lse_out=l_full, stream=st))
    ia.device_status()

    # End to end: every step copies its inputs from pinned host memory to the
    # device and its output (o, lse) back. The copies run on their own streams,
    # double-buffered, so step i+1's inputs travel while step i computes and
    # step i's output returns while step i+1 computes.
    hq = q.cpu().pin_memory()
    hk = k.cpu().pin_memory()
    hv = v.cpu().pin_memory()
    hb = bias.cpu().pin_memory()
    host_in = (hq, hk, hv, hb)
    ins = [(q, k, v, bias), tuple(torch.empty_like(t) for t in (q, k, v, bias))]
    outs = [(o_core, l_core), (torch.empty_like(o_core), torch.empty_like(l_core))]
    host_out = [(torch.empty(o_core.shape, dtype=o_core.dtype).pin_memory(),
                 torch.empty(l_core.shape, dtype=torch.float32).pin_memory()) for _ in range(2)]
    e2e_steps = max(3, min(args.steps, 20))
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = sum(t.numel() * t.element_size() for t in host_out[0])
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)

    def e2e_run(n):
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_done = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]

        def copy_in(j):
            for t, ht in zip(ins[j], host_in):
                t.copy_(ht, non_blocking=True)
            ev_in[j].record(s_in)

        s_in.wait_stream(stream)
        s_out.wait_stream(stream)
        with torch.cuda.stream(s_in):
            copy_in(0)
        for i in range(n):
            j = i % 2
            stream.wait_event(ev_in[j])
            if i >= 2:
                stream.wait_event(ev_out[j])   # step i-2's output has left outs[j]
            step(ins=ins[j], outs=outs[j])
            ev_done[j].record(stream)
            if i + 1 < n:
                with torch.cuda.stream(s_in):
                    if i >= 1:
                        s_in.wait_event(ev_done[1 - j])  # step i-1 has read ins[1-j]
                    copy_in(1 - j)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_done[j])
                host_out[j][0].copy_(outs[j][0], non_blocking=True)
                host_out[j][1].copy_(outs[j][1], non_blocking=True)
                ev_out[j].record(s_out)
        stream.wait_stream(s_in)
        stream.wait_stream(s_out)

    e2e_run(2)
    torch.cuda.synchronize()
    if pg:
        pg.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_run(e2e_steps)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    if pg:
        e2e_ms = dist_max(e2e_ms, pg, dev)
    ia.device_status()
    # the pipelined copies gave the same answer as the plain step
    torch.cuda.synchronize()
    step(ins=ins[0], outs=outs[1])
    torch.cuda.synchronize()
    e2e_ok = bool(torch.equal(host_out[(e2e_steps - 1) % 2][0], outs[1][0].cpu()))

    hbm, bf16, bf16_sus, peak_kind = peaks()
    achieved = att_ops / (att_ms * 1e-3) / 1e12
    # compulsory bytes of the quantize pass: Q and K read once (16-bit), codes
    # written (int8), one fp32 scale per row and the fp32 K mean; a second read
    # of K (the codes need the mean first) is not counted
    quant_bytes = B * H * (Sq + Sk) * D * (2 + 1) + B * H * (Sq + Sk) * 4 + B * H * D * 4
    # The second bound of the attention launches: the softmax's ALU and MUFU
    # work, one exp2 per score at the measured 32 ex2/clk/SM, and its issue
    # slots at 4 warp instructions per clock per SM. Per 8 scores of a 128-key
    # row the fast path issues 2 shared loads of k scales, 4 f32x2 multiplies,
    # 4 three-input maxima, 4 f32x2 FMAs, 8 ex2, 4 f32x2 adds (row sum) and 4
    # packing conversions: 30 instructions, 3.75 per score.
    sm_count = torch.cuda.get_device_properties(dev).multi_processor_count
    sm_mhz = (clocks or {}).get("sm_mhz") or 2070.0
    scores = att_ops / (4 * D) / args.steps  # one score per 4*D operations
    per_sec = sm_count * sm_mhz * 1e6
    alu = {"bound": "alu", "scores_per_step": scores, "ex2_per_clk_per_sm": 32,
           "issue_per_score": 3.75, "sm_count": sm_count, "sm_mhz": sm_mhz,
           "mufu_ms": scores / (32 * per_sec) * 1e3,
           "issue_ms": scores * 3.75 / (128 * per_sec) * 1e3,
           "tensor_ms": att_ops / args.steps / (bf16 * 1e12) * 1e3,
           "attention_ms": att_ms / args.steps}
    alu["frac_mufu"] = alu["mufu_ms"] / alu["attention_ms"]
    alu["frac_issue"] = alu["issue_ms"] / alu["attention_ms"]
    if rank != 0:
        if pg:
            pg.destroy_process_group()
        return
    others = None if args.no_extra else time_workloads(ia, torch)
    mask_forms = None if args.no_extra else time_mask_forms(ia, torch, q8, k8, qs, ks, v, bias,
                                                            o_full)
    prologue = None if args.no_extra else time_prologue(ia, torch)
    cpu = None if args.no_cpu_baseline else cpu_baseline()
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": value / (ops / (PAGE_SPLIT_MS * 1e-3) / 1e12),
        "vs_baseline_ref": "RTX 5090 core+skirt split of the same problem, 11.05 ms "
                           "(comfy-kitchen issue #177); another machine: context only",
        "dtype": "int8 QK (exact, fp16-coded MMA) / bf16 PV, fp32 accumulate",
        "data": "synthetic",
        "config": {"workload": "banded cross-window attention B1 H56 Q4096 K33600 D128 bf16: "
                               "quantise Q/K, core 20160 keys unmasked + two 6720-key skirts "
                               "with the per-key raised-cosine bias, LSE merges",
                   "B": B, "H": H, "Sq": Sq, "Sk": Sk, "D": D,
                   "l2": "no flush: inputs (q+k+v = 1.02 GB) are larger than L2"},
        "calls_ms": {"unmasked_all_keys": unmasked_ms, "bias_all_keys": bias_ms,
                     "bias_over_unmasked": bias_ms / unmasked_ms, "quantize_qk": quant_ms,
                     "merge_lse": merge_ms,
                     "step_two_pass": step_ms, "step_fused_q": step_fused_ms,
                     "unmasked_tops": ops / (unmasked_ms * 1e-3) / 1e12,
                     "bias_tops": ops / (bias_ms * 1e-3) / 1e12,
                     "quantize_gbs": quant_bytes / (quant_ms * 1e-3) / 1e9},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": bf16, "unit": "TFLOP/s",
                     "frac": achieved / bf16,
                     "traffic": attn_traffic_per_launch(H, Sq, [hi - lo, lo, Sk - hi], D),
                     "algorithmic_bytes": sum(H * (Sq * D * 3 + Sq * 8 + n * (D * 3 + 4))
                                              for n in (hi - lo, lo, Sk - hi)) / 3,
                     "kernel": "attn_fwd_kernel (CTA pairs, QS=2, BN=128, D=128); per launch = mean of "
                               "the step's three attention launches",
                     "peak_source": f"{peak_kind} bf16 dense burst (MEASURED_PEAKS.json)",
                     "frac_of_sustained": achieved / bf16_sus if bf16_sus else None,
                     "second_bound": alu},
        "e2e": {"value": weak_value(ws, ops, e2e_ms), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "copies": "pinned host <-> device every step on two copy streams, double-"
                          "buffered so that they overlap the neighbouring steps' kernels",
                "output_matches_device_step": e2e_ok},
        "workloads": others,
        "mask_forms": mask_forms,
        "prologue": prologue,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()


if __name__ == "__main__":
    main()

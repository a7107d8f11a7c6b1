"""Benchmark: causal attention forward + backward on one GB300 (per rank).

One step = the whole hot path over one batch of synthetic input:
  permute Q, K, V, dO to the partition's worker-major order
  -> forward over every (worker, ring step) chunk pair in one launch
     (online-softmax merge of the ring steps on chip)
  -> backward (D preprocess, recomputation kernel, dQ conversion)
  -> un-permute O, LSE, dQ, dK, dV to natural order.
Workload: Llama-7B attention layer at N = 131072 (B=1, H=32, d=128, causal,
bf16 N(0,1) inputs from seed 2 with 1% of query rows x8), P = 8 striped.
Throughput counts causal FLOPs only: fwd 4 d pairs, bwd 10 d pairs,
pairs = B H N (N+1) / 2.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
Under torchrun each rank runs its own replica (weak scaling); rank 0 prints
one JSON line.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "causal attn fwd+bwd TFLOPS (bf16, 1 GB300) and % of dense BF16 tensor peak"
WORKLOAD = "llama7b_128k"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def reduce_max(x: float, device=None) -> float:
    """Max of a per-rank value over the default process group (identity when
    no group is initialised).  Used only for timing, never on the data path."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


class ClockSampler:
    """nvidia-smi clock / throttle sampling during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = [r for r in csv.reader(io.StringIO(self.out or "")) if len(r) >= 9]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        sm = sorted(float(r[1]) for r in rows)
        mx = max(float(r[2]) for r in rows)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4)
                          if r[5 + i].strip().lower() == "active"})
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": mx, "reasons": reasons,
                "samples": len(rows)}


KERNEL_SOURCES = {
    "attn_bwd_kernel": ("dfa_bwd.cu", "dfa_ptx.cuh", "dfa_params.h", "dfa_api.cu"),
    "attn_fwd_kernel": ("dfa_fwd.cu", "dfa_ptx.cuh", "dfa_params.h", "dfa_api.cu"),
}


def source_hash(kernel: str) -> str:
    """First 16 hex digits of the SHA-256 over the sources that shape a
    kernel's launch (its .cu, the PTX helpers, the parameter structs and the
    host code that orders its work units), in a fixed order."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "long_context_flashattention_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def kernel_traffic(summary: str, kernel: str):
    """DRAM bytes (read + write) per launch from a committed ncu summary
    (`key: value` lines), or None unless it was taken on the current sources
    of the kernel."""
    p = os.path.join(ROOT, "profiles", summary)
    if not os.path.exists(p):
        return None
    fields = {}
    with open(p) as f:
        for line in f:
            if ":" in line and not line.startswith(("#", "|", " ")):
                key, _, val = line.partition(":")
                fields[key.strip()] = val.strip().strip("`")
    if fields.get("source_sha256_16") != source_hash(kernel):
        return None
    try:
        return int(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def schedule_summary(N: int, P: int, kind: str) -> dict:
    """How evenly the workload's partition spreads the causal (query, key)
    pairs over a P-worker ring (dfa_make_schedule, host only; Striped
    Attention Guide, "Workload Balance Theorem"; DistFlashAttn Guide, "The
    Causal Imbalance Crisis"): eta_slots is the share of (worker, step) slots
    with any work, eta_flops the lockstep utilisation, total pairs over P
    times the sum of each step's largest per-worker load."""
    from long_context_flashattention_gb300 import dfa
    s = dfa.make_schedule(N, P, kind, items=False)
    return {"P": P, "partition": kind, "total_pairs": s["total_pairs"],
            "eta_slots": round(s["eta_slots"], 6), "eta_flops": round(s["eta_flops"], 6)}


# ----------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------
def run_gpu(args):
    from long_context_flashattention_gb300 import dfa
    from long_context_flashattention_gb300.inputs import WORKLOADS, make_workload

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    w = WORKLOADS[args.workload]
    if args.heads:
        # profiling aid: the same sequence and partition with fewer heads
        # (heads are independent units processed one after another, so a
        # launch's work and traffic scale with the head count)
        import dataclasses
        w = dataclasses.replace(w, name=f"{w.name} (heads {args.heads})", Hq=args.heads,
                                Hkv=max(1, args.heads * w.Hkv // w.Hq))
    P, kind = w.P, w.partitions[0]
    dfa.lib()

    # inputs, resident in HBM before timing (larger than L2: 1 GiB per tensor)
    q, k, v, do = make_workload(w)
    host = [t.pin_memory() for t in (q, k, v, do)]
    qg, kg, vg, dog = (t.to(dev) for t in host)
    bufs = {
        "perm": [torch.empty_like(t) for t in (qg, kg, vg, dog)],
        "o": torch.empty_like(qg), "lse": torch.empty(w.B, w.Hq, w.N, device=dev),
        "dq": torch.empty_like(qg), "dk": torch.empty_like(kg), "dv": torch.empty_like(vg),
        "out": [torch.empty_like(qg), torch.empty(w.B, w.Hq, w.N, device=dev),
                torch.empty_like(qg), torch.empty_like(kg), torch.empty_like(vg)],
    }
    desc = dfa.desc_for(qg, kg, P=P, partition=kind)
    ws = dfa.new_workspace(desc, dfa.OP_BWD, dev)
    stream = torch.cuda.current_stream(dev)
    ev = {n: torch.cuda.Event(enable_timing=True) for n in ("f0", "f1", "b0", "b1")}

    def step(inputs, record=False):
        pq, pk, pv, pdo = bufs["perm"]
        for src, dst in zip(inputs, bufs["perm"]):
            dfa.permute(src, P, kind, out=dst)
        if record:
            ev["f0"].record(stream)
        dfa.attn_fwd(pq, pk, pv, P=P, partition=kind, ws=ws, out=bufs["o"], lse=bufs["lse"])
        if record:
            ev["f1"].record(stream)
            ev["b0"].record(stream)
        dfa.attn_bwd(pq, pk, pv, bufs["o"], pdo, bufs["lse"], P=P, partition=kind, ws=ws,
                     dq=bufs["dq"], dk=bufs["dk"], dv=bufs["dv"])
        if record:
            ev["b1"].record(stream)
        for src, dst in zip((bufs["o"], bufs["lse"], bufs["dq"], bufs["dk"], bufs["dv"]),
                            bufs["out"]):
            dfa.permute(src, P, kind, inverse=True, out=dst)

    # permutes in, forward, backward (preprocess, main kernel, dQ conversion;
    # with query blocking above 64K rows per head also dK and dV conversions),
    # permutes out
    blocked = w.N * (w.Hq // w.Hkv) > 131072
    launches_per_step = 4 + 1 + (5 if blocked else 3) + 5

    def barrier():
        torch.cuda.synchronize(dev)
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    for _ in range(args.warmup):
        step((qg, kg, vg, dog))
    dfa.stream_status(ws)
    barrier()

    fwd_ms, bwd_ms = [], []
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier()
        t0.record(stream)
        for _ in range(args.steps):
            step((qg, kg, vg, dog), record=True)
            # per-call events; read after the region (no sync inside)
            fwd_ms.append((ev["f0"], ev["f1"]))
            bwd_ms.append((ev["b0"], ev["b1"]))
            ev = {n: torch.cuda.Event(enable_timing=True) for n in ("f0", "f1", "b0", "b1")}
        t1.record(stream)
        barrier()
    dfa.stream_status(ws)
    step_ms = t0.elapsed_time(t1) / args.steps
    fwd_call_ms = sum(a.elapsed_time(b) for a, b in fwd_ms) / len(fwd_ms)
    bwd_call_ms = sum(a.elapsed_time(b) for a, b in bwd_ms) / len(bwd_ms)
    step_ms = reduce_max(step_ms, dev)

    if args.only_step:
        pk, src = peaks()
        flops = w.flops_fwd + w.flops_bwd
        print(json.dumps({"only_step": True, "workload": w.name, "ms_per_step": round(step_ms, 3),
                          "fwd_ms": round(fwd_call_ms, 3), "bwd_ms": round(bwd_call_ms, 3),
                          "tflops": round(flops / (step_ms * 1e-3) / 1e12, 2),
                          "clocks": clk.summary()}), flush=True)
        return

    # end to end through the C ABI with HOST buffers (dfa_attn_steps_host, the
    # steps of the timed region in one call): every step uploads its inputs
    # from pinned host memory and downloads O, LSE, dQ, dK, dV, in groups of
    # key/value heads whose copies overlap the compute, across step boundaries
    h_out = tuple(torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in bufs["out"])
    h_desc = dfa.make_desc(w.B, w.Hq, w.Hkv, w.N, w.d, P=P, partition=kind)
    h_ws = dfa.step_host_workspace(h_desc, 0, dev)
    e2e_steps = max(1, min(args.steps, 64))  # the call takes at most 64 steps

    def e2e_steps_call(n):
        dfa.attn_steps_host([tuple(host)] * n, P=P, partition=kind, outs=[h_out] * n, ws=h_ws)

    e2e_steps_call(1)
    dfa.stream_status(h_ws)
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_steps_call(e2e_steps)
    e1.record(stream)
    barrier()
    dfa.stream_status(h_ws)
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    h2d = sum(t.numel() * t.element_size() for t in host)
    d2h = sum(t.numel() * t.element_size() for t in h_out)
    del h_ws

    # the same copies alone, one after another on one stream (what the
    # overlap hides)
    torch.cuda.synchronize(dev)
    e0.record(stream)
    for h, dsrc in zip(host, bufs["perm"]):
        dsrc.copy_(h, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    h2d_ms = e0.elapsed_time(e1)
    e0.record(stream)
    for h, dres in zip(h_out, bufs["out"]):
        h.copy_(dres, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    d2h_ms = e0.elapsed_time(e1)

    # standalone LSE merge at this workload's size (k = P partials per row;
    # at most 4M rows, 17 GB of partials at k = 8, so that the largest
    # workload's merge stays within memory beside its step buffers)
    rows = min(w.B * w.Hq * w.N, 1 << 22)
    parts_o = torch.randn(P, rows, w.d, device=dev)
    parts_l = 4 * torch.randn(P, rows, device=dev)
    m_out = torch.empty(rows, w.d, dtype=torch.bfloat16, device=dev)
    m_lse = torch.empty(rows, device=dev)
    for _ in range(3):
        dfa.lse_merge(parts_o, parts_l, out_fp32=False, o_out=m_out, lse_out=m_lse)
    m0 = torch.cuda.Event(enable_timing=True)
    m1 = torch.cuda.Event(enable_timing=True)
    reps = 10
    torch.cuda.synchronize(dev)
    m0.record(stream)
    for _ in range(reps):
        dfa.lse_merge(parts_o, parts_l, out_fp32=False, o_out=m_out, lse_out=m_lse)
    m1.record(stream)
    torch.cuda.synchronize(dev)
    merge_ms = m0.elapsed_time(m1) / reps
    merge_bytes = rows * (P * (4 * w.d + 4) + (2 * w.d + 4))
    del parts_o, parts_l

    # the same merge at the grouped-query 64K workload's size: B2 Hq32 N65536
    # rows (as many as here), k = 16 partials (P = 16)
    rows16, k16 = 2 * 32 * 65536, 16
    parts_o = torch.randn(k16, rows16, w.d, device=dev)
    parts_l = 4 * torch.randn(k16, rows16, device=dev)
    m_out = torch.empty(rows16, w.d, dtype=torch.bfloat16, device=dev)
    m_lse = torch.empty(rows16, device=dev)
    for _ in range(3):
        dfa.lse_merge(parts_o, parts_l, out_fp32=False, o_out=m_out, lse_out=m_lse)
    torch.cuda.synchronize(dev)
    m0.record(stream)
    for _ in range(reps):
        dfa.lse_merge(parts_o, parts_l, out_fp32=False, o_out=m_out, lse_out=m_lse)
    m1.record(stream)
    torch.cuda.synchronize(dev)
    merge16_ms = m0.elapsed_time(m1) / reps
    merge16_bytes = rows16 * (k16 * (4 * w.d + 4) + (2 * w.d + 4))
    del parts_o, parts_l, m_out, m_lse

    # the plain permute of Q into worker-major order
    p_out = torch.empty_like(qg)
    for _ in range(3):
        dfa.permute(qg, P, kind, out=p_out)
    torch.cuda.synchronize(dev)
    m0.record(stream)
    for _ in range(reps):
        dfa.permute(qg, P, kind, out=p_out)
    m1.record(stream)
    torch.cuda.synchronize(dev)
    perm_ms = m0.elapsed_time(m1) / reps
    perm_bytes = 2 * qg.numel() * qg.element_size()
    del p_out

    # permute fused with the rotary embedding at global positions, on Q
    r_out = torch.empty_like(qg)
    for _ in range(3):
        dfa.permute_rope(qg, P, kind, out=r_out)
    torch.cuda.synchronize(dev)
    m0.record(stream)
    for _ in range(reps):
        dfa.permute_rope(qg, P, kind, out=r_out)
    m1.record(stream)
    torch.cuda.synchronize(dev)
    rope_ms = m0.elapsed_time(m1) / reps
    rope_bytes = 2 * qg.numel() * qg.element_size()
    del r_out

    # the ring schedule on one GPU (P workers, K/V hand-over on a second stream)
    n = w.N // P
    pq, pk, pv = bufs["perm"][:3]
    qc, kc, vc = ([t[:, :, p * n:(p + 1) * n].contiguous() for p in range(P)]
                  for t in (pq, pk, pv))
    slots = [torch.empty(4 * kc[0].numel(), dtype=torch.bfloat16, device=dev) for _ in range(P)]
    outs = dfa.ring_fwd(qc, kc, vc, kind, slots=slots)
    ring_ws = dfa.new_workspace(dfa.make_desc(w.B, w.Hq, w.Hkv, w.N, w.d, P=P, partition=kind),
                                dfa.OP_RING_FWD, dev)

    def timed(fn, rep=2):
        torch.cuda.synchronize(dev)
        m0.record(stream)
        for _ in range(rep):
            fn()
        m1.record(stream)
        torch.cuda.synchronize(dev)
        return m0.elapsed_time(m1) / rep

    ring_ov = timed(lambda: dfa.ring_fwd(qc, kc, vc, kind, slots=slots, outs=outs, ws=ring_ws))
    ring_se = timed(lambda: dfa.ring_fwd(qc, kc, vc, kind, slots=slots, outs=outs, ws=ring_ws,
                                         overlap=False))

    def copies_alone():
        for _ in range(P - 1):
            for p in range(P):
                slots[p][:kc[0].numel()].copy_(kc[(p - 1) % P].view(-1))
                slots[p][kc[0].numel():2 * kc[0].numel()].copy_(vc[(p - 1) % P].view(-1))

    ring_cp = timed(copies_alone)
    del qc, kc, vc, slots, outs, ring_ws

    # split-KV decoding: one new token per head against this workload's K/V as the cache
    dq_in = qg[:, :, -1:].contiguous()
    dec_out = dfa.decode(dq_in, kg, vg, split_len=1024)
    dec_ms = timed(lambda: dfa.decode(dq_in, kg, vg, split_len=1024, out=dec_out[0],
                                      lse=dec_out[1]), rep=10)
    dec_bytes = 2 * kg.numel() * kg.element_size()
    del dq_in, dec_out

    pk, src = peaks()
    flops = w.flops_fwd + w.flops_bwd
    value = flops * world / (step_ms * 1e-3) / 1e12
    bwd_tflops = w.flops_bwd / (bwd_call_ms * 1e-3) / 1e12
    fwd_tflops = w.flops_fwd / (fwd_call_ms * 1e-3) / 1e12
    peak_s = pk["bf16_tflops_sustained"]
    merge_gbs = merge_bytes / (merge_ms * 1e-3) / 1e9
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(step_ms, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16, 1% of query rows x8)",
        "config": {"workload": f"{w.name} causal, P={P} {kind} partition, fused ring steps",
                   "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "N": w.N, "d": w.d, "P": P,
                   "partition": kind, "per_rank_batch": w.B,
                   "l2": "inputs larger than L2 (1 GiB per tensor), no flush"},
        "pct_of_peak": round(100 * value / world / pk["bf16_tflops"], 2),
        "pct_of_peak_basis": f"bf16_tflops {pk['bf16_tflops']} ({src} dense bf16 GEMM, burst)",
        "pct_of_peak_sustained": round(100 * value / world / peak_s, 2),
        "pct_of_peak_sustained_basis": f"bf16_tflops_sustained {peak_s} ({src}, seconds-long "
                                       f"loop under the power cap)",
        "fwd_tflops": round(fwd_tflops, 2),
        "bwd_tflops": round(bwd_tflops, 2),
        "fwd_ms": round(fwd_call_ms, 3),
        "bwd_ms": round(bwd_call_ms, 3),
        "roofline": {
            "kernel": "dfa::bwd::attn_bwd_kernel (timed over the dfa_attn_bwd call: D "
                      "preprocess + main kernel + dQ convert)",
            "bound": "tensor", "achieved": round(bwd_tflops, 2), "peak": peak_s,
            "unit": "TFLOP/s", "frac": round(bwd_tflops / peak_s, 4),
            "peak_source": f"{src} bf16_tflops_sustained",
            # the committed DRAM capture covers the 128K workload only
            "traffic": (kernel_traffic("attn_bwd_kernel_llama7b_128k_traffic.md",
                                       "attn_bwd_kernel")
                        if args.workload == "llama7b_128k" and not args.heads else None),
        },
        "merge": {"kernel": "dfa::lse_merge_kernel", "k": P, "rows": rows,
                  "bytes": merge_bytes, "ms": round(merge_ms, 4),
                  "achieved": round(merge_gbs, 1), "peak": pk["hbm_gbs"], "unit": "GB/s",
                  "frac": round(merge_gbs / pk["hbm_gbs"], 4)},
        "merge_k16": {"kernel": "dfa::lse_merge_kernel", "k": k16, "rows": rows16,
                      "size": "grouped-query attention B2 Hq32 N65536 output rows, P = 16",
                      "bytes": merge16_bytes, "ms": round(merge16_ms, 4),
                      "achieved": round(merge16_bytes / (merge16_ms * 1e-3) / 1e9, 1),
                      "peak": pk["hbm_gbs"], "unit": "GB/s",
                      "frac": round(merge16_bytes / (merge16_ms * 1e-3) / 1e9 / pk["hbm_gbs"],
                                    4)},
        "permute": {"kernel": "dfa::permute_kernel", "tensor": "Q", "bytes": perm_bytes,
                    "ms": round(perm_ms, 4),
                    "achieved": round(perm_bytes / (perm_ms * 1e-3) / 1e9, 1),
                    "peak": pk["hbm_gbs"], "unit": "GB/s",
                    "frac": round(perm_bytes / (perm_ms * 1e-3) / 1e9 / pk["hbm_gbs"], 4)},
        "rope_permute": {"kernel": "dfa::permute_rope_kernel", "tensor": "Q",
                         "bytes": rope_bytes, "ms": round(rope_ms, 4),
                         "achieved": round(rope_bytes / (rope_ms * 1e-3) / 1e9, 1),
                         "peak": pk["hbm_gbs"], "unit": "GB/s",
                         "frac": round(rope_bytes / (rope_ms * 1e-3) / 1e9 / pk["hbm_gbs"], 4)},
        "schedule": schedule_summary(w.N, P, kind),
        "ring_fwd": {"P": P, "partition": kind, "ms_overlap": round(ring_ov, 3),
                     "ms_serial": round(ring_se, 3), "ms_copies_alone": round(ring_cp, 3),
                     "tflops_overlap": round(w.flops_fwd / (ring_ov * 1e-3) / 1e12, 2),
                     "copy_hidden_frac": round(max(0.0, ring_se - ring_ov) / ring_cp, 3)
                     if ring_cp > 0 else None},
        "decode": {"kernel": "dfa::dec::decode_split_kernel + lse_merge", "T": 1,
                   "L": w.N, "split_len": 1024, "bytes": dec_bytes, "ms": round(dec_ms, 4),
                   "achieved": round(dec_bytes / (dec_ms * 1e-3) / 1e9, 1),
                   "peak": pk["hbm_gbs"], "unit": "GB/s",
                   "frac": round(dec_bytes / (dec_ms * 1e-3) / 1e9 / pk["hbm_gbs"], 4)},
        "e2e": {"value": round(flops / (e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                "ms_per_step": round(e2e_ms, 3), "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "call": "dfa_attn_steps_host (the timed steps in one call; pinned host "
                        "buffers, groups of key/value heads, copies on two streams beside "
                        "the compute and across step boundaries)", "steps": e2e_steps,
                "h2d_alone_ms": round(h2d_ms, 3), "d2h_alone_ms": round(d2h_ms, 3),
                "h2d_gbs": round(h2d / (h2d_ms * 1e-3) / 1e9, 1),
                "d2h_gbs": round(d2h / (d2h_ms * 1e-3) / 1e9, 1)},
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clk.summary(),
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(q, k, v, do, w, budget_s=args.cpu_seconds)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------
# CPU oracle arm (baseline / reference)
# ----------------------------------------------------------------------------
def cpu_baseline(q, k, v, do, w, budget_s=15.0):
    """The fp64 oracle, as it stands, on the host cores: forward and dQ of
    seeded sampled query rows of the same workload, in batches until the time
    budget is used.  FLOPs counted: 4 d (i+1) per forward row and 6 d (i+1)
    per dQ row (scores, dP and dQ), i the row's position."""
    import numpy as np

    import oracle
    from long_context_flashattention_gb300.inputs import sample_rows
    cores = oracle.num_threads()
    rows_all = np.array(sample_rows(w.B, w.Hq, w.N, 1 << 16, seed=w.seed + 2000))
    rng = np.random.default_rng(w.seed)
    rng.shuffle(rows_all)
    done, flops, t_used, batch = 0, 0.0, 0.0, 64
    while t_used < budget_s and done < len(rows_all):
        r = rows_all[done:done + batch]
        t0 = time.perf_counter()
        oracle.attn_fwd(q, k, v, rows=r)
        oracle.attn_bwd_q_rows(q, k, v, do, r)
        t_used += time.perf_counter() - t0
        i = (r % w.N) + 1
        flops += float((4 * w.d * i).sum() + (6 * w.d * i).sum())
        done += len(r)
        batch = min(batch * 2, 512)
    value = flops / t_used / 1e12
    # the whole oracle (forward and every gradient) on the tiny workload, in full
    from long_context_flashattention_gb300.inputs import WORKLOADS, make_workload
    tw = WORKLOADS["tiny"]
    tq, tk, tv, tdo = make_workload(tw)
    t0 = time.perf_counter()
    oracle.attn_fwd(tq, tk, tv)
    oracle.attn_bwd(tq, tk, tv, tdo)
    tiny_s = time.perf_counter() - t0
    return {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
            "sample": f"{done} seeded sampled query rows of {w.name}: fp64 forward row + dQ "
                      f"row each ({t_used:.1f} s)",
            "seconds": round(t_used, 2),
            "extrapolated_full_s": round((w.flops_fwd + w.flops_bwd) / (value * 1e12), 1),
            "extrapolated_basis": "forward and backward FLOPs of the whole workload at the "
                                  "sampled rows' rate (extrapolated, not run)",
            "tiny_full_s": round(tiny_s, 4),
            "tiny_full_tflops": round((tw.flops_fwd + tw.flops_bwd) / tiny_s / 1e12, 6)}


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    from long_context_flashattention_gb300.inputs import WORKLOADS, make_workload
    w = WORKLOADS[args.workload]
    q, k, v, do = make_workload(w)
    per = []
    for _ in range(args.warmup):
        cpu_baseline(q, k, v, do, w, budget_s=2.0)
    t_total = 0.0
    for _ in range(args.steps):
        t0 = time.perf_counter()
        cb = cpu_baseline(q, k, v, do, w, budget_s=args.cpu_seconds / max(1, args.steps))
        t_total += time.perf_counter() - t0
        per.append(cb["value"])
    value = sum(per) / len(per)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * t_total / args.steps, 1), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{w.name} causal, P={w.P} {w.partitions[0]} partition",
                   "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "N": w.N, "d": w.d},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cb["cores"],
                         "kind": "oracle", "sample": cb["sample"]},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="dfa", choices=["dfa", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only-step", action="store_true",
                    help="time the step only (no end-to-end, merge, permute, ring, decode legs, "
                         "no CPU baseline): the command the profiler captures run")
    ap.add_argument("--heads", type=int, default=0,
                    help="profiling aid: override the workload's query heads (key/value heads "
                         "scaled alike)")
    ap.add_argument("--workload", default=WORKLOAD,
                    help="workload name from inputs.WORKLOADS (default: the 128K Llama-7B layer)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()

"""Benchmark of the multi-tenant LoRA decode layer on GB300 (one JSON line).

A "step" is one Llama-3.1-8B-shaped decoder layer's four projections (qkv,
o, gate_up, down), each a full pass of the hot path through the C ABI's fused
entry (per-token quantizer, multi-adapter shrink, tcgen05 GEMM with the LoRA
epilogue: for a few tokens one persistent kernel per projection, otherwise
the shrink grid and the GEMM as its programmatic dependent), replayed as one
CUDA graph. The L2 cache is flushed between steps (a write and a read of
buffers twice its size) outside the timed events.

Default workload: M = 1 decode token, one tenant with a rank-64 adapter, FP8
E4M3 weights with per-channel scales and per-token FP8 activations. Measured
in the same run: 32 tenants (M = 32, one distinct rank-64 adapter per token)
with bf16 and with stored FP8 adapters, an NVFP4 base at several M and ranks,
multi-slice qkv / gate_up, the wide-batch layers against the tensor peak,
per-projection exposure controls, and the oracle on the host cores.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload 8b_m1_fp8|8b_m32_fp8|8b_m1_nvfp4|...]

Under torchrun (N > 1) every rank runs an independent replica on its own GPU
(the layer needs no exchange between GPUs); rank 0 prints the line with the
slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import subprocess
import sys
import tempfile
import time

# The oracle's workers run single-threaded (one process per core) so that
# "cores" is exact.
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fused FP8/NVFP4+LoRA layer µs @M=1, tokens/s @32 tenants, % HBM roofline"
PROJ8B = (("qkv", 4096, 6144), ("o", 4096, 4096), ("gate_up", 4096, 28672), ("down", 14336, 4096))
PROJ70B = (("qkv", 8192, 10240), ("o", 8192, 8192), ("gate_up", 8192, 57344), ("down", 28672, 8192))
# wide token tiles (tensor-bound): (name, projections, M, fmt, L, r, idx_mode, mask_mode, n_decode, description)
LARGE_WORKLOADS = (
    ("70b_prefill2048_fp8", PROJ70B, 2112, 0, 512, 16, "zipf", "prefill_chunk", 64,
     "Llama-3.1-70B layer, 64 decode tokens (mask 0) + one 2048-token prefill chunk (mask 1, one adapter), "
     "512 resident rank-16 adapters, Zipf(1.1) indices, FP8"),
    ("8b_m512_nvfp4", PROJ8B, 512, 1, 128, 64, "zipf", "all", 0,
     "Llama-3.1-8B layer, M=512, NVFP4, 128 resident rank-64 adapters, Zipf(1.1) indices"),
)

WORKLOADS = {
    # name: (M, fmt, L, r, idx_mode, description)
    "8b_m1_fp8": (1, 0, 1, 64, "single",
                  "Llama-3.1-8B decode layer (qkv 4096->6144, o 4096->4096, gate_up 4096->28672, "
                  "down 14336->4096), M=1, one tenant rank-64 bf16 adapter, FP8 E4M3 per-channel weights, "
                  "per-token FP8 activations"),
    "8b_m32_fp8": (32, 0, 32, 64, "per_token",
                   "Llama-3.1-8B decode layer, M=32 tokens, 32 tenants each with a distinct rank-64 adapter, FP8"),
    "8b_m1_nvfp4": (1, 1, 128, 64, "zipf",
                    "Llama-3.1-8B decode layer, M=1, NVFP4 weights/activations, 128 resident rank-64 adapters"),
    "8b_m32_nvfp4": (32, 1, 128, 64, "zipf",
                     "Llama-3.1-8B decode layer, M=32, NVFP4, 128 resident rank-64 adapters, Zipf(1.1) indices"),
}


def csrc_sha256(files=None) -> str:
    """sha256 over the named files of the kernel sources (all of them by
    default), in name order."""
    h = hashlib.sha256()
    d = os.path.join(ROOT, "precision_gemm_token_gb300", "csrc")
    for f in sorted(files or os.listdir(d)):
        with open(os.path.join(d, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()


def read_profile_traffic(workload: str, kernel: str = "gemm_gate_up"):
    """dram bytes per launch of the dominant kernel from the committed ncu
    summary, if it was taken on the current kernel sources."""
    path = os.path.join(ROOT, "profiles", f"{kernel}_{workload}.md")
    if not os.path.exists(path):
        return None
    txt = open(path).read()
    m = re.search(r"dram_bytes_per_launch:\s*([0-9.eE+]+)", txt)
    # the hash of the files the kernel is compiled from (listed), else of all
    # kernel sources
    srcs = re.search(r"kernel_sources:\s*([\w. ]+)", txt)
    s = re.search(r"sources_sha256:\s*([0-9a-f]+)", txt) or re.search(r"csrc_sha256:\s*([0-9a-f]+)", txt)
    files = srcs.group(1).split() if srcs else None
    if not m or not s or s.group(1) != csrc_sha256(files):
        return None
    return float(m.group(1))


# ----------------------------------------------------------------------------
# distributed plumbing (replicas only: one barrier and one max-reduction)
# ----------------------------------------------------------------------------
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if os.environ.get("EPILORA_BENCH_BACKEND", "nccl") == "nccl" else "gloo"
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, world: int, device) -> float:
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------
# clocks sampled during the timed region
# ----------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for nm, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(nm)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------
def algorithmic_bytes(M, K, N, fmt, r, n_distinct, with_adapter=True):
    """Bytes a perfect kernel must move for one projection (see the design
    notes): weight codes + weight scales + bf16 X + bf16 Y + per distinct
    active adapter its A (r x K) and B slice (N x r) in bf16 + S written and
    read once (fp32) + quantized activations written and read once."""
    wbytes = N * K if fmt == 0 else N * K // 2 + N * K // 16
    wscale = N * 4 if fmt == 0 else 4
    xq = M * K if fmt == 0 else M * K // 2 + M * K // 16
    b = wbytes + wscale + M * K * 2 + M * N * 2 + 2 * xq
    if with_adapter:
        b += n_distinct * (r * K * 2 + N * r * 2) + 2 * M * r * 4
    return b


def gemm_kernel_bytes(M, K, N, fmt, r, n_distinct):
    """Algorithmic bytes of one GEMM-with-epilogue launch: W codes and scales,
    quantized X, S, the tile slices of B of the distinct active adapters, Y."""
    wbytes = N * K if fmt == 0 else N * K // 2 + N * K // 16
    wscale = N * 4 if fmt == 0 else 4
    xq = M * K + M * 4 if fmt == 0 else M * K // 2 + M * K // 16
    return wbytes + wscale + xq + M * r * 4 + n_distinct * N * r * 2 + M * N * 2


def kernels_per_call(fmt, M, N, K, r):
    """Kernels one layer call enqueues with a workspace of
    epilora_layer_workspace_bytes: epilora_layer_forward_kernels, plus the
    expand pass where that workspace holds its fp32 term."""
    from precision_gemm_token_gb300 import _binding as E
    k = E.epilora_layer_forward_kernels(fmt, M, K, r)
    if k == 2 and E.epilora_layer_workspace_bytes(fmt, M, N, K, r) > E.epilora_workspace_bytes(fmt, M, K, r):
        k += 1
    return k


def run_ours(args, rank, world, local):
    import numpy as np
    import torch

    import precision_gemm_token_gb300 as E
    from precision_gemm_token_gb300 import tensors as T
    from synth import make_projection

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0:
        E.build()
    barrier(world)
    E.load()
    peaks = {}
    pk = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(pk):
        peaks = json.load(open(pk))

    def make_layer(workload, seed, spec=None, M=None, r=None, adapters="bf16", slices=None):
        """One layer's projections. adapters: "bf16" tables or "fp8" stored
        tables; slices: {projection: [slice ends]} for multi-slice
        projections (one rank-r adapter pair per slice)."""
        if spec is None:
            M0, fmt, L, r0, idx_mode, _ = WORKLOADS[workload]
            plist, mask_mode, n_decode = PROJ8B, "all", 0
            M = M or M0
            r = r or r0
        else:
            _, plist, M, fmt, L, r, idx_mode, mask_mode, n_decode, _ = spec
        projs = []
        for i, (name, K, N) in enumerate(plist):
            ends = (slices or {}).get(name)
            rr = r * len(ends) if ends else r
            p = make_projection(M, K, N, L, rr, seed=seed + i, idx_mode=idx_mode, mask_mode=mask_mode,
                                n_decode=n_decode, device=str(dev))
            if ends:
                p.B = p.B[:, :, :r].contiguous()     # B [L, N, r]; A stacks the slices' rank-r blocks
            w = T.quantize_weight(p.W, fmt)
            del p.W
            gx = T.nvfp4_global_scale(p.X) if fmt == 1 else None
            ws = T.LayerWorkspace(dev)
            ws.get(fmt, M, K, rr, N)
            Y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
            q = dict(name=name, K=K, N=N, r=rr, p=p, w=w, gx=gx, ws=ws, Y=Y, ends=ends, ad=None,
                     st=torch.zeros(1, dtype=torch.int32, device=dev))
            if adapters == "fp8":
                q["ad"] = T.quantize_adapters_fp8(p.A, p.B)
            projs.append(q)
        torch.cuda.synchronize()
        return projs

    def layer(projs, stream=None):
        for q in projs:
            p = q["p"]
            if q["ad"] is not None:
                T.layer_forward_fp8_adapters(p.X, q["w"], q["ad"], p.idx, p.mask, x_global_scale=q["gx"],
                                             workspace=q["ws"], status=q["st"], stream=stream, Y=q["Y"])
            elif q["ends"]:
                T.layer_forward_slices(p.X, q["w"], p.A, p.B, p.idx, q["ends"], p.mask, x_global_scale=q["gx"],
                                       workspace=q["ws"], status=q["st"], stream=stream, Y=q["Y"])
            else:
                T.layer_forward(p.X, q["w"], p.A, p.B, p.idx, p.mask, x_global_scale=q["gx"], workspace=q["ws"],
                                status=q["st"], stream=stream, Y=q["Y"])

    def layer_line(projs, fmt, steps, warmup, desc, M, layers=1):
        """Layer time (graph replay, L2 flushed) and the layer's HBM
        fraction over its algorithmic bytes; `layers` layers of distinct
        weights in one graph are reported per layer."""
        ms, _, _, _ = time_graph(projs, steps, warmup)
        ms = max_over_ranks(ms, world, dev) / layers
        byts = 0
        for q in projs:
            pq = q["p"]
            act = [int(i) for i, m in zip(pq.idx.tolist(), pq.mask.tolist()) if i >= 0 and m != 0]
            nd = len(set(act))
            b = algorithmic_bytes(M, q["K"], q["N"], fmt, q["r"], nd)
            if q["ad"] is not None:       # stored FP8 tables: 1 byte per element + a scale per row
                b -= nd * (q["r"] * q["K"] + q["N"] * q["r"]) - nd * (q["r"] + q["N"]) * 4
            byts += b
        byts //= layers
        gbs = byts / (ms / 1000) / 1e9
        return {"workload": desc, "M": M, "layer_us": round(ms * 1000, 2),
                "tokens_per_s": round(world * M / (ms / 1000), 1), "algorithmic_bytes": int(byts),
                "hbm_gbs": round(gbs, 1), "hbm_frac_of_measured": round(gbs / peaks.get("hbm_gbs", 6800.0), 4),
                "kernels_per_projection": [kernels_per_call(fmt, M, q["N"], q["K"], q["r"])
                                           for q in projs[:len(projs) // layers]]}

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush_buf = torch.empty(2 * l2 // 4 + 1024, dtype=torch.int32, device=dev)
    clean_buf = torch.ones(2 * l2 // 4 + 1024, dtype=torch.int32, device=dev)
    clean_out = torch.empty((), dtype=torch.int64, device=dev)

    class _Flush:
        """Write a buffer of twice the L2 size, then read another one: nothing
        of the workload stays in L2, and the flush's own dirty lines are
        written back before the timed events rather than inside them."""

        @staticmethod
        def fill_(v):
            flush_buf.fill_(v)
            torch.sum(clean_buf, dim=0, dtype=torch.int64, out=clean_out)

    flush = _Flush()

    def time_graph(projs, steps, warmup, sampler=None):
        s = torch.cuda.Stream(device=dev)
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            layer(projs, s)           # warm the kernels' attributes before capture
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            layer(projs, s)
        for _ in range(warmup):
            flush.fill_(1)
            g.replay()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        barrier(world)
        torch.cuda.synchronize()
        if sampler:
            sampler.start()
            time.sleep(0.3)
        t_wall = time.perf_counter()
        for a, b in evs:
            flush.fill_(1)
            a.record()
            g.replay()
            b.record()
        torch.cuda.synchronize()
        t_wall = time.perf_counter() - t_wall
        clocks = sampler.stop() if sampler else None
        barrier(world)
        per = [a.elapsed_time(b) for a, b in evs]
        for q in projs:
            if int(q["st"].item()) != 0:
                raise RuntimeError(f"device status {int(q['st'].item())} in {q['name']}")
        return float(np.mean(per)), float(np.median(per)), t_wall, clocks

    def time_calls(fn, steps, warmup):
        """Median and mean (ms) of `fn` (one projection's enqueue) captured as
        a CUDA graph, each replay behind an L2 flush outside the events."""
        s = torch.cuda.Stream(device=dev)
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            fn(s)
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            fn(s)
        for _ in range(warmup):
            flush.fill_(1)
            g.replay()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        torch.cuda.synchronize()
        for a, b in evs:
            flush.fill_(1)
            a.record()
            g.replay()
            b.record()
        torch.cuda.synchronize()
        per = sorted(a.elapsed_time(b) for a, b in evs)
        return per[len(per) // 2], float(np.mean(per))

    def exposure_controls(projs, steps, warmup):
        """Per projection (EpiLoRA, Evaluation › Kernels, Tables 10-12 and 17):
        T(fused call), T(no adapter: the same call with A = B = NULL),
        T(GEMM, h given: the standalone GEMM with its adapter epilogue reading
        a precomputed S and quantized X), T(serial: quantizer, shrink and GEMM
        as three ordinary launches), and exposed = T(fused) - T(h given), the
        adapter cost added = T(fused) - T(no adapter). Medians in us."""
        out, tot = {}, {}
        for q in projs:
            p, w, gx, Y = q["p"], q["w"], q["gx"], q["Y"]
            Mq, Kq = p.X.shape
            Xq, xs = T.quant_act(p.X, w.fmt, global_scale=gx)
            S = T.lora_shrink(p.X, p.A, p.idx, p.mask)
            ws0 = T.LayerWorkspace(dev)
            torch.cuda.synchronize()
            fns = {
                "fused": lambda st, p=p, w=w, gx=gx, Y=Y, ws=q["ws"]: T.layer_forward(
                    p.X, w, p.A, p.B, p.idx, p.mask, x_global_scale=gx, workspace=ws, stream=st, Y=Y),
                "no_adapter": lambda st, p=p, w=w, gx=gx, Y=Y, ws=ws0: T.layer_forward(
                    p.X, w, x_global_scale=gx, workspace=ws, stream=st, Y=Y),
                "h_given": lambda st, p=p, w=w, gx=gx, Y=Y, Xq=Xq, xs=xs, S=S, Mq=Mq, Kq=Kq: T.gemm_lora_epilogue(
                    Xq, xs, w, Mq, Kq, S=S, B=p.B, idx=p.idx, mask=p.mask, x_global_scale=gx, stream=st, Y=Y),
            }

            def serial(st, p=p, w=w, gx=gx, Y=Y, Mq=Mq, Kq=Kq, Xq=Xq, xs=xs, S=S):
                T.quant_act_into(p.X, w.fmt, Xq, xs, global_scale=gx, stream=st)
                T.lora_shrink_into(p.X, p.A, p.idx, p.mask, S, stream=st)
                T.gemm_lora_epilogue(Xq, xs, w, Mq, Kq, S=S, B=p.B, idx=p.idx, mask=p.mask, x_global_scale=gx,
                                     stream=st, Y=Y)
            fns["serial"] = serial
            row = {}
            for k, fn in fns.items():
                med, _ = time_calls(fn, steps, warmup)
                row[k] = round(med * 1000, 2)
            row["exposed_vs_h_given"] = round(row["fused"] - row["h_given"], 2)
            row["adapter_cost_vs_no_adapter"] = round(row["fused"] - row["no_adapter"], 2)
            out[q["name"]] = row
            for k, v in row.items():
                tot[k] = round(tot.get(k, 0.0) + v, 2)
        out["sum"] = tot
        return out

    workload = args.workload
    M, fmt, L, r, idx_mode, desc = WORKLOADS[workload]
    projs = make_layer(workload, seed=100)
    sampler = ClockSampler(local)
    ms_mean, ms_med, t_wall, clocks = time_graph(projs, args.steps, args.warmup, sampler)
    ms_max = max_over_ranks(ms_mean, world, dev)
    value_us = ms_max * 1000.0

    controls = None
    if not args.skip_controls:
        controls = exposure_controls(projs, max(args.steps // 2, 10), args.warmup)

    # more decode layers of the configurations: 32 tenants (FP8 base with bf16
    # adapters, the same with stored FP8 adapters, an NVFP4 base), the NVFP4
    # layer over M and rank, and multi-slice projections
    t32 = t32_fp8ad = t32_nv = nv = slices_line = chain_line = None
    nv_sweep = []
    xsteps = max(args.steps // 4, 5)
    if not args.skip_tenants:
        w32 = "8b_m32_fp8"
        pr = make_layer(w32, seed=200)
        t32 = layer_line(pr, 0, xsteps, args.warmup, WORKLOADS[w32][5], 32)
        y_bf = pr[3]["Y"].float().clone()
        pd = pr[3]
        y_base = T.layer_forward(pd["p"].X, pd["w"]).float()
        del pr, pd
        torch.cuda.empty_cache()
        pr = make_layer(w32, seed=200, adapters="fp8")
        t32_fp8ad = layer_line(pr, 0, xsteps, args.warmup,
                               WORKLOADS[w32][5] + ", adapters stored as E4M3 codes with one fp32 scale per row", 32)
        y_q = pr[3]["Y"].float()
        # the stored tables' price: their adapter term against the bf16
        # tables' term (down projection, all 32 tokens)
        t32_fp8ad["adapter_term_rel_err_vs_bf16"] = round(float((y_q - y_bf).norm() / (y_bf - y_base).norm()), 5)
        del pr, y_bf, y_q, y_base
        torch.cuda.empty_cache()
        pr = make_layer("8b_m32_nvfp4", seed=210)
        t32_nv = layer_line(pr, 1, xsteps, args.warmup, WORKLOADS["8b_m32_nvfp4"][5], 32)
        del pr
        torch.cuda.empty_cache()
        pr = make_layer("8b_m1_nvfp4", seed=400)
        nv = layer_line(pr, 1, xsteps, args.warmup, WORKLOADS["8b_m1_nvfp4"][5], 1)
        del pr
        torch.cuda.empty_cache()
        for (Mv, rv) in ((1, 16), (1, 128), (8, 64), (32, 16), (32, 128)):
            pr = make_layer("8b_m1_nvfp4", seed=420 + Mv + rv, M=Mv, r=rv)
            nv_sweep.append(layer_line(pr, 1, xsteps, args.warmup,
                                       f"Llama-3.1-8B layer, NVFP4, M={Mv}, 128 resident rank-{rv} adapters, "
                                       "Zipf(1.1) indices", Mv))
            del pr
            torch.cuda.empty_cache()
        pr = make_layer("8b_m1_fp8", seed=500, slices={"qkv": [4096, 5120, 6144], "gate_up": [14336, 28672]})
        slices_line = layer_line(pr, 0, xsteps, args.warmup,
                                 "Llama-3.1-8B layer, M=1, FP8, qkv as three slices (q, k, v) and gate_up as two "
                                 "(gate, up), one rank-64 adapter pair per slice", 1)
        del pr
        torch.cuda.empty_cache()
        # four layers of distinct weights in one graph, as a decode step runs
        # them (0.9 GB, far larger than L2; the flush stays outside the
        # events): the cost of one layer inside a chain
        pr = []
        for li in range(4):
            pr += make_layer("8b_m1_fp8", seed=600 + 10 * li)
        chain_line = layer_line(pr, 0, xsteps, args.warmup,
                                "four Llama-3.1-8B decode layers of distinct weights in one graph, M=1, FP8, one "
                                "rank-64 adapter each; per layer", 1, layers=4)
        del pr
        torch.cuda.empty_cache()

    # wide token tiles: tensor-pipe fraction of the fused layer (FP8 peak =
    # measured bf16 burst x 2, NVFP4 = x 6: the nominal dense ratios)
    large = None
    if not args.skip_large:
        large = []
        bf16 = peaks.get("bf16_tflops", 1900.0)
        for spec in LARGE_WORKLOADS:
            name, plist, Ml, fl, _, _, _, _, _, desc_l = spec
            projs_l = make_layer(None, seed=300, spec=spec)
            ms_l, _, _, _ = time_graph(projs_l, 5, args.warmup)
            ms_l = max_over_ranks(ms_l, world, dev)
            flops = sum(2.0 * Ml * N * K for _, K, N in plist)
            peak_l = bf16 * (2.0 if fl == 0 else 6.0)
            tf = flops / (ms_l / 1000) / 1e12
            # the same layer against HBM: distinct adapters active per projection
            bytes_l = 0
            for q, (_, K, N) in zip(projs_l, plist):
                pq = q["p"]
                act = [int(i) for i, m in zip(pq.idx.tolist(), pq.mask.tolist()) if i >= 0 and m != 0]
                bytes_l += algorithmic_bytes(Ml, K, N, fl, spec[5], len(set(act)))
            gbs_l = bytes_l / (ms_l / 1000) / 1e9
            # the layer's roofline: the slower of its HBM time (algorithmic
            # bytes at the measured copy bandwidth) and its tensor time
            t_hbm = bytes_l / (peaks.get("hbm_gbs", 6800.0) * 1e9)
            t_tc = flops / (peak_l * 1e12)
            large.append({"workload": desc_l, "M": Ml, "layer_us": round(ms_l * 1000, 1), "tflops": round(tf, 1),
                          "algorithmic_bytes": int(bytes_l), "hbm_gbs": round(gbs_l, 1),
                          "hbm_frac_of_measured": round(gbs_l / peaks.get("hbm_gbs", 6800.0), 4),
                          "peak_tflops": round(peak_l, 1), "tensor_frac": round(tf / peak_l, 4),
                          "bound": "hbm" if t_hbm > t_tc else "tensor",
                          "roofline_us": round(max(t_hbm, t_tc) * 1e6, 1),
                          "frac": round(max(t_hbm, t_tc) / (ms_l / 1000), 4),
                          "peak_source": "measured bf16 burst x " + ("2 (FP8)" if fl == 0 else "6 (NVFP4)")
                                         + "; measured copy bandwidth",
                          "kernels_per_projection": [kernels_per_call(fl, Ml, N, K, spec[5]) for _, K, N in plist]})
            del projs_l
            torch.cuda.empty_cache()

    # dominant kernel, gate_up, timed alone behind an L2 flush: the single
    # decode kernel (the whole projection) where the library takes that path,
    # else the GEMM with its LoRA epilogue reading S already in memory
    q = projs[2]
    p = q["p"]
    n_distinct = len(set(int(i) for i in p.idx.tolist() if i >= 0))
    single = E.epilora_layer_forward_kernels(fmt, M, q["K"], r) == 1
    if single:
        kern = lambda: T.layer_forward(p.X, q["w"], p.A, p.B, p.idx, p.mask, x_global_scale=q["gx"],  # noqa
                                       workspace=q["ws"], Y=q["Y"])
        kbytes = algorithmic_bytes(M, q["K"], q["N"], fmt, r, n_distinct)
        kname, prof = f"fused_decode_kernel gate_up {q['K']}->{q['N']} M={M}", "fused_decode_gate_up"
    else:
        Xq, xs = T.quant_act(p.X, fmt, global_scale=q["gx"])
        S = T.lora_shrink(p.X, p.A, p.idx, p.mask)
        kern = lambda: T.gemm_lora_epilogue(Xq, xs, q["w"], M, q["K"], S=S, B=p.B, idx=p.idx, mask=p.mask,  # noqa
                                            x_global_scale=q["gx"], Y=q["Y"])
        kbytes = gemm_kernel_bytes(M, q["K"], q["N"], fmt, r, n_distinct)
        kname, prof = f"gemm_lora_kernel gate_up {q['K']}->{q['N']} M={M}", "gemm_gate_up"
    torch.cuda.synchronize()
    # eager launches on the current stream, each queued behind the L2 flush
    # (kernels of tens of microseconds): the host has submitted the start
    # event and the kernel before the flush ends, so the events bracket the
    # kernel's execution only
    for _ in range(args.warmup):
        flush.fill_(1)
        kern()
    ke = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    torch.cuda.synchronize()
    for a, b in ke:
        flush.fill_(1)
        a.record()
        kern()
        b.record()
    torch.cuda.synchronize()
    k_ms = float(np.mean([a.elapsed_time(b) for a, b in ke]))
    peak = peaks.get("hbm_gbs")
    peak_src = "measured" if peak else "fallback"
    peak = peak or 6800.0
    achieved = kbytes / (k_ms / 1000) / 1e9
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": read_profile_traffic(workload, prof),
                "kernel": kname, "kernel_us": round(k_ms * 1000, 2),
                "algorithmic_bytes": kbytes, "peak_source": peak_src}

    layer_bytes = sum(algorithmic_bytes(M, K, N, fmt, r, max(n_distinct, 1)) for _, K, N in PROJ8B)

    # end-to-end through the public API with host buffers
    e2e = None
    if not args.skip_e2e:
        # the step's inputs staged in one pinned host buffer and its outputs
        # gathered in one device buffer: one copy each way per step (the
        # projections' X and Y are views of those buffers)
        nx = [q["p"].X.numel() for q in projs]
        ny = [q["Y"].numel() for q in projs]
        hx = torch.empty(sum(nx), dtype=torch.bfloat16).pin_memory()
        dx = torch.empty(sum(nx), dtype=torch.bfloat16, device=dev)
        hy = torch.empty(sum(ny), dtype=torch.bfloat16).pin_memory()
        dy = torch.empty(sum(ny), dtype=torch.bfloat16, device=dev)
        xv, yv = [], []
        ox = oy = 0
        for q, a, b in zip(projs, nx, ny):
            hx[ox:ox + a].copy_(q["p"].X.reshape(-1).cpu())
            xv.append(dx[ox:ox + a].view(q["p"].X.shape))
            yv.append(dy[oy:oy + b].view(q["Y"].shape))
            ox += a
            oy += b
        h2d = hx.numel() * hx.element_size()
        d2h = hy.numel() * hy.element_size()
        st = torch.cuda.current_stream()

        # each projection's call bound once (PreparedLayer: one C call per
        # projection and step)
        calls = [T.PreparedLayer(xq, q["w"], q["p"].A, q["p"].B, q["p"].idx, q["p"].mask, x_global_scale=q["gx"],
                                 workspace=q["ws"], status=q["st"], stream=st, Y=yq)
                 for q, xq, yq in zip(projs, xv, yv)]

        def e2e_layer():
            for c in calls:
                c()

        dx.copy_(hx)
        for _ in range(args.warmup):
            e2e_layer()
        torch.cuda.synchronize()
        times = []
        for _ in range(args.steps):
            flush.fill_(1)
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            dx.copy_(hx, non_blocking=True)
            e2e_layer()
            hy.copy_(dy, non_blocking=True)
            torch.cuda.synchronize()
            times.append(time.perf_counter() - t0)
        # the results equal a call on the device-resident inputs (same kernels,
        # same inputs)
        for q, yq in zip(projs, yv):
            p = q["p"]
            ref = T.layer_forward(p.X, q["w"], p.A, p.B, p.idx, p.mask, x_global_scale=q["gx"], workspace=q["ws"])
            if not torch.equal(yq, ref):
                raise RuntimeError(f"end-to-end output differs in {q['name']}")
        e2e_us = max_over_ranks(float(np.mean(times)) * 1e6, world, dev)
        e2e = {"value": round(e2e_us, 2), "unit": "us", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "how": "eager C-ABI calls per projection from Python (no graph; tensors.PreparedLayer, the "
                      "arguments bound once); the step's X from one pinned host buffer in one copy, its Y out in "
                      "one copy"}

    line = {
        "metric": METRIC, "value": round(value_us, 3), "unit": "us", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_max, 5), "higher_is_better": False, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp8_e4m3" if fmt == 0 else "nvfp4_e2m1", "data": "synthetic",
        "config": {"workload": desc, "M": M, "rank": r, "tenants": L if idx_mode != "single" else 1,
                   "parallelism": f"replicas{world}", "cuda_graph": True,
                   "l2": "flushed between steps outside the timed events: write of a 2x-L2 buffer, then a read "
                         "of another 2x-L2 buffer (the write's dirty lines leave L2 before the timed region)",
                   "timed": "CUDA events around each graph replay of the 4 projections"},
        "tokens_per_s": round(world * M / (ms_max / 1000), 1),
        "layer_hbm_gbs": round(layer_bytes / (ms_max / 1000) / 1e9, 1),
        "layer_hbm_frac_of_measured": round(layer_bytes / (ms_max / 1000) / 1e9 / peak, 4),
        "roofline": roofline,
        "exposure": controls,
        "tenants32": t32,
        "tenants32_fp8_adapters": t32_fp8ad,
        "tenants32_nvfp4": t32_nv,
        "nvfp4_m1": nv,
        "nvfp4_sweep": nv_sweep,
        "multi_slice": slices_line,
        "layers_chained": chain_line,
        "large_m": large,
        "e2e": e2e,
        # per projection: one persistent kernel (single-kernel decode path) or
        # the shrink grid and the GEMM, as the library reports for the shape
        "gpu_launches": args.steps * sum(E.epilora_layer_forward_kernels(fmt, M, K, r) for _, K, _ in PROJ8B),
        "clocks": clocks,
        "median_ms_per_step": round(ms_med, 5),
    }
    if rank == 0 and not args.skip_cpu:
        line["cpu_baseline"] = cpu_baseline(workload, args.cpu_seconds)
    return line


# ----------------------------------------------------------------------------
# the oracle on the host (cpu baseline and the reference arm)
# ----------------------------------------------------------------------------
def oracle_prepare(workload, frac, seed=100):
    """Inputs of one layer step restricted to a column sample of every
    projection (the same fraction of each projection's output columns, full
    K and M), with the weights quantized by the oracle."""
    from oracle import epilora_oracle as O
    from synth import make_projection

    M, fmt, L, r, idx_mode, _ = WORKLOADS[workload]
    out = []
    for i, (name, K, N) in enumerate(PROJ8B):
        ncol = max(8, min(N, int(round(frac * N))))
        Ls = L if idx_mode == "per_token" else min(L, 4)
        p = make_projection(M, K, ncol, Ls, r, seed=seed + i, idx_mode=idx_mode if idx_mode != "zipf" else "uniform")
        x, Wn = p.X.float().numpy(), p.W.float().numpy()
        d = dict(name=name, K=K, N=N, ncol=ncol, x=x, A=p.A.float().numpy(), B=p.B.float().numpy(),
                 idx=p.idx.numpy(), mask=p.mask.numpy())
        if fmt == 0:
            d["wq"], d["sw"] = O.quant_fp8_rows(Wn)
        else:
            d["gw"] = O.nvfp4_global_scale(Wn)
            d["wq"], d["sbw"] = O.quant_nvfp4_rows(Wn, d["gw"])
            d["gx"] = O.nvfp4_global_scale(x)
        out.append(d)
    return out


def _oracle_job(job):
    """One column chunk of one projection through the oracle (a pool worker)."""
    from oracle import epilora_oracle as O

    fmt, d = job
    if fmt == 0:
        O.layer_fp8(d["x"], d["wq"], d["sw"], d["A"], d["B"], d["idx"], d["mask"])
    else:
        O.layer_nvfp4(d["x"], d["gx"], d["wq"], d["sbw"], d["gw"], d["A"], d["B"], d["idx"], d["mask"])
    return d["ncol"]


class OraclePool:
    """The oracle on the host cores: one single-threaded worker process per
    core (spawned, so no GPU state is inherited), each taking column chunks
    of the projections."""

    def __init__(self):
        import multiprocessing as mp
        try:
            self.n = len(os.sched_getaffinity(0))
        except AttributeError:
            self.n = os.cpu_count() or 1
        self.pool = mp.get_context("spawn").Pool(self.n)

    def close(self):
        self.pool.close()
        self.pool.join()

    def step(self, workload, sample):
        """Wall time of one pass over the sample, extrapolated to the whole
        layer by the ratio of multiply-adds (us), and the sample's detail."""
        import numpy as np

        fmt = WORKLOADS[workload][1]
        jobs = []
        for d in sample:
            for ch in np.array_split(np.arange(d["ncol"]), self.n):
                if ch.size == 0:
                    continue
                sl = slice(int(ch[0]), int(ch[-1]) + 1)
                e = dict(d, ncol=int(ch.size), wq=d["wq"][sl], B=d["B"][:, sl, :])
                if fmt == 0:
                    e["sw"] = d["sw"][sl]
                else:
                    e["sbw"] = d["sbw"][sl]
                jobs.append((fmt, e))
        t0 = time.perf_counter()
        self.pool.map(_oracle_job, jobs, chunksize=1)
        dt = time.perf_counter() - t0
        scale = sum(d["K"] * d["N"] for d in sample) / sum(d["K"] * d["ncol"] for d in sample)
        detail = ", ".join(f"{d['name']} {d['ncol']}/{d['N']}" for d in sample)
        return dt * scale * 1e6, detail


def cpu_baseline(workload, seconds_target=10.0):
    """The oracle on all host cores, on a column sample sized to about
    seconds_target of wall time."""
    pool = OraclePool()
    try:
        pool.step(workload, oracle_prepare(workload, 0.002))          # workers up
        probe_us, _ = pool.step(workload, oracle_prepare(workload, 0.01))
        frac = min(1.0, max(0.002, 0.01 * seconds_target * 1e6 / max(probe_us * 0.01, 1.0) / 2))
        us, detail = pool.step(workload, oracle_prepare(workload, frac))
    finally:
        pool.close()
    return {"value": round(us, 1), "unit": "us", "cores": pool.n, "kind": "oracle",
            "sample": f"output columns sampled per projection (sampled/total: {detail}) at full K and M, "
                      f"spread over {pool.n} single-threaded worker processes, wall time extrapolated by "
                      "the ratio of multiply-adds"}


def run_reference(args, rank, world):
    """The oracle as the reference arm: rank 0 only, on the host cores, each
    step a column sample of the same workload sized so that the whole run
    stays within about two minutes."""
    if rank != 0:
        return None
    workload = args.workload
    M, fmt, L, r, idx_mode, desc = WORKLOADS[workload]
    pool = OraclePool()
    try:
        pool.step(workload, oracle_prepare(workload, 0.002))
        probe_us, _ = pool.step(workload, oracle_prepare(workload, 0.01))
        budget_us = 120e6 / (args.steps + args.warmup)
        frac = min(1.0, max(0.001, 0.01 * budget_us / max(probe_us * 0.01, 1.0) / 2))
        sample = oracle_prepare(workload, frac)
        for _ in range(args.warmup):
            pool.step(workload, sample)
        per, detail = [], ""
        for _ in range(args.steps):
            v, detail = pool.step(workload, sample)
            per.append(v)
    finally:
        pool.close()
    value = sum(per) / len(per)
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": "us", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(value / 1000, 3),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": desc, "M": M, "rank": r, "tenants": L if idx_mode != "single" else 1,
                   "parallelism": "host oracle, rank 0 only"},
        "cpu_baseline": {"value": round(value, 1), "unit": "us", "cores": pool.n, "kind": "oracle",
                         "sample": f"output columns per projection per step (sampled/total: {detail}) at full K "
                                   f"and M over {pool.n} worker processes, extrapolated by the ratio of "
                                   "multiply-adds"},
        "e2e": {"value": round(value, 1), "unit": "us", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_profile(args):
    """The dominant kernel alone, for ncu: quantize X and run the shrink
    once, then launch the gate_up GEMM with its LoRA epilogue five times
    (ordinary launches, S already in memory)."""
    import torch

    import precision_gemm_token_gb300 as E
    from precision_gemm_token_gb300 import tensors as T
    from synth import make_projection

    E.build()
    E.load()
    M, fmt, L, r, idx_mode, _ = WORKLOADS[args.workload]
    _, K, N = PROJ8B[2]
    p = make_projection(M, K, N, L, r, seed=102, idx_mode=idx_mode, device="cuda")
    w = T.quantize_weight(p.W, fmt)
    gx = T.nvfp4_global_scale(p.X) if fmt == 1 else None
    Xq, xs = T.quant_act(p.X, fmt, global_scale=gx)
    S = T.lora_shrink(p.X, p.A, p.idx, p.mask)
    Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    for _ in range(5):
        T.gemm_lora_epilogue(Xq, xs, w, M, K, S=S, B=p.B, idx=p.idx, mask=p.mask, x_global_scale=gx, Y=Y)
    torch.cuda.synchronize()
    print(json.dumps({"profile": args.workload, "kernel": f"gate_up {K}->{N} M={M}", "ok": True}))


def run_profile_fused(args):
    """One fused layer call alone, for ncu: the workload's gate_up projection
    (4096 -> 28672) through epilora_layer_forward five times on one
    workspace, on the single-kernel decode path (for a few tokens; both
    formats)."""
    import torch

    import precision_gemm_token_gb300 as E
    from precision_gemm_token_gb300 import tensors as T
    from synth import make_projection

    E.build()
    E.load()
    E.epilora_set_decode_path(E.DECODE_PATH_SINGLE)
    M, fmt, L, r, idx_mode, _ = WORKLOADS[args.workload]
    _, K, N = PROJ8B[2]
    p = make_projection(M, K, N, L, r, seed=102, idx_mode=idx_mode, device="cuda")
    w = T.quantize_weight(p.W, fmt)
    gx = T.nvfp4_global_scale(p.X) if fmt == 1 else None
    ws = T.LayerWorkspace("cuda")
    Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(5):
        T.layer_forward(p.X, w, p.A, p.B, p.idx, p.mask, x_global_scale=gx, workspace=ws, status=st, Y=Y)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    print(json.dumps({"profile": args.workload, "kernel": f"fused gate_up {K}->{N} M={M}",
                      "kernels_per_call": E.epilora_layer_forward_kernels(fmt, M, K, r), "ok": True}))


def run_profile_large(args):
    """The 8B NVFP4 M = 512 layer's gate_up projection alone, for ncu: three
    fused layer calls (shrink grid, expand pass, wide-tile GEMM) on
    Zipf-indexed rank-64 adapters out of 128; with --profile-large-base the
    same calls without adapters (quantizer grid and base GEMM)."""
    import torch

    import precision_gemm_token_gb300 as E
    from precision_gemm_token_gb300 import tensors as T
    from synth import make_projection

    E.build()
    E.load()
    _, plist, M, fmt, L, r, idx_mode, mask_mode, n_decode, _ = LARGE_WORKLOADS[1]
    _, K, N = plist[2]
    p = make_projection(M, K, N, L, r, seed=302, idx_mode=idx_mode, mask_mode=mask_mode, n_decode=n_decode,
                        device="cuda")
    w = T.quantize_weight(p.W, fmt)
    del p.W
    gx = T.nvfp4_global_scale(p.X)
    ws = T.LayerWorkspace("cuda")
    Y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    A, B = (None, None) if getattr(args, "profile_large_base", False) else (p.A, p.B)
    for _ in range(3):
        T.layer_forward(p.X, w, A, B, p.idx, p.mask, x_global_scale=gx, workspace=ws, status=st, Y=Y)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    print(json.dumps({"profile": "8b_m512_nvfp4", "kernel": f"gate_up {K}->{N} M={M}",
                      "adapters": A is not None, "ok": True}))


def run_profile_wide(args):
    """A wide-tile fused layer call alone, for ncu: the Llama-3.1-70B gate_up
    projection's quarter column slice (K 8192 -> N 14336: 1008 tiles of
    256x128, the persistent kernel) over the prefill-chunk batch (64 mask-0
    decode tokens + 2048 prefill tokens on one adapter, 512 resident rank-16
    adapters, Zipf(1.1) indices, FP8), five layer_forward calls (shrink grid
    + GEMM each)."""
    import torch

    import precision_gemm_token_gb300 as E
    from precision_gemm_token_gb300 import tensors as T
    from synth import make_projection

    E.build()
    E.load()
    M, K, N = 2112, 8192, 57344 // 4
    p = make_projection(M, K, N, 512, 16, seed=5, idx_mode="zipf", mask_mode="prefill_chunk", n_decode=64,
                        device="cuda")
    w = T.quantize_weight(p.W, 0)
    ws = T.LayerWorkspace("cuda")
    for _ in range(5):
        T.layer_forward(p.X, w, p.A, p.B, p.idx, p.mask, workspace=ws)
    torch.cuda.synchronize()
    print(json.dumps({"profile": "70b_gate_up_quarter_prefill2112_fp8", "kernel": f"gate_up {K}->{N} M={M}",
                      "ok": True}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="8b_m1_fp8", choices=sorted(WORKLOADS))
    ap.add_argument("--skip-tenants", action="store_true")
    ap.add_argument("--skip-large", action="store_true", help="skip the wide-tile (tensor-bound) layers")
    ap.add_argument("--skip-e2e", action="store_true")
    ap.add_argument("--skip-controls", action="store_true", help="skip the per-projection exposure controls")
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--profile", action="store_true", help="run the dominant kernel alone (for ncu)")
    ap.add_argument("--profile-wide", action="store_true", help="run one wide-tile fused layer call alone (for ncu)")
    ap.add_argument("--profile-large", action="store_true",
                    help="run the 8B NVFP4 M=512 gate_up fused call alone (for ncu)")
    ap.add_argument("--profile-large-base", action="store_true",
                    help="the same calls without adapters (the base GEMM alone, for ncu)")
    ap.add_argument("--profile-fused", action="store_true",
                    help="run the workload's fused gate_up layer call alone (for ncu)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.profile:
        run_profile(args)
        return
    if args.profile_wide:
        run_profile_wide(args)
        return
    if args.profile_fused:
        run_profile_fused(args)
        return
    if args.profile_large or args.profile_large_base:
        run_profile_large(args)
        return
    rank, world, local = dist_setup()
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        line = run_ours(args, rank, world, local)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

"""Throughput of the fused LM-head forward + backward on GB300.

One step = the whole scoring path on one batch of synthetic inputs:
keep mask from the loss mask (next-token shift) -> compaction -> chunked
tcgen05 projection with the online-softmax epilogue -> split-V merge ->
expansion; then the backward: compaction, logit recomputation with the dZ
epilogue, dHidden (scattered back) and dW contractions per chunk.

Default workload: 30B-MoE-shaped RL head, N=65536 packed tokens, H=4096,
V=151936, bf16, sequences of length ~U[512, 8192] whose first half (prompt
fraction 0.5) is masked, so half the rows are kept (32767 of 65536),
differentiable entropy (grad_entropy = -0.01).  `--workload moe30b_rl` draws
the prompt fraction ~U[0.3, 0.7] instead (55% kept).

With --gpus N > 1 the step runs data-parallel on N ranks (one process per
GPU, under torch.distributed.run; started by this script when it is run
without one): every rank scores its own batch and the weight gradients are
summed by one all-reduce after the backward, inside the timed region.

Prints one JSON line.  `--impl reference` times the float64 CPU oracle on a
bounded sample of kept rows of the same workload instead.
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

METRIC = "fused LM-head fwd+bwd kept-tokens/s and TFLOP/s (% of GB300 bf16 tensor peak)"
UNIT = "kept-tokens/s"


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d["bf16_tflops"], d["bf16_tflops_sustained"], d["hbm_gbs"], "measured"
    except Exception:
        return 1900.0, 1700.0, 6800.0, "fallback"


def kernel_source_digest():
    """sha256 over the library's CUDA sources (csrc/), in name order."""
    import hashlib
    d = os.path.join(ROOT, "sft_keep_mask_gb300", "csrc")
    h = hashlib.sha256()
    for name in sorted(os.listdir(d)):
        if name.endswith((".cu", ".cuh", ".h")):
            h.update(name.encode())
            with open(os.path.join(d, name), "rb") as f:
                h.update(f.read())
    return h.hexdigest()


def recorded_traffic(kernel, config):
    """DRAM bytes per launch of `kernel` for this workload from an ncu capture
    (of a smaller case of it, scaled as the record states), or None if no
    capture of the current kernel sources exists for this workload."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except Exception:
        return None
    if rec.get("source_sha256") != kernel_source_digest():
        return None
    for key in ("workload", "N", "H", "V", "chunk_rows", "mode", "keep_mask", "rows", "entropy"):
        if rec.get("config", {}).get(key) != config.get(key):
            return None
    k = rec.get("kernels", {}).get(kernel)
    return None if k is None else dict(k, scaling=rec.get("scaling", ""),
                                       capture=rec.get("capture", {}))


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def launch_plan(gpus, env):
    """What `--gpus N` asks for, given the environment: "run" (this process
    is one of the N ranks, or N == 1), "spawn" (no launcher: start N ranks
    under torch.distributed.run) or an error message (a launcher started a
    different number of ranks)."""
    if gpus < 1:
        return f"--gpus must be at least 1, got {gpus}"
    if "WORLD_SIZE" not in env:
        return "run" if gpus == 1 else "spawn"
    world = int(env["WORLD_SIZE"])
    if world != gpus:
        return f"--gpus {gpus} but the launcher started {world} ranks"
    return "run"


def spawn_ranks(gpus, argv):
    """Re-runs this script as `gpus` ranks on this node (torch.distributed.run,
    rendezvous on 127.0.0.1) and returns its exit code."""
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={gpus}", "--master-addr=127.0.0.1", f"--master-port={port}",
           os.path.abspath(__file__), *argv]
    return subprocess.call(cmd)


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        import threading
        self.lines = []
        first = threading.Event()
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.gpu)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return self

        def reader():
            for ln in self.proc.stdout:
                if ln.strip():
                    self.lines.append(ln)
                    first.set()
            first.set()

        self.thread = threading.Thread(target=reader, daemon=True)
        self.thread.start()
        # the timed region starts only once the sampler is up and sampling
        first.wait(timeout=15.0)
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.thread.join(timeout=5)

    def summary(self):
        sm, mx, reasons, power = [], None, set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            try:
                power.append(float(parts[3]))
            except ValueError:
                pass
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm),
                "power_w": statistics.median(power) if power else None}


def _oracle_sample(inp, keep, rows, want_grad=True):
    """Float64 oracle on `rows` kept rows (full forward + backward work)."""
    import numpy as np
    from oracle import lmhead_oracle as O
    idx = np.flatnonzero(keep)
    pick = idx[np.linspace(0, len(idx) - 1, rows).astype(np.int64)]
    h = inp["hidden"][pick].float().cpu().double().numpy()
    y = inp["targets"][pick].cpu().numpy()
    g1 = inp["grad_logprob"][pick].cpu().double().numpy()
    g2 = (inp["grad_entropy"][pick].cpu().double().numpy()
          if inp["grad_entropy"] is not None else None)
    return h, y, g1, g2


def cpu_oracle_rate(inp, keep_np, W64, rows, mode="fwdbwd", entropy_grad=True):
    """Oracle time for `rows` sampled kept rows: the forward, plus for
    mode "fwdbwd" the dhidden and dW contributions (with the entropy term
    when `entropy_grad`).  The timed oracle is the C float64 one (plain
    loops, OpenMP over the host's cores)."""
    from oracle import lmhead_oracle_c as OC
    h, y, g1, g2 = _oracle_sample(inp, keep_np, rows)
    if mode != "fwdbwd":
        g1 = g2 = None
    elif not entropy_grad:
        g2 = None
    t0 = time.perf_counter()
    OC.score_rows(h, W64, y, g1, g2)
    dt = time.perf_counter() - t0
    return rows / dt, dt


def _oracle_cores():
    from oracle import lmhead_oracle_c as OC
    return OC.threads()


L2_BYTES = 126.5e6


def run_config(args, N, H, V, nk, world, entropy_grad):
    """The `config` object of the JSON line (both arms)."""
    w_bytes, h_bytes = V * H * 2, N * H * 2
    big = w_bytes + h_bytes > L2_BYTES
    return {"workload": args.workload, "N": N, "H": H, "V": V, "kept_rows": nk,
            "kept_frac": nk / N if N else 0.0, "chunk_rows": args.chunk_rows or 8192,
            "entropy": "differentiable" if entropy_grad else "metric-only",
            "mode": args.mode, "keep_mask": "off" if args.keep_off else "on",
            "rows": "block-sparse tiles" if args.blocksparse else "compacted",
            "l2": ("inputs larger than L2" if big else "inputs fit in L2 (no flush)")
                  + f" (W {w_bytes / 1e9:.2f} GB, hidden {h_bytes / 1e9:.2f} GB)",
            "parallelism": f"dp{world}" if world > 1 else "single GPU"}


def entropy_grad_of(args, inp):
    """Whether the step differentiates the entropy (the workload's default
    unless --entropy-grad says otherwise)."""
    if args.entropy_grad < 0:
        return inp["grad_entropy"] is not None
    return bool(args.entropy_grad) and inp["grad_entropy"] is not None


def _workload(args):
    from sft_keep_mask_gb300 import synth
    over = {}
    if args.rows:
        over["N"] = args.rows
    if args.vocab:
        over["V"] = args.vocab
    return synth.workload(args.workload, **over)


def reduce_over_ranks(elapsed, kept, world, device):
    """(max elapsed over ranks, sum of kept rows over ranks).

    Every rank scores its own batch (data-parallel, weak scaling), so the
    job's time is the slowest rank's and its work is the sum of all ranks'
    rows.
    """
    if world <= 1:
        return float(elapsed), float(kept)
    import torch
    import torch.distributed as dist
    mx = torch.tensor([float(elapsed)], dtype=torch.float64, device=device)
    sm = torch.tensor([float(kept)], dtype=torch.float64, device=device)
    dist.all_reduce(mx, op=dist.ReduceOp.MAX)
    dist.all_reduce(sm, op=dist.ReduceOp.SUM)
    return float(mx[0]), float(sm[0])


def _cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count()


def run_reference(args):
    """Reference arm: the float64 CPU oracle, timed on host cores."""
    world, rank, _ = _dist()
    if rank != 0:
        return
    import numpy as np
    import torch
    from oracle import lmhead_oracle as O
    from sft_keep_mask_gb300 import synth
    w = _workload(args)
    inp = synth.make_inputs(w, device="cpu")
    if args.keep_off:
        keep = np.ones(w.N, dtype=np.uint8)
    elif "components" in inp:
        keep = O.build_keep_mask([c.numpy() for c in inp["components"]], inp["seq_lens"])
    else:
        keep = inp["keep"].numpy()
    nk = int(keep.sum())
    ent_grad = entropy_grad_of(args, inp)
    W64 = inp["weight"].float().double().numpy()
    rows = min(args.ref_rows, nk)
    for _ in range(args.warmup):
        cpu_oracle_rate(inp, keep, W64, rows, args.mode, ent_grad)
    times = []
    for _ in range(args.steps):
        _, dt = cpu_oracle_rate(inp, keep, W64, rows, args.mode, ent_grad)
        times.append(dt)
    tot = sum(times)
    value = rows * args.steps / tot
    flops = (8.0 if args.mode == "fwdbwd" else 2.0) * rows * w.H * w.V * args.steps
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * tot / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        # the GPU arm's config exactly; the sample size is a key of its own
        "config": run_config(args, w.N, w.H, w.V, nk, world, ent_grad),
        "sample_rows_per_step": rows,
        "tflops": flops / tot / 1e12,
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": _oracle_cores(), "kind": "oracle",
                         "sample": f"{rows} kept rows per step, full H and V, forward"
                                   + (" + dhidden + dW contribution" if args.mode == "fwdbwd"
                                      else "") + ", C float64 oracle (OpenMP)"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args):
    import numpy as np
    import torch
    from sft_keep_mask_gb300 import lmhead as L
    from sft_keep_mask_gb300 import synth
    from sft_keep_mask_gb300.api import LMHeadScorer, allreduce_weight_grad

    world, rank, local = _dist()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    L.lib()

    w = _workload(args)
    base_seed = w.seed
    if world > 1:
        # data-parallel ranks: one weight, a batch per rank
        w = synth.workload(args.workload, N=w.N, V=w.V, seed=w.seed + 100 * rank)
    inp = synth.make_inputs(w, device=dev, active_frac=args.active_frac,
                            weight_seed=base_seed if world > 1 else None)
    sc = LMHeadScorer(w.N, w.H, w.V, chunk_rows=args.chunk_rows, device=dev,
                      blocksparse=args.blocksparse)
    comps = inp.get("components")
    lens = inp.get("seq_lens")
    offsets = None
    if comps is not None:
        off = np.zeros(len(lens) + 1, np.int32)
        off[1:] = np.cumsum(lens)
        offsets = torch.from_numpy(off).to(dev)
    N, H, V = w.N, w.H, w.V
    keep = torch.empty(N, dtype=torch.uint8, device=dev)
    lp = torch.empty(N, dtype=torch.float32, device=dev)
    ent = torch.empty(N, dtype=torch.float32, device=dev)
    lse = torch.empty(N, dtype=torch.float32, device=dev)
    dh = torch.empty(N, H, dtype=torch.bfloat16, device=dev)
    dW = torch.empty(V, H, dtype=torch.float32, device=dev)
    ws = sc.workspace
    use_ent_grad = entropy_grad_of(args, inp)
    g_ent = inp["grad_entropy"] if use_ent_grad else None
    stream = torch.cuda.current_stream(dev)

    keep_arg = None if args.keep_off else keep  # keep-off arm: every row scored

    def step(hidden, targets, loss_mask, offs, g_lp, g_e, mid=None):
        if args.keep_off:
            pass
        elif loss_mask is not None:
            L.lmhead_build_keep_mask(loss_mask, None, None, offs, keep, stream)
        else:
            keep.copy_(inp["keep"])
        fwd = L.lmhead_fwd_blocksparse if args.blocksparse else L.lmhead_fwd
        bwd = L.lmhead_bwd_blocksparse if args.blocksparse else L.lmhead_bwd
        fwd(hidden, inp["weight"], targets, keep_arg, True, lp, ent, lse, ws, args.chunk_rows,
            stream)
        if mid is not None:
            mid.record(stream)  # end of the forward pass
        if args.mode == "fwdbwd":
            bwd(hidden, inp["weight"], targets, keep_arg, lse, ent, g_lp, g_e, dh, dW, False, ws,
                args.chunk_rows, stream)
            # data-parallel ranks: one all-reduce of dW after the backward
            allreduce_weight_grad(dW)

    loss_mask = comps[0] if comps is not None else None
    dev_args = (inp["hidden"], inp["targets"], loss_mask, offsets, inp["grad_logprob"], g_ent)
    for _ in range(args.warmup):
        step(*dev_args)
    torch.cuda.synchronize(dev)
    status = L.lmhead_get_status(ws)
    if status != 0:
        raise RuntimeError(f"device status {status} after warm-up "
                           f"(timeout record {L.lmhead_get_timeout_record(ws)})")
    nk = N if args.keep_off else int(keep.sum().item())

    # ---------------------------------------------------------- device-timed
    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)

    L.lmhead_profile_enable(True)
    L.lmhead_profile_read()
    launches0 = L.lmhead_launch_count()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    # one event per step boundary as well, for the spread of the step times
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    mids = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    with ClockSampler(local) as clk:
        barrier()
        ev0.record(stream)
        marks[0].record(stream)
        for i in range(args.steps):
            step(*dev_args, mid=mids[i])
            marks[i + 1].record(stream)
        ev1.record(stream)
        barrier()
    step_ms = [marks[i].elapsed_time(marks[i + 1]) for i in range(args.steps)]
    # forward (keep mask build included) and backward parts of each step
    fwd_ms = [marks[i].elapsed_time(mids[i]) for i in range(args.steps)]
    bwd_ms = [mids[i].elapsed_time(marks[i + 1]) for i in range(args.steps)]
    L.lmhead_profile_enable(False)
    launches = L.lmhead_launch_count() - launches0
    status_timed = L.lmhead_get_status(ws)
    if status_timed != 0:
        raise RuntimeError(f"device status {status_timed} after the timed steps "
                           f"(timeout record {L.lmhead_get_timeout_record(ws)})")
    prof = L.lmhead_profile_read()
    ms = ev0.elapsed_time(ev1)
    ms_max, nk_total = reduce_over_ranks(ms, nk, world, dev)
    sec = ms_max / 1e3
    value = nk_total * args.steps / sec
    per_row = 8.0 if args.mode == "fwdbwd" else 2.0
    flops_step = per_row * nk_total * H * V
    tflops = flops_step * args.steps / sec / 1e12
    # the same work counted without the backward's recompute of the logits
    # (2 Nk H V forward + 4 Nk H V backward)
    per_row_rf = 6.0 if args.mode == "fwdbwd" else 2.0
    tflops_rf = per_row_rf * nk_total * H * V * args.steps / sec / 1e12
    burst, sustained, hbm, peak_src = _peaks()

    # dominant kernel of the step (largest summed device time)
    kinds = {k: v for k, v in prof.items() if v[0] > 0}
    tot_ms = sum(v[1] for v in kinds.values()) or 1.0
    gemm_flops = {"gemm_fwd": 2.0, "gemm_dz": 2.0, "gemm_dh": 2.0, "gemm_dw": 2.0}
    dom = max(kinds, key=lambda k: kinds[k][1])
    dom_ms = kinds[dom][1]
    if dom in gemm_flops:
        alg = gemm_flops[dom] * nk * H * V * args.steps  # flops of this kernel in the region
        achieved = alg / (dom_ms / 1e3) / 1e12
        roof = {"bound": "tensor", "kernel": dom, "achieved": achieved, "peak": sustained,
                "unit": "TFLOP/s", "frac": achieved / sustained,
                "frac_of_burst_peak": achieved / burst, "peak_source": f"{peak_src} sustained",
                "traffic": None}
    else:
        roof = {"bound": "hbm", "kernel": dom, "achieved": None, "peak": hbm, "unit": "GB/s",
                "frac": None, "traffic": None}
    kernels = {k: {"launches": v[0], "ms": v[1], "share": v[1] / tot_ms} for k, v in kinds.items()}
    gemm_ms = sum(kinds[k][1] for k in gemm_flops if k in kinds)
    gemm_tflops = per_row * nk * H * V * args.steps / (gemm_ms / 1e3) / 1e12 if gemm_ms else None

    # ---------------------------------------------------------- end to end
    e2e = None
    if not args.no_e2e:
        pin = lambda t: t.cpu().pin_memory() if t is not None else None  # noqa: E731
        host = [pin(inp["hidden"]), pin(inp["targets"]), pin(loss_mask), pin(offsets),
                pin(inp["grad_logprob"]), pin(g_ent)]
        h2d = sum(t.numel() * t.element_size() for t in host if t is not None)
        d2h = 2 * N * 4
        if args.keep_off:
            host[2] = host[3] = None
            h2d = sum(t.numel() * t.element_size() for t in host if t is not None)

        from sft_keep_mask_gb300.api import StepPipeline
        pipe = StepPipeline(step, lambda: (lp, ent), host, device=dev)
        pipe.run([host] * 2)
        barrier()
        t0 = time.perf_counter()
        pipe.run([host] * args.steps)
        barrier()
        el = time.perf_counter() - t0
        el, _ = reduce_over_ranks(el, 0, world, dev)
        if L.lmhead_get_status(ws) != 0:
            raise RuntimeError("device status non-zero after the end-to-end steps")
        e2e = {"value": nk_total * args.steps / el, "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": 1e3 * el / args.steps,
               "copies": "in: hidden, targets, loss mask, sequence offsets, grad_logprob, "
                         "grad_entropy; out: logprob and entropy. dhidden and dW stay on the "
                         "device (they feed the caller's backward and optimizer)"}

    # ---------------------------------------------------------- CPU oracle
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import numpy as np
        # the keep-off arm scores every row (its keep buffer is never filled)
        keep_np = np.ones(N, np.uint8) if args.keep_off else keep.cpu().numpy()
        W64 = inp["weight"].float().cpu().double().numpy()
        rows = min(args.cpu_rows, nk)
        rate, dt = cpu_oracle_rate(inp, keep_np, W64, rows, args.mode, g_ent is not None)
        what = "forward + dhidden + dW contribution" if args.mode == "fwdbwd" else "forward"
        cpu = {"value": rate, "unit": UNIT, "cores": _oracle_cores(), "kind": "oracle",
               "sample": f"{rows} kept rows, full H and V: {what} in the C float64 oracle "
                         f"(OpenMP, {dt:.1f} s)"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": run_config(args, N, H, V, nk, world, g_ent is not None),
            "peak_device_mem_gb": torch.cuda.max_memory_allocated(dev) / 1e9,
            "logits_bf16_gb_avoided": N * V * 2 / 1e9,
            "step_ms": {"min": min(step_ms), "median": statistics.median(step_ms),
                        "max": max(step_ms)},
            "pass_ms": {"fwd": statistics.median(fwd_ms),
                        "bwd": statistics.median(bwd_ms) if args.mode == "fwdbwd" else None},
            "tflops": tflops, "frac_of_peak": tflops / burst,
            "frac_of_sustained_peak": tflops / sustained,
            "tflops_recompute_free": tflops_rf,
            "gemm_tflops": gemm_tflops,
            "roofline": roof, "kernels": kernels, "gpu_launches": launches,
            "clocks": clk.summary(), "device_status": status_timed, "e2e": e2e,
            "cpu_baseline": cpu,
        }
        # under the power limit the step time is energy / power: the median
        # board power over the timed region times the step time (this GPU).
        # The board's power reading trails the load by a fraction of a
        # second, so it is used only over timed regions of 1.5 s or more.
        pw = line["clocks"]["power_w"]
        if pw is not None and world == 1 and sec >= 1.5 and line["clocks"]["samples"] >= 10:
            j = pw * ms_max / args.steps / 1e3
            line["energy"] = {"board_w_median": pw, "j_per_step": j,
                              "pj_per_flop": j / flops_step * 1e12 if flops_step else None}
        rec = recorded_traffic(roof["kernel"], line["config"])
        if rec is not None:
            roof["traffic"] = rec["dram_bytes_per_launch"]
            cap = rec["capture"]
            roof["traffic_note"] = (
                "ncu dram__bytes_read.sum + dram__bytes_write.sum of this kernel (current sources) "
                f"on the same workload at V = {cap.get('V')}: {rec['scaling']}; algorithmic "
                f"bytes per launch {rec['algorithmic_bytes_per_launch']:.4g}")
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def run_sls(args):
    """Scoring of existing bf16 logits (selective_log_softmax), fwd + bwd."""
    import torch
    from sft_keep_mask_gb300 import lmhead as L
    from sft_keep_mask_gb300 import synth
    world, rank, local = _dist()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    L.lib()
    N, V = (args.rows or 16384), (args.vocab or 151936)
    d = synth.make_logits(N, V, seed=60 + rank, device=dev)
    z = d["logits"]
    lp = torch.empty(N, device=dev)
    ent = torch.empty(N, device=dev)
    lse = torch.empty(N, device=dev)
    dz = torch.empty_like(z)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        L.lmhead_selective_log_softmax_fwd(z, d["targets"], None, True, lp, ent, lse, st, stream)
        L.lmhead_selective_log_softmax_bwd(z, d["targets"], None, lse, ent, d["grad_logprob"],
                                           d["grad_entropy"], dz, st, stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    L.lmhead_profile_enable(True)
    L.lmhead_profile_read()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
    L.lmhead_profile_enable(False)
    prof = L.lmhead_profile_read()
    if int(st.item()) != 0:
        raise RuntimeError("device status non-zero")
    ms = e0.elapsed_time(e1)
    _, _, hbm, src = _peaks()
    elem = float(N) * V
    fwd_ms, bwd_ms = prof["sls_fwd"][1], prof["sls_bwd"][1]
    fwd_gbs = 2 * elem * args.steps / (fwd_ms / 1e3) / 1e9
    bwd_gbs = 4 * elem * args.steps / (bwd_ms / 1e3) / 1e9
    dom, ach = ("sls_bwd", bwd_gbs) if bwd_ms >= fwd_ms else ("sls_fwd", fwd_gbs)
    line = {
        "metric": "selective_log_softmax fwd+bwd rows/s (HBM GB/s of measured peak)",
        "value": N * args.steps / (ms / 1e3), "unit": "rows/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": "selective_log_softmax", "N": N, "V": V,
                   "logits": "bf16 ~N(0, 4)", "l2": "inputs larger than L2 (5 GB logits)"},
        "gbs": {"sls_fwd": fwd_gbs, "sls_bwd": bwd_gbs},
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": ach, "peak": hbm, "unit": "GB/s",
                     "frac": ach / hbm, "peak_source": src, "traffic": None},
        "clocks": clk.summary(),
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="moe30b_rl_half")
    ap.add_argument("--chunk-rows", type=int, default=0)
    ap.add_argument("--rows", type=int, default=0, help="override N (profiling cases)")
    ap.add_argument("--vocab", type=int, default=0, help="override V (profiling cases)")
    ap.add_argument("--entropy-grad", type=int, default=-1,
                    help="1: differentiable entropy, 0: metric-only (default: the workload's)")
    ap.add_argument("--mode", default="fwdbwd", choices=["fwdbwd", "fwd"])
    ap.add_argument("--keep-off", action="store_true",
                    help="score every row (keep mask off), the comparison arm")
    ap.add_argument("--blocksparse", action="store_true",
                    help="score the active 256-row tiles in place instead of compacting")
    ap.add_argument("--active-frac", type=float, default=1.0,
                    help="active suffix fraction of the entropy_bonus workload")
    ap.add_argument("--ref-rows", type=int, default=32,
                    help="kept rows the oracle scores per step of --impl reference")
    ap.add_argument("--cpu-rows", type=int, default=256,
                    help="kept rows of the cpu_baseline sample (about 16 s of oracle work "
                         "at the default shape on 16 Arm cores)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    plan = launch_plan(args.gpus, os.environ)
    if plan == "spawn":
        sys.exit(spawn_ranks(args.gpus, sys.argv[1:]))
    if plan != "run":
        print(plan, file=sys.stderr)
        sys.exit(2)
    if args.impl == "reference":
        run_reference(args)
    elif args.workload == "selective_log_softmax":
        run_sls(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()

"""Runtime behaviour of the C ABI: CUDA-graph capture of a whole forward +
backward step and the device-side kept-row count."""

import numpy as np
import pytest
import torch

from sft_keep_mask_gb300 import lmhead as L
from sft_keep_mask_gb300 import synth
from sft_keep_mask_gb300.api import LMHeadScorer

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_forward_backward_step_replays_from_a_cuda_graph():
    w = synth.workload("moe30b_rl", seed=130, N=2048, H=256, V=3000)
    inp = synth.make_inputs(w, device=DEV)
    sc = LMHeadScorer(w.N, w.H, w.V, chunk_rows=512)
    off = np.zeros(len(inp["seq_lens"]) + 1, np.int32)
    off[1:] = np.cumsum(inp["seq_lens"])
    offsets = torch.from_numpy(off).to(DEV)
    keep = torch.empty(w.N, dtype=torch.uint8, device=DEV)
    lp = torch.empty(w.N, device=DEV)
    ent = torch.empty(w.N, device=DEV)
    lse = torch.empty(w.N, device=DEV)
    dh = torch.empty_like(inp["hidden"])
    dW = torch.empty(w.V, w.H, device=DEV)

    def step():
        s = torch.cuda.current_stream()
        L.lmhead_build_keep_mask(inp["components"][0], None, None, offsets, keep, s)
        L.lmhead_fwd(inp["hidden"], inp["weight"], inp["targets"], keep, True, lp, ent, lse,
                     sc.workspace, 512, s)
        L.lmhead_bwd(inp["hidden"], inp["weight"], inp["targets"], keep, lse, ent,
                     inp["grad_logprob"], inp["grad_entropy"], dh, dW, False, sc.workspace,
                     512, s)

    step()  # eager; also the one-time per-process set-up of the library
    torch.cuda.synchronize()
    want = [t.clone() for t in (keep, lp, ent, lse, dh, dW)]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for t in (keep, lp, ent, lse, dh, dW):
        t.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert sc.status() == 0
    for got, exp in zip((keep, lp, ent, lse, dh, dW), want):
        assert torch.equal(got, exp)


def test_kept_rows_on_the_device():
    w = synth.workload("tiny", seed=131, N=999, H=64, V=500)
    inp = synth.make_inputs(w, device=DEV)
    sc = LMHeadScorer(w.N, w.H, w.V)
    sc.forward(inp["hidden"], inp["weight"], inp["targets"], inp["keep"])
    torch.cuda.synchronize()
    assert int(sc.kept_rows().item()) == int(inp["keep"].sum().item())


def test_step_pipeline_overlapped_copies_give_the_same_results():
    # three different batches in pinned host memory; the pipeline copies batch
    # i+1 while batch i computes and must return what direct calls return
    from sft_keep_mask_gb300.api import StepPipeline
    w = synth.workload("tiny", seed=132, N=800, H=128, V=2000)
    batches, direct = [], []
    sc = LMHeadScorer(w.N, w.H, w.V, chunk_rows=256)
    weight = synth.make_inputs(w, device=DEV)["weight"]
    for k in range(3):
        inp = synth.make_inputs(synth.workload("tiny", seed=133 + k, N=800, H=128, V=2000),
                                device=DEV)
        lp, ent, _ = sc.forward(inp["hidden"], weight, inp["targets"], inp["keep"])
        torch.cuda.synchronize()
        direct.append((lp.cpu(), ent.cpu()))
        batches.append([inp["hidden"].cpu().pin_memory(), inp["targets"].cpu().pin_memory(),
                        inp["keep"].cpu().pin_memory()])
    lp = torch.empty(w.N, device=DEV)
    ent = torch.empty(w.N, device=DEV)
    lse = torch.empty(w.N, device=DEV)
    seen = []

    def step(hidden, targets, keep):
        sc.forward(hidden, weight, targets, keep, out=(lp, ent, lse))

    def result():
        return lp, ent

    pipe = StepPipeline(step, result, batches[0], device=DEV)
    for b, want in zip(batches, direct):
        out = pipe.run([b])
        seen.append((out[0].clone(), out[1].clone()))
    out = pipe.run(batches)  # all three back to back: the last one is returned
    assert torch.equal(out[0], direct[-1][0]) and torch.equal(out[1], direct[-1][1])
    for (a, b), (c, d) in zip(seen, direct):
        assert torch.equal(a, c) and torch.equal(b, d)


def test_plain_c_caller():
    # the C ABI used from C alone: cudaMalloc'd buffers, lmhead_fwd /
    # lmhead_bwd, property checks on the results (see the example's header)
    import subprocess
    from sft_keep_mask_gb300 import build as b
    exe = b.build_example()
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "0 bad rows" in r.stdout


def _step_outputs(sc, inp, stream=None):
    lp, ent, lse = sc.forward(inp["hidden"], inp["weight"], inp["targets"], inp["keep"],
                              stream=stream)
    dh, dW = sc.backward(inp["hidden"], inp["weight"], inp["targets"], inp["keep"], lse, ent,
                         inp["grad_logprob"], inp["grad_entropy"], stream=stream)
    return lp, ent, lse, dh, dW


def test_side_streams_and_two_concurrent_scorers_match_sequential_runs():
    # two independent problems, each with its own workspace: run one after
    # the other on the default stream, then concurrently on two side streams;
    # the persistent kernels share the SMs but no state, so every output must
    # be bit-identical
    wa = synth.workload("tiny", seed=140, N=1500, H=320, V=5000)
    wb = synth.workload("tiny", seed=141, N=1100, H=256, V=3300)
    ia, ib = synth.make_inputs(wa, device=DEV), synth.make_inputs(wb, device=DEV)
    sa = LMHeadScorer(wa.N, wa.H, wa.V, chunk_rows=256)
    sb = LMHeadScorer(wb.N, wb.H, wb.V, chunk_rows=256)
    ref_a = _step_outputs(sa, ia)
    ref_b = _step_outputs(sb, ib)
    torch.cuda.synchronize()
    ref_a = [t.clone() for t in ref_a]
    ref_b = [t.clone() for t in ref_b]

    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    s1.wait_stream(torch.cuda.current_stream())
    s2.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s1):
        got_a = _step_outputs(sa, ia)  # the binding picks up s1 as the current stream
    with torch.cuda.stream(s2):
        got_b = _step_outputs(sb, ib, stream=s2)
    torch.cuda.synchronize()
    assert sa.status() == 0 and sb.status() == 0
    names = ("lp", "ent", "lse", "dh", "dW")
    for name, r, g in zip([f"a.{n}" for n in names] + [f"b.{n}" for n in names],
                          list(ref_a) + list(ref_b), list(got_a) + list(got_b)):
        assert torch.equal(r, g), name


def test_one_scorer_serves_smaller_batches():
    # the workspace of an N-row scorer serves any batch of at most N rows; the
    # results equal those of a scorer sized for the batch, bit for bit
    big = LMHeadScorer(1000, 192, 3000, chunk_rows=256)
    for n, seed in ((600, 150), (1000, 151), (37, 152)):
        w = synth.workload("tiny", seed=seed, N=n, H=192, V=3000)
        inp = synth.make_inputs(w, device=DEV)
        exact = LMHeadScorer(n, 192, 3000, chunk_rows=256)
        got = _step_outputs(big, inp)
        want = _step_outputs(exact, inp)
        torch.cuda.synchronize()
        assert big.status() == 0
        for g, r in zip(got, want):
            assert g.shape == r.shape and torch.equal(g, r)
    w = synth.workload("tiny", seed=153, N=1001, H=192, V=3000)
    inp = synth.make_inputs(w, device=DEV)
    with pytest.raises(ValueError, match="capacity"):
        big.forward(inp["hidden"], inp["weight"], inp["targets"], inp["keep"])


_ALLOC_SCRIPT = """
import torch
from sft_keep_mask_gb300 import synth
from sft_keep_mask_gb300.api import LMHeadScorer
w = synth.workload("tiny", seed=5, N=600, H=128, V=2000)
inp = synth.make_inputs(w, device="cuda")
sc = LMHeadScorer(w.N, w.H, w.V)
lp, ent, lse = sc.forward(inp["hidden"], inp["weight"], inp["targets"], inp["keep"])
dh, dW = sc.backward(inp["hidden"], inp["weight"], inp["targets"], inp["keep"], lse, ent,
                     inp["grad_logprob"], inp["grad_entropy"])
torch.cuda.synchronize()
assert sc.status() == 0
print(repr(float(lp.double().sum())), repr(float(dW.double().abs().sum())))
"""


def test_memory_from_every_torch_allocator_mode_is_accepted():
    # the entry points refuse pointers that are not device memory of the
    # current device; tensors from the expandable-segment (virtual memory)
    # and cudaMallocAsync allocators are device memory and must pass, with
    # the same results as the default allocator
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    outs = []
    for conf in (None, "expandable_segments:True", "backend:cudaMallocAsync"):
        env = dict(os.environ)
        env.pop("PYTORCH_CUDA_ALLOC_CONF", None)
        if conf:
            env["PYTORCH_CUDA_ALLOC_CONF"] = conf
        r = subprocess.run([sys.executable, "-c", _ALLOC_SCRIPT], env=env, cwd=root,
                           capture_output=True, text=True, timeout=600)
        assert r.returncode == 0, (conf, r.stderr[-2000:])
        outs.append(r.stdout.strip().splitlines()[-1])
    assert len(set(outs)) == 1, outs


def test_two_host_threads_with_their_own_streams_and_scorers():
    # ctypes releases the GIL during library calls, so two host threads drive
    # the library at the same time (the launch counter, profiling records and
    # the per-device set-up are shared host state); each thread repeats its
    # own problem on its own stream, and every result must equal a
    # single-threaded run bit for bit
    import threading
    problems = []
    for seed, (N, H, V) in ((160, (1200, 256, 4000)), (161, (900, 192, 3100))):
        w = synth.workload("tiny", seed=seed, N=N, H=H, V=V)
        inp = synth.make_inputs(w, device=DEV)
        sc = LMHeadScorer(N, H, V, chunk_rows=256)
        ref = [t.clone() for t in _step_outputs(sc, inp)]
        problems.append((sc, inp, ref))
    torch.cuda.synchronize()
    errors = []

    def worker(sc, inp, ref):
        try:
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.default_stream())
            with torch.cuda.stream(s):
                for _ in range(5):
                    got = _step_outputs(sc, inp)
                    s.synchronize()
                    if sc.status() != 0 or not all(torch.equal(a, b) for a, b in zip(got, ref)):
                        errors.append("mismatch")
                        return
        except Exception as e:  # surfaced by the assertion below
            errors.append(repr(e))

    L.lmhead_profile_enable(True)
    try:
        threads = [threading.Thread(target=worker, args=p) for p in problems]
        for t in threads:
            t.start()
        for t in threads:
            t.join()
    finally:
        L.lmhead_profile_enable(False)
        L.lmhead_profile_read()
    assert not errors, errors

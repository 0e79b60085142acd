#!/usr/bin/env python3
"""Decode-step benchmark: one hybrid decode layer (KDA + routed MoE) plus one speculative
window (verify, accept, replay) per step, through the C-ABI library.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Workload of one step (synthetic, seeded):
  * hybrid decode layer, batch 64: RMSNorm(7168) -> q/k/v/gate/beta projection
    (7168 -> 32x128 x4 + 32) -> KDA step on 64 fp32 states [32,128,128] -> output
    projection 4096 -> 7168 + residual -> RMSNorm -> router (256 experts, top-8, sigmoid)
    -> routed SwiGLU experts (intermediate 2048, ~22.5 GB of bf16 weights) + 1 shared
    expert + residual, with the side-stream L2 prefetch;
  * speculative window on 16 other sequences, 4 drafted tokens each: verify (no state
    write), accepted-length bookkeeping (accepted length uniform in 0..4), replay of the
    accepted prefix from the committed state.
The metric is achieved HBM bandwidth over the step: algorithmic bytes (weights streamed,
states read and written, activations; scratch traffic not credited) / step time.  The
step's working set (~20 GB) is far larger than the 129 MB L2, so every step reads cold.

The one JSON line also carries: µs per step, a roofline entry for the dominant kernel
(routed-expert gate/up streaming, timed live with CUDA events on its launching stream),
an end-to-end number through host buffers, clocks sampled during the timed region, the
number of library kernel launches, batch sweeps, and the fp64 oracle timed on the host
cores as the CPU baseline.  `--impl reference` times that oracle alone as the reference
arm on a bounded sample of the same workload.
"""

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode µs/step and achieved HBM GB/s (KDA + MoE) vs GB300 peak at batch 1–64"
CFG = dict(M=64, Hd=7168, H=32, d=128, E=256, k=8, I=2048, n_shared=1, eps=1e-6,
           spec_B=16, spec_T=4)
# draft length of the spec sweep's windows (the headline step keeps spec_T = 4)
SWEEP_T = int(os.environ.get("HLA_BENCH_SPEC_T", "4"))
ROTATE = 4  # distinct input batches cycled through the timed steps


# ----------------------------------------------------------------------------- bytes

def layer_bytes(M, U, c=CFG):
    """Algorithmic HBM bytes of one decode layer over M sequences with U active experts."""
    Hd, H, d, E, k, I, ns = c["Hd"], c["H"], c["d"], c["E"], c["k"], c["I"], c["n_shared"]
    Nq = 4 * H * d + H
    b = dict(
        rmsnorm=2 * (2 * M * Hd * 2 + Hd * 2),
        qkvg=Nq * Hd * 2 + M * Hd * 2 + 3 * M * H * d * 2 + M * H * d * 4 + M * H * 4,
        kda=M * H * (8 * d * d + 3 * d * 2 + d * 4 + 4 + d * 2),
        oproj=Hd * H * d * 2 + M * H * d * 2 + 2 * M * Hd * 2,
        router=E * Hd * 2 + M * Hd * 2 + M * k * 8,
        experts=(U + ns) * 3 * I * Hd * 2 + 3 * M * Hd * 2,
    )
    return b


def spec_bytes(B, T, accepted, c=CFG):
    H, d = c["H"], c["d"]
    tok = 3 * d * 2 + d * 4 + 4
    return dict(verify=B * H * (4 * d * d + T * (tok + 4 * d)),
                accept=2 * B * T * 4 + 3 * B * 4,
                replay=sum(H * (8 * d * d + int(a) * tok) for a in accepted if a > 0))


def gateup_bytes(M, U, c=CFG):
    """Algorithmic bytes of one routed+shared gate/up launch."""
    P = M * (c["k"] + c["n_shared"])
    return (U + c["n_shared"]) * 2 * c["I"] * c["Hd"] * 2 + M * c["Hd"] * 2 + P * c["I"] * 2


def kda_bytes(B, c=CFG, o_bytes=4):
    H, d = c["H"], c["d"]
    return B * H * (8 * d * d + 3 * d * 2 + d * 4 + 4 + d * o_bytes)


# ----------------------------------------------------------------------------- host helpers

def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms while measuring."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu, self.proc, self.path = gpu_index, None, None

    def start(self):
        try:
            self.path = os.path.join(tempfile.mkdtemp(prefix="hla_clocks_"), f"clocks_rank{self.gpu}.csv")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.5)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return dict(sm_mhz=None, sm_max_mhz=None, reasons=["unsampled"], samples=0)
        time.sleep(0.3)
        self.proc.terminate()
        self.proc.wait()
        sm, smax, reasons, n = [], [], set(), 0
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            n += 1
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return dict(sm_mhz=statistics.median(sm) if sm else None,
                    sm_max_mhz=max(smax) if smax else None, reasons=sorted(reasons), samples=n)


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def round_up16(n):
    return (n + 15) // 16 * 16


def reduce_over_ranks(elapsed_s, nbytes, world):
    """(max elapsed over ranks, total bytes over ranks); identity on one rank."""
    if world <= 1:
        return elapsed_s, nbytes
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=dev)
    b = torch.tensor([float(nbytes)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(b, op=dist.ReduceOp.SUM)
    return float(t.item()), float(b.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------------------- GPU arm

class launch_chain:
    """Brackets library calls queued back to back on the current stream as one launch chain
    (hla_chain_begin / hla_chain_end) unless HLA_BENCH_CHAIN=0."""

    def __init__(self, hla):
        self.hla = hla
        self.on = os.environ.get("HLA_BENCH_CHAIN", "1") == "1"

    def __enter__(self):
        if self.on:
            self.hla.hla_chain_begin()

    def __exit__(self, *exc):
        if self.on:
            self.hla.hla_chain_end()
        return False


class Workload:
    """Device-resident weights, states, rotating inputs and workspaces of one step."""

    def __init__(self, dev, rank, prefetch=True):
        import torch
        from hybrid_linear_attention_gated_gb300 import hla, inputs
        self.torch, self.hla, self.inputs, self.dev = torch, hla, inputs, dev
        c = CFG
        seed = 100 * rank
        self.w = inputs.moe_weights(c["E"], c["Hd"], c["I"], c["n_shared"],
                                    inputs.generator(seed + 3, dev), device=dev)
        self.w.update(inputs.layer_weights(c["Hd"], c["H"], c["d"], c["d"],
                                           inputs.generator(seed + 4, dev), device=dev))
        self.L = hla.make_layer(c["Hd"], c["H"], c["d"], c["d"], c["E"], c["k"], c["I"],
                                c["n_shared"], c["eps"], self.w)
        M, H, d = c["M"], c["H"], c["d"]
        g = inputs.generator(seed + 5, dev)
        self.S = self.warm_states(M, g)
        self.S_spec = self.warm_states(c["spec_B"], g)
        self.x = [inputs.activations(M, c["Hd"], g, dev) for _ in range(ROTATE)]
        B, T = c["spec_B"], c["spec_T"]
        self.win, self.ids = [], []
        for _ in range(ROTATE):
            self.win.append(inputs.kda_inputs((B, T), H, d, d, g, dev))
            dr, tg, a = inputs.accept_ids(B, T, g, dev)
            self.ids.append((dr, tg, a.cpu().numpy()))
        self.y = torch.empty(M, c["Hd"], dtype=torch.bfloat16, device=dev)
        self.o_spec = torch.empty(B, T, H, d, device=dev)
        self.acc = torch.zeros(B, dtype=torch.int32, device=dev)
        self.com = torch.zeros(B, dtype=torch.int32, device=dev)
        self.ws_bytes = hla.hla_decode_layer_workspace_size(self.L, M)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=dev)
        self.side = torch.cuda.Stream(device=dev) if prefetch else 0

    def warm_states(self, B, g):
        """States after 256 prior updates from zero, produced by the decode kernel itself."""
        torch, hla, inputs = self.torch, self.hla, self.inputs
        H, d = CFG["H"], CFG["d"]
        S = torch.zeros(B, H, d, d, device=self.dev)
        o = torch.empty(B, H, d, device=self.dev)
        for _ in range(256):
            u = inputs.kda_inputs((B,), H, d, d, g, self.dev)
            hla.kda_decode_step(B, H, d, d, S, None, u["q"], u["k"], u["v"], u["alpha"], u["beta"], o)
        return S

    def step(self, i, x=None, win=None, ids=None):
        hla, c = self.hla, CFG
        r = i % ROTATE
        x = self.x[r] if x is None else x
        win = self.win[r] if win is None else win
        dr, tg = (self.ids[r][0], self.ids[r][1]) if ids is None else ids
        B, T, H, d = c["spec_B"], c["spec_T"], c["H"], c["d"]
        # one launch chain: the layer's kernels, then the window's, back to back on this stream
        with launch_chain(hla):
            hla.hla_decode_layer(self.L, c["M"], x, self.S, None, self.y, self.ws, self.ws_bytes,
                                 prefetch_stream=self.side)
            hla.kda_spec_verify_replay(hla.HLA_SPEC_VERIFY, B, T, H, d, d, self.S_spec, None, win["q"],
                                       win["k"], win["v"], win["alpha"], win["beta"], None, self.o_spec)
            hla.spec_accept_prefix(B, T, dr, tg, self.acc, self.com)
            hla.kda_spec_verify_replay(hla.HLA_SPEC_REPLAY, B, T, H, d, d, self.S_spec, None, win["q"],
                                       win["k"], win["v"], win["alpha"], win["beta"], self.acc, None)

    def active_experts(self):
        torch = self.torch
        ip, _ = self.hla.hla_decode_layer_routing(self.L, CFG["M"], self.ws)
        idx = torch.empty(CFG["M"] * CFG["k"], dtype=torch.int32, device=self.dev)
        # copy from the workspace address into a tensor
        src = self.ws[ip - self.ws.data_ptr(): ip - self.ws.data_ptr() + idx.numel() * 4]
        idx.view(torch.uint8).copy_(src)
        return int(torch.unique(idx).numel())


def time_steps(torch, fn, steps, world, label="timed"):
    """Run fn(0..steps-1) between two CUDA events on the current stream, bracketed by a
    barrier and a device synchronise on both sides, inside an NVTX start/end range."""
    barrier(world)
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    rid = torch.cuda.nvtx.range_start(label)
    e0.record(st)
    for i in range(steps):
        fn(i)
    e1.record(st)
    torch.cuda.synchronize()
    torch.cuda.nvtx.range_end(rid)
    barrier(world)
    return e0.elapsed_time(e1) / 1e3


def graph_time(torch, fn, iters, reps=3):
    """Capture `iters` calls of fn(i) in one CUDA graph; median replay time per call (s)."""
    fn(0)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for i in range(iters):
                fn(i)
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    out = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        out.append(e0.elapsed_time(e1) / 1e3 / iters)
    del g
    return statistics.median(out)


def kda_sweep(torch, hla, inputs, dev, peak):
    """KDA decode step alone at B in {1,2,8,32,64}: states rotated over a 512 MB pool (> 3x L2)."""
    H, d = CFG["H"], CFG["d"]
    pool_slots = 512 * 2 ** 20 // (H * d * d * 4)
    pool = torch.randn(pool_slots, H, d, d, device=dev).mul_(0.05)
    res = []
    for B in (1, 2, 8, 32, 64):
        iters = max(8, min(200, pool_slots // B))
        g = inputs.generator(7000 + B, dev)
        u = inputs.kda_inputs((B,), H, d, d, g, dev)
        o = torch.empty(B, H, d, device=dev)
        idxs = [torch.arange(i * B, (i + 1) * B, dtype=torch.int32, device=dev) % pool_slots
                for i in range(iters)]

        def fn(i):
            hla.kda_decode_step(B, H, d, d, pool, idxs[i], u["q"], u["k"], u["v"], u["alpha"],
                                u["beta"], o)
        t = graph_time(torch, fn, iters)
        gbs = kda_bytes(B) / t / 1e9
        res.append(dict(batch=B, us=round(t * 1e6, 2), tokens_per_s=round(B / t), gbs=round(gbs, 1),
                        frac=round(gbs / peak, 3), variant=hla.hla_last_variant()))
    del pool
    return res


def moe_sweep(torch, hla, inputs, wl, dev, peak):
    """Router + experts alone at M in {1,2,8,32,64} (the weights are ~22.5 GB: always cold), the two
    calls bracketed as one launch chain (HLA_BENCH_CHAIN=0: plain)."""
    c = CFG
    res = []
    for M in (1, 2, 8, 32, 64):
        g = inputs.generator(8000 + M, dev)
        xs = [inputs.activations(M, c["Hd"], g, dev) for _ in range(ROTATE)]
        idx = torch.empty(M, c["k"], dtype=torch.int32, device=dev)
        wt = torch.empty(M, c["k"], device=dev)
        rb = hla.moe_route_topk_workspace_size(M, c["Hd"], c["E"])
        rws = torch.empty(max(rb, 256), dtype=torch.uint8, device=dev)
        nb = hla.moe_expert_forward_workspace_size(M, c["Hd"], c["I"], c["E"], c["k"], c["n_shared"])
        mws = torch.empty(nb, dtype=torch.uint8, device=dev)
        y = torch.empty(M, c["Hd"], dtype=torch.bfloat16, device=dev)
        w = wl.w
        us = []
        for r in range(ROTATE):
            hla.moe_route_topk(M, c["Hd"], c["E"], c["k"], xs[r], w["W_r"], idx, wt, None, rws, rb)
            us.append(int(torch.unique(idx).numel()))

        def fn(i):
            x = xs[i % ROTATE]
            with launch_chain(hla):  # the router's top-k and the dispatch as one chain, as in the layer
                hla.moe_route_topk(M, c["Hd"], c["E"], c["k"], x, w["W_r"], idx, wt, None, rws, rb)
                hla.moe_expert_forward(M, c["Hd"], c["I"], c["E"], c["k"], c["n_shared"], x, idx, wt,
                                       w["W_gate"], w["W_up"], w["W_down"], w["Ws_gate"], w["Ws_up"],
                                       w["Ws_down"], None, y, mws, nb)
        t = graph_time(torch, fn, 4 * ROTATE)
        U = statistics.mean(us)
        nbytes = layer_bytes(M, U)["router"] + layer_bytes(M, U)["experts"]
        gbs = nbytes / t / 1e9
        res.append(dict(tokens=M, active_experts=U, us=round(t * 1e6, 1), tokens_per_s=round(M / t),
                        gbs=round(gbs, 1), frac=round(gbs / peak, 3), variant=hla.hla_last_variant()))
    return res


def extend_sweep(torch, hla, inputs, dev, peak):
    """Mixed batches through kda_extend: decoding sequences (1 token) next to prefill chunks,
    states in a rotating pool larger than L2.  Tokens of one sequence are applied in order
    (the recurrent form), so a long chunk is a serial chain."""
    c = CFG
    H, d = c["H"], c["d"]
    tok_bytes = 3 * d * 2 + d * 4 + 4 + 4 * d
    pool_slots = 512 * 2 ** 20 // (H * d * d * 4)
    pool = torch.randn(pool_slots, H, d, d, device=dev).mul_(0.05)
    res = []
    for name, lens in (("64 decode", [1] * 64), ("60 decode + 4 x 32-token chunks", [1] * 60 + [32] * 4),
                       ("60 decode + 4 x 128-token chunks", [1] * 60 + [128] * 4),
                       ("4 x 512-token chunks", [512] * 4)):
        B = len(lens)
        cu = torch.tensor([0] + list(__import__("itertools").accumulate(lens)), dtype=torch.int32, device=dev)
        N = int(cu[-1])
        u = inputs.kda_inputs((N,), H, d, d, inputs.generator(7800 + N, dev), dev)
        o = torch.empty(N, H, d, device=dev)
        iters = max(4, min(32, pool_slots // B))
        idxs = [torch.arange(i * B, (i + 1) * B, dtype=torch.int32, device=dev) % pool_slots
                for i in range(iters)]

        def fn(i, B=B, cu=cu, u=u, o=o, idxs=idxs):
            hla.kda_extend(B, cu, H, d, d, pool, idxs[i % len(idxs)], u["q"], u["k"], u["v"],
                           u["alpha"], u["beta"], o)
        t = graph_time(torch, fn, iters)
        nbytes = B * H * 8 * d * d + N * H * tok_bytes
        res.append(dict(batch=name, tokens=N, us=round(t * 1e6, 2), tokens_per_s=round(N / t),
                        gbs=round(nbytes / t / 1e9, 1), frac=round(nbytes / t / 1e9 / peak, 3)))
    del pool
    return res


def spec_sweep(torch, hla, inputs, wl, dev, peak):
    """Speculative window, T=4, accepted length uniform in 0..4, at B=16 and B=64, two forms per
    step: separate (verify + accept + replay) and fused (replay of the previous window with the
    verify of the next + accept); and the verify and replay programs each alone.  Each step takes
    the next B committed states of a 768 MB pool (> 3x L2) through state_idx, so every step reads
    its states from HBM; the inputs rotate through 4 windows.  tokens/s counts accepted tokens
    (verify alone: the drafted tokens it scores)."""
    c = CFG
    T, H, d = SWEEP_T, c["H"], c["d"]
    tok = 3 * d * 2 + d * 4 + 4
    pool_slots = 768 * 2 ** 20 // (H * d * d * 4)
    pool = torch.randn(pool_slots, H, d, d, device=dev).mul_(0.05)
    res = []
    for B in (16, 64):
        if B == c["spec_B"] and T == c["spec_T"]:
            wins, ids = wl.win, wl.ids
        else:
            g = inputs.generator(7700 + B, dev)
            wins, ids = [], []
            for _ in range(ROTATE):
                wins.append(inputs.kda_inputs((B, T), H, d, d, g, dev))
                dr, tg, a = inputs.accept_ids(B, T, g, dev)
                ids.append((dr, tg, a.cpu().numpy()))
        o = torch.empty(B, T, H, d, device=dev)
        acc = torch.zeros(B, dtype=torch.int32, device=dev)
        com = torch.zeros(B, dtype=torch.int32, device=dev)
        iters = 4 * ROTATE
        sets = pool_slots // B
        idxs = [torch.arange((i % sets) * B, (i % sets + 1) * B, dtype=torch.int32, device=dev)
                for i in range(iters)]

        def separate(i, B=B, wins=wins, ids=ids, o=o, acc=acc, com=com, idxs=idxs):
            w = wins[i % ROTATE]
            dr, tg, _ = ids[i % ROTATE]
            with launch_chain(hla):
                hla.kda_spec_verify_replay(hla.HLA_SPEC_VERIFY, B, T, H, d, d, pool, idxs[i], w["q"], w["k"],
                                           w["v"], w["alpha"], w["beta"], None, o)
                hla.spec_accept_prefix(B, T, dr, tg, acc, com)
                hla.kda_spec_verify_replay(hla.HLA_SPEC_REPLAY, B, T, H, d, d, pool, idxs[i], w["q"], w["k"],
                                           w["v"], w["alpha"], w["beta"], acc, None)

        def fused(i, B=B, wins=wins, ids=ids, o=o, acc=acc, com=com, idxs=idxs):
            p_, w = wins[(i + ROTATE - 1) % ROTATE], wins[i % ROTATE]
            dr, tg, _ = ids[i % ROTATE]
            with launch_chain(hla):
                hla.kda_spec_replay_verify(B, T, T, H, d, d, pool, idxs[i], p_["q"], p_["k"], p_["v"],
                                           p_["alpha"], p_["beta"], acc, w["q"], w["k"], w["v"],
                                           w["alpha"], w["beta"], o)
                hla.spec_accept_prefix(B, T, dr, tg, acc, com)
        accs = [torch.from_numpy(ids[r][2].astype("int32")).to(dev) for r in range(ROTATE)]

        def verify_only(i, B=B, wins=wins, o=o, idxs=idxs):
            w = wins[i % ROTATE]
            hla.kda_spec_verify_replay(hla.HLA_SPEC_VERIFY, B, T, H, d, d, pool, idxs[i], w["q"], w["k"],
                                       w["v"], w["alpha"], w["beta"], None, o)

        def replay_only(i, B=B, wins=wins, accs=accs, idxs=idxs):
            w = wins[i % ROTATE]
            hla.kda_spec_verify_replay(hla.HLA_SPEC_REPLAY, B, T, H, d, d, pool, idxs[i], w["q"], w["k"],
                                       w["v"], w["alpha"], w["beta"], accs[i % ROTATE], None)
        mean_sep = statistics.mean(sum(spec_bytes(B, T, ids[r][2]).values()) for r in range(ROTATE))
        mean_ver = statistics.mean(spec_bytes(B, T, ids[r][2])["verify"] for r in range(ROTATE))
        mean_rep = statistics.mean(spec_bytes(B, T, ids[r][2])["replay"] for r in range(ROTATE))
        mean_fused = statistics.mean(
            B * H * 4 * d * d + sum(H * (4 * d * d + int(a) * tok) for a in ids[r][2] if a > 0)
            + B * H * T * (tok + 4 * d) + 2 * B * T * 4 + 3 * B * 4 for r in range(ROTATE))
        accepted = statistics.mean(float(sum(ids[r][2])) for r in range(ROTATE))
        for name, fn, nbytes, ntok in (("separate", separate, mean_sep, accepted),
                                       ("fused", fused, mean_fused, accepted),
                                       ("verify alone", verify_only, mean_ver, float(B * T)),
                                       ("replay alone", replay_only, mean_rep, accepted)):
            t = graph_time(torch, fn, iters)
            res.append(dict(batch=B, form=name, us=round(t * 1e6, 2), bytes=round(nbytes),
                            accepted_tokens=accepted, tokens_per_s=round(ntok / t),
                            gbs=round(nbytes / t / 1e9, 1), frac=round(nbytes / t / 1e9 / peak, 3)))
    del pool
    return res


def layer_sweep(torch, hla, inputs, wl, dev, peak):
    c = CFG
    res = []
    for M in (1, 8, 64):
        g = inputs.generator(9000 + M, dev)
        xs = [inputs.activations(M, c["Hd"], g, dev) for _ in range(ROTATE)]
        S = wl.S[:M].clone()
        y = torch.empty(M, c["Hd"], dtype=torch.bfloat16, device=dev)
        nb = hla.hla_decode_layer_workspace_size(wl.L, M)
        ws = torch.empty(nb, dtype=torch.uint8, device=dev)

        def fn(i):
            hla.hla_decode_layer(wl.L, M, xs[i % ROTATE], S, None, y, ws, nb, prefetch_stream=wl.side)
        t = graph_time(torch, fn, 4 * ROTATE)
        ip, _ = hla.hla_decode_layer_routing(wl.L, M, ws)
        off = ip - ws.data_ptr()
        U = int(torch.unique(ws[off:off + M * c["k"] * 4].view(torch.int32)).numel())
        nbytes = sum(layer_bytes(M, U).values())
        gbs = nbytes / t / 1e9
        res.append(dict(batch=M, active_experts=U, us=round(t * 1e6, 1), tokens_per_s=round(M / t),
                        gbs=round(gbs, 1), frac=round(gbs / peak, 3)))
    return res


def traffic_entry(kernel, units):
    """DRAM bytes per launch from a committed ncu capture (per streamed unit, times the units
    of this launch), or None when the kernel sources changed since the counters were taken."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
            t = json.load(f)[kernel]
    except (OSError, KeyError, ValueError):
        return None
    import hashlib
    h = hashlib.sha256()
    for rel in t["sources"]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    if h.hexdigest() != t["sources_sha256"]:
        return None
    return dict(t, bytes_per_launch=round(t["per_unit_bytes"] * units))


def cpu_baseline(steps=3, warmup=3):
    """The fp64 oracle, as it stands, on the host cores: the reference arm's bounded sample (per
    step the decode layer for one of the 64 sequences and the speculative window for one of the
    16), run in child processes with the BLAS / OpenMP thread pools limited to 1 thread and to
    every core the process may use.  Reported beside the GPU number, not a target."""
    cores = len(os.sched_getaffinity(0))
    runs = {}
    for threads in (cores, 1):
        env = dict(os.environ)
        for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS"):
            env[var] = str(threads)
        cmd = [sys.executable, os.path.abspath(__file__), "--impl", "reference", "--steps", str(steps),
               "--warmup", str(warmup), "--threads", str(threads)]
        r = subprocess.run(cmd, env=env, capture_output=True, text=True, cwd=ROOT)
        line = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
        if r.returncode != 0 or not line:
            runs[threads] = dict(error=(r.stderr or r.stdout)[-300:])
            continue
        runs[threads] = json.loads(line[-1])
    best = runs.get(cores, {})
    one = runs.get(1, {})
    return dict(value=best.get("value"), unit="GB/s", cores=cores, kind="oracle",
                ms_per_step=best.get("ms_per_step"),
                single_thread=dict(value=one.get("value"), unit="GB/s", cores=1,
                                   ms_per_step=one.get("ms_per_step")),
                sample=(best.get("config") or {}).get("sample", "") +
                f" ({steps} timed steps after {warmup} warm-up steps per thread count; weights drawn "
                f"from the same distributions on the host; {os.uname().machine}, {cores} cores)",
                **({"errors": {k: v["error"] for k, v in runs.items() if "error" in v}}
                   if any("error" in v for v in runs.values()) else {}))


def run_ours(args):
    import torch
    from hybrid_linear_attention_gated_gb300 import build, hla, inputs
    world, rank, local = dist_setup()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", init_method="env://")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    build.build()
    hla.load()
    peak, peak_kind = peaks()
    wl = Workload(dev, rank, prefetch=not args.no_prefetch)
    c = CFG
    for i in range(args.warmup):
        wl.step(i)
    torch.cuda.synchronize()

    sampler = ClockSampler(local)
    sampler.start()
    # the states as they enter the timed region: the same steps are replayed from them afterwards
    # to read each timed step's routing (the kernels are deterministic, so the replay takes the
    # same routing decisions; its final states are checked bit for bit against the timed run's)
    snap = [t.clone() for t in (wl.S, wl.S_spec, wl.acc, wl.com)]
    hla.hla_trace_enable("moe_gateup", args.steps)
    n0 = hla.hla_launch_count()
    elapsed = time_steps(torch, wl.step, args.steps, world)
    launches = hla.hla_launch_count() - n0
    gu_ms = hla.hla_trace_read(args.steps)
    hla.hla_trace_enable(None, 0)

    # active experts of every timed step, from the deterministic replay
    final = [t.clone() for t in (wl.S, wl.S_spec, wl.acc, wl.com)]
    for t, s0 in zip((wl.S, wl.S_spec, wl.acc, wl.com), snap):
        t.copy_(s0)
    Us = []
    for i in range(args.steps):
        wl.step(i)
        torch.cuda.synchronize()
        Us.append(wl.active_experts())
    replay_bitwise = all(torch.equal(a, b) for a, b in zip((wl.S, wl.S_spec, wl.acc, wl.com), final))
    del snap, final
    U = statistics.mean(Us)
    layer_total = sum(sum(layer_bytes(c["M"], u).values()) for u in Us)
    per_step = layer_bytes(c["M"], U)
    accepted = [wl.ids[i % ROTATE][2] for i in range(args.steps)]
    spec_total = sum(sum(spec_bytes(c["spec_B"], c["spec_T"], a).values()) for a in accepted)
    local_bytes = layer_total + spec_total
    # tokens a step advances: one per decoding sequence, plus the accepted drafted tokens
    local_tokens = c["M"] * args.steps + sum(int(sum(a)) for a in accepted)
    t_max, all_bytes = reduce_over_ranks(elapsed, local_bytes, world)
    _, all_tokens = reduce_over_ranks(elapsed, local_tokens, world)

    # end to end through host buffers: pinned host inputs in, results out, every step.  A step's
    # inputs sit in one pinned buffer and go over in one copy (the library reads them through
    # views of a device staging buffer); its outputs are written into views of one device buffer
    # and come back in one copy.  As a serving loop would, the copies run on a second stream,
    # double-buffered: step i+1's inputs go over and step i-1's outputs come back while step i
    # computes.  The first copy starts after the timer, and the last read-back is joined before
    # it stops.
    def packed(tensors):
        """(pinned uint8 host buffer holding the tensors back to back, [(offset, tensor)])."""
        offs, o = [], 0
        for t in tensors:
            offs.append(o)
            o += round_up16(t.numel() * t.element_size())
        buf = torch.empty(o, dtype=torch.uint8).pin_memory()
        for off, t in zip(offs, tensors):
            n = t.numel() * t.element_size()
            buf[off:off + n].copy_(t.detach().cpu().contiguous().view(-1).view(torch.uint8))
        return buf, list(zip(offs, tensors))

    def view_of(buf, off, like):
        n = like.numel() * like.element_size()
        return buf[off:off + n].view(like.dtype).view(like.shape)

    win_keys = list(wl.win[0].keys())
    stage_h, layout = [], None
    for r in range(ROTATE):
        buf, layout = packed([wl.x[r]] + [wl.win[r][k2] for k2 in win_keys] + [wl.ids[r][0], wl.ids[r][1]])
        stage_h.append(buf)
    out_like = [wl.y, wl.o_spec, wl.acc]
    o_offs, o = [], 0
    for t in out_like:
        o_offs.append(o)
        o += round_up16(t.numel() * t.element_size())
    stage_d = [torch.empty(stage_h[0].numel(), dtype=torch.uint8, device=dev) for _ in range(2)]
    out_d = [torch.empty(o, dtype=torch.uint8, device=dev) for _ in range(2)]
    out_h = [torch.empty(o, dtype=torch.uint8).pin_memory() for _ in range(2)]
    in_views = [[view_of(sd, off, t) for off, t in layout] for sd in stage_d]
    out_views = [[view_of(od, off, t) for off, t in zip(o_offs, out_like)] for od in out_d]
    h2d = stage_h[0].numel()
    d2h = out_h[0].numel()
    cs = torch.cuda.Stream(device=dev)
    ev = {name: [torch.cuda.Event() for _ in range(2)] for name in ("h2d", "comp", "d2h")}

    class E2E:
        """Pipelined end-to-end steps 0..n-1 (call reset(n) before each run)."""

        def reset(self, n):
            self.n = n

        def __call__(self, i):
            main = torch.cuda.current_stream()
            b = i % 2
            if i == 0:
                cs.wait_stream(main)
                with torch.cuda.stream(cs):
                    stage_d[0].copy_(stage_h[0], non_blocking=True)
                    ev["h2d"][0].record(cs)
            if i + 1 < self.n:  # next step's inputs, once step i-1 (same buffer) has computed
                nb = (i + 1) % 2
                if i >= 1:
                    cs.wait_event(ev["comp"][nb])
                with torch.cuda.stream(cs):
                    stage_d[nb].copy_(stage_h[(i + 1) % ROTATE], non_blocking=True)
                    ev["h2d"][nb].record(cs)
            main.wait_event(ev["h2d"][b])
            if i >= 2:
                main.wait_event(ev["d2h"][b])  # step i-2's outputs are back on the host
            v = in_views[b]
            wl.y, wl.o_spec, wl.acc = out_views[b]
            wl.step(i, x=v[0], win=dict(zip(win_keys, v[1:1 + len(win_keys)])), ids=(v[-2], v[-1]))
            ev["comp"][b].record(main)
            cs.wait_event(ev["comp"][b])
            with torch.cuda.stream(cs):
                out_h[b].copy_(out_d[b], non_blocking=True)
                ev["d2h"][b].record(cs)
            if i == self.n - 1:
                main.wait_stream(cs)

    e2e_step = E2E()
    e2e_step.reset(2)
    for i in range(2):
        e2e_step(i)
    torch.cuda.synchronize()
    e2e_step.reset(args.steps)
    e2e_elapsed = time_steps(torch, e2e_step, args.steps, world, label="e2e")
    e2e_max, _ = reduce_over_ranks(e2e_elapsed, 0, world)

    sweeps = {}
    if not args.no_sweep and rank == 0:
        sweeps["kda_decode"] = kda_sweep(torch, hla, inputs, dev, peak)
        sweeps["moe"] = moe_sweep(torch, hla, inputs, wl, dev, peak)
        sweeps["layer"] = layer_sweep(torch, hla, inputs, wl, dev, peak)
        sweeps["spec_window"] = spec_sweep(torch, hla, inputs, wl, dev, peak)
        sweeps["kda_extend"] = extend_sweep(torch, hla, inputs, dev, peak)
    clocks = sampler.stop()

    if rank != 0:
        return
    value = all_bytes / t_max / 1e9
    gu_avg_s = statistics.mean(gu_ms) / 1e3 if gu_ms else None
    # the gate/up launches timed above, each with its own step's routing
    gu_b = statistics.mean(gateup_bytes(c["M"], u) for u in Us[:len(gu_ms)]) if gu_ms else gateup_bytes(c["M"], U)
    achieved = gu_b / gu_avg_s / 1e9 if gu_avg_s else None  # bytes per launch / mean launch time
    tr = traffic_entry("moe_gateup_kernel", U + c["n_shared"])
    out = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(t_max / args.steps * 1e3, 4),
        "us_per_step": round(t_max / args.steps * 1e6, 1),
        "tokens_per_s": round(all_tokens / t_max),
        "tokens_note": "tokens advanced per step: one per decoding sequence of the layer (64) plus "
                       "the accepted drafted tokens of the speculative window",
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "dtype_note": "bf16 weights and activations with fp32 accumulation; fp32 KDA state and arithmetic",
        "data": "synthetic (seeded; random-init weights of the layer's shapes)",
        "config": {
            "workload": "hybrid decode layer at batch 64 (hidden 7168; KDA 32 heads x 128, fp32 "
                        "state; 256 routed experts top-8 + 1 shared, intermediate 2048; L2 prefetch "
                        "on a side stream) + speculative window B=16, T=4 (verify, accept, replay)",
            "batch": c["M"], "spec_batch": c["spec_B"], "draft_len": c["spec_T"],
            "active_experts_mean": U, "active_experts_per_timed_step": Us,
            "routing_from": "a deterministic replay of the timed steps from their starting states "
                            f"(final states bit-identical to the timed run: {replay_bitwise})",
            "bytes_per_step": round(local_bytes / args.steps),
            "l2": "working set ~20 GB per step >> 129 MB L2 (inputs larger than L2; no flush)",
            "parallelism": f"replicas x{world} (no collective on the data path)",
            "launch": "eager launches on torch's current stream; prefetch on a second stream",
        },
        "breakdown_bytes_per_step": {**{k: v for k, v in per_step.items()},
                                     **{"spec_" + k: v for k, v in spec_bytes(
                                         c["spec_B"], c["spec_T"], wl.ids[0][2]).items()}},
        "clocks": {k: clocks[k] for k in ("sm_mhz", "sm_max_mhz", "reasons")},
        "clock_samples": clocks["samples"],
        "e2e": {"value": round(all_bytes / e2e_max / 1e9, 1), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "us_per_step": round(e2e_max / args.steps * 1e6, 1)},
        "gpu_launches": int(launches),
        "roofline": {
            "kernel": "moe_gateup_kernel (routed + shared expert gate/up weight streaming)",
            "bound": "hbm",
            "achieved": round(achieved, 1) if achieved else None,
            "peak": peak,
            "peak_kind": f"{peak_kind} (MEASURED_PEAKS hbm_gbs copy bandwidth)" if peak_kind == "measured" else peak_kind,
            "unit": "GB/s",
            "frac": round(achieved / peak, 3) if achieved else None,
            "traffic": tr["bytes_per_launch"] if tr else None,
            "algorithmic_bytes_per_launch": gu_b,
            "avg_launch_us": round(gu_avg_s * 1e6, 1) if gu_avg_s else None,
            "launches_timed": len(gu_ms),
        },
        "sweeps": sweeps,
    }
    if not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline()
    print(json.dumps(out))


# ----------------------------------------------------------------------------- ncu cases

def run_profile(kind, iters=3):
    """Small cases of the hot kernels for `ncu --set full` captures: a few GB on the
    device, inputs still larger than L2.  Prints one JSON line describing the case."""
    import torch
    from hybrid_linear_attention_gated_gb300 import build, hla, inputs
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    build.build()
    c = CFG
    g = inputs.generator(500, dev)
    info = dict(case=kind)
    if kind == "moe":
        # 48 experts, 32 tokens, top-8: the same kernel variants as the batch-64 workload
        # (16-token tile, cross-item load rings, no K split), 4.2 GB of weights
        E, M = 48, 32
        w = inputs.moe_weights(E, c["Hd"], c["I"], c["n_shared"], g, device=dev)
        x = inputs.activations(M, c["Hd"], g, dev)
        idx = torch.empty(M, c["k"], dtype=torch.int32, device=dev)
        wt = torch.empty(M, c["k"], device=dev)
        rb = hla.moe_route_topk_workspace_size(M, c["Hd"], E)
        rws = torch.empty(max(rb, 256), dtype=torch.uint8, device=dev)
        nb = hla.moe_expert_forward_workspace_size(M, c["Hd"], c["I"], E, c["k"], c["n_shared"])
        mws = torch.empty(nb, dtype=torch.uint8, device=dev)
        y = torch.empty(M, c["Hd"], dtype=torch.bfloat16, device=dev)
        hla.moe_route_topk(M, c["Hd"], E, c["k"], x, w["W_r"], idx, wt, None, rws, rb)
        U = int(torch.unique(idx).numel())
        for _ in range(iters):
            hla.moe_expert_forward(M, c["Hd"], c["I"], E, c["k"], c["n_shared"], x, idx, wt,
                                   w["W_gate"], w["W_up"], w["W_down"], w["Ws_gate"], w["Ws_up"],
                                   w["Ws_down"], None, y, mws, nb)
        info.update(E=E, M=M, active_experts=U, gateup_bytes=gateup_bytes(M, U),
                    variant=hla.hla_last_variant())
    elif kind == "kda":
        B, H, d = 64, c["H"], c["d"]
        S = torch.randn(B, H, d, d, device=dev).mul_(0.05)
        u = inputs.kda_inputs((B,), H, d, d, g, dev)
        o = torch.empty(B, H, d, device=dev)
        for _ in range(iters):
            hla.kda_decode_step(B, H, d, d, S, None, u["q"], u["k"], u["v"], u["alpha"], u["beta"], o)
        info.update(B=B, bytes=kda_bytes(B), variant=hla.hla_last_variant())
    elif kind == "spec":
        # speculative window at batch 64 (134 MB of committed state, > L2): verify, accept, replay
        B, T, H, d = 64, c["spec_T"], c["H"], c["d"]
        S = torch.randn(B, H, d, d, device=dev).mul_(0.05)
        w = inputs.kda_inputs((B, T), H, d, d, g, dev)
        dr, tg, a = inputs.accept_ids(B, T, g, dev)
        o = torch.empty(B, T, H, d, device=dev)
        acc = torch.zeros(B, dtype=torch.int32, device=dev)
        com = torch.zeros(B, dtype=torch.int32, device=dev)
        for _ in range(iters):
            hla.kda_spec_verify_replay(hla.HLA_SPEC_VERIFY, B, T, H, d, d, S, None, w["q"], w["k"],
                                       w["v"], w["alpha"], w["beta"], None, o)
            verify_variant = hla.hla_last_variant()
            hla.spec_accept_prefix(B, T, dr, tg, acc, com)
            hla.kda_spec_verify_replay(hla.HLA_SPEC_REPLAY, B, T, H, d, d, S, None, w["q"], w["k"],
                                       w["v"], w["alpha"], w["beta"], acc, None)
        info.update(B=B, T=T, accepted=a.tolist(), verify_bytes=spec_bytes(B, T, a.cpu().numpy())["verify"],
                    replay_bytes=spec_bytes(B, T, a.cpu().numpy())["replay"],
                    variant=[verify_variant, hla.hla_last_variant()])
    elif kind == "fused":
        # the fused speculative step at batch 64: the previous window's accepted prefix replayed and
        # committed, then this window verified, in one pass over the state (134 MB, > L2)
        B, T, H, d = 64, c["spec_T"], c["H"], c["d"]
        S = torch.randn(B, H, d, d, device=dev).mul_(0.05)
        prev = inputs.kda_inputs((B, T), H, d, d, g, dev)
        w = inputs.kda_inputs((B, T), H, d, d, g, dev)
        _, _, a = inputs.accept_ids(B, T, g, dev)
        acc = a.to(torch.int32)
        o = torch.empty(B, T, H, d, device=dev)
        for _ in range(iters):
            hla.kda_spec_replay_verify(B, T, T, H, d, d, S, None, prev["q"], prev["k"], prev["v"],
                                       prev["alpha"], prev["beta"], acc, w["q"], w["k"], w["v"],
                                       w["alpha"], w["beta"], o)
        an = a.cpu().numpy()
        tok = 3 * d * 2 + d * 4 + 4
        nbytes = (B * H * 4 * d * d + sum(H * (4 * d * d + int(x) * tok) for x in an if x > 0)
                  + B * H * T * (tok + 4 * d))
        info.update(B=B, T=T, accepted=an.tolist(), bytes=int(nbytes), variant=hla.hla_last_variant())
    elif kind == "extend":
        # four 512-token prefill chunks through kda_extend: each (sequence, head) is one serial
        # chain of 512 steps (8 MB of state; the kernel is bound by its step latency, not HBM)
        B, L, H, d = 4, 512, c["H"], c["d"]
        S = torch.randn(B, H, d, d, device=dev).mul_(0.05)
        cu = torch.arange(0, (B + 1) * L, L, dtype=torch.int32, device=dev)
        u = inputs.kda_inputs((B * L,), H, d, d, g, dev)
        o = torch.empty(B * L, H, d, device=dev)
        for _ in range(iters):
            hla.kda_extend(B, cu, H, d, d, S, None, u["q"], u["k"], u["v"], u["alpha"], u["beta"], o)
        info.update(B=B, tokens=B * L, variant=hla.hla_last_variant())
    elif kind in ("layer1", "layer8"):
        # the decode layer at batch 1 or 8 with the full-size weights: three warm-up calls, then
        # `iters` calls in the NVTX range "timed" (for an ncu launch list of the small-batch layer)
        M = 1 if kind == "layer1" else 8
        wl = Workload(dev, 0)
        x = inputs.activations(M, c["Hd"], g, dev)
        S = wl.S[:M].clone()
        y = torch.empty(M, c["Hd"], dtype=torch.bfloat16, device=dev)
        nb = hla.hla_decode_layer_workspace_size(wl.L, M)
        ws = torch.empty(nb, dtype=torch.uint8, device=dev)

        def layer_call(i):
            hla.hla_decode_layer(wl.L, M, x, S, None, y, ws, nb, prefetch_stream=wl.side)
        for i in range(3):
            layer_call(i)
        t = time_steps(torch, layer_call, iters, 1)
        info.update(M=M, calls=iters, us_per_call_eager=round(t / iters * 1e6, 1),
                    variant=hla.hla_last_variant())
    elif kind in ("dense", "dense16"):
        # the input projection at batch 64 (tensor-core path) or 16 (streaming path)
        M, H, d = (64 if kind == "dense" else 16), c["H"], c["d"]
        W = inputs.weight((4 * H * d + H, c["Hd"]), g, dev)
        x = inputs.activations(M, c["Hd"], g, dev)
        outs = [torch.empty(M, H, d, dtype=torch.bfloat16, device=dev) for _ in range(3)]
        al, be = torch.empty(M, H, d, device=dev), torch.empty(M, H, device=dev)
        nb = hla.kda_qkvg_proj_workspace_size(M, c["Hd"], H, d, d, 0)
        ws = torch.empty(nb, dtype=torch.uint8, device=dev)
        for _ in range(iters):
            hla.kda_qkvg_proj(M, c["Hd"], H, d, d, x, W, *outs, al, be, 0, ws, nb)
        info.update(M=M, weight_bytes=W.numel() * 2, variant=hla.hla_last_variant())
    torch.cuda.synchronize()
    print(json.dumps(info))


# ----------------------------------------------------------------------------- prefetch A/B

def run_prefetch_ab(reps=4):
    """Layer time at batch 1 / 8 / 64 for every side-stream prefetch mask (interleaved
    repetitions, CUDA graph of 8 calls each), with clocks; one JSON line."""
    import torch
    from hybrid_linear_attention_gated_gb300 import build, hla, inputs
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    build.build()
    wl = Workload(dev, 0, prefetch=True)
    c = CFG
    masks = ["none", "0", "1", "2", "3", "7"]
    sampler = ClockSampler(0)
    sampler.start()
    table = {}
    for M in (1, 8, 64):
        g = inputs.generator(9000 + M, dev)
        xs = [inputs.activations(M, c["Hd"], g, dev) for _ in range(ROTATE)]
        S = wl.S[:M].clone()
        y = torch.empty(M, c["Hd"], dtype=torch.bfloat16, device=dev)
        nb = hla.hla_decode_layer_workspace_size(wl.L, M)
        ws = torch.empty(nb, dtype=torch.uint8, device=dev)
        res = {m: [] for m in masks}
        for _ in range(reps):
            for m in masks:
                os.environ.pop("HLA_PREFETCH_MASK", None)
                if m != "none":
                    os.environ["HLA_PREFETCH_MASK"] = m
                pf = 0 if m == "none" else wl.side

                def fn(i, pf=pf):
                    hla.hla_decode_layer(wl.L, M, xs[i % ROTATE], S, None, y, ws, nb, prefetch_stream=pf)
                res[m].append(graph_time(torch, fn, 8) * 1e6)
        os.environ.pop("HLA_PREFETCH_MASK", None)
        table[M] = {m: round(statistics.median(v), 1) for m, v in res.items()}
    clocks = sampler.stop()
    print(json.dumps({"prefetch_ab_us_per_layer": table, "clocks": clocks,
                      "masks": "none = no prefetch stream; 1 = W_o+W_r during KDA; 2 = shared gate/up "
                               "during dispatch; 4 = shared down"}))


# ----------------------------------------------------------------------------- layer A/B

def run_layer_ab(spec, reps=5, batches=(1, 2, 8, 32, 64)):
    """Layer time (CUDA graph of 8 calls, with the prefetch stream) at several batch sizes for
    each value of one tuning switch, e.g. ``HLA_PDL=0,1`` (``-`` = the switch unset); repetitions
    are interleaved so that the values see the same clocks.  One JSON line with the medians and
    the clocks."""
    import torch
    from hybrid_linear_attention_gated_gb300 import build, hla, inputs
    var, vals = spec.split("=")
    vals = vals.split(",")
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    build.build()
    wl = Workload(dev, 0, prefetch=True)
    c = CFG
    sampler = ClockSampler(0)
    sampler.start()
    table = {}
    for M in batches:
        g = inputs.generator(9000 + M, dev)
        xs = [inputs.activations(M, c["Hd"], g, dev) for _ in range(ROTATE)]
        S = wl.S[:M].clone() if M <= c["M"] else None
        if S is None:
            continue
        y = torch.empty(M, c["Hd"], dtype=torch.bfloat16, device=dev)

        def set_switch(v):
            if v == "-":
                os.environ.pop(var, None)
            else:
                os.environ[var] = v
        nbs = {}
        for v in vals:  # a switch may change the workspace size (e.g. a forced split)
            set_switch(v)
            nbs[v] = hla.hla_decode_layer_workspace_size(wl.L, M)
        ws = torch.empty(max(nbs.values()), dtype=torch.uint8, device=dev)
        res = {v: [] for v in vals}
        for _ in range(reps):
            for v in vals:
                set_switch(v)
                nb = nbs[v]

                def fn(i, nb=nb):
                    hla.hla_decode_layer(wl.L, M, xs[i % ROTATE], S, None, y, ws, nb, prefetch_stream=wl.side)
                res[v].append(graph_time(torch, fn, 8) * 1e6)
        os.environ.pop(var, None)
        table[M] = {v: round(statistics.median(t), 2) for v, t in res.items()}
    clocks = sampler.stop()
    print(json.dumps({"layer_ab_us_per_call": table, "switch": var, "reps": reps, "clocks": clocks}))


def run_spec_ab(spec, reps=3):
    """The speculative-window sweep (B = 16 and 64, separate and fused forms, states rotated past
    L2) for each value of one tuning switch, e.g. ``HLA_KDA_CW=0,32`` (0: the default width);
    repetitions interleaved.
    One JSON line with the median microseconds and fractions of the peak."""
    import torch
    from hybrid_linear_attention_gated_gb300 import build, hla, inputs
    var, vals = spec.split("=")
    vals = vals.split(",")
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    build.build()
    peak, _ = peaks()

    class _Wl:  # the spec sweep needs only the B=16 windows
        pass
    wl = _Wl()
    g = inputs.generator(5, dev)
    wl.win, wl.ids = [], []
    for _ in range(ROTATE):
        wl.win.append(inputs.kda_inputs((CFG["spec_B"], CFG["spec_T"]), CFG["H"], CFG["d"], CFG["d"], g, dev))
        dr, tg, a = inputs.accept_ids(CFG["spec_B"], CFG["spec_T"], g, dev)
        wl.ids.append((dr, tg, a.cpu().numpy()))
    sampler = ClockSampler(0)
    sampler.start()
    res = {v: [] for v in vals}
    for _ in range(reps):
        for v in vals:
            os.environ[var] = v
            res[v].append(spec_sweep(torch, hla, inputs, wl, dev, peak))
    os.environ.pop(var, None)
    clocks = sampler.stop()
    table = {}
    for v, runs in res.items():
        for i, row in enumerate(runs[0]):
            us = statistics.median(r[i]["us"] for r in runs)
            key = f"B{row['batch']}_{row['form']}"
            table.setdefault(key, {})[v] = dict(us=round(us, 2), frac=round(row["bytes"] / us / 1e3 / peak, 3))
    print(json.dumps({"spec_ab": table, "switch": var, "reps": reps, "clocks": clocks}))


# ----------------------------------------------------------------------------- reference arm

def run_reference(args):
    """The fp64 oracle on the host cores, each step a bounded sample of the workload:
    the decode layer for one of the 64 sequences and the speculative window for one of
    the 16 sequences."""
    world, rank, _ = dist_setup()
    if rank != 0:
        return
    import numpy as np
    import torch
    import oracle
    if args.threads > 0:
        torch.set_num_threads(args.threads)
    from hybrid_linear_attention_gated_gb300 import inputs
    c = CFG
    f = lambda t: t.float().numpy()  # noqa: E731  (exact for bf16; the oracle upcasts)
    g = inputs.generator(11)
    lw = inputs.layer_weights(c["Hd"], c["H"], c["d"], c["d"], g)
    W_r = inputs.weight((c["E"], c["Hd"]), g)
    p = dict(H=c["H"], dk=c["d"], dv=c["d"], top_k=c["k"], eps=c["eps"],
             gamma_attn=f(lw["gamma_attn"]), gamma_moe=f(lw["gamma_moe"]),
             W_qkvgb=f(lw["W_qkvgb"]), W_o=f(lw["W_o"]), W_r=f(W_r))
    cache = {}

    def experts(e):  # each expert's weights drawn on first use from its own seed
        if e not in cache:
            ge = inputs.generator(3_000_000 + int(e))
            cache[e] = tuple(f(inputs.weight(s, ge)) for s in
                             ((c["I"], c["Hd"]), (c["I"], c["Hd"]), (c["Hd"], c["I"])))
        return cache[e]
    gs = inputs.generator(12)
    shared = [tuple(f(inputs.weight(s, gs)) for s in
                    ((c["I"], c["Hd"]), (c["I"], c["Hd"]), (c["Hd"], c["I"])))]
    H, d, T = c["H"], c["d"], c["spec_T"]
    u = inputs.warm_update_inputs(256, 2 * H, d, d, inputs.generator(13))
    pool = oracle.kda.warm_state((2 * H, d, d), *(f(u[k]) for k in ("q", "k", "v", "alpha", "beta")))
    S = pool[:H][None]
    S_spec = pool[H:][None]
    xs = [inputs.activations(1, c["Hd"], inputs.generator(20 + i)) for i in range(ROTATE)]
    wins = [{k: f(v) for k, v in inputs.kda_inputs((1, T), H, d, d, inputs.generator(30 + i)).items()}
            for i in range(ROTATE)]
    accs = [inputs.accept_ids(1, T, inputs.generator(40 + i))[2].numpy() for i in range(ROTATE)]
    for r in range(ROTATE):  # convert every expert the sample will touch before timing
        oracle.layer.decode_layer(f(xs[r]), S, p, experts, shared)

    def one(i):
        r = i % ROTATE
        _, _, aux = oracle.layer.decode_layer(f(xs[r]), S, p, experts, shared)
        w = wins[r]
        oracle.kda.spec_verify(S_spec, w["q"], w["k"], w["v"], w["alpha"], w["beta"])
        oracle.kda.spec_replay(S_spec, w["q"], w["k"], w["v"], w["alpha"], w["beta"], accs[r])
        U = len(set(int(e) for e in aux["topk_idx"][0]))
        return sum(layer_bytes(1, U).values()) + sum(spec_bytes(1, T, accs[r]).values())
    for i in range(args.warmup):
        one(i)
    t0 = time.perf_counter()
    nbytes = sum(one(i) for i in range(args.steps))
    dt = time.perf_counter() - t0
    value = nbytes / dt / 1e9
    cores = args.threads if args.threads > 0 else len(os.sched_getaffinity(0))
    sample = ("per step: the decode layer for 1 of the 64 sequences and the speculative window "
              "for 1 of the 16 sequences, fp64 numpy oracle; bytes credited as for that sample")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 2), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": {"workload": "bounded sample of: hybrid decode layer batch 64 + speculative "
                               "window B=16, T=4", "sample": sample},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }))
    del np, torch


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-prefetch", action="store_true")
    ap.add_argument("--threads", type=int, default=0,
                    help="reference arm: host threads the oracle may use (0 = every core); the "
                         "BLAS thread count is fixed by its environment variables at start-up")
    ap.add_argument("--profile", choices=["moe", "kda", "spec", "fused", "extend", "dense", "dense16", "layer1",
                                          "layer8"],
                    help="run one small case of a hot kernel (for ncu captures) and exit")
    ap.add_argument("--prefetch-ab", action="store_true",
                    help="time the layer under every side-stream prefetch mask and exit")
    ap.add_argument("--layer-ab", metavar="VAR=v1,v2",
                    help="time the layer at batch 1-64 for each value of one tuning switch and exit")
    ap.add_argument("--ab-batches", default="1,2,8,32,64", help="batch sizes of --layer-ab")
    ap.add_argument("--spec-ab", metavar="VAR=v1,v2",
                    help="time the speculative window for each value of one tuning switch and exit")
    args = ap.parse_args()
    if args.profile:
        return run_profile(args.profile)
    if args.prefetch_ab:
        return run_prefetch_ab()
    if args.layer_ab:
        return run_layer_ab(args.layer_ab, batches=tuple(int(b) for b in args.ab_batches.split(",")))
    if args.spec_ab:
        return run_spec_ab(args.spec_ab)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()

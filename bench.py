"""Benchmark: MoE-layer decode throughput on GB300.

Workload (one step): one token through 48 stacked routed-expert layers with a
residual stream, H=2048, 512 experts per layer, expert width I=768, top-10,
2-bit block-quantised experts (36.2 GB resident), a bf16 shared expert
(I=768) and an fp32 router biased for Zipf(1.1) expert popularity; seeded
synthetic data.  Each step is one launch of moe_decode_forward (all 48
layers in one persistent kernel); ``--path modular`` times instead a CUDA
graph of the per-layer calls router_topk -> permute -> shared_expert ->
expert_forward.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line.  Besides the headline (one-token decode) it carries
``verify_4tok`` (4-token verify windows through the same 48-layer stack) and
``prefill_32k`` (one layer over a 32,768-token prompt: router, permutation,
shared expert and the grouped expert GEMMs, with the tensor roofline of the
expert call), ``prefill_32k_fp8`` (the same on e4m3 operands, an opt-in
approximation) and ``prefill_3bit_4k`` (4,096 tokens through a 48-layer stack
of 3-bit experts, uniform and Zipf(1.4) routing reported separately, with
both the tensor and the HBM fraction) and ``tiny_layer`` (the tiny
configuration's time per layer call on each path); ``--no-extra`` skips
those four.  ``--impl reference`` times the
oracle (plain scalar CPU code) on a bounded sample of the same workload
instead.  Under torchrun
every rank runs an independent replica (the layer does not shard across GPUs
here); rank 0 prints the whole-job throughput.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

LAYERS, H, E, I, K_TOP, IS = 48, 2048, 512, 768, 10, 768
# DRAM bytes (read + write) of one 48-layer fused decode launch, median of the
# 18 plain launches after the first in an ncu capture of `bench.py --only-hot`
# (dram__bytes_read.sum + dram__bytes_write.sum),
# valid for the decode source whose code (comments and whitespace removed) has
# this SHA-256 prefix; reported as null once that code changes, until it is
# captured again.
DECODE_TRAFFIC = (1_363_879_552, "f50f7317dca4e112")
EXPERT_BYTES = 1_474_560
ROUTER_BYTES = E * H * 4
SHARED_BYTES = 3 * H * IS * 2
BYTES_PER_TOKEN = LAYERS * (K_TOP * EXPERT_BYTES + ROUTER_BYTES + SHARED_BYTES)  # 1,362,100,224
KERNELS_PER_LAYER = 10  # rms_norm_bf16, router gemv, topk, permute, shared (2 gemv + add), experts (2 gemv + combine)
WORKLOAD = ("decode: 1 token x 48 layers, H=2048, E=512, I=768, top-10, 2-bit experts (32-weight blocks, fp16 "
            "scales) + bf16 shared expert I=768, fp32 router with Zipf(1.1) bias, fp32 residual stream "
            "normalised (RMS) in front of each layer")


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def peaks_bf16():
    """Dense bf16 tensor peak (TFLOP/s), burst: the prefill GEMMs are timed alone."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["bf16_tflops"]), "measured"
    return 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([c.strip() for c in line.split(",")])

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=2)
        sm = []
        smax = 0.0
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in self.rows:
            try:
                sm.append(float(r[0]))
                smax = max(smax, float(r[1]))
                for n, v in zip(names, r[4:8]):
                    if v.lower() == "active":
                        reasons.add(n)
            except (ValueError, IndexError):
                continue
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": smax or None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl" if os.environ.get("BENCH_GLOO") is None else "gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(world, v: float) -> float:
    if world == 1:
        return v
    import torch
    import torch.distributed as dist

    dev = "cpu" if dist.get_backend() == "gloo" else "cuda"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------- oracle leg

def oracle_decode_sample(n_layers: int, seed: int = 0, step: int = 0):
    """Time the oracle on one token through `n_layers` layers of the workload.

    Returns (seconds of oracle compute, layers).  Weights of the experts the
    token picks are regenerated on the host from the seeded generator; that
    generation is not timed.
    """
    import oracle
    from bit_expert_ffn_gb300 import synth

    x = synth.activations(seed, 1, H, step=step)
    xres = synth.bf16_bits_to_f32(x).astype(np.float64)
    t_oracle = 0.0
    for layer in range(n_layers):
        t0 = time.perf_counter()
        xn = oracle.rms_norm(xres.astype(np.float32), 1e-6)
        t_oracle += time.perf_counter() - t0
        xb = synth.f32_to_bf16_bits(xn.astype(np.float32))
        wr = synth.router_weights(seed, layer, E, H)
        b = synth.zipf_bias(seed, layer, E, 1.1)
        shared = synth.shared_weights(seed, layer, H, IS)
        t0 = time.perf_counter()
        logits = oracle.router_logits(xb, wr, b).astype(np.float32)
        ids, w = oracle.topk(logits, K_TOP)
        t_oracle += time.perf_counter() - t0
        parts = [[], [], [], [], [], []]
        for e in ids[0]:
            g, u, d = synth.expert_codes(seed, layer, int(e), 2, H, I)
            gus, ds = synth.expert_scales(seed, layer, int(e), H, I)
            for lst, a in zip(parts, (g, gus[0], u, gus[1], d, ds)):
                lst.append(a)
        arena = [np.stack(p) for p in parts]
        t0 = time.perf_counter()
        y = oracle.moe_layer(2, xb, np.arange(K_TOP, dtype=np.int32)[None, :], w, *arena, shared=shared)
        t_oracle += time.perf_counter() - t0
        xres = xres + y
    return t_oracle, n_layers


def activation_rows(seed, tokens, step=0):
    """Rows `tokens` of synth.activations(seed, T, H, step) (bf16 bits), drawn alone."""
    from bit_expert_ffn_gb300 import synth

    key = synth.stream_key(seed, synth.TAG_X, step)
    return np.stack([synth.f32_to_bf16_bits(synth.normal(key, H, start=int(t) * H)) for t in tokens])


def oracle_prefill_sample(seed, layer, bits, x_bf16, zipf_s, threads):
    """Seconds the oracle takes for the tokens x_bf16 [n][H] through one prefill layer, spread over
    `threads` host threads (the oracle is C code called through ctypes, which releases the GIL): router
    logits and top-10 of every token first, then the layer (shared expert and routed experts) on the
    oracle's own routing.  The weights of the experts those tokens pick are drawn by the device generator
    in between, untimed."""
    from concurrent.futures import ThreadPoolExecutor

    import oracle
    from bit_expert_ffn_gb300 import synth
    from bit_expert_ffn_gb300.model import draw_expert_parts

    wr = synth.router_weights(seed, layer, E, H)
    b = synth.zipf_bias(seed, layer, E, zipf_s)
    shared = synth.shared_weights(seed, layer, H, IS)
    n = x_bf16.shape[0]
    with ThreadPoolExecutor(max_workers=threads) as pool:
        t0 = time.perf_counter()
        routed = list(pool.map(lambda t: oracle.topk(oracle.router_logits(x_bf16[t:t + 1], wr, b).astype(np.float32),
                                                     K_TOP), range(n)))
        t_route = time.perf_counter() - t0
        ids = np.concatenate([r[0] for r in routed])
        w = np.concatenate([r[1] for r in routed])
        used = sorted(set(ids.ravel().tolist()))
        remap = {e: i for i, e in enumerate(used)}
        arena = draw_expert_parts(seed, layer, used, bits, H, I)
        cids = np.vectorize(remap.get)(ids).astype(np.int32)
        t0 = time.perf_counter()
        list(pool.map(lambda t: oracle.moe_layer(bits, x_bf16[t:t + 1], cids[t:t + 1], w[t:t + 1], *arena,
                                                 shared=shared), range(n)))
        t_layer = time.perf_counter() - t0
    return t_route + t_layer


def prefill_cpu_baselines(n_tokens: int = 48):
    """The oracle timed on token samples of the two prefill workloads, on every host core."""
    import oracle
    from bit_expert_ffn_gb300 import synth

    threads = os.cpu_count() or 1
    toks = sorted(np.random.default_rng(11).choice(32768, n_tokens, replace=False))
    t = oracle_prefill_sample(1, 0, 2, activation_rows(1, toks), 1.1, threads)
    c3 = {"value": n_tokens / t, "unit": "tokens/s", "cores": threads, "kind": "oracle",
          "sample": f"{n_tokens} of the 32,768 prompt tokens through the layer (router, top-10, shared and routed "
                    f"experts), fp64 scalar C, {threads} host threads over the tokens"}
    toks = sorted(np.random.default_rng(12).choice(4096, n_tokens, replace=False))
    xin = activation_rows(4, toks)
    xn = synth.f32_to_bf16_bits(oracle.rms_norm(synth.bf16_bits_to_f32(xin), 1e-6).astype(np.float32))
    t = oracle_prefill_sample(4, 0, 3, xn, 0.0, threads)
    c4 = {"value": n_tokens / (t * LAYERS), "unit": "tokens/s", "cores": threads, "kind": "oracle",
          "sample": f"{n_tokens} of the 4,096 tokens through layer 0 of the 3-bit stack (uniform routing), "
                    f"extrapolated to the 48 layers (x48), fp64 scalar C, {threads} host threads over the tokens"}
    return c3, c4


def run_reference(args, world, rank):
    if rank != 0:
        return
    t_total = 0.0
    layers_total = 0
    for s in range(args.warmup):
        oracle_decode_sample(1, step=s)
    for s in range(args.steps):
        t, n = oracle_decode_sample(1, step=1000 + s)
        t_total += t
        layers_total += n
    tok_s = layers_total / LAYERS / t_total
    sample = f"{args.steps} steps, each one token through 1 of the 48 layers (oracle compute only), scaled by 1/48"
    line = {"impl": "reference", "metric": "decode tokens/s (48-layer MoE stack, 1 token per step)", "value": tok_s,
            "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 * t_total / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded generator)",
            "config": {"workload": WORKLOAD, "tokens_per_step": 1, "layers": LAYERS},
            "cpu_baseline": {"value": tok_s, "unit": "tokens/s", "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": tok_s, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- our leg

READOUT_VOCAB = 8192


def readout_head(H_: int):
    """A seeded random readout W [V][H] ~ N(0, 2/sqrt(H)) (fp32, host): with trained weights absent it stands in
    for the model's output head when the route-tail skip's effect on next-token distributions is measured
    (logits of standard deviation about 2 for a unit-RMS hidden state)."""
    from bit_expert_ffn_gb300 import synth

    return synth.normal_sigma(synth.stream_key(77, 12), READOUT_VOCAB * H_, 2.0 / np.sqrt(H_)).reshape(READOUT_VOCAB, H_)


def readout_compare(head, xe: np.ndarray, xs: np.ndarray):
    """KL(p_exact || p_skip) per token and top-1 agreement of the readout distributions of two hidden states."""
    def logp(x):
        x = x.astype(np.float64)
        z = (x / np.sqrt(np.mean(x * x, axis=1, keepdims=True) + 1e-6)) @ head.T.astype(np.float64)
        z -= z.max(axis=1, keepdims=True)
        return z - np.log(np.exp(z).sum(axis=1, keepdims=True))
    le, ls = logp(xe), logp(xs)
    kl = np.sum(np.exp(le) * (le - ls), axis=1)
    return kl, np.argmax(le, axis=1) == np.argmax(ls, axis=1)


def bench_verify(m, lib, layers, descs, dev, stream, steps: int, warmup: int, tail_skip: int = 0):
    """4-token verify windows through the same stack (moe_decode_forward, T=4).

    Bytes per step are counted from the routing the kernel reports for the
    timed windows themselves (each timed call writes its ids into its own
    slice of a device buffer, 1,920 ints per window): the union of the 4
    tokens' experts in every layer (with tail_skip, the experts the skip
    keeps), plus every layer's router and shared expert.  With tail_skip the
    calls go through moe_decode_forward_ex and the line also reports the
    skip's effect on the output against the exact path: relative L2 of the
    48-layer output and, through a seeded readout head, the KL divergence and
    top-1 agreement of next-token distributions (on 16 of the windows).
    """
    import ctypes

    import torch

    from bit_expert_ffn_gb300 import synth

    T, NL = 4, len(layers)
    nb = m.moe_decode_workspace_size(T, H, I, E, K_TOP, IS)
    ws = torch.empty(nb, dtype=torch.uint8, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    n_steps = warmup + steps
    ids = torch.empty(n_steps, NL, T, K_TOP, dtype=torch.int32, device=dev)
    wts = torch.empty(n_steps, NL, T, K_TOP, dtype=torch.float32, device=dev)
    X = torch.stack([torch.from_numpy(synth.bf16_bits_to_f32(synth.verify_window(100 + i, T, H))) for i in range(n_steps)]).to(dev)
    x = torch.zeros(T, H, dtype=torch.float32, device=dev)
    sptr = ctypes.c_void_p(stream.cuda_stream)

    opts = m.moe_decode_options(tail_skip, None)

    def call(i, skip=True):
        if tail_skip and skip:
            r = lib.moe_decode_forward_ex(descs, NL, x.data_ptr(), T, K_TOP, m.RMS_EPS, ctypes.byref(opts),
                                          ids[i].data_ptr(), wts[i].data_ptr(), ws.data_ptr(), nb, st.data_ptr(), sptr)
        else:
            r = lib.moe_decode_forward(descs, NL, x.data_ptr(), T, K_TOP, m.RMS_EPS, ids[i].data_ptr(),
                                       wts[i].data_ptr(), ws.data_ptr(), nb, st.data_ptr(), sptr)
        if r:
            raise m.MoeError(r, m.moe_last_error())

    with torch.cuda.stream(stream):
        for i in range(warmup):
            x.copy_(X[i])
            call(i)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(warmup, n_steps):
            x.copy_(X[i])
            call(i)
        e1.record(stream)
    torch.cuda.synchronize()
    assert m.moe_check_status(st) == 0, m.moe_last_error()
    ms = e0.elapsed_time(e1) / steps
    timed = ids[warmup:].cpu().numpy()

    def kept(i, l):
        sel = timed[i, l]
        if not tail_skip:
            return set(sel.ravel().tolist())
        early = set(sel[:, :tail_skip].ravel().tolist())
        return early | {int(e) for e in sel[:, tail_skip:].ravel() if int(e) in early}

    u = float(np.mean([sum(len(kept(i, l)) for l in range(NL)) for i in range(steps)]))
    bytes_step = u * EXPERT_BYTES + NL * (ROUTER_BYTES + SHARED_BYTES)
    res = {"workload": f"verify window: 4 tokens x {NL} layers, same stack (c + N(0, 0.3^2) per token)"
                       + (f", route-tail skip from rank {tail_skip} (an approximation)" if tail_skip else ""),
           "value": T / (ms / 1000.0), "unit": "tokens/s", "ms_per_step": ms,
           "mean_experts_per_step": u, "bytes_per_step": bytes_step,
           "achieved_gbs": bytes_step / (ms / 1000.0) / 1e9}
    if tail_skip:
        head = readout_head(H)
        kls, agree, rels = [], [], []
        with torch.cuda.stream(stream):
            for i in range(warmup, min(n_steps, warmup + 16)):
                x.copy_(X[i])
                call(i, skip=False)
                xe = x.cpu().numpy()
                x.copy_(X[i])
                call(i, skip=True)
                xs = x.cpu().numpy()
                kl, ag = readout_compare(head, xe, xs)
                kls.extend(kl.tolist())
                agree.extend(ag.tolist())
                rels.append(float(np.linalg.norm(xs - xe) / np.linalg.norm(xe - X[i].cpu().numpy())))
        assert m.moe_check_status(st) == 0, m.moe_last_error()
        res["quality_vs_exact"] = {"kl_mean": float(np.mean(kls)), "kl_max": float(np.max(kls)),
                                   "top1_agreement": float(np.mean(agree)),
                                   "rel_l2_of_stack_update": float(np.mean(rels)), "tokens": len(kls),
                                   "readout": f"seeded N(0, 2/sqrt(H)) head over {READOUT_VOCAB} outputs on the "
                                              "RMS-normalised 48-layer output (stands in for the model's head)"}
    return res


HOT_BUDGET = 96 * 1024 * 1024  # bytes of expert weights kept in L2 (of its 129 MB) by the hot-expert hints


def bench_decode_hot(m, lib, descs, dev, stream, X, steps: int, warmup: int, profile_steps: int = 16):
    """The decode step (one token, 48 layers) with hot-expert L2 hints (moe_decode_forward_ex).

    The hot set is learned as the pages' adaptive cache learns it: from the
    routing that `profile_steps` earlier decode steps reported (ids_out), the
    most often picked experts over all layers are marked until their weights
    fill HOT_BUDGET.  The results are bit-identical to the plain decode; the
    line reports the time per step and the share of routed expert reads that
    fall on hot experts (those bytes come from L2 instead of HBM once warm).
    """
    import ctypes

    import torch

    NL = len(descs)
    nb = m.moe_decode_workspace_size(1, H, I, E, K_TOP, IS)
    ws = torch.empty(nb, dtype=torch.uint8, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    x = torch.zeros(1, H, dtype=torch.float32, device=dev)
    ids = torch.empty(profile_steps + steps, NL, 1, K_TOP, dtype=torch.int32, device=dev)
    wts = torch.empty(profile_steps + steps, NL, 1, K_TOP, dtype=torch.float32, device=dev)
    sptr = ctypes.c_void_p(stream.cuda_stream)
    n_in = X.shape[0]

    def run(i, opts, out_i=None):
        r = lib.moe_decode_forward_ex(descs, NL, x.data_ptr(), 1, K_TOP, m.RMS_EPS, ctypes.byref(opts) if opts else None,
                                      ids[out_i].data_ptr() if out_i is not None else None,
                                      wts[out_i].data_ptr() if out_i is not None else None,
                                      ws.data_ptr(), nb, st.data_ptr(), sptr)
        if r:
            raise m.MoeError(r, m.moe_last_error())

    with torch.cuda.stream(stream):
        for i in range(profile_steps):  # the routing profile
            x.copy_(X[i % n_in:i % n_in + 1])
            run(i, None, i)
    torch.cuda.synchronize()
    prof = ids[:profile_steps].cpu().numpy().reshape(profile_steps, NL, K_TOP)
    counts = np.zeros((NL, E), np.int64)
    for l in range(NL):
        np.add.at(counts[l], prof[:, l].ravel(), 1)
    order = np.argsort(-counts, axis=None, kind="stable")
    n_hot = int(HOT_BUDGET // EXPERT_BYTES)
    mask = np.zeros((NL, (E + 31) // 32), np.uint32)
    hot = np.zeros((NL, E), bool)
    for f in order[:n_hot]:
        l, e = divmod(int(f), E)
        hot[l, e] = True
        mask[l, e // 32] |= np.uint32(1 << (e % 32))
    hot_dev = torch.from_numpy(mask.view(np.int32)).to(dev)
    opts = m.moe_decode_options(0, hot_dev.data_ptr())
    with torch.cuda.stream(stream):
        for i in range(warmup):
            x.copy_(X[i % n_in:i % n_in + 1])
            run(i, opts)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(steps):
            x.copy_(X[(warmup + i) % n_in:(warmup + i) % n_in + 1])
            run(i, opts, profile_steps + i)
        e1.record(stream)
    torch.cuda.synchronize()
    assert m.moe_check_status(st) == 0, m.moe_last_error()
    ms = e0.elapsed_time(e1) / steps
    timed = ids[profile_steps:].cpu().numpy().reshape(steps, NL, K_TOP)
    share = float(np.mean([hot[l, timed[i, l]].mean() for i in range(steps) for l in range(NL)]))
    return {"workload": "decode: 1 token x 48 layers (the headline workload), hot-expert L2 hints",
            "value": 1000.0 / ms, "unit": "tokens/s", "ms_per_step": ms,
            "hot_experts": n_hot, "hot_bytes": n_hot * EXPERT_BYTES,
            "profile": f"picks of {profile_steps} earlier decode steps, most picked experts over all layers",
            "hot_share_of_routed_reads": share,
            "routed_bytes_from_l2_per_token_est": share * NL * K_TOP * EXPERT_BYTES,
            "note": "bit-identical to the plain decode; bytes from L2 assume the hot lines stay resident"}


def bench_prefill(m, dev, reps: int = 3, T: int = 32768, fp8: bool = False):
    """One routed-expert layer over a 32,768-token prompt: router_topk ->
    permute -> shared_expert -> expert_forward (prefill path, or its FP8
    variant), CUDA events around each call."""
    import torch

    from bit_expert_ffn_gb300 import synth
    from bit_expert_ffn_gb300.model import LayerShape, MoeLayer, StepBuffers, Workspace

    s = LayerShape(bits=2)
    L = MoeLayer(s, dev)
    L.fill_device(seed=1, layer=0, zipf_s=1.1)
    x = torch.from_numpy(synth.activations(1, T, s.H).view(np.int16)).to(dev)
    bufs = StepBuffers(T, s.E, s.k, dev)
    wsp = Workspace(dev)
    out = torch.zeros(T, s.H, dtype=torch.float32, device=dev)
    pws = m.moe_permute_workspace_size(T, s.k, s.E)
    path = m.MOE_PATH_PREFILL_FP8 if fp8 else m.MOE_PATH_PREFILL
    ews = m.moe_expert_forward_workspace_size(L.arena, T, s.k, path)
    sws = m.moe_shared_expert_workspace_size(s.H, s.Is, T)
    rws = m.moe_router_workspace_size(T, s.H, s.E, True)
    buf = wsp.get(max(pws, ews, sws, rws))
    res = {}
    for r in range(reps + 2):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
        ev[0].record()
        m.moe_router_topk(x, T, s.H, L.router_w, L.router_b, s.E, s.k, bufs.logits, bufs.ids, bufs.w, buf, rws,
                          dev_status=L.status)
        ev[1].record()
        m.moe_permute(bufs.ids, T, s.k, s.E, bufs.offsets, bufs.perm, bufs.inv, buf, pws, dev_status=L.status)
        ev[2].record()
        m.moe_shared_expert(*L.shared, s.H, s.Is, x, T, out, m.MOE_F32, False, buf, sws, L.status)
        ev[3].record()
        m.moe_expert_forward(L.arena, x, T, bufs.ids, bufs.w, s.k, bufs.offsets, bufs.perm, bufs.inv, out, m.MOE_F32,
                             True, path, buf, ews, dev_status=L.status)
        ev[4].record()
        torch.cuda.synchronize()
        if r >= 2:
            for name, i0, i1 in (("router", 0, 1), ("permute", 1, 2), ("shared", 2, 3), ("experts", 3, 4),
                                 ("total", 0, 4)):
                res.setdefault(name, []).append(ev[i0].elapsed_time(ev[i1]))
    assert m.moe_check_status(L.status) == 0, m.moe_last_error()
    assert bool(torch.isfinite(out).all()), "prefill output is not finite"
    ms = {k: float(np.median(v)) for k, v in res.items()}
    flop = 2.0 * T * s.k * 3 * s.H * s.I  # routed experts: gate, up, down
    tflops = flop / (ms["experts"] / 1000.0) / 1e12
    peak = peaks_bf16()
    if fp8:
        # e4m3 runs at twice the bf16 rate (nominal 4.5 vs 2.25 PFLOP/s dense): the measured bf16 peak x 2
        return {"workload": f"FP8 prefill (an approximation): {T} tokens x 1 layer, H=2048, E=512, I=768, top-10, "
                            "2-bit, Zipf(1.1), routed experts on e4m3 operands",
                "value": T / (ms["total"] / 1000.0), "unit": "tokens/s", "ms": ms,
                "experts_tflops": tflops, "experts_flop": flop,
                "rel_l2_vs_exact_layer": "about 3e-2 (tests/test_gpu_prefill_fp8.py; the 2e-2 target is not met)",
                "tensor_roofline": {"kernel": "moe_expert_forward FP8 prefill (row exponents, e4m3 gather, gate/up "
                                              "GEMM, h to e4m3, down GEMM, combine)",
                                    "bound": "tensor", "achieved": tflops, "peak": 2 * peak[0], "unit": "TFLOP/s",
                                    "frac": tflops / (2 * peak[0]), "peak_kind": peak[1] + " bf16 x 2",
                                    "note": "e4m3 operands (kind::f8f6f4)"}}
    return {"workload": f"prefill: {T} tokens x 1 layer, H=2048, E=512, I=768, top-10, 2-bit, Zipf(1.1)",
            "value": T / (ms["total"] / 1000.0), "unit": "tokens/s", "ms": ms,
            "experts_tflops": tflops, "experts_flop": flop,
            "tensor_roofline": {"kernel": "moe_expert_forward prefill (gather, gate/up GEMM, down GEMM, combine)",
                                "bound": "tensor", "achieved": tflops, "peak": peak[0], "unit": "TFLOP/s",
                                "frac": tflops / peak[0], "peak_kind": peak[1],
                                "note": "fp16 operands (kind::f16, the bf16 rate)"}}


def bench_tiny(m, dev, reps: int = 200):
    """The tiny configuration (8 tokens, H=256, E=16, I=128, top-2, bf16 shared expert I=128): one layer
    call (router, permutation, shared expert, routed experts) per path, CUDA events around `reps` calls;
    launch latency bounds it, so only the time per call is reported."""
    import torch

    from bit_expert_ffn_gb300 import synth
    from bit_expert_ffn_gb300.model import LayerShape, MoeLayer, StepBuffers, Workspace

    T = 8
    s = LayerShape(H=256, I=128, E=16, k=2, Is=128, bits=2)
    L = MoeLayer(s, dev)
    L.fill_device(seed=0, layer=0)
    x = torch.from_numpy(synth.activations(0, T, s.H).view(np.int16)).to(dev)
    out = torch.zeros(T, s.H, dtype=torch.float32, device=dev)
    bufs, wsp = StepBuffers(T, s.E, s.k, dev), Workspace(dev)
    res = {"workload": "tiny layer: 8 tokens, H=256, E=16, I=128, top-2, 2-bit, bf16 shared expert I=128"}
    for name, path in (("decode_path_us", m.MOE_PATH_DECODE), ("prefill_path_us", m.MOE_PATH_PREFILL)):
        for _ in range(10):
            L.forward(x, T, out, wsp, bufs, accumulate=False, path=path)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            L.forward(x, T, out, wsp, bufs, accumulate=False, path=path)
        e1.record()
        torch.cuda.synchronize()
        assert m.moe_check_status(L.status) == 0, m.moe_last_error()
        res[name] = 1000.0 * e0.elapsed_time(e1) / reps
    return res


def bench_prefill3(m, dev, T: int = 4096, n_layers: int = LAYERS, reps: int = 3):
    """3-bit prefill: T tokens through the 48-layer residual stack (RMS-normalised bf16 input to each
    layer, fp32 residual stream), prefill path, with uniform and with Zipf(1.4) routing (the same weights,
    only the router bias changes).  CUDA events around each full 48-layer pass.  The same passes through
    the FP8 prefill (an approximation) are reported under "fp8", against twice the bf16 peak."""
    import torch

    from bit_expert_ffn_gb300 import synth
    from bit_expert_ffn_gb300.model import LayerShape, MoeLayer, StepBuffers, Workspace

    s = LayerShape(bits=3)
    layers = []
    for l in range(n_layers):
        L = MoeLayer(s, dev)
        L.fill_device(seed=4, layer=l, zipf_s=0.0)
        layers.append(L)
    x0 = torch.from_numpy(synth.bf16_bits_to_f32(synth.activations(4, T, s.H))).to(dev)
    x = torch.empty_like(x0)
    xb = torch.empty(T, s.H, dtype=torch.int16, device=dev)
    wsp = Workspace(dev)
    bufs = StepBuffers(T, s.E, s.k, dev)
    cgu, sgu = m.moe_packed_size(3, 2 * s.I, s.H)
    cd, sd = m.moe_packed_size(3, s.H, s.I)
    expert_bytes = cgu + sgu + cd + sd  # 2,064,384 for H=2048, I=768
    fixed_bytes = s.E * s.H * 4 + 3 * s.Is * s.H * 2  # router fp32 + shared bf16, every layer
    flop_layer = 2.0 * T * s.k * 3 * s.H * s.I
    peak_t, kind_t = peaks_bf16()
    peak_b, kind_b = peaks()

    def one_pass(path):
        for L in layers:
            m.moe_rms_norm_bf16(x, xb, T, s.H, m.RMS_EPS)
            L.forward(xb, T, x, wsp, bufs, accumulate=True, path=path)

    res, res8 = {}, {}
    for (name, zs), path in [(z, p) for p in (m.MOE_PATH_PREFILL, m.MOE_PATH_PREFILL_FP8)
                             for z in (("uniform", 0.0), ("zipf_1.4", 1.4))]:
        fp8 = path == m.MOE_PATH_PREFILL_FP8
        out, pk = (res8, 2 * peak_t) if fp8 else (res, peak_t)
        for l, L in enumerate(layers):
            L.router_b.copy_(torch.from_numpy(synth.zipf_bias(4, l, s.E, zs)))
        # experts touched per layer (untimed pass, layer by layer)
        x.copy_(x0)
        used = 0
        for L in layers:
            m.moe_rms_norm_bf16(x, xb, T, s.H, m.RMS_EPS)
            L.forward(xb, T, x, wsp, bufs, accumulate=True, path=path)
            used += int((torch.diff(bufs.offsets) > 0).sum().item())
        times = []
        for r in range(reps + 2):
            x.copy_(x0)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            one_pass(path)
            e1.record()
            torch.cuda.synchronize()
            if r >= 2:
                times.append(e0.elapsed_time(e1))
        for L in layers:
            assert m.moe_check_status(L.status) == 0, m.moe_last_error()
        assert bool(torch.isfinite(x).all()), "3-bit prefill output is not finite"
        ms = float(np.median(times))
        nbytes = used * expert_bytes + n_layers * fixed_bytes
        tfl = flop_layer * n_layers / (ms / 1000.0) / 1e12
        gbs = nbytes / (ms / 1000.0) / 1e9
        out[name] = {"value": T / (ms / 1000.0), "unit": "tokens/s", "ms_per_pass": ms,
                     "experts_used_per_layer": used / n_layers,
                     "tensor": {"achieved": tfl, "peak": pk, "unit": "TFLOP/s", "frac": tfl / pk,
                                "peak_kind": kind_t + (" bf16 x 2 (e4m3)" if fp8 else ""),
                                "flop": flop_layer * n_layers, "note": "routed expert FLOP only"},
                     "hbm": {"achieved": gbs, "peak": peak_b, "unit": "GB/s", "frac": gbs / peak_b,
                             "peak_kind": kind_b, "bytes": nbytes,
                             "note": "touched experts + router + shared expert, each read once"}}
    del layers
    torch.cuda.empty_cache()
    return {"workload": f"3-bit prefill: {T} tokens x {n_layers} layers (residual stack), H=2048, E=512, I=768, "
                        "top-10, 3-bit experts (8 levels, 32-weight blocks, fp16 scales), bf16 shared expert",
            **res,
            "fp8": {"workload": "the same passes through the FP8 prefill (e4m3 operands, an approximation; "
                                "tests/test_gpu_prefill_fp8.py reports its error against the exact layer)", **res8}}


def run_ours(args, world, rank, local):
    import ctypes

    import torch

    import bit_expert_ffn_gb300 as m
    from bit_expert_ffn_gb300 import synth
    from bit_expert_ffn_gb300.model import LayerShape, MoeLayer, StepBuffers, Workspace, residual_step

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    lib = m.load()
    shape = LayerShape(H=H, I=I, E=E, k=K_TOP, Is=IS, bits=2)
    NL = args.layers
    bytes_per_token = NL * (K_TOP * EXPERT_BYTES + ROUTER_BYTES + SHARED_BYTES)
    layers = []
    for layer in range(NL):
        L = MoeLayer(shape, dev)
        L.fill_device(seed=0, layer=layer, zipf_s=1.1)
        layers.append(L)
    torch.cuda.synchronize()
    for L in layers:
        assert m.moe_check_status(L.status) == 0, m.moe_last_error()

    n_steps = args.warmup + args.steps
    X = torch.from_numpy(synth.bf16_bits_to_f32(synth.activations(0, n_steps, H, step=rank)).reshape(n_steps, H)).to(dev)
    x_res = torch.zeros(1, H, dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    sptr = ctypes.c_void_p(stream.cuda_stream)

    if args.path == "fused":
        descs = (m.moe_layer_weights * NL)(*[L.weights() for L in layers])
        nb = m.moe_decode_workspace_size(1, H, I, E, K_TOP, IS)
        ws = torch.empty(nb, dtype=torch.uint8, device=dev)
        kernels_per_step = 1

        def call():
            st = lib.moe_decode_forward(descs, NL, x_res.data_ptr(), 1, K_TOP, m.RMS_EPS, None, None,
                                        ws.data_ptr(), nb, status.data_ptr(), sptr)
            if st:
                raise m.MoeError(st, m.moe_last_error())
    else:
        x_bf16 = torch.zeros(1, H, dtype=torch.int16, device=dev)
        bufs = StepBuffers(1, E, K_TOP, dev)
        wsp = Workspace(dev)
        wsp.get(8 << 20)
        kernels_per_step = KERNELS_PER_LAYER * NL
        with torch.cuda.stream(stream):
            residual_step(layers, x_res, x_bf16, 1, wsp, bufs)  # eager warm-up (sizes the workspace)
            stream.synchronize()
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                residual_step(layers, x_res, x_bf16, 1, wsp, bufs)
        torch.cuda.synchronize()

        def call():
            graph.replay()

    def step(i):
        x_res.copy_(X[i:i + 1])
        call()

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(i)
    torch.cuda.synchronize()
    assert m.moe_check_status(status) == 0, m.moe_last_error()
    for L in layers:
        assert m.moe_check_status(L.status) == 0, m.moe_last_error()
    assert bool(torch.isfinite(x_res).all()), "residual stream is not finite"

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for i in range(args.warmup, n_steps):
            step(i)
        e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop()
    assert m.moe_check_status(status) == 0, m.moe_last_error()
    ms = e0.elapsed_time(e1)
    ms = max_over_ranks(world, ms)
    tok_s = world * args.steps / (ms / 1000.0)

    # -- the dominant kernel, timed per launch with events on its own stream
    evs = []
    with torch.cuda.stream(stream):
        for i in range(min(args.steps, 20)):
            x_res.copy_(X[i:i + 1])
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            call()
            b.record(stream)
            evs.append((a, b))
    torch.cuda.synchronize()
    call_ms = float(np.mean([a.elapsed_time(b) for a, b in evs]))
    peak, peak_kind = peaks()
    achieved = bytes_per_token / (call_ms / 1000.0) / 1e9

    # -- end to end through host buffers: pinned x in, result out, every step
    x_host = torch.empty(1, H, dtype=torch.float32, pin_memory=True)
    y_host = torch.empty(1, H, dtype=torch.float32, pin_memory=True)
    x_host.copy_(X[0:1].cpu())
    n_e2e = min(args.steps, 50)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for _ in range(n_e2e):
            x_res.copy_(x_host, non_blocking=True)
            call()
            y_host.copy_(x_res, non_blocking=True)
            stream.synchronize()
    e2e_s = time.perf_counter() - t0
    e2e_s = max_over_ranks(world, e2e_s)
    e2e = {"value": world * n_e2e / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": 4 * H,
           "d2h_bytes_per_step": 4 * H}

    extra = {}
    if args.path == "fused" and not args.no_extra and NL == LAYERS:
        extra["verify_4tok"] = bench_verify(m, lib, layers, descs, dev, stream, steps=min(args.steps, 50), warmup=3)
        extra["verify_4tok_tail_skip"] = bench_verify(m, lib, layers, descs, dev, stream, steps=min(args.steps, 50),
                                                      warmup=3, tail_skip=7)
        extra["decode_l2_hot"] = bench_decode_hot(m, lib, descs, dev, stream, X, steps=min(args.steps, 50),
                                                  warmup=args.warmup)
    if not args.no_extra:  # the decode stack stays resident (36 GB of 288 GB)
        extra["prefill_32k"] = bench_prefill(m, dev)
        extra["prefill_32k_fp8"] = bench_prefill(m, dev, fp8=True)
        extra["prefill_3bit_4k"] = bench_prefill3(m, dev)
        extra["tiny_layer"] = bench_tiny(m, dev)

    if rank == 0:
        cpu = None
        if not args.no_cpu_baseline:
            t_or, n_l = oracle_decode_sample(2)
            cpu = {"value": n_l / LAYERS / t_or, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                   "sample": "one token through 2 of the 48 layers, oracle compute only, scaled by 1/24 "
                             "(fp64 scalar C, one host core)"}
            if "prefill_32k" in extra and "prefill_3bit_4k" in extra:
                c3, c4 = prefill_cpu_baselines()
                extra["prefill_32k"]["cpu_baseline"] = c3
                extra["prefill_3bit_4k"]["cpu_baseline"] = c4
        kernel = (f"decode_kernel (moe_decode_forward: {NL} layers, one cooperative launch)" if args.path == "fused"
                  else f"whole modular step (CUDA graph of {kernels_per_step} launches)")
        line = {
            "metric": "decode tokens/s (48-layer MoE stack, 1 token per step)",
            "value": tok_s, "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32", "data": "synthetic (seeded generator, weights drawn on the GPU)",
            "config": {"workload": WORKLOAD if NL == LAYERS else WORKLOAD.replace("48 layers", f"{NL} layers"),
                       "tokens_per_step": 1, "layers": NL, "parallelism": "replicas",
                       "path": args.path,
                       "l2": "no flush: each step reads 1.36 GB of weights, 10x the 129 MB L2"},
            "hbm_roofline": {"bytes_per_token": bytes_per_token,
                             "achieved_gbs": bytes_per_token * tok_s / world / 1e9,
                             "frac_of_measured": bytes_per_token * tok_s / world / 1e9 / peak},
            "roofline": {"kernel": kernel, "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": decode_traffic(args.path, NL), "peak_kind": peak_kind,
                         "bytes_per_launch": bytes_per_token, "avg_launch_ms": call_ms},
            "clocks": clocks,
            "e2e": e2e,
            "gpu_launches": kernels_per_step * args.steps,
            "cpu_baseline": cpu,
        }
        line.update(extra)
        print(json.dumps(line), flush=True)


def run_only_hot(local: int):
    """Profiling aid: 3 plain 48-layer decode steps, then bench_decode_hot (16 steps that record the routing,
    3 warm-up and 3 timed steps with the hot masks), so one capture holds launches of both variants."""
    import torch

    import bit_expert_ffn_gb300 as m
    from bit_expert_ffn_gb300 import synth
    from bit_expert_ffn_gb300.model import LayerShape, MoeLayer

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    lib = m.load()
    s = LayerShape()
    layers = []
    for layer in range(LAYERS):
        L = MoeLayer(s, dev)
        L.fill_device(seed=0, layer=layer, zipf_s=1.1)
        layers.append(L)
    descs = (m.moe_layer_weights * LAYERS)(*[L.weights() for L in layers])
    X = torch.from_numpy(synth.bf16_bits_to_f32(synth.activations(0, 40, H)).reshape(40, H)).to(dev)
    nb = m.moe_decode_workspace_size(1, H, I, E, K_TOP, IS)
    ws = torch.empty(nb, dtype=torch.uint8, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    x = torch.empty(1, H, device=dev)
    for i in range(3):
        x.copy_(X[i:i + 1])
        m.moe_decode_forward([L.weights() for L in layers], x, 1, K_TOP, m.RMS_EPS, None, None, ws, nb, st)
    torch.cuda.synchronize()
    r = bench_decode_hot(m, lib, descs, dev, torch.cuda.Stream(device=dev), X, steps=3, warmup=3)
    print(json.dumps({k: v for k, v in r.items() if k != "workload"}), flush=True)


def decode_traffic(path: str, n_layers: int):
    """The captured DRAM bytes of the timed launch, if they belong to the current source."""
    if path != "fused" or n_layers != LAYERS:
        return None
    return DECODE_TRAFFIC[0] if decode_source_digest().startswith(DECODE_TRAFFIC[1]) else None


def decode_source_digest() -> str:
    """SHA-256 of the decode kernel's source with comments and whitespace removed (comment edits keep it)."""
    import hashlib
    import re

    src = os.path.join(os.path.dirname(os.path.abspath(__file__)), "bit_expert_ffn_gb300", "csrc", "decode_fused.cu")
    with open(src, encoding="utf-8") as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return hashlib.sha256("".join(text.split()).encode()).hexdigest()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="skip the verify-window and prefill measurements")
    ap.add_argument("--only-prefill", action="store_true", help="run only the 32K-prefill measurement (profiling)")
    ap.add_argument("--fp8", action="store_true", help="with --only-prefill: the FP8 variant")
    ap.add_argument("--only-prefill3", action="store_true",
                    help="run only the 3-bit 4,096-token 48-layer prefill measurement (profiling)")
    ap.add_argument("--only-hot", action="store_true",
                    help="run only the decode with hot-expert L2 hints, after 3 plain decode steps (profiling)")
    ap.add_argument("--path", default="fused", choices=["fused", "modular"])
    ap.add_argument("--layers", type=int, default=LAYERS, help="layers per step (48 is the workload; fewer only "
                    "for profiling captures)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world, rank, local = dist_setup()
    if args.only_prefill3:
        import torch

        import bit_expert_ffn_gb300 as m

        torch.cuda.set_device(local)
        m.load()
        print(json.dumps(bench_prefill3(m, torch.device("cuda", local), n_layers=args.layers)), flush=True)
        return
    if args.only_prefill:
        import torch

        import bit_expert_ffn_gb300 as m

        torch.cuda.set_device(local)
        m.load()
        print(json.dumps(bench_prefill(m, torch.device("cuda", local), fp8=args.fp8)), flush=True)
        return
    if args.only_hot:
        run_only_hot(local)
        return
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()

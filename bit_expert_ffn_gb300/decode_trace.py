"""Phase trace of the fused decode (a development tool).

    python -m bit_expert_ffn_gb300.decode_trace [--T 1] [--layers 48]

Builds a copy of the library with the decode kernel's trace hooks compiled in
(MOE_DECODE_TRACE: thread 0 of every CTA stamps the global timer at each
phase boundary of every layer) into ``_build_trace/`` next to this file, runs
the benchmark's decode stack (H=2048, E=512, I=768, top-10, 2-bit, Zipf(1.1),
seeded weights drawn on the device) for T tokens, and prints, per phase, the
mean over layers of the mean and of the maximum over CTAs of its duration.
The product build (``build.py``) never defines MOE_DECODE_TRACE.
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import ctypes
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
OUT = os.path.join(HERE, "_build_trace")
PHASES = ["x gather", "rms + operands + router rows in", "router + shared rows", "logits in", "routing",
          "copy issue + gate/up", "h barrier", "shared-down rows in", "shared down + staged h", "down items",
          "combine"]


def build_traced() -> str:
    from . import build as b

    os.makedirs(OUT, exist_ok=True)
    srcs = [f for f in sorted(glob.glob(os.path.join(b.CSRC, "*.cu"))) if not f.endswith(b.SYNTH_SRC)]

    def comp(f):
        o = os.path.join(OUT, os.path.basename(f)[:-3] + ".o")
        extra = ["-DMOE_DECODE_TRACE"] if f.endswith("decode_fused.cu") else []
        subprocess.run([b.nvcc()] + b.NVFLAGS + extra + ["-c", f, "-o", o], check=True)
        return o

    with cf.ThreadPoolExecutor(8) as ex:
        objs = list(ex.map(comp, srcs))
    lib = os.path.join(OUT, "libmoe_gb300.so")
    subprocess.run([b.nvcc()] + b.ARCH + ["-shared", "-cudart", "shared", "-o", lib] + objs +
                   ["-Xlinker", "-rpath", "-Xlinker", "/usr/local/cuda/lib64"], check=True)
    return lib


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--T", type=int, default=1)
    ap.add_argument("--layers", type=int, default=48)
    args = ap.parse_args()
    lib_path = build_traced()
    import numpy as np
    import torch

    import bit_expert_ffn_gb300 as m

    m.LIB_PATH = lib_path
    lib = m.load()
    lib.moe_decode_trace_read.argtypes = [ctypes.c_void_p]
    from . import synth
    from .model import LayerShape, MoeLayer

    T, NL = args.T, args.layers
    s = LayerShape()
    layers = []
    for l in range(NL):
        L = MoeLayer(s, "cuda")
        L.fill_device(0, l, zipf_s=1.1)
        layers.append(L)
    descs = [L.weights() for L in layers]
    nb = m.moe_decode_workspace_size(T, s.H, s.I, s.E, s.k, s.Is)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    x0 = torch.from_numpy(synth.bf16_bits_to_f32(synth.activations(0, T, s.H))).cuda()
    x = x0.clone()
    for _ in range(5):
        x.copy_(x0)
        m.moe_decode_forward(descs, x, T, s.k, m.RMS_EPS, None, None, ws, nb, st)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(10):
        x.copy_(x0)
        m.moe_decode_forward(descs, x, T, s.k, m.RMS_EPS, None, None, ws, nb, st)
    e1.record()
    torch.cuda.synchronize()
    print(f"T={T}, {NL} layers: {e0.elapsed_time(e1) / 10:.4f} ms per step (traced build), status "
          f"{m.moe_check_status(st)}")
    buf = np.zeros((64, 160, 12), np.uint64)
    if lib.moe_decode_trace_read(buf.ctypes.data_as(ctypes.c_void_p)) != 0:
        sys.exit("reading the trace failed")
    G = torch.cuda.get_device_properties(0).multi_processor_count
    b = buf[:NL, :G, :].astype(np.float64) / 1000.0
    d = np.diff(b, axis=2)
    print(f"layer (CTA mean): {(b[:, :, 11] - b[:, :, 0]).mean():.2f} us")
    for i, n in enumerate(PHASES):
        print(f"  {n:34s} mean {d[:, :, i].mean():6.2f} us   max over CTAs {d[:, :, i].max(1).mean():6.2f} us")


if __name__ == "__main__":
    main()

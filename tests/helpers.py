"""Shared setup for the GPU parity tests: seeded host inputs and the oracle
comparison helpers.  Inputs come from bit_expert_ffn_gb300.synth only."""
import numpy as np

from bit_expert_ffn_gb300 import synth


def host_layer(seed=0, layer=0, bits=2, H=256, I=128, E=16, Is=128, zipf=0.0):
    """Logical codes/scales of every expert, router weights/bias and shared weights."""
    gate, up, down, gsc, usc, dsc = [], [], [], [], [], []
    for e in range(E):
        g, u, d = synth.expert_codes(seed, layer, e, bits, H, I)
        gus, ds = synth.expert_scales(seed, layer, e, H, I)
        gate.append(g); up.append(u); down.append(d)
        gsc.append(gus[0]); usc.append(gus[1]); dsc.append(ds)
    arena = [np.stack(a) for a in (gate, gsc, up, usc, down, dsc)]
    wr = synth.router_weights(seed, layer, E, H)
    b = synth.zipf_bias(seed, layer, E, zipf)
    shared = synth.shared_weights(seed, layer, H, Is) if Is else None
    return arena, wr, b, shared


def rel_l2(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def u16(t):
    """Device int16 tensor holding bf16/fp16 bits -> host uint16 array."""
    return t.cpu().numpy().view(np.uint16)


def bf16_rne(a):
    return synth.f32_to_bf16_bits(np.asarray(a, np.float32))

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


def device_expert_parts(seed, layer, experts, bits, H, I):
    """The picked experts' logical codes and scales, drawn by the device generator (model.draw_expert_parts)."""
    from bit_expert_ffn_gb300.model import draw_expert_parts

    return draw_expert_parts(seed, layer, experts, bits, H, I)


def oracle_sampled_layer(seed, layer, bits, H, I, x_bf16, ids, w, shared, pool=None, fp8=False):
    """oracle.moe_layer for the tokens of x_bf16 [T][H] with the given routing,
    regenerating only the experts they picked (on the device generator);
    fp8=True takes the routed experts in their FP8 variant.
    With a thread pool the tokens run in parallel (the oracle is C code called
    through ctypes, which releases the GIL)."""
    import oracle

    used = sorted(set(int(e) for e in np.asarray(ids).ravel()))
    remap = {e: i for i, e in enumerate(used)}
    arena = device_expert_parts(seed, layer, used, bits, H, I)
    cids = np.vectorize(remap.get)(np.asarray(ids)).astype(np.int32).reshape(np.shape(ids))
    w = np.asarray(w, np.float64)

    def one(t):
        return oracle.moe_layer(bits, x_bf16[t:t + 1], cids[t:t + 1], w[t:t + 1], *arena, shared=shared,
                                fp8=fp8)[0]

    T = x_bf16.shape[0]
    rows = list(pool.map(one, range(T))) if pool is not None else [one(t) for t in range(T)]
    return np.stack(rows)

"""GPU parity of moe_decode_forward (the fused multi-layer decode) against the
oracle, teacher-forced layer by layer with the routing the kernel reports,
plus its batch invariance and the grid barrier's time limit."""
import numpy as np
import pytest
import torch

import bit_expert_ffn_gb300 as m
import oracle
from bit_expert_ffn_gb300 import synth
from bit_expert_ffn_gb300.model import LayerShape, MoeLayer, StepBuffers, Workspace, residual_step
from helpers import host_layer, rel_l2

pytestmark = pytest.mark.gpu
DEV = "cuda"


def tiny_stack(n_layers, bits=2, H=256, I=128, E=16, k=2, Is=128, zipf=1.1):
    layers, hosts = [], []
    for l in range(n_layers):
        arena, wr, b, shared = host_layer(seed=40 + l, layer=l, bits=bits, H=H, I=I, E=E, Is=Is, zipf=zipf)
        L = MoeLayer(LayerShape(H=H, I=I, E=E, k=k, Is=Is, bits=bits), DEV)
        L.load_host(arena[0], arena[1], arena[2], arena[3], arena[4], arena[5], wr, b, shared)
        layers.append(L)
        hosts.append((arena, wr, b, shared))
    return layers, hosts


def run_fused(layers, x0, k):
    T, H = x0.shape
    s = layers[0].s
    x = torch.from_numpy(x0.copy()).to(DEV)
    n = len(layers)
    ids = torch.empty(n, T, k, dtype=torch.int32, device=DEV)
    w = torch.empty(n, T, k, dtype=torch.float32, device=DEV)
    nb = m.moe_decode_workspace_size(T, s.H, s.I, s.E, k, s.Is)
    ws = torch.empty(nb, dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    m.moe_decode_forward([L.weights() for L in layers], x, T, k, m.RMS_EPS, ids, w, ws, nb, st)
    assert m.moe_check_status(st) == 0, m.moe_last_error()
    return x.cpu().numpy(), ids.cpu().numpy(), w.cpu().numpy()


def layer_input(xr):
    """bf16 of the normalised residual stream, as the stacked layers take it."""
    return synth.f32_to_bf16_bits(oracle.rms_norm(xr.astype(np.float32), m.RMS_EPS).astype(np.float32))


def oracle_stack(bits, x0, ids, w, host_arenas):
    """Residual stack in fp64, routing taken from the kernel, normalised bf16 inputs per layer."""
    xr = x0.astype(np.float64)
    for l, (arena, wr, b, shared) in enumerate(host_arenas):
        xr = xr + oracle.moe_layer(bits, layer_input(xr), ids[l], w[l].astype(np.float64), *arena, shared=shared)
    return xr


@pytest.mark.parametrize("T", [1, 2, 3, 4])
@pytest.mark.parametrize("bits", [2, 3])
def test_one_layer_matches_oracle(moe, T, bits):
    layers, hosts = tiny_stack(1, bits=bits)
    x0 = synth.bf16_bits_to_f32(synth.verify_window(5, T, 256))
    x1, ids, w = run_fused(layers, x0, 2)
    want = oracle_stack(bits, x0, ids, w, hosts)
    assert rel_l2(x1 - x0, want - x0) <= 2e-5
    # routing: the oracle's own selection on its own logits agrees (no near-ties at this size)
    wr, b = hosts[0][1], hosts[0][2]
    lg = oracle.router_logits(layer_input(x0), wr, b)
    oids, ow = oracle.topk(lg.astype(np.float32), 2)
    assert np.array_equal(oids, ids[0])
    np.testing.assert_allclose(w[0], ow, rtol=2e-6, atol=1e-7)


def test_three_layers_teacher_forced(moe):
    layers, hosts = tiny_stack(3, k=4)
    x0 = synth.bf16_bits_to_f32(synth.verify_window(6, 4, 256))
    x3, ids, w = run_fused(layers, x0, 4)
    want = oracle_stack(2, x0, ids, w, hosts)
    assert rel_l2(x3 - x0, want - x0) <= 1e-4


def test_batch_invariance(moe):
    """Each token's result is bit-identical alone and inside a 4-token window."""
    layers, _ = tiny_stack(2, k=4)
    x0 = synth.bf16_bits_to_f32(synth.verify_window(7, 4, 256))
    group, gids, _ = run_fused(layers, x0, 4)
    for t in range(4):
        alone, aids, _ = run_fused(layers, x0[t:t + 1], 4)
        assert np.array_equal(aids[:, 0], gids[:, t])
        assert np.array_equal(alone[0], group[t])


def test_agrees_with_modular_path(moe):
    layers, _ = tiny_stack(2, k=2)
    x0 = synth.bf16_bits_to_f32(synth.verify_window(8, 3, 256))
    fused, ids, _ = run_fused(layers, x0, 2)
    x = torch.from_numpy(x0.copy()).to(DEV)
    xb = torch.empty(3, 256, dtype=torch.int16, device=DEV)
    residual_step(layers, x, xb, 3, Workspace(DEV), StepBuffers(3, 16, 2, DEV), path=m.MOE_PATH_DECODE)
    assert rel_l2(fused - x0, x.cpu().numpy() - x0) <= 2e-5


def test_full_size_two_layers_sampled(moe):
    """H=2048, E=512, I=768, top-10, 2-bit, Zipf(1.1), bf16 shared I=768, T=4 verify window."""
    seed = 3
    s = LayerShape()
    layers = []
    for l in range(2):
        L = MoeLayer(s, DEV)
        L.fill_device(seed, l, zipf_s=1.1)
        layers.append(L)
    x0 = synth.bf16_bits_to_f32(synth.verify_window(seed, 4, s.H))
    x2, ids, w = run_fused(layers, x0, 10)
    xr = x0.astype(np.float64)
    for l in range(2):
        used = sorted(set(int(e) for e in ids[l].ravel()))
        remap = {e: i for i, e in enumerate(used)}
        parts = [[], [], [], [], [], []]
        for e in used:
            g, u, d = synth.expert_codes(seed, l, e, 2, s.H, s.I)
            gus, ds = synth.expert_scales(seed, l, e, s.H, s.I)
            for lst, a in zip(parts, (g, gus[0], u, gus[1], d, ds)):
                lst.append(a)
        arena = [np.stack(p) for p in parts]
        cids = np.vectorize(remap.get)(ids[l]).astype(np.int32)
        shared = synth.shared_weights(seed, l, s.H, s.Is)
        xr = xr + oracle.moe_layer(2, layer_input(xr), cids, w[l].astype(np.float64), *arena, shared=shared)
    assert rel_l2(x2 - x0, xr - x0) <= 1e-4
    # layer 0's selection is the oracle's top-10 of its own logits, up to
    # near-ties that fp32 summation order may flip
    lg = oracle.router_logits(layer_input(x0), synth.router_weights(seed, 0, s.E, s.H),
                              synth.zipf_bias(seed, 0, s.E, 1.1))
    oids, _ = oracle.topk(lg.astype(np.float32), 10)
    for t in range(4):
        if set(ids[0][t]) != set(oids[t]):
            kth = np.sort(lg[t])[::-1][9]
            assert all(abs(lg[t][e] - kth) <= 1e-5 * max(1.0, abs(kth)) for e in set(ids[0][t]) ^ set(oids[t]))


def tie_layer(bias, E=512, H=256, I=128, Is=128):
    """One small-expert layer whose router weights are zero, so the logits are the bias exactly."""
    arena, _, _, shared = host_layer(seed=60, layer=0, bits=2, H=H, I=I, E=E, Is=Is)
    wr = np.zeros((E, H), np.float32)
    b = np.asarray(bias, np.float32)
    L = MoeLayer(LayerShape(H=H, I=I, E=E, k=10, Is=Is, bits=2), DEV)
    L.load_host(arena[0], arena[1], arena[2], arena[3], arena[4], arena[5], wr, b, shared)
    return L, (arena, wr, b, shared)


def _ties_case(name, E=512):
    b = np.full(E, -1.0, np.float32)
    if name == "spread":    # 12 equal logits in 12 lists of 32: 12 survive the threshold
        b[[3, 40, 77, 100, 150, 200, 260, 300, 333, 401, 450, 500]] = 1.0
    elif name == "cluster":  # 9 lists led by 2.0, one list of twenty 1.0s: 29 survive
        b[[45, 90, 130, 170, 210, 250, 290, 330, 370]] = 2.0
        b[0:20] = 1.0
    elif name == "all":      # every logit equal: all survive, so the list merge decides
        b[:] = 0.5
    elif name == "dense":    # 70 top logits in 3 lists: more than 64 survive
        b[100:170] = 3.0 + np.arange(70, dtype=np.float32) % 3
    return b


@pytest.mark.parametrize("case", ["spread", "cluster", "all", "dense"])
@pytest.mark.parametrize("T", [1, 4])
def test_topk_ties_lower_id_first(moe, case, T):
    """Exact ties at E=512, k=10 are broken by the lower expert id, on both the
    threshold-filtered path and the list merge it falls back to."""
    b = _ties_case(case)
    L, host = tie_layer(b)
    x0 = synth.bf16_bits_to_f32(synth.verify_window(9, T, 256))
    x1, ids, w = run_fused([L], x0, 10)
    oids, ow = oracle.topk(np.tile(b, (T, 1)), 10)
    assert np.array_equal(ids[0], oids)
    np.testing.assert_allclose(w[0], ow, rtol=2e-6, atol=1e-7)
    want = oracle_stack(2, x0, ids, w, [host])
    assert rel_l2(x1 - x0, want - x0) <= 2e-5


def test_barrier_completes_and_times_out(moe):
    ws = torch.zeros(16, dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    m.moe_selftest_barrier(0, 1000, ws, 16, st)
    assert m.moe_check_status(st) == 0
    passed = ws.view(torch.int32)[1].item()
    assert passed == torch.cuda.get_device_properties(0).multi_processor_count
    # an unreachable target: every CTA gives up after 200 ms and reports the timeout
    m.moe_selftest_barrier(1, 200, ws, 16, st)
    assert m.moe_check_status(st, reset=True) == m.MOE_ERR_TIMEOUT
    assert ws.view(torch.int32)[1].item() == 0
    # the context is still usable
    m.moe_selftest_barrier(0, 1000, ws, 16, st)
    assert m.moe_check_status(st) == 0


def test_rms_norm_bf16_matches_oracle(moe):
    rng = np.random.default_rng(11)
    x = (rng.normal(0, 3, (5, 2048)) * rng.uniform(0.1, 50, (5, 1))).astype(np.float32)
    out = torch.empty(5, 2048, dtype=torch.int16, device=DEV)
    m.moe_rms_norm_bf16(torch.from_numpy(x).to(DEV), out, 5, 2048)
    got = synth.bf16_bits_to_f32(out.cpu().numpy().view(np.uint16)).astype(np.float64)
    want = oracle.rms_norm(x, m.RMS_EPS)
    assert np.all(np.abs(got - want) <= np.abs(want) * 2.0 ** -8 + 1e-30)  # within one bf16 rounding
    exact = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(want.astype(np.float32)))
    assert np.mean(got == exact) > 0.999


def test_long_stack_stays_finite(moe):
    """Twenty normalised layers keep the residual stream finite (the plain residual sum would not)."""
    layers, _ = tiny_stack(20, k=2)
    x0 = synth.bf16_bits_to_f32(synth.activations(12, 2, 256))
    x, ids, w = run_fused(layers, x0, 2)
    assert np.all(np.isfinite(x))


# ---------------------------------------------------------------- options: route-tail skip, hot-expert hints

def run_fused_ex(layers, x0, k, tail=0, hot=None):
    T, H = x0.shape
    s = layers[0].s
    x = torch.from_numpy(x0.copy()).to(DEV)
    n = len(layers)
    ids = torch.empty(n, T, k, dtype=torch.int32, device=DEV)
    w = torch.empty(n, T, k, dtype=torch.float32, device=DEV)
    nb = m.moe_decode_workspace_size(T, s.H, s.I, s.E, k, s.Is)
    ws = torch.empty(nb, dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    m.moe_decode_forward_ex([L.weights() for L in layers], x, T, k, m.RMS_EPS, tail, hot, ids, w, ws, nb, st)
    assert m.moe_check_status(st) == 0, m.moe_last_error()
    return x.cpu().numpy(), ids.cpu().numpy(), w.cpu().numpy()


def hot_masks(n_layers, E, hot_sets):
    words = (E + 31) // 32
    mask = np.zeros((n_layers, words), np.uint32)
    for l, hs in enumerate(hot_sets):
        for e in hs:
            mask[l, e // 32] |= np.uint32(1 << (e % 32))
    return torch.from_numpy(mask.view(np.int32)).to(DEV)


@pytest.mark.parametrize("T,rank", [(1, 7), (4, 7), (4, 3), (3, 1)])
def test_route_tail_skip_matches_oracle(moe, T, rank):
    """One layer with the skip: the oracle's layer with the left-out pairs' weights set to zero."""
    layers, hosts = tiny_stack(1, k=10, E=24)
    x0 = synth.bf16_bits_to_f32(synth.verify_window(13 + T, T, 256))
    x1, ids, w = run_fused_ex(layers, x0, 10, tail=rank)
    drop = oracle.route_tail_skip(ids[0], rank)
    if T == 1:
        assert drop.sum() == 10 - rank
    assert drop.any()
    weff = np.where(drop, 0.0, w[0].astype(np.float64))
    want = oracle_stack(2, x0, ids, weff[None], hosts)
    assert rel_l2(x1 - x0, want - x0) <= 2e-5
    # and the exact layer differs by the left-out terms
    exact, ids2, _ = run_fused(layers, x0, 10)
    assert np.array_equal(ids, ids2)
    assert not np.array_equal(exact, x1)


def test_route_tail_skip_three_layers(moe):
    layers, hosts = tiny_stack(3, k=10, E=24)
    x0 = synth.bf16_bits_to_f32(synth.verify_window(17, 4, 256))
    x3, ids, w = run_fused_ex(layers, x0, 10, tail=7)
    weff = np.stack([np.where(oracle.route_tail_skip(ids[l], 7), 0.0, w[l].astype(np.float64)) for l in range(3)])
    want = oracle_stack(2, x0, ids, weff, hosts)
    assert rel_l2(x3 - x0, want - x0) <= 1e-4


@pytest.mark.parametrize("T", [1, 4])
def test_options_off_and_hot_masks_keep_the_exact_bits(moe, T):
    """route_tail_skip 0 or k leaves nothing out; hot-expert masks only add cache hints."""
    layers, _ = tiny_stack(2, k=10, E=24)
    x0 = synth.bf16_bits_to_f32(synth.verify_window(19, T, 256))
    exact, ids, w = run_fused(layers, x0, 10)
    rng = np.random.default_rng(T)
    hot = hot_masks(2, 24, [rng.choice(24, 5, replace=False), rng.choice(24, 5, replace=False)])
    for tail, hm in ((0, None), (10, None), (0, hot)):
        got, gids, gw = run_fused_ex(layers, x0, 10, tail=tail, hot=hm)
        assert np.array_equal(got.view(np.uint32), exact.view(np.uint32))
        assert np.array_equal(gids, ids) and np.array_equal(gw.view(np.uint32), w.view(np.uint32))


def test_route_tail_skip_keeps_hot_experts(moe):
    layers, hosts = tiny_stack(1, k=10, E=24)
    x0 = synth.bf16_bits_to_f32(synth.verify_window(23, 4, 256))
    _, ids, _ = run_fused(layers, x0, 10)
    tail_experts = sorted(set(ids[0][:, 7:].ravel().tolist()))
    hot_set = tail_experts[:2]
    x1, ids1, w1 = run_fused_ex(layers, x0, 10, tail=7, hot=hot_masks(1, 24, [hot_set]))
    drop = oracle.route_tail_skip(ids1[0], 7, hot=hot_set)
    weff = np.where(drop, 0.0, w1[0].astype(np.float64))
    want = oracle_stack(2, x0, ids1, weff[None], hosts)
    assert rel_l2(x1 - x0, want - x0) <= 2e-5

"""Invariants of the layer on the GPU paths (the FP8 prefill included), which
hold whatever the oracle says: all block scales zero leaves only the shared expert; identical experts
make the routed sum one expert's output (the weights sum to one); renaming
the experts together with their router rows and biases changes nothing."""
import numpy as np
import pytest
import torch

import bit_expert_ffn_gb300 as m
from bit_expert_ffn_gb300 import synth
from bit_expert_ffn_gb300.model import LayerShape, MoeLayer, StepBuffers, Workspace
from helpers import host_layer, rel_l2

pytestmark = pytest.mark.gpu
DEV = "cuda"
H, I, E, K, IS, T = 256, 128, 16, 2, 128, 8
PATHS = [m.MOE_PATH_DECODE, m.MOE_PATH_PREFILL, m.MOE_PATH_PREFILL_FP8]


def layer(arena, wr, b, shared, bits=2):
    L = MoeLayer(LayerShape(H=H, I=I, E=E, k=K, Is=IS, bits=bits), DEV)
    L.load_host(*arena, wr, b, shared)
    return L


def forward(L, x, path, with_shared=True):
    bufs = StepBuffers(T, E, K)
    out = torch.zeros(T, H, dtype=torch.float32, device=DEV)
    xd = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).to(DEV)
    L.forward(xd, T, out, Workspace(DEV), bufs, accumulate=False, path=path, with_shared=with_shared)
    assert m.moe_check_status(L.status) == 0, m.moe_last_error()
    return out.cpu().numpy(), bufs.ids.cpu().numpy()


def fused(layers, x0, T_):
    x = torch.from_numpy(x0.copy()).to(DEV)
    nb = m.moe_decode_workspace_size(T_, H, I, E, K, IS)
    ws = torch.empty(nb, dtype=torch.uint8, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    m.moe_decode_forward([L.weights() for L in layers], x, T_, K, m.RMS_EPS, None, None, ws, nb, st)
    assert m.moe_check_status(st) == 0, m.moe_last_error()
    return x.cpu().numpy()


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("bits", [2, 3])
def test_zero_scales_leave_the_shared_expert(moe, path, bits):
    arena, wr, b, shared = host_layer(seed=31, bits=bits, H=H, I=I, E=E, Is=IS, zipf=1.1)
    arena = [a if i % 2 == 0 else np.zeros_like(a) for i, a in enumerate(arena)]  # every scale +0
    L = layer(arena, wr, b, shared, bits)
    x = synth.activations(31, T, H)
    got, _ = forward(L, x, path)
    out = torch.zeros(T, H, dtype=torch.float32, device=DEV)
    nb = m.moe_shared_expert_workspace_size(H, IS, T)
    ws = torch.empty(max(nb, 1), dtype=torch.uint8, device=DEV)
    xd = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).to(DEV)
    m.moe_shared_expert(*L.shared, H, IS, xd, T, out, m.MOE_F32, False, ws, nb)
    assert np.array_equal(got, out.cpu().numpy())  # the routed sum adds exact zeros


def test_zero_scales_fused_decode_is_residual_plus_shared(moe):
    arena, wr, b, shared = host_layer(seed=32, bits=2, H=H, I=I, E=E, Is=IS)
    zero = [a if i % 2 == 0 else np.zeros_like(a) for i, a in enumerate(arena)]
    L = layer(zero, wr, b, shared)
    Ls = layer(zero, wr, b, None)  # no shared expert either: the layer adds nothing
    x0 = synth.bf16_bits_to_f32(synth.verify_window(32, 3, H))
    assert np.array_equal(fused([Ls], x0, 3), x0)
    x1 = fused([L], x0, 3)
    # the shared output of the normalised input, through the library calls
    out = torch.zeros(3, H, dtype=torch.float32, device=DEV)
    ub = torch.empty(3, H, dtype=torch.int16, device=DEV)
    m.moe_rms_norm_bf16(torch.from_numpy(x0.copy()).to(DEV), ub, 3, H, m.RMS_EPS)
    nb = m.moe_shared_expert_workspace_size(H, IS, 3)
    ws = torch.empty(max(nb, 1), dtype=torch.uint8, device=DEV)
    m.moe_shared_expert(*L.shared, H, IS, ub, 3, out, m.MOE_F32, False, ws, nb)
    # fp32 sums in another order, and u from the library's own RMS normalisation
    assert rel_l2(x1 - x0, out.cpu().numpy()) <= 1e-4


@pytest.mark.parametrize("path", PATHS)
def test_identical_experts_sum_to_one_expert(moe, path):
    arena, wr, b, shared = host_layer(seed=33, bits=2, H=H, I=I, E=E, Is=IS, zipf=1.1)
    same = [np.repeat(a[:1], E, axis=0) for a in arena]  # expert 0 everywhere
    L = layer(same, wr, b, None)
    x = synth.activations(33, T, H)
    got, _ = forward(L, x, path, with_shared=False)
    # the same tokens through a layer whose router always picks expert 0 with weight 1 in slot 0
    wr1 = np.zeros_like(wr)
    b1 = np.full(E, -30.0, np.float32)
    b1[0] = 30.0
    L1 = layer(same, wr1, b1, None)
    one, ids = forward(L1, x, path, with_shared=False)
    assert (ids[:, 0] == 0).all()
    assert rel_l2(got, one) <= 2e-6  # the weights sum to one within fp32 rounding


@pytest.mark.parametrize("path", PATHS)
def test_relabelled_experts_give_the_same_layer(moe, path):
    arena, wr, b, shared = host_layer(seed=34, bits=2, H=H, I=I, E=E, Is=IS, zipf=1.1)
    perm = np.random.default_rng(34).permutation(E)  # new id of old expert e is perm[e]
    inv = np.argsort(perm)
    arena2 = [a[inv] for a in arena]                # new expert j holds old expert inv[j]
    L1, L2 = layer(arena, wr, b, shared), layer(arena2, wr[inv], b[inv], shared)
    x = synth.activations(34, T, H)
    out1, ids1 = forward(L1, x, path)
    out2, ids2 = forward(L2, x, path)
    assert np.array_equal(perm[ids1], ids2)  # the same experts, under their new names, in the same slots
    assert rel_l2(out2, out1) <= 1e-6

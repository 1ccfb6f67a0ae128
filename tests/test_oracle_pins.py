"""Pins of the oracle against facts that do not come from the oracle itself.

Each test ties one oracle function to something fixed outside it: a value the
pages print, a hand-worked byte pattern, a closed form, a library routine, a
brute-force enumeration, or an invariant of the mathematics.  Together they
are chosen so that a dropped term, a wrong sign, offset or index, or a
transposed operand in the oracle fails at least one of them
(tests/test_oracle_mutants.py plants such mistakes and checks that).
"""
import itertools
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
from scipy.special import expit, softmax

import oracle
from bit_expert_ffn_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
pytestmark = pytest.mark.usefixtures("oracle_lib")


# ---------------------------------------------------------------------------
# number formats and the dequantised value
# ---------------------------------------------------------------------------

def test_fp16_decode_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.fp16_to_double(b) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # signed zeros keep their sign
    assert math.copysign(1.0, oracle.fp16_to_double(0x8000)) == -1.0


def test_bf16_decode_patterns():
    bits = np.arange(0, 65536, 7, dtype=np.uint32).astype(np.uint16)
    with np.errstate(invalid="ignore"):
        ref = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    got = np.array([oracle.bf16_to_double(b) for b in bits])
    nan = np.isnan(ref)
    assert np.array_equal(got[~nan], ref[~nan])


@pytest.mark.parametrize("bits", [2, 3])
def test_dequant_exact_closed_form(bits):
    """(c - (2^bits-1)/2) * s, exactly, for every code over a sweep of fp16 scales."""
    scales = [0x0000, 0x0001, 0x03FF, 0x0400, 0x2E66, 0x3C00, 0x3555, 0x7BFF, 0x8001, 0xBC00, 0xFBFF]
    scales += list(range(0x1000, 0x7C00, 0x0357))
    mid = Fraction(2 ** bits - 1, 2)
    for s in scales:
        sv = Fraction(float(np.uint16(s).view(np.float16)))
        for c in range(2 ** bits):
            want = (c - mid) * sv
            got = oracle.dequant(bits, c, s)
            assert Fraction(got) == want, (bits, c, hex(s))


def test_dequant_levels_symmetric():
    s = 0x3C00  # 1.0
    assert [oracle.dequant(2, c, s) for c in range(4)] == [-1.5, -0.5, 0.5, 1.5]
    assert [oracle.dequant(3, c, s) for c in range(8)] == [-3.5, -2.5, -1.5, -0.5, 0.5, 1.5, 2.5, 3.5]


# ---------------------------------------------------------------------------
# packed format
# ---------------------------------------------------------------------------

def test_pack_hand_worked_examples():
    cases = json.load(open(os.path.join(GOLDEN, "pack_examples.json")))["cases"]
    for case in cases:
        codes = np.array(case["codes"], np.uint8)[None, :]
        got = oracle.pack(case["bits"], codes)[0]
        assert got.tobytes().hex() == case["packed_hex_row"], case["name"]
        assert np.array_equal(oracle.unpack(case["bits"], got[None, :], 32)[0], codes[0])


def test_pack_2bit_every_byte_value_round_trips():
    # 256 bytes -> 1024 codes -> 32 rows of 32 codes
    byte_values = np.arange(256, dtype=np.uint8).reshape(32, 8)
    codes = oracle.unpack(2, byte_values, 32)
    assert codes.max() <= 3
    assert np.array_equal(oracle.pack(2, codes), byte_values)
    # each packed byte holds exactly its four codes, the first in the low bits
    assert np.array_equal(codes.reshape(-1, 4) @ np.array([1, 4, 16, 64]), np.arange(256))


def test_pack_3bit_every_code_every_position():
    rows = []
    for pos in range(32):
        for c in range(8):
            r = np.zeros(32, np.uint8)
            r[pos] = c
            rows.append(r)
    codes = np.stack(rows)
    packed = oracle.pack(3, codes)
    assert packed.shape == (256, 12)
    assert np.array_equal(oracle.unpack(3, packed, 32), codes)
    # a single nonzero code sets bits in at most one low byte and one high bit
    for r, p in zip(codes, packed):
        c = int(r.max())
        ones = sum(bin(b).count("1") for b in p)
        assert ones == bin(c).count("1")


def test_pack_rejects_wide_codes():
    with pytest.raises(oracle.OracleError):
        oracle.pack(2, np.full((1, 32), 4, np.uint8))
    with pytest.raises(oracle.OracleError):
        oracle.pack(3, np.full((1, 32), 8, np.uint8))


@pytest.mark.parametrize("bits,cols", [(2, 64), (2, 2048), (3, 768), (3, 96)])
def test_pack_random_round_trip(bits, cols):
    codes = synth.codes(synth.stream_key(7, 99), 5 * cols, bits).reshape(5, cols)
    packed = oracle.pack(bits, codes)
    assert packed.shape[1] == oracle.packed_row_bytes(bits, cols)
    assert np.array_equal(oracle.unpack(bits, packed, cols), codes)


def test_census_matches_pages():
    """The pages' byte census: 34.0 GB stored, 0.66 GB per token of routed experts."""
    g = json.load(open(os.path.join(GOLDEN, "census.json")))
    H, I = g["hidden"], g["expert_width"]
    per_expert = 0
    for rows, cols in ((2 * I, H), (H, I)):
        per_expert += rows * oracle.packed_row_bytes(2, cols) + rows * (cols // 32) * 2
    assert per_expert == 1_474_560
    gib = 2.0 ** 30
    stored = per_expert * g["layers"] * g["experts_per_layer"] / gib
    per_token = per_expert * g["layers"] * g["active_per_layer"] / gib
    assert abs(stored - g["stored_routed_gib_printed"]) <= g["stored_tolerance_gib"]
    assert abs(per_token - g["per_token_routed_gib_printed"]) <= g["per_token_tolerance_gib"]
    # 3-bit: 3.5 bits per weight
    per_expert3 = sum(r * oracle.packed_row_bytes(3, c) + r * (c // 32) * 2 for r, c in ((2 * I, H), (H, I)))
    assert per_expert3 == 2_064_384


# ---------------------------------------------------------------------------
# router and top-k
# ---------------------------------------------------------------------------

def brute_force_topk(l, k):
    """rank_e = #{e' : l_e' > l_e or (l_e' == l_e and e' < e)}; position = rank."""
    E = len(l)
    ids = [None] * k
    for e in range(E):
        rank = sum(1 for f in range(E) if l[f] > l[e] or (l[f] == l[e] and f < e))
        if rank < k:
            ids[rank] = e
    return ids


def test_router_logits_vs_library_matmul():
    T, H, E = 5, 256, 16
    x = synth.activations(3, T, H)
    w = synth.router_weights(3, 0, E, H)
    b = synth.zipf_bias(3, 0, E, 1.1)
    got = oracle.router_logits(x, w, b)
    ref = synth.bf16_bits_to_f32(x).astype(np.float64) @ w.astype(np.float64).T + b.astype(np.float64)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)
    # without a bias
    np.testing.assert_allclose(oracle.router_logits(x, w), ref - b, rtol=1e-12, atol=1e-12)


def test_topk_brute_force_random_and_ties():
    rng = np.random.default_rng(1)
    for trial in range(200):
        E = int(rng.integers(1, 40))
        k = int(rng.integers(1, E + 1))
        if trial % 3 == 0:
            l = rng.integers(-3, 3, E).astype(np.float32)  # many ties
        else:
            l = rng.normal(0, 1, E).astype(np.float32)
        ids, w = oracle.topk(l[None, :], k)
        assert list(ids[0]) == brute_force_topk(list(l), k)
        assert abs(w.sum() - 1.0) < 1e-12


def test_topk_exhaustive_E4():
    vals = [0.0, 1.0, 2.0, 3.0]
    for pattern in itertools.product(vals, repeat=4):
        l = np.array(pattern, np.float32)
        for k in range(1, 5):
            ids, _ = oracle.topk(l[None, :], k)
            assert list(ids[0]) == brute_force_topk(list(l), k), (pattern, k)


def test_topk_signed_zero_and_infinities():
    l = np.array([-0.0, 0.0, -1.0, 0.0], np.float32)
    ids, w = oracle.topk(l[None, :], 3)
    assert list(ids[0]) == [0, 1, 3]  # -0 == +0: lower id first
    np.testing.assert_allclose(w[0], [1 / 3] * 3, rtol=1e-15)
    l = np.array([1.0, np.inf, 5.0, np.inf, -np.inf], np.float32)
    ids, w = oracle.topk(l[None, :], 3)
    assert list(ids[0]) == [1, 3, 2]
    np.testing.assert_allclose(w[0], [0.5, 0.5, 0.0])
    l = np.full(4, -np.inf, np.float32)
    ids, w = oracle.topk(l[None, :], 2)
    assert list(ids[0]) == [0, 1]
    np.testing.assert_allclose(w[0], [0.5, 0.5])


def test_topk_nan_is_an_error():
    l = np.array([[0.0, np.nan, 1.0]], np.float32)
    with pytest.raises(oracle.OracleError) as e:
        oracle.topk(l, 1)
    assert e.value.status == oracle.ERR_NONFINITE


def test_renorm_weights():
    rng = np.random.default_rng(2)
    l = rng.normal(0, 2, (6, 12)).astype(np.float32)
    # k == E: the weights are the full softmax, in id order of selection
    ids, w = oracle.topk(l, 12)
    full = softmax(l.astype(np.float64), axis=1)
    for t in range(6):
        np.testing.assert_allclose(w[t], full[t, ids[t]], rtol=1e-13)
    # k < E: renormalised softmax of the kept logits == softmax over the kept logits
    ids, w = oracle.topk(l, 4)
    for t in range(6):
        np.testing.assert_allclose(w[t], softmax(l[t, ids[t]].astype(np.float64)), rtol=1e-13)
        assert np.all(np.diff(w[t]) <= 0)  # weights follow the logit order
    # all logits equal -> ids 0..k-1 and w = 1/k
    ids, w = oracle.topk(np.zeros((1, 9), np.float32), 5)
    assert list(ids[0]) == [0, 1, 2, 3, 4]
    np.testing.assert_allclose(w[0], 0.2, rtol=1e-15)


# ---------------------------------------------------------------------------
# permutation
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("T,k,E", [(1, 1, 1), (8, 2, 16), (33, 10, 512), (64, 3, 5), (0, 4, 7)])
def test_permute_brute_force(T, k, E):
    rng = np.random.default_rng(T * 1000 + k)
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]).astype(np.int32) if T else np.zeros((0, k), np.int32)
    offsets, perm, inv = oracle.permute(ids, E)
    flat = ids.reshape(-1)
    order = sorted(range(T * k), key=lambda f: (flat[f], f))
    assert list(perm) == order
    assert offsets[0] == 0 and offsets[E] == T * k
    for e in range(E):
        assert offsets[e + 1] - offsets[e] == int((flat == e).sum())
    assert np.array_equal(inv[perm], np.arange(T * k))


def test_permute_rejects_out_of_range():
    with pytest.raises(oracle.OracleError) as e:
        oracle.permute(np.array([[0, 5]], np.int32), 5)
    assert e.value.status == oracle.ERR_BOUNDS


# ---------------------------------------------------------------------------
# experts and the layer
# ---------------------------------------------------------------------------

def dense(bits, codes, scales):
    """Independent dense expansion: numpy broadcast of the block scales."""
    mid = (2 ** bits - 1) / 2.0
    s = scales.view(np.float16).astype(np.float64)
    return (codes.astype(np.float64) - mid) * np.repeat(s, 32, axis=-1)


def numpy_ffn(bits, gc, gs, uc, us, dc, ds, x):
    g = dense(bits, gc, gs) @ x
    u = dense(bits, uc, us) @ x
    h = g * expit(g) * u
    return dense(bits, dc, ds) @ h


@pytest.mark.parametrize("bits,H,I", [(2, 256, 128), (3, 96, 64), (2, 64, 32)])
def test_expert_ffn_vs_dense_numpy(bits, H, I):
    gc, uc, dc = synth.expert_codes(5, 0, 3, bits, H, I)
    gus, ds = synth.expert_scales(5, 0, 3, H, I)
    x = synth.bf16_bits_to_f32(synth.activations(5, 1, H))[0].astype(np.float64)
    got = oracle.expert_ffn(bits, gc, gus[0], uc, gus[1], dc, ds, x)
    ref = numpy_ffn(bits, gc, gus[0], uc, gus[1], dc, ds, x)
    assert np.linalg.norm(got - ref) <= 1e-12 * np.linalg.norm(ref)


def test_expert_ffn_closed_form_one_hot():
    """One-hot x picks one input column; single-block matrices give a closed form."""
    H, I = 32, 32
    gc = np.full((I, H), 3, np.uint8)  # +1.5 s
    uc = np.full((I, H), 0, np.uint8)  # -1.5 s
    dc = np.full((H, I), 2, np.uint8)  # +0.5 s
    one = np.uint16(0x3C00)
    gs = np.full((I, 1), one, np.uint16)
    us = np.full((I, 1), one, np.uint16)
    ds = np.full((H, 1), np.uint16(0x4000), np.uint16)  # 2.0
    x = np.zeros(H)
    x[7] = 2.0
    g, u = 3.0, -3.0  # 1.5 * 2, -1.5 * 2
    h = g / (1 + math.exp(-g)) * u
    y = I * (0.5 * 2.0) * h
    got = oracle.expert_ffn(2, gc, gs, uc, us, dc, ds, x)
    np.testing.assert_allclose(got, np.full(H, y), rtol=1e-14)


def test_shared_expert_vs_dense_numpy():
    H, I = 128, 64
    wg, wu, wd = synth.shared_weights(4, 0, H, I)
    x = synth.bf16_bits_to_f32(synth.activations(4, 1, H))[0].astype(np.float64)
    got = oracle.shared_expert(wg, wu, wd, x)
    f = lambda a: synth.bf16_bits_to_f32(a).astype(np.float64)
    g, u = f(wg) @ x, f(wu) @ x
    ref = f(wd) @ (g * expit(g) * u)
    assert np.linalg.norm(got - ref) <= 1e-12 * np.linalg.norm(ref)


def small_layer(seed=0, bits=2, T=8, H=256, I=128, E=16, k=2, Is=128):
    gate, up, down, gsc, usc, dsc = [], [], [], [], [], []
    for e in range(E):
        g, u, d = synth.expert_codes(seed, 0, e, bits, H, I)
        gus, ds = synth.expert_scales(seed, 0, e, H, I)
        gate.append(g); up.append(u); down.append(d)
        gsc.append(gus[0]); usc.append(gus[1]); dsc.append(ds)
    arena = [np.stack(a) for a in (gate, gsc, up, usc, down, dsc)]
    shared = synth.shared_weights(seed, 0, H, Is)
    x = synth.activations(seed, T, H)
    wr = synth.router_weights(seed, 0, E, H)
    return x, wr, arena, shared, k


def test_layer_equals_per_token_sum_of_dense_experts():
    x, wr, arena, shared, k = small_layer()
    logits = oracle.router_logits(x, wr).astype(np.float32)
    ids, w = oracle.topk(logits, k)
    out = oracle.moe_layer(2, x, ids, w, *arena, shared=shared)
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    gate, gsc, up, usc, down, dsc = arena
    for t in range(x.shape[0]):
        ref = oracle.shared_expert(*shared, xf[t])
        for j in range(k):
            e = ids[t, j]
            ref = ref + w[t, j] * numpy_ffn(2, gate[e], gsc[e], up[e], usc[e], down[e], dsc[e], xf[t])
        assert np.linalg.norm(out[t] - ref) <= 1e-12 * np.linalg.norm(ref)


def test_replicated_expert_invariant():
    """All experts identical: the routed part equals one expert, whatever the routing (sum w = 1)."""
    x, wr, arena, shared, k = small_layer(seed=1, k=4)
    rep = [np.repeat(a[:1], a.shape[0], axis=0) for a in arena]
    ids, w = oracle.topk(oracle.router_logits(x, wr).astype(np.float32), k)
    out = oracle.moe_layer(2, x, ids, w, *rep, shared=None)
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    for t in range(x.shape[0]):
        one = oracle.expert_ffn(2, rep[0][0], rep[1][0], rep[2][0], rep[3][0], rep[4][0], rep[5][0], xf[t])
        assert np.linalg.norm(out[t] - one) <= 1e-12 * np.linalg.norm(one)


def test_zero_expert_invariant():
    """All scales zero: the layer output is the shared expert, exactly."""
    x, wr, arena, shared, k = small_layer(seed=2)
    zero = list(arena)
    for i in (1, 3, 5):
        zero[i] = np.zeros_like(arena[i])
    ids, w = oracle.topk(oracle.router_logits(x, wr).astype(np.float32), k)
    out = oracle.moe_layer(2, x, ids, w, *zero, shared=shared)
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    for t in range(x.shape[0]):
        assert np.array_equal(out[t], oracle.shared_expert(*shared, xf[t]))


def test_relabelling_invariant():
    """Permuting expert ids together with router rows leaves the layer output unchanged."""
    x, wr, arena, shared, k = small_layer(seed=3, k=3)
    E = wr.shape[0]
    b = synth.zipf_bias(3, 0, E, 1.1)
    ids, w = oracle.topk(oracle.router_logits(x, wr, b).astype(np.float32), k)
    out = oracle.moe_layer(2, x, ids, w, *arena, shared=shared)
    sigma = np.random.default_rng(0).permutation(E)  # new id of old expert e is sigma[e]
    inv = np.argsort(sigma)
    wr2, b2 = wr[inv], b[inv]
    arena2 = [a[inv] for a in arena]
    ids2, w2 = oracle.topk(oracle.router_logits(x, wr2, b2).astype(np.float32), k)
    assert np.array_equal(np.sort(sigma[ids], axis=1), np.sort(ids2, axis=1))
    out2 = oracle.moe_layer(2, x, ids2, w2, *arena2, shared=shared)
    np.testing.assert_allclose(out2, out, rtol=1e-12, atol=1e-14)


def test_layer_tokens_independent():
    x, wr, arena, shared, k = small_layer(seed=4, T=4)
    ids, w = oracle.topk(oracle.router_logits(x, wr).astype(np.float32), k)
    out = oracle.moe_layer(2, x, ids, w, *arena, shared=shared)
    for t in range(4):
        one = oracle.moe_layer(2, x[t:t + 1], ids[t:t + 1], w[t:t + 1], *arena, shared=shared)
        assert np.array_equal(one[0], out[t])


def test_layer_rejects_bad_ids():
    x, wr, arena, shared, k = small_layer(seed=5, T=2)
    ids = np.array([[0, 1], [2, 16]], np.int32)
    with pytest.raises(oracle.OracleError) as e:
        oracle.moe_layer(2, x, ids, np.full((2, 2), 0.5), *arena, shared=shared)
    assert e.value.status == oracle.ERR_BOUNDS


def test_layer_3bit_vs_dense_numpy():
    x, wr, arena, shared, k = small_layer(seed=6, bits=3, T=3, H=64, I=32, E=5, k=2, Is=32)
    ids, w = oracle.topk(oracle.router_logits(x, wr).astype(np.float32), k)
    out = oracle.moe_layer(3, x, ids, w, *arena, shared=None)
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    gate, gsc, up, usc, down, dsc = arena
    for t in range(3):
        ref = sum(w[t, j] * numpy_ffn(3, gate[e], gsc[e], up[e], usc[e], down[e], dsc[e], xf[t])
                  for j, e in enumerate(ids[t]))
        assert np.linalg.norm(out[t] - ref) <= 1e-12 * np.linalg.norm(ref)


# ---------------------------------------------------------------------------
# the FP8 variant: e4m3 and fp16 rounding, the scaling exponent, the expert
# ---------------------------------------------------------------------------

def e4m3_table():
    """Every e4m3 byte decoded by torch's float8_e4m3fn (a library routine)."""
    torch = pytest.importorskip("torch")
    b = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return b.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_e4m3_decode_all_codes():
    ref = e4m3_table()
    got = np.array([oracle.e4m3_to_double(b) for b in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan) and nan.sum() == 2  # 0x7F, 0xFF
    assert np.array_equal(got[~nan], ref[~nan])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9 and got[0x08] == 2.0 ** -6 and got[0x38] == 1.0


def brute_e4m3(v, table):
    """Nearest finite e4m3 value by enumeration; a tie goes to the code whose
    mantissa is even (the byte's lowest bit clear)."""
    codes = [c for c in range(256) if not np.isnan(table[c])]
    d = np.array([abs(v - table[c]) for c in codes])
    best = np.flatnonzero(d == d.min())
    cands = [codes[i] for i in best]
    if len(cands) > 1:
        even = [c for c in cands if c & 1 == 0]
        cands = even or cands
    val = table[cands[0]]
    return math.copysign(abs(val), v) if val == 0 else val


def test_e4m3_round_brute_force_and_library():
    torch = pytest.importorskip("torch")
    table = e4m3_table()
    rng = np.random.default_rng(11)
    fin = np.unique(table[~np.isnan(table)])
    mids = (fin[1:] + fin[:-1]) / 2  # exact ties
    vals = np.concatenate([
        np.exp2(rng.uniform(-14, 10, 3000)) * rng.choice([-1, 1], 3000),
        mids, -mids, mids * (1 + 2.0 ** -30), mids * (1 - 2.0 ** -30),
        [448.0, 455.9, 464.0, 479.0, 480.0, 1e4, 1e6, -1e4, 2.0 ** -10, 2.0 ** -11, 3 * 2.0 ** -11],
    ])
    got = oracle.e4m3_round(vals)
    want = np.array([brute_e4m3(v, table) for v in vals])
    assert np.array_equal(got, want)
    # torch's own conversion agrees inside the finite range (inputs exact in fp32)
    v32 = vals.astype(np.float32)
    inr = np.abs(v32) < 448
    t = torch.from_numpy(v32[inr]).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(oracle.e4m3_round(v32[inr].astype(np.float64)), t)
    assert list(oracle.e4m3_round([np.inf, 1e30, -1e30])) == [448.0, 448.0, -448.0] and np.isnan(oracle.e4m3_round([np.nan])[0])


def test_fp16_round_vs_numpy():
    rng = np.random.default_rng(12)
    f16 = np.arange(0, 0x7C00, 37, dtype=np.uint32).astype(np.uint16).view(np.float16).astype(np.float64)
    ulp = np.spacing(f16.astype(np.float16)).astype(np.float64)
    vals = np.concatenate([
        np.exp2(rng.uniform(-26, 16, 3000)) * rng.choice([-1, 1], 3000),
        f16 + ulp / 2, f16 + ulp / 2 * (1 + 2.0 ** -40), -(f16 + ulp / 2),
        [65504.0, 65519.0, 65520.0, 70000.0, 2.0 ** -25, 3 * 2.0 ** -26],
    ])
    got = oracle.fp16_round(vals)
    with np.errstate(over="ignore"):
        want = vals.astype(np.float16).astype(np.float64)
    assert np.array_equal(got, want)


def test_fp8_exponent_closed_forms():
    cases = {1.0: 7, 1.999: 7, 2.0: 6, 0.75: 8, 255.0: 0, 256.0: -1, 2.0 ** -57: 64, 2.0 ** -60: 64,
             2.0 ** 71: -64, 2.0 ** 70: -63, 0.0: 0, float("inf"): 0}
    for a, e in cases.items():
        assert oracle.fp8_exponent(a) == e, a
    rng = np.random.default_rng(13)
    for a in np.exp2(rng.uniform(-50, 60, 500)):
        e = oracle.fp8_exponent(a)
        assert 128 <= a * 2.0 ** e < 256


def fp8_closed_form_expert():
    """H = I = 64.  Gate rows: +0.5 * 128 on block 0, scale 0 on block 1, so
    g = 64 (silu(64) = 64 in double); up rows: +0.5 on both blocks, so
    u = (1 + 2^-4 + 2^-12) / 2 and h = 32 (1 + 2^-4 + 2^-12); down rows:
    +1.5 with block scales 1 and 4.  x = (1 at 0, 2^-4 at 32, 2^-12 at 33).
    Every operand but h is exact in e4m3 after its scaling.  h rounds to
    fp16 34 = 32 * 1.0625, then h * 2^2 = 136 is an e4m3 tie between 128 and
    144 and goes to 128: the effective h is 32 in every row, and
    y_o = 32 * 1.5 * 32 + 32 * (1.5 * 4) * 32 = 7680."""
    H = I = 64
    gc = np.full((I, H), 2, np.uint8)
    uc = np.full((I, H), 2, np.uint8)
    dc = np.full((H, I), 3, np.uint8)
    f16 = lambda v: np.float16(v).view(np.uint16)
    gs = np.tile(np.array([f16(128.0), f16(0.0)], np.uint16), (I, 1))
    us = np.full((I, 2), f16(1.0), np.uint16)
    ds = np.tile(np.array([f16(1.0), f16(4.0)], np.uint16), (H, 1))
    x = np.zeros(H)
    x[0], x[32], x[33] = 1.0, 2.0 ** -4, 2.0 ** -12
    return gc, gs, uc, us, dc, ds, x


def test_expert_ffn_fp8_closed_form():
    gc, gs, uc, us, dc, ds, x = fp8_closed_form_expert()
    got = oracle.expert_ffn_fp8(2, gc, gs, uc, us, dc, ds, x)
    assert np.array_equal(got, np.full(64, 7680.0))
    # the exact expert on the same input: h = 32 (1 + 2^-4 + 2^-12) unrounded
    exact = oracle.expert_ffn(2, gc, gs, uc, us, dc, ds, x)
    np.testing.assert_allclose(exact, np.full(64, 240.0 * 32 * (1 + 2.0 ** -4 + 2.0 ** -12)), rtol=1e-14)


@pytest.mark.parametrize("bits", [2, 3])
def test_expert_ffn_fp8_vs_library_roundings(bits):
    """The FP8 expert rebuilt from library roundings (torch's e4m3 cast,
    numpy's fp16 cast) and numpy's dense products, the exponents by frexp."""
    torch = pytest.importorskip("torch")
    H, I = 256, 128
    maxc = (2 ** bits - 1) / 2.0
    gc, uc, dc = synth.expert_codes(7, 0, 2, bits, H, I)
    gus, ds = synth.expert_scales(7, 0, 2, H, I)
    x = synth.bf16_bits_to_f32(synth.activations(7, 1, H))[0].astype(np.float64)

    def expo(a):
        m, e = np.frexp(a)
        return np.where(a == 0, 0, np.clip(8 - e, -64, 64))

    def e4m3(v):  # v exact in fp32 here
        return torch.from_numpy(np.asarray(v, np.float32)).to(torch.float8_e4m3fn).to(torch.float64).numpy()

    def fp8_dense(codes, scales):
        w = dense(bits, codes, scales)
        kw = expo(maxc * np.abs(scales.view(np.float16).astype(np.float64)).max(axis=1))
        return e4m3(w * np.exp2(kw)[:, None]), kw

    ex = expo(np.abs(x).max())
    x8 = e4m3(x * 2.0 ** ex)
    wg, kg = fp8_dense(gc, gus[0])
    wu, ku = fp8_dense(uc, gus[1])
    wd, kd = fp8_dense(dc, ds)
    g = (wg @ x8) * np.exp2(-(kg + ex))
    u = (wu @ x8) * np.exp2(-(ku + ex))
    h = (g * expit(g) * u).astype(np.float16).astype(np.float64)
    eh = expo(np.abs(h).max())
    h8 = e4m3(h * 2.0 ** eh)
    want = (wd @ h8) * np.exp2(-(kd + eh))
    got = oracle.expert_ffn_fp8(bits, gc, gus[0], uc, gus[1], dc, ds, x)
    assert np.linalg.norm(got - want) <= 1e-12 * np.linalg.norm(want)
    # and it is an approximation of the exact expert at the size e4m3 implies
    exact = oracle.expert_ffn(bits, gc, gus[0], uc, gus[1], dc, ds, x)
    err = np.linalg.norm(got - exact) / np.linalg.norm(exact)
    assert 5e-3 < err < 0.15, err


def test_expert_ffn_fp8_power_of_two_scalings():
    """Scaling a down row's block scales by 2^j scales that output by 2^j
    exactly; scaling every up scale by 2^j scales the whole output by 2^j
    (h moves by 2^j in fp16's normal range, its exponent absorbs it)."""
    bits, H, I = 2, 128, 64
    gc, uc, dc = synth.expert_codes(8, 0, 1, bits, H, I)
    gus, ds = synth.expert_scales(8, 0, 1, H, I)
    x = synth.bf16_bits_to_f32(synth.activations(8, 1, H))[0].astype(np.float64)
    base = oracle.expert_ffn_fp8(bits, gc, gus[0], uc, gus[1], dc, ds, x)
    sc = lambda a, j: (a.view(np.float16).astype(np.float64) * 2.0 ** j).astype(np.float16).view(np.uint16)
    ds2 = ds.copy()
    ds2[5] = sc(ds[5], 3)
    got = oracle.expert_ffn_fp8(bits, gc, gus[0], uc, gus[1], dc, ds2, x)
    want = base.copy()
    want[5] *= 8.0
    assert np.array_equal(got, want)
    got = oracle.expert_ffn_fp8(bits, gc, gus[0], uc, sc(gus[1], -2), dc, ds, x)
    assert np.array_equal(got, base / 4.0)


def test_expert_ffn_fp8_nonfinite():
    gc, gs, uc, us, dc, ds, x = fp8_closed_form_expert()
    x2 = x.copy()
    x2[3] = np.inf
    with pytest.raises(oracle.OracleError) as e:
        oracle.expert_ffn_fp8(2, gc, gs, uc, us, dc, ds, x2)
    assert e.value.status == oracle.ERR_NONFINITE
    us2 = us.copy()
    us2[0, 0] = np.uint16(0x7C00)  # +inf scale
    with pytest.raises(oracle.OracleError):
        oracle.expert_ffn_fp8(2, gc, gs, uc, us2, dc, ds, x)


def test_layer_fp8_equals_per_token_sum():
    x, wr, arena, shared, k = small_layer(seed=9)
    ids, w = oracle.topk(oracle.router_logits(x, wr).astype(np.float32), k)
    out = oracle.moe_layer(2, x, ids, w, *arena, shared=shared, fp8=True)
    xf = synth.bf16_bits_to_f32(x).astype(np.float64)
    gate, gsc, up, usc, down, dsc = arena
    for t in range(x.shape[0]):
        ref = oracle.shared_expert(*shared, xf[t])
        for j in range(k):
            e = ids[t, j]
            ref = ref + w[t, j] * oracle.expert_ffn_fp8(2, gate[e], gsc[e], up[e], usc[e], down[e], dsc[e], xf[t])
        assert np.linalg.norm(out[t] - ref) <= 1e-12 * np.linalg.norm(ref)
    # zero scales leave exactly the shared expert
    zero = list(arena)
    for i in (1, 3, 5):
        zero[i] = np.zeros_like(arena[i])
    out0 = oracle.moe_layer(2, x, ids, w, *zero, shared=shared, fp8=True)
    for t in range(x.shape[0]):
        assert np.array_equal(out0[t], oracle.shared_expert(*shared, xf[t]))


# ---------------------------------------------------------------------------
# residual-stream normalisation in front of each stacked layer
# ---------------------------------------------------------------------------

def test_rms_norm_closed_forms():
    H = 64
    c = np.full((1, H), 3.0, np.float32)
    np.testing.assert_allclose(oracle.rms_norm(c, 0.0), 1.0, rtol=1e-15)
    # eps enters under the root: mean(x^2) = 9, so each entry is 3 / sqrt(9 + eps)
    np.testing.assert_allclose(oracle.rms_norm(c, 7.0), 3.0 / 4.0, rtol=1e-15)
    x = np.zeros((1, H), np.float32)
    x[0, 5] = -2.0  # mean(x^2) = 4/H
    y = oracle.rms_norm(x, 0.0)
    np.testing.assert_allclose(y[0, 5], -2.0 / np.sqrt(4.0 / H), rtol=1e-15)
    assert np.count_nonzero(y) == 1


def test_rms_norm_properties():
    rng = np.random.default_rng(3)
    x = rng.normal(0, 5, (4, 2048)).astype(np.float32)
    y = oracle.rms_norm(x, 0.0)
    np.testing.assert_allclose((y ** 2).mean(axis=1), 1.0, rtol=1e-12)  # unit mean square
    np.testing.assert_allclose(oracle.rms_norm(x * np.float32(8.0), 0.0), y, rtol=1e-12)  # scale invariant
    ref = x.astype(np.float64) / np.sqrt((x.astype(np.float64) ** 2).mean(axis=1, keepdims=True) + 1e-6)
    np.testing.assert_allclose(oracle.rms_norm(x, 1e-6), ref, rtol=1e-13)


# ---------------------------------------------------------------- route-tail skip
# "How Strata runs a 125-billion-parameter model ...", Step 2, "Verify-window
# route tail skip": experts every token of the window ranks 7..9 are skipped,
# experts ranked 0..6 by at least one token and fast-tier ones are kept.

def test_route_tail_skip_single_token_drops_ranks_7_to_9():
    ids = np.array([[40, 41, 42, 43, 44, 45, 46, 47, 48, 49]])
    got = oracle.route_tail_skip(ids, 7)
    assert got.tolist() == [[False] * 7 + [True] * 3]


def test_route_tail_skip_keeps_an_expert_another_token_ranks_early():
    # token 1 ranks expert 9 first: token 0's rank-9 pair is kept; expert 8 is
    # at the tail for both tokens: both its pairs go; expert 7 only in token 0's tail
    ids = np.array([[0, 1, 2, 3, 4, 5, 6, 7, 8, 9],
                    [9, 10, 11, 12, 13, 14, 15, 16, 8, 17]])
    got = oracle.route_tail_skip(ids, 7)
    want = np.zeros((2, 10), bool)
    want[0, 7] = want[0, 8] = True   # 7 and 8 nobody ranks early; 9 is kept
    want[1, 7] = want[1, 8] = want[1, 9] = True  # 16, 8, 17
    assert np.array_equal(got, want)


def test_route_tail_skip_hot_experts_and_off():
    ids = np.array([[0, 1, 2, 3, 4, 5, 6, 7, 8, 9]])
    assert oracle.route_tail_skip(ids, 7, hot=[8]).tolist() == [[False] * 7 + [True, False, True]]
    assert not oracle.route_tail_skip(ids, 0).any()
    assert not oracle.route_tail_skip(ids, 10).any()
    # a threshold of 1 keeps only what some token ranks first
    ids2 = np.array([[3, 1], [1, 3]])
    assert not oracle.route_tail_skip(ids2, 1).any()
    assert oracle.route_tail_skip(np.array([[3, 1], [2, 4]]), 1).tolist() == [[False, True], [False, True]]


def test_route_tail_skip_brute_force_definition():
    """Against the definition enumerated over every (token, slot) of random windows."""
    rng = np.random.default_rng(3)
    for _ in range(200):
        T, k, E = rng.integers(1, 5), rng.integers(1, 11), rng.integers(10, 30)
        ids = np.stack([rng.permutation(E)[:k] for _ in range(T)])
        r = int(rng.integers(0, k + 1))
        hot = set(rng.choice(E, 3, replace=False).tolist())
        got = oracle.route_tail_skip(ids, r, hot)
        for t in range(T):
            for j in range(k):
                e = ids[t, j]
                early = any(ids[tt, jj] == e for tt in range(T) for jj in range(k) if jj < r)
                assert got[t, j] == (r > 0 and j >= r and e not in hot and not early)

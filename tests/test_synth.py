"""The seeded input generator: determinism, distributions and the Zipf routing shape."""
import numpy as np

import oracle
from bit_expert_ffn_gb300 import synth


def test_splitmix64_reference_values():
    # SplitMix64 seeded with 0 (state += golden gamma, then the output mix):
    # first outputs as published with the generator's reference C code.
    outs = synth.u64(0, np.arange(3, dtype=np.uint64))
    assert [int(v) for v in outs] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_deterministic_and_stream_separated():
    k1 = synth.stream_key(0, synth.TAG_GU_CODES, 3, 7)
    k2 = synth.stream_key(0, synth.TAG_GU_CODES, 3, 8)
    a = synth.codes(k1, 1000, 2)
    assert np.array_equal(a, synth.codes(k1, 1000, 2))
    assert not np.array_equal(a, synth.codes(k2, 1000, 2))
    # a window starting mid-stream equals the slice of the full stream
    assert np.array_equal(synth.codes(k1, 100, 2, start=400), a[400:500])
    assert np.array_equal(synth.normal(k1, 50, start=10), synth.normal(k1, 60)[10:])


def test_code_distribution_uniform():
    for bits in (2, 3):
        c = synth.codes(synth.stream_key(1, 1), 400_000, bits)
        counts = np.bincount(c, minlength=2 ** bits)
        assert len(counts) == 2 ** bits
        expect = len(c) / 2 ** bits
        chi2 = ((counts - expect) ** 2 / expect).sum()
        assert chi2 < 40


def test_normal_moments():
    z = synth.normal(synth.stream_key(2, 2), 1_000_000).astype(np.float64)
    assert abs(z.mean()) < 5e-3
    assert abs(z.std() - 1.0) < 5e-3
    assert np.abs(z).max() < 4.9
    kurt = ((z - z.mean()) ** 4).mean() / z.var() ** 2
    assert 2.7 < kurt < 3.0  # Irwin-Hall(8): 3 - 1.2/8 = 2.85


def test_bf16_rounding_is_nearest_even():
    v = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -9, -2.5], np.float32)
    got = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(v))
    assert list(got) == [1.0, 1.0, 1.0 + 4 * 2 ** -8, 1.0, -2.5]


def test_zipf_slope_and_uniform():
    """Router bias from the generator gives a Zipf(1.1) pick-count slope on 4,096 tokens."""
    H, E, K, T = 2048, 512, 10, 4096
    w = synth.router_weights(0, 0, E, H).astype(np.float64)
    x = synth.bf16_bits_to_f32(synth.activations(0, T, H, step=1000)).astype(np.float64)
    rank = synth.zipf_rank(0, 0, E)
    assert sorted(rank) == list(range(E))
    for s in (1.1, 1.4):
        logits = (x @ w.T + synth.zipf_bias(0, 0, E, s)).astype(np.float32)
        ids, _ = oracle.topk(logits, K)
        by_rank = np.bincount(ids.ravel(), minlength=E)[np.argsort(rank)]
        r = np.arange(1, E + 1)
        m = (by_rank < 0.5 * T) & (by_rank > 0)
        slope = np.polyfit(np.log(r[m]), np.log(by_rank[m]), 1)[0]
        assert abs(slope + s) < 0.05, (s, slope)
    assert np.all(synth.zipf_bias(0, 0, E, 0) == 0)

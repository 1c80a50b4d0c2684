"""The seeded generator: determinism, slicing, and distribution shape."""
import numpy as np

from bit_expert_weight_gb300 import synth as S


def test_splitmix64_reference_values():
    """SplitMix64 seeded with 0 (state += gamma, then mix) is a published
    sequence: 0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F."""
    got = S.words(0, 0, 3)
    assert [int(v) for v in got] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4,
                                     0x06C45D188009454F]


def test_streams_are_sliceable_and_deterministic():
    key = S.stream_key(3, 1, 2, 0)
    a = S.values_f32(key, 1000, 0.02, p_out=0.01)
    b = S.values_f32(key, 300, 0.02, p_out=0.01, start=700)
    assert np.array_equal(a[700:], b)
    assert np.array_equal(a, S.values_f32(key, 1000, 0.02, p_out=0.01, chunk=37))
    assert not np.array_equal(a, S.values_f32(S.stream_key(3, 1, 2, 1), 1000, 0.02))


def test_distribution_shape():
    key = S.stream_key(0, 0, 0, 0)
    v = S.values_f32(key, 200000, 0.02, p_out=0.01, p_zero=0.2)
    zeros = np.mean(v == 0.0)
    assert abs(zeros - 0.2) < 0.01
    nz = v[v != 0]
    big = np.mean(np.abs(nz) > 0.02 * 7)  # only outliers exceed ~6 sigma
    assert 0.004 < big < 0.012
    core = S.values_f32(key, 200000, 1.0)
    assert abs(core.std() - 1.0) < 0.01 and abs(core.mean()) < 0.01
    assert np.abs(core).max() <= 6.0


def test_bf16_rounding_is_nearest_even():
    v = np.array([1.0, 1.00390625, 1.01171875, -2.5, 3.0e-3], np.float32)
    bits = S._f32_to_bf16_rne(v)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7 -> even (1.0)
    assert S.bf16_to_f32(bits)[1] == 1.0
    assert S.bf16_to_f32(bits)[2] == np.float32(1.015625)
    ref = v.astype(np.float32)
    assert np.all(np.abs(S.bf16_to_f32(bits) - ref) <= np.abs(ref) * 2.0 ** -8)


def test_zipf_bias_construction():
    """The batched Qwen-like workload's selection-only bias: a seeded
    permutation of Zipf(1.1) popularities, tau calibrated so the most popular
    expert is in the top-k of ~p_1 of the tokens (checked on a 1024-token
    sample, with the margin widened for the smaller sample)."""
    wl = S.WORKLOADS["qwen235b_batched"]
    rank = wl.zipf_ranks()
    assert sorted(rank.tolist()) == list(range(1, wl.E + 1))
    p = wl.zipf_p()
    assert abs(p.sum() - 1.0) < 1e-12
    assert np.allclose(p * (rank.astype(float) ** 1.1), p[np.argmin(rank)])
    b = wl.zipf_bias()
    assert b.dtype == np.float32 and np.array_equal(b, wl.zipf_bias())
    target = float(p.max())
    lg = wl.zipf_logits(0, 1024)
    s_lo, s_mid, s_hi = (wl.zipf_share(0, t, 1024, lg) for t in (0.25, wl.zipf_tau, 0.5))
    assert s_lo < s_mid < s_hi
    assert abs(s_mid - target) <= 0.2 * target


def test_c_twin_matches_the_numpy_definition():
    """values_bf16 runs the plain-C twin of the generator; it must give the
    numpy definition's bits for every parameter mix (outliers, zeros, an
    offset start, the tiny layer's 20 % zeros, unit-sigma activations)."""
    cases = [
        (S.stream_key(1, 0, 3, S.ROLE_GATE), 50_000, 0.02, 0.01, 0.0, 0),
        (S.stream_key(2, 93, 127, S.ROLE_DOWN), 20_000, 0.02, 0.01, 0.0, 123_457),
        (S.stream_key(0, 0, 5, S.ROLE_UP), 30_000, 0.02, 0.01, 0.20, 0),
        (S.stream_key(3, 0, 0, S.ROLE_X), 10_000, 1.0, 0.0, 0.0, 4096 * 7),
        (S.stream_key(4, 1, S.SHARED_EXPERT, S.ROLE_SHARED_GATE), 2048, 0.02, 0.0, 0.0, 0),
    ]
    for key, n, sigma, p_out, p_zero, start in cases:
        a = S.values_bf16(key, n, sigma, p_out=p_out, p_zero=p_zero, start=start)
        b = S.values_bf16_numpy(key, n, sigma, p_out=p_out, p_zero=p_zero, start=start)
        assert a.dtype == np.uint16 and a.shape == (n,)
        assert np.array_equal(a, b), (key, start)


def test_bf16_activations_are_the_rounded_fp32_stream():
    """Workload.activations takes bf16 tokens from the C twin; they must be
    the bf16 rounding of the fp32 stream (the definition), also at an
    offset token."""
    wl = S.WORKLOADS["deepseek16b"]
    for start in (0, 7):
        x, bits = wl.activations(3, 5, start_token=start)
        key = S.stream_key(wl.seed, 3, 0, S.ROLE_X)
        v = S.values_f32(key, 5 * wl.d, 1.0, start=start * wl.d).reshape(5, wl.d)
        assert np.array_equal(bits, S._f32_to_bf16_rne(v))
        assert np.array_equal(x, S.bf16_to_f32(bits))

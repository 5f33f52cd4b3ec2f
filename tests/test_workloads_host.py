"""The seeded input generators (no GPU): the recipe the tests and the bench
rely on -- one PCG64 generator per rank seeded base + r, fp32 draws rounded to
bf16 to nearest-even, the stated ranges and special-value mix, and the Llama
bucket workload's sizes -- so that inputs are reproducible from the recipe
alone."""
import numpy as np
import pytest

from ring_allreduce_rank_gb300 import workloads as W


def _pcg(seed):
    return np.random.Generator(np.random.PCG64(seed))


@pytest.mark.parametrize("fn", [lambda N, K, b: W.normal_bf16(N, K, seed_base=b),
                                lambda N, K, b: W.uniform_fp32(N, K, seed_base=b),
                                lambda N, K, b: W.mixed_fp32(N, K, seed_base=b),
                                lambda N, K, b: W.mixed_bf16(N, K, seed_base=b)])
def test_rank_r_is_drawn_from_seed_base_plus_r(fn):
    N, K, b = 5, 1001, 40
    x = fn(N, K, b)
    assert x.shape == (N, K)
    for r in range(N):
        np.testing.assert_array_equal(x[r], fn(1, K, b + r)[0])
    np.testing.assert_array_equal(x, fn(N, K, b))  # deterministic


def test_normal_bf16_recipe():
    K, std = 1 << 20, 1e-3
    bits = W.normal_bf16(1, K, std=std, seed_base=7)[0]
    x = _pcg(7).standard_normal(K, dtype=np.float32) * np.float32(std)
    np.testing.assert_array_equal(bits, W.to_bf16_bits(x))
    v = W.bf16_bits_to_f32(bits).astype(np.float64)
    assert abs(v.std() / std - 1) < 0.01 and abs(v.mean()) < 5 * std / np.sqrt(K)


def test_bf16_rounding_is_to_nearest_even():
    f = lambda *b: np.array(b, dtype=np.uint32).view(np.float32)
    got = W.to_bf16_bits(f(0x3f808000, 0x3f818000, 0x3f808001, 0x7f800000, 0xff800000, 0x80000000, 0x00000001))
    # ties go to the even neighbour; above a tie rounds up; inf, -0 and the
    # smallest subnormal (rounded to +0) keep their meaning
    assert [hex(v) for v in got] == ["0x3f80", "0x3f82", "0x3f81", "0x7f80", "0xff80", "0x8000", "0x0"]
    nan = W.to_bf16_bits(f(0x7fc00000, 0x7f800001))
    assert all((v & 0x7f80) == 0x7f80 and (v & 0x7f) for v in nan)


def test_integers_and_uniform_ranges():
    x = W.integers_fp32(4, 1 << 16, seed=0)
    assert x.min() == -8 and x.max() == 8 and (x == np.round(x)).all()
    u = W.uniform_fp32(3, 1 << 16, lo=-1.0, hi=1.0, seed_base=2)
    assert u.min() >= -1.0 and u.max() < 1.0 and u.dtype == np.float32


def test_mixed_values_carry_the_special_cases():
    x = W.mixed_fp32(2, 1 << 16, seed_base=3)
    frac = np.isin(x.view(np.uint32), W.special_values_fp32().view(np.uint32)).mean()
    assert 0.04 < frac < 0.07  # 5 % drawn from the specials (plus chance matches)
    b = x.view(np.uint32)
    assert np.isnan(x).any() and np.isinf(x).any()
    assert ((b & 0x7f800000) == 0).any() and (b == 0x80000000).any()  # subnormals and -0
    mags = np.abs(x[np.isfinite(x) & (x != 0)])
    assert mags.min() < 2.0 ** -25 and mags.max() > 2.0 ** 25  # magnitudes spread over 2^±30


def test_llama_bucket_workload_sizes():
    numels = W.llama_layer_numels(4)
    assert len(numels) == 36 and sum(numels) == 809_533_440
    assert numels[:9] == [4096, 4096 ** 2, 4096 ** 2, 4096 ** 2, 4096 ** 2, 4096, 4096 * 11008, 4096 * 11008,
                          11008 * 4096]
    assert W.bucket_elems(25 * W.MiB, 2) == 13_107_200


def test_bucket_gradients_draw_tensors_in_registration_order():
    numels = [5, 300, 1, 70]
    g = W.bucket_gradients_bf16(3, numels, std=1e-3, seed_base=11)
    for r in range(3):
        gen = _pcg(11 + r)
        for t, n in enumerate(numels):
            x = gen.standard_normal(n, dtype=np.float32) * np.float32(1e-3)
            np.testing.assert_array_equal(g[r][t], W.to_bf16_bits(x))


def test_zipf_routing_is_seeded_and_skewed():
    c = W.zipf_expert_counts(8, 4096, 64, 1.2, 1000)
    np.testing.assert_array_equal(c, W.zipf_expert_counts(8, 4096, 64, 1.2, 1000))
    assert (c.sum(axis=1) == 4096).all()
    recv = c.sum(axis=0)
    assert recv[0] == recv.max() and recv[0] > 2 * recv.mean()  # the hot receiver holds experts 0..7

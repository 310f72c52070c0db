"""The seeded input generator: determinism, independence of streams, moments."""
import numpy as np

import datagen


def _splitmix64(z):
    m = (1 << 64) - 1
    z = (z + 0x9E3779B97F4A7C15) & m
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & m
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & m
    return z ^ (z >> 31)


def test_counter_hash_is_splitmix64_of_the_stated_key():
    # published splitmix64 finaliser; key(seed, tag) = sm(seed ^ sm(tag + 1))
    m = (1 << 64) - 1
    for seed, tag, i in [(0, 0, 0), (0, 4, 12345), (7, 3, 2 ** 40 + 3)]:
        key = _splitmix64(seed ^ _splitmix64(tag + 1))
        assert datagen.raw_u64(seed, tag, i) == _splitmix64((key + i * 0x9E3779B97F4A7C15) & m)


def test_deterministic_and_offsettable():
    a = datagen.normal_bf16(0, 1, (1000,), 0.02)
    b = datagen.normal_bf16(0, 1, (1000,), 0.02)
    np.testing.assert_array_equal(a, b)
    c = datagen.normal_bf16(0, 1, (500,), 0.02, start=500)
    np.testing.assert_array_equal(a[500:], c)
    assert not np.array_equal(a, datagen.normal_bf16(0, 2, (1000,), 0.02))
    assert not np.array_equal(a, datagen.normal_bf16(1, 1, (1000,), 0.02))


def test_normal_moments():
    z = datagen.bf16_to_f32(datagen.normal_bf16(0, 9, (1 << 20,), 1.0)).astype(np.float64)
    assert abs(z.mean()) < 5e-3
    assert abs(z.std() - 1.0) < 5e-3
    assert abs((z ** 4).mean() / (z ** 2).mean() ** 2 - 3.0) < 0.05
    assert abs((z > 1.96).mean() - 0.025) < 2e-3


def test_partial_expert_draw_matches_full_draw():
    w = datagen.WORKLOADS["tiny"]
    g, u, d = datagen.expert_weights(w)
    gp, up, dp = datagen.expert_weights(w, experts=[3, 200])
    for full, part in ((g, gp), (u, up), (d, dp)):
        np.testing.assert_array_equal(full[[3, 200]], part[[3, 200]])
        assert not part[4].any()


def test_permutation_is_a_permutation():
    p = datagen.permutation(0, 5, 256)
    assert sorted(p.tolist()) == list(range(256))
    assert p.tolist() != list(range(256))


def test_bf16_rounding_helpers():
    v = np.array([1.0, 1.00390625, 1.005859375, -3.14159, 0.0], np.float32)
    b = datagen.f32_to_bf16(v)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: goes to the even mantissa (1.0)
    assert datagen.bf16_to_f32(b).tolist()[:3] == [1.0, 1.0, 1.0078125]
    assert datagen.bf16_to_f32(b)[4] == 0.0

"""Pins of the randomized Walsh-Hadamard rotation (trefon.com "Matematyka cache
KV", section "Jak 4-bitowemu cache to uchodzi: najpierw obrot": sign flip,
transform, sign flip; orthonormal; dot products survive the rotation)."""

import numpy as np
import pytest

from oracle import kvq_oracle as O


def test_sylvester_orthogonality_exact():
    H = O.sylvester(128)
    assert np.array_equal(H @ H.T, 128 * np.eye(128, dtype=np.int64))
    assert np.array_equal(H, H.T)
    # Sylvester recursion: H_2n = [[H, H], [H, -H]]
    h64 = O.sylvester(64)
    assert np.array_equal(H, np.block([[h64, h64], [h64, -h64]]))


def test_butterfly_equals_matrix_on_integers():
    rng = np.random.default_rng(0)
    x = rng.integers(-1000, 1000, (20, 128)).astype(np.float32)
    y = O.fwht_f32(x)
    assert np.array_equal(y.astype(np.int64), x.astype(np.int64) @ O.sylvester(128).T)


def test_butterfly_close_to_matrix_on_reals():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((50, 128)).astype(np.float32)
    y = O.fwht_f32(x).astype(np.float64)
    ref = x.astype(np.float64) @ O.sylvester(128).T.astype(np.float64)
    assert np.max(np.abs(y - ref)) < 1e-4


def test_scale_constant_bits():
    assert int(np.asarray(O.HADAMARD_SCALE_F32).view(np.uint32)) == 0x3DB504F3


def test_splitmix64_published_value():
    # SplitMix64 seeded with 0: first output 0xE220A8397B1DCDAF.
    assert O.splitmix64_stream(0, 1)[0] == 0xE220A8397B1DCDAF


def test_seed_zero_is_plain_sylvester():
    d1, d2 = O.hadamard_signs(0)
    assert np.all(d1 == 1) and np.all(d2 == 1)
    x = np.random.default_rng(2).standard_normal((3, 128))
    assert np.allclose(O.rotate_f64(x, d1, d2), x @ O.sylvester(128).T / np.sqrt(128), atol=1e-13)


def test_seeded_signs_are_pm1_and_differ():
    d1, d2 = O.hadamard_signs(12345)
    for d in (d1, d2):
        assert set(np.unique(d)) == {-1.0, 1.0}
        assert 30 < np.sum(d < 0) < 98
    assert not np.array_equal(d1, d2)
    assert not np.array_equal(d1, O.hadamard_signs(12346)[0])


@pytest.mark.parametrize("seed", [0, 7, 2 ** 63 + 5])
def test_rotation_orthonormal_and_invertible(seed):
    d1, d2 = O.hadamard_signs(seed)
    R = O.rotation_matrix_f64(d1, d2)
    assert np.max(np.abs(R @ R.T - np.eye(128))) < 1e-14
    rng = np.random.default_rng(3)
    x = rng.standard_normal((4, 256))
    y = O.rotate_f64(x, d1, d2)
    assert np.allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-13)
    assert np.allclose(O.unrotate_f64(y, d1, d2), x, atol=1e-13)


@pytest.mark.parametrize("seed", [0, 99])
def test_dot_products_survive(seed):
    """q.k = (Rq).(Rk), per 128-chunk and over the whole head vector."""
    d1, d2 = O.hadamard_signs(seed)
    rng = np.random.default_rng(4)
    q, k = rng.standard_normal((2, 10, 256))
    lhs = np.sum(O.rotate_f64(q, d1, d2) * O.rotate_f64(k, d1, d2), axis=-1)
    assert np.allclose(lhs, np.sum(q * k, axis=-1), atol=1e-12)


def test_fp32_path_matches_fp64_path():
    d1, d2 = O.hadamard_signs(5)
    x = np.random.default_rng(6).standard_normal((30, 128)).astype(np.float32)
    y32 = O.rotate_f32(x, d1, d2)
    y64 = O.rotate_f64(x.astype(np.float64), d1, d2)
    assert np.max(np.abs(y32 - y64)) < 2e-6


def test_outlier_energy_is_spread():
    """A single outlier coordinate spreads to magnitude |x|/sqrt(128) on every
    coordinate, so one block scale no longer stretches to it."""
    d1, d2 = O.hadamard_signs(11)
    x = np.zeros(128)
    x[37] = 100.0
    y = O.rotate_f64(x, d1, d2)
    assert np.allclose(np.abs(y), 100.0 / np.sqrt(128), rtol=1e-13)

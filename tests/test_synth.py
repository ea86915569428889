"""Pins of the seeded input generator (shared by the CUDA path and the oracle)."""
import numpy as np

from rank_weight_reconstruction_gb300 import synth


def test_splitmix64_reference_vector():
    # First five outputs of splitmix64 started at state 1234567, the test vector
    # published with the generator's reference C implementation.
    want = [6457827717110365317, 3203168211198807973, 9817491932198370423,
            4593380528125082431, 16408922859458223821]
    assert [int(v) for v in synth.splitmix64(1234567, np.arange(5))] == want


def test_counter_based_and_chunk_independent():
    st = synth.stream_seed("t", 1)
    a = synth.normal_f64(st, 10_000_000)
    b = synth.normal_f64(st, 1000)
    assert np.array_equal(a[:1000], b)
    assert synth.stream_seed("t", 1) != synth.stream_seed("t", 2)


def test_distribution_moments():
    n = 2_000_000
    v = synth.normal_f64(synth.stream_seed("m"), n, sigma=0.02)
    assert abs(v.mean()) < 5 * 0.02 / np.sqrt(n)
    assert abs(v.std() / 0.02 - 1) < 5 / np.sqrt(2 * n)
    u = synth.uniform_f64(synth.stream_seed("u"), n, 0.9, 1.1)
    assert u.min() >= 0.9 and u.max() < 1.1 and abs(u.mean() - 1.0) < 1e-3


def test_theta_layout_and_padding():
    th = synth.make_theta(("x",), 10, 12, 4)
    assert th.W0.shape == (10, 16) and th.U.shape == (10, 8) and th.V.shape == (12, 8)
    assert not th.W0[:, 12:].any() and not th.U[:, 4:].any() and not th.V[:, 4:].any()
    W0, s, U, V = th.f64()
    assert W0.shape == (10, 12) and U.shape == (10, 4) and V.shape == (12, 4)
    assert np.all((s >= 0.89) & (s <= 1.11))
    # values are exactly bf16
    assert np.array_equal(synth.bf16_bits_from_f64(W0), th.W0[:, :12])


def test_small_int_theta_ranges():
    th = synth.small_int_theta(("i",), 9, 17, 3)
    W0, s, U, V = th.f64()
    for a in (W0, U, V):
        assert np.all(a == np.round(a)) and np.abs(a).max() <= 3
    assert set(np.unique(s)) <= {0.5, 1.0, 2.0}


def test_row_scaled_x():
    x = synth.bf16_bits_to_f64(synth.make_x(("rs",), 64, 256, row_scale=(0.5, 2.0)))
    norms = np.linalg.norm(x, axis=1) / 16.0
    assert norms.min() > 0.4 and norms.max() < 2.3 and norms.max() / norms.min() > 2

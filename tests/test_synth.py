"""The seeded input generator: deterministic, sliceable, the stated distributions."""
import numpy as np

import synth


def test_slices_equal_whole():
    whole = synth.normal_bf16(1000, synth.S_X, seed=3)
    part = synth.normal_bf16(301, synth.S_X, offset=457, seed=3)
    assert np.array_equal(whole[457:758], part)


def test_streams_and_seeds_differ():
    a = synth.normal_bf16(64, 1)
    assert not np.array_equal(a, synth.normal_bf16(64, 2))
    assert not np.array_equal(a, synth.normal_bf16(64, 1, seed=1))


def test_normal_moments():
    x = synth.bf16_to_f32(synth.normal_bf16(1 << 20, 9, std=0.5)).astype(np.float64)
    assert abs(x.mean()) < 3e-3 and abs(x.std() - 0.5) < 3e-3


def test_bf16_rounding_matches_generator():
    f = synth.normal_f32(4096, 11)
    assert np.array_equal(synth.f32_to_bf16(f), synth.normal_bf16(4096, 11))


def test_integer_values():
    v = synth.bf16_to_f32(synth.int_bf16(5000, 4, -2, 2))
    assert set(np.unique(v).tolist()) == {-2.0, -1.0, 0.0, 1.0, 2.0}


def test_expert_slices():
    wl = synth.scaled(synth.WORKLOADS["tiny"], E=5)
    full = synth.make_w_down(wl)
    sub = synth.make_w_down(wl, experts=[3, 1])
    assert np.array_equal(full[3], sub[0]) and np.array_equal(full[1], sub[1])
    rows = synth.make_x(wl, rows=np.array([7, 2]))
    assert np.array_equal(synth.make_x(wl)[[7, 2]], rows)

"""The seeded input generator: deterministic, chunk-parallel, correct distribution, RNE rounding."""
import numpy as np

from backward_split_linear_gb300 import synth


def test_deterministic_and_seed_dependent():
    a = synth.stage_inputs("transformer", 2, 256, 512, 4, 2, 64, tokens=33, n_mb=2, seed=0)
    b = synth.stage_inputs("transformer", 2, 256, 512, 4, 2, 64, tokens=33, n_mb=2, seed=0)
    c = synth.stage_inputs("transformer", 2, 256, 512, 4, 2, 64, tokens=33, n_mb=2, seed=1)
    for la, lb, lc in zip(a["params"], b["params"], c["params"]):
        for k in la:
            assert np.array_equal(la[k], lb[k])
            assert not np.array_equal(la[k], lc[k])
    assert all(np.array_equal(x, y) for x, y in zip(a["x"], b["x"]))
    assert not np.array_equal(a["x"][0], a["x"][1])


def test_chunks_are_independent_of_threads():
    big = synth.normal(3, 7, (3 * synth.CHUNK + 5,))
    # chunk j is the same draw whatever else is generated
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence(3, spawn_key=(7, 2))))
    ref = g.standard_normal(synth.CHUNK, dtype=np.float32)
    assert np.array_equal(big[2 * synth.CHUNK: 3 * synth.CHUNK], ref)


def test_distribution():
    w = synth.bf16_to_f64(synth.bf16_bits(synth.normal(0, 0, (1 << 20,), synth.WEIGHT_STD)))
    assert abs(w.mean()) < 1e-4 and abs(w.std() - 0.02) < 2e-4


def test_round_to_nearest_even():
    a = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8), 3.0e38, 1e-40], dtype=np.float32)
    got = synth.bf16_to_f64(synth.bf16_bits(a))
    # ties go to the even mantissa: 1 + 2^-8 -> 1, 1 + 3 * 2^-8 -> 1 + 2^-6
    assert got[0] == 1.0 and got[1] == 1.0 and got[2] == 1.0 + 2 ** -6 and got[3] == -1.0
    assert np.isfinite(got[4]) and got[5] >= 0

"""The seeded input generator: determinism, thread independence, distributions, rounding."""
import math

import numpy as np

import synth


def test_splitmix64_reference_values():
    """SplitMix64 seeded with 0 gives the published first outputs; the counter form reproduces them."""
    # first three outputs of SplitMix64(seed=0) (Steele, Lea & Flood 2014; the standard test vector)
    expected = [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]
    gamma = 0x9E3779B97F4A7C15
    def mix(z):
        z &= (1 << 64) - 1
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & ((1 << 64) - 1)
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & ((1 << 64) - 1)
        return z ^ (z >> 31)
    assert [mix((i + 1) * gamma) for i in range(3)] == expected
    # counter form: stream key = mix(seed + (stream + 1) * gamma), draw i = mix(key + (i + 1) * gamma)
    key = mix(7 + 1 * gamma)  # seed 7, stream 0
    for i in range(5):
        assert synth.draw(7, 0, i) == mix(key + (i + 1) * gamma)


def test_thread_count_does_not_change_values():
    a = synth.normal(3, 5, (1000, 7), threads=1)
    b = synth.normal(3, 5, (1000, 7), threads=7)
    assert np.array_equal(a, b)
    a = synth.unit_rows(3, 5, (333, 2, 16), synth.BF16, threads=1)
    b = synth.unit_rows(3, 5, (333, 2, 16), synth.BF16, threads=5)
    assert np.array_equal(a, b)


def test_distributions():
    x = synth.normal(1, 1, (200000,), dtype=synth.F64)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1) < 0.01
    u = synth.uniform(1, 2, 100000)
    assert u.min() > 0 and u.max() < 1 and abs(u.mean() - 0.5) < 0.01
    g = synth.log_decay(1, 3, (100000,), -2.0, 1.0)
    assert g.max() < 0 and g.min() >= -5.0
    ref = -np.log1p(np.exp(-2.0 + synth.normal(1, 3, (100000,), dtype=synth.F64)))
    np.testing.assert_allclose(g, ref.astype(np.float32), rtol=1e-6)
    b = synth.sigmoid_normal(1, 4, (100000,))
    assert 0 < b.min() and b.max() < 1 and abs(b.mean() - 0.5) < 0.01


def test_unit_rows_and_bf16_rounding():
    x = synth.unit_rows(9, 1, (100, 3, 128), synth.F64)
    np.testing.assert_allclose(np.linalg.norm(x, axis=-1), 1.0, rtol=1e-14)
    bf = synth.unit_rows(9, 1, (100, 3, 128), synth.BF16)
    assert np.array_equal(bf, synth.f32_to_bf16(x.astype(np.float32)))
    # round-to-nearest-even on exact ties
    t = np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -1.0 - 2 ** -8], np.float32)
    assert list(synth.bf16_to_f32(synth.f32_to_bf16(t))) == [1.0, 1.0 + 2 ** -6, -1.0]


def test_workloads_shapes():
    p = synth.tiny()
    assert p.q.shape == (64, 2, 16) and p.q.dtype == np.float32 and p.init_zero
    v = synth.varlen(n_seqs=4, lo=100, hi=300, H=2, d=16, num_slots=8, num_extra=8)
    assert v.N == 4 and len(set(v.slot_ids.tolist())) == 4
    assert len(set(v.extra_slot_ids.ravel().tolist())) == 8
    assert np.all(v.lengths >= 100) and np.all(v.lengths <= 300)
    dv = synth.decode_verify(B=64, W=8, H=2, d=16, num_slots=128)
    assert dv.wq.shape == (64, 8, 2, 16) and dv.accepted.min() >= 0 and dv.accepted.max() <= 8
    assert len(set(dv.slot_ids.tolist())) == 64


def test_poisson_clipped_mean():
    a = synth.poisson_clipped(4, synth.S_ACCEPT, 20000, 2.7, 8)
    # E[min(Poisson(2.7), 8)] computed from the pmf
    pmf = [math.exp(-2.7) * 2.7 ** k / math.factorial(k) for k in range(8)]
    mean = sum(k * p for k, p in enumerate(pmf)) + 8 * (1 - sum(pmf))
    assert abs(a.mean() - mean) < 0.05

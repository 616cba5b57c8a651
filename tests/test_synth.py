"""The seeded input generator against its published definitions (SplitMix64, Box-Muller, bf16
round-to-nearest-even), its moments, and the stand-in drafter of the speculative rounds."""
import numpy as np

import synth

M64 = (1 << 64) - 1


def sm64(x):
    """SplitMix64's output for state x (Steele, Lea and Flood 2014; Vigna's finaliser)."""
    z = (x + 0x9E3779B97F4A7C15) & M64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M64
    return z ^ (z >> 31)


def test_splitmix64_reference_outputs():
    # the first three outputs of SplitMix64 started from state 0, as published with the generator
    assert [sm64(0), sm64(0x9E3779B97F4A7C15), sm64(2 * 0x9E3779B97F4A7C15 & M64)] == \
        [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_words_are_the_counter_generator():
    for seed, t in [(0, 0), (7, synth.tid("layer3.w_in")), (2 ** 40 + 3, 12345)]:
        key = sm64(seed ^ sm64(t ^ 0xA5A5A5A5A5A5A5A5))
        assert synth.words(seed, t, 5).tolist() == [sm64((key + i) & M64) for i in range(5)]


def test_normals_are_box_muller_of_the_words():
    seed, t, n = 3, synth.tid("gdn.q"), 64
    w = synth.words(seed, t, 2 * n).tolist()
    u1 = np.array([((x >> 11) + 1.0) / 2.0 ** 53 for x in w[0::2]])
    u2 = np.array([(x >> 11) / 2.0 ** 53 for x in w[1::2]])
    ref = np.sqrt(-2.0 * np.log(u1)) * np.cos(2 * np.pi * u2)
    np.testing.assert_allclose(synth.normal_f64(seed, t, n), ref, rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(synth.normal_f64(seed, t, n, sigma=0.02, mean=1.0), 1.0 + 0.02 * ref, rtol=1e-14)


def test_bf16_is_round_to_nearest_even_of_the_float_sample():
    seed, t, n = 4, synth.tid("w"), 1 << 16
    f = synth.normal_f64(seed, t, n, sigma=0.02).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    ref = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)   # no NaN or infinity here
    assert np.array_equal(synth.normal_bf16(seed, t, n, sigma=0.02), ref)


def test_moments_and_independence():
    n = 1 << 20
    x = synth.normal_f64(11, synth.tid("moments"), n)
    assert abs(x.mean()) < 5 / np.sqrt(n)
    assert abs(x.std() - 1.0) < 0.005
    assert abs(np.mean(np.abs(x) < 1.0) - 0.682689) < 0.003
    y = synth.normal_f64(11, synth.tid("moments2"), n)
    assert abs(np.corrcoef(x, y)[0, 1]) < 5 / np.sqrt(n)
    assert np.array_equal(x, synth.normal_f64(11, synth.tid("moments"), n))   # a pure function


def test_uniform_integers_cover_their_range():
    v = synth.uniform_i32(5, synth.tid("ids"), 200000, 3, 103)
    assert v.min() == 3 and v.max() == 102
    counts = np.bincount(v - 3, minlength=100)
    assert counts.min() > 1700 and counts.max() < 2300


def test_replay_drafter_acceptance():
    from bit_exact_speculative_gb300.speculative import ReplayDrafter
    ref = list(range(1000, 2000))
    assert ReplayDrafter(ref, 5000, 1.0).propose(10, 8) == ref[11:19]
    d0 = ReplayDrafter(ref, 5000, 0.0, seed=1)
    assert all(a != b for a, b in zip(d0.propose(10, 200), ref[11:211]))
    d = ReplayDrafter(ref, 5000, 0.6, seed=2)
    hits = sum(a == b for a, b in zip(d.propose(0, 900), ref[1:901]))
    assert 0.55 < hits / 900 < 0.65

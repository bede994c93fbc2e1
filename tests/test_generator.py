"""The seeded generator: determinism, distributions, and agreement of its Q4
quantiser with the oracle's independently written one."""
import numpy as np

import gen
from gen import configs, synth
from oracle import oracle as orc

M64 = (1 << 64) - 1


def _splitmix_outputs(seed_state, n):
    """SplitMix64 as published (Steele et al. 2014): state += golden gamma,
    then the variant-13 finaliser."""
    out, s = [], seed_state
    for _ in range(n):
        s = (s + 0x9E3779B97F4A7C15) & M64
        z = s
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M64
        out.append(z ^ (z >> 31))
    return out


def test_draws_are_splitmix64_stream():
    seed, tid = 7, 123
    base = _splitmix_outputs(((seed << 32) + tid) & M64, 1)[0]
    want = _splitmix_outputs(base, 5)
    got = [int(v) for v in gen.raw_draws(seed, tid, 5)]
    assert got == want


def test_determinism_and_thread_independence():
    a = gen.q4_matrix(3, 11, 64, 512, 0.02, nthreads=1)
    b = gen.q4_matrix(3, 11, 64, 512, 0.02, nthreads=5)
    assert np.array_equal(a, b)
    c = gen.q4_matrix(4, 11, 64, 512, 0.02, nthreads=1)
    assert not np.array_equal(a, c)


def test_normal_moments():
    """Box-Muller deviates: mean 0, variance 1, the normal's kurtosis 3 (a
    four-term Irwin-Hall sum would give 2.7 and never pass 3.47), tails past
    4 sigma at about the normal rate, and the normal CDF at a few points."""
    z = gen.normal_f64(0, 9, 400000)
    assert abs(z.mean()) < 0.01
    assert abs(z.std() - 1.0) < 0.01
    k = np.mean(z ** 4)
    assert abs(k - 3.0) < 0.05
    assert np.abs(z).max() > 4.0
    tail = np.mean(np.abs(z) > 3.0)  # 2 * (1 - Phi(3)) = 0.0026998
    assert abs(tail - 0.0026998) < 0.0006
    for x, phi in ((-1.0, 0.1586553), (0.5, 0.6914625), (2.0, 0.9772499)):
        assert abs(np.mean(z <= x) - phi) < 0.003


def test_normal_deviates_are_box_muller_of_the_draws():
    """Each deviate is sqrt(-2 ln u1) cos(2 pi u2) of its own 64-bit draw
    (u1, u2 from the high and low 32-bit halves), to within the error of the
    generator's own ln/cos series."""
    n = 2000
    raw = gen.raw_draws(4, 21, n)
    z = gen.normal_f64(4, 21, n)
    hi = (raw >> np.uint64(32)).astype(np.float64)
    lo = (raw & np.uint64(0xFFFFFFFF)).astype(np.float64)
    u1, u2 = (hi + 0.5) / 2.0 ** 32, (lo + 0.5) / 2.0 ** 32
    want = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
    assert np.max(np.abs(z - want)) < 1e-12


def test_generator_q4_equals_oracle_quantiser():
    rows, k = 48, 1024
    raw = gen.normal_f64(5, 42, rows * k, sigma=0.02)
    blocks = gen.q4_matrix(5, 42, rows, k, 0.02, nthreads=2).reshape(-1, 144)
    again = orc.q4_encode(raw)
    assert np.array_equal(blocks, again)


def test_tokens_and_permutation():
    t = gen.uniform_tokens(1, 2, 10000, 2048)
    assert t.min() >= 0 and t.max() < 2048
    assert len(np.unique(t)) > 1900
    p = gen.permutation(3, 70000, 8448)
    assert sorted(p.tolist()) == list(range(8448))
    assert not np.array_equal(p, np.arange(8448))


def test_q8_blocks_range():
    c, s = synth.q8_blocks(1, 50003, (8, 256))
    assert c.min() >= -127 and c.max() <= 127
    vals = np.array([orc.half_value(int(x)) for x in s.ravel()])
    assert np.all(vals > 2.0 / 127 * 0.99) and np.all(vals < 4.0 / 127 * 1.01)


def test_inventory_sizes():
    m = configs.QWEN27
    inv = configs.tensor_inventory(m)
    q4_weights = sum(r * k for _, _, kind, (r, k) in
                     [(n, i, kd, sh) for n, i, kd, sh in inv if kd == "q4"] if True)
    # streamed per step: everything but the embedding (gathered, not streamed)
    streamed = q4_weights - m["vocab"] * m["hidden"]
    assert abs(streamed / 1e9 - 25.62) < 0.05
    assert abs(streamed * 0.5625 / 1e9 - 14.41) < 0.03

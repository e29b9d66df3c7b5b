"""The seeded input generator (no GPU): stream definition, distributions,
quantisation, and the workload shapes."""
import numpy as np

import workloads as W


def _sequential_splitmix64(seed, n):
    """The published stateful form: x += gamma; z = mix(x)."""
    x, out = seed, []
    for _ in range(n):
        x = (x + 0x9E3779B97F4A7C15) & (2 ** 64 - 1)
        z = x
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & (2 ** 64 - 1)
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & (2 ** 64 - 1)
        out.append(z ^ (z >> 31))
    return out


def test_splitmix64_known_vector():
    # First outputs for seed 1234567 of the reference splitmix64.c.
    want = [6457827717110365317, 3203168211198807973, 9817491932198370423,
            4593380528125082431, 16408922859458223821]
    got = [int(v) for v in W.splitmix64(1234567, np.arange(5, dtype=np.uint64))]
    assert got == want
    assert _sequential_splitmix64(1234567, 5) == want


def test_counter_form_equals_sequential():
    for seed in (0, 1, 3, 2 ** 63 + 5):
        got = [int(v) for v in W.splitmix64(seed, np.arange(100, dtype=np.uint64))]
        assert got == _sequential_splitmix64(seed, 100)


def test_uniform_is_exact_binary32_in_range():
    x = W._uniform_f32(0, np.arange(1 << 16, dtype=np.uint64))
    assert x.dtype == np.float32
    assert x.min() >= -1.0 and x.max() < 1.0
    assert np.all((x.astype(np.float64) + 1) * 2 ** 23 == np.round((x.astype(np.float64) + 1) * 2 ** 23))
    assert abs(float(x.mean())) < 0.01


def test_normal_moments():
    x = W._normal_f32(1, np.arange(1 << 18, dtype=np.uint64), 4.0).astype(np.float64)
    assert abs(x.mean()) < 0.05
    assert abs(x.var() - 16.0) < 0.3


def test_quantise_e4m3fn_saturates():
    x = np.array([1000.0, -1000.0, 448.0, 463.9, 0.0], np.float32)
    assert list(W.quantise(x, "e4m3fn")) == [0x7E, 0xFE, 0x7E, 0x7E, 0x00]


def test_rank_input_blocks_and_samples_agree():
    count = (1 << 22) + 37
    full = W.rank_input("normal", 2, "fp16", count, rank=1)
    idx = np.array([0, 1, 12345, (1 << 22) - 1, 1 << 22, count - 1])
    s = W.sample_inputs("normal", 2, "fp16", count, 2, idx)
    assert np.array_equal(s[1], full[idx])
    assert np.array_equal(W.rank_input("normal", 2, "fp16", 100, rank=1),
                          W.draw("normal", 2, np.arange(100, 200, dtype=np.uint64), "fp16"))


def test_workload_shapes():
    assert (W.C1.nranks, W.C1.dtype, W.C1.bytes_per_rank) == (2, "bf16", 1 << 20)
    assert (W.C2.nranks, W.C2.dtype, W.C2.bytes_per_rank) == (8, "fp16", 64 << 20)
    assert [w.bytes_per_rank for w in W.C3] == [16 << 10 << (2 * k) for k in range(8)]
    assert (W.C4.nranks, W.C4.dtype, W.C4.bytes_per_rank, W.C4.sigma) == (8, "e4m3fn", 16 << 20, 4.0)
    assert sorted({w.dtype for w in W.C5}) == ["bf16", "fp32"]
    assert sorted({w.bytes_per_rank for w in W.C5}) == [1 << 10 << (2 * k) for k in range(6)]
    assert W.C2.algo_bytes == 2 * 8 * (64 << 20)

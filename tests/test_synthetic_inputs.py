"""The seeded input generators (CPU only)."""
import numpy as np
import torch

import synthetic_inputs as si


def test_splitmix64_reference_values():
    # SplitMix64 from state 0 (increment then finalise): the generator's
    # published first outputs, 0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4.
    with np.errstate(over="ignore"):
        states = np.array([si.GAMMA, np.uint64(2) * si.GAMMA], dtype=np.uint64)
    out = si._mix(states)
    assert int(out[0]) == 0xE220A8397B1DCDAF
    assert int(out[1]) == 0x6E789E6AA1B965F4


def test_deterministic_and_counter_based():
    a = si.draws(5, 3, 100)
    assert np.array_equal(a, si.draws(5, 3, 100))
    assert np.array_equal(a[40:], si.draws(5, 3, 60, start=40))
    assert not np.array_equal(a, si.draws(5, 4, 100))
    assert not np.array_equal(a, si.draws(6, 3, 100))


def test_uniform_range_and_moments():
    u = si.uniform_pm1(0, 1, (200000,))
    assert u.dtype == np.float32
    assert u.min() >= -1.0 and u.max() < 1.0
    assert abs(u.mean()) < 0.01 and abs(u.var() - 1 / 3) < 0.01
    # 24-bit grid: every value is k * 2^-23 - 1
    k = (u.astype(np.float64) + 1.0) * 2.0 ** 23
    assert np.array_equal(k, np.round(k))


def test_normal_moments():
    z = si.normal(0, 2, (200000,), 0.0, 0.02)
    assert abs(z.mean()) < 2e-4 and abs(z.std() - 0.02) < 4e-4


def test_bf16_rounding_matches_torch():
    x = np.concatenate([si.normal(1, 1, (50000,)), si.uniform_pm1(1, 2, (50000,)) * 1e3,
                        np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -0.0, 65504.0], np.float32)])
    ours = si.to_bf16_bits(x)
    theirs = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, theirs)
    assert np.array_equal(si.bf16_bits_to_f32(ours), torch.from_numpy(ours.view(np.int16)).view(torch.bfloat16).float().numpy())


def test_workload_shapes():
    assert si.SKINNY_16x4096.algorithmic_bytes() == 2 * (16 * 4096 + 4096 * 4096) + 2 * 16 * 4096 + 4 * 4096
    X, W, b = si.make_inputs(si.Layer("t", 3, 5, 8, si.PREC_BF16, bias=True))
    assert X.shape == (3, 8) and W.shape == (5, 8) and b.shape == (5,)
    assert np.array_equal(si.round_bf16(X), X)


def test_block_generation_equals_plain_definition(monkeypatch):
    """Generation in reused blocks gives the same bits as the definition written
    out on whole arrays, across block boundaries."""
    import math

    monkeypatch.setattr(si, "CHUNK", 1000)

    def plain_draws(seed, tid, count):
        base = si.stream_base(seed, tid)
        idx = np.arange(1, count + 1, dtype=np.uint64)
        with np.errstate(over="ignore"):
            return si._mix(base + idx * si.GAMMA)

    for n in (1, 999, 1000, 2501):
        assert np.array_equal(si.draws(3, 4, n), plain_draws(3, 4, n))
        u = (plain_draws(3, 4, n) >> np.uint64(40)).astype(np.float64)
        assert np.array_equal(si.uniform_pm1(3, 4, (n,)), (u * 2.0 ** -23 - 1.0).astype(np.float32))
        d = plain_draws(5, 6, 2 * n)
        u1 = ((d[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0 ** -53
        u2 = (d[1::2] >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
        z = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)
        assert np.array_equal(si.normal(5, 6, (n,), 0.1, 0.02), (0.1 + 0.02 * z).astype(np.float32))
        x = si.normal(7, 8, (n,))
        b = x.view(np.uint32).astype(np.uint64)
        plain_bits = ((b + ((b >> 16) & 1) + 0x7FFF) >> 16).astype(np.uint16)
        assert np.array_equal(si.to_bf16_bits(x), plain_bits)


def test_qkv_recipe():
    """The attention input: (B*T) x 3C values drawn N(0, 1) from stream 4 and
    rounded to bf16, the same for every call with the same seed."""
    att = si.Attention("t", 2, 7, 3, 64, causal=True, seed=5)
    a = si.make_qkv(att)
    assert a.shape == (14, 3 * 192) and a.dtype == np.float32
    assert np.array_equal(a, si.make_qkv(att))
    assert np.array_equal(a, si.round_bf16(si.normal(5, 4, (14, 3 * 192), 0.0, 1.0)))
    big = si.make_qkv(si.GPT2_ATTN_B64)
    assert big.shape == (64 * 128, 3 * 768)
    assert abs(float(big.mean())) < 0.01 and abs(float(big.std()) - 1.0) < 0.01

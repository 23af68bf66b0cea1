"""The shared seeded generator (harness/gen.py) against its stated
definition: the 32-bit finaliser, the stream key, the Irwin-Hall draw and
its fp32 scale, round-to-nearest-even to bf16, slices that match longer
draws, and the distribution the docstring promises.  The restatement below
uses plain Python integers, not the module's torch code."""
import math
import struct

import numpy as np
import pytest
import torch

from harness import gen

M = 0xFFFFFFFF


def mix32_int(x: int) -> int:
    x ^= x >> 16
    x = (x * 0x45D9F3B) & M
    x ^= x >> 16
    x = (x * 0x45D9F3B) & M
    x ^= x >> 16
    return x


def f32(v: float) -> float:
    return struct.unpack("<f", struct.pack("<f", v))[0]


def normal_int(seed: int, stream: int, n: int, sigma: float) -> float:
    key = mix32_int(mix32_int(seed & M) ^ (stream & M))
    w0 = mix32_int((key + 2 * n) & M)
    w1 = mix32_int((key + 2 * n + 1) & M)
    c = (w0 & 0xFFFF) + (w0 >> 16) + (w1 & 0xFFFF) + (w1 >> 16) - 2 * 65535
    scale = f32(sigma * math.sqrt(3.0) / 65536.0)
    return f32(float(c) * scale)  # c is exact in fp32 (|c| < 2^17); one IEEE multiply


def bf16_rne_bits(v: np.ndarray) -> np.ndarray:
    b = v.astype(np.float32).view(np.uint32).astype(np.uint64)
    return ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)


@pytest.mark.parametrize("x", [0, 1, 2, 0x7FFFFFFF, 0x80000000, 0xFFFFFFFF, 0x12345678, 0xDEADBEEF])
def test_mix32_is_the_stated_finaliser(x):
    assert int(gen.mix32(torch.tensor([x], dtype=torch.int64))[0]) == mix32_int(x)


def test_mix32_is_a_bijection_on_a_sample():
    xs = np.random.default_rng(0).integers(0, 2 ** 32, 200_000, dtype=np.uint64)
    ys = gen.mix32(torch.from_numpy(xs.astype(np.int64))).numpy()
    assert len(np.unique(xs)) == len(np.unique(ys))


@pytest.mark.parametrize("seed,stream,sigma", [(1, gen.stream_id(gen.KIND_X), 1.0),
                                               (2, gen.stream_id(gen.KIND_EXPERT, 3, 77), 0.02),
                                               (0xFFFFFFFF, 0, 0.5)])
def test_normal_draws_match_the_definition(seed, stream, sigma):
    got = gen.normal_f32(seed, stream, 64, sigma, start=1000).numpy()
    want = np.array([normal_int(seed, stream, 1000 + i, sigma) for i in range(64)], dtype=np.float32)
    assert np.array_equal(got, want)


def test_slices_equal_the_same_elements_of_a_longer_draw():
    full = gen.normal_f32(5, 9, 5000, 1.0).numpy()
    assert np.array_equal(gen.normal_f32(5, 9, 300, 1.0, start=2700).numpy(), full[2700:3000])
    assert np.array_equal(gen.uniform_words(5, 9, 10, start=40).numpy(), gen.uniform_words(5, 9, 50).numpy()[40:])


def test_bf16_draws_round_to_nearest_even():
    v = gen.normal_f32(3, 4, 100_000, 0.02)
    got = gen.normal_bf16(3, 4, 100_000, 0.02).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, bf16_rne_bits(v.numpy()))


def test_distribution_is_the_promised_one():
    sigma = 0.7
    v = gen.normal_f32(11, 12, 2_000_000, sigma).double().numpy()
    assert abs(v.mean()) < 0.002 * sigma
    assert abs(v.std() / sigma - 1.0) < 0.002
    assert np.abs(v).max() <= 2 * 65535 * f32(sigma * math.sqrt(3.0) / 65536.0) * (1 + 1e-6)  # about 3.46 sigma
    # Irwin-Hall(4) has excess kurtosis -1.2 / 4 = -0.3 (a normal has 0)
    k = ((v - v.mean()) ** 4).mean() / v.var() ** 2 - 3.0
    assert abs(k + 0.3) < 0.02


def test_streams_and_permutations():
    a = gen.normal_f32(1, gen.stream_id(gen.KIND_X, 0, 0), 1000, 1.0)
    b = gen.normal_f32(1, gen.stream_id(gen.KIND_X, 0, 1), 1000, 1.0)
    assert not torch.equal(a, b)
    p = gen.permutation(7, 3, 1000)
    assert np.array_equal(np.sort(p), np.arange(1000))
    assert np.array_equal(p, gen.permutation(7, 3, 1000))
    assert not np.array_equal(p, gen.permutation(7, 4, 1000))
    assert gen.stream_id(0x3, 0x12, 0x3456) == (0x3 << 24) | (0x12 << 16) | 0x3456


def test_budget_slots_follow_the_page_profile():
    # "Betelgeuse ... on an RTX 3060", "Arrival-Slack VRAM Slot Pool": 240 slots per layer on layers 0-4,
    # 92 in the middle, 60 at the tail, about 5,000 in all for 48 layers of 512 experts
    from harness import configs as C
    b = C.budget_slots(512, 48)
    assert b[:5] == (240,) * 5 and b[5:43] == (92,) * 38 and b[43:] == (60,) * 5
    assert abs(sum(b) - 5000) < 25
    s = C.budget_slots(288, 48)
    assert s[0] == 135 and s[20] == 52 and s[47] == 34
    assert [C.layer_S(C.STACK_BUDGET, l) for l in (0, 4, 5, 42, 43, 47)] == [135, 135, 52, 52, 34, 34]
    assert len(C.initial_residency(C.STACK_BUDGET, 47)) == 34

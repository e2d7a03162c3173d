"""The seeded input generator against its published definition (SplitMix64 + Box-Muller)."""
import math
import struct

import numpy as np

import workload

M64 = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15


def mix(z):
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & M64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & M64
    return z ^ (z >> 31)


def ref_key(seed, stream):
    return mix((mix(seed ^ 0x5851F42D4C957F2D) + stream * GAMMA) & M64)


def ref_draw(key, i):
    return mix((key + (i + 1) * GAMMA) & M64)


def ref_normal(seed, stream, i, std):
    k = ref_key(seed, stream)
    p = i // 2
    u1 = 1.0 - (ref_draw(k, 2 * p) >> 11) * 2.0 ** -53
    u2 = (ref_draw(k, 2 * p + 1) >> 11) * 2.0 ** -53
    r = math.sqrt(-2.0 * math.log(u1))
    z = r * math.cos(2 * math.pi * u2) if i % 2 == 0 else r * math.sin(2 * math.pi * u2)
    return struct.unpack("f", struct.pack("f", std * z))[0]


def test_splitmix_reference_vector():
    # SplitMix64 seeded with 1234567: first outputs of the published generator
    state = 1234567
    outs = []
    for _ in range(3):
        state = (state + GAMMA) & M64
        outs.append(mix(state))
    assert outs[0] == 6457827717110365317
    assert outs[1] == 3203168211198807973
    assert outs[2] == 9817491932198370423


def test_key_and_draw_match_definition():
    for seed, stream in ((0, 0), (1, 5), (2, 1 << 33), (123456789, 3 << 32)):
        k = workload.key(seed, stream)
        assert k == ref_key(seed, stream)
        for i in (0, 1, 2, 1000, 10 ** 9):
            assert workload.draw(k, i) == ref_draw(k, i)


def test_normal_matches_definition():
    a = workload.normal(3, 77, (50,), 0.02, "f32", first=1000)
    for e in range(50):
        assert abs(a[e] - ref_normal(3, 77, 1000 + e, 0.02)) <= 2e-9
    b = workload.normal(3, 77, (50,), 0.02, "bf16", first=1000)
    bf = workload.bf16_bits_to_f32(b)
    assert np.max(np.abs(bf - a)) <= np.max(np.abs(a)) * 2 ** -8


def test_normal_statistics_and_counter_property():
    a = workload.normal(5, 9, (200000,), 0.02, "f32")
    assert abs(a.mean()) < 3e-4 and abs(a.std() - 0.02) < 3e-4
    tail = workload.normal(5, 9, (100,), 0.02, "f32", first=150000)
    assert np.array_equal(tail, a[150000:150100])


def test_tokens_and_permutation():
    t = workload.tokens(1, 2, 1000, 50)
    assert t.min() >= 0 and t.max() < 50
    k = ref_key(1, 2)
    assert all(int(t[i]) == ref_draw(k, i) % 50 for i in range(20))
    p = workload.permutation(7, 8, 16)
    assert sorted(p.tolist()) == list(range(16))


def test_request_layout():
    spec = workload.WORKLOADS["llama8b-8k"]
    r = workload.make_request(spec, 3, 0.15)
    assert r.tokens.shape == (spec.n_tokens,)
    assert [c[1] for c in r.chunks] == [i * 512 for i in range(16)]
    assert all(c[0] == 0 and c[2] == 512 for c in r.chunks)

"""The seeded input generator: Philox4x32-10 known-answer vectors and the value recipes."""
import numpy as np

import inputgen as ig


def test_philox_known_answers():
    # Known-answer vectors published with the Random123 library for philox4x32-10
    # (Salmon et al., "Parallel Random Numbers: As Easy as 1, 2, 3", SC'11).
    assert ig.philox4x32_10([0, 0, 0, 0], [0, 0]) == (0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8)
    assert ig.philox4x32_10([0xFFFFFFFF] * 4, [0xFFFFFFFF] * 2) == \
        (0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD)
    assert ig.philox4x32_10([0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344],
                            [0xA4093822, 0x299F31D0]) == (0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1)


def test_streams_are_deterministic_and_offsettable():
    a = np.empty(1001, np.uint16)
    b = np.empty(1001, np.uint16)
    ig.fill_bf16(a, ig.normal(1.0), 0, 3, 1)
    ig.fill_bf16(b, ig.normal(1.0), 0, 3, 1)
    assert np.array_equal(a, b)
    c = np.empty(400, np.uint16)
    ig.fill_bf16(c, ig.normal(1.0), 0, 3, 1, first=333)
    assert np.array_equal(c, a[333:733])
    d = np.empty(1001, np.uint16)
    ig.fill_bf16(d, ig.normal(1.0), 0, 4, 1)      # another rank: another stream
    assert not np.array_equal(a, d)


def test_value_recipes():
    n = 1 << 20
    u = ig.bf16_bits_to_f32(ig.fill_bf16(np.empty(n, np.uint16), ig.UNIFORM_PM1, 0, 0, 0))
    assert u.min() >= -1.0 and u.max() <= 1.0
    assert abs(u.mean()) < 5e-3 and abs(u.var() - 1 / 3) < 5e-3
    z = ig.bf16_bits_to_f32(ig.fill_bf16(np.empty(n, np.uint16), ig.normal(1 / 512), 0, 0, 1))
    assert abs(z.mean()) < 1e-3 and abs(z.var() * 512 - 1) < 1e-2     # second parameter = variance
    k = ig.bf16_bits_to_f32(ig.fill_bf16(np.empty(n, np.uint16), ig.INTEGER_PM2, 0, 0, 0))
    assert set(np.unique(k).tolist()) == {-2.0, -1.0, 0.0, 1.0, 2.0}


def test_workload_table():
    w = ig.WORKLOADS["ar_mlp_down_p8_m8192_n8192_k3584"]
    assert (w.P, w.M, w.N, w.Kr) == (8, 8192, 8192, 3584) and w.flops == 2 * 8192 * 8192 * 28672
    assert ig.sweep_workload(256).M == 256
    A, B = ig.make_operands(ig.WORKLOADS["ar_p2_m128_n128_k256"])
    assert len(A) == 2 and A[0].shape == (128, 256) and B[1].shape == (256, 128)

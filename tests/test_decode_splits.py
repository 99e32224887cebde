"""The automatic key-range count of the split-KV decode (diffattn_decode_auto_splits).

Host arithmetic only: no GPU.  The chooser minimises a cost model of the split
kernel; these tests check it on recorded B300 timings and on the invariants
every count it returns must satisfy.

MEASURED holds graph-replayed latencies (us per call) of the decode at fixed
split counts, on one B300 (148 SMs), d = 64, dv = 128, with the caches rotated
over more than 2x the L2 so every call reads HBM.  They are timings, not
results of the computation, so they say nothing about parity: they are the
data the cost model was fitted to, kept so that a change to the model is
checked against them.
"""
import pytest

import transformer_attention_07_b300 as da
from transformer_attention_07_b300 import build as dabuild

SMS = 148

MEASURED = {
    (1, 32, 1024): {1: 15.84, 2: 12.43, 3: 12.09, 4: 10.73, 5: 14.93, 6: 15.59, 8: 14.87, 9: 15.27, 10: 15.65,
                    12: 18.88, 14: 19.57, 16: 22.48},
    (1, 32, 4096): {1: 42.69, 2: 26.02, 3: 21.47, 4: 18.5, 5: 27.2, 6: 25.62, 8: 22.89, 9: 23.64, 10: 28.67,
                    12: 26.85, 14: 27.71, 16: 31.6, 18: 32.38, 20: 34.58, 24: 35.56, 28: 39.93, 32: 43.38,
                    40: 50.47, 48: 58.37, 64: 76.49},
    (1, 8, 8192): {1: 77.15, 2: 43.27, 3: 32.37, 4: 25.65, 5: 23.07, 6: 21.56, 8: 18.59, 9: 18.64, 10: 18.87,
                   12: 17.95, 14: 18.42, 16: 18.1, 18: 19.91, 20: 24.64, 24: 25.03, 28: 26.47, 32: 26.76,
                   40: 33.36, 48: 36.72, 64: 44.08},
    (4, 32, 4096): {1: 47.11, 2: 51.14, 3: 56.38, 4: 58.22, 5: 62.23, 6: 64.98, 8: 65.57, 9: 68.13, 10: 73.33,
                    12: 76.75, 14: 81.78, 16: 89.36, 18: 89.22, 20: 97.33, 24: 103.58, 28: 114.98, 32: 129.29,
                    40: 135.71, 48: 163.9, 64: 213.61},
    (1, 32, 16384): {1: 149.07, 2: 79.46, 3: 57.51, 4: 48.11, 5: 73.19, 6: 65.45, 8: 53.83, 9: 54.18,
                     10: 66.46, 12: 60.06, 14: 69.78, 16: 65.8, 18: 64.85, 20: 70.8, 24: 77.53, 28: 76.04,
                     32: 79.84, 40: 90.69, 48: 101.86, 64: 119.02},
    (8, 32, 8192): {1: 165.6, 2: 178.8, 3: 187.17, 4: 173.78, 5: 179.6, 6: 189.37, 8: 194.44, 9: 197.55,
                    10: 207.56, 12: 206.0, 14: 216.09, 16: 237.43, 18: 239.46, 20: 252.86, 24: 261.66,
                    28: 280.98, 32: 321.18, 40: 336.6, 48: 364.71, 64: 463.0},
    (2, 8, 32768): {1: 289.95, 2: 150.05, 3: 104.16, 4: 79.6, 5: 66.76, 6: 58.76, 8: 49.43, 9: 50.33,
                    10: 76.31, 12: 67.11, 14: 63.39, 16: 58.22, 18: 59.95, 20: 71.55, 24: 67.25, 28: 74.69,
                    32: 75.13, 40: 83.95, 48: 93.93, 64: 99.42},
}


@pytest.fixture(scope="module")
def lib():
    dabuild.build()
    return da.load()


def pick(B, H, Nk, d=64, dv=128, sms=SMS, cap=0):
    return da.decode_auto_splits(B, H, Nk, d, dv, sms, cap)


@pytest.mark.parametrize("shape", sorted(MEASURED))
def test_pick_is_within_3_percent_of_the_fastest_measured_count(lib, shape):
    s = pick(*shape)
    times = MEASURED[shape]
    assert s in times, f"{shape}: picked {s}, not among the measured counts"
    assert times[s] <= 1.03 * min(times.values()), (shape, s, times[s], min(times.values()))


def test_every_pick_is_a_valid_key_range_split(lib):
    for B, H in ((1, 1), (1, 8), (1, 32), (2, 16), (4, 32), (8, 32), (32, 32), (1, 300), (64, 128)):
        for Nk in (1, 31, 32, 33, 255, 256, 257, 1000, 1024, 4096, 8191, 32768, 131072, 1 << 20):
            for cap in (0, 1, 5, 64):
                s = pick(B, H, Nk, cap=cap)
                assert 1 <= s <= (cap or 32)
                per = ((Nk + s - 1) // s + 31) // 32 * 32
                assert (s - 1) * per < Nk, "the last key range would be empty"
                assert s == 1 or per >= 256 or Nk < 512, (B, H, Nk, s)


def test_full_waves_of_heads_take_one_range(lib):
    # As many heads as SMs or more: every extra range only adds waves.
    assert pick(32, 32, 32768) == 1
    assert pick(4, 32, 4096) == 1
    assert pick(8, 32, 8192) == 1
    assert pick(1, 300, 16384, cap=26) <= 26


def test_few_heads_with_long_caches_spread_over_the_sms(lib):
    # 16 heads x 1M keys: 8 ranges = 128 CTAs, one wave.
    assert pick(1, 16, 1 << 20) == 8
    assert pick(1, 1, 1 << 20) == 32
    assert pick(1, 1, 1 << 20, cap=5) == 5


def test_invalid_arguments_return_zero(lib):
    assert pick(0, 1, 100) == 0
    assert pick(1, 0, 100) == 0
    assert pick(1, 1, 0) == 0
    assert pick(1, 1, 100, sms=0) == 0
    assert pick(1, 1, 100, cap=65) == 0
    assert pick(1, 1, 100, cap=-1) == 0
    assert pick(1, 1, 100, d=48) == 0
    assert pick(1, 1, 100, d=32, dv=64) == 1

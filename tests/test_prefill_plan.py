"""The prefill's launch plan (host arithmetic behind `diffattn_prefill_plan`,
the same function the launcher uses), pinned on the shapes of the workloads
and at the edges of each rule, for a 148-SM B300.

Every form computes the same bits (the GPU tests compare them); what these
tests fix is which form a shape gets:
  * persistent (one CTA per SM) when there are more query tiles than SMs and
    Nk <= 4096, or Nk <= 8192 when the tile list is weight-major;
  * the list is weight-major under causal masking when all heads' K and V
    (bf16: 4d + 2dv bytes per key; fp8 Q/K: 2d + 2dv) fit in 64 MiB,
    (b, h)-major otherwise;
  * otherwise one CTA per query tile: a 1-D grid over groups of heads under
    causal masking when at least four heads' K and V fit in 16 MiB, else the
    (tile, h, b) grid;
  * 1-D orders only below 2^30 tiles.
"""
import pytest

import transformer_attention_07_b300 as da

SMS = 148
MiB = 1 << 20


@pytest.mark.parametrize("name,B,H,Nq,Nk,causal,form,ctas", [
    # the workloads
    ("causal_2k", 4, 8, 2048, 2048, True, "persistent_weight", SMS),          # K/V 32 MiB
    ("cancel_8k", 2, 16, 8192, 8192, True, "tile_grouped", 2 * 16 * 64),     # K/V 128 MiB: groups of 4 heads
    ("long_64k", 1, 16, 65536, 65536, True, "tile_grid", 16 * 512),
    ("long_128k", 1, 8, 131072, 131072, True, "tile_grid", 8 * 1024),
    # the bench's other lengths
    ("2k_b8h16", 8, 16, 2048, 2048, True, "persistent", SMS),                # K/V 128 MiB
    ("4k_b16h16", 16, 16, 4096, 4096, True, "persistent", SMS),
    ("8k_b1h16", 1, 16, 8192, 8192, True, "persistent_weight", SMS),         # K/V exactly 64 MiB
    ("16k_b4h16", 4, 16, 16384, 16384, True, "tile_grid", 4 * 16 * 128),     # 8 MiB per head: groups of 2 < 4
    # edges
    ("148 tiles", 1, 148, 128, 128, True, "tile_grouped", 148),              # not more tiles than SMs
    ("149 tiles", 1, 149, 128, 128, True, "persistent_weight", SMS),
    ("8k_b1h17", 1, 17, 8192, 8192, True, "tile_grouped", 17 * 64),          # 68 MiB: not weight-major, Nk > 4096
    ("noncausal_4k", 4, 16, 4096, 4096, False, "persistent", SMS),           # weight-major needs causal masking
    ("noncausal_8k", 1, 16, 8192, 8192, False, "tile_grid", 16 * 64),        # no groups without causal masking
    ("one head", 1, 1, 2048, 2048, True, "tile_grid", 16),                   # one head is no group of four
    ("empty", 0, 16, 2048, 2048, True, "tile_grid", 0),
])
def test_prefill_plan_bf16(name, B, H, Nq, Nk, causal, form, ctas):
    assert da.prefill_plan(B, H, Nq, Nk, 64, 128, causal=causal, sms=SMS) == (form, ctas), name


def test_weight_major_threshold_is_64_mib_of_k_and_v():
    # bf16, d = 64, dv = 128: 512 bytes per key and head.
    per_key = 4 * 64 + 2 * 128
    assert 1 * 16 * 8192 * per_key == 64 * MiB
    assert da.prefill_plan(1, 16, 8192, 8192)[0] == "persistent_weight"
    # One more key per head tips it over: (b, h)-major, and past 4096 keys that
    # is no longer persistent; 4.0002 MiB per head also leaves only three
    # heads per 16 MiB group, so the (tile, h, b) grid.
    assert da.prefill_plan(1, 16, 8064, 8193) == ("tile_grid", 16 * 63)


def test_fp8_counts_one_byte_per_query_key_element():
    # 21 heads of 8192 keys: 66,060,288 bytes of K and V with e4m3 Q/K (384
    # bytes per key), within 64 MiB, so weight-major; 88,080,384 with bf16 Q/K
    # (512 bytes per key), so (b, h)-major.
    assert 21 * 8192 * (2 * 64 + 2 * 128) < 64 * MiB < 21 * 8192 * (4 * 64 + 2 * 128)
    assert da.prefill_plan(1, 21, 8192, 8192, fp8=True)[0] == "persistent_weight"
    assert da.prefill_plan(1, 21, 8192, 8192, fp8=False)[0] == "tile_grouped"


def test_d32_widths():
    # d = 32, dv = 64: 256 bytes per key, so 32 heads of 8192 keys fit 64 MiB.
    assert da.prefill_plan(1, 32, 8192, 8192, 32, 64) == ("persistent_weight", SMS)
    assert da.prefill_plan(1, 33, 8192, 8192, 32, 64)[0] == "tile_grouped"


def test_tile_count_limit_of_the_1d_orders():
    # 2^30 tiles or more: the (tile, h, b) grid, whatever else holds.
    B, H = 1 << 15, 1 << 15
    assert da.prefill_plan(B, H, 128, 128) == ("tile_grid", B * H)
    assert da.prefill_plan(B, H - 1, 128, 128) == ("persistent", SMS)


def test_plan_rejects_bad_arguments():
    for args, kw in (((1, 1, 128, 128, 48, 128), {}), ((1, 1, 256, 128), {"causal": True}),
                     ((1, 1, 128, 0), {}), ((-1, 1, 128, 128), {}), ((1, 1, 128, 128), {"sms": 0})):
        with pytest.raises(da.DiffAttnError):
            da.prefill_plan(*args, **kw)

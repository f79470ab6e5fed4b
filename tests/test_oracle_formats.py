"""Oracle format codecs pinned to library casts, the OCP MX table and exact rationals."""
import pins


def test_e4m3_decode_matches_torch(orc):
    assert pins.pin_e4m3_decode(orc) == []


def test_e2m1_decode_matches_ocp_table(orc):
    assert pins.pin_e2m1_decode(orc) == []


def test_ue8m0_decode_matches_torch(orc):
    assert pins.pin_ue8m0_decode(orc) == []


def test_bf16_encode_matches_torch(orc):
    assert pins.pin_bf16_encode(orc) == []


def test_e4m3_encode_matches_torch_and_saturates(orc):
    assert pins.pin_e4m3_encode(orc) == []


def test_e4m3_round_trip_all_finite_codes(orc):
    import numpy as np
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF, 0x80)], np.uint8)
    assert np.array_equal(orc.encode_e4m3(orc.decode_e4m3(codes)), codes)


def test_requant_code_is_smallest_power_of_two(orc):
    assert pins.pin_requant_code(orc) == []

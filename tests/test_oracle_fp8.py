"""Pins for the oracle's FP8 E4M3 code (CPU only).

The FP8 KV cache of the decode engine on the ORL paper card (Table 11
caption: the NVFP4 configurations use an FP8 KV cache) stores K and V as
OCP E4M3 codes with a per-head scale.  oracle.c restates the format from its
definition; these checks tie it to things other than itself:
- decoding: all 256 codes against torch's float8_e4m3fn conversion;
- encoding: every bf16 value and a million random fp32 values below the
  saturation boundary against torch's conversion (round to nearest even);
  at and beyond 464 (torch returns NaN there) the definition's saturation to
  448; NaN stays NaN;
- closed forms: the largest finite value 448, the smallest subnormal 2^-9,
  ties at halfway points go to the even code, round trips are exact;
- the KV quantiser divides in fp32 before encoding.
"""
import numpy as np
import torch

import oracle


def _torch_encode(x32):
    return torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32)).to(
        torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_decode_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    d = oracle.e4m3_decode(codes)
    t = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(d), np.isnan(t))
    assert np.array_equal(d[~np.isnan(d)], t[~np.isnan(t)])
    assert np.isnan(d[0x7F]) and np.isnan(d[0xFF]) and np.isnan(d).sum() == 2
    assert d[0x7E] == 448.0 and d[0x01] == 2.0 ** -9 and d[0x08] == 2.0 ** -6


def test_encode_every_bf16_value():
    bits = np.arange(1 << 16, dtype=np.uint32) << 16
    x = bits.view(np.float32)
    got = oracle.e4m3_encode(x)
    finite = np.isfinite(x)
    small = finite & (np.abs(x) < 464.0)
    assert np.array_equal(got[small], _torch_encode(x[small]))
    big = ~np.isnan(x) & ~small  # >= 464 in magnitude, or infinite: saturate
    assert np.all((got[big] & 0x7F) == 0x7E)
    assert np.array_equal(got[big] >> 7, (np.signbit(x[big])).astype(np.uint8))
    assert np.all((got[np.isnan(x)] & 0x7F) == 0x7F)


def test_encode_random_fp32_values():
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(1_000_000) * np.exp2(rng.uniform(-14, 9, 1_000_000))).astype(np.float32)
    x = x[np.abs(x) < 464.0]
    assert np.array_equal(oracle.e4m3_encode(x), _torch_encode(x))


def test_ties_round_to_even_and_round_trips():
    # halfway between 1.0 (m=0) and 1.125 (m=1): to the even code m=0
    assert oracle.e4m3_encode(np.float32(1.0625)) == 0x38
    # halfway between 1.125 (m=1) and 1.25 (m=2): to m=2
    assert oracle.e4m3_encode(np.float32(1.1875)) == 0x3A
    # halfway between 0 and the smallest subnormal: to zero
    assert oracle.e4m3_encode(np.float32(2.0 ** -10)) == 0x00
    assert oracle.e4m3_encode(np.float32(-3.0 * 2.0 ** -10)) == 0x82  # -1.5 sub -> -2 sub
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    back = oracle.e4m3_encode(oracle.e4m3_decode(codes).astype(np.float32))
    same = (back == codes) | ((codes & 0x7F) == 0)  # -0 and +0 both decode to 0
    assert same.all()


def test_kv_quantiser_divides_in_fp32():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((64, 4, 16)).astype(np.float32)
    scale = np.array([0.01, 0.3, 1.0 / 3.0, 7.0], dtype=np.float32)
    want = _torch_encode(np.clip(x / scale.reshape(1, -1, 1), -463.0, 463.0))
    got = oracle.quantize_kv_e4m3(x, scale)
    q = x / scale.reshape(1, -1, 1)
    sat = np.abs(q) >= 464.0
    assert np.array_equal(got[~sat], want[~sat]) and np.all((got[sat] & 0x7F) == 0x7E)
    deq = oracle.dequantize_kv_e4m3(got, scale)
    assert np.allclose(deq[~sat], x[~sat], rtol=2.0 ** -4, atol=float(scale.max()) * 2.0 ** -9)

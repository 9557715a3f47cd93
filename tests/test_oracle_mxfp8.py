"""Pins for the oracle's MXFP8 codec.

* E4M3 decode: spec values (tests/golden/e4m3_spec_values.txt) and all 256
  codes against PyTorch's float8_e4m3fn conversion;
* E4M3 encode: round-to-nearest-even against PyTorch's fp32 -> float8_e4m3fn
  cast on in-range values, identity on every finite code, saturation at 448;
* E8M0 scale: closed forms of floor(log2 amax) - 8 + 127;
* block quantisation: error at most half a unit in the last place of the
  scaled element (unless saturated), exact dequantisation of known payloads.
"""
import os

import numpy as np
import pytest
import torch

from oracle import mxfp8 as M

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _spec_table():
    rows = []
    with open(os.path.join(GOLDEN, "e4m3_spec_values.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                c, v = line.split()
                rows.append((int(c, 16), float(v)))
    return rows


def test_decode_spec_values():
    for code, val in _spec_table():
        got = float(M.e4m3_decode(np.uint8(code)))
        if np.isnan(val):
            assert np.isnan(got), hex(code)
        else:
            assert got == val and np.signbit(got) == np.signbit(val), hex(code)


def test_decode_all_codes_against_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = M.e4m3_decode(codes)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])


def test_encode_rne_against_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(50000) * 50, rng.standard_normal(50000) * 1e-2,
                        rng.uniform(-448, 448, 20000)]).astype(np.float32)
    # exact midpoints between neighbours: ties go to the even code
    finite = M.e4m3_decode(np.arange(0x7E, dtype=np.uint8))
    mids = ((finite[:-1] + finite[1:]) / 2).astype(np.float32)
    x = np.concatenate([x, mids, -mids])
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = M.e4m3_encode(x.astype(np.float64))
    assert np.array_equal(got, ref)


def test_encode_roundtrip_and_saturation():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    assert np.array_equal(M.e4m3_encode(M.e4m3_decode(codes)), codes)
    assert M.e4m3_encode(np.array([1000.0, -1e9, 448.0, 464.0, 470.0]) ).tolist() == [0x7E, 0xFE, 0x7E, 0x7E, 0x7E]
    assert M.e4m3_encode(np.array([np.nan]))[0] == 0x7F


@pytest.mark.parametrize("amax,code", [(1.0, 119), (1.99, 119), (2.0, 120), (448.0, 127), (0.75, 118),
                                       (2.0 ** -130, 0), (0.0, 0), (3e38, 246), (2.0 ** 140, 254)])
def test_scale_code_closed_form(amax, code):
    assert int(M.e8m0_scale_code(np.array(amax))) == code


def test_quantize_error_bound_and_axes():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((8, 128)) * np.exp(rng.standard_normal((8, 1)) * 3)
    x[0, :32] = 0.0                                          # an all-zero block
    q, s = M.quantize(x, axis=1)
    assert s.shape == (8, 4) and q.shape == x.shape
    assert s[0, 0] == 0 and np.all(q[0, :32] == 0)
    deq = M.dequantize(q, s, axis=1)
    scale = np.repeat(M.e8m0_value(s), 32, axis=1)
    y = x / scale                                            # the scaled elements
    assert np.all(np.abs(y) < 512)
    mag = np.abs(y)
    e = np.floor(np.log2(np.maximum(mag, 2.0 ** -6)))
    half_ulp = 2.0 ** (e - 3) / 2                           # 3 mantissa bits
    sat = mag > 448
    err = np.abs(deq - x) / scale
    assert np.all(err[~sat] <= half_ulp[~sat] * (1 + 1e-12))
    assert np.all(np.abs(deq[sat]) == 448 * scale[sat])
    # quantising along axis 0 equals quantising the transpose along axis 1
    q0, s0 = M.quantize(x[:, :64].T.copy(), axis=0)
    q1, s1 = M.quantize(x[:, :64], axis=1)
    assert np.array_equal(q0, q1.T) and np.array_equal(s0, s1.T)


def test_dequantize_known_payload():
    payload = np.array([[0x38, 0x40, 0xB8, 0x00] + [0] * 28], np.uint8)   # 1, 2, -1, 0
    scale = np.array([[130]], np.uint8)                                     # 2^3
    deq = M.dequantize(payload, scale, axis=1)
    assert deq[0, :4].tolist() == [8.0, 16.0, -8.0, 0.0]


def test_input_quantiser_agrees_with_the_oracle_codec():
    """The seeded MXFP8 input weights (PyTorch float8 cast) follow the same OCP MX
    rule as the oracle's codec, so both describe the same weights."""
    import moe_inputs as MI
    g = torch.Generator().manual_seed(3)
    w = (torch.randn(2, 64, 96, generator=g) * 0.02).to(torch.bfloat16)
    w[0, :32, :32] = 0                                     # all-zero blocks
    for axis, np_axis in ((-1, 2), (-2, 1)):
        q, s = MI.mxfp8_quantize_torch(w, axis)
        rq, rs = M.quantize(w.double().numpy(), axis=np_axis)
        assert np.array_equal(q.numpy(), rq) and np.array_equal(s.numpy(), rs)

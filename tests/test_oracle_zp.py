"""Pins of the oracle's asymmetric (scale + zero point) blocks, the next row
after symmetric KIVI (nalar.dev, "Granularitas kuantisasi mengendalikan
rentang...": low-bit codes need a scale and sometimes a zero point; the
error budget compares representations at equal bytes).

* exact round trip of representable grids (codes 0 and 2^b - 1 present,
  power-of-two scale, fp16 zero);
* the error bound: |x - x_hat| <= s/2 plus the fp16 rounding of the zero
  and the scale;
* brute force on small blocks: each code is a nearest level c*s + z;
* byte layout: fp16 scale, fp16 zero, then the unbiased codes in the
  format's bit fields;
* the error budget at 2 bits: four levels beat the ternary symmetric code on
  Gaussian blocks at 2 more bytes per block, and the cache round trip keeps
  the bound.
"""

import numpy as np
import pytest

from oracle import kvq_oracle as O


@pytest.mark.parametrize("bits", [2, 3, 4, 8])
def test_representable_grid_round_trips(bits):
    rng = np.random.default_rng(bits)
    qlev = (1 << bits) - 1
    for e in (-9, -3, 0, 2):
        s = 2.0 ** e
        z = float(np.float16(rng.standard_normal() * 4))
        c = rng.integers(0, qlev + 1, size=(64, 32))
        c[:, 0], c[:, 1] = 0, qlev
        x = (c * s + z).astype(np.float32)
        assert np.array_equal(x.astype(np.float64), c * s + z)  # exactly representable
        s16, z16, codes = O.quantize_zp(x, bits)
        assert np.all(s16.astype(np.float64) == s) and np.all(z16.astype(np.float64) == z)
        assert np.array_equal(codes, c)
        assert np.array_equal(O.dequantize_zp_f64(s16, z16, codes), x.astype(np.float64))


@pytest.mark.parametrize("bits", [2, 4])
def test_error_bound_and_nearest_level(bits):
    rng = np.random.default_rng(10 + bits)
    qlev = (1 << bits) - 1
    x = (rng.standard_normal((2000, 32)) * rng.lognormal(0, 1.5, (2000, 1)) + rng.standard_normal((2000, 1))
         ).astype(np.float16).astype(np.float32)
    s16, z16, codes = O.quantize_zp(x, bits)
    sf = s16.astype(np.float64)[:, None]
    zf = z16.astype(np.float64)[:, None]
    xh = O.dequantize_zp_f64(s16, z16, codes)
    mn, mx = x.min(-1, keepdims=True).astype(np.float64), x.max(-1, keepdims=True).astype(np.float64)
    bound = 0.5 * sf + qlev * sf * 2.0 ** -10 + (np.abs(mn) + np.abs(mx)) * 2.0 ** -10
    assert np.all(np.abs(x - xh) <= bound)
    # brute force: the chosen level is a nearest one (up to fp32 rounding of the quotient)
    levels = np.arange(qlev + 1)[None, None, :] * sf[..., None] + zf[..., None]
    d = np.abs(x[..., None].astype(np.float64) - levels)
    chosen = np.take_along_axis(d, codes[..., None].astype(np.int64), -1)[..., 0]
    assert np.all(chosen <= d.min(-1) + 1e-6 * sf)
    assert codes.min() == 0 and codes.max() == qlev


def test_zero_range_block():
    x = np.full((3, 32), 1.25, np.float32)
    x[1] = 0.0
    s16, z16, codes = O.quantize_zp(x, 4)
    assert np.all(s16 == 0) and np.all(codes == 0)
    assert np.array_equal(O.dequantize_zp_f64(s16, z16, codes), x.astype(np.float64))


def test_signed_zero_minimum_is_stored_as_plus_zero():
    x = np.abs(np.random.default_rng(3).standard_normal((4, 32))).astype(np.float32)
    x[0, 5], x[0, 9] = -0.0, 0.0
    x[1, 0] = -0.0
    x[2, :] = -0.0
    x[3, 7] = -0.0
    x[3, 8] = -1.0
    s16, z16, codes = O.quantize_zp(x, 4)
    assert list(z16[:3].view(np.uint16)) == [0, 0, 0]
    assert z16[3] == -1.0 and s16[2] == 0 and np.all(codes[2] == 0)
    blob = O.encode_blocks(x, 4, zp=True)
    assert np.all(blob[:3, 2:4] == 0)


def test_byte_layout():
    x = np.arange(32, dtype=np.float32) / 2 - 3.0  # min -3, step 0.5: scale 15.5/15 -> fp16
    blob = O.encode_blocks(x[None], 4, zp=True)[0]
    assert blob.shape == (O.block_bytes(4, 32, zp=True),) == (20,)
    s16, z16, codes = O.quantize_zp(x[None], 4)
    assert blob[0:2].view(np.float16)[0] == s16[0] and blob[2:4].view(np.float16)[0] == z16[0]
    c = codes[0].astype(np.int64)
    assert np.array_equal(blob[4:], (c[0::2] | (c[1::2] << 4)).astype(np.uint8))
    blob2 = O.encode_blocks(x[None], 2, zp=True)[0]
    s2, z2, c2 = O.quantize_zp(x[None], 2)
    c2 = c2[0].astype(np.int64).reshape(8, 4)
    assert np.array_equal(blob2[4:], (c2[:, 0] | c2[:, 1] << 2 | c2[:, 2] << 4 | c2[:, 3] << 6).astype(np.uint8))
    assert O.block_bytes(2, 32, zp=True) == 12 and O.block_bytes(4, 32) == 18


def test_two_bit_error_budget():
    """At 2 bits the zero point buys four levels instead of the ternary
    symmetric code: lower MSE on Gaussian blocks, for 12 B instead of 10 B
    per 32 values."""
    rng = np.random.default_rng(7)
    x = rng.standard_normal((4000, 32)).astype(np.float32)
    s, c = O.quantize(x, 2)
    mse_sym = np.mean((O.dequantize_f64(s, c) - x) ** 2)
    s16, z16, cz = O.quantize_zp(x, 2)
    mse_zp = np.mean((O.dequantize_zp_f64(s16, z16, cz) - x) ** 2)
    assert len(np.unique(cz)) == 4 and len(np.unique(c)) == 3
    assert mse_zp < 0.8 * mse_sym, (mse_zp, mse_sym)


def test_zp_cache_round_trip():
    cfg = O.Config(L=1, H_kv=2, H_q=2, D=128, batch=1, max_T=256, in_dtype=O.DT_F16,
                   k_fmt=O.Fmt(4, 32, O.AXIS_CHANNEL, zp=True), v_fmt=O.Fmt(4, 32, zp=True),
                   k_cold=O.Fmt(2, 32, O.AXIS_CHANNEL, zp=True), v_cold=O.Fmt(2, 32, zp=True),
                   hot_window=64, residual_window=32)
    bufs = O.new_buffers(cfg)
    rng = np.random.default_rng(8)
    T = 200
    k = (rng.standard_normal((T, 2, 128)) + 0.5).astype(np.float16)
    v = rng.standard_normal((T, 2, 128)).astype(np.float16)
    O.append(cfg, bufs, 0, k.view(np.uint16), v.view(np.uint16), [T], [0])
    K, V = O.dequantize(cfg, bufs, 0, 0, T)
    qe, ce = O.q_end(cfg, T), O.c_end(cfg, T)
    assert 0 < ce < qe < T
    kf = k.astype(np.float64)
    # hot tier (4-bit) and window are close; cold (2-bit) coarser; window exact
    assert np.array_equal(K[qe:], kf[qe:])
    hot_err = np.abs(K[ce:qe] - kf[ce:qe]).max()
    cold_err = np.abs(K[:ce] - kf[:ce]).max()
    assert hot_err < 0.6 and cold_err < 2.5 and hot_err < cold_err

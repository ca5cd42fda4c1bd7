"""The seeded block-scaled quantiser (input preparation for the MX and
NVFP4 parity cases), checked on the CPU with the oracle's pinned decoders."""
import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si

FORMATS = [("e4m3", 32, "e8m0"), ("e5m2", 32, "e8m0"), ("e2m1", 32, "e8m0"), ("e2m1", 16, "ue4m3")]


def _decode(codes, scodes, elem, block, scale):
    if elem == "e2m1":
        nib = np.stack([codes & 15, codes >> 4], axis=-1).reshape(codes.shape[0], -1)
        vals = oracle.e2m1_to_f64(nib)
    else:
        vals = oracle.e4m3_to_f64(codes) if elem == "e4m3" else oracle.e5m2_to_f64(codes)
    svals = oracle.e8m0_to_f64(scodes) if scale == "e8m0" else oracle.ue4m3_to_f64(scodes)
    K = vals.shape[1]
    return vals * np.repeat(svals, block, axis=1)[:, :K], vals


@pytest.mark.parametrize("elem,block,scale", FORMATS)
def test_block_scaled_quantiser_error_and_range(elem, block, scale):
    """Every element is within half a step of its format at its block's
    scale, or, where the MX rule's scale 2^(floor(log2 amax) - emax) puts
    it above the format's largest value (E4M3: 448 = 1.75 * 2^8), is clamped
    to that value, as the MX definition says (K = 200: a partial last block)."""
    t = si.normal((6, 200), 11) * 3.0
    codes, scodes = si.to_block_scaled(t, elem, block, scale)
    got, vals = _decode(codes, scodes, elem, block, scale)
    x = t.to(torch.float64).numpy()
    assert np.isfinite(got).all()
    mant = {"e4m3": 3, "e5m2": 2, "e2m1": 1}[elem]
    # a value's step is 2^(floor(log2|v|) - mant) in its binade; the bound
    # below takes the step of the block's largest binade, which covers all
    svals = (oracle.e8m0_to_f64(scodes) if scale == "e8m0" else oracle.ue4m3_to_f64(scodes))
    amax_blocks = np.abs(np.pad(x, ((0, 0), (0, -x.shape[1] % block)))).reshape(6, -1, block).max(axis=-1)
    step = 2.0 ** (np.floor(np.log2(amax_blocks)) - mant + 1)
    sfull = np.repeat(svals, block, axis=1)[:, :200]
    top = si._ELEM_MAX[elem][0] * sfull
    clamped = np.abs(x) > top
    assert np.array_equal(np.abs(got[clamped]), top[clamped])
    assert np.all(np.sign(got[clamped]) == np.sign(x[clamped]))
    ok = ~clamped
    assert np.all(np.abs(got - x)[ok] <= (np.repeat(step, block, axis=1)[:, :200] * 0.5)[ok])
    assert np.all(svals > 0)
    if scale == "ue4m3":
        # NVFP4's scale is amax / 6 rounded to E4M3: a scale rounded down by
        # at most 1/16 clamps the block's largest element by at most that much
        assert np.all(np.abs(x[clamped]) <= top[clamped] * (1 + 1 / 16))


@pytest.mark.parametrize("elem,block,scale", FORMATS[:3])
def test_block_scaled_quantiser_is_exact_on_representable_values(elem, block, scale):
    """Values that are already element values times a power-of-two scale
    come back unchanged."""
    rng = np.random.default_rng(12)
    rows, K = 3, 2 * block
    if elem == "e2m1":
        vals = np.array(si.E2M1_MAGNITUDES)[rng.integers(1, 8, size=(rows, K))]
        vals[:, ::block] = 6.0  # each block reaches the top of the format
    else:
        codes = rng.integers(0x30, 0x60, size=(rows, K), dtype=np.uint8)
        vals = oracle.e4m3_to_f64(codes) if elem == "e4m3" else oracle.e5m2_to_f64(codes)
        vals[:, ::block] = si._ELEM_MAX[elem][0]
    x = vals * np.where(rng.random((rows, K)) < 0.5, -1.0, 1.0) * 2.0 ** -20
    codes, scodes = si.to_block_scaled(torch.from_numpy(x), elem, block, scale)
    got, _ = _decode(codes, scodes, elem, block, scale)
    assert np.array_equal(got, x)


def test_e2m1_rounding_ties_to_even():
    x = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 7.0, -0.75, -5.0])
    want = [0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0, 6.0, -1.0, -4.0]
    got = oracle.e2m1_to_f64(si._e2m1_codes(x))
    assert got.tolist() == want


def test_nvfp4_scale_stays_in_range_for_huge_and_tiny_runs():
    """A run whose amax / 6 is above E4M3's largest value takes the largest
    scale (448) and clips to +-6 x 448; one below the smallest subnormal
    takes the smallest scale (2^-9): neither gets a NaN or zero scale."""
    x = np.zeros((2, 32))
    x[0, :16] = np.linspace(-6000.0, 6000.0, 16)  # amax / 6 = 1000 > 448
    x[0, 16:] = np.linspace(-1e-5, 1e-5, 16)      # amax / 6 ~ 1.7e-6 < 2^-9 ~ 1.95e-3
    x[1, :16] = 1.0
    codes, scodes = si.to_block_scaled(torch.from_numpy(x), "e2m1", 16, "ue4m3")
    svals = oracle.ue4m3_to_f64(scodes)
    assert svals[0, 0] == 448.0 and svals[0, 1] == 2.0 ** -9
    assert np.all(np.isfinite(svals)) and np.all(svals > 0)
    got, _ = _decode(codes, scodes, "e2m1", 16, "ue4m3")
    assert got[0, 0] == -6.0 * 448.0 and got[0, 15] == 6.0 * 448.0  # clipped at the top of the range
    assert np.all(np.abs(got[0, 16:] - x[0, 16:]) <= 2.0 ** -9 * 0.5)  # below one step of the smallest scale
    assert svals[1, 0] == 0.171875  # an in-range run keeps amax / 6 rounded to E4M3

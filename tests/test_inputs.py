"""The seeded input recipes do what the workloads state (CPU only)."""
import numpy as np
import pytest
import torch

import oracle
from dense_gemm_preshuffle_gb300 import inputs


def test_seeded_and_deterministic():
    a = inputs.make_operands("e4m3", 16, 32, 128, seed=inputs.SEED_BASE)
    b = inputs.make_operands("e4m3", 16, 32, 128, seed=inputs.SEED_BASE)
    assert np.array_equal(a.a, b.a) and np.array_equal(a.scale_b, b.scale_b)
    c = inputs.make_operands("e4m3", 16, 32, 128, seed=inputs.SEED_BASE + 1)
    assert not np.array_equal(a.a, c.a)


def test_e4m3_rows_amax_maps_to_448():
    g = inputs._gen(1)
    q, s = inputs.e4m3_rows(64, 512, g)
    v = oracle.decode_e4m3(q)
    assert not np.isnan(v).any()
    assert np.all(np.abs(v).max(axis=1) == 448.0)
    # dequantised values are close to an N(0,1) draw: |x| < 7 essentially always
    assert np.all(np.abs(v * s[:, None]) < 7.0)


def test_e4m3_rows_match_plain_quantisation():
    g = inputs._gen(5)
    x = torch.randn((8, 256), generator=g)
    amax = x.abs().amax(dim=1)
    q, s = inputs.e4m3_rows(8, 256, inputs._gen(5))
    assert np.array_equal(s, (amax / 448.0).numpy())
    # each code is the nearest E4M3 value to x/s (ties: even code)
    vals = oracle.decode_e4m3(np.arange(256, dtype=np.uint8))
    finite = ~np.isnan(vals)
    y = (x / (amax / 448.0)[:, None]).numpy().astype(np.float64)
    got = oracle.decode_e4m3(q)
    d_got = np.abs(got - y)
    d_best = np.min(np.abs(y[..., None] - vals[finite][None, None, :]), axis=-1)
    assert np.all(d_got == d_best)


def test_int8_range():
    x = inputs.int8_rows(64, 4096, inputs._gen(2))
    assert x.dtype == np.int8 and x.min() == -127 and x.max() == 127


def test_bf16_scale():
    x = oracle.decode_bf16(inputs.bf16_rows(64, 4096, inputs._gen(3)))
    assert abs(x.std() * np.sqrt(4096) - 1.0) < 0.02


@pytest.mark.parametrize("amax,e", [(6.0, 0), (6.0 * (1 + 2.0 ** -23), 1), (3.0, -1), (0.0, 0),
                                    (12.0, 1), (12.000001, 2), (0.75, -3), (1e-30, -102)])
def test_ue8m0_exponent_rule(amax, e):
    assert int(inputs.ue8m0_block_exponent(np.array([amax]))[0]) == e


@pytest.mark.parametrize("v,val", [(0.25, 0.0), (0.75, 1.0), (1.25, 1.0), (1.75, 2.0), (2.5, 2.0),
                                   (3.5, 4.0), (5.0, 4.0), (0.2, 0.0), (0.3, 0.5), (5.1, 6.0),
                                   (6.0, 6.0), (-2.5, -2.0), (-0.74, -0.5)])
def test_e2m1_round_to_nearest_even(v, val):
    code = inputs.e2m1_encode(np.array([v]))
    assert oracle.decode_e2m1(code)[0] == val


def test_mxfp4_blocks_fit_and_use_the_range():
    pa, ea = inputs.mxfp4_rows(32, 1024, inputs._gen(4))
    codes = oracle.unpack_e2m1_rows(pa, 1024)
    vals = oracle.decode_e2m1(codes).reshape(32, 32, 32)
    scale = oracle.decode_ue8m0(ea)
    # the block maximum lands in (3, 6]: amax/2^e is in (3, 6] before rounding
    m = np.abs(vals).max(axis=2)
    assert np.all((m >= 3.0) & (m <= 6.0))
    # reconstruct and compare to the draw (relative to the block scale)
    g = inputs._gen(4)
    x = torch.randn((32, 1024), generator=g).numpy().reshape(32, 32, 32)
    err = np.abs(vals * scale[:, :, None] - x) / scale[:, :, None]
    assert err.max() <= 1.0  # half the widest E2M1 gap (4 -> 6)

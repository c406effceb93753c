"""GPU parity of the halo-tile conv kernel (grids at least 128 pixels wide).

Every conv op of small decodes whose upper levels are 128-256 pixels wide is
checked against the oracle's conv applied to the op's captured input, covering
plain 3x3 convs, causal 3x3x3 convs, the four-phase upsample conv, residuals,
shortcut outputs and ragged row tiles; then whole decodes against the oracle
and across band counts.
"""
import numpy as np
import pytest

import synth
from gpu_helpers import Case, assert_bf16_parity, max_abs, oracle_op, parse_shape, rel_l2

pytestmark = pytest.mark.gpu


def check_conv_ops(case, n_bands, min_width=128):
    checked = 0
    for op in range(case.dec.num_ops(case.shape, n_bands)):
        d = case.dec.op_desc(case.shape, n_bands, op)
        if d["kind"] != "conv" or parse_shape(d["in"])[3] < min_width:
            continue
        d, x, aux, y = case.capture(n_bands, op)
        ref = oracle_op(d, case.W, case.arch, x.reshape(parse_shape(d["in"])), aux)
        err = rel_l2(y.reshape(ref.shape), ref)
        assert err <= 6e-3, f"op {op} {d}: rel-L2 {err:.3e}"
        checked += 1
    assert checked > 0
    return checked


@pytest.fixture(scope="module")
def kl_wide():
    # levels 4x32 -> 8x64 -> 16x128 -> 32x256
    return Case(synth.KL_ZIMAGE, "bf16", (1, 16, 4, 32))


def test_kl_halo_conv_ops(kl_wide):
    assert check_conv_ops(kl_wide, 2) >= 10


def test_kl_halo_decode_matches_oracle(kl_wide):
    assert bool((kl_wide.decode(1).cpu() == kl_wide.decode(4).cpu()).all())
    out = kl_wide.decode(2).float().cpu().numpy()
    ref = kl_wide.oracle()
    assert_bf16_parity(out, ref)


@pytest.fixture(scope="module")
def wan_wide():
    # levels 4x32 -> 8x64 -> 16x128 -> 32x256, frames 2 -> 3 -> 5
    return Case(synth.WAN, "bf16", (1, 16, 2, 4, 32))


def test_wan_halo_conv_ops(wan_wide):
    assert check_conv_ops(wan_wide, 2) >= 8


def test_wan_halo_decode_matches_oracle(wan_wide):
    out = wan_wide.decode(2).float().cpu().numpy()
    ref = wan_wide.oracle()
    assert_bf16_parity(out, ref)

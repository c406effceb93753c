"""Degenerate shapes on the GPU against the float64 oracle: one-pixel and one-row/one-column
latents, one-row bands (n_bands = H) and a single frame for the causal decoder.

The fp32 path takes any size; the bf16 tensor-core path needs latent H*W to be a multiple of 8
(its attention streams 16-byte key rows), so its narrowest grids are 1 x 8 and 8 x 1, and its
narrowest two-wide grids 2 x 4, 4 x 2, 2 x 8 and 8 x 2.  Bars as in the other parity tests (fp32
rel-L2 <= 1e-4; bf16 max-abs <= 3e-2 and rel-L2 <= 1e-2, whole output), and the output is bit for
bit the same for every band count and split axis.

The one-wide bf16 grids (1 x 8, 8 x 1) sit above the whole-decode rel-L2 bar: every op is at the
bf16 rounding floor (rel-L2 ~2e-3 per op), but the ~40 roundings of the decode compound to a
rel-L2 of 1.09-1.18% on those outputs (measured on GB300).  The bar is therefore claimed from
two-wide grids up, where all four cases meet both bars in full; the one-wide grids are checked
op by op (every op against the oracle applied to that op's own GPU input, at one band and at
one-row bands), against the whole-decode max-abs bar, and for band and axis invariance.
"""
import pytest

import synth
from gpu_helpers import BF16_MAX_ABS, Case, assert_bf16_parity, check_all_ops, max_abs, rel_l2

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("shape", [(1, 4, 1, 1), (1, 4, 1, 5), (1, 4, 3, 1), (2, 4, 2, 3)])
def test_fp32_degenerate_latents(shape):
    c = Case(synth.KL_TINY, "fp32", shape)
    ref = c.oracle()
    out = c.decode(1)
    got = out.cpu().numpy()
    assert got.shape == ref.shape
    assert rel_l2(got, ref) <= 1e-4
    torch = c.torch
    for n in range(2, shape[2] + 1):               # up to one-row bands
        assert bool((c.decode(n).cpu() == out.cpu()).all()), n
    for n in range(2, shape[3] + 1):
        o = c.dec.decode(c.z_dev, n, axis="width")
        torch.cuda.synchronize()
        assert bool((o.cpu() == out.cpu()).all()), ("width", n)


@pytest.mark.parametrize("shape", [(1, 16, 1, 8), (1, 16, 8, 1)])
def test_bf16_one_row_and_one_column_latents(shape):
    c = Case(synth.KL_ZIMAGE, "bf16", shape)
    kinds = check_all_ops(c, 1)
    assert {"conv:k3", "conv:up2x_k3", "groupnorm:", "attention:"} <= kinds
    if shape[2] > 1:
        check_all_ops(c, shape[2], stride=3)       # one-row bands
    ref = c.oracle()
    out = c.decode(1)
    got = out.float().cpu().numpy()
    assert got.shape == ref.shape
    e_abs = max_abs(got, ref)
    assert e_abs <= BF16_MAX_ABS, f"max-abs {e_abs:.4f} (rel-L2 {rel_l2(got, ref):.4e})"
    if shape[2] > 1:
        assert bool((c.decode(shape[2]).cpu() == out.cpu()).all())
    if shape[3] > 1:
        o = c.dec.decode(c.z_dev, shape[3], axis="width")
        c.torch.cuda.synchronize()
        assert bool((o.cpu() == out.cpu()).all())


@pytest.mark.parametrize("shape", [(1, 16, 2, 4), (1, 16, 4, 2), (1, 16, 2, 8), (1, 16, 8, 2)])
def test_bf16_two_wide_latents_meet_both_bars(shape):
    c = Case(synth.KL_ZIMAGE, "bf16", shape)
    ref = c.oracle()
    out = c.decode(1)
    got = out.float().cpu().numpy()
    assert got.shape == ref.shape
    assert_bf16_parity(got, ref)
    for n in range(2, shape[2] + 1):               # down to one-row bands
        assert bool((c.decode(n).cpu() == out.cpu()).all()), n
    for n in range(2, shape[3] + 1):
        o = c.dec.decode(c.z_dev, n, axis="width")
        c.torch.cuda.synchronize()
        assert bool((o.cpu() == out.cpu()).all()), ("width", n)


def test_wan_single_frame():
    c = Case(synth.WAN, "bf16", (1, 16, 1, 4, 6))    # T = 1: the temporal upsamples keep 1 frame
    ref = c.oracle()
    out = c.decode(4)                                # one-row bands
    got = out.float().cpu().numpy()
    assert got.shape == ref.shape == (1, 3, 1, 32, 48)
    assert_bf16_parity(got.reshape(-1), ref.reshape(-1))
    assert bool((c.decode(1).cpu() == out.cpu()).all())

"""GPU parity: the CUDA decode (through the C ABI) against the float64 oracle.

Per-op checks trace every op of the decode (its captured input, residual and
output) and compare the output with the oracle's op applied to the same input.
End-to-end checks compare whole decodes with the oracle's decode within the
stated tolerances: bf16 tensor-core path max-abs <= 3e-2 and rel-L2 <= 1e-2,
fp32 path rel-L2 <= 1e-4.  Band-count invariance is checked bit for bit.
"""
import dataclasses

import numpy as np
import pytest

import synth
from gpu_helpers import Case, assert_bf16_parity, check_all_ops, rel_l2

pytestmark = pytest.mark.gpu

BF16_MAX_ABS = 3e-2
BF16_REL_L2 = 1e-2
F32_REL_L2 = 1e-4

# ---------------------------------------------------------------- fp32 path
@pytest.fixture(scope="module")
def tiny():
    w = synth.WORKLOADS["kl_tiny_fp32"]
    return Case(w.arch, w.dtype, w.latent_shape)


def test_tiny_fp32_every_op(tiny):
    kinds = check_all_ops(tiny, 2)
    assert {"conv:k3", "conv:up2x_k3", "groupnorm:", "attention:"} <= kinds


def test_tiny_fp32_decode_matches_oracle(tiny):
    out = tiny.decode(2)
    ref = tiny.oracle()
    got = out.float().cpu().numpy()
    assert got.shape == ref.shape
    assert rel_l2(got, ref) <= F32_REL_L2


def test_tiny_fp32_band_count_bitwise(tiny):
    base = tiny.decode(1).cpu()
    for nb in (2, 3, 16):
        assert bool((tiny.decode(nb).cpu() == base).all()), nb


# ---------------------------------------------------------------- bf16 KL path
@pytest.fixture(scope="module")
def kl_ops():
    # full Z-Image channel widths on a small, ragged latent (6 x 12)
    return Case(synth.KL_ZIMAGE, "bf16", (1, 16, 6, 12))


def test_kl_bf16_every_op(kl_ops):
    kinds = check_all_ops(kl_ops, 3)
    assert {"conv:k3", "conv:k1", "conv:up2x_k3", "groupnorm:", "attention:"} <= kinds


@pytest.fixture(scope="module")
def kl_small():
    return Case(synth.KL_ZIMAGE, "bf16", (1, 16, 12, 20))


def test_kl_bf16_decode_matches_oracle(kl_small):
    out = kl_small.decode(3).float().cpu().numpy()
    ref = kl_small.oracle()
    assert out.shape == ref.shape == (1, 3, 96, 160)
    assert_bf16_parity(out, ref)


def test_kl_bf16_band_count_bitwise(kl_small):
    base = kl_small.decode(1).cpu()
    for nb in (2, 3, 5, 12):
        assert bool((kl_small.decode(nb).cpu() == base).all()), nb


def test_kl_bf16_batch2_uneven_bands():
    # batch 2, 10 latent rows in 3 bands (4/3/3): element-count-weighted merge, unequal halos
    case = Case(synth.KL_ZIMAGE, "bf16", (2, 16, 10, 8), zseed=3)
    assert bool((case.decode(1).cpu() == case.decode(3).cpu()).all())
    out = case.decode(3).float().cpu().numpy()
    ref = case.oracle(3)
    assert_bf16_parity(out, ref)


# ---------------------------------------------------------------- bf16 Wan path
@pytest.fixture(scope="module")
def wan_small():
    return Case(synth.WAN, "bf16", (1, 16, 2, 6, 8))


def test_wan_bf16_every_op(wan_small):
    kinds = check_all_ops(wan_small, 2)
    assert {"conv:causal3", "conv:time", "conv:up2x_k3", "rmsnorm:", "attention:"} <= kinds


def test_wan_bf16_decode_matches_oracle(wan_small):
    out = wan_small.decode(2).float().cpu().numpy()
    ref = wan_small.oracle()
    assert out.shape == ref.shape == (1, 3, 5, 48, 64)
    assert_bf16_parity(out, ref)


def test_wan_bf16_band_count_bitwise(wan_small):
    base = wan_small.decode(1).cpu()
    for nb in (2, 3, 6):
        assert bool((wan_small.decode(nb).cpu() == base).all()), nb


# ---------------------------------------------------------------- host-side errors with a live handle
def test_bad_band_counts_rejected(kl_small):
    import row_band_layerwise_gb300 as rbl
    for nb in (0, 13, -1):
        with pytest.raises(rbl.VaedecError):
            kl_small.dec.decode(kl_small.z_dev, nb)
    # the handle stays usable
    assert kl_small.decode(2).shape == (1, 3, 96, 160)


def test_shape_above_max_rejected(kl_small):
    import torch
    import row_band_layerwise_gb300 as rbl
    z = torch.zeros((1, 16, 13, 20), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(rbl.VaedecError):
        kl_small.dec.decode(z, 1)


def test_bf16_grid_the_attention_cannot_take_is_unsupported(kl_small):
    """The bf16 path's fused attention streams keys as 16-byte rows: a latent grid whose H*W is
    not a multiple of 8 is refused with UNSUPPORTED before any launch, and the handle stays usable."""
    import torch
    import row_band_layerwise_gb300 as rbl
    n0 = kl_small.dec.launch_count()
    for shp in ((1, 16, 3, 5), (1, 16, 1, 7), (1, 16, 5, 9)):
        z = torch.zeros(shp, dtype=torch.bfloat16, device="cuda")
        with pytest.raises(rbl.VaedecError) as ei:
            kl_small.dec.decode(z, 1)
        assert ei.value.status == 2, str(ei.value)
        assert "multiple of 8" in str(ei.value)
    assert kl_small.dec.launch_count() == n0
    assert kl_small.decode(2).shape == (1, 3, 96, 160)


def test_one_workspace_layout_serves_every_smaller_shape():
    """The workspace arena is laid out once, at create time, for max_latent; every smaller latent
    reuses that layout.  A 16x16-bounded handle decodes an 8x8 latent (whose last stage is too
    narrow for the fused 1x1 shortcut, so the walk takes the other branch) and a 16x12 one, bit for
    bit as handles created for exactly those shapes, and within the bars of the oracle."""
    from gpu_helpers import Case
    import torch
    big = Case(synth.KL_ZIMAGE, "bf16", (1, 16, 16, 16))
    for shp in [(1, 16, 8, 8), (1, 16, 16, 12)]:
        exact = Case(synth.KL_ZIMAGE, "bf16", shp)
        z = exact.z_dev
        a = big.dec.decode(z, 2)
        torch.cuda.synchronize()
        big.dec.sync()
        b = exact.decode(2)
        assert bool((a == b).all()), shp
        assert_bf16_parity(a.float().cpu().numpy(), exact.oracle())
        exact.dec.close()
    big.dec.close()

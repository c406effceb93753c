"""GPU parity of the AutoencoderKLFlux2 latent front-end ("VAEP：VAE 并行解码", 不同模型如何复用:
the adapter keeps the latent BatchNorm and the patch conversion) against the float64 oracle.

The decode input is the transformer-side latent: 2x2-patchified and normalised by an inference
BatchNorm.  The library's first kernel undoes the BatchNorm and unpatchifies into the decoder's
channels-last latent; checked here as an op (one rounding of its output to the model dtype), in
whole decodes on the bf16 tensor-core path and the fp32 path, and for band-count and band-axis
invariance (bit for bit).
"""
import dataclasses

import numpy as np
import pytest

import synth
from gpu_helpers import Case, assert_bf16_parity, rel_l2
from oracle import decoder as odec

pytestmark = pytest.mark.gpu

FLUX2_TINY = dataclasses.replace(synth.KL_TINY, latent_channels=4, latent_patch=2, latent_bn_eps=1e-4)


@pytest.fixture(scope="module")
def flux2_bf16():
    # full FLUX.2-style widths on a small ragged patch grid (4 x 6 -> 8 x 12 decoder latent)
    return Case(synth.FLUX2, "bf16", (1, 128, 4, 6))


def test_frontend_op_matches_oracle(flux2_bf16):
    c = flux2_bf16
    d, x, aux, y = c.capture(2, 0)
    assert d["kind"] == "latent"
    ref = odec.latent_frontend(c.arch, c.W, x.reshape(c.shape))          # [B, C, 2H, 2W]
    got = y.reshape(ref.shape[0], ref.shape[2], ref.shape[3], ref.shape[1]).transpose(0, 3, 1, 2)
    assert rel_l2(got, ref) <= 4e-3           # one bf16 rounding of the output
    np.testing.assert_allclose(got, ref, rtol=8e-3, atol=1e-6)


def test_flux2_bf16_decode_matches_oracle(flux2_bf16):
    out = flux2_bf16.decode(3)
    ref = flux2_bf16.oracle()
    got = out.float().cpu().numpy()
    assert got.shape == ref.shape == (1, 3, 64, 96)
    assert_bf16_parity(got.reshape(-1), ref.reshape(-1))


def test_flux2_bf16_band_invariance(flux2_bf16):
    torch = flux2_bf16.torch
    base = flux2_bf16.decode(1)
    for n in (2, 5, 8):
        for axis in ("height", "width", "auto"):
            out = flux2_bf16.dec.decode(flux2_bf16.z_dev, n, axis=axis)
            torch.cuda.synchronize()
            assert bool((out == base).all()), (n, axis)


def test_flux2_fp32_decode_matches_oracle():
    c = Case(FLUX2_TINY, "fp32", (1, 16, 8, 8))
    out = c.decode(2)
    ref = c.oracle()
    got = out.cpu().numpy()
    assert got.shape == ref.shape == (1, 3, 32, 32)
    assert rel_l2(got, ref) <= 1e-4
    assert bool((c.decode(1).cpu() == out.cpu()).all())


def test_flux2_rejects_an_unpatched_latent(flux2_bf16):
    c = flux2_bf16
    z = c.torch.zeros((1, 32, 4, 6), dtype=c.torch.bfloat16, device="cuda")
    with pytest.raises(c.rbl.VaedecError):
        c.dec.decode(z, 1)

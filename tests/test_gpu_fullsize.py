"""GPU parity at the full workload sizes, in the launch configuration the bench times.

The float64 oracle needs minutes to an hour per full-size decode, so its outputs
are precomputed by ``tests/golden/make_decode_samples.py`` (which calls only the
seeded input generators and the oracle) and stored whole: the complete output of
every image workload, and for the video workload its first, middle and last
frames complete plus every output row within three rows of a band boundary in
every frame ("Static Layer-Wise VAE Decode", Tests: full tensors are compared,
boundary rows included).  Here the CUDA decode of the same workload (same seeds,
same band count as the bench) must match every stored element within the bf16
bars (max-abs <= 3e-2, rel-L2 <= 1e-2), and the decode must be bit for bit the
same for one band and for the workload's band count, checked on the whole output.
"""
import glob
import os

import numpy as np
import pytest

import synth
from gpu_helpers import assert_bf16_parity, max_abs, rel_l2, require_gpu

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
# workloads whose fixtures must be present (their oracle decodes take minutes to an hour)
REQUIRED = ("kl_zimage_512", "kl_zimage_1024", "kl_zimage_b2_800x1088", "wan_17x480x832")


def fixture_names():
    return sorted(os.path.basename(p)[len("decode_full_"):-4]
                  for p in glob.glob(os.path.join(GOLDEN, "decode_full_*.npz")))


def stored_pairs(ref, got_all):
    """(GPU values, oracle values) over every stored element of the fixture."""
    if "out" in ref:
        return got_all.reshape(-1), ref["out"].astype(np.float64).reshape(-1)
    frames, rows = ref["frames"], ref["rows"]
    g = [got_all[:, :, frames].reshape(-1), got_all[:, :, :, rows].reshape(-1)]
    r = [ref["frame_out"].reshape(-1), ref["row_out"].reshape(-1)]
    return np.concatenate(g), np.concatenate(r).astype(np.float64)


def test_required_fixtures_present():
    names = fixture_names()
    for r in REQUIRED:
        assert r in names, f"missing tests/golden/decode_full_{r}.npz"


@pytest.mark.parametrize("name", fixture_names())
def test_full_size_decode_matches_oracle(name):
    torch, rbl = require_gpu()
    w = synth.WORKLOADS[name]
    ref = dict(np.load(os.path.join(GOLDEN, f"decode_full_{name}.npz")))
    W = synth.make_weights(w.arch, w.dtype)
    z = synth.make_latent(w.latent_shape, w.dtype)
    shp = w.latent_shape
    max_latent = (shp[0], 1, shp[2], shp[3]) if len(shp) == 4 else (shp[0], shp[2], shp[3], shp[4])
    dec = rbl.Decoder(w.arch, W, w.dtype, max_latent)
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    zd = torch.from_numpy(z).to("cuda").to(tdt).contiguous()
    out = dec.decode(zd, w.n_bands)
    torch.cuda.synchronize()
    dec.sync()
    assert tuple(out.shape) == tuple(ref["shape"])
    got_all = out.float().cpu().numpy().astype(np.float64)
    assert np.isfinite(got_all).all()
    # band-count invariance over the whole output
    one = dec.decode(zd, 1)
    torch.cuda.synchronize()
    dec.sync()
    assert bool((one == out).all()), "1-band decode differs from the banded decode"
    dec.close()
    got, exp = stored_pairs(ref, got_all)
    print(f"\n{name}: {exp.size} elements compared, max-abs {max_abs(got, exp):.5f}, "
          f"rel-L2 {rel_l2(got, exp):.5e}")
    assert_bf16_parity(got, exp)

"""Pins for the oracle's decoders (CPU only).

* banded == unbanded: the pages' invariant that the layer-wise banded decode
  keeps whole-image semantics ("Static Layer-Wise VAE Decode", "Semantics and
  Communication"; "VAEP：VAE 并行解码", 按高度分片，逐层解码).
* the decoder composed from PyTorch CPU float64 library modules (conv2d,
  conv3d, group_norm, silu, interpolate, scaled_dot_product_attention) equals
  the oracle on tiny instances of both families.  This pins each layer's
  arithmetic and the wiring against a second, independent composition; the
  wiring's match with the Diffusers modules themselves is unpinned (neither
  Diffusers nor pretrained weights are available).
"""
import dataclasses

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import synth
from oracle import decoder

KL_SMALL = dataclasses.replace(
    synth.KL_ZIMAGE, mid_channels=16, stage_channels=(16, 16, 8, 8), stage_resnets=(1, 2, 1, 2),
    stage_up_channels=(16, 16, 8, 0), norm_groups=4)
WAN_SMALL = dataclasses.replace(
    synth.WAN, mid_channels=16, stage_channels=(16, 16, 8, 4), stage_resnets=(1, 1, 2, 1),
    stage_up_channels=(8, 8, 4, 0))


def _t(a):
    return torch.from_numpy(np.asarray(a, dtype=np.float64))


def torch_decode_kl(arch, W, z):
    T = {k: _t(v) for k, v in W.items()}
    G, eps = arch.norm_groups, arch.eps

    def conv(x, p):
        w = T[p + ".weight"]
        return F.conv2d(x, w, T[p + ".bias"], padding=w.shape[-1] // 2)

    def gn(x, p):
        return F.group_norm(x, G, T[p + ".weight"], T[p + ".bias"], eps)

    def resnet(x, p):
        h = conv(F.silu(gn(x, p + ".norm1")), p + ".conv1")
        h = conv(F.silu(gn(h, p + ".norm2")), p + ".conv2")
        sc = conv(x, p + ".conv_shortcut") if p + ".conv_shortcut.weight" in T else x
        return sc + h

    def attn(x, p):
        n, c, h, w = x.shape
        t = gn(x, p + ".group_norm").reshape(n, c, h * w).transpose(1, 2)
        q = F.linear(t, T[p + ".to_q.weight"], T[p + ".to_q.bias"])
        k = F.linear(t, T[p + ".to_k.weight"], T[p + ".to_k.bias"])
        v = F.linear(t, T[p + ".to_v.weight"], T[p + ".to_v.bias"])
        o = F.scaled_dot_product_attention(q, k, v)
        o = F.linear(o, T[p + ".to_out.0.weight"], T[p + ".to_out.0.bias"])
        return x + o.transpose(1, 2).reshape(n, c, h, w)

    x = conv(_t(z), "conv_in")
    x = resnet(x, "mid_block.resnets.0")
    x = attn(x, "mid_block.attentions.0")
    x = resnet(x, "mid_block.resnets.1")
    for s in range(len(arch.stage_channels)):
        for r in range(arch.stage_resnets[s]):
            x = resnet(x, f"up_blocks.{s}.resnets.{r}")
        if arch.stage_upsample[s]:
            x = conv(F.interpolate(x, scale_factor=2, mode="nearest"), f"up_blocks.{s}.upsamplers.0.conv")
    x = F.silu(gn(x, "conv_norm_out"))
    return conv(x, "conv_out").numpy()


def torch_decode_wan(arch, W, z):
    """Wan decoder run frame-chunk by frame-chunk with the causal feature cache.

    This follows the original module's streaming protocol (first latent frame
    alone, then one latent frame per call, a 2-frame cache per causal conv,
    the time_conv skipped on the first chunk), so it also pins the oracle's
    whole-sequence reading of that protocol.
    """
    T = {k: _t(v) for k, v in W.items()}

    def rms(x, g):
        return F.normalize(x, dim=1) * (x.shape[1] ** 0.5) * g.view(1, -1, *([1] * (x.ndim - 2)))

    caches = {}

    def cconv(x, p, key):
        w = T[p + ".weight"]
        kt, kh = w.shape[2], w.shape[3]
        prev = caches.get(key)
        need = kt - 1
        if need:
            if prev is None:
                prev = torch.zeros(x.shape[0], x.shape[1], 0, x.shape[3], x.shape[4], dtype=x.dtype)
            xin = torch.cat([prev, x], dim=2)
            xin = F.pad(xin, (0, 0, 0, 0, need - prev.shape[2], 0))
            caches[key] = xin[:, :, -need:]
        else:
            xin = x
        return F.conv3d(F.pad(xin, (kh // 2,) * 4), w, T[p + ".bias"])

    def resnet(x, p):
        h = cconv(F.silu(rms(x, T[p + ".norm1.gamma"])), p + ".conv1", p + ".conv1")
        h = cconv(F.silu(rms(h, T[p + ".norm2.gamma"])), p + ".conv2", p + ".conv2")
        sc = cconv(x, p + ".conv_shortcut", p + ".sc") if p + ".conv_shortcut.weight" in T else x
        return sc + h

    def attn(x, p):
        n, c, t, h, w = x.shape
        f = x.permute(0, 2, 1, 3, 4).reshape(n * t, c, h, w)
        f = rms(f, T[p + ".norm.gamma"])
        qkv = F.conv2d(f, T[p + ".to_qkv.weight"], T[p + ".to_qkv.bias"])
        qkv = qkv.reshape(n * t, 3 * c, h * w).transpose(1, 2)
        q, k, v = qkv[..., :c], qkv[..., c:2 * c], qkv[..., 2 * c:]
        o = F.scaled_dot_product_attention(q, k, v).transpose(1, 2).reshape(n * t, c, h, w)
        o = F.conv2d(o, T[p + ".proj.weight"], T[p + ".proj.bias"])
        return x + o.reshape(n, t, c, h, w).permute(0, 2, 1, 3, 4)

    def upsample(x, s, first_chunk):
        pre = f"up_blocks.{s}.upsamplers.0"
        if arch.stage_upsample[s] == 2 and not first_chunk:
            y = cconv(x, pre + ".time_conv", pre + ".time_conv")
            n, c2, t, h, w = y.shape
            c = c2 // 2
            x = torch.stack((y[:, :c], y[:, c:]), dim=3).reshape(n, c, 2 * t, h, w)
        n, c, t, h, w = x.shape
        f = x.permute(0, 2, 1, 3, 4).reshape(n * t, c, h, w)
        f = F.conv2d(F.interpolate(f, scale_factor=2, mode="nearest-exact"), T[pre + ".resample.1.weight"],
                     T[pre + ".resample.1.bias"], padding=1)
        return f.reshape(n, t, -1, 2 * h, 2 * w).permute(0, 2, 1, 3, 4)

    def chunk(x, first):
        x = cconv(x, "conv_in", "conv_in")
        x = resnet(x, "mid_block.resnets.0")
        x = attn(x, "mid_block.attentions.0")
        x = resnet(x, "mid_block.resnets.1")
        for s in range(len(arch.stage_channels)):
            for r in range(arch.stage_resnets[s]):
                x = resnet(x, f"up_blocks.{s}.resnets.{r}")
            if arch.stage_upsample[s]:
                x = upsample(x, s, first)
        x = F.silu(rms(x, T["norm_out.gamma"]))
        return cconv(x, "conv_out", "conv_out")

    zt = _t(z)
    outs = [chunk(zt[:, :, i:i + 1], i == 0) for i in range(zt.shape[2])]
    return torch.cat(outs, dim=2).numpy()


@pytest.fixture(scope="module")
def kl_small():
    W = synth.make_weights(KL_SMALL, "fp32", seed=5)
    z = synth.make_latent((2, 16, 7, 5), "fp32", seed=6)
    return W, z, decoder.decode(KL_SMALL, W, z)


@pytest.fixture(scope="module")
def wan_small():
    W = synth.make_weights(WAN_SMALL, "fp32", seed=7)
    z = synth.make_latent((1, 16, 3, 5, 4), "fp32", seed=8)
    return W, z, decoder.decode(WAN_SMALL, W, z)


def test_kl_decoder_matches_torch_composition(kl_small):
    W, z, y = kl_small
    assert y.shape == decoder.output_shape(KL_SMALL, z.shape)
    np.testing.assert_allclose(y, torch_decode_kl(KL_SMALL, W, z), rtol=1e-10, atol=1e-10)


def test_wan_decoder_matches_streaming_torch_composition(wan_small):
    W, z, y = wan_small
    assert y.shape == decoder.output_shape(WAN_SMALL, z.shape)
    np.testing.assert_allclose(y, torch_decode_wan(WAN_SMALL, W, z), rtol=1e-10, atol=1e-10)


def test_tiny_workload_matches_torch_composition():
    w = synth.WORKLOADS["kl_tiny_fp32"]
    W = synth.make_weights(w.arch, w.dtype)
    z = synth.make_latent(w.latent_shape, w.dtype)
    np.testing.assert_allclose(decoder.decode(w.arch, W, z), torch_decode_kl(w.arch, W, z),
                               rtol=1e-10, atol=1e-10)


@pytest.mark.parametrize("n_bands", [2, 3, 7])
def test_kl_banded_equals_unbanded(kl_small, n_bands):
    W, z, y = kl_small
    yb = decoder.decode(KL_SMALL, W, z, n_bands)
    np.testing.assert_allclose(yb, y, rtol=0, atol=1e-12 * np.abs(y).max())


@pytest.mark.parametrize("n_bands", [2, 5])
def test_wan_banded_equals_unbanded(wan_small, n_bands):
    W, z, y = wan_small
    yb = decoder.decode(WAN_SMALL, W, z, n_bands)
    np.testing.assert_allclose(yb, y, rtol=0, atol=1e-12 * np.abs(y).max())


def test_banded_without_halo_differs():
    """A banded conv that used zero padding at interior cuts (no halo) would
    differ from the unbanded decode at the band boundaries: the halo matters."""
    W, z = synth.make_weights(KL_SMALL, "fp32", seed=5), synth.make_latent((1, 16, 6, 5), "fp32", seed=9)
    from oracle import ops
    x = z.astype(np.float64)
    w, b = W["conv_in.weight"], W["conv_in.bias"]
    whole = ops.conv2d_same(x, w, b)
    cut = np.concatenate([ops.conv2d_same(x[:, :, :3], w, b), ops.conv2d_same(x[:, :, 3:], w, b)], axis=2)
    halo = decoder.Banded(2).join(decoder.Banded(2).conv(decoder.Banded(2).split(x), w, b))
    assert np.abs(cut - whole)[:, :, 2:4].max() > 1e-3
    np.testing.assert_allclose(halo, whole, rtol=0, atol=1e-13)


def test_too_many_bands_rejected():
    W, z, _ = None, synth.make_latent((1, 16, 3, 4), "fp32"), None
    with pytest.raises(ValueError):
        decoder.decode(KL_SMALL, synth.make_weights(KL_SMALL, "fp32"), z, 4)


# ---- width column bands (the pages' second spatial split axis) -------------------------------
@pytest.mark.parametrize("n_bands", [2, 3])
def test_kl_width_banded_equals_unbanded(kl_small, n_bands):
    W, z, y = kl_small
    yb = decoder.decode(KL_SMALL, W, z, n_bands, axis="width")
    np.testing.assert_allclose(yb, y, rtol=0, atol=1e-12 * np.abs(y).max())


def test_wan_width_banded_equals_unbanded(wan_small):
    W, z, y = wan_small
    yb = decoder.decode(WAN_SMALL, W, z, 2, axis="width")
    np.testing.assert_allclose(yb, y, rtol=0, atol=1e-12 * np.abs(y).max())


def test_width_banded_conv_needs_the_column_halo():
    """Zero padding at an interior column cut differs from the whole conv near the cut; the
    banded conv with neighbour columns as halo equals it."""
    W = synth.make_weights(KL_SMALL, "fp32", seed=5)
    x = synth.make_latent((1, 16, 5, 6), "fp32", seed=9).astype(np.float64)
    from oracle import ops
    w, b = W["conv_in.weight"], W["conv_in.bias"]
    whole = ops.conv2d_same(x, w, b)
    cut = np.concatenate([ops.conv2d_same(x[..., :3], w, b), ops.conv2d_same(x[..., 3:], w, b)], axis=-1)
    ex = decoder.Banded(2, "width")
    halo = ex.join(ex.conv(ex.split(x), w, b))
    assert np.abs(cut - whole)[..., 2:4].max() > 1e-3
    np.testing.assert_allclose(halo, whole, rtol=0, atol=1e-13)


def test_width_bands_take_the_remainder_first():
    ex = decoder.Banded(3, "width")
    parts = ex.split(np.zeros((1, 2, 4, 136)))
    assert [p.shape[-1] for p in parts] == [46, 45, 45]


@pytest.mark.parametrize("h,w,n,axis,want", [
    (128, 128, 8, "auto", "width"),      # square: width wins the tie
    (100, 136, 3, "auto", "width"),      # the longer axis
    (136, 100, 3, "auto", "height"),
    (20, 3, 4, "auto", "height"),        # width cannot hold 4 bands
    (3, 20, 4, "auto", "width"),
    (16, 16, 4, "height", "height"),
    (16, 16, 4, "width", "width"),
])
def test_band_axis_rule(h, w, n, axis, want):
    assert decoder.band_axis(h, w, n, axis) == want


@pytest.mark.parametrize("h,w,n,axis", [(3, 3, 4, "auto"), (3, 20, 4, "height"), (20, 3, 4, "width"),
                                        (8, 8, 0, "auto"), (8, 8, 2, "diagonal")])
def test_band_axis_rejects(h, w, n, axis):
    with pytest.raises(ValueError):
        decoder.band_axis(h, w, n, axis)


# ---- AutoencoderKLFlux2 latent front-end (inverse latent BatchNorm, 2x2 unpatchify) -----------
def test_unpatchify_inverts_pixel_unshuffle():
    """torch's pixel_unshuffle groups each channel's 2x2 patch into channels c*4 + py*2 + px; the
    oracle's unpatchify must invert it exactly."""
    x = np.random.default_rng(2).standard_normal((2, 3, 8, 6))
    from oracle import ops
    patched = F.pixel_unshuffle(torch.from_numpy(x), 2).numpy()
    np.testing.assert_array_equal(ops.unpatchify(patched, 2), x)
    np.testing.assert_array_equal(F.pixel_shuffle(torch.from_numpy(patched), 2).numpy(), ops.unpatchify(patched, 2))


def test_inverse_batch_norm_inverts_torch_batch_norm():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((2, 12, 5, 7))
    mean, var, eps = rng.normal(0, 0.5, 12), rng.uniform(0.25, 4.0, 12), 1e-4
    from oracle import ops
    y = ops.inverse_batch_norm(x, mean, var, eps)
    back = F.batch_norm(torch.from_numpy(y), torch.from_numpy(mean), torch.from_numpy(var), training=False,
                        eps=eps).numpy()
    np.testing.assert_allclose(back, x, rtol=1e-13, atol=1e-13)


FLUX2_SMALL = dataclasses.replace(KL_SMALL, latent_channels=8, latent_patch=2, latent_bn_eps=1e-4)


def test_flux2_decode_is_the_kl_decode_of_the_frontend_output():
    """The front-end is a pure prefix: decoding the patchified, normalised latent equals decoding
    (with the same decoder body) the latent that torch's batch_norm + pixel_unshuffle would turn
    into it."""
    W = synth.make_weights(FLUX2_SMALL, "fp32", seed=3)
    rng = np.random.default_rng(6)
    z = rng.standard_normal((1, 8, 6, 4))                                  # decoder-grid latent
    zp = F.pixel_unshuffle(torch.from_numpy(z), 2)
    zp = F.batch_norm(zp, torch.from_numpy(W["bn.running_mean"].astype(np.float64)),
                      torch.from_numpy(W["bn.running_var"].astype(np.float64)), training=False,
                      eps=FLUX2_SMALL.latent_bn_eps).numpy()                # what the pipeline hands in
    body = dataclasses.replace(FLUX2_SMALL, latent_patch=1)
    want = decoder.decode(body, W, z)
    got = decoder.decode(FLUX2_SMALL, W, zp)
    assert got.shape == decoder.output_shape(FLUX2_SMALL, zp.shape) == want.shape
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12 * np.abs(want).max())
    np.testing.assert_allclose(decoder.decode(FLUX2_SMALL, W, zp, 3), got, rtol=0,
                               atol=1e-12 * np.abs(got).max())

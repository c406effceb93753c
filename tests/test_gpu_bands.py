"""Band split axis on the GPU: height row bands, width column bands and the auto choice all give
the same bits ("VAE Parallel", Strategy Selection Contract: spatial_shard_height / _width / auto).

On one GPU a band only decides which queries one attention pass holds (a width band's queries are
gathered into a dense buffer and its output scattered back), so the whole decode must be bit for
bit the same for every axis and band count; the height-band decode itself is checked against the
float64 oracle in the other GPU tests, so equality carries that parity over.
"""
import pytest

import synth
from gpu_helpers import max_latent_for, require_gpu

pytestmark = pytest.mark.gpu

CASES = [
    ("kl", (1, 16, 64, 64), [4, 7]),          # 512x512 output, width bands of 16 / 10-9 columns
    ("kl", (2, 16, 40, 68), [3, 5]),          # batch 2, ragged width bands (23/23/22 columns)
    ("wan", (1, 16, 3, 24, 40), [3, 8]),      # per-frame attention, 9 output frames
]


@pytest.mark.parametrize("arch_name,shape,bands", CASES)
def test_width_bands_bitwise_equal_height_bands(arch_name, shape, bands):
    torch, rbl = require_gpu()
    arch = synth.KL_ZIMAGE if arch_name == "kl" else synth.WAN
    W = synth.make_weights(arch, "bf16")
    dec = rbl.Decoder(arch, W, "bf16", max_latent_for(shape))
    z = torch.from_numpy(synth.make_latent(shape, "bf16", seed=3)).cuda().to(torch.bfloat16).contiguous()
    ref = dec.decode(z, 1).clone()
    for n in bands:
        for axis in ("height", "width", "auto"):
            if axis == "height" and n > shape[-2]:
                continue
            out = dec.decode(z, n, axis=axis)
            torch.cuda.synchronize()
            dec.sync()
            assert bool((out == ref).all()), f"{axis} x {n} bands differs from the 1-band decode"
    dec.close()


def test_width_bands_beyond_the_width_rejected():
    torch, rbl = require_gpu()
    shape = (1, 16, 64, 8)
    dec = rbl.Decoder(synth.KL_ZIMAGE, synth.make_weights(synth.KL_ZIMAGE, "bf16"), "bf16", max_latent_for(shape))
    z = torch.from_numpy(synth.make_latent(shape, "bf16")).cuda().to(torch.bfloat16).contiguous()
    with pytest.raises(rbl.VaedecError):
        dec.decode(z, 9, axis="width")
    assert rbl.band_axis(shape, 9, "auto") == "height"
    out = dec.decode(z, 9, axis="auto")        # auto falls back to the height axis
    torch.cuda.synchronize()
    assert bool((out == dec.decode(z, 1)).all())
    dec.close()

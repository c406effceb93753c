"""vaedec_decode_host: host buffers in and out (copies inside the call, synchronous).

It gives the bits of the device-buffer decode and enqueues the same kernels, also on repeated calls,
after a change of shape or band count, and with per-op profiling on.
"""
import pytest

import synth
from gpu_helpers import require_gpu

pytestmark = pytest.mark.gpu


def _check(torch, dec, shape, n_bands, seed):
    z = synth.make_latent(shape, "bf16", seed=seed)
    n0 = dec.launch_count()
    ref = dec.decode(torch.from_numpy(z).cuda().to(torch.bfloat16), n_bands).cpu()
    torch.cuda.synchronize()
    n_dev = dec.launch_count() - n0
    zh = torch.from_numpy(z).to(torch.bfloat16).pin_memory()
    oh = torch.empty(dec.output_shape(shape), dtype=torch.bfloat16).pin_memory()
    n0 = dec.launch_count()
    dec.decode_host(zh, oh, n_bands)
    assert torch.equal(oh, ref), (shape, n_bands)
    # the same kernels as the device-buffer decode
    assert dec.launch_count() - n0 == n_dev


@pytest.mark.parametrize("arch_name,shapes,max_latent", [
    ("kl", [((1, 16, 12, 20), 3), ((1, 16, 16, 16), 2)], (1, 1, 16, 20)),
    ("wan", [((1, 16, 3, 24, 40), 3), ((1, 16, 2, 16, 24), 2)], (1, 3, 24, 40)),
])
def test_host_decode_matches_device_decode(arch_name, shapes, max_latent):
    torch, rbl = require_gpu()
    arch = synth.KL_ZIMAGE if arch_name == "kl" else synth.WAN
    dec = rbl.Decoder(arch, synth.make_weights(arch, "bf16"), "bf16", max_latent)
    for rnd in range(2):
        for i, (shape, nb) in enumerate(shapes):
            _check(torch, dec, shape, nb, seed=10 * rnd + i)
    dec.profile(True)
    _check(torch, dec, *shapes[0], seed=3)
    dec.profile(False)
    dec.sync()


def test_decode_checks_its_buffers():
    """Output buffers of the wrong place, shape or dtype are refused before any copy or launch (a host
    buffer too small for the output would otherwise be overrun by the download)."""
    torch, rbl = require_gpu()
    shape = (1, 16, 8, 8)
    W = synth.make_weights(synth.KL_ZIMAGE, "bf16")
    dec = rbl.Decoder(synth.KL_ZIMAGE, W, "bf16", (1, 1, 8, 8))
    z = torch.from_numpy(synth.make_latent(shape, "bf16")).to(torch.bfloat16)
    oshape = dec.output_shape(shape)
    zd = z.cuda()
    with pytest.raises(ValueError):
        dec.decode(zd, 1, out=torch.empty(oshape, dtype=torch.bfloat16))                  # host output
    with pytest.raises(ValueError):
        dec.decode(zd, 1, out=torch.empty((1, 3, 64, 32), dtype=torch.bfloat16, device="cuda"))
    with pytest.raises(ValueError):
        dec.decode(zd, 1, out=torch.empty(oshape, dtype=torch.float32, device="cuda"))
    with pytest.raises(ValueError):
        dec.decode_host(z, torch.empty((1, 3, 64, 32), dtype=torch.bfloat16), 1)          # too small
    with pytest.raises(ValueError):
        dec.decode_host(zd, torch.empty(oshape, dtype=torch.bfloat16), 1)                 # device latent
    out = dec.decode_host(z, torch.empty(oshape, dtype=torch.bfloat16), 1)
    assert tuple(out.shape) == tuple(oshape)
    dec.close()

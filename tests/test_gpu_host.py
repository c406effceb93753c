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

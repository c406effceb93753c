"""A decode captured into a CUDA graph replays with exactly the bits of the eager decode.

The library's decode is stream-ordered device work only (kernel launches on the caller's stream,
each programmatically dependent on the previous kernel), so a caller can capture it once and replay
it, the usual way to take per-launch host cost out of a serving loop.  The replay must also follow a new latent written
into the captured input buffer.
"""
import pytest

import synth
from gpu_helpers import max_latent_for, require_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("arch_name,shape,n_bands", [
    ("kl", (1, 16, 64, 64), 4),          # Z-Image decoder, 512x512 output, attention over 4096 keys
    ("wan", (1, 16, 3, 24, 40), 3),      # Wan causal decoder, 9 frames 192x320
])
def test_graph_replay_matches_eager(arch_name, shape, n_bands):
    torch, rbl = require_gpu()
    arch = synth.KL_ZIMAGE if arch_name == "kl" else synth.WAN
    W = synth.make_weights(arch, "bf16")
    dec = rbl.Decoder(arch, W, "bf16", max_latent_for(shape))
    z1 = torch.from_numpy(synth.make_latent(shape, "bf16", seed=11)).cuda().to(torch.bfloat16).contiguous()
    z2 = torch.from_numpy(synth.make_latent(shape, "bf16", seed=12)).cuda().to(torch.bfloat16).contiguous()
    eager1 = dec.decode(z1, n_bands).clone()
    eager2 = dec.decode(z2, n_bands).clone()
    torch.cuda.synchronize()
    dec.sync()

    zin = z1.clone()
    out = torch.empty_like(eager1)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        dec.decode(zin, n_bands, out=out, stream=s)   # warm-up outside the capture
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        dec.decode(zin, n_bands, out=out, stream=s)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    dec.sync()
    assert bool((out == eager1).all()), "graph replay differs from the eager decode"
    zin.copy_(z2)
    g.replay()
    torch.cuda.synchronize()
    dec.sync()
    assert bool((out == eager2).all()), "graph replay does not follow the new latent"
    dec.close()

"""GroupNorm through the no-allocation entry point (``vaedec_groupnorm_noalloc``).

That entry point exists for callers that cannot allocate device memory while the
op runs (plugin hosts that forbid cudaMalloc in their enqueue callback, real-time
pipelines with memory fixed at start-up, code under a foreign allocator): its
scratch is a fixed array inside the library instead of the decoder's workspace.
This test captures one GroupNorm op of a real decode (input and output, through
the C ABI's inspection call), runs the same normalisation twice in a row through
the no-allocation entry point, and requires both results to match the decoder's
within the per-op tolerance (they are in fact expected to be bit-identical: the
same kernels on the same input).  It also checks that sizes beyond the fixed
scratch are refused before anything is launched.  The file name sorts last so a
run that stops at the first failure has already run every other test.
"""
import numpy as np
import pytest

import synth
from gpu_helpers import Case, parse_shape, rel_l2, to_numpy

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def case():
    return Case(synth.KL_ZIMAGE, "bf16", (1, 16, 6, 12))


def _first_groupnorm(case, n_bands):
    for op in range(case.dec.num_ops(case.shape, n_bands)):
        d = case.dec.op_desc(case.shape, n_bands, op)
        if d["kind"] == "groupnorm" and d["in_dt"] == "f32":
            return op, d
    raise AssertionError("no groupnorm op")


def test_noalloc_groupnorm_matches_decoder_twice(case):
    import torch
    import row_band_layerwise_gb300 as rbl

    op, d = _first_groupnorm(case, 2)
    d_, x, _, y_ref = case.capture(2, op)
    B, T, H, W, C = parse_shape(d["in"])
    x_dev = torch.from_numpy(x.astype(np.float32)).reshape(B, T * H, W, C).cuda()
    gamma = torch.from_numpy(case.W[d["name"] + ".weight"]).float().cuda()
    beta = torch.from_numpy(case.W[d["name"] + ".bias"]).float().cuda()
    silu = d["silu"] == "1"
    outs = []
    for _ in range(2):
        y = torch.empty((B, T * H, W, C), dtype=torch.bfloat16, device="cuda")
        rbl.groupnorm_noalloc(x_dev, y, int(d["groups"]), gamma, beta, synth.KL_ZIMAGE.eps, silu)
        torch.cuda.synchronize()
        outs.append(to_numpy(y).reshape(-1))
    for got in outs:
        assert rel_l2(got, y_ref) <= 6e-3
        np.testing.assert_array_equal(got, y_ref)
    np.testing.assert_array_equal(outs[0], outs[1])


def test_noalloc_rejects_sizes_beyond_the_scratch():
    import torch
    import row_band_layerwise_gb300 as rbl

    x = torch.empty((1, 8192, 1, 32), dtype=torch.float32, device="cuda")   # rows * G = 262144 > 131072
    y = torch.empty_like(x, dtype=torch.bfloat16)
    g = torch.ones(32, device="cuda")
    b = torch.zeros(32, device="cuda")
    with pytest.raises(rbl.VaedecError, match="scratch limit"):
        rbl.groupnorm_noalloc(x, y, 32, g, b, 1e-6, True)

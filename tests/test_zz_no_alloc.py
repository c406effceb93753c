"""GroupNorm through the no-allocation entry point (``vaedec_groupnorm_noalloc``).

That entry point exists for callers that cannot allocate device memory while the
op runs (plugin hosts that forbid cudaMalloc in their enqueue callback, real-time
pipelines with memory fixed at start-up, code under a foreign allocator): its
scratch is a fixed array inside the library instead of the decoder's workspace.

The tests run it twice in a row on seeded inputs and check each result against
the float64 oracle's GroupNorm (+ SiLU), for every dtype pair it takes, with and
without SiLU, for groups narrower than one 8-channel vector (C/G = 4) and wider
ones; the two calls must agree bit for bit.  One test also captures a GroupNorm
op of a real decode through the C ABI's inspection call and requires the
entry point to reproduce the decoder's own output.  Sizes beyond the fixed
scratch and malformed tensors are refused before anything is launched.  The
file name sorts last so a run that stops at the first failure has already run
every other test.
"""
import numpy as np
import pytest

import synth
from gpu_helpers import Case, parse_shape, rel_l2, to_numpy
from oracle import ops

pytestmark = pytest.mark.gpu

# per-op bars: one bf16 rounding of the output, or fp32 arithmetic against float64
TOL = {"bf16": 6e-3, "fp32": 1e-5}


def _torch_rbl():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import row_band_layerwise_gb300 as rbl
    from gpu_helpers import require_gpu
    require_gpu()
    return torch, rbl


@pytest.mark.parametrize("in_dt,out_dt", [("fp32", "bf16"), ("bf16", "bf16"), ("fp32", "fp32")])
@pytest.mark.parametrize("silu", [True, False])
@pytest.mark.parametrize("shape,G", [((2, 6, 40, 128), 32), ((1, 5, 24, 512), 32), ((1, 3, 16, 64), 8)])
def test_noalloc_groupnorm_matches_oracle_twice(in_dt, out_dt, silu, shape, G):
    torch, rbl = _torch_rbl()
    B, rows, W, C = shape
    rng = np.random.default_rng(11)
    x = rng.standard_normal(shape) * 1.5 + 0.3
    gamma = rng.uniform(0.5, 1.5, C)
    beta = rng.uniform(-0.2, 0.2, C)
    tdt = {"fp32": torch.float32, "bf16": torch.bfloat16}
    x_dev = torch.from_numpy(x.astype(np.float32)).to("cuda").to(tdt[in_dt]).contiguous()
    x_used = to_numpy(x_dev)                                 # the values the kernel reads
    g_dev = torch.from_numpy(gamma.astype(np.float32)).cuda()
    b_dev = torch.from_numpy(beta.astype(np.float32)).cuda()
    g_used, b_used = to_numpy(g_dev), to_numpy(b_dev)
    # oracle on channels-first [B, C, rows, W]
    ref = ops.group_norm(np.moveaxis(x_used, -1, 1), G, g_used, b_used, 1e-6)
    if silu:
        ref = ops.silu(ref)
    ref = np.moveaxis(ref, 1, -1)
    outs = []
    for _ in range(2):
        y = torch.empty(shape, dtype=tdt[out_dt], device="cuda")
        rbl.groupnorm_noalloc(x_dev, y, G, g_dev, b_dev, 1e-6, silu)
        torch.cuda.synchronize()
        outs.append(to_numpy(y))
    for got in outs:
        err = rel_l2(got, ref)
        assert err <= TOL[out_dt], f"rel-L2 {err:.3e}"
    np.testing.assert_array_equal(outs[0], outs[1])


def test_noalloc_groupnorm_matches_decoder_op():
    torch, rbl = _torch_rbl()
    case = Case(synth.KL_ZIMAGE, "bf16", (1, 16, 6, 12))
    op = next(i for i in range(case.dec.num_ops(case.shape, 2))
              if case.dec.op_desc(case.shape, 2, i)["kind"] == "groupnorm"
              and case.dec.op_desc(case.shape, 2, i)["in_dt"] == "f32")
    d, x, _, y_ref = case.capture(2, op)
    B, T, H, W, C = parse_shape(d["in"])
    x_dev = torch.from_numpy(x.astype(np.float32)).reshape(B, T * H, W, C).cuda()
    gamma = torch.from_numpy(case.W[d["name"] + ".weight"]).float().cuda()
    beta = torch.from_numpy(case.W[d["name"] + ".bias"]).float().cuda()
    for _ in range(2):
        y = torch.empty((B, T * H, W, C), dtype=torch.bfloat16, device="cuda")
        rbl.groupnorm_noalloc(x_dev, y, int(d["groups"]), gamma, beta, synth.KL_ZIMAGE.eps, d["silu"] == "1")
        torch.cuda.synchronize()
        np.testing.assert_array_equal(to_numpy(y).reshape(-1), y_ref)
    case.dec.close()


def test_noalloc_rejects_sizes_beyond_the_scratch_and_bad_tensors():
    torch, rbl = _torch_rbl()
    x = torch.empty((1, 8192, 1, 32), dtype=torch.float32, device="cuda")   # rows * G = 262144 > 131072
    y = torch.empty_like(x, dtype=torch.bfloat16)
    g = torch.ones(32, device="cuda")
    b = torch.zeros(32, device="cuda")
    with pytest.raises(rbl.VaedecError, match="scratch limit"):
        rbl.groupnorm_noalloc(x, y, 32, g, b, 1e-6, True)
    x = torch.zeros((1, 4, 8, 32), dtype=torch.float32, device="cuda")
    with pytest.raises(ValueError):                                           # y too small
        rbl.groupnorm_noalloc(x, torch.empty((1, 4, 4, 32), device="cuda"), 8, g, b, 1e-6, True)
    with pytest.raises(ValueError):                                           # gamma too short
        rbl.groupnorm_noalloc(x, torch.empty_like(x), 8, g[:16], b, 1e-6, True)
    with pytest.raises(ValueError):                                           # not contiguous
        rbl.groupnorm_noalloc(x.transpose(1, 2), torch.empty_like(x).transpose(1, 2), 8, g, b, 1e-6, True)
    with pytest.raises(ValueError):                                           # host tensor
        rbl.groupnorm_noalloc(x.cpu(), torch.empty_like(x), 8, g, b, 1e-6, True)

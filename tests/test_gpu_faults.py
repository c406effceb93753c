"""Failure handling on the GPU, with no GPU fault, trap or hang.

* Allocation failures injected on the host make vaedec_create return OOM after
  releasing everything it had allocated (device free memory is unchanged), and a
  following create works.
* A refused kernel launch makes the decode return an error; the next decode on
  the same handle is bit-identical to a clean one.
* A kernel whose bounded wait is on a barrier nothing completes (the same wait
  the decode kernels use, its limit lowered to 1 ms) records a timeout in the
  handle's status word and returns; vaedec_sync reports TIMEOUT once and the
  same handle then decodes bit-identically again.
"""
import numpy as np
import pytest

import synth
from gpu_helpers import Case, require_gpu

pytestmark = pytest.mark.gpu

SHAPE = (1, 16, 8, 16)   # widths where the channel-major conv, the GEMM and the narrow conv all run


@pytest.fixture(scope="module")
def case():
    return Case(synth.KL_ZIMAGE, "bf16", SHAPE)


@pytest.fixture(scope="module")
def clean(case):
    return case.decode(2).cpu()


def _free_bytes(torch):
    torch.cuda.synchronize()
    return torch.cuda.mem_get_info()[0]


def test_injected_allocation_failure_releases_everything(case):
    torch, rbl = require_gpu()
    W = case.W
    before = _free_bytes(torch)
    for nth in (1, 5, 17):
        rbl.inject_fault("alloc", nth)
        with pytest.raises(rbl.VaedecError) as ei:
            rbl.Decoder(synth.KL_ZIMAGE, W, "bf16", (1, 1, SHAPE[2], SHAPE[3]))
        assert ei.value.status == 3   # OOM
        assert abs(_free_bytes(torch) - before) <= 2 << 20
    rbl.inject_fault("off")
    dec = rbl.Decoder(synth.KL_ZIMAGE, W, "bf16", (1, 1, SHAPE[2], SHAPE[3]))
    out = dec.decode(case.z_dev, 2)
    torch.cuda.synchronize()
    dec.sync()
    assert bool((out.cpu() == case.decode(2).cpu()).all())
    dec.close()


def test_refused_launch_then_clean_decode(case, clean):
    torch, rbl = require_gpu()
    rbl.inject_fault("launch", 7)
    with pytest.raises(rbl.VaedecError) as ei:
        case.decode(2)
    assert ei.value.status == 4   # CUDA
    rbl.inject_fault("off")
    assert bool((case.decode(2).cpu() == clean).all())


def test_bounded_wait_runs_out_and_the_handle_recovers(case, clean):
    torch, rbl = require_gpu()
    rbl.set_wait_limit(1_000_000)   # 1 ms
    try:
        case.dec.wait_probe()
        torch.cuda.synchronize()
        with pytest.raises(rbl.VaedecError) as ei:
            case.dec.sync()
        assert ei.value.status == 5   # TIMEOUT
        case.dec.sync()               # the status word was cleared when it was reported
    finally:
        rbl.set_wait_limit(0)
    assert bool((case.decode(2).cpu() == clean).all())


@pytest.mark.parametrize("axis", ["height", "width"])
def test_refused_launch_at_every_point_of_the_attention_op(case, clean, axis):
    """A decode stopped at any launch inside the attention op (norm, projections, width-band
    gathers, the fused attention kernel, its key-split merge, scatters, output projection) leaves
    nothing half-done that the next decode could see: the next decode on the same handle is
    bit-identical to a clean one."""
    torch, rbl = require_gpu()
    n_bands = 4
    ops = case.dec.ops(SHAPE, n_bands)
    # launches before the attention op = launches of a decode stopped just before it
    first = None
    total = 0
    counts = []
    for i, d in enumerate(ops):
        if d["kind"] == "attention":
            first = i
            break
    assert first is not None
    before = case.dec.launch_count()
    case.dec.run_until(case.z_dev, n_bands, first - 1)
    torch.cuda.synchronize()
    n_pre = case.dec.launch_count() - before
    before = case.dec.launch_count()
    case.dec.run_until(case.z_dev, n_bands, first)
    torch.cuda.synchronize()
    n_attn = case.dec.launch_count() - before - n_pre
    assert n_attn > 6
    for k in range(1, n_attn + 1):
        rbl.inject_fault("launch", n_pre + k)
        with pytest.raises(rbl.VaedecError):
            case.dec.decode(case.z_dev, n_bands, axis=axis)
        rbl.inject_fault("off")
        torch.cuda.synchronize()
        out = case.dec.decode(case.z_dev, n_bands, axis=axis)
        torch.cuda.synchronize()
        case.dec.sync()
        assert bool((out.cpu() == clean).all()), f"stop at attention launch {k}"

"""C-ABI checks that need no GPU: the library loads, exports every symbol the
header declares, and rejects bad arguments on the host before touching CUDA."""
import ctypes
import os
import re

import pytest

import synth
import row_band_layerwise_gb300 as rbl
from row_band_layerwise_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "vaedec.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(build.lib_path()):
        build.build()
    return rbl.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(vaedec_[a-z_]+)\s*\(", text)))


def test_header_declares_the_binding_symbols():
    assert declared_functions() == sorted(rbl.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_create_rejects_bad_config_without_cuda(lib):
    cfg = rbl.make_config(synth.KL_TINY, "fp32", (1, 1, 16, 16))
    h = ctypes.c_void_p()
    cfg.family = 7
    assert lib.vaedec_create(ctypes.byref(cfg), None, 0, ctypes.byref(h)) == 1
    assert b"family" in lib.vaedec_last_error()
    cfg = rbl.make_config(synth.KL_TINY, "fp32", (1, 1, 16, 16))
    cfg.norm_groups = 5   # does not divide 64
    assert lib.vaedec_create(ctypes.byref(cfg), None, 0, ctypes.byref(h)) == 1
    cfg = rbl.make_config(synth.KL_TINY, "bf16", (1, 1, 16, 16))   # latent channels 4: not a bf16 tile
    assert lib.vaedec_create(ctypes.byref(cfg), None, 0, ctypes.byref(h)) == 2
    cfg = rbl.make_config(synth.KL_TINY, "fp32", (1, 2, 16, 16))   # T must be 1 for the 2D decoder
    assert lib.vaedec_create(ctypes.byref(cfg), None, 0, ctypes.byref(h)) == 1
    assert not h.value


def test_null_arguments_rejected(lib):
    assert lib.vaedec_create(None, None, 0, None) == 1
    assert lib.vaedec_decode(None, None, None, 0, None, 1, None) == 1
    assert lib.vaedec_sync(None, None) == 1
    lib.vaedec_destroy(None)


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(RuntimeError, match="not built"):
        rbl.load_library(str(tmp_path / "nope.so"))


def test_fault_injection_arguments_checked_without_cuda(lib):
    assert lib.vaedec_debug_inject_fault(7, 1) == 1
    assert lib.vaedec_debug_inject_fault(1, 0) == 1
    assert lib.vaedec_debug_inject_fault(0, 0) == 0


@pytest.mark.parametrize("shape", [(1, 16, 128, 128), (2, 16, 100, 136), (1, 16, 136, 100), (1, 16, 5, 60, 104),
                                   (1, 4, 20, 3), (1, 4, 3, 20)])
@pytest.mark.parametrize("n_bands", [1, 3, 4, 8])
@pytest.mark.parametrize("axis", ["height", "width", "auto"])
def test_band_axis_rule_matches_the_oracle(lib, shape, n_bands, axis):
    """vaedec_band_axis (host logic) makes the same choice as the oracle's rule, and rejects
    exactly the requests the rule rejects."""
    from oracle import decoder
    h, w = shape[-2], shape[-1]
    try:
        want = decoder.band_axis(h, w, n_bands, axis)
    except ValueError:
        with pytest.raises(rbl.VaedecError):
            rbl.band_axis(shape, n_bands, axis)
        return
    assert rbl.band_axis(shape, n_bands, axis) == want


def test_band_axis_rejects_bad_arguments(lib):
    out = ctypes.c_int(-1)
    shp = (ctypes.c_int64 * 4)(1, 16, 8, 8)
    assert lib.vaedec_band_axis(shp, 4, 2, 7, ctypes.byref(out)) != 0      # unknown axis
    assert lib.vaedec_band_axis(shp, 3, 2, 0, ctypes.byref(out)) != 0      # ndim
    assert lib.vaedec_band_axis(shp, 4, 0, 2, ctypes.byref(out)) != 0      # n_bands < 1
    assert lib.vaedec_band_axis(None, 4, 2, 2, ctypes.byref(out)) != 0


def test_latent_frontend_config_checked_without_cuda(lib):
    import dataclasses
    h = ctypes.c_void_p()
    flux = dataclasses.replace(synth.KL_TINY, latent_patch=2, latent_bn_eps=1e-4)
    cfg = rbl.make_config(flux, "fp32", (1, 1, 8, 8))
    cfg.latent_patch = 3                                    # only 2x2 patches
    assert lib.vaedec_create(ctypes.byref(cfg), None, 0, ctypes.byref(h)) == 2
    cfg = rbl.make_config(flux, "fp32", (1, 1, 8, 8))
    cfg.latent_bn_eps = 0.0
    assert lib.vaedec_create(ctypes.byref(cfg), None, 0, ctypes.byref(h)) == 1
    cfg = rbl.make_config(dataclasses.replace(synth.WAN, latent_patch=2), "bf16", (1, 2, 8, 8))
    assert lib.vaedec_create(ctypes.byref(cfg), None, 0, ctypes.byref(h)) == 1   # a KL2D option only
    assert not h.value


def test_bf16_attention_width_checked_without_cuda(lib):
    """The bf16 path's fused mid-block attention takes a multiple of 128 channels up to 512:
    other widths are refused at create time, before any device work."""
    import dataclasses
    h = ctypes.c_void_p()
    narrow = dataclasses.replace(synth.KL_TINY, latent_channels=16, mid_channels=64, stage_channels=(64,))
    cfg = rbl.make_config(narrow, "bf16", (1, 1, 16, 16))
    assert lib.vaedec_create(ctypes.byref(cfg), None, 0, ctypes.byref(h)) == 2
    assert b"128" in lib.vaedec_last_error()
    wide = dataclasses.replace(narrow, mid_channels=640, stage_channels=(640,))
    cfg = rbl.make_config(wide, "bf16", (1, 1, 16, 16))
    assert lib.vaedec_create(ctypes.byref(cfg), None, 0, ctypes.byref(h)) == 2
    assert not h.value


def test_band_attention_workspace_and_arguments_checked_without_cuda(lib):
    """Host logic of vaedec_band_attention: the key-split workspace size (one split per 2048 keys,
    at most 4; each split holds an fp32 output row and a (max, sum) pair per query) and the argument
    checks, all before any device work (the pointers below are never dereferenced)."""
    n = ctypes.c_size_t(7)
    assert lib.vaedec_band_attention_work_bytes(1, 128, 128, 512, ctypes.byref(n)) == 0
    assert n.value == 4 * 16384 * (512 * 4 + 8)
    assert lib.vaedec_band_attention_work_bytes(5, 60, 104, 384, ctypes.byref(n)) == 0
    assert n.value == 3 * 5 * 6240 * (384 * 4 + 8)
    assert lib.vaedec_band_attention_work_bytes(1, 32, 32, 512, ctypes.byref(n)) == 0
    assert n.value == 0                                     # 1024 keys: one split, no workspace
    assert lib.vaedec_band_attention_work_bytes(0, 8, 8, 512, ctypes.byref(n)) != 0
    fake = ctypes.c_void_p(1 << 20)                         # 16-byte aligned, never touched
    st = ctypes.c_void_p(1 << 21)
    call = lib.vaedec_band_attention
    assert call(None, fake, fake, fake, 1, 8, 8, 512, 1, None, 0, st, None) == 1           # NULL q
    assert call(fake, fake, fake, fake, 1, 8, 8, 512, 1, None, 0, None, None) == 1         # NULL status
    assert call(fake, fake, fake, fake, 1, 8, 8, 96, 1, None, 0, st, None) == 1            # C not x128
    assert call(fake, fake, fake, fake, 1, 8, 8, 1024, 1, None, 0, st, None) == 1          # C > 512
    assert call(fake, fake, fake, fake, 1, 3, 5, 512, 1, None, 0, st, None) == 1           # 15 keys
    assert call(fake, fake, fake, fake, 1, 8, 8, 512, 9, None, 0, st, None) == 1           # bands > rows
    assert call(fake, fake, fake, fake, 1, 8, 8, 512, 0, None, 0, st, None) == 1           # no bands
    assert call(ctypes.c_void_p((1 << 20) + 8), fake, fake, fake, 1, 8, 8, 512, 1, None, 0, st,
                None) == 1                                                                # misaligned
    assert call(fake, fake, fake, fake, 1, 64, 64, 512, 1, None, 0, st, None) == 1        # needs work
    assert b"work" in lib.vaedec_last_error()


def test_workspace_plan_is_the_largest_layers_live_set(lib):
    """The band scheduler's workspace (row a15): every activation and the attention's scratch share
    one arena, placed by lifetime.  For the Z-Image decoder the largest live set is the first
    GroupNorm of the last stage at full resolution: its fp32 input (256 channels), the bf16
    normalised output and the bf16 operand copy for the fused 1x1 shortcut, i.e.
    B * H_out * W_out * 256 * (4 + 2 + 2) bytes; the placement reaches that bound exactly (plus a
    1 MiB guard), and everything else the handle owns is small."""
    mib = 1 << 20
    for name in ("kl_zimage_512", "kl_zimage_1024", "kl_zimage_b2_800x1088", "flux2_1024"):
        w = synth.WORKLOADS[name]
        b, _, h, wd = w.latent_shape
        p = w.arch.latent_patch
        h_out, w_out = h * p * 8, wd * p * 8
        plan = rbl.plan_workspace(w.arch, w.dtype, (b, 1, h, wd))
        assert plan["peak_live"] == b * h_out * w_out * 256 * 8, name
        assert plan["arena"] == plan["peak_live"] + mib, name
        assert plan["peak_live"] <= plan["bytes"] <= plan["arena"] + 40 * mib, (name, plan)
    # the 1024x1024 decode: 2.07 GiB in all (five whole-image buffers used to take 5.6 GB)
    w = synth.WORKLOADS["kl_zimage_1024"]
    assert rbl.plan_workspace(w.arch, w.dtype, (1, 1, 128, 128))["bytes"] <= 2.2e9
    # linear in the pixel count: twice the width, twice the arena
    a1 = rbl.plan_workspace(w.arch, w.dtype, (1, 1, 64, 64))["peak_live"]
    a2 = rbl.plan_workspace(w.arch, w.dtype, (1, 1, 64, 128))["peak_live"]
    assert a2 == 2 * a1


def test_workspace_plan_rejects_bad_configs(lib):
    cfg = rbl.make_config(synth.KL_TINY, "fp32", (1, 1, 16, 16))
    cfg.family = 7
    n = ctypes.c_size_t()
    assert lib.vaedec_plan_workspace(ctypes.byref(cfg), ctypes.byref(n), None, None) == 1
    assert lib.vaedec_plan_workspace(None, ctypes.byref(n), None, None) == 1
    cfg = rbl.make_config(synth.WAN, "bf16", (1, 5, 60, 104))
    assert lib.vaedec_plan_workspace(ctypes.byref(cfg), ctypes.byref(n), None, None) == 0
    assert n.value > 0


def test_band_attention_binding_checks_operands_without_cuda():
    """The binding rejects operands it cannot pass safely as raw pointers (host tensors, wrong shapes
    or dtypes) before the library sees them."""
    torch = pytest.importorskip("torch")
    import row_band_layerwise_gb300 as rbl
    q = torch.zeros((1, 64, 128), dtype=torch.bfloat16)
    vt = torch.zeros((1, 128, 64), dtype=torch.bfloat16)
    st = torch.zeros(1, dtype=torch.int32)
    with pytest.raises(ValueError):
        rbl.band_attention(q, q, vt, q, 8, 8, 1, None, st)            # host tensors
    with pytest.raises(ValueError):
        rbl.band_attention(q[0], q, vt, q, 8, 8, 1, None, st)         # q not [F, ntok, C]
    with pytest.raises(ValueError):
        rbl.band_attention(q, q, vt, q, 8, 7, 1, None, st)            # tokens do not fill the grid

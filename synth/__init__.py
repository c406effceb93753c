"""Seeded synthetic inputs for the layerwise row-band VAE decode.

This module is shared by the oracle, the tests and the benchmark.  It holds
no arithmetic of the decode itself: only the workload definitions (decoder
hyper-parameters, latent shapes, band counts), the weight naming and shapes,
and seeded random generation of latents and weights.

Weights are drawn in a fixed order from ``numpy.random.default_rng(seed)``:
every conv / linear weight and bias is U(-1/sqrt(fan_in), 1/sqrt(fan_in)) with
fan_in = C_in * k_t * k_h * k_w; every norm scale is 1 and every norm shift is
0.  Latents are N(0, 1) from ``default_rng(seed)``.  For bf16 workloads both
are rounded to bf16 (round-to-nearest-even) and kept as float32 arrays that
hold bf16-exact values.

Weight names follow the Diffusers state-dict keys of ``Decoder`` (the
AutoencoderKL 2D decoder) and ``WanDecoder3d`` (the Wan causal 3D decoder).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, List, Tuple

import numpy as np

__all__ = [
    "Arch", "Workload", "WORKLOADS", "weight_spec", "make_weights",
    "make_latent", "round_bf16",
]


@dataclass(frozen=True)
class Arch:
    """Decoder hyper-parameters shared by both families.

    Stage ``s`` runs ``stage_resnets[s]`` residual blocks ending at
    ``stage_channels[s]`` channels, then an optional upsample
    (0 = none, 1 = nearest-2x in space, 2 = temporal 2x + nearest-2x in space)
    whose 3x3 conv maps to ``stage_up_channels[s]`` channels.  The input
    channel count of stage ``s`` is ``mid_channels`` for s = 0, else the
    channel count leaving stage ``s - 1``.
    """

    family: str                      # "kl2d" | "wan3d"
    latent_channels: int
    mid_channels: int
    stage_channels: Tuple[int, ...]
    stage_resnets: Tuple[int, ...]
    stage_upsample: Tuple[int, ...]
    stage_up_channels: Tuple[int, ...]
    norm_groups: int = 32            # GroupNorm groups (kl2d only)
    eps: float = 1e-6                # GroupNorm epsilon (kl2d only)
    out_channels: int = 3
    # AutoencoderKLFlux2-style front-end (kl2d only): the decode input is the 2x2-patchified latent
    # (latent_patch**2 * latent_channels channels on a half-size grid) normalised by an inference
    # BatchNorm without affine terms (weights bn.running_mean / bn.running_var)
    latent_patch: int = 1
    latent_bn_eps: float = 1e-4

    def stage_in_channels(self) -> List[int]:
        cins = []
        c = self.mid_channels
        for s in range(len(self.stage_channels)):
            cins.append(c)
            c = self.stage_up_channels[s] if self.stage_upsample[s] else self.stage_channels[s]
        return cins

    def final_channels(self) -> int:
        s = len(self.stage_channels) - 1
        return self.stage_up_channels[s] if self.stage_upsample[s] else self.stage_channels[s]


# Tiny AutoencoderKL-style decoder: conv_in 4->64, mid (resnet, attn, resnet)
# at 64, one up stage (1 resnet 64->64, nearest-2x + conv3x3 64->32),
# GroupNorm(8) -> SiLU -> conv_out 32->3.
KL_TINY = Arch(
    family="kl2d", latent_channels=4, mid_channels=64,
    stage_channels=(64,), stage_resnets=(1,), stage_upsample=(1,),
    stage_up_channels=(32,), norm_groups=8, eps=1e-6,
)

# FLUX.1 / Z-Image AutoencoderKL decoder: block_out_channels (128,256,512,512)
# reversed for decoding, 3 resnets per up block, upsample after the first three.
KL_ZIMAGE = Arch(
    family="kl2d", latent_channels=16, mid_channels=512,
    stage_channels=(512, 512, 256, 128), stage_resnets=(3, 3, 3, 3),
    stage_upsample=(1, 1, 1, 0), stage_up_channels=(512, 512, 256, 0),
    norm_groups=32, eps=1e-6,
)

# FLUX.2-style AutoencoderKLFlux2 decoder: the Z-Image / FLUX.1 decoder body with 32 latent
# channels, fed through the latent front-end (inverse BatchNorm over the 128 patchified channels,
# then 2x2 unpatchify).
FLUX2 = Arch(
    family="kl2d", latent_channels=32, mid_channels=512,
    stage_channels=(512, 512, 256, 128), stage_resnets=(3, 3, 3, 3),
    stage_upsample=(1, 1, 1, 0), stage_up_channels=(512, 512, 256, 0),
    norm_groups=32, eps=1e-6, latent_patch=2, latent_bn_eps=1e-4,
)

# Wan 2.1 VAE decoder: base dim 96, dim_mult (1,2,4,4); stages 0 and 1 end in a
# temporal+spatial upsample, stage 2 in a spatial-only upsample; each upsample
# conv halves the channels.
WAN = Arch(
    family="wan3d", latent_channels=16, mid_channels=384,
    stage_channels=(384, 384, 192, 96), stage_resnets=(3, 3, 3, 3),
    stage_upsample=(2, 2, 1, 0), stage_up_channels=(192, 192, 96, 0),
    norm_groups=0, eps=0.0,
)


@dataclass(frozen=True)
class Workload:
    name: str
    arch: Arch
    dtype: str                              # "fp32" | "bf16"
    latent_shape: Tuple[int, ...]           # NCHW or NCTHW
    n_bands: int
    description: str = ""


WORKLOADS: Dict[str, Workload] = {
    w.name: w for w in [
        Workload("kl_tiny_fp32", KL_TINY, "fp32", (1, 4, 16, 16), 2,
                 "tiny AutoencoderKL-style decoder, 16x16 latent -> 32x32, fp32, 2 bands"),
        Workload("kl_zimage_512", KL_ZIMAGE, "bf16", (1, 16, 64, 64), 4,
                 "Z-Image AutoencoderKL decoder, 64x64 latent -> 512x512, bf16, 4 bands"),
        Workload("kl_zimage_1024", KL_ZIMAGE, "bf16", (1, 16, 128, 128), 8,
                 "Z-Image AutoencoderKL decoder, 128x128 latent -> 1024x1024, bf16, 8 bands"),
        Workload("kl_zimage_b2_800x1088", KL_ZIMAGE, "bf16", (2, 16, 100, 136), 3,
                 "Z-Image AutoencoderKL decoder, batch 2, 100x136 latent -> 800x1088, bf16, "
                 "3 uneven bands (34/33/33)"),
        Workload("wan_17x480x832", WAN, "bf16", (1, 16, 5, 60, 104), 4,
                 "Wan causal 3D decoder, 5x60x104 latent -> 17x480x832, bf16, 4 bands"),
        Workload("flux2_1024", FLUX2, "bf16", (1, 128, 64, 64), 8,
                 "FLUX.2-style decoder, patchified 128x64x64 latent (32x128x128 after the front-end) "
                 "-> 1024x1024, bf16, 8 bands"),
    ]
}


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); returns float32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) & 0xFFFF0000
    return u.astype(np.uint32).view(np.float32)


def _conv_entries(name: str, cin: int, cout: int, k: Tuple[int, ...]):
    fan_in = cin * int(np.prod(k))
    return [(name + ".weight", (cout, cin) + tuple(k), fan_in, "uniform"),
            (name + ".bias", (cout,), fan_in, "uniform")]


def _norm_entries_gn(name: str, c: int):
    return [(name + ".weight", (c,), 0, "ones"), (name + ".bias", (c,), 0, "zeros")]


def _norm_entries_rms(name: str, c: int):
    return [(name + ".gamma", (c,), 0, "ones")]


def weight_spec(arch: Arch) -> List[Tuple[str, Tuple[int, ...], int, str]]:
    """(name, shape, fan_in, init kind) for every parameter, in generation order."""
    spec: List = []
    if arch.family == "kl2d":
        k3, k1 = (3, 3), (1, 1)

        def resnet(prefix, cin, cout):
            e = _norm_entries_gn(prefix + ".norm1", cin)
            e += _conv_entries(prefix + ".conv1", cin, cout, k3)
            e += _norm_entries_gn(prefix + ".norm2", cout)
            e += _conv_entries(prefix + ".conv2", cout, cout, k3)
            if cin != cout:
                e += _conv_entries(prefix + ".conv_shortcut", cin, cout, k1)
            return e

        C = arch.mid_channels
        if arch.latent_patch > 1:
            cp = arch.latent_channels * arch.latent_patch ** 2
            spec += [("bn.running_mean", (cp,), 0, "bn_mean"), ("bn.running_var", (cp,), 0, "bn_var")]
        spec += _conv_entries("conv_in", arch.latent_channels, C, k3)
        spec += resnet("mid_block.resnets.0", C, C)
        a = "mid_block.attentions.0"
        spec += _norm_entries_gn(a + ".group_norm", C)
        for p in ("to_q", "to_k", "to_v", "to_out.0"):
            spec += [(f"{a}.{p}.weight", (C, C), C, "uniform"), (f"{a}.{p}.bias", (C,), C, "uniform")]
        spec += resnet("mid_block.resnets.1", C, C)
        cins = arch.stage_in_channels()
        for s, cout in enumerate(arch.stage_channels):
            cin = cins[s]
            for r in range(arch.stage_resnets[s]):
                spec += resnet(f"up_blocks.{s}.resnets.{r}", cin if r == 0 else cout, cout)
            if arch.stage_upsample[s]:
                spec += _conv_entries(f"up_blocks.{s}.upsamplers.0.conv", cout,
                                      arch.stage_up_channels[s], k3)
        cf = arch.final_channels()
        spec += _norm_entries_gn("conv_norm_out", cf)
        spec += _conv_entries("conv_out", cf, arch.out_channels, k3)
    elif arch.family == "wan3d":
        k3, k1 = (3, 3, 3), (1, 1, 1)

        def resnet(prefix, cin, cout):
            e = _norm_entries_rms(prefix + ".norm1", cin)
            e += _conv_entries(prefix + ".conv1", cin, cout, k3)
            e += _norm_entries_rms(prefix + ".norm2", cout)
            e += _conv_entries(prefix + ".conv2", cout, cout, k3)
            if cin != cout:
                e += _conv_entries(prefix + ".conv_shortcut", cin, cout, k1)
            return e

        C = arch.mid_channels
        spec += _conv_entries("conv_in", arch.latent_channels, C, k3)
        spec += resnet("mid_block.resnets.0", C, C)
        a = "mid_block.attentions.0"
        spec += _norm_entries_rms(a + ".norm", C)
        spec += _conv_entries(a + ".to_qkv", C, 3 * C, (1, 1))
        spec += _conv_entries(a + ".proj", C, C, (1, 1))
        spec += resnet("mid_block.resnets.1", C, C)
        cins = arch.stage_in_channels()
        for s, cout in enumerate(arch.stage_channels):
            cin = cins[s]
            for r in range(arch.stage_resnets[s]):
                spec += resnet(f"up_blocks.{s}.resnets.{r}", cin if r == 0 else cout, cout)
            if arch.stage_upsample[s] == 2:
                spec += _conv_entries(f"up_blocks.{s}.upsamplers.0.time_conv", cout, 2 * cout, (3, 1, 1))
            if arch.stage_upsample[s]:
                spec += _conv_entries(f"up_blocks.{s}.upsamplers.0.resample.1", cout,
                                      arch.stage_up_channels[s], (3, 3))
        cf = arch.final_channels()
        spec += _norm_entries_rms("norm_out", cf)
        spec += _conv_entries("conv_out", cf, arch.out_channels, k3)
    else:
        raise ValueError(f"unknown family {arch.family!r}")
    return spec


def make_weights(arch: Arch, dtype: str, seed: int = 1) -> Dict[str, np.ndarray]:
    """Seeded random-init weights as float32 arrays (bf16-exact when dtype is bf16)."""
    rng = np.random.default_rng(seed)
    out: Dict[str, np.ndarray] = {}
    for name, shape, fan_in, kind in weight_spec(arch):
        if kind == "uniform":
            bound = 1.0 / np.sqrt(fan_in)
            v = rng.uniform(-bound, bound, size=shape).astype(np.float32)
        elif kind == "ones":
            v = np.ones(shape, np.float32)
        elif kind == "bn_mean":
            v = rng.normal(0.0, 0.5, size=shape).astype(np.float32)
        elif kind == "bn_var":
            v = rng.uniform(0.25, 4.0, size=shape).astype(np.float32)
        else:
            v = np.zeros(shape, np.float32)
        out[name] = round_bf16(v) if dtype == "bf16" else v
    return out


def make_latent(shape: Tuple[int, ...], dtype: str, seed: int = 0) -> np.ndarray:
    """Seeded N(0,1) latent as float32 (bf16-exact when dtype is bf16)."""
    rng = np.random.default_rng(seed)
    z = rng.standard_normal(size=shape).astype(np.float32)
    return round_bf16(z) if dtype == "bf16" else z

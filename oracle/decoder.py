"""The two decoders, unbanded or as the pages' banded layer-wise algorithm.

Architecture readings (the pages name the decoders but do not spell out
their blocks; the plainest reading of the Diffusers modules is taken):

AutoencoderKL-style 2D decoder (Diffusers ``Decoder``)
  conv_in 3x3 -> mid [resnet, attention, resnet] -> up stages (resnets, then
  optional nearest-2x + conv3x3) -> GroupNorm -> SiLU -> conv_out 3x3.
  resnet(x) = shortcut(x) + conv2(SiLU(GN2(conv1(SiLU(GN1(x)))))), shortcut a
  1x1 conv when channels change, else identity.
  attention(x) = x + W_o softmax(Q K^T / sqrt(C)) V + b_o with
  Q, K, V = W_{q,k,v} GN(x) + b: one head over all H*W tokens.

WanDecoder3d-style causal 3D decoder
  Causal 3x3x3 convs (time padded (2, 0), space 1), channel RMSNorm, per-frame
  attention (RMSNorm -> 1x1 to_qkv -> softmax attention over one frame's
  tokens -> 1x1 proj + residual), upsample3d = time_conv (causal 3x1x1,
  C -> 2C) over frames 1..T-1 with frame 0 passed through, each frame's two
  channel halves becoming two consecutive frames, then nearest-2x + Conv2d 3x3
  per frame; upsample2d = the spatial part only.  The frame-chunked causal
  cache of the original module equals this whole-sequence causal form.

Banded mode runs "VAEP：VAE 并行解码" / "Static Layer-Wise VAE Decode" as
written: the latent height is cut into row bands (section 按高度分片，逐层解码;
table "Semantics and Communication"); every conv takes kernel-radius halo rows
from the adjacent bands and zero padding only at the global top/bottom edge
(section 卷积：交换边界行); GroupNorm computes per-band central moments and
merges them with the element-count-weighted rule (section GroupNorm：合并全局统计量);
attention keeps Q band-local and attends over K/V gathered from all bands
(section Attention：本地 Q，全局 K/V); pointwise ops, channel RMSNorm and
nearest upsample run per band.  The same algorithm runs over width column bands
(the pages' second spatial split axis, "Parallel modes": spatial_shard_width):
halo columns from the left/right neighbours, zero padding only at the global
left/right edge, height padded as in the original.

TEST INFRASTRUCTURE ONLY: see the package docstring.
"""
from __future__ import annotations

from typing import Dict, List, Optional, Sequence, Tuple

import numpy as np

from . import ops


def band_axis(h: int, w: int, n_bands: int, axis: str) -> str:
    """The split axis a request gets: "height", "width", or for "auto" the longer latent axis
    that can hold every band (at least one latent row or column each), width winning ties
    ("Parallel modes", auto: the longer axis that can cover every rank, width wins ties).
    Raises ValueError when the requested axis (or, for auto, neither axis) can hold n_bands."""
    if n_bands < 1:
        raise ValueError("n_bands must be >= 1")
    if axis == "height":
        if n_bands > h:
            raise ValueError(f"n_bands={n_bands} exceeds the latent height {h}")
        return axis
    if axis == "width":
        if n_bands > w:
            raise ValueError(f"n_bands={n_bands} exceeds the latent width {w}")
        return axis
    if axis != "auto":
        raise ValueError(axis)
    fits = [a for a, n in (("width", w), ("height", h)) if n >= n_bands]
    if not fits:
        raise ValueError(f"neither axis ({h} x {w}) can hold {n_bands} bands")
    return max(fits, key=lambda a: w if a == "width" else h)   # first maximum: width on ties


def band_rows(h: int, n_bands: int) -> List[int]:
    """Latent rows per band: floor(h/n) each, the first (h mod n) bands one more.

    Uneven splits keep their actual lengths ("Static Layer-Wise VAE Decode",
    "Semantics and Communication"); the remainder-first rule is the one the
    100-row, 3-band workload (34/33/33) fixes.
    """
    if n_bands < 1 or n_bands > h:
        raise ValueError(f"n_bands={n_bands} must be in [1, {h}]")
    q, r = divmod(h, n_bands)
    return [q + (1 if i < r else 0) for i in range(n_bands)]


def output_shape(arch, latent_shape: Sequence[int]) -> Tuple[int, ...]:
    """Decoded output shape: 2x space per upsampling stage, T -> 2T - 1 per temporal one."""
    n_up = sum(1 for u in arch.stage_upsample if u)
    f = 2 ** n_up
    if arch.family == "kl2d":
        b, _, h, w = latent_shape
        f *= arch.latent_patch          # the front-end's unpatchify doubles the grid when patched
        return (b, arch.out_channels, h * f, w * f)
    b, _, t, h, w = latent_shape
    for u in arch.stage_upsample:
        if u == 2:
            t = 2 * t - 1
    return (b, arch.out_channels, t, h * f, w * f)


# ---------------------------------------------------------------------------
# Executors: the same decoder body runs on a whole tensor or on a band list.
# Height is always axis -2 and width axis -1 (NCHW and NCTHW).
# ---------------------------------------------------------------------------
class Dense:
    """Unbanded: every operator on the whole tensor."""

    def split(self, z):
        return ops._f64(z)

    def join(self, x):
        return x

    def conv(self, x, w, b):
        w = np.asarray(w)
        if w.ndim == 5:
            return ops.causal_conv3d(x, w, b)
        if x.ndim == 5:                      # per-frame 2D conv on a video
            n, c, t, h, wd = x.shape
            xf = x.transpose(0, 2, 1, 3, 4).reshape(n * t, c, h, wd)
            y = ops.conv2d_same(xf, w, b)
            return y.reshape(n, t, -1, h, wd).transpose(0, 2, 1, 3, 4)
        return ops.conv2d_same(x, w, b)

    def map(self, fn, *xs):
        return fn(*xs)

    def group_norm(self, x, groups, gamma, beta, eps):
        return ops.group_norm(x, groups, gamma, beta, eps)


class Banded:
    """The pages' layer-wise algorithm over height row bands or width column bands."""

    def __init__(self, n_bands: int, axis: str = "height"):
        if axis not in ("height", "width"):
            raise ValueError(axis)
        self.n_bands = n_bands
        self.ax = -2 if axis == "height" else -1

    def split(self, z):
        z = ops._f64(z)
        sizes = band_rows(z.shape[self.ax], self.n_bands)
        out, y = [], 0
        for r in sizes:
            sl = [slice(None)] * z.ndim
            sl[self.ax] = slice(y, y + r)
            out.append(z[tuple(sl)].copy())
            y += r
        return out

    def join(self, xs):
        return np.concatenate(xs, axis=self.ax)

    def conv(self, xs, w, b):
        """Each band convolves [halo, own rows or columns, halo] with no padding along the split axis.

        The halo is the kernel radius of the neighbouring band along the split
        axis; at the global edge it is zeros (the original padding).  The other
        spatial axis keeps its original zero padding.
        """
        w = np.asarray(w)
        kh, kw = w.shape[-2], w.shape[-1]
        if kh % 2 != 1 or kw % 2 != 1:
            raise ValueError("banded conv needs centred odd kernels")
        ax = self.ax
        r = (kh if ax == -2 else kw) // 2
        pad = (0, 0, kw // 2, kw // 2) if ax == -2 else (kh // 2, kh // 2, 0, 0)

        def take(a, lo, hi):
            sl = [slice(None)] * a.ndim
            sl[ax] = slice(lo, hi)
            return a[tuple(sl)]

        outs = []
        for i, xb in enumerate(xs):
            if r > 0 and xb.shape[ax] < r:
                raise ValueError("band smaller than the conv halo")
            zshape = list(xb.shape)
            zshape[ax] = r
            lo = take(xs[i - 1], -r, None) if (i > 0 and r > 0) else np.zeros(zshape)
            hi = take(xs[i + 1], 0, r) if (i + 1 < len(xs) and r > 0) else np.zeros(zshape)
            xin = np.concatenate([lo, xb, hi], axis=ax) if r > 0 else xb
            if w.ndim == 5:
                y = ops.causal_conv3d(xin, w, b, pad_hw=pad)
            elif xin.ndim == 5:
                n, c, t, h, wd = xin.shape
                xf = xin.transpose(0, 2, 1, 3, 4).reshape(n * t, c, h, wd)
                y = ops.conv2d(xf, w, b, pad)
                y = y.reshape(n, t, -1, y.shape[-2], y.shape[-1]).transpose(0, 2, 1, 3, 4)
            else:
                y = ops.conv2d(xin, w, b, pad)
            assert y.shape[ax] == xb.shape[ax]
            outs.append(y)
        return outs

    def map(self, fn, *xs):
        return [fn(*parts) for parts in zip(*xs)]

    def group_norm(self, xs, groups, gamma, beta, eps):
        """Per-band central moments, weighted merge, then the shared statistics per band."""
        parts = [ops.group_moments(xb, groups) for xb in xs]
        _, mean, var = ops.merge_moments(parts)
        return [ops.group_norm_apply(xb, groups, mean, var, gamma, beta, eps) for xb in xs]


# ---------------------------------------------------------------------------
# Decoder bodies
# ---------------------------------------------------------------------------
def _kl_resnet(ex, W, p, x, groups, eps):
    h = ex.group_norm(x, groups, W[p + ".norm1.weight"], W[p + ".norm1.bias"], eps)
    h = ex.map(ops.silu, h)
    h = ex.conv(h, W[p + ".conv1.weight"], W[p + ".conv1.bias"])
    h = ex.group_norm(h, groups, W[p + ".norm2.weight"], W[p + ".norm2.bias"], eps)
    h = ex.map(ops.silu, h)
    h = ex.conv(h, W[p + ".conv2.weight"], W[p + ".conv2.bias"])
    if p + ".conv_shortcut.weight" in W:
        sc = ex.conv(x, W[p + ".conv_shortcut.weight"], W[p + ".conv_shortcut.bias"])
    else:
        sc = x
    return ex.map(lambda a, b: a + b, sc, h)


def _tokens(x):
    """[B, C, H, W] -> [B, H*W, C] (row-major pixel order)."""
    n, c = x.shape[0], x.shape[1]
    return x.reshape(n, c, -1).transpose(0, 2, 1)


def _kl_attention(ex, W, p, x, groups, eps):
    hn = ex.group_norm(x, groups, W[p + ".group_norm.weight"], W[p + ".group_norm.bias"], eps)

    def q_fn(h):
        return np.stack([ops.linear(t, W[p + ".to_q.weight"], W[p + ".to_q.bias"]) for t in _tokens(h)])

    def kv_fn(h):
        tk = _tokens(h)
        k = np.stack([ops.linear(t, W[p + ".to_k.weight"], W[p + ".to_k.bias"]) for t in tk])
        v = np.stack([ops.linear(t, W[p + ".to_v.weight"], W[p + ".to_v.bias"]) for t in tk])
        return k, v

    def out_fn(xb, q, k, v):
        n, c, h, w = xb.shape
        o = np.stack([ops.sdpa(q[i], k[i], v[i]) for i in range(n)])
        o = np.stack([ops.linear(o[i], W[p + ".to_out.0.weight"], W[p + ".to_out.0.bias"])
                      for i in range(n)])
        return xb + o.transpose(0, 2, 1).reshape(n, c, h, w)

    if isinstance(ex, Banded):
        qs = [q_fn(hb) for hb in hn]
        kvs = [kv_fn(hb) for hb in hn]
        k_all = np.concatenate([kv[0] for kv in kvs], axis=1)
        v_all = np.concatenate([kv[1] for kv in kvs], axis=1)
        return [out_fn(xb, q, k_all, v_all) for xb, q in zip(x, qs)]
    return out_fn(x, q_fn(hn), *kv_fn(hn))


def latent_frontend(arch, W: Dict[str, np.ndarray], z: np.ndarray) -> np.ndarray:
    """AutoencoderKLFlux2 front-end (kl2d with latent_patch > 1): undo the latent BatchNorm over the
    patchified channels, then unpatchify to the decoder's latent grid.  Identity otherwise."""
    if arch.latent_patch <= 1:
        return z
    x = ops.inverse_batch_norm(z, W["bn.running_mean"], W["bn.running_var"], arch.latent_bn_eps)
    return ops.unpatchify(x, arch.latent_patch)


def decode_kl2d(arch, W: Dict[str, np.ndarray], z: np.ndarray, ex) -> np.ndarray:
    G, eps = arch.norm_groups, arch.eps
    z = latent_frontend(arch, W, z)
    x = ex.split(z)
    x = ex.conv(x, W["conv_in.weight"], W["conv_in.bias"])
    x = _kl_resnet(ex, W, "mid_block.resnets.0", x, G, eps)
    x = _kl_attention(ex, W, "mid_block.attentions.0", x, G, eps)
    x = _kl_resnet(ex, W, "mid_block.resnets.1", x, G, eps)
    for s in range(len(arch.stage_channels)):
        for r in range(arch.stage_resnets[s]):
            x = _kl_resnet(ex, W, f"up_blocks.{s}.resnets.{r}", x, G, eps)
        if arch.stage_upsample[s]:
            x = ex.map(ops.upsample_nearest2x, x)
            x = ex.conv(x, W[f"up_blocks.{s}.upsamplers.0.conv.weight"],
                        W[f"up_blocks.{s}.upsamplers.0.conv.bias"])
    x = ex.group_norm(x, G, W["conv_norm_out.weight"], W["conv_norm_out.bias"], eps)
    x = ex.map(ops.silu, x)
    x = ex.conv(x, W["conv_out.weight"], W["conv_out.bias"])
    return ex.join(x)


def _wan_resnet(ex, W, p, x):
    h = ex.map(lambda a: ops.silu(ops.rms_norm_channels(a, W[p + ".norm1.gamma"])), x)
    h = ex.conv(h, W[p + ".conv1.weight"], W[p + ".conv1.bias"])
    h = ex.map(lambda a: ops.silu(ops.rms_norm_channels(a, W[p + ".norm2.gamma"])), h)
    h = ex.conv(h, W[p + ".conv2.weight"], W[p + ".conv2.bias"])
    if p + ".conv_shortcut.weight" in W:
        sc = ex.conv(x, W[p + ".conv_shortcut.weight"], W[p + ".conv_shortcut.bias"])
    else:
        sc = x
    return ex.map(lambda a, b: a + b, sc, h)


def _wan_attention(ex, W, p, x):
    """Per-frame attention: tokens are one frame's H*W pixels (global over bands)."""
    c = x[0].shape[1] if isinstance(x, list) else x.shape[1]
    wq = W[p + ".to_qkv.weight"].reshape(3 * c, c)
    bq = W[p + ".to_qkv.bias"]
    wo = W[p + ".proj.weight"].reshape(c, c)
    bo = W[p + ".proj.bias"]

    def frames_tokens(a):
        n, cc, t, h, w = a.shape
        return a.transpose(0, 2, 1, 3, 4).reshape(n * t, cc, h * w).transpose(0, 2, 1)

    hn = ex.map(lambda a: ops.rms_norm_channels(a, W[p + ".norm.gamma"]), x)

    def qkv(hb):
        tk = frames_tokens(hb)                             # [N*T, tokens, C]
        qkv_ = np.stack([ops.linear(t, wq, bq) for t in tk])
        return qkv_[..., :c], qkv_[..., c:2 * c], qkv_[..., 2 * c:]

    def out_fn(xb, q, k, v):
        n, cc, t, h, w = xb.shape
        o = np.stack([ops.sdpa(q[i], k[i], v[i]) for i in range(q.shape[0])])
        o = np.stack([ops.linear(o[i], wo, bo) for i in range(q.shape[0])])
        o = o.transpose(0, 2, 1).reshape(n, t, cc, h, w).transpose(0, 2, 1, 3, 4)
        return xb + o

    if isinstance(ex, Banded):
        parts = [qkv(hb) for hb in hn]
        k_all = np.concatenate([pp[1] for pp in parts], axis=1)
        v_all = np.concatenate([pp[2] for pp in parts], axis=1)
        return [out_fn(xb, pp[0], k_all, v_all) for xb, pp in zip(x, parts)]
    q, k, v = qkv(hn)
    return out_fn(x, q, k, v)


def temporal_upsample(a: np.ndarray, w: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Wan upsample3d time step: frame 0 kept; frames 1..T-1 -> time_conv -> 2 frames each.

    time_conv is causal over the frames 1..T-1 (zero frames before frame 1)
    and maps C -> 2C channels; channels [0, C) become the first and [C, 2C)
    the second of the two output frames.  T frames become 2T - 1.
    """
    n, c, t, h, wd = a.shape
    if t == 1:
        return a
    y = ops.causal_conv3d(a[:, :, 1:], w, b, pad_hw=(0, 0, 0, 0))   # [n, 2c, t-1, h, w]
    out = np.empty((n, c, 1 + 2 * (t - 1), h, wd))
    out[:, :, 0] = a[:, :, 0]
    out[:, :, 1::2] = y[:, :c]
    out[:, :, 2::2] = y[:, c:]
    return out


def decode_wan3d(arch, W: Dict[str, np.ndarray], z: np.ndarray, ex) -> np.ndarray:
    x = ex.split(z)
    x = ex.conv(x, W["conv_in.weight"], W["conv_in.bias"])
    x = _wan_resnet(ex, W, "mid_block.resnets.0", x)
    x = _wan_attention(ex, W, "mid_block.attentions.0", x)
    x = _wan_resnet(ex, W, "mid_block.resnets.1", x)
    for s in range(len(arch.stage_channels)):
        for r in range(arch.stage_resnets[s]):
            x = _wan_resnet(ex, W, f"up_blocks.{s}.resnets.{r}", x)
        up = arch.stage_upsample[s]
        pre = f"up_blocks.{s}.upsamplers.0"
        if up == 2:
            x = ex.map(lambda a: temporal_upsample(a, W[pre + ".time_conv.weight"],
                                                   W[pre + ".time_conv.bias"]), x)
        if up:
            x = ex.map(ops.upsample_nearest2x, x)
            x = ex.conv(x, W[pre + ".resample.1.weight"], W[pre + ".resample.1.bias"])
    x = ex.map(lambda a: ops.silu(ops.rms_norm_channels(a, W["norm_out.gamma"])), x)
    x = ex.conv(x, W["conv_out.weight"], W["conv_out.bias"])
    return ex.join(x)


def decode(arch, W: Dict[str, np.ndarray], z: np.ndarray,
           n_bands: Optional[int] = None, axis: str = "height") -> np.ndarray:
    """Decode ``z`` in float64; unbanded when ``n_bands`` is None, else banded along ``axis``
    ("height", "width" or "auto", see band_axis)."""
    if n_bands is not None:
        p = arch.latent_patch if arch.family == "kl2d" else 1   # bands split the decoder's latent grid
        axis = band_axis(z.shape[-2] * p, z.shape[-1] * p, n_bands, axis)
    ex = Dense() if n_bands is None else Banded(n_bands, axis)
    if arch.family == "kl2d":
        return decode_kl2d(arch, W, z, ex)
    if arch.family == "wan3d":
        return decode_wan3d(arch, W, z, ex)
    raise ValueError(arch.family)

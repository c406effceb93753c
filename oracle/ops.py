"""Single-layer operators of the decode, float64, as their plain definitions.

Layouts follow the PyTorch modules the pages reuse: images are NCHW, videos
NCTHW, conv weights [C_out, C_in, k...].  Every function computes in float64.

TEST INFRASTRUCTURE ONLY: see the package docstring.
"""
from __future__ import annotations

from typing import List, Sequence, Tuple

import numpy as np

F64 = np.float64


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=F64)


# ---------------------------------------------------------------------------
# Convolution
# ---------------------------------------------------------------------------
def conv2d(x: np.ndarray, w: np.ndarray, b: np.ndarray,
           pad: Tuple[int, int, int, int]) -> np.ndarray:
    """Stride-1 2D cross-correlation with explicit zero padding.

    ``pad = (top, bottom, left, right)``.  With xp the zero-padded input,
    out[n, o, y, x] = b[o] + sum_{c, i, j} w[o, c, i, j] * xp[n, c, y + i, x + j].
    One matrix product per kernel tap (w[:, :, i, j] times the shifted input)
    realises the sum; the tap loop is the definition's (i, j) sum.
    """
    x, w, b = _f64(x), _f64(w), _f64(b)
    n_b, c_in, h, wd = x.shape
    c_out, c_in2, kh, kw = w.shape
    assert c_in == c_in2, (c_in, c_in2)
    top, bot, lef, rig = pad
    xp = np.zeros((n_b, c_in, h + top + bot, wd + lef + rig), F64)
    xp[:, :, top:top + h, lef:lef + wd] = x
    ho, wo = h + top + bot - kh + 1, wd + lef + rig - kw + 1
    out = np.empty((n_b, c_out, ho, wo), F64)
    out[:] = b[None, :, None, None]
    for n in range(n_b):
        acc = out[n].reshape(c_out, ho * wo)
        for i in range(kh):
            for j in range(kw):
                patch = np.ascontiguousarray(xp[n, :, i:i + ho, j:j + wo]).reshape(c_in, ho * wo)
                acc += w[:, :, i, j] @ patch
    return out


def conv2d_same(x: np.ndarray, w: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Centred odd-kernel conv with zero padding (k-1)/2 on every side."""
    kh, kw = w.shape[2], w.shape[3]
    assert kh % 2 == 1 and kw % 2 == 1, "centred odd kernels only"
    return conv2d(x, w, b, (kh // 2, kh // 2, kw // 2, kw // 2))


def causal_conv3d(x: np.ndarray, w: np.ndarray, b: np.ndarray,
                  pad_hw: Tuple[int, int, int, int] | None = None) -> np.ndarray:
    """Causal 3D conv (WanCausalConv3d): time padded (k_t - 1, 0), space as given.

    ``pad_hw = (top, bottom, left, right)``, default (k_h-1)/2 and (k_w-1)/2 on
    each side.  With xp the padded input,
    out[n, o, t, y, x] = b[o] + sum_{c, s, i, j} w[o, c, s, i, j] * xp[n, c, t + s, y + i, x + j],
    so output frame t sees input frames t - k_t + 1 .. t, and frames before 0
    are zero.
    """
    x, w, b = _f64(x), _f64(w), _f64(b)
    n_b, c_in, t, h, wd = x.shape
    c_out, c_in2, kt, kh, kw = w.shape
    assert c_in == c_in2
    if pad_hw is None:
        pad_hw = (kh // 2, kh // 2, kw // 2, kw // 2)
    top, bot, lef, rig = pad_hw
    xp = np.zeros((n_b, c_in, t + kt - 1, h + top + bot, wd + lef + rig), F64)
    xp[:, :, kt - 1:, top:top + h, lef:lef + wd] = x
    ho, wo = h + top + bot - kh + 1, wd + lef + rig - kw + 1
    out = np.empty((n_b, c_out, t, ho, wo), F64)
    out[:] = b[None, :, None, None, None]
    for n in range(n_b):
        acc = out[n].reshape(c_out, t * ho * wo)
        for s in range(kt):
            for i in range(kh):
                for j in range(kw):
                    patch = np.ascontiguousarray(
                        xp[n, :, s:s + t, i:i + ho, j:j + wo]).reshape(c_in, t * ho * wo)
                    acc += w[:, :, s, i, j] @ patch
    return out


# ---------------------------------------------------------------------------
# Pointwise and local operators
# ---------------------------------------------------------------------------
def unpatchify(x: np.ndarray, p: int) -> np.ndarray:
    """[B, C p^2, H, W] -> [B, C, p H, p W]: input channel c p^2 + py p + px holds output pixel
    (p y + py, p x + px) of channel c (the inverse of the p x p space-to-depth that groups each
    channel's p x p patch into consecutive channels; AutoencoderKLFlux2's latent patch conversion,
    "VAEP：VAE 并行解码", 不同模型如何复用)."""
    x = _f64(x)
    b, cp, h, w = x.shape
    c = cp // (p * p)
    out = np.empty((b, c, h * p, w * p))
    for py in range(p):
        for px in range(p):
            out[:, :, py::p, px::p] = x[:, py * p + px::p * p]
    return out


def inverse_batch_norm(x: np.ndarray, mean: np.ndarray, var: np.ndarray, eps: float) -> np.ndarray:
    """Undo an inference BatchNorm without affine terms, per channel (axis 1):
    x sqrt(var + eps) + mean (the latent BatchNorm the AutoencoderKLFlux2 front-end keeps)."""
    x = _f64(x)
    shape = (1, -1) + (1,) * (x.ndim - 2)
    return x * np.sqrt(_f64(var) + eps).reshape(shape) + _f64(mean).reshape(shape)


def silu(x: np.ndarray) -> np.ndarray:
    """SiLU(x) = x / (1 + exp(-x))."""
    x = _f64(x)
    return x / (1.0 + np.exp(-x))


def upsample_nearest2x(x: np.ndarray) -> np.ndarray:
    """Nearest-neighbour 2x in the last two (spatial) axes: up[.., Y, X] = x[.., Y // 2, X // 2]."""
    x = _f64(x)
    h, w = x.shape[-2], x.shape[-1]
    yi = np.arange(2 * h) // 2
    xi = np.arange(2 * w) // 2
    return x[..., yi, :][..., :, xi]


def rms_norm_channels(x: np.ndarray, gamma: np.ndarray, eps: float = 1e-12) -> np.ndarray:
    """Wan channel RMSNorm: x / max(||x||_2 over channels, eps) * sqrt(C) * gamma.

    Channels are axis 1; the norm is taken per pixel (and per frame).
    """
    x = _f64(x)
    c = x.shape[1]
    nrm = np.sqrt(np.sum(x * x, axis=1, keepdims=True))
    g = _f64(gamma).reshape((1, c) + (1,) * (x.ndim - 2))
    return x / np.maximum(nrm, eps) * np.sqrt(c) * g


# ---------------------------------------------------------------------------
# GroupNorm: whole-tensor two-pass statistics, per-band moments and their merge
# ---------------------------------------------------------------------------
def group_moments(x: np.ndarray, groups: int) -> Tuple[int, np.ndarray, np.ndarray]:
    """Two-pass moments per (sample, group): count n, mean, biased variance.

    mean = sum(x) / n, then var = sum((x - mean)^2) / n, over the group's
    channels and every spatial (and temporal) position of ``x``.
    """
    x = _f64(x)
    n_b, c = x.shape[0], x.shape[1]
    assert c % groups == 0
    xg = x.reshape(n_b, groups, -1)
    n = xg.shape[2]
    mean = xg.sum(axis=2) / n
    var = ((xg - mean[:, :, None]) ** 2).sum(axis=2) / n
    return n, mean, var


def merge_moments(parts: Sequence[Tuple[int, np.ndarray, np.ndarray]]
                  ) -> Tuple[int, np.ndarray, np.ndarray]:
    """Merge per-band central moments with the weighted rule.

    From "VAEP：VAE 并行解码", section "GroupNorm：合并全局统计量", and
    "Static Layer-Wise VAE Decode", section "Semantics and Communication":
    with w_i = n_i / N the band's share of the elements,
      mean = sum_i w_i * mean_i
      var  = sum_i w_i * (var_i + (mean_i - mean)^2).
    """
    total = sum(p[0] for p in parts)
    mean = sum((p[0] / total) * p[1] for p in parts)
    var = sum((p[0] / total) * (p[2] + (p[1] - mean) ** 2) for p in parts)
    return total, mean, var


def group_norm_apply(x: np.ndarray, groups: int, mean: np.ndarray, var: np.ndarray,
                     gamma: np.ndarray, beta: np.ndarray, eps: float) -> np.ndarray:
    """y = (x - mean_g) / sqrt(var_g + eps) * gamma_c + beta_c, per (sample, group)."""
    x = _f64(x)
    n_b, c = x.shape[0], x.shape[1]
    shp = (n_b, groups, c // groups) + x.shape[2:]
    xg = x.reshape(shp)
    ext = (n_b, groups) + (1,) * (xg.ndim - 2)
    y = (xg - mean.reshape(ext)) / np.sqrt(var.reshape(ext) + eps)
    y = y.reshape(x.shape)
    cshape = (1, c) + (1,) * (x.ndim - 2)
    return y * _f64(gamma).reshape(cshape) + _f64(beta).reshape(cshape)


def group_norm(x: np.ndarray, groups: int, gamma: np.ndarray, beta: np.ndarray,
               eps: float) -> np.ndarray:
    """GroupNorm with two-pass whole-tensor statistics (biased variance, eps inside the root)."""
    _, mean, var = group_moments(x, groups)
    return group_norm_apply(x, groups, mean, var, gamma, beta, eps)


# ---------------------------------------------------------------------------
# Attention
# ---------------------------------------------------------------------------
def softmax_rows(s: np.ndarray) -> np.ndarray:
    """Row softmax: subtract the row max, exponentiate, divide by the row sum."""
    s = _f64(s)
    m = s.max(axis=-1, keepdims=True)
    e = np.exp(s - m)
    return e / e.sum(axis=-1, keepdims=True)


def sdpa(q: np.ndarray, k: np.ndarray, v: np.ndarray) -> np.ndarray:
    """Single-head attention softmax(q k^T / sqrt(d)) v; q [Nq, d], k/v [Nk, d]."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    d = q.shape[-1]
    return softmax_rows(q @ k.T / np.sqrt(d)) @ v


def linear(x_tok: np.ndarray, w: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Per-token affine map: x_tok [N, C_in] @ w[C_out, C_in]^T + b."""
    return _f64(x_tok) @ _f64(w).T + _f64(b)[None, :]

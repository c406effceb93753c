"""Helpers for the GPU parity tests: decoders from seeded workloads, layout
conversions, the oracle's version of one traced op, and error metrics."""
from __future__ import annotations

import os
from typing import Dict, Tuple

import numpy as np
import pytest

import synth
from oracle import decoder as odec
from oracle import ops


def require_gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import row_band_layerwise_gb300 as rbl
    from row_band_layerwise_gb300 import build
    if not os.path.exists(build.lib_path()):
        build.build()
    return torch, rbl


def max_latent_for(shape) -> Tuple[int, int, int, int]:
    if len(shape) == 4:
        return (shape[0], 1, shape[2], shape[3])
    return (shape[0], shape[2], shape[3], shape[4])


def rel_l2(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))


def max_abs(a, b) -> float:
    return float(np.max(np.abs(np.asarray(a, np.float64) - np.asarray(b, np.float64))))


BF16_MAX_ABS = 3e-2     # the workload's bars for the bf16 tensor-core path
BF16_REL_L2 = 1e-2


def assert_bf16_parity(out, ref):
    """Whole-decode parity of the bf16 path: max-abs <= 3e-2 and rel-L2 <= 1e-2."""
    e_abs, e_rel = max_abs(out, ref), rel_l2(out, ref)
    assert e_rel <= BF16_REL_L2, f"rel-L2 {e_rel:.4e} > {BF16_REL_L2} (max-abs {e_abs:.4f})"
    assert e_abs <= BF16_MAX_ABS, f"max-abs {e_abs:.4f} > {BF16_MAX_ABS} (rel-L2 {e_rel:.4e})"
    return e_abs, e_rel


def to_numpy(t) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def parse_shape(s: str):
    return tuple(int(v) for v in s.split(","))


def cl_to_cf(x: np.ndarray) -> np.ndarray:
    """[B,T,H,W,C] -> [B,C,T,H,W]."""
    return np.ascontiguousarray(x.transpose(0, 4, 1, 2, 3))


def oracle_op(d: Dict[str, str], W, arch, x_cl: np.ndarray, aux_cl):
    """The oracle's output of one traced op, in the op's output layout.

    Channels-last ops return [B,T,H,W,C]; the final conv returns the
    channels-first decoder output (NCHW or NCTHW).
    """
    kind = d["kind"]
    x = cl_to_cf(x_cl)                      # [B,C,T,H,W]
    two_d = arch.family == "kl2d"
    if kind == "conv":
        name, conv = d["name"], d["conv"]
        w, b = W[name + ".weight"], W[name + ".bias"]
        if conv in ("k3", "k1", "up2x_k3"):
            n, c, t, h, wd = x.shape
            xf = x.transpose(0, 2, 1, 3, 4).reshape(n * t, c, h, wd)
            w4 = w if w.ndim == 4 else w.reshape(w.shape[0], w.shape[1], 1, 1)
            if conv == "up2x_k3":
                xf = ops.upsample_nearest2x(xf)
            y = ops.conv2d_same(xf, w4, b)
            y = y.reshape(n, t, y.shape[1], y.shape[2], y.shape[3]).transpose(0, 2, 1, 3, 4)
        elif conv == "causal3":
            y = ops.causal_conv3d(x, w, b)
        elif conv == "time":
            y = odec.temporal_upsample(x, w, b)
        else:
            raise ValueError(conv)
        if d.get("shortcut"):
            # 1x1 shortcut of the block fused into this conv: aux is its input
            sw, sb = W[d["shortcut"] + ".weight"], W[d["shortcut"] + ".bias"]
            a = cl_to_cf(aux_cl)
            n, c, t, h, wd = a.shape
            af = a.transpose(0, 2, 1, 3, 4).reshape(n * t, c, h, wd)
            s = ops.conv2d_same(af, sw.reshape(sw.shape[0], sw.shape[1], 1, 1), sb)
            y = y + s.reshape(n, t, s.shape[1], h, wd).transpose(0, 2, 1, 3, 4)
        elif d.get("res") == "1":
            y = y + cl_to_cf(aux_cl)
        if d.get("final") == "1":
            return y[:, :, 0] if two_d else y
        return y.transpose(0, 2, 3, 4, 1)
    if kind == "groupnorm":
        p = d["name"]
        y = ops.group_norm(x, int(d["groups"]), W[p + ".weight"], W[p + ".bias"], arch.eps)
        if d["silu"] == "1":
            y = ops.silu(y)
        return y.transpose(0, 2, 3, 4, 1)
    if kind == "rmsnorm":
        y = ops.rms_norm_channels(x, W[d["name"] + ".gamma"])
        if d["silu"] == "1":
            y = ops.silu(y)
        return y.transpose(0, 2, 3, 4, 1)
    if kind == "attention":
        if two_d:
            y = odec._kl_attention(odec.Dense(), W, d["name"], x[:, :, 0], arch.norm_groups, arch.eps)
            return y[:, :, None].transpose(0, 2, 3, 4, 1)
        y = odec._wan_attention(odec.Dense(), W, d["name"], x)
        return y.transpose(0, 2, 3, 4, 1)
    raise ValueError(kind)


class Case:
    """A seeded decoder instance plus its GPU handle."""

    def __init__(self, arch, dtype, latent_shape, wseed=1, zseed=0, max_latent=None):
        self.torch, self.rbl = require_gpu()
        self.arch, self.dtype, self.shape = arch, dtype, tuple(latent_shape)
        self.W = synth.make_weights(arch, dtype, seed=wseed)
        self.z = synth.make_latent(self.shape, dtype, seed=zseed)
        self.dec = self.rbl.Decoder(arch, self.W, dtype, max_latent or max_latent_for(self.shape))
        tdt = self.torch.bfloat16 if dtype == "bf16" else self.torch.float32
        self.z_dev = self.torch.from_numpy(self.z).to("cuda").to(tdt).contiguous()

    def decode(self, n_bands):
        out = self.dec.decode(self.z_dev, n_bands)
        self.torch.cuda.synchronize()
        self.dec.sync()
        return out

    def oracle(self, n_bands=None):
        return odec.decode(self.arch, self.W, self.z, n_bands)

    def capture(self, n_bands, op):
        torch = self.torch
        d = self.dec.op_desc(self.shape, n_bands, op)
        tdt = {"bf16": torch.bfloat16, "f32": torch.float32}
        in_shape = parse_shape(d["in"])
        out_shape = parse_shape(d["out"])
        t_in = torch.empty(int(np.prod(in_shape)), dtype=tdt[d["in_dt"]], device="cuda")
        t_out = torch.empty(int(np.prod(out_shape)), dtype=tdt[d["out_dt"]], device="cuda")
        aux_shape = parse_shape(d["aux"]) if "aux" in d else None
        t_aux = (torch.empty(int(np.prod(aux_shape)), dtype=tdt[d["aux_dt"]], device="cuda")
                 if aux_shape is not None else None)
        self.dec.run_until(self.z_dev, n_bands, op, t_in, t_aux, t_out)
        torch.cuda.synchronize()
        x = to_numpy(t_in)
        y = to_numpy(t_out)
        aux = to_numpy(t_aux).reshape(aux_shape) if t_aux is not None else None
        return d, x, aux, y


# Per-op tolerances: one bf16 rounding of the output dominates (2^-9 relative).
OP_TOL = {"bf16": dict(rel=6e-3, attn_rel=1.2e-2), "fp32": dict(rel=1e-5, attn_rel=1e-5)}


def check_all_ops(case: Case, n_bands: int, stride: int = 1):
    """Every traced op of one decode (every `stride`-th) against the oracle applied to that
    op's own GPU input, within OP_TOL; returns the set of "kind:conv" seen."""
    n_ops = case.dec.num_ops(case.shape, n_bands)
    assert n_ops > 5
    tol = OP_TOL[case.dtype]
    seen = set()
    for op in range(0, n_ops, stride):
        d, x, aux, y = case.capture(n_bands, op)
        seen.add(d["kind"] + ":" + d.get("conv", ""))
        in_shape = parse_shape(d["in"])
        if d["kind"] == "latent":
            xin = x.reshape(case.shape)
            exp = np.moveaxis(xin, 1, -1)
            np.testing.assert_array_equal(y.reshape(exp.shape), exp)
            continue
        ref = oracle_op(d, case.W, case.arch, x.reshape(in_shape), aux)
        got = y.reshape(ref.shape)
        lim = tol["attn_rel"] if d["kind"] == "attention" else tol["rel"]
        err = rel_l2(got, ref)
        assert err <= lim, f"op {op} {d}: rel-L2 {err:.3e} > {lim}"
    return seen

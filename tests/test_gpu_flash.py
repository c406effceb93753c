"""GPU parity of the fused band-attention kernel through its C entry point.

O = softmax(Q K^T / sqrt(C)) V per frame, every query against every key of its frame (the
pages' band-local Q against global K/V), compared with the float64 oracle (oracle.ops.sdpa)
on the same bf16-rounded Q, K, V.  The cases cover: key counts that leave a ragged last
128-key block (240, 4400), one to four key splits (a function of the key count), C = 384
and 512, two frames, queries whose running maximum keeps rising over the key blocks (so
the accumulator is rescaled), and band plans down to one-row bands, whose output must be
bit-identical to the one-band output.

Bar: rel-L2 <= 4e-3 and max-abs <= 1e-2 * max|O|.  The kernel's roundings are the bf16
probabilities fed to the tensor core (2^-9 relative, averaging out over the keys) and the
final bf16 output (at most 2^-9 relative per element, ~1.3e-3 rel-L2), so 4e-3 leaves room
without hiding a dropped block (a missing 128-key block moves O by far more).
"""
import numpy as np
import pytest

from gpu_helpers import max_abs, rel_l2, require_gpu
from oracle import ops

pytestmark = pytest.mark.gpu

REL = 4e-3
ABS_FRAC = 1e-2


def _inputs(seed, F, ntok, C, q_scale=2.0, ramp=0.0):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((F, ntok, C)) * q_scale
    k = rng.standard_normal((F, ntok, C))
    v = rng.standard_normal((F, ntok, C))
    if ramp:
        # scores of every query rise along the keys: channel 0 of the keys grows with the key index
        q[:, :, 0] = ramp
        k[:, :, 0] = np.linspace(-1.0, 1.0, ntok)[None, :] * 4.0
    return q.astype(np.float32), k.astype(np.float32), v.astype(np.float32)


def _run(torch, rbl, q, k, v, gh, gw, n_bands):
    dev = torch.device("cuda")
    F, ntok, C = q.shape
    tq = torch.from_numpy(q).to(dev).to(torch.bfloat16).contiguous()
    tk = torch.from_numpy(k).to(dev).to(torch.bfloat16).contiguous()
    tvt = torch.from_numpy(np.ascontiguousarray(v.transpose(0, 2, 1))).to(dev).to(torch.bfloat16).contiguous()
    out = torch.empty((F, ntok, C), dtype=torch.bfloat16, device=dev)
    nb = rbl.band_attention_work_bytes(F, gh, gw, C)
    work = torch.empty(max(nb, 16), dtype=torch.uint8, device=dev) if nb else None
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    rbl.band_attention(tq, tk, tvt, out, gh, gw, n_bands, work, status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    # the oracle sees exactly the bf16 operands the kernel read
    rq = tq.float().cpu().numpy().astype(np.float64)
    rk = tk.float().cpu().numpy().astype(np.float64)
    rv = tvt.float().cpu().numpy().astype(np.float64).transpose(0, 2, 1)
    return out.float().cpu().numpy().astype(np.float64), rq, rk, rv


def _check(got, rq, rk, rv, rows=None):
    for f in range(got.shape[0]):
        sel = np.arange(got.shape[1]) if rows is None else rows
        ref = ops.sdpa(rq[f, sel], rk[f], rv[f])
        g = got[f, sel]
        e_rel, e_abs = rel_l2(g, ref), max_abs(g, ref)
        assert e_rel <= REL, f"frame {f}: rel-L2 {e_rel:.3e}"
        assert e_abs <= ABS_FRAC * np.abs(ref).max(), f"frame {f}: max-abs {e_abs:.3e}"


@pytest.mark.parametrize("F,gh,gw,C,bands", [
    (1, 12, 20, 512, (1, 5, 12)),     # 240 keys: two key blocks, the second holding 112
    (2, 50, 88, 384, (1, 3)),         # 4400 keys: two key splits, ragged last block, two frames
    (2, 50, 88, 512, (1, 2)),         # the same at C = 512: CTAs whose first tile ends a frame run
                                      # their softmax warps unevenly (the per-block hand-off must hold)
    (1, 41, 200, 512, (1, 7)),        # 8200 keys: four key splits
])
def test_fused_attention_matches_oracle(F, gh, gw, C, bands):
    torch, rbl = require_gpu()
    q, k, v = _inputs(7, F, gh * gw, C)
    base = None
    for nb in bands:
        got, rq, rk, rv = _run(torch, rbl, q, k, v, gh, gw, nb)
        if base is None:
            base = got
            rows = None if gh * gw <= 4400 else np.random.default_rng(3).choice(gh * gw, 700, replace=False)
            _check(got, rq, rk, rv, rows)
        else:
            np.testing.assert_array_equal(got, base)   # bands only pick the query tiles


def test_fused_attention_rising_maximum():
    """Scores that climb over ~25 powers of two across the keys: the running maximum moves many
    times, every move past 2^8 rescales the accumulator, and the result still matches."""
    torch, rbl = require_gpu()
    gh, gw, C = 16, 64, 512
    q, k, v = _inputs(11, 1, gh * gw, C, ramp=100.0)
    got, rq, rk, rv = _run(torch, rbl, q, k, v, gh, gw, 4)
    _check(got, rq, rk, rv)


def test_fused_attention_rejects_bad_arguments():
    torch, rbl = require_gpu()
    dev = torch.device("cuda")

    def qkv(ntok, C):
        t = torch.zeros((1, ntok, C), dtype=torch.bfloat16, device=dev)
        return t, torch.zeros((1, C, ntok), dtype=torch.bfloat16, device=dev)

    st = torch.zeros(1, dtype=torch.int32, device=dev)
    t, tv = qkv(64, 512)
    with pytest.raises(rbl.VaedecError):
        rbl.band_attention(t, t, tv, t, 8, 8, 9, None, st)        # more bands than grid rows
    t2, tv2 = qkv(64, 96)
    with pytest.raises(rbl.VaedecError):
        rbl.band_attention(t2, t2, tv2, t2, 8, 8, 1, None, st)    # C not a multiple of 128
    t3, tv3 = qkv(64, 1024)
    with pytest.raises(rbl.VaedecError):
        rbl.band_attention(t3, t3, tv3, t3, 8, 8, 1, None, st)    # C above 512
    t4, tv4 = qkv(4400, 384)
    with pytest.raises(ValueError):
        rbl.band_attention(t4, t4, tv4, t4, 50, 88, 1, None, st)  # key splits need a work buffer
    small = torch.empty(16, dtype=torch.uint8, device=dev)
    with pytest.raises(ValueError):
        rbl.band_attention(t4, t4, tv4, t4, 50, 88, 1, small, st)  # ... of at least the stated size
    with pytest.raises(ValueError):
        rbl.band_attention(t, t, t, t, 8, 8, 1, None, st)          # V^T must be [F, C, ntok]
    with pytest.raises(ValueError):
        rbl.band_attention(t, t, tv, t, 8, 9, 1, None, st)         # tokens must fill the grid
    with pytest.raises(ValueError):
        rbl.band_attention(t, t, tv, t.cpu(), 8, 8, 1, None, st)   # every operand on the device
    with pytest.raises(ValueError):
        rbl.band_attention(t, t, tv, t, 8, 8, 1, None, st.float())  # status is int32

"""The multi-rank row-band split on CPU ranks (gloo, world size 2 and 3).

Each rank holds one height band of a seeded whole tensor.  The exchanges must rebuild exactly what
the whole-tensor computation reads ("VAEP：VAE 并行解码", 卷积：交换边界行 / GroupNorm：合并全局统计量 /
Attention：本地 Q，全局 K/V):

* halos: the band plus one row of each neighbour equals the slice of the zero-padded whole tensor,
  and a 3x3 conv of it (zero padding along the width only) equals the band's rows of the whole conv;
* moments: the gathered per-band moments, merged with the weighted rule, equal the whole tensor's
  two-pass moments (the oracle's functions, float64);
* K/V: the gathered rows equal the whole tensor's rows;
* the leader gather returns the whole tensor on rank 0 only.

Uneven bands (7 rows over 2 ranks, 3 over 3: one-row bands) are included.
"""
import multiprocessing as mp
import os
import socket

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, h, q):
    import sys
    sys.path.insert(0, ROOT)
    import numpy as np
    import torch
    import torch.distributed as dist
    import torch.nn.functional as F
    from oracle import ops
    from row_band_layerwise_gb300 import multirank as mr

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        rng = np.random.default_rng(5)
        B, C, W, G = 2, 8, 6, 4
        X = torch.from_numpy(rng.standard_normal((B, C, h, W)) * 2.0 + 0.5)        # whole tensor, float64
        band = mr.rank_bands(h, world)[rank]
        xb = X[:, :, band.row0:band.row0 + band.rows].contiguous()
        res = {}
        # halo rows
        xh = mr.halo_exchange(xb, r=1, axis=2)
        Xp = F.pad(X, (0, 0, 1, 1))
        res["halo"] = bool(torch.equal(xh, Xp[:, :, band.row0:band.row0 + band.rows + 2]))
        wgt = torch.from_numpy(rng.standard_normal((5, C, 3, 3)))
        bias = torch.from_numpy(rng.standard_normal(5))
        yb = F.conv2d(xh, wgt, bias, padding=(0, 1))
        Y = F.conv2d(X, wgt, bias, padding=1)
        res["conv"] = float((yb - Y[:, :, band.row0:band.row0 + band.rows]).abs().max())
        # moments: one (n, mean, var) triple per (sample, group) per band, gathered in band order
        n, mean, var = ops.group_moments(xb.numpy(), G)
        part = torch.from_numpy(np.stack([np.full_like(mean, n), mean, var], axis=-1))[None]   # [1, B, G, 3]
        parts = mr.allgather_rows(part, axis=0).numpy()
        merged = ops.merge_moments([(int(p[0, 0, 0]), p[..., 1], p[..., 2]) for p in parts])
        n_all, m_all, v_all = ops.group_moments(X.numpy(), G)
        res["moments"] = (merged[0] == n_all, float(np.max(np.abs(merged[1] - m_all) / (np.abs(m_all) + 1))),
                          float(np.max(np.abs(merged[2] - v_all) / v_all)))
        # K/V: token rows of this band, gathered
        tok = xb.permute(0, 2, 3, 1).reshape(B, band.rows * W, C)
        kv = mr.allgather_rows(tok, axis=1)
        res["kv"] = bool(torch.equal(kv, X.permute(0, 2, 3, 1).reshape(B, h * W, C)))
        # leader gather
        whole = mr.gather_to_leader(xb, axis=2)
        res["gather"] = (whole is None) if rank != 0 else bool(torch.equal(whole, X))
        dist.barrier()
    finally:
        dist.destroy_process_group()
    q.put((rank, res))


@pytest.mark.parametrize("world,h", [(2, 7), (2, 2), (3, 3), (3, 10)])
def test_band_exchanges_rebuild_the_whole_tensor(world, h):
    pytest.importorskip("torch")
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, world, port, h, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = dict(q.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, res in out.items():
        assert res["halo"], rank
        assert res["conv"] < 1e-12, (rank, res["conv"])
        same_n, e_mean, e_var = res["moments"]
        assert same_n and e_mean < 1e-12 and e_var < 1e-12, (rank, res["moments"])
        assert res["kv"], rank
        assert res["gather"], rank


def test_band_plan_matches_the_library_rule():
    from row_band_layerwise_gb300 import multirank as mr
    assert mr.band_rows(100, 3) == [34, 33, 33]
    bands = mr.rank_bands(100, 3)
    assert [(b.row0, b.rows) for b in bands] == [(0, 34), (34, 33), (67, 33)]
    assert bands[1].at(8) == mr.RankBand(1, 272, 264)
    with pytest.raises(ValueError):
        mr.band_rows(2, 3)


def test_exchange_schedule_of_the_1024_decode():
    """Two ranks, Z-Image 1024x1024: one halo exchange per 3x3 conv (31 of them: conv_in, 2 per
    resnet, 3 upsample convs, conv_out), one moment gather per GroupNorm (30), one K/V gather, one
    output gather; the halo volume of a rank is one row per conv at that conv's input width."""
    import synth
    from row_band_layerwise_gb300 import multirank as mr
    arch = synth.KL_ZIMAGE
    steps = mr.exchange_schedule(arch, (1, 16, 128, 128), 2)
    kinds = [s["kind"] for s in steps]
    assert kinds.count("halo") == 1 + 2 * (2 + 12) + 3 + 1
    assert kinds.count("moments") == 2 * (2 + 12) + 1 + 1
    assert kinds.count("kv") == 1 and kinds[-1] == "gather"
    # K and V of a 64-row band at C = 512, bf16
    kv = next(s for s in steps if s["kind"] == "kv")
    assert kv["bytes"] == 2 * 64 * 128 * 512 * 2
    out = steps[-1]
    assert out["bytes"] == 3 * 512 * 1024 * 2
    conv_out = [s for s in steps if s["layer"] == "conv_out"][0]
    assert conv_out["bytes"] == 1024 * 128 * 2          # one 1024-pixel row of 128 channels, bf16

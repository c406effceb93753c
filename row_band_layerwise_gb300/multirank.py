"""Row-band split of one decode across ranks: the exchange plan and its host-side collectives.

On one GPU the library runs every band: a conv reads its neighbour band's rows in place, GroupNorm
merges fixed row chunks, and attention's band-local queries see every key already resident.  Split
across GPUs, each rank holds one band and four exchanges keep the decode exact ("VAEP：VAE 并行解码",
按高度分片，逐层解码, 卷积：交换边界行, GroupNorm：合并全局统计量, Attention：本地 Q，全局 K/V;
"Static Layer-Wise VAE Decode", Semantics and Communication):

* every 3x3 conv: the kernel radius (r = 1 row) from each neighbouring band, zero rows at the
  global image edges only (``halo_exchange``);
* every GroupNorm: the per-band partial moments (count, mean, sum of squared deviations) of every
  (sample, group), gathered by every rank in global band order (``allgather_rows``), so each rank
  merges the same list in the same order with the weighted rule;
* mid-block attention: every rank's K and V rows gathered into local buffers (``allgather_rows``),
  queries stay local;
* at the end, the output bands gathered on the leader (``gather_to_leader``).

Remote data is always copied into a local tensor before use: nothing reads a peer's memory in
place and nothing uses multicast.  The collectives are torch.distributed calls (NCCL on GPUs, gloo
on the CPU); ``exchange_schedule`` lists the exchanges of a whole decode with their sizes.  This
split is exercised on CPU ranks only: no call in this project runs on more than one GPU.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import List, Optional, Sequence

__all__ = ["band_rows", "RankBand", "rank_bands", "halo_exchange", "allgather_rows", "gather_to_leader",
           "exchange_schedule"]


def band_rows(h: int, n: int) -> List[int]:
    """Rows per band: floor(h / n) each, the first h mod n bands one more (the pages' 34/33/33
    split of 100 rows into 3)."""
    if n < 1 or h < n:
        raise ValueError(f"cannot split {h} rows into {n} non-empty bands")
    return [h // n + (1 if i < h % n else 0) for i in range(n)]


@dataclass(frozen=True)
class RankBand:
    """One rank's band of latent rows [row0, row0 + rows)."""
    rank: int
    row0: int
    rows: int

    def at(self, factor: int) -> "RankBand":
        """The same band at a resolution `factor` times the latent's (nearest-2x upsamples double it)."""
        return RankBand(self.rank, self.row0 * factor, self.rows * factor)


def rank_bands(h: int, world: int) -> List[RankBand]:
    out, r0 = [], 0
    for rank, r in enumerate(band_rows(h, world)):
        out.append(RankBand(rank, r0, r))
        r0 += r
    return out


def _dist():
    import torch.distributed as dist
    return dist


def halo_exchange(x, r: int = 1, axis: int = -2, group=None):
    """``x`` (this rank's band, rows along ``axis``) with ``r`` rows of each neighbouring band
    attached, and ``r`` zero rows where the band meets the global image edge.

    Each rank sends its first ``r`` rows to the rank above and its last ``r`` rows to the rank
    below, and receives theirs into local buffers (paired non-blocking send/recv)."""
    import torch
    dist = _dist()
    rank, world = dist.get_rank(group), dist.get_world_size(group)
    ax = axis % x.dim()
    n = x.shape[ax]
    if r < 0 or (r > n and world > 1):
        raise ValueError(f"halo of {r} rows needs bands of at least {r} rows (this band has {n})")
    if r == 0:
        return x
    shape = list(x.shape)
    shape[ax] = r
    top = torch.zeros(shape, dtype=x.dtype, device=x.device)
    bot = torch.zeros(shape, dtype=x.dtype, device=x.device)
    ops = []
    if rank > 0:
        ops.append(dist.P2POp(dist.isend, x.narrow(ax, 0, r).contiguous(), _peer(rank - 1, group), group))
        ops.append(dist.P2POp(dist.irecv, top, _peer(rank - 1, group), group))
    if rank + 1 < world:
        ops.append(dist.P2POp(dist.isend, x.narrow(ax, n - r, r).contiguous(), _peer(rank + 1, group), group))
        ops.append(dist.P2POp(dist.irecv, bot, _peer(rank + 1, group), group))
    if ops:
        for req in dist.batch_isend_irecv(ops):
            req.wait()
    return torch.cat([top, x, bot], dim=ax)


def _peer(group_rank: int, group):
    dist = _dist()
    return group_rank if group is None else dist.get_global_rank(group, group_rank)


def allgather_rows(x, axis: int = 0, group=None):
    """Every rank's ``x`` concatenated along ``axis`` in rank order, on every rank.  The ranks'
    extents along ``axis`` may differ (uneven bands); the other dimensions must agree."""
    import torch
    dist = _dist()
    world = dist.get_world_size(group)
    ax = axis % x.dim()
    n = torch.tensor([x.shape[ax]], dtype=torch.int64, device=x.device)
    sizes = [torch.zeros_like(n) for _ in range(world)]
    dist.all_gather(sizes, n, group=group)
    sizes = [int(s.item()) for s in sizes]
    top = max(sizes)
    pad_shape = list(x.shape)
    pad_shape[ax] = top - x.shape[ax]
    xp = torch.cat([x, torch.zeros(pad_shape, dtype=x.dtype, device=x.device)], dim=ax) if pad_shape[ax] else x
    bufs = [torch.empty_like(xp.contiguous()) for _ in range(world)]
    dist.all_gather(bufs, xp.contiguous(), group=group)
    return torch.cat([b.narrow(ax, 0, s) for b, s in zip(bufs, sizes)], dim=ax)


def gather_to_leader(x, axis: int = -2, leader: int = 0, group=None):
    """The whole tensor (every rank's band along ``axis``, in rank order) on ``leader``; None on
    the other ranks."""
    dist = _dist()
    whole = allgather_rows(x, axis=axis, group=group)
    return whole if dist.get_rank(group) == leader else None


def exchange_schedule(arch, latent_shape: Sequence[int], world: int, bytes_per_value: int = 2) -> List[dict]:
    """Every exchange of one decode split into ``world`` height bands, in decode order, with the
    bytes one rank sends in it (largest band; halo rows both ways for an inner band).

    ``arch`` is a decoder description as in ``synth`` (KL 2D or Wan 3D).  Convs with a 3x3 spatial
    kernel exchange one row per neighbour (an upsample conv exchanges one low-resolution row: the
    nearest-2x rows it needs above and below come from it); 1x1 convs and the time conv exchange
    nothing; every GroupNorm gathers 3 fp32 values per (sample, group) per band; RMSNorm and SiLU
    are local; attention gathers K and V; the decode ends with a gather of the output bands.
    """
    kl = arch.family == "kl2d"
    b = latent_shape[0]
    t = 1 if kl else latent_shape[2]
    h, w = latent_shape[-2], latent_shape[-1]
    if kl and getattr(arch, "latent_patch", 1) > 1:
        h, w = h * arch.latent_patch, w * arch.latent_patch
    bands = rank_bands(h, world)
    big = max(bands, key=lambda bb: bb.rows)
    inner = 2 if world > 2 else (1 if world == 2 else 0)
    steps: List[dict] = []
    f = 1

    def halo(name, c, tt):
        steps.append({"kind": "halo", "layer": name, "rows": 1, "bytes": inner * b * tt * (w * f) * c * bytes_per_value})

    def moments(name):
        if kl:
            steps.append({"kind": "moments", "layer": name, "bytes": b * arch.norm_groups * 3 * 4})

    def resnet(p, cin, cout, tt):
        moments(p + ".norm1")
        halo(p + ".conv1", cin, tt)
        moments(p + ".norm2")
        halo(p + ".conv2", cout, tt)

    c = arch.mid_channels
    halo("conv_in", arch.latent_channels, t)
    resnet("mid_block.resnets.0", c, c, t)
    moments("mid_block.attentions.0.group_norm")
    steps.append({"kind": "kv", "layer": "mid_block.attentions.0",
                  "bytes": 2 * b * t * big.rows * w * c * bytes_per_value})
    resnet("mid_block.resnets.1", c, c, t)
    for s, cout in enumerate(arch.stage_channels):
        for r in range(arch.stage_resnets[s]):
            resnet(f"up_blocks.{s}.resnets.{r}", c, cout, t)
            c = cout
        up = arch.stage_upsample[s]
        if up:
            if up == 2:
                t = 2 * t - 1
            # the upsample conv reads one low-resolution halo row per neighbour
            halo(f"up_blocks.{s}.upsamplers.0", c, t)
            c = arch.stage_up_channels[s]
            f *= 2
    moments("conv_norm_out" if kl else "norm_out")
    halo("conv_out", c, t)
    steps.append({"kind": "gather", "layer": "output",
                  "bytes": b * arch.out_channels * t * big.rows * f * w * f * bytes_per_value})
    return steps

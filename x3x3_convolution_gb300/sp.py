"""Row-band parallel decode of a causal convolution stack over several ranks.

The FastVideo wan22_vae_decode commit message describes a decode split over a sequence-parallel group
of 2, 4 or 8 GPUs whose ranks agree on whether every one of them could build the kernel, and the
head.cu page's kernel takes a band of the output plane (its row offset and the global height). Here
each rank owns a contiguous band of rows of every layer's plane (all layers keep the plane's height).
Per layer and pass the ranks exchange one halo row with each neighbour - a rank's first input row is
the rank above's lower halo, its last row the rank below's upper halo - and then run the layer in the
library's banded mode (``make_desc(..., band_lo=, band_rows=, H_global=)``). Each layer's two-frame
history is kept per rank with the halo rows included, i.e. the last two frames of the assembled band
input. At the end the output bands are gathered. Bands concatenate to the whole plane bit for bit
(the banded mode is exact), so the parallel decode gives the single-GPU result.

This module is host-side plumbing: the exchange goes through torch.distributed point-to-point calls
(NCCL between GPUs, gloo between CPU processes) or, for ranks emulated one after another in one
process, through plain copies (``LocalBands``); every convolution runs in the callable given per layer,
normally a banded ``Conv`` of the library.
"""
from __future__ import annotations

from . import dist as _xd


def band_rows(H: int, world: int):
    """[(band_lo, band_rows)] of each rank: contiguous, sizes differing by at most one."""
    return [(r.start, len(r)) for r in (_xd.shard(H, k, world) for k in range(world))]


def halo_rows(band_lo: int, rows: int, H: int):
    """Global input rows [lo, hi) the band needs: its rows plus the halo rows that exist."""
    return max(band_lo - 1, 0), min(band_lo + rows + 1, H)


class DistBands:
    """Halo exchange and gather over torch.distributed (one band per rank)."""

    def __init__(self, H: int, row_axis: int):
        import torch.distributed as dist
        self.dist = dist
        self.rank, self.world = dist.get_rank(), dist.get_world_size()
        self.H, self.axis = H, row_axis
        self.bands = band_rows(H, self.world)
        self.band_lo, self.rows = self.bands[self.rank]

    def with_halo(self, x):
        """x: this rank's rows of a layer input; returns them with the neighbours' boundary rows attached
        (the row above from rank - 1, the row below from rank + 1, where those ranks exist)."""
        import torch
        dist, ax = self.dist, self.axis
        first = x.narrow(ax, 0, 1).contiguous()
        last = x.narrow(ax, x.shape[ax] - 1, 1).contiguous()
        up = torch.empty_like(first) if self.rank > 0 else None
        down = torch.empty_like(last) if self.rank < self.world - 1 else None
        ops = []
        if self.rank > 0:
            ops.append(dist.P2POp(dist.isend, first, self.rank - 1))
            ops.append(dist.P2POp(dist.irecv, up, self.rank - 1))
        if self.rank < self.world - 1:
            ops.append(dist.P2POp(dist.isend, last, self.rank + 1))
            ops.append(dist.P2POp(dist.irecv, down, self.rank + 1))
        if ops:
            for req in dist.batch_isend_irecv(ops):
                req.wait()
        parts = ([up] if up is not None else []) + [x] + ([down] if down is not None else [])
        return torch.cat(parts, dim=ax)

    def gather(self, y, scale: int = 1):
        """All ranks' output bands concatenated along the row axis (each band has `scale` output rows per
        plane row, e.g. 2 after a 2x2 unpatchify), on every rank."""
        import torch
        dist, ax = self.dist, self.axis
        most = max(r for _, r in self.bands) * scale
        pad = list(y.shape)
        pad[ax] = most
        buf = torch.zeros(pad, dtype=y.dtype, device=y.device)
        buf.narrow(ax, 0, y.shape[ax]).copy_(y)
        got = [torch.empty_like(buf) for _ in range(self.world)]
        dist.all_gather(got, buf)
        return torch.cat([g.narrow(ax, 0, r * scale) for g, (_, r) in zip(got, self.bands)], dim=ax)


class LocalBands:
    """The same decode with `world` ranks emulated one after another in one process: the halo rows are
    copied from the neighbouring bands' current inputs instead of being sent."""

    def __init__(self, H: int, row_axis: int, world: int):
        self.H, self.axis, self.world = H, row_axis, world
        self.bands = band_rows(H, world)


def decode_bands(layers, x_band, carries, carry_valid: bool, exchange, time_axis: int = 1):
    """One pass of a causal stack over this rank's band.

    layers:  per layer, a callable run(x_with_halo, carry_or_None) -> the band's output rows, computing
             the layer in banded mode for this rank's band (input rows = band rows + existing halos).
    x_band:  this rank's rows of the first layer's input (frames along `time_axis`).
    carries: per layer, a tensor to hold the layer's two-frame history with halo rows, or None; read
             when carry_valid, then overwritten with the last two frames of the assembled band input.
    exchange: a DistBands of this rank.
    Returns this rank's rows of the last layer's output.
    """
    import torch
    cur = x_band
    for i, run in enumerate(layers):
        inp = exchange.with_halo(cur)
        c = carries[i] if carries is not None else None
        hist = c if (c is not None and carry_valid) else None
        out = run(inp, hist)
        if c is not None:
            seq = inp if hist is None else torch.cat([hist, inp], dim=time_axis)
            if seq.shape[time_axis] < 2:
                seq = torch.cat([torch.zeros_like(seq), seq], dim=time_axis)
            c.copy_(seq.narrow(time_axis, seq.shape[time_axis] - 2, 2))
        cur = out
    return cur


def decode_bands_local(layers_per_rank, x, carries_per_rank, carry_valid: bool, bands: LocalBands,
                       time_axis: int = 1):
    """decode_bands for `bands.world` ranks emulated in one process. layers_per_rank[r][i] runs layer i on
    rank r's band; x is the whole first-layer input; carries_per_rank[r] as for decode_bands. Returns the
    ranks' output bands (to be concatenated along the row axis)."""
    import torch
    ax = bands.axis
    cur = [x.narrow(ax, lo, rows) for lo, rows in bands.bands]
    n_layers = len(layers_per_rank[0])
    for i in range(n_layers):
        inps = []
        for r in range(bands.world):
            parts = []
            if r > 0:
                parts.append(cur[r - 1].narrow(ax, cur[r - 1].shape[ax] - 1, 1))
            parts.append(cur[r])
            if r < bands.world - 1:
                parts.append(cur[r + 1].narrow(ax, 0, 1))
            inps.append(torch.cat(parts, dim=ax).contiguous())
        outs = []
        for r in range(bands.world):
            c = carries_per_rank[r][i] if carries_per_rank is not None else None
            hist = c if (c is not None and carry_valid) else None
            outs.append(layers_per_rank[r][i](inps[r], hist))
            if c is not None:
                seq = inps[r] if hist is None else torch.cat([hist, inps[r]], dim=time_axis)
                if seq.shape[time_axis] < 2:
                    seq = torch.cat([torch.zeros_like(seq), seq], dim=time_axis)
                c.copy_(seq.narrow(time_axis, seq.shape[time_axis] - 2, 2))
        cur = outs
    return cur


def banded_conv(conv_factory, desc_kwargs: dict, band_lo: int, rows: int, H_global: int):
    """A library Conv for one rank's band of a layer whose whole-plane descriptor is desc_kwargs (H =
    H_global): conv_factory(desc) builds it (with the layer's weights)."""
    from . import make_desc
    lo, hi = halo_rows(band_lo, rows, H_global)
    d = dict(desc_kwargs, H=hi - lo, band_lo=band_lo, band_rows=rows, H_global=H_global)
    return conv_factory(make_desc(**d))

"""Row-band parallel decode across ranks (x3x3_convolution_gb300.sp), tested as gloo processes on CPU
at world sizes 2 and 3: each rank holds a band of rows, exchanges one halo row with each neighbour per
layer, keeps its layers' two-frame histories with the halo rows, and the gathered output of two passes
must equal the single-rank decode bit for bit. The layers here are the oracle run on each band (its
rows plus halo rows, cropped to the band), so the test exercises the exchange, history and gather
logic; the library's banded kernels are checked against the whole plane in tests/test_gpu_band.py."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from x3x3_convolution_gb300 import sp

H, W, D = 11, 7, 3
CHANS = [4, 6, 5, 3]
ACTS = ["relu", "relu", "clamp"]


def _layers():
    rng = np.random.default_rng(9100)
    out = []
    for ci, co, act in zip(CHANS[:-1], CHANS[1:], ACTS):
        w = rng.integers(-1, 2, (co, ci, 3, 3, 3)).astype(np.float32)
        b = rng.integers(-1, 2, co).astype(np.float32)
        out.append(dict(w=w, b=b, act=act))
    return out


def _inputs():
    rng = np.random.default_rng(9101)
    return [rng.integers(-2, 3, (1, D, H, W, CHANS[0])).astype(np.float32) for _ in range(2)]


def _band_layer(oracle, L, band_lo, rows):
    lo, hi = sp.halo_rows(band_lo, rows, H)

    def run(inp, hist):
        y = oracle.conv3d_causal(inp.numpy(), L["w"], L["b"], carry=None if hist is None else hist.numpy(),
                                 act=L["act"], layout="NDHWC")
        y = oracle.round_to(y, "bf16")[0]
        return torch.from_numpy(np.ascontiguousarray(y[:, :, band_lo - lo:band_lo - lo + rows]))
    return run


def _reference(oracle):
    """Two passes of the stack on the whole plane, each layer rounded to bf16, histories carried."""
    layers, xs = _layers(), _inputs()
    hist = [None] * len(layers)
    outs = []
    for x in xs:
        cur = x
        for i, L in enumerate(layers):
            seq = cur if hist[i] is None else np.concatenate([hist[i], cur], axis=1)
            new_hist = seq[:, -2:].copy()
            cur = oracle.round_to(oracle.conv3d_causal(cur, L["w"], L["b"], carry=hist[i], act=L["act"],
                                                       layout="NDHWC"), "bf16")[0]
            hist[i] = new_hist
        outs.append(cur)
    return outs


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    import oracle
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ex = sp.DistBands(H, row_axis=2)
        lo, rows = ex.band_lo, ex.rows
        in_lo, in_hi = sp.halo_rows(lo, rows, H)
        runs = [_band_layer(oracle, L, lo, rows) for L in _layers()]
        carries = [torch.zeros((1, 2, in_hi - in_lo, W, c)) for c in CHANS[:-1]]
        outs = []
        for p, x in enumerate(_inputs()):
            y = sp.decode_bands(runs, torch.from_numpy(x[:, :, lo:lo + rows].copy()), carries, p > 0, ex)
            outs.append(ex.gather(y).numpy())
        q.put((rank, outs, None))
    except Exception as e:  # report to the parent instead of hanging it
        q.put((rank, None, repr(e)))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_band_decode_over_ranks_equals_one_rank(world, oracle_mod):
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = [q.get(timeout=180) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    ref = _reference(oracle_mod)
    for rank, outs, err in results:
        assert err is None, (rank, err)
        for got, want in zip(outs, ref):
            assert got.shape == want.shape
            assert np.array_equal(got, want), rank


def test_band_rows_split():
    assert sp.band_rows(11, 3) == [(0, 4), (4, 4), (8, 3)]
    assert sp.halo_rows(0, 4, 11) == (0, 5) and sp.halo_rows(4, 4, 11) == (3, 9) and sp.halo_rows(8, 3, 11) == (7, 11)


def test_local_band_decode_equals_one_rank(oracle_mod):
    """The same decode with the ranks emulated in one process (plain copies for the halo rows)."""
    world = 3
    bands = sp.LocalBands(H, row_axis=2, world=world)
    layers = _layers()
    runs = [[_band_layer(oracle_mod, L, lo, rows) for L in layers] for lo, rows in bands.bands]
    carries = []
    for lo, rows in bands.bands:
        a, b = sp.halo_rows(lo, rows, H)
        carries.append([torch.zeros((1, 2, b - a, W, c)) for c in CHANS[:-1]])
    ref = _reference(oracle_mod)
    for p, x in enumerate(_inputs()):
        parts = sp.decode_bands_local(runs, torch.from_numpy(x), carries, p > 0, bands)
        assert np.array_equal(torch.cat(parts, dim=2).numpy(), ref[p])

"""Host-side checks of the C ABI (no GPU): the library loads, exports every function that
include/x3conv.h declares, validates descriptors and arguments before any launch, and plans
tilings whose shared-memory staging covers every MMA read.
"""
import os
import re
import subprocess

import numpy as np
import pytest

import x3x3_convolution_gb300 as x3
from x3x3_convolution_gb300 import build as xb

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "x3conv.h")


@pytest.fixture(scope="module")
def lib():
    xb.build()
    return x3.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w \*]*?\b(conv_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("conv_plan_create", "conv_forward", "conv_stack_forward", "conv_plan_destroy",
                     "conv_pack_weights", "conv_stack_workspace_bytes", "conv_last_error"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", xb.LIB], capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT (\w+)$", out, flags=re.M))
    missing = [n for n in declared_functions() if n not in exported]
    assert not missing, missing
    for n in declared_functions():
        assert hasattr(lib, n)


def test_selftest_limits_validated_on_host(lib):
    for bad in (0, -5, 2001):
        assert lib.conv_selftest_wait_timeout(bad, None) == x3.X3_ERR_INVALID


def test_version(lib):
    assert "sm_103a" in x3.conv_version()


def _status(desc):
    import ctypes
    plan = ctypes.c_void_p()
    st = x3.load().conv_plan_create(ctypes.byref(desc), ctypes.byref(plan))
    if plan.value:
        x3.conv_plan_destroy(plan.value)
    return st


BAD = {
    "dims4": dict(dims=4),
    "zero_channels": dict(C_in=0),
    "stride3": dict(stride=3),
    "3d_stride2": dict(dims=3, layout="NDHWC", stride=2),
    "2d_with_3d_layout": dict(layout="NDHWC"),
    "3d_with_2d_layout": dict(dims=3, layout="NCHW"),
    "unpatch_needs_12": dict(unpatchify2x2=True, C_out=16),
    "zero_width": dict(W=0),
}


@pytest.mark.parametrize("name", sorted(BAD))
def test_invalid_descriptors_rejected(lib, name):
    kw = dict(dims=2, N=1, C_in=16, C_out=16, H=8, W=8, layout="NCHW", dtype="f16")
    kw.update(BAD[name])
    d = x3.make_desc(**kw)
    if name == "dims4":
        d.dims = 4
    assert _status(d) == x3.X3_ERR_INVALID
    assert x3.conv_last_error() != ""


LIMITS = [  # (descriptor changes, accepted) around the boundary's size limits
    (dict(H=32768, W=32768), True),                  # a plane of 2^30 positions
    (dict(H=32768, W=32769), False),
    (dict(C_in=65536), True),
    (dict(C_in=65537), False),
    (dict(C_out=65536), True),
    (dict(C_out=65537), False),
    (dict(N=1 << 30, H=1, W=1), True),               # 2^30 frames
    (dict(N=(1 << 30) + 1, H=1, W=1), False),
    (dict(dims=3, layout="NDHWC", dtype="bf16", D=(1 << 30) - 2, H=1, W=1), True),  # N (D + 2) = 2^30
    (dict(dims=3, layout="NDHWC", dtype="bf16", D=(1 << 30) - 1, H=1, W=1), False),
]


@pytest.mark.parametrize("i", range(len(LIMITS)))
def test_size_limits(lib, i):
    """Tensors up to the limits plan; one step past a limit is X3_ERR_INVALID ("tensor too large")."""
    kw = dict(dims=2, N=1, C_in=16, C_out=16, H=8, W=8, layout="NCHW", dtype="f16")
    change, ok = LIMITS[i]
    kw.update(change)
    st = _status(x3.make_desc(**kw))
    if ok:
        assert st == x3.X3_OK, x3.conv_last_error()
    else:
        assert st == x3.X3_ERR_INVALID and "too large" in x3.conv_last_error()


@pytest.mark.parametrize("H,kernel", [(65535, "igemm_tcgen05_sw128_head_stencil"),
                                      (65536, "igemm_tcgen05_sw128_head")])
def test_head_rows_past_the_stencil_limit(lib, H, kernel):
    """The stencil head keeps output rows in 16 bits: 65535 rows plan it, one more goes to the
    single-pass head."""
    p = x3.conv_plan_create(x3.make_desc(3, 1, 256, 12, H, 64, D=3, layout="NDHWC", dtype="bf16", act="clamp",
                                         unpatchify2x2=True))
    try:
        assert x3.conv_plan_kernel_name(p) == kernel
    finally:
        x3.conv_plan_destroy(p)


def test_plan_creation_from_threads(lib):
    """Eight threads create and destroy plans at once (ctypes releases the GIL during each call), half of
    them from descriptors that fail with a message naming the thread's own numbers: every status is
    right, every thread reads back its own last error (thread-local), and a success clears it."""
    import ctypes
    import threading

    failures = []

    def worker(i):
        try:
            for k in range(200):
                plan = ctypes.c_void_p()
                if (i + k) % 2:
                    d = x3.make_desc(2, 1, 16, 16, 8, 8 + i, layout="NCHW", dtype="f16")
                    assert lib.conv_plan_create(ctypes.byref(d), ctypes.byref(plan)) == x3.X3_OK
                    assert plan.value and x3.conv_last_error() == ""
                    x3.conv_plan_destroy(plan.value)
                else:
                    d = x3.make_desc(2, 1, 16, 16, 8, 8, layout="NCHW", dtype="f16",
                                     band_lo=0, band_rows=200 + i, H_global=100 + i)
                    assert lib.conv_plan_create(ctypes.byref(d), ctypes.byref(plan)) == x3.X3_ERR_INVALID
                    assert not plan.value
                    want = f"band [0, {200 + i}) is not inside the {100 + i}-row image"
                    assert want in x3.conv_last_error(), (i, x3.conv_last_error())
        except Exception as e:  # reported by the main thread
            failures.append((i, repr(e)))

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(8)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not failures, failures[:3]


def test_forced_igemm_unsupported_is_reported(lib):
    d = x3.make_desc(2, 1, 16, 16, 9, 9, layout="NCHW", dtype="f16", kernel="igemm")  # W % 8 != 0
    assert _status(d) == x3.X3_ERR_UNSUPPORTED
    d = x3.make_desc(2, 1, 16, 16, 9, 9, layout="NCHW", dtype="f16")
    assert _status(d) == x3.X3_OK


def test_forward_null_pointers_rejected_without_launch(lib):
    p = x3.conv_plan_create(x3.make_desc(2, 1, 16, 16, 8, 8, dtype="f16"))
    try:
        st = lib.conv_forward(p, None, None, None, None, None, None)
        assert st == x3.X3_ERR_INVALID
        st = lib.conv_forward(p, 16, None, 256, None, 4096, None)  # bias required (has_bias=1)
        assert st == x3.X3_ERR_INVALID
        st = lib.conv_forward(p, 18, None, 256, 2, 4096, None)     # misaligned x
        assert st == x3.X3_ERR_INVALID
        st = lib.conv_pack_weights(p, 2, 100, None)                 # misaligned packed buffer
        assert st == x3.X3_ERR_INVALID
    finally:
        x3.conv_plan_destroy(p)


def test_empty_stack_rejected(lib):
    for fn in (lib.conv_stack_forward, lib.conv_stack_forward_noalloc):
        assert fn(None, 0, 16, None, 0, None, None, 256, *((None, 0) if fn is lib.conv_stack_forward else ()),
                  None) == x3.X3_ERR_INVALID
        assert "layers" in x3.conv_last_error()
    assert lib.conv_stack_workspace_bytes(None, 0) == 0


def test_stack_validation(lib):
    a = x3.conv_plan_create(x3.make_desc(3, 1, 16, 32, 8, 8, D=2))
    b = x3.conv_plan_create(x3.make_desc(3, 1, 16, 8, 8, 8, D=2))   # C_in 16 != 32
    try:
        with pytest.raises(x3.X3Error) as e:
            x3.conv_stack_forward([a, b], 16, None, 0, [256, 256], [2, 2], 4096, 256, 1 << 20)
        assert e.value.status == x3.X3_ERR_INVALID
        c = x3.conv_plan_create(x3.make_desc(3, 1, 32, 8, 8, 8, D=2))
        need = x3.conv_stack_workspace_bytes([a, c])
        assert need >= 8 * 8 * 2 * 32 * 2
        with pytest.raises(x3.X3Error) as e:
            x3.conv_stack_forward([a, c], 16, None, 0, [256, 256], [2, 2], 4096, 256, need - 1)
        assert e.value.status == x3.X3_ERR_OOM
        x3.conv_plan_destroy(c)
    finally:
        x3.conv_plan_destroy(a)
        x3.conv_plan_destroy(b)


WORKLOADS = {
    "conv2d_16x16_64": dict(dims=2, N=1, C_in=16, C_out=16, H=64, W=64, dtype="f16", layout="NCHW"),
    "taesd_3to64_256": dict(dims=2, N=4, C_in=3, C_out=64, H=256, W=256, dtype="f16", layout="NCHW"),
    "taesd_64_256": dict(dims=2, N=4, C_in=64, C_out=64, H=256, W=256, dtype="f16", layout="NCHW"),
    "taesd_64_128": dict(dims=2, N=4, C_in=64, C_out=64, H=128, W=128, dtype="f16", layout="NCHW"),
    "causal_256_88x156": dict(dims=3, N=1, C_in=256, C_out=256, D=4, H=88, W=156),
    "causal_128_352x624": dict(dims=3, N=1, C_in=128, C_out=128, D=4, H=352, W=624),
    "causal_256to128_176x312": dict(dims=3, N=1, C_in=256, C_out=128, D=4, H=176, W=312),
    "head_256to12": dict(dims=3, N=1, C_in=256, C_out=12, D=4, H=352, W=624, unpatchify2x2=True, kernel="igemm"),
    "head_stencil_256to12": dict(dims=3, N=1, C_in=256, C_out=12, D=4, H=352, W=624, unpatchify2x2=True),
    "ragged_3d": dict(dims=3, N=2, C_in=40, C_out=72, D=3, H=7, W=301),
    "ragged_3d_wide": dict(dims=3, N=2, C_in=40, C_out=136, D=3, H=7, W=301),
    "nhwc_2d_256": dict(dims=2, N=3, C_in=64, C_out=256, H=33, W=97, layout="NHWC"),
    "nhwc_2d_64_tn": dict(dims=2, N=4, C_in=64, C_out=64, H=256, W=256, layout="NHWC", dtype="f16"),
    "nhwc_2d_80_tn": dict(dims=2, N=1, C_in=136, C_out=80, H=19, W=301, layout="NHWC"),
    "nhwc_2d_16_tn": dict(dims=2, N=2, C_in=8, C_out=16, H=7, W=9, layout="NHWC"),
    "head_two_pass_256to12": dict(dims=3, N=1, C_in=256, C_out=12, D=4, H=352, W=624, unpatchify2x2=True,
                                  kernel="head_two_pass"),
}


def _check_tn_plan(g, C_in, C_out):
    """Positions-as-M form with the horizontal taps in N: a tile is four whole raster rows of pitch 32
    (30 outputs and two junk columns each, one row per epilogue warp, so the kw shifts stay inside a
    warp); A = 128 staged positions from kh P (kh <= 2); N = 3 x C_out padded to 16 rows of resident
    weights; two TMEM buffers of N columns at a 256-column stride."""
    P, HR, Wt = g["P"], g["HR"], g["Wt"]
    assert g["tn"] == 1 and g["m64"] == 0 and g["win_adv"] == 128
    assert g["tk"] == (C_in == 8)
    assert (P, Wt, HR) == (32, 30, 7 if g["tk"] else 6)
    for win in range(min(g["windows"], 4 * P)):
        pos_off = (128 * win) % P
        assert pos_off == 0
        if g["tk"]:
            # taps in K: the ninth tap's rows (offset 2P + 2) and its zero partner one position on,
            # 16 bytes per position
            need = pos_off + 127 + 2 * P + 2 + 1 + 1
            assert need <= HR * P and need * 16 <= g["h_bytes"]
        else:
            need = pos_off + 127 + 2 * P + 1
            assert need <= HR * P and need * 128 <= g["h_bytes"]
    cp = (C_out + 15) // 16 * 16
    assert 3 * cp <= 256 and g["h_bytes"] % 1024 == 0 and g["smem_bytes"] <= 232448
    assert 2 <= g["n_h"] <= 4
    assert g["strips"] * Wt >= g["W_out"] or g.get("sub2")
    return cp


def _check_sw128_plan(g):
    """Channels-last swapped engine: 256-position windows of strip rasters of pitch P."""
    P, HR, Wt = g["P"], g["HR"], g["Wt"]
    if g.get("tn"):
        assert g["windows"] * 128 >= g["H_out"] * P
        assert g["tiles"] == g["strips"] * g["windows"] * g["frames"]
        return
    assert P == Wt + 2 and P <= 256 and HR <= 256
    # the furthest halo row read: a window starting at offset P-1 of a row (or 0 when P divides
    # 256), its last position, tap (kh=2, kw=2)
    adv = g["win_adv"]
    # a tile is one window of 256 positions (254 in the head form), or two (512) in the W2 form
    assert adv == (254 if g["kwm"] else (512 if g["w2"] else 256))
    span = 512 if g["w2"] else 256
    # furthest halo row read by a tile: its start offset in the first row, its last column,
    # kh = 2 (+2P) and, unless kw is folded into M, kw = 2 (+2); every such row is staged by the box
    for win in range(min(g["windows"], 4 * P)):
        pos_off = (adv * win) % P
        need = pos_off + span - 1 + 2 * P + (0 if g["kwm"] else 2) + 1
        assert need <= HR * P and need * 128 <= g["h_bytes"]
    assert g["h_bytes"] % 1024 == 0 and g["smem_bytes"] <= 232448
    assert g["strips"] * Wt >= g["W_out"] and g["windows"] * adv >= g["H_out"] * P
    assert g["tiles"] == g["strips"] * g["windows"] * g["frames"] * g["n_tiles"]


def stn_segments(H, strips, runs_max):
    """The stencil head's row segments: with fewer strips than runs each strip is cut into k segments
    (at least 16 rows each) so that there are about as many segments as runs; part p of strip s is
    segment p * strips + s. Returns (segment count, rows per segment)."""
    k = -(-runs_max // strips) if strips < runs_max else 1
    seg_rows = -(-H // k)
    if k > 1:
        seg_rows += (6 - seg_rows % 8) % 8  # rows + 2 a multiple of 8: the windows fill exactly
    if seg_rows < 16:
        seg_rows = min(H, 16)
    k = -(-H // seg_rows)
    return strips * k, seg_rows


def stn_plan(H, strips, runs_max):
    """The assignment of 8-row windows to runs: whole segments in rounds (run r takes r, r + R, ...)
    when there are at least as many segments as runs, then the greedy over the segments left (a run
    takes segment remainders while its windows last, else the 8 n - 2 rows its last n windows yield).
    Returns per run its pieces (strip, first output row, windows, segment end) and the windows of the
    longest run (the plan's `windows`)."""
    nseg, seg_rows = stn_segments(H, strips, runs_max)

    def bounds(sg):
        lo = (sg // strips) * seg_rows
        return sg % strips, lo, min(lo + seg_rows, H)

    full = nseg // runs_max if nseg >= runs_max else 0
    R = runs_max if full else 0
    runs = []
    for r in range(R):
        pieces = []
        for j in range(full):
            st, lo, hi = bounds(r + j * R)
            pieces.append((st, lo, (hi - lo + 9) // 8, hi))
        runs.append(pieces)
    left0 = full * R
    whole = [sum(p[2] for p in r) for r in runs] + [0] * (runs_max - len(runs))
    if left0 < nseg:
        T = max(whole)
        while True:
            sg, o, tail = left0, bounds(left0)[1], [[] for _ in range(runs_max)]
            for c in range(runs_max):
                cap = T - whole[c]
                if sg >= nseg or cap <= 0:
                    continue
                rem = cap
                while rem > 0 and sg < nseg:
                    st, lo, hi = bounds(sg)
                    need = (hi - o + 9) // 8
                    if need <= rem:
                        tail[c].append((st, o, need, hi))
                        rem -= need
                        sg += 1
                        if sg < nseg:
                            o = bounds(sg)[1]
                    else:
                        tail[c].append((st, o, rem, hi))
                        o += 8 * rem - 2
                        rem = 0
            if sg >= nseg:
                break
            T += 1
        used = max((c + 1 for c in range(runs_max) if tail[c]), default=0)
        for c in range(max(used, len(runs))):
            if c < len(runs):
                runs[c] += tail[c]
            else:
                runs.append(tail[c])
    return runs, max(sum(p[2] for p in r) for r in runs)


def _check_stn_runs(g):
    """The runs the plan implies cover every output row of every strip exactly once (a piece of nb
    windows from row o0 stores rows o0 .. o0 + 8 nb - 3, clipped at its segment's end), each run by
    one CTA per frame group (the fewest frames per group that divide the frames and leave no more groups
    than CTAs), with no more CTAs than SMs."""
    H, strips, n, F = g["H_out"], g["strips"], g["windows"], g["frames"]
    ctas = min(g["sms"], 256)
    fpc = 1
    while F % fpc or F // fpc > ctas:
        fpc += 1
    groups = F // fpc
    runs_max = ctas // groups
    runs, n_model = stn_plan(H, strips, runs_max)
    assert n == n_model
    assert len(runs) * groups == g["grid"] <= ctas
    assert g["tiles"] == sum(p[2] for r in runs for p in r) * g["frames"]
    cover = np.zeros((strips, H), np.int32)
    for r in runs:
        for s, o0, nb, hi in r:
            cover[s, o0:min(o0 + 8 * nb - 2, hi)] += 1
    assert np.all(cover == 1)


@pytest.mark.parametrize("H,W,D,N", [(352, 624, 4, 1), (17, 33, 1, 1), (100, 300, 2, 2), (5, 2000, 3, 1),
                                     (1000, 14, 2, 1), (64, 64, 8, 1), (40, 60, 7, 1), (20, 30, 100, 2)])
def test_stencil_head_runs(lib, H, W, D, N):
    d = x3.make_desc(3, N, 256, 12, H, W, D=D, act="clamp", unpatchify2x2=True, kernel="head_stencil")
    p = x3.conv_plan_create(d)
    try:
        g = x3.conv_plan_describe(p)
    finally:
        x3.conv_plan_destroy(p)
    assert g["stn"] == 1 and g["frames"] == N * D
    _check_stn_runs(g)


def test_stencil_head_run_model_rejects_bad_runs():
    """The coverage check above fails for runs that overlap or leave gaps (a run yielding 16 nb - 1
    or 16 nb - 3 rows per piece), so it constrains the piece arithmetic."""
    def cover(step):
        c = np.zeros((3, 100), np.int32)
        s = o = 0
        while s < 3:
            need = (100 - o + 17) // 16
            nb = min(need, 2)
            c[s, o:min(o + 16 * nb + step, 100)] += 1
            if nb == need:
                s, o = s + 1, 0
            else:
                o += 16 * nb - 2
        return c
    assert np.all(cover(-2) == 1)
    assert not np.all(cover(-1) == 1) and not np.all(cover(-3) == 1)


@pytest.mark.parametrize("name", sorted(WORKLOADS))
def test_igemm_plans_cover_their_reads(lib, name):
    _check_plan_of(WORKLOADS[name])


def _random_descs(n, seed):
    """Seeded random stride-1 channels-last layers: causal 3D (NDHWC bf16) and 2D (NHWC, f16 or bf16),
    channel counts around the engines' thresholds and tile sizes, ragged planes."""
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        if i % 3:
            out.append(dict(dims=3, N=int(rng.integers(1, 4)), C_in=int(rng.choice([8, 16, 24, 40, 64, 96, 128, 136, 256, 320])),
                            C_out=int(rng.choice([8, 16, 32, 64, 72, 96, 128, 136, 200, 256])), D=int(rng.integers(1, 7)),
                            H=int(rng.integers(1, 400)), W=int(rng.integers(1, 700)),
                            act=str(rng.choice(["none", "relu", "clamp"]))))
        else:
            out.append(dict(dims=2, N=int(rng.integers(1, 5)), C_in=int(rng.choice([8, 16, 24, 64, 136])),
                            C_out=int(rng.choice([8, 16, 24, 48, 64, 80, 96, 128, 256])), H=int(rng.integers(1, 300)),
                            W=int(rng.integers(1, 600)), layout="NHWC", dtype=str(rng.choice(["f16", "bf16"])),
                            act=str(rng.choice(["none", "relu"]))))
    return out


def test_random_plans_cover_their_reads(lib):
    """300 seeded random layers plan without error, and every tensor-core plan among them passes the
    same geometry checks as the workloads above (staged halo covers every read, tiles cover the
    output, shared memory and TMEM within their limits)."""
    kinds = set()
    for wl in _random_descs(300, seed=7500):
        kinds.add(_check_plan_of(wl))
    assert {"igemm_tcgen05_sw128", "tn"} <= kinds, kinds


def _check_plan_of(wl):
    """Plan the layer and check its geometry; returns the form checked."""
    p = x3.conv_plan_create(x3.make_desc(**wl))
    try:
        g = x3.conv_plan_describe(p)
        if g["kernel"] == "direct_simt":
            return "direct_simt"
        if g.get("stn"):
            # stencil head: 32 x 8 raster windows (30 output columns), one stage per (kt, chunk)
            # holding the window (32 KB) and its weight block (16 KB); every CTA runs at most `windows`
            # consecutive windows down the strips
            assert g["P"] == 32 and g["Wt"] == 30 and g["HR"] == 8 and g["win_adv"] == 256
            assert g["strips"] * 30 >= g["W_out"]
            assert g["h_bytes"] == 16 * 16 * 128 + 128 * 64 * 2 and g["smem_bytes"] <= 232448
            _check_stn_runs(g)
            return "stn"
        if wl.get("kernel") == "head_two_pass":
            # the temporal pass stages no halo: windows of 256 consecutive positions of a frame, each
            # stage holding the window (32 KB) and its (kt, chunk) weight block (16 KB)
            assert g["P"] == g["Wt"] == g["W_out"] and g["strips"] == 1
            assert g["windows"] * 256 >= g["H_out"] * g["W_out"] and g["h_bytes"] == 256 * 128 + 128 * 64 * 2
            assert g["tiles"] == g["windows"] * g["frames"] and g["smem_bytes"] <= 232448
            return "two_pass"
        if g["kernel"] in ("igemm_tcgen05_sw128", "igemm_tcgen05_sw128_head"):
            if g.get("tn"):
                _check_tn_plan(g, wl["C_in"], wl["C_out"])
            _check_sw128_plan(g)
            return "tn" if g.get("tn") else g["kernel"]
        assert g["kernel"] == "igemm_tcgen05"
        P, Rt, Wt, NSUB, spr = g["P"], g["Rt"], g["Wt"], g["NSUB"], g["spr"]
        assert P == Wt + 2 and P <= 256
        # every output of the tile is covered by a subtile row
        offs = [((s // spr) * P + (s % spr) * 128) if spr else 128 * s for s in range(NSUB)]
        covered = set()
        for o in offs:
            covered.update(range(o, o + 128))
        for r in range(Rt):
            for c in range(Wt):
                assert r * P + c in covered
        # the furthest A read (tap kh=2, kw=2 of the last subtile row) stays inside one A stage
        max_read = max(offs) + 127 + 2 * P + 2
        kpl = g["CK"] // 8
        assert (kpl - 1) * g["plane_stride"] + (max_read + 1) * 16 <= g["a_bytes"]
        assert g["tmem_cols"] <= 512 and g["NSUB"] * g["BN"] * g["acc_bufs"] <= g["tmem_cols"]
        assert g["smem_bytes"] <= 232448
        assert g["tiles"] == g["col_tiles"] * g["row_tiles"] * g["frames"] * g["n_tiles"]
        assert g["col_tiles"] * Wt >= g["W_out"] and g["row_tiles"] * Rt >= g["H_out"]
        return "igemm_tcgen05"
    finally:
        x3.conv_plan_destroy(p)


def test_head_two_pass_plan(lib):
    """The two-pass head is only offered for the conv_out head's shape, and its plan runs only
    through conv_head_two_pass, with a caller-provided 112-channel bf16 g plane."""
    good = dict(dims=3, N=2, C_in=256, C_out=12, D=3, H=20, W=30, unpatchify2x2=True, kernel="head_two_pass")
    p = x3.conv_plan_create(x3.make_desc(**good))
    try:
        assert x3.conv_plan_kernel_name(p) == "head_two_pass"
        assert x3.conv_head_g_bytes(p) == 2 * 3 * 9 * 20 * 30 * 12 * 2      # [N][D][9][H][W][12] bf16
        assert x3.conv_packed_weight_bytes(p) == 3 * 4 * 128 * 64 * 2   # [kt][chunk] A tiles, centre tap only
        g = x3.conv_plan_describe(p)
        assert g["win_adv"] == 256 and not g["kwm"] and g["n_tiles"] == 1
        st = lib.conv_forward(p, 16, None, 256, 32, 1 << 40, None)
        assert st == x3.X3_ERR_INVALID and "conv_head_two_pass" in x3.conv_last_error()
        assert lib.conv_head_two_pass(p, 16, None, 256, None, 1 << 40, 1 << 41, None) == x3.X3_ERR_INVALID  # bias
        assert lib.conv_head_two_pass(p, 16, None, 256, 32, (1 << 40) + 4, 1 << 41, None) == x3.X3_ERR_INVALID   # g align
        assert lib.conv_head_two_pass(p, 16, None, 256, 32, 4096, 1 << 41, None) == x3.X3_ERR_INVALID  # g overlaps x
        assert "overlap" in x3.conv_last_error()
        assert lib.conv_head_two_pass(p, 1 << 42, None, 256, 32, 1 << 40, (1 << 40) + 4096, None) == x3.X3_ERR_INVALID
    finally:
        x3.conv_plan_destroy(p)
    q = x3.conv_plan_create(x3.make_desc(3, 1, 64, 64, 8, 8, D=2))
    try:
        assert x3.conv_head_g_bytes(q) == 0
        assert lib.conv_head_two_pass(q, 16, None, 256, 32, 4096, 8192, None) == x3.X3_ERR_INVALID
    finally:
        x3.conv_plan_destroy(q)
    s = x3.conv_plan_create(x3.make_desc(**{**good, "kernel": "head_split"}))
    try:
        assert x3.conv_plan_kernel_name(s) == "head_split"
        assert x3.conv_head_g_bytes(s) == 2 * 3 * 9 * 20 * 30 * 12 * 4    # fp32 G
    finally:
        x3.conv_plan_destroy(s)
    for bad in (dict(unpatchify2x2=False), dict(layout="NCDHW"), dict(dtype="f16")):
        with pytest.raises(x3.X3Error) as e:
            x3.conv_plan_create(x3.make_desc(**{**good, **bad}))
        assert e.value.status == x3.X3_ERR_UNSUPPORTED


SHADOW_WORKLOADS = {
    "taesd_3to64_256": dict(dims=2, N=4, C_in=3, C_out=64, H=256, W=256, dtype="f16"),
    "taesd_64_256": dict(dims=2, N=4, C_in=64, C_out=64, H=256, W=256, dtype="f16"),
    "taesd_64_256_s2": dict(dims=2, N=4, C_in=64, C_out=64, H=256, W=256, stride=2, dtype="f16"),
    "taesd_64_128": dict(dims=2, N=4, C_in=64, C_out=64, H=128, W=128, dtype="f16"),
    "odd_5to24": dict(dims=2, N=1, C_in=5, C_out=24, H=37, W=83),
    "odd_72to136": dict(dims=2, N=1, C_in=72, C_out=136, H=19, W=42),
}


@pytest.mark.parametrize("name", sorted(SHADOW_WORKLOADS))
def test_nchw_layers_have_channels_last_forms(lib, name):
    """A 2D NCHW layer's channels-last form (used between the layers of a stack) stages every halo
    row its windows read, covers the stride-1 raster of its input, and puts its weight blocks after
    the layer's own packed weights unless the two share one format."""
    cfg = SHADOW_WORKLOADS[name]
    p = x3.conv_plan_create(x3.make_desc(**cfg))
    try:
        g = x3.conv_plan_describe(p)
        s = g["shadow"]
        P, HR, Wt = s["P"], s["HR"], s["Wt"]
        s2 = cfg.get("stride", 1) == 2
        assert s["s2"] == s2 and s["sub2"] == 0  # stride 2 from the four input phases
        if s2:
            # output raster of pitch Wt + 1; each phase box spans 2P x 2HR input positions (<= 256)
            Ho, Wo = (cfg["H"] + 1) // 2, (cfg["W"] + 1) // 2
            assert P == Wt + 1 and 2 * P <= 256 and 2 * HR <= 256
            for win in range(min(s["windows"], 4 * P)):
                assert (256 * win) % P + 255 + P + 1 + 1 <= HR * P  # shifts of one row and one column
        elif cfg["C_out"] <= 80:
            # stride 1 with at most 80 output channels: positions as M, horizontal taps in N
            Ho, Wo = cfg["H"], cfg["W"]
            assert s["tn"] == 1 and s["m64"] == 0 and (P, Wt, HR) == (32, 30, 7 if s["tk"] else 6)
            assert s["tk"] == ((cfg["C_in"] + 7) // 8 * 8 == 8)
            for win in range(min(s["windows"], 4 * P)):
                assert (128 * win) % P + 127 + 2 * P + 1 <= HR * P
        else:
            Ho, Wo = cfg["H"], cfg["W"]
            assert P == Wt + 2 and P <= 256 and HR <= 256
            for win in range(min(s["windows"], 4 * P)):
                assert (256 * win) % P + 255 + 2 * P + 2 + 1 <= HR * P
        adv = 128 if s["tn"] else 256
        assert s["strips"] * Wt >= Wo and s["windows"] * adv >= Ho * P
        assert s["n_chunks"] == (cfg["C_in"] + 63) // 64
        assert s["n_tiles"] == (1 if s["tn"] else (cfg["C_out"] + (63 if s["m64"] else 127)) // (64 if s["m64"] else 128))
        assert s["smem_bytes"] <= 232448 and s["w_off"] % 256 == 0
        assert s["m64"] == (cfg["C_out"] <= 64 and not s["tn"])
        cp = (cfg["C_out"] + 15) // 16 * 16
        shadow_bytes = (5 * cp * 32 if s.get("tk") else s["n_chunks"] * 3 * 3 * cp * 128 if s["tn"] else
                        s["n_tiles"] * s["n_chunks"] * 9 * (64 if s["m64"] else 128) * 64 * 2)
        assert x3.conv_packed_weight_bytes(p) == s["w_off"] + shadow_bytes or \
            (s["w_off"] == 0 and x3.conv_packed_weight_bytes(p) == shadow_bytes)
    finally:
        x3.conv_plan_destroy(p)


def test_stack_workspace_covers_the_channels_last_input(lib):
    """A two-layer NCHW stack run channels-last holds the converted input and one intermediate."""
    a = x3.conv_plan_create(x3.make_desc(2, 2, 64, 8, 16, 24))
    b = x3.conv_plan_create(x3.make_desc(2, 2, 8, 8, 16, 24))
    try:
        need = x3.conv_stack_workspace_bytes([a, b])
        assert need == 2 * ((2 * 16 * 24 * 64 * 2 + 255) // 256 * 256)
    finally:
        x3.conv_plan_destroy(a)
        x3.conv_plan_destroy(b)


@pytest.mark.parametrize("shape", [(4, 64, 64, 256, 256), (1, 64, 64, 33, 97), (2, 8, 32, 17, 255),
                                   (1, 64, 128, 20, 66), (1, 96, 64, 15, 40)], ids=str)
@pytest.mark.parametrize("form", ["phases", "raster"])
def test_stride2_channels_last_forms_planned(lib, shape, form, monkeypatch):
    """Stride-2 NHWC layers plan the four-input-phase form by default (output raster of pitch
    Wt + 1, each phase box spanning 2P x 2HR input positions, at most 256 a side) and, with
    X3CONV_S2=0, the stride-1 raster over the input plane with even positions kept. Plan geometry
    only: no GPU needed."""
    monkeypatch.setenv("X3CONV_S2", "1" if form == "phases" else "0")
    N, Ci, Co, H, W = shape
    p = x3.conv_plan_create(x3.make_desc(2, N, Ci, Co, H, W, stride=2, layout="NHWC", dtype="bf16"))
    try:
        g = x3.conv_plan_describe(p)
        Ho, Wo = (H + 1) // 2, (W + 1) // 2
        assert (g["H_out"], g["W_out"]) == (Ho, Wo)
        if form == "phases":
            assert (g["s2"], g["sub2"]) == (1, 0)
            P, HR, Wt = g["P"], g["HR"], g["Wt"]
            assert P == Wt + 1 and 2 * P <= 256 and 2 * HR <= 256
            assert g["strips"] * Wt >= Wo and g["windows"] * 256 >= Ho * P
            # every window's rows, shifted by one row and one column, stay inside its phase box
            for win in range(min(g["windows"], 4 * P)):
                assert (256 * win) % P + 255 + P + 1 + 1 <= HR * P
            assert g["h_bytes"] >= HR * P * 128 and g["h_bytes"] % 1024 == 0
            assert g["m64"] == (Co <= 64 and Ci <= 64)
        else:
            assert (g["s2"], g["sub2"]) == (0, 1)
            adv = 128 if g["tn"] else 256
            assert g["tn"] == (Co <= 80)
            assert g["P"] == g["Wt"] + 2 and g["strips"] * g["Wt"] >= W and g["windows"] * adv >= H * g["P"]
        assert g["smem_bytes"] <= 232448
    finally:
        x3.conv_plan_destroy(p)


# ------------------------------------------------------------------ banded mode (validation only)

def _band_desc(band_lo, band_rows, H_global, H=None, **kw):
    lo, hi = x3.band_input_rows(band_lo, band_rows, H_global)
    d = dict(dims=3, N=1, C_in=128, C_out=128, D=2, W=40)
    d.update(kw)
    return x3.make_desc(H=hi - lo if H is None else H, band_lo=band_lo, band_rows=band_rows, H_global=H_global, **d)


@pytest.mark.parametrize("band", [(0, 5, 20), (5, 6, 20), (11, 9, 20), (0, 20, 20), (19, 1, 20)], ids=str)
def test_band_plans(lib, band):
    """A band of output rows [lo, lo + rows) of an H_global-row image: its input holds the band's rows and
    the halo rows that exist globally; the plan's output height is the band's and its input starts one
    row above the band unless the band is at the top."""
    lo, rows, Hg = band
    p = x3.conv_plan_create(_band_desc(lo, rows, Hg))
    try:
        g = x3.conv_plan_describe(p)
        assert g["H_out"] == rows and g["row_shift"] == (1 if lo > 0 else 0)
    finally:
        x3.conv_plan_destroy(p)


def test_band_validation(lib):
    """Bands that miss a halo row which exists globally, lie outside the image, use stride 2 or the
    two-pass head, or give band rows without H_global, are rejected before any launch."""
    cases = [
        dict(band_lo=5, band_rows=6, H_global=20, H=7),    # the row below is missing
        dict(band_lo=5, band_rows=6, H_global=20, H=6),    # both halo rows missing
        dict(band_lo=0, band_rows=6, H_global=20, H=8),    # one row too many
        dict(band_lo=15, band_rows=6, H_global=20),        # past the bottom
        dict(band_lo=-1, band_rows=6, H_global=20, H=7),
        dict(band_lo=3, band_rows=0, H_global=20, H=2),
    ]
    for c in cases:
        lo, rows, Hg = c["band_lo"], c["band_rows"], c["H_global"]
        H = c.get("H", 8)
        with pytest.raises(x3.X3Error) as e:
            x3.conv_plan_create(_band_desc(lo, rows, Hg, H=H))
        assert e.value.status == x3.X3_ERR_INVALID
    with pytest.raises(x3.X3Error) as e:
        x3.conv_plan_create(_band_desc(5, 6, 20, H=7))
    assert "halo rows" in str(e.value)
    with pytest.raises(x3.X3Error):
        x3.conv_plan_create(_band_desc(4, 4, 16, dims=2, D=1, stride=2, layout="NHWC"))
    with pytest.raises(x3.X3Error):
        x3.conv_plan_create(_band_desc(4, 4, 16, C_in=256, C_out=12, unpatchify2x2=True, kernel="head_two_pass"))
    with pytest.raises(x3.X3Error):
        x3.conv_plan_create(x3.make_desc(3, 1, 8, 8, 10, 10, D=1, band_lo=2, band_rows=3))


def test_band_plans_do_not_chain(lib):
    """conv_stack_forward rejects banded layers: a band's output is narrower than the next band's input
    (the halo rows come from the neighbouring bands)."""
    a = x3.conv_plan_create(_band_desc(4, 8, 32))
    b = x3.conv_plan_create(_band_desc(4, 8, 32))
    try:
        plans, k1 = x3._ptrs([a, b])
        w, k2 = x3._ptrs([256, 256])
        bias, k3 = x3._ptrs([32, 32])
        st = lib.conv_stack_forward(plans, 2, 16, None, 0, w, bias, 1 << 40, 1 << 41, 1 << 30, None)
        assert st == x3.X3_ERR_INVALID
    finally:
        x3.conv_plan_destroy(a)
        x3.conv_plan_destroy(b)


def test_stencil_head_runs_random_planes(lib):
    """60 seeded random head planes (1 to 2000 rows, 1 to 4000 columns, 1 to 8 frames, batch 1 to 3):
    every plan's runs cover each output row of each strip exactly once and agree with the model."""
    rng = np.random.default_rng(8100)
    for _ in range(60):
        H, W = int(rng.integers(1, 2001)), int(rng.integers(1, 4001))
        D, N = int(rng.integers(1, 9)), int(rng.integers(1, 4))
        d = x3.make_desc(3, N, 256, 12, H, W, D=D, act="clamp", unpatchify2x2=True, kernel="head_stencil")
        p = x3.conv_plan_create(d)
        try:
            g = x3.conv_plan_describe(p)
        finally:
            x3.conv_plan_destroy(p)
        assert g["stn"] == 1, (H, W, D, N)
        _check_stn_runs(g)

"""Shared helpers of the GPU parity tests: device transfer, decoding and the tolerance checks.

Tolerances on random data: max|d| <= 1.5e-2 * max|ref| and rms(d) <= 4e-3 * rms(ref) against the
oracle's fp32 result; on integer-valued data the result must equal the oracle's value rounded
once to the storage type. Decoded outputs of the head: PSNR >= 55 dB over the [-1,1] range and
SSIM >= 0.998 (tests/ssim.py).
"""
import numpy as np
import torch

import oracle

MAX_TOL = 1.5e-2
RMS_TOL = 4e-3
PSNR_MIN = 55.0
SSIM_MIN = 0.998


def dev(t):
    """synth.Tensor -> torch tensor on cuda:0."""
    return t.torch("cuda")


def host_values(y: torch.Tensor, dtype: str) -> np.ndarray:
    bits = y.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    if dtype == "f16":
        return bits.view(np.float16).astype(np.float32)
    return (bits.astype(np.uint32) << 16).view(np.float32)


def assert_exact(got: np.ndarray, ref_f32: np.ndarray, dtype: str):
    ref, _ = oracle.round_to(ref_f32, dtype)
    bad = np.nonzero(got != ref)
    assert bad[0].size == 0, (f"{bad[0].size} of {got.size} values differ; first at {tuple(b[0] for b in bad)}: "
                              f"got {got[tuple(b[0] for b in bad)]} want {ref[tuple(b[0] for b in bad)]}")


def errors(got, ref):
    d = got.astype(np.float64) - ref.astype(np.float64)
    max_ratio = np.max(np.abs(d)) / max(np.max(np.abs(ref)), 1e-30)
    rms_ratio = np.sqrt(np.mean(d * d)) / max(np.sqrt(np.mean(ref.astype(np.float64) ** 2)), 1e-30)
    return max_ratio, rms_ratio


def assert_close(got, ref):
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got))
    m, r = errors(got, ref)
    assert m <= MAX_TOL and r <= RMS_TOL, f"max ratio {m:.3e} (<= {MAX_TOL}), rms ratio {r:.3e} (<= {RMS_TOL})"


def psnr(got, ref):
    mse = np.mean((got.astype(np.float64) - ref.astype(np.float64)) ** 2)
    return float("inf") if mse == 0 else 10.0 * np.log10(4.0 / mse)


def crops_3d(seq: np.ndarray, positions):
    """Zero-padded 3x3x3 windows of an NDHWC frame sequence [1, F, H, W, C] around output
    positions (t, h, w), where output frame t reads sequence frames t..t+2."""
    _, F, H, W, C = seq.shape
    out = np.zeros((len(positions), 3, 3, 3, C), np.float32)
    for i, (t, h, w) in enumerate(positions):
        for dh in range(3):
            hh = h + dh - 1
            if hh < 0 or hh >= H:
                continue
            w0, w1 = max(w - 1, 0), min(w + 2, W)
            out[i, :, dh, w0 - (w - 1):w1 - (w - 1)] = seq[0, t:t + 3, hh, w0:w1]
    return out


def oracle_sampled_3d(seq, w, b, act, positions, threads=0):
    """Oracle outputs at sampled positions, each from the oracle run on its own window.
    Returns [len(positions), C_out] fp32."""
    cr = crops_3d(seq, positions)
    y = oracle.conv3d_causal(cr[:, 2:3], w, b, carry=cr[:, 0:2], act=act, layout="NDHWC", threads=threads)
    return y[:, 0, 1, 1, :]


def sample_positions(D, H, W, n_random, seed, tile_w=128):
    rng = np.random.default_rng(seed)
    pos = set()
    for t in range(D):
        for h in (0, H - 1):
            for w in (0, 1, W - 2, W - 1):
                pos.add((t, h, w))
        for w in range(tile_w - 1, W, tile_w):
            for h in (0, H // 2, H - 1):
                pos.add((t, h, w))
                if w + 1 < W:
                    pos.add((t, h, w + 1))
    while len(pos) < n_random + 32:
        pos.add((int(rng.integers(D)), int(rng.integers(H)), int(rng.integers(W))))
    return sorted(pos)

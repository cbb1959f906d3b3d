"""Pins of the oracle's chain helpers, ``oracle.conv2d_chain`` and ``oracle.conv3d_chain``.

Each chain is checked against a reference built independently from torch's float64 ``conv2d`` /
``conv3d`` (the library special case of the definitions: TAESD conv page, ``taesd_conv3x3_impl``,
pad-1 cross-correlation with stride, bias-initialised accumulator, ReLU; FastVideo head.cu header
comment, causal 3x3x3 over [2 carried frames, current frames]); the causal chain's new histories
are checked against explicit slices of each layer's input sequence. Integer data give exact
results on both sides; random data agree within the fp32 summation bound of each layer.

The mutant tests build plausible wrong chains (a dropped activation, an ignored stride, a dropped bias,
rounding between layers, an ignored, misordered or misplaced history, a history taken from the output) and check
that the same pin rejects every one of them, so the pin is sensitive to those mistakes.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle


def _t(a):
    return torch.from_numpy(np.asarray(a, np.float64))


def torch_chain2d(x, layers):
    y = _t(x)
    for L in layers:
        y = F.conv2d(y, _t(L["w"]), None if L.get("b") is None else _t(L["b"]), stride=L.get("stride", 1), padding=1)
        if L.get("act", "none") == "relu":
            y = torch.relu(y)
        elif L.get("act") == "clamp":
            y = y.clamp(-1.0, 1.0)
    return y.numpy()


def torch_chain3d(x, layers, carries):
    """NCDHW; returns (y, new_carries) with new carry = last two frames of [carry, input]."""
    y = _t(x)
    news = []
    for i, L in enumerate(layers):
        c = _t(np.zeros(y.shape[:2] + (2,) + y.shape[3:])) if carries is None or carries[i] is None else _t(carries[i])
        seq = torch.cat([c, y], dim=2)
        news.append(seq[:, :, -2:].numpy().copy())
        y = F.conv3d(seq, _t(L["w"]), None if L.get("b") is None else _t(L["b"]), padding=(0, 1, 1))
        if L.get("act", "none") == "relu":
            y = torch.relu(y)
        elif L.get("act") == "clamp":
            y = y.clamp(-1.0, 1.0)
    return y.numpy(), news


def _layers2d(rng, integer):
    spec = [(3, 5, 1, "relu"), (5, 4, 2, "none"), (4, 6, 1, "relu"), (6, 3, 2, "relu")]
    out = []
    for ci, co, s, a in spec:
        if integer:
            w = rng.integers(-2, 3, (co, ci, 3, 3)).astype(np.float32)
            b = rng.integers(-2, 3, co).astype(np.float32)
        else:
            w = rng.standard_normal((co, ci, 3, 3)).astype(np.float32) / 3
            b = rng.uniform(-0.1, 0.1, co).astype(np.float32)
        out.append(dict(w=w, b=b, stride=s, act=a))
    return out


def _layers3d(rng, integer):
    spec = [(3, 4, "relu"), (4, 5, "none"), (5, 2, "relu")]
    out = []
    for ci, co, a in spec:
        if integer:
            w = rng.integers(-2, 3, (co, ci, 3, 3, 3)).astype(np.float32)
            b = rng.integers(-2, 3, co).astype(np.float32)
        else:
            w = rng.standard_normal((co, ci, 3, 3, 3)).astype(np.float32) / 5
            b = rng.uniform(-0.1, 0.1, co).astype(np.float32)
        out.append(dict(w=w, b=b, act=a))
    return out


def _fixture2d(integer):
    rng = np.random.default_rng(8101 if integer else 8102)
    x = (rng.integers(-2, 3, (2, 3, 11, 13)) if integer else rng.uniform(-1, 1, (2, 3, 11, 13))).astype(np.float32)
    return x, _layers2d(rng, integer)


def _fixture3d(integer, D=3):
    rng = np.random.default_rng(8201 if integer else 8202)
    draw = (lambda s: rng.integers(-2, 3, s)) if integer else (lambda s: rng.standard_normal(s))
    x = draw((2, 3, D, 7, 9)).astype(np.float32)
    layers = _layers3d(rng, integer)
    chans = [3, 4, 5]
    carries = [draw((2, c, 2, 7, 9)).astype(np.float32) for c in chans]
    return x, layers, carries


def _close(got, ref, integer):
    if integer:
        return got.shape == ref.shape and np.array_equal(got, ref)
    tol = 1e-4 * max(1.0, float(np.abs(ref).max()))
    return got.shape == ref.shape and float(np.abs(got - ref).max()) <= tol


def pin2d_ok(chain, integer):
    x, layers = _fixture2d(integer)
    return _close(np.asarray(chain(x, layers), np.float64), torch_chain2d(x, layers), integer)


def pin3d_ok(chain, integer, D=3, with_carries=True):
    x, layers, carries = _fixture3d(integer, D)
    cs = carries if with_carries else None
    y, news = chain(x, layers, carries=cs)
    ry, rnews = torch_chain3d(x, layers, cs)
    if not _close(np.asarray(y, np.float64), ry, integer):
        return False
    # new histories: the first layer's is exact input data; later ones are exact on integer data
    for i, (a, b) in enumerate(zip(news, rnews)):
        if not _close(np.asarray(a, np.float64), b, integer or i == 0):
            return False
    return True


@pytest.mark.parametrize("integer", [True, False])
def test_conv2d_chain_against_torch(integer):
    assert pin2d_ok(oracle.conv2d_chain, integer)


@pytest.mark.parametrize("with_carries", [True, False])
@pytest.mark.parametrize("D", [1, 3])
@pytest.mark.parametrize("integer", [True, False])
def test_conv3d_chain_against_torch(integer, D, with_carries):
    assert pin3d_ok(oracle.conv3d_chain, integer, D, with_carries)


def test_conv3d_chain_ndhwc_equals_ncdhw():
    x, layers, carries = _fixture3d(True)
    y1, n1 = oracle.conv3d_chain(x, layers, carries=carries)
    perm = (0, 2, 3, 4, 1)
    y2, n2 = oracle.conv3d_chain(x.transpose(perm), layers, carries=[c.transpose(perm) for c in carries],
                                 layout="NDHWC")
    assert np.array_equal(y2, y1.transpose(perm))
    for a, b in zip(n1, n2):
        assert np.array_equal(b, a.transpose(perm))


# ------------------------------------------------------------------ mutants of the chain helpers

def _m2d_no_act(x, layers):
    y = x
    for i, L in enumerate(layers):
        y = oracle.conv2d(y, L["w"], L["b"], stride=L["stride"], act="none" if i == 0 else L["act"])
    return y


def _m2d_no_stride(x, layers):
    y = x
    for L in layers:
        y = oracle.conv2d(y, L["w"], L["b"], stride=1, act=L["act"])
    return y[..., ::2, ::2] if y.shape[-1] > 4 else y


def _m2d_no_bias(x, layers):
    y = x
    for i, L in enumerate(layers):
        y = oracle.conv2d(y, L["w"], None if i == 1 else L["b"], stride=L["stride"], act=L["act"])
    return y


def _m2d_round_between(x, layers):
    y = x
    for L in layers:
        y = oracle.round_to(oracle.conv2d(y, L["w"], L["b"], stride=L["stride"], act=L["act"]), "bf16")[0]
    return y


@pytest.mark.parametrize("mutant", [_m2d_no_act, _m2d_no_stride, _m2d_no_bias, _m2d_round_between],
                         ids=lambda f: f.__name__)
def test_conv2d_chain_pin_rejects_mutants(mutant):
    assert pin2d_ok(oracle.conv2d_chain, False)
    # the rounding mutant is invisible on integer data of this size; the others fail either way
    assert not pin2d_ok(mutant, False)
    if mutant is not _m2d_round_between:
        assert not pin2d_ok(mutant, True)


def _m3d(kind):
    def chain(x, layers, carries=None):
        y = x
        news = []
        order = list(range(len(layers)))
        for i in order:
            L = layers[i]
            c = None if (carries is None or kind == "ignore_carry") else carries[i]
            if c is not None and kind == "carry_frames_swapped":
                c = c[:, :, ::-1]
            seq = y if c is None else np.concatenate([c, y], axis=2)
            if seq.shape[2] < 2:
                seq = np.concatenate([np.zeros_like(seq), seq], axis=2)
            news.append(seq[:, :, :2] if kind == "history_first_frames" else seq[:, :, -2:])
            act = "none" if (kind == "no_act" and i == 0) else L["act"]
            out = oracle.conv3d_causal(y, L["w"], L["b"], carry=c, act=act)
            if kind == "history_from_output":
                news[-1] = out[:, :, -2:] if out.shape[2] >= 2 else news[-1]
            y = out
        return y, news
    chain.__name__ = kind
    return chain


@pytest.mark.parametrize("kind", ["no_act", "ignore_carry", "carry_frames_swapped", "history_first_frames",
                                  "history_from_output"])
def test_conv3d_chain_pin_rejects_mutants(kind):
    assert pin3d_ok(oracle.conv3d_chain, True)
    assert not pin3d_ok(_m3d(kind), True)

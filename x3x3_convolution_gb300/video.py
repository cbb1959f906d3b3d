"""Pass-by-pass decoding of a long frame sequence through a causal stack.

The decoder of FastVideo wan22_vae_decode (commit message) carries a few latent frames per pass and
frees intermediates early, so that the peak memory of a long video stays bounded ("a 5 s video
peaks at 20.3 GiB, down from 94.6 GiB ... with the same output"). Here a ConvStack (one plan per
layer for `pass_frames` frames) is run over consecutive chunks of the sequence; each layer's
two-frame history lives in a small device buffer that conv_stack_forward reads and rewrites, the
intermediates live in the stack's two ping-pong workspace buffers, and only one pass of input and
output frames is on the device at a time. The output equals one pass over the whole sequence
(tests/test_gpu_video.py). Argument plumbing only: every convolution runs in libx3conv's kernels.
"""
from __future__ import annotations

from . import ConvStack, Conv, conv_plan_create, conv_plan_destroy, conv_packed_weight_bytes, make_desc


class PassDecoder:
    """Decodes [1, T, H, W, C] channels-last sequences pass by pass through causal 3D layers.

    layers: list of (Conv) built for `pass_frames` frames, chained (C_out[i] == C_in[i+1]).
    A final shorter pass (T % pass_frames frames) gets plans of its own that reuse the packed weights.
    """

    def __init__(self, layers, pass_frames: int):
        import torch
        self.layers = list(layers)
        self.D = pass_frames
        for L in self.layers:
            if L.desc.dims != 3 or L.desc.D != pass_frames:
                raise ValueError("PassDecoder needs 3D layers planned for pass_frames frames")
        self.stack = ConvStack(self.layers)
        d0 = self.layers[0].desc
        self.carries = [torch.zeros((1, 2, L.desc.H, L.desc.W, L.desc.C_in), dtype=torch.bfloat16
                                    if L.desc.dtype == 1 else torch.float16, device="cuda") for L in self.layers]
        self._short = {}
        self.in_shape = (1, pass_frames, d0.H, d0.W, d0.C_in)

    def _stack_for(self, frames):
        if frames == self.D:
            return self.stack
        if frames not in self._short:
            convs = []
            for L in self.layers:
                d = L.desc
                sd = make_desc(3, d.N, d.C_in, d.C_out, d.H, d.W, D=frames,
                               dtype="bf16" if d.dtype == 1 else "f16", act={0: "none", 1: "relu", 2: "clamp"}[d.act],
                               has_bias=bool(d.has_bias), unpatchify2x2=bool(d.unpatchify2x2))
                c = Conv.__new__(Conv)  # same packed weights, a plan for the shorter pass
                c.desc = sd
                c.plan = conv_plan_create(sd)
                if conv_packed_weight_bytes(c.plan) != conv_packed_weight_bytes(L.plan):
                    conv_plan_destroy(c.plan)
                    raise RuntimeError("the shorter pass packs its weights differently")
                c.kernel_name = L.kernel_name
                c.w_packed, c._wp, c.bias = L.w_packed, L._wp, L.bias
                convs.append(c)
            self._short[frames] = ConvStack(convs)
        return self._short[frames]

    def decode(self, frames, out=None, stream=None):
        """frames: [1, T, H, W, C] on the host (pinned for overlap) or the device. Returns the output
        sequence on the same side as `out` (default: host if the input is on the host)."""
        import torch
        T = frames.shape[1]
        last = self.layers[-1]
        if out is None:
            shape = list(last.out_shape())
            shape[1] = T
            out = torch.empty(shape, dtype=frames.dtype, device=frames.device,
                              pin_memory=(frames.device.type == "cpu"))
        x_dev = torch.empty(self.in_shape, dtype=frames.dtype, device="cuda")
        y_dev = torch.empty(last.out_shape(), dtype=frames.dtype, device="cuda")
        for p, t0 in enumerate(range(0, T, self.D)):
            n = min(self.D, T - t0)
            stack = self._stack_for(n)
            xin = x_dev[:, :n]
            xin.copy_(frames[:, t0:t0 + n], non_blocking=True)
            yout = y_dev[:, :n]
            stack(xin, carries=self.carries, carry_valid=p > 0, out=yout, stream=stream)
            out[:, t0:t0 + n].copy_(yout, non_blocking=True)
        torch.cuda.current_stream().synchronize()
        return out

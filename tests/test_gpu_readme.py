"""The README's Python example runs as written on one GPU and gives the shapes it states."""
import pathlib
import re

import pytest
import torch

pytestmark = pytest.mark.gpu


def test_readme_python_example():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    text = (pathlib.Path(__file__).resolve().parents[1] / "README.md").read_text()
    code = re.search(r"```python\n(.*?)```", text, re.S).group(1)
    ns = {}
    exec(compile(code, "README.md", "exec"), ns)
    torch.cuda.synchronize()
    assert tuple(ns["y"].shape) == (1, 4, 352, 624, 128)
    assert tuple(ns["head"].out_shape()) == (1, 4, 704, 1248, 3)
    assert ns["conv"].kernel_name == "igemm_tcgen05_sw128"
    assert ns["head"].kernel_name == "igemm_tcgen05_sw128_head_stencil"
    # the stack equals its two layers run one after the other with zero history
    x, carry = ns["x"], ns["carry"]
    zero = torch.zeros_like(carry)
    y2 = ns["conv2"](ns["conv"](x, zero), zero)
    torch.cuda.synchronize()
    assert torch.equal(ns["y"].view(torch.int16), y2.view(torch.int16))

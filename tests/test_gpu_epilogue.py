"""Kc, the fused bias + cast epilogue, run alone and compared bit for bit
with PyTorch's round-to-nearest-even casts of the same fp32 sums."""
import numpy as np
import pytest
import torch

import depthwise_convolution_forward_gb300 as gc
from depthwise_convolution_forward_gb300 import inputs
from gpu_util import require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def special_values(dt):
    """fp32 values that sit on rounding boundaries of the target type."""
    t = inputs.DTYPES[dt]
    base = torch.tensor([1.0, 3.0, -7.5, 65504.0, 1e-7, 6e-5, 0.0, -0.0, 1e30, -1e30], dtype=torch.float32)
    if t == torch.float32:
        return base
    lo = base.to(t).float()
    ulp = (torch.nextafter(base.to(t), torch.tensor(float("inf")).to(t)).float() - lo)
    halfway = lo + ulp / 2  # exact ties: round to even
    return torch.cat([base, halfway, -halfway, lo + ulp * 0.49, lo + ulp * 0.51])


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
@pytest.mark.parametrize("with_bias", [True, False])
def test_epilogue_bit_exact(dt, with_bias):
    t = inputs.DTYPES[dt]
    g = torch.Generator().manual_seed(5)
    cols = 24
    sv = special_values(dt)
    rows = 1000
    acc = torch.randn(rows, cols, generator=g) * 3
    acc.view(-1)[: sv.numel()] = sv
    bias = (torch.rand(cols, generator=g) - 0.5).to(t) if with_bias else None
    want = (acc + (bias.float() if with_bias else 0.0)).to(t)
    dev = torch.device("cuda:0")
    y = torch.empty(rows, cols, dtype=t, device=dev)
    gc.gconv_epilogue_apply(acc.to(dev), bias.to(dev) if with_bias else None, y, rows, cols,
                            gc.DTYPE_CODES[dt], torch.cuda.current_stream())
    torch.cuda.synchronize()
    iv = torch.int32 if t == torch.float32 else torch.int16
    got = y.cpu()
    same = (got.view(iv) == want.view(iv)) | (torch.isnan(got) & torch.isnan(want))
    assert bool(same.all()), f"{int((~same).sum())} mismatches"

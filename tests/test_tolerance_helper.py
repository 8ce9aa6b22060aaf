"""The parity tests' one-ulp bound: its spacing of the 16-bit formats agrees
with numpy's (fp16) and torch's next representable value (bf16)."""
import numpy as np
import torch

from gpu_helpers import ulp


def _values():
    rng = np.random.default_rng(0)
    x = rng.standard_normal(2000) * np.exp2(rng.integers(-30, 12, 2000))
    return np.concatenate([x, [1.0, 0.5, 0.75, 2.0, -1.0, 60000.0, 6.1e-5]])


def test_fp16_spacing_matches_numpy():
    x = _values()
    h = x.astype(np.float16)
    h = h[np.isfinite(h) & (h != 0)]
    ref = np.spacing(np.abs(h)).astype(np.float64)
    assert np.array_equal(ulp(h.astype(np.float64), torch.float16), ref)


def test_bf16_spacing_matches_torch_nextafter():
    x = torch.from_numpy(_values()).to(torch.bfloat16)
    x = x[x != 0].abs()
    up = torch.nextafter(x, torch.full_like(x, float("inf")))
    ref = (up.double() - x.double()).numpy()
    assert np.array_equal(ulp(x.double().numpy(), torch.bfloat16), ref)

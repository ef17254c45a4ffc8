"""Helpers shared by the GPU parity tests: move stored inputs to the device,
bring results back as float64, and apply the stated tolerances.

Tolerances (relative to rms(y_oracle), the root mean square of the oracle's
output over the compared elements):
  fp32 storage        max |diff| <= 1e-4 * rms
  fp16 / bf16 / Q4    max |diff| <= 2e-2 * rms  and  mean |diff| <= 4e-3 * rms
"""

from __future__ import annotations

import numpy as np

import oracle

F32_MAX = 1e-4
BF16_MAX = 2e-2
BF16_MEAN = 4e-3


def to_dev(a: np.ndarray, dtype: str):
    import torch
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def to_host64(t) -> np.ndarray:
    import torch
    if t.dtype == torch.bfloat16:
        return oracle.widen(t.view(torch.int16).cpu().numpy().view(np.uint16), "bf16")
    return t.cpu().numpy().astype(np.float64)


def errors(y: np.ndarray, ref: np.ndarray):
    rms = float(np.sqrt(np.mean(ref * ref)))
    d = np.abs(y - ref)
    return rms, float(d.max()) / rms, float(d.mean()) / rms


def assert_f32(y, ref):
    assert np.all(np.isfinite(y))
    rms, mx, _ = errors(y, ref)
    assert mx <= F32_MAX, f"max |diff| = {mx:.3e} * rms (bound {F32_MAX})"


def assert_lowp(y, ref):
    assert np.all(np.isfinite(y))
    rms, mx, mean = errors(y, ref)
    assert mx <= BF16_MAX, f"max |diff| = {mx:.3e} * rms (bound {BF16_MAX})"
    assert mean <= BF16_MEAN, f"mean |diff| = {mean:.3e} * rms (bound {BF16_MEAN})"


def assert_dtype(y, ref, dtype: str):
    (assert_f32 if dtype == "f32" else assert_lowp)(y, ref)


def q4_dev(inp: dict, name: str):
    import torch
    return (torch.from_numpy(inp["qs_" + name]).cuda(),
            torch.from_numpy(inp["sc_" + name].view(np.int16)).cuda())


def fp8_dev(inp: dict, name: str):
    import torch
    return (torch.from_numpy(np.ascontiguousarray(inp["c_" + name])).cuda(),
            torch.from_numpy(np.ascontiguousarray(inp["s_" + name])).cuda())


def q8_dev(inp: dict, name: str):
    import torch
    return (torch.from_numpy(np.ascontiguousarray(inp["q8_" + name])).cuda(),
            torch.from_numpy(np.ascontiguousarray(inp["q8s_" + name]).view(np.int16)).cuda())

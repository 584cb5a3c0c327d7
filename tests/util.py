"""Helpers shared by the GPU tests: tensor -> numpy marshalling for the
oracle and the parity bounds."""
import numpy as np
import torch

# fp32: max-abs error 1e-5; bf16 (fp32 accumulation): |gpu - ref| <= 2e-2 + 1e-2 |ref|;
# fp16 (fp32 accumulation, 3 more mantissa bits than bf16): 1e-2 + 5e-3 |ref|
TOL = {"f32": (1e-5, 0.0), "bf16": (2e-2, 1e-2), "f16": (1e-2, 5e-3)}


def to_np(t: torch.Tensor):
    """(array, dtype tag) for the oracle: bf16 as raw uint16 patterns."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16), "bf16"
    if t.dtype == torch.float32:
        return t.numpy(), "f32"
    if t.dtype == torch.float16:
        return t.numpy(), "f16"
    raise TypeError(t.dtype)


def bits(t: torch.Tensor) -> np.ndarray:
    """Raw bit patterns, for bit-exact comparisons."""
    t = t.detach().cpu().contiguous()
    if t.element_size() == 2:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.view(torch.int32).numpy().view(np.uint32)


def assert_close(got64: np.ndarray, ref64: np.ndarray, dtype: str, what: str = ""):
    atol, rtol = TOL[dtype]
    err = np.abs(got64 - ref64)
    bound = atol + rtol * np.abs(ref64)
    bad = ~(err <= bound)
    if bad.any():
        idx = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {err.size} outside {atol}+{rtol}|ref|; "
            f"worst at {idx}: got {got64[idx]!r} ref {ref64[idx]!r}")
    return float(err.max()) if err.size else 0.0

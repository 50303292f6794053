"""Helpers for the GPU parity tests: host arrays to device tensors and back
(uint32 data travels as int32 tensors holding the same bits), and the fp32
tolerance check."""
import numpy as np
import torch

F32_RTOL = 1e-5   # |gpu_i - ref_i| <= 1e-5 * sum_{j<=i} |x_j|


def to_dev(a: np.ndarray) -> torch.Tensor:
    if a.dtype == np.uint32:
        a = a.view(np.int32)
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def from_dev(t: torch.Tensor, dtype) -> np.ndarray:
    a = t.cpu().numpy()
    return a.view(dtype) if np.dtype(dtype) == np.uint32 else a


def assert_f32_within(got: np.ndarray, ref64: np.ndarray, abs_prefix: np.ndarray, what: str = ""):
    err = np.abs(got.astype(np.float64) - ref64)
    bound = F32_RTOL * abs_prefix
    bad = np.nonzero(err > bound)[0]
    assert bad.size == 0, (f"{what}: {bad.size} elements outside 1e-5*prefix|x|; first at {bad[0]}: "
                           f"got {got[bad[0]]!r} ref {ref64[bad[0]]!r} bound {bound[bad[0]]!r}")

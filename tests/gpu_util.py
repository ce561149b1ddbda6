"""Helpers for the GPU parity tests: device placement of numpy arrays in the
storage layouts the library must handle (dense, padded row stride, base
offset by one element so rows are not 16-byte aligned)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bitwise_reproducible_fp32_gb300 import build, detlib
    build.build()
    detlib.load()
    return torch.device("cuda:0")


def to_dev(a: np.ndarray, layout: str = "dense"):
    """Device copy of a 2-D array with the requested storage layout:
    dense  -- row stride = row length
    padded -- row stride rounded up to a multiple of 4, plus 4
    offset -- base pointer one float past a 16-byte boundary, stride + 1
    """
    a = np.ascontiguousarray(a)
    if a.ndim == 1 or layout == "dense":
        return torch.from_numpy(a).cuda()
    rows, cols = a.shape
    if layout == "padded":
        ld = (cols + 3) // 4 * 4 + 4
        buf = torch.full((rows, ld), float("nan"), dtype=torch.float32, device="cuda")
        buf[:, :cols] = torch.from_numpy(a).cuda()
        return buf[:, :cols]
    if layout == "offset":
        buf = torch.full((rows, cols + 1), float("nan"), dtype=torch.float32,
                         device="cuda")
        buf[:, 1:] = torch.from_numpy(a).cuda()
        return buf[:, 1:]
    raise ValueError(layout)


def empty_dev(rows: int, cols: int, layout: str = "dense"):
    return to_dev(np.full((rows, cols), np.nan, np.float32), layout)


def host(t) -> np.ndarray:
    return t.detach().cpu().numpy()

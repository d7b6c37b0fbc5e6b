"""Shared helpers of the GPU parity tests: moving seeded numpy inputs to the
device, and the element-wise tolerance checks."""
import numpy as np
import torch

# Tolerances of the path: |gpu - ref| <= ATOL + RTOL * |ref|, ref in fp64.
SHRINK_ATOL, SHRINK_RTOL = 1e-3, 2e-3
EXPAND_ATOL, EXPAND_RTOL = 1e-2, 1e-2


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    a = np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16)
    return torch.from_numpy(a).view(torch.bfloat16).cuda()


def host_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def bits_to_f64(bits: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.to(torch.float64).numpy()


def dev_i32(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def dev_f32(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def assert_close(got: np.ndarray, ref: np.ndarray, atol: float, rtol: float, what: str):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.isfinite(got).all(), "%s: non-finite output" % what
    err = np.abs(got - ref)
    bound = atol + rtol * np.abs(ref)
    bad = err > bound
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError("%s: %d of %d elements out of tolerance; first %s; max err %.3g"
                             % (what, int(bad.sum()), bad.size, idx.tolist(), float(err.max())))

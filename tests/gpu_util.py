"""Helpers shared by the GPU parity tests: moving seeded inputs to the device
and comparing against the oracle with the stated tolerances."""
import numpy as np
import pytest
import torch

# bf16 attention outputs: max-abs 2e-2 and mean-abs 2e-3 against the fp64
# oracle; fp32 paths: 1e-4.
BF16_MAX_ABS, BF16_MEAN_ABS = 2e-2, 2e-3
F32_MAX_ABS = 1e-4


def need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.float().cpu().numpy().astype(np.float64)
    return t.cpu().numpy()


def assert_close_bf16(got, want, what=""):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert got.shape == want.shape, (got.shape, want.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - want)
    assert err.max() <= BF16_MAX_ABS, f"{what}: max-abs {err.max():.3e} > {BF16_MAX_ABS}"
    assert err.mean() <= BF16_MEAN_ABS, f"{what}: mean-abs {err.mean():.3e} > {BF16_MEAN_ABS}"
    return err.max(), err.mean()


def assert_close_f32(got, want, what=""):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert got.shape == want.shape, (got.shape, want.shape)
    err = np.abs(got - want)
    assert err.max() <= F32_MAX_ABS, f"{what}: max-abs {err.max():.3e} > {F32_MAX_ABS}"
    return err.max()


def no_device_errors():
    import sliding_window_kv_swa_gb300 as nd
    torch.cuda.synchronize()
    assert nd.nd_device_errors(clear=True) == 0

"""Shared helpers of the GPU parity tests."""
import numpy as np
import pytest
import torch

import cohere_compass_decoder_gb300._lib as L


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    if not __import__("os").path.exists(L.LIB_PATH):
        from cohere_compass_decoder_gb300.build import build
        build()
    L.lib()


def bf16_dev(x_np_f32, device="cuda"):
    """float array -> bf16 device tensor (rounded by torch's cast)."""
    return torch.from_numpy(np.ascontiguousarray(x_np_f32, dtype=np.float32)).to(device).to(torch.bfloat16)


def f64(t):
    return t.detach().float().cpu().numpy().astype(np.float64)


def err_stats(got, want):
    d = np.abs(np.asarray(got, np.float64) - np.asarray(want, np.float64))
    return float(d.max()), float(d.mean())


def assert_close(got, want, max_abs, mean_abs, what=""):
    mx, mn = err_stats(got, want)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    assert mx <= max_abs and mn <= mean_abs, f"{what}: max-abs {mx:.3g} (<= {max_abs}), mean-abs {mn:.3g} (<= {mean_abs})"
    return mx, mn

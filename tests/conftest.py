import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: takes more than a few seconds on CPU")


def read_golden(name):
    """Non-comment lines of a golden fixture, split into tokens."""
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.lstrip().startswith("#")]


@pytest.fixture(scope="session")
def golden():
    return read_golden


def pytest_runtest_setup(item):
    if "gpu" in item.keywords:
        import torch
        if not torch.cuda.is_available():
            pytest.skip("needs a CUDA device")


@pytest.fixture(scope="session")
def va():
    import linear_attention_video_fwd_b300 as mod
    return mod


@pytest.fixture(scope="session")
def dev():
    import torch
    return torch.device("cuda", 0)


_INPUT_CACHE = {}


def cached_video_qkv(B, heads, T, H, W, d, seed, dtype="bf16"):
    """Session cache of synth.video_qkv (the full-size inputs take seconds)."""
    import synth
    key = (B, heads, T, H, W, d, seed, dtype)
    if key not in _INPUT_CACHE:
        _INPUT_CACHE.clear()
        _INPUT_CACHE[key] = synth.video_qkv(B, heads, T, H, W, d, seed, dtype)
    return _INPUT_CACHE[key]


def assert_bf16_close(got, want, max_abs=2e-2, mean_abs=2e-3):
    """The bf16 parity bar: max-abs <= 2e-2 and mean-abs <= 2e-3 vs the fp64 oracle."""
    import numpy as np
    err = np.abs(np.asarray(got, dtype=np.float64) - np.asarray(want, dtype=np.float64))
    assert np.isfinite(err).all(), "non-finite output"
    assert err.max() <= max_abs and err.mean() <= mean_abs, (float(err.max()), float(err.mean()))
    return float(err.max()), float(err.mean())

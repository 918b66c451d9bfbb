import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")


def read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


import pytest  # noqa: E402


@pytest.fixture(scope="session")
def ftlib():
    """The built libft binding (builds the library in-tree when it is missing or stale)."""
    import importlib.util
    spec = importlib.util.spec_from_file_location(
        "_ft_build", os.path.join(ROOT, "expert_cache_streaming_fp32_b300", "build.py"))
    b = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(b)
    b.build()
    import expert_cache_streaming_fp32_b300 as ft
    return ft


def rel_fro(a, b):
    import numpy as np
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def assert_close_layer(got, ref, fro=5e-3, maxrel=2e-2):
    """The floating-point bar: relative Frobenius error and max |err| against max |ref|."""
    import numpy as np
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape
    rf = rel_fro(got, ref)
    mx = float(np.abs(got - ref).max()) if got.size else 0.0
    scale = float(np.abs(ref).max()) if ref.size else 0.0
    assert rf <= fro, f"relative Frobenius error {rf:.3e} > {fro}"
    assert mx <= maxrel * scale + 1e-30, f"max |err| {mx:.3e} > {maxrel} * max|ref| ({scale:.3e})"
    return rf, mx


CC_MAX_ASSIGNMENTS = 8   # FT_CC_MAX_ASSIGNMENTS in include/ft.h


def bf16_act_round(T, k):
    """The oracle's rounding of the intermediate silu(G)*U for bf16 experts evaluated T*k
    assignments at a time: bf16 on the tensor cores, none (fp32) on the CUDA cores, which take
    batches of at most CC_MAX_ASSIGNMENTS assignments."""
    from oracle import formats
    return None if T * k <= CC_MAX_ASSIGNMENTS else formats.round_to_bf16

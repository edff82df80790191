"""Shared helpers of the GPU parity tests (compare a CUDA result with the oracle)."""
import numpy as np

# Parity bar for bf16 inputs/outputs with fp32 accumulation: element-wise
# max-abs and mean-abs error against the float64 oracle.
MAX_ABS = 2e-2
MEAN_ABS = 2e-3


def assert_close(got, ref, max_abs=MAX_ABS, mean_abs=MEAN_ABS, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    mx, mean = float(err.max()) if err.size else 0.0, float(err.mean()) if err.size else 0.0
    assert mx <= max_abs and mean <= mean_abs, f"{what}: max|err| {mx:.3e} mean|err| {mean:.3e}"
    return mx, mean


def sample_rows(S, n, seed, must=()):
    """n distinct query rows in [0, S): the given ones plus seeded picks."""
    rng = np.random.default_rng(seed)
    rows = {int(r) for r in must if 0 <= r < S}
    while len(rows) < min(n, S):
        rows.add(int(rng.integers(0, S)))
    return np.array(sorted(rows), np.int64)

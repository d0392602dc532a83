"""Shared helpers of the GPU parity tests (comparison against the oracle)."""
import math

import numpy as np

# Tolerances: bf16 inputs, fp32 accumulation; max |dO| and relative L2 error of
# O against the fp64 oracle on the same bf16-rounded inputs, and |d lse|.
MAX_ABS_O = 2e-2
REL_L2_O = 5e-3
MAX_ABS_LSE = 1e-3


def to64(t):
    return t.detach().to("cpu").double().numpy()


def assert_close(o, o_ref, lse=None, lse_ref=None, what="", elem_rel=0.0):
    """The gates above; elem_rel > 0 widens the per-element bound to
    MAX_ABS_O + elem_rel * |o_ref| (for inputs outside the configurations,
    where |O| can approach the largest |V|)."""
    o = np.asarray(o, dtype=np.float64)
    o_ref = np.asarray(o_ref, dtype=np.float64)
    assert o.shape == o_ref.shape, (o.shape, o_ref.shape)
    assert np.all(np.isfinite(o)), f"{what}: non-finite output"
    err = np.abs(o - o_ref)
    nref = np.linalg.norm(o_ref)
    rel = np.linalg.norm(o - o_ref) / nref if nref > 0 else np.linalg.norm(o - o_ref)
    msg = f"{what}: max|dO| {err.max():.3e} rel {rel:.3e}"
    assert np.all(err <= MAX_ABS_O + elem_rel * np.abs(o_ref)), msg
    assert rel <= REL_L2_O, msg
    if lse is not None:
        lse = np.asarray(lse, dtype=np.float64)
        lse_ref = np.asarray(lse_ref, dtype=np.float64)
        fin = np.isfinite(lse_ref)
        assert np.array_equal(fin, np.isfinite(lse)), f"{what}: lse finiteness differs"
        if fin.any():
            le = np.abs(lse[fin] - lse_ref[fin]).max()
            assert le <= MAX_ABS_LSE, f"{what}: max|dlse| {le:.3e}"


def scale_of(d):
    return 1.0 / math.sqrt(d)

"""Comparison helpers and the parity bars shared by the GPU tests.

Bars (per the method's stated tolerances):
  * int32 A: bit-exact when both sides consume the same codes.
  * Q codes from the pack: equal except +-1 on at most 1e-4 of the elements
    (an fp32 rotation computed in a different order can move a quotient
    across a rounding boundary); s scales within 1e-6 relative.
  * Y: max |Y_gpu - Y_oracle| / max |Y_oracle| <= 1e-3 per output tensor; when
    both sides use the same codes and scales Y is compared bit-exactly
    (the reconstruction is the same ordered fp32 arithmetic).
"""
import numpy as np

Q_MISMATCH_FRAC = 1e-4
S_REL = 1e-6
Y_REL = 1e-3


def code_mismatch(Q_gpu, Q_ref):
    Q_gpu = np.asarray(Q_gpu).astype(np.int32)
    Q_ref = np.asarray(Q_ref).astype(np.int32)
    d = np.abs(Q_gpu - Q_ref)
    n = int(np.count_nonzero(d))
    return n, (int(d.max()) if d.size else 0), n / max(d.size, 1)


def assert_codes(Q_gpu, Q_ref, what="Q"):
    n, dmax, frac = code_mismatch(Q_gpu, Q_ref)
    assert dmax <= 1, f"{what}: a code differs by {dmax}"
    assert frac <= Q_MISMATCH_FRAC, f"{what}: {n} codes differ ({frac:.2e} > {Q_MISMATCH_FRAC})"
    return n


def assert_scales(s_gpu, s_ref, what="s"):
    s_gpu = np.asarray(s_gpu, np.float64)
    s_ref = np.asarray(s_ref, np.float64)
    den = np.where(s_ref == 0, 1.0, np.abs(s_ref))
    rel = np.abs(s_gpu - s_ref) / den
    assert np.all((s_ref != 0) | (s_gpu == 0)), f"{what}: zero-row scale not zero"
    assert rel.max(initial=0.0) <= S_REL, f"{what}: max rel err {rel.max():.3e}"
    return float(rel.max(initial=0.0))


def y_rel_err(Y_gpu, Y_ref):
    Y_gpu = np.asarray(Y_gpu, np.float64)
    Y_ref = np.asarray(Y_ref, np.float64)
    den = np.max(np.abs(Y_ref)) if Y_ref.size else 1.0
    return float(np.max(np.abs(Y_gpu - Y_ref)) / max(den, 1e-30)) if Y_ref.size else 0.0


def assert_y(Y_gpu, Y_ref, what="Y"):
    e = y_rel_err(Y_gpu, Y_ref)
    assert e <= Y_REL, f"{what}: max rel err {e:.3e} > {Y_REL}"
    return e

"""Pins for the CPU oracle: facts that the pages and mathematics fix.

None of these tests re-types an oracle formula. Each compares the oracle with
something independent of it: the H4 matrix as printed on the page, NumPy's
Kronecker product, orthogonality and symmetry, exact rational arithmetic,
closed forms for one-hot rows, brute-force integer loops, and error bounds.
The last group plants plausible mistakes in the oracle and checks that some
pin fails for each of them.
"""
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import convrot_oracle as orc
from int8_hadamard_rotated_gb300 import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
GROUPS = (1, 4, 16, 64, 256, 1024)


def printed_h4():
    rows = []
    with open(os.path.join(GOLDEN, "h4.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append([int(v) for v in line.split()])
    return np.array(rows, dtype=np.float64) / 2.0


def kron_power(H, G):
    R = np.ones((1, 1))
    while R.shape[0] < G:
        R = np.kron(R, H)
    return R


# --------------------------------------------------------------------------
# R_G ("INT8 Convrot Safetensors" -- How INT8 convrot works)
# --------------------------------------------------------------------------

def check_h4(mod=orc):
    np.testing.assert_array_equal(mod.H4, printed_h4())


def check_R_kron(mod=orc):
    H = printed_h4()
    for G in (4, 16, 64, 256):
        R = mod.hadamard_matrix(G)
        np.testing.assert_array_equal(R, kron_power(H, G))
        if G > 4:
            # the factors are identical, so either nesting gives R_G
            np.testing.assert_array_equal(R, np.kron(H, kron_power(H, G // 4)))


def check_R_algebra(mod=orc):
    for G in GROUPS:
        R = mod.hadamard_matrix(G)
        eye = np.eye(G)
        np.testing.assert_allclose(R @ R.T, eye, atol=1e-12)   # orthogonal
        np.testing.assert_array_equal(R, R.T)                  # symmetric
        np.testing.assert_allclose(R @ R, eye, atol=1e-12)     # hence an involution
        np.testing.assert_allclose(R.sum(axis=1), np.ones(G), atol=1e-12)  # regular
        np.testing.assert_array_equal(np.abs(R), np.full((G, G), 1.0 / np.sqrt(G)))


def test_h4_is_the_printed_matrix():
    check_h4()


def test_R_is_the_kronecker_power():
    check_R_kron()


def test_R_orthogonal_symmetric_regular():
    check_R_algebra()


def test_group_rule():
    for G in GROUPS:
        assert orc.is_valid_group(G, 3 * G)
    for G in (2, 3, 8, 12, 32, 128, 512, 0, -4):
        assert not orc.is_valid_group(G, 4096)
    assert not orc.is_valid_group(256, 1000)
    with pytest.raises(ValueError):
        orc.rotate(np.zeros((2, 96), np.float32), 64)


# --------------------------------------------------------------------------
# rotation
# --------------------------------------------------------------------------

def _exact_fp32_round(fr: Fraction) -> np.float32:
    """Round an exact rational to the nearest fp32 (ties to even), by search."""
    x = np.float32(float(fr))           # within a few ulp of the answer
    cands = [x]
    for _ in range(3):
        cands.append(np.nextafter(cands[-1], np.float32(np.inf)))
    y = x
    for _ in range(3):
        y = np.nextafter(y, np.float32(-np.inf))
        cands.append(y)
    best = min(cands, key=lambda c: (abs(Fraction(float(c)) - fr),
                                     int(np.array(c).view(np.int32)) & 1))
    return np.float32(best)


def check_rotate_exact(mod=orc):
    """Brute force: each output is the exact dot product with the group's
    R column (exact rationals), rounded once to fp32."""
    rng = workloads.rng_for(11)
    H = printed_h4()
    for G, K in ((4, 12), (16, 32), (64, 64)):
        X = workloads.activations(rng, 3, K, outlier_frac=0.1, outlier_mult=30.0)
        Rf = [[Fraction(v) for v in row] for row in kron_power(H, G)]
        got = mod.rotate(X, G)
        for r in range(3):
            for c in range(K):
                g0 = (c // G) * G
                acc = Fraction(0)
                for i in range(G):
                    acc += Fraction(float(X[r, g0 + i])) * Rf[i][c - g0]
                assert got[r, c] == _exact_fp32_round(acc), (G, r, c)


def test_rotate_is_the_correctly_rounded_product():
    check_rotate_exact()


def test_rotation_identity_fp64():
    """X R (W R)^T = X W^T (How INT8 convrot works), fp64 on small inputs."""
    rng = workloads.rng_for(12)
    for G in (4, 16, 64, 256):
        K = 2 * G
        X = rng.standard_normal((5, K))
        W = rng.standard_normal((7, K))
        R = np.kron(np.eye(K // G), orc.hadamard_matrix(G))
        lhs = (X @ R) @ (W @ R).T
        np.testing.assert_allclose(lhs, X @ W.T, rtol=1e-12, atol=1e-12)


def test_rotation_keeps_row_norms_and_groups():
    rng = workloads.rng_for(13)
    X = workloads.activations(rng, 8, 1024, outlier_frac=0.02, outlier_mult=40.0)
    for G in GROUPS:
        Y = orc.rotate(X, G).astype(np.float64)
        x64 = X.astype(np.float64)
        for g in range(1024 // G):
            sl = slice(g * G, (g + 1) * G)
            np.testing.assert_allclose(np.linalg.norm(Y[:, sl], axis=1),
                                       np.linalg.norm(x64[:, sl], axis=1), rtol=1e-6)
    np.testing.assert_array_equal(orc.rotate(X, 1), X)   # G = 1 is the identity


def test_rotation_of_group_constant_rows():
    """Rows of R sum to 1, so a row constant on each group is unchanged."""
    for G in (4, 16, 64, 256, 1024):
        X = np.repeat(np.array([[1.5, -2.0, 0.25]], np.float32), G, axis=1)
        np.testing.assert_array_equal(orc.rotate(X, G), X)


def test_one_hot_closed_form():
    """x = c e_j spreads to +-c/sqrt(G) over its group: |Q| = 127 there,
    zero elsewhere, s = (|c|/sqrt G)/127 (the outlier-spreading purpose)."""
    K = 2048
    for G in (4, 16, 64, 256, 1024):
        for j, c in ((0, 3.0), (G + 5, -40.0), (K - 1, 1000.0)):
            X = np.zeros((1, K), np.float32)
            X[0, j] = c
            Q, s = orc.pack(X, G)
            g0 = (j // G) * G
            mag = np.float32(abs(c) / np.sqrt(G))
            assert s[0] == np.float32(mag / np.float32(127))
            R = orc.hadamard_matrix(G)
            expect = np.zeros(K, np.int8)
            expect[g0:g0 + G] = (np.sign(c) * np.sign(R[j - g0])).astype(np.int8) * 127
            np.testing.assert_array_equal(Q[0], expect)


# --------------------------------------------------------------------------
# quantizer (Runtime activation quantization / Weight quantization)
# --------------------------------------------------------------------------

def check_round_half_even(mod=orc):
    # row max 254 -> s = 2 exactly; x/s lands exactly on k + 1/2
    X = np.array([[254, 1, 3, 5, -1, -3, 7, 0]], np.float32)
    Q, s = mod.quantize_rows(X)
    assert s[0] == np.float32(2.0)
    np.testing.assert_array_equal(Q[0], np.array([127, 0, 2, 2, 0, -2, 4, 0], np.int8))


def test_round_half_to_even():
    check_round_half_even()


def check_quantizer_invariants(mod=orc):
    rng = workloads.rng_for(14)
    X = workloads.activations(rng, 64, 512, outlier_frac=0.01, outlier_mult=50.0)
    for G in (1, 4, 64, 256):
        Xr = mod.rotate(X, G)
        Q, s = mod.quantize_rows(Xr)
        assert Q.dtype == np.int8 and s.dtype == np.float32
        assert Q.min() >= -127 and Q.max() <= 127
        np.testing.assert_array_equal(np.abs(Q).max(axis=1), 127)
        amax = np.abs(Xr).max(axis=1).astype(np.float64)
        np.testing.assert_allclose(s.astype(np.float64), amax / 127.0, rtol=2**-23)
        err = np.abs(Xr.astype(np.float64) - Q.astype(np.float64) * s[:, None])
        assert np.all(err <= s[:, None] * (0.5 + 1e-5))
        # odd symmetry and monotonicity of the quantizer within each row
        Qn, sn = mod.quantize_rows(-Xr)
        np.testing.assert_array_equal(Qn, -Q)
        np.testing.assert_array_equal(sn, s)
        order = np.argsort(Xr, axis=1, kind="stable")
        assert np.all(np.diff(np.take_along_axis(Q.astype(np.int32), order, axis=1), axis=1) >= 0)


def test_quantizer_invariants():
    check_quantizer_invariants()


def test_zero_rows():
    X = np.zeros((3, 256), np.float32)
    X[1, 7] = 2.0
    Q, s = orc.pack(X, 256)
    assert s[0] == 0 and s[2] == 0 and s[1] > 0
    assert not Q[0].any() and not Q[2].any()


def test_g1_is_plain_absmax_quantization():
    """G = 1: the rotation is the identity and the pack is textbook per-row
    absmax quantization; compare with a direct Fraction-based evaluation of
    round(x / s) where s and x/s are fp32 results."""
    rng = workloads.rng_for(15)
    X = workloads.activations(rng, 4, 32, outlier_frac=0.1, outlier_mult=20.0)
    Q, s = orc.pack(X, 1)
    for r in range(4):
        a = max(abs(Fraction(float(v))) for v in X[r])
        s_r = _exact_fp32_round(a / 127)
        assert s[r] == s_r
        for i in range(32):
            qf = _exact_fp32_round(Fraction(float(X[r, i])) / Fraction(float(s_r)))
            qi = int(np.rint(np.float64(qf)))
            assert Q[r, i] == max(-127, min(127, qi))


# --------------------------------------------------------------------------
# integer GEMM and reconstruction
# --------------------------------------------------------------------------

def check_gemm_bruteforce(mod=orc):
    rng = workloads.rng_for(16)
    Qx = workloads.random_codes(rng, 5, 48)
    Qw = workloads.random_codes(rng, 7, 48)
    A = mod.gemm_s32(Qx, Qw)
    assert A.dtype == np.int32 and A.shape == (5, 7)
    for r in range(5):
        for o in range(7):
            assert A[r, o] == sum(int(Qx[r, i]) * int(Qw[o, i]) for i in range(48))


def test_gemm_bruteforce():
    check_gemm_bruteforce()


def test_gemm_extremes():
    K = 133144  # largest K whose worst case fits int32: 133144 * 127^2 < 2^31
    Qx = np.full((2, K), 127, np.int8)
    Qw = np.full((2, K), 127, np.int8)
    Qw[1] = -127
    A = orc.gemm_s32(Qx, Qw)
    assert A[0, 0] == K * 127 * 127 and A[0, 1] == -K * 127 * 127
    with pytest.raises(OverflowError):
        orc.gemm_s32(np.zeros((1, K + 1), np.int8), np.zeros((1, K + 1), np.int8))


def check_reconstruct_exact(mod=orc):
    A = np.array([[3, -8], [0, 1 << 20]], np.int32)
    s_x = np.array([0.5, 2.0], np.float32)
    s_w = np.array([0.25, 4.0], np.float32)
    b = np.array([1.0, -0.5], np.float32)
    Y = mod.reconstruct(A, s_x, s_w, b)
    np.testing.assert_array_equal(Y, np.array([[1.375, -16.5], [1.0, 8.0 * (1 << 20) - 0.5]], np.float32))
    np.testing.assert_array_equal(mod.reconstruct(A, s_x), np.array([[1.5, -4.0], [0.0, 2.0 * (1 << 20)]], np.float32))
    np.testing.assert_array_equal(mod.reconstruct(A, s_x, None, b), np.array([[2.5, -4.5], [1.0, 2.0 * (1 << 20) - 0.5]], np.float32))


def test_reconstruct_exact_cases():
    check_reconstruct_exact()


def test_reconstruct_rounds_int32_once():
    """|A| above 2^24 is itself rounded when converted to fp32."""
    A = np.array([[(1 << 24) + 1]], np.int32)
    Y = orc.reconstruct(A, np.array([1.0], np.float32), np.array([1.0], np.float32), np.array([0.0], np.float32))
    assert Y[0, 0] == np.float32(1 << 24)


def check_linear_error_bound(mod=orc):
    """Y differs from X W^T + b by at most the quantization error bound
    sum_i |x_rot_i| s_w/2 + |q_w,i s_w| s_x/2 (plus fp32 rounding)."""
    case = workloads.make_case(workloads.get("tiny"))
    X, W, b = case.X, case.Ws[0], case.bs[0]
    G = 256
    Qw, s_w = mod.prepare_weight(W, G)
    Y = mod.linear(X, Qw, s_w, b, G)
    ref = X.astype(np.float64) @ W.astype(np.float64).T + b
    Xr = mod.rotate(X, G).astype(np.float64)
    _, s_x = mod.pack(X, G)
    wq = Qw.astype(np.float64) * s_w[:, None]
    bound = (np.abs(Xr) @ np.ones_like(wq.T)) * (s_w[None, :] / 2) \
        + (np.ones_like(Xr) @ np.abs(wq).T) * (s_x[:, None] / 2)
    err = np.abs(Y - ref)
    assert np.all(err <= bound * 1.001 + 1e-5), float(np.max(err / bound))
    # and the approximation is useful: error well below the output scale
    assert np.max(err) < 0.05 * np.max(np.abs(ref))


def test_linear_within_quantization_error():
    check_linear_error_bound()


def test_rotation_spreads_outliers():
    """With a channel outlier the rotated quantization error is smaller than
    the unrotated one (the purpose stated in How INT8 convrot works)."""
    rng = workloads.rng_for(17)
    X = workloads.activations(rng, 64, 1024, outlier_kind="channel",
                              outlier_frac=0.005, outlier_mult=30.0)
    def rel_err(G):
        Q, s = orc.pack(X, G)
        Xr = orc.rotate(X, G).astype(np.float64)
        return np.linalg.norm(Xr - Q * s[:, None].astype(np.float64)) / np.linalg.norm(Xr)
    assert rel_err(256) < 0.5 * rel_err(1)


def test_gelu_reference_points():
    y = np.array([0.0, 1.0, -1.0, 3.0], np.float32)
    # Phi(1) = 0.8413447460685429..., Phi(3) = 0.9986501019683699
    expect = np.array([0.0, 0.8413447460685429, -0.15865525393145707, 3 * 0.9986501019683699])
    np.testing.assert_allclose(orc.gelu(y), expect.astype(np.float32), rtol=1e-7)


# --------------------------------------------------------------------------
# planted mistakes: each must trip at least one pin
# --------------------------------------------------------------------------

class _Mutant:
    """A copy of the oracle namespace with one function replaced."""

    def __init__(self, **over):
        for k in dir(orc):
            if not k.startswith("__"):
                setattr(self, k, getattr(orc, k))
        for k, v in over.items():
            setattr(self, k, v)
        # rebind helpers that call each other through the module
        me = self

        def pack(X, G):
            return me.quantize_rows(me.rotate(X, G))

        def prepare_weight(W, G):
            return me.quantize_rows(me.rotate(W, G))

        def linear(X, Qw, s_w, bias, G):
            Qx, s_x = me.pack(X, G)
            return me.reconstruct(me.gemm_s32(Qx, Qw), s_x, s_w, bias)

        for name, fn in (("pack", pack), ("prepare_weight", prepare_weight), ("linear", linear)):
            if name not in over:
                setattr(self, name, fn)


def _fails(mod, checks):
    for chk in checks:
        try:
            chk(mod)
        except AssertionError:
            return True
    return False


ALL_CHECKS = (check_h4, check_R_kron, check_R_algebra, check_rotate_exact,
              check_round_half_even, check_quantizer_invariants,
              check_gemm_bruteforce, check_reconstruct_exact, check_linear_error_bound)


def _bad_h4():
    H = orc.H4.copy()
    H[2, 3] = -H[2, 3]
    return H


def _rotate_wrong_axis(X, G):
    M, K = X.shape
    R = orc.hadamard_matrix(G)
    x = X.astype(np.float64).reshape(M, K // G, G)
    # groups taken with stride K/G instead of contiguous
    x = X.astype(np.float64).reshape(M, G, K // G).transpose(0, 2, 1)
    y = np.einsum("rgi,ij->rgj", x, R)
    return y.transpose(0, 2, 1).reshape(M, K).astype(np.float32)


def _rotate_unnormalised(X, G):
    return (orc.rotate(X, G).astype(np.float64) * np.sqrt(G)).astype(np.float32)


def _quant_half_away(Xrot):
    Xrot = np.asarray(Xrot, np.float32)
    s = (np.abs(Xrot).max(axis=1) / np.float32(127)).astype(np.float32)
    q = Xrot / s[:, None]
    q = np.sign(q) * np.floor(np.abs(q) + 0.5)
    return np.clip(q, -127, 127).astype(np.int8), s


def _quant_scale_255(Xrot):
    Xrot = np.asarray(Xrot, np.float32)
    s = (np.abs(Xrot).max(axis=1) / np.float32(255)).astype(np.float32)
    q = np.rint(Xrot / s[:, None])
    return np.clip(q, -128, 127).astype(np.int8), s


def _gemm_transposed(Qx, Qw):
    return orc.gemm_s32(Qx, Qw[::-1])


def _gemm_offby(Qx, Qw):
    return orc.gemm_s32(Qx[:, 1:], Qw[:, :-1])


def _recon_no_sw(A, s_x, s_w=None, bias=None):
    return orc.reconstruct(A, s_x, None, bias)


def _recon_minus_bias(A, s_x, s_w=None, bias=None):
    Y = orc.reconstruct(A, s_x, s_w, None)
    return Y if bias is None else (Y - np.asarray(bias, np.float32)[None, :]).astype(np.float32)


@pytest.mark.parametrize("mutant", [
    dict(H4=_bad_h4()),
    dict(rotate=_rotate_wrong_axis),
    dict(rotate=_rotate_unnormalised),
    dict(quantize_rows=_quant_half_away),
    dict(quantize_rows=_quant_scale_255),
    dict(gemm_s32=_gemm_transposed),
    dict(gemm_s32=_gemm_offby),
    dict(reconstruct=_recon_no_sw),
    dict(reconstruct=_recon_minus_bias),
], ids=["h4-sign", "rotate-strided-groups", "rotate-unnormalised", "round-half-away",
        "scale-255", "gemm-transposed", "gemm-shifted", "recon-no-sw", "recon-minus-bias"])
def test_planted_mistakes_are_caught(mutant):
    if "H4" in mutant:
        # H4 feeds hadamard_matrix through the module global
        bad = mutant["H4"]

        def hm(G, _bad=bad):
            n = 0
            while 4**n < G:
                n += 1
            R = np.ones((G, G))
            idx = np.arange(G)
            for k in range(n):
                d = (idx // 4**k) % 4
                R *= _bad[d[:, None], d[None, :]]
            return R
        mutant = dict(mutant, hadamard_matrix=hm)
    assert _fails(_Mutant(**mutant), ALL_CHECKS)


def test_oracle_package_exports():
    for name in ("H4", "hadamard_matrix", "rotate", "quantize_rows", "pack",
                 "prepare_weight", "gemm_s32", "reconstruct", "linear", "gelu"):
        assert hasattr(oracle, name)


def test_chunk_plan_reference_rule():
    """The plan reference (tests/chunk_plan_ref.py) on hand-checkable rows:
    all-127 rows allow 16 K-blocks exactly (16 * 64 * 127 * 127 < 2^24 but
    17 blocks would not), all-1 rows allow the whole K."""
    import numpy as np
    from chunk_plan_ref import plan, plan_is_safe
    K = 64 * 48
    full = np.full((128, K), 127, np.int8)
    assert plan(full).tolist() == [16]
    assert 127 * 127 * 64 * 16 <= (1 << 24) - 1 < 127 * 127 * 64 * 17
    ones = np.ones((130, K), np.int8)
    assert plan(ones).tolist() == [48, 48]
    mixed = ones.copy()
    mixed[129] = 127       # the second block holds a dense row
    p = plan(mixed)
    assert p.tolist() == [48, 16] and plan_is_safe(mixed, p)
    assert not plan_is_safe(full, np.array([32], np.int32))


def test_linear_scaled_pins():
    """linear_scaled against what the definition fixes: scale 1 is the plain
    linear; a power-of-two scale commutes exactly with every fp32 step (the
    absmax, both divisions and every product scale by the same power of two),
    so the output equals the plain linear bit for bit; any other scale moves
    codes by at most one step, so Y stays within the quantization error."""
    import numpy as np
    rng = np.random.default_rng(5)
    M, K, N, G = 24, 256, 40, 64
    X = rng.standard_normal((M, K)).astype(np.float32)
    X[3, 7] = 60.0
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    b = (rng.standard_normal(N) * 0.01).astype(np.float32)
    Qw, s_w = oracle.prepare_weight(W, G)
    Y = oracle.linear(X, Qw, s_w, b, G)
    np.testing.assert_array_equal(oracle.linear_scaled(X, Qw, s_w, b, G, 1.0), Y)
    for a in (0.25, 8.0, 2.0 ** -10):
        np.testing.assert_array_equal(oracle.linear_scaled(X, Qw, s_w, b, G, a), Y)
    for a in (3.0, 0.37, 1.7):
        Ys = oracle.linear_scaled(X, Qw, s_w, b, G, a)
        # one code step of X_rot is s_x; through the weights it moves Y by at most
        # s_x * s_w * sum |Q_w| per row/column pair
        Qx, s_x = oracle.pack(X, G)
        bound = np.outer(s_x, s_w * np.abs(Qw.astype(np.float64)).sum(axis=1)) + 1e-6
        assert np.all(np.abs(Ys.astype(np.float64) - Y) <= bound)
        assert not np.array_equal(Ys, Y) or a == 1.0
    # a forgotten unscale is caught: the output would be a times too large
    Qx, s_x = oracle.pack((X * np.float32(3.0)).astype(np.float32), G)
    wrong = oracle.reconstruct(oracle.gemm_s32(Qx, Qw), s_x, s_w, b)
    assert np.max(np.abs(wrong - Y)) > 0.5 * np.max(np.abs(Y))


def check_prologue(mod=orc):
    """The modulation prologue on hand-computed values where every step of
    its definition shows: the RMS norm divides by sqrt(mean(x^2) + eps), with
    eps under the square root and the mean over the row's length; then the
    weight; then (x + x * scale) + shift."""
    f32 = np.float32
    # rows of +-1 (mean x^2 = 1) with eps = 3: 1 / sqrt(1 + 3) = 0.5 exactly,
    # where eps outside the root, 1 / (sqrt(1) + 3), would give 0.25
    x = np.array([[1.0, -1.0, 1.0, 1.0], [-1.0, -1.0, 1.0, -1.0]], f32)
    np.testing.assert_array_equal(mod.prologue(x, rmsnorm=True, eps=3.0), x * f32(0.5))
    # the mean, not the sum: a row of +-2 of length 4 has mean x^2 = 4;
    # eps = 12 gives 1 / sqrt(16) = 0.25, so x * r = +-0.5
    y = np.array([[2.0, -2.0, 2.0, 2.0]], f32)
    np.testing.assert_array_equal(mod.prologue(y, rmsnorm=True, eps=12.0), y * f32(0.25))
    # the order of the per-channel steps: ((x * r) * w + (x * r) * w * scale) + shift
    z = np.array([[1.0, -1.0, 1.0, -1.0]], f32)
    got = mod.prologue(z, rmsnorm=True, eps=3.0, weight=np.full(4, 4.0, f32), scale=np.full(4, 0.5, f32),
                       shift=np.full(4, 1.0, f32))
    # x r = +-0.5; times 4 = +-2; (+-2 + +-2 * 0.5) = +-3; + 1 = 4 or -2
    np.testing.assert_array_equal(got, np.array([[4.0, -2.0, 4.0, -2.0]], f32))


def test_prologue_eps_and_order():
    check_prologue()


def _prologue_eps_outside_root(X, rmsnorm=False, eps=1e-6, weight=None, scale=None, shift=None):
    x = np.asarray(X).astype(np.float32)
    if rmsnorm:
        ms = (x.astype(np.float64) ** 2).mean(axis=1)
        x = (x / (np.sqrt(ms) + eps)[:, None]).astype(np.float32)
    return orc.prologue(x, False, eps, weight, scale, shift)


def _prologue_sum_not_mean(X, rmsnorm=False, eps=1e-6, weight=None, scale=None, shift=None):
    x = np.asarray(X).astype(np.float32)
    if rmsnorm:
        ss = (x.astype(np.float64) ** 2).sum(axis=1)
        x = (x / np.sqrt(ss + eps)[:, None]).astype(np.float32)
    return orc.prologue(x, False, eps, weight, scale, shift)


def _prologue_shift_then_scale(X, rmsnorm=False, eps=1e-6, weight=None, scale=None, shift=None):
    x = orc.prologue(X, rmsnorm, eps, weight, None, shift)
    return orc.prologue(x, False, eps, None, scale, None)


@pytest.mark.parametrize("bad", [_prologue_eps_outside_root, _prologue_sum_not_mean, _prologue_shift_then_scale],
                         ids=["eps-outside-root", "sum-not-mean", "shift-before-scale"])
def test_planted_prologue_mistakes_are_caught(bad):
    assert _fails(_Mutant(prologue=bad), (check_prologue,))


def test_prologue_pins():
    """The modulation prologue against values fixed by its definition."""
    import numpy as np
    f32 = np.float32
    # nothing requested: identity
    X = np.random.default_rng(3).standard_normal((5, 64)).astype(f32)
    np.testing.assert_array_equal(oracle.prologue(X), X)
    # (x + x * scale) + shift, not x * scale + shift: 2 + 2 * 0.5 + 1 = 4
    one = np.array([[2.0]], f32)
    assert oracle.prologue(one, scale=np.array([0.5], f32), shift=np.array([1.0], f32))[0, 0] == 4.0
    assert oracle.prologue(one, weight=np.array([3.0], f32))[0, 0] == 6.0
    # RMS norm of a constant power-of-two row with eps = 0 is exactly +-1
    c = np.full((2, 256), 4.0, f32)
    c[1] = -0.25
    np.testing.assert_array_equal(oracle.prologue(c, rmsnorm=True, eps=0.0), np.sign(c))
    # RMS norm rescales each row by one factor, which the absmax quantizer
    # divides out: the codes stay (up to rare rounding) and s_x shrinks by r
    X = np.random.default_rng(4).standard_normal((16, 512)).astype(f32) * 7.0
    Xn = oracle.prologue(X, rmsnorm=True, eps=1e-6)
    Q0, s0 = oracle.pack(X, 64)
    Q1, s1 = oracle.pack(Xn, 64)
    assert np.count_nonzero(Q0 != Q1) <= 0.001 * Q0.size and np.abs(Q0.astype(int) - Q1).max() <= 1
    rms = np.sqrt((X.astype(np.float64) ** 2).mean(axis=1) + 1e-6)
    np.testing.assert_allclose(s1, s0 / rms, rtol=1e-5)


def test_unpack_w4_pins():
    """Packed INT4 layout: low nibble first, two's complement in [-8, 7]."""
    import numpy as np
    packed = np.array([[0x8F, 0x71, 0x00, 0xF8]], np.uint8)
    assert oracle.unpack_w4(packed).tolist() == [[-1, -8, 1, 7, 0, 0, -8, -1]]
    # every byte value round-trips through its two nibbles
    allb = np.arange(256, dtype=np.uint8)[None, :]
    q = oracle.unpack_w4(allb).astype(np.int16)
    back = ((q[:, 0::2] & 0xF) | ((q[:, 1::2] & 0xF) << 4)).astype(np.uint8)
    np.testing.assert_array_equal(back, allb)
    assert q.min() == -8 and q.max() == 7


def check_silu_mul(mod=orc):
    """silu(g) * u against facts of the logistic function: silu(0) = 0;
    silu(1) = e / (1 + e) and silu(-1) = -1 / (1 + e); silu(g) - silu(-g) = g;
    silu(g) = g (1 + tanh(g / 2)) / 2; silu saturates to g for large g and to
    0 for very negative g; the gate is the silu argument, the up input only
    scales it."""
    import math
    f32 = np.float32
    e = math.e
    one = np.ones(5, f32)
    g = np.array([0.0, 1.0, -1.0, 40.0, -200.0], f32)
    h = mod.silu_mul(g, one).astype(np.float64)
    expect = [0.0, e / (1 + e), -1 / (1 + e), 40.0, 0.0]
    np.testing.assert_allclose(h, np.array(expect, f32), rtol=1e-7, atol=1e-30)
    x = np.linspace(-6, 6, 49).astype(f32)
    d = mod.silu_mul(x, np.ones_like(x)).astype(np.float64) - mod.silu_mul(-x, np.ones_like(x)).astype(np.float64)
    np.testing.assert_allclose(d, x.astype(np.float64), rtol=1e-6, atol=1e-6)
    th = x.astype(np.float64) * (1 + np.tanh(x.astype(np.float64) / 2)) / 2
    np.testing.assert_allclose(mod.silu_mul(x, np.ones_like(x)), th.astype(f32), rtol=1e-6, atol=1e-7)
    # the up input scales the result linearly; the gate is not symmetric with it
    u = np.full_like(x, 3.0)
    np.testing.assert_allclose(mod.silu_mul(x, u), 3.0 * mod.silu_mul(x, np.ones_like(x)), rtol=1e-6, atol=1e-6)
    assert mod.silu_mul(np.array([2.0], f32), np.array([-1.0], f32))[0] != \
        mod.silu_mul(np.array([-1.0], f32), np.array([2.0], f32))[0]


def test_silu_mul_pins():
    check_silu_mul()


def _silu_swapped(gate, up):
    return orc.silu_mul(up, gate)


def _sigmoid_only(gate, up):
    g = np.asarray(gate, np.float64)
    return (np.asarray(up, np.float64) / (1.0 + np.exp(-g))).astype(np.float32)


@pytest.mark.parametrize("bad", [_silu_swapped, _sigmoid_only], ids=["gate-up-swapped", "sigmoid-not-silu"])
def test_planted_silu_mistakes_are_caught(bad):
    assert _fails(_Mutant(silu_mul=bad), (check_silu_mul,))


def test_linear_swiglu_is_the_two_linears():
    """linear_swiglu is silu_mul of the two convrot linears on the same pack."""
    rng = np.random.default_rng(8)
    M, K, N, G = 12, 256, 40, 64
    X = rng.standard_normal((M, K)).astype(np.float32)
    Wg = (rng.standard_normal((N, K)) * 0.05).astype(np.float32)
    Wu = (rng.standard_normal((N, K)) * 0.05).astype(np.float32)
    Qg, sg = oracle.prepare_weight(Wg, G)
    Qu, su = oracle.prepare_weight(Wu, G)
    h = oracle.linear_swiglu(X, Qg, sg, None, Qu, su, None, G)
    np.testing.assert_array_equal(h, oracle.silu_mul(oracle.linear(X, Qg, sg, None, G), oracle.linear(X, Qu, su, None, G)))
    # and it approximates silu(X Wg^T) * (X Wu^T) within the quantization error
    ref = X.astype(np.float64) @ Wg.T.astype(np.float64)
    ref = ref / (1 + np.exp(-ref)) * (X.astype(np.float64) @ Wu.T.astype(np.float64))
    assert np.max(np.abs(h - ref)) <= 0.05 * np.max(np.abs(ref))


"""Pins of the value rotation R_V = U_S H P_br (OSCAR page, section "attention-statistics rotation
+ Triton kernels": C_S = (1/N) V^T S^T S V, score-weighted value covariance) and of its absorption
into the value and output projections, checked against linear-algebra facts: two associations of
C_S, the eigen-decomposition it must produce, orthogonality, and an unchanged attention output."""
import numpy as np
import scipy.linalg

D = 128


def _calibration(seed, n=96, t=300):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((n, D)) * np.linspace(2.0, 0.2, D)        # anisotropic queries
    k = rng.standard_normal((t, D))
    v = rng.standard_normal((t, D)) * np.exp(0.5 * rng.standard_normal(D))
    return q, k, v


def test_value_covariance_two_associations(orc):
    q, k, v = _calibration(1)
    y = orc.score_weighted_values(q, k, v)              # rows of S V
    c_rows = y.T @ y / q.shape[0]                       # (1/N) (S V)^T (S V)
    c_def = orc.value_covariance(q, k, v)               # (1/N) V^T (S^T S) V, as printed
    assert np.allclose(c_rows, c_def, rtol=1e-12, atol=1e-14)
    # the softmax rows of S sum to one: S V of a constant value column is that constant
    vc = np.tile(np.linspace(-1, 1, D), (k.shape[0], 1))
    assert np.allclose(orc.score_weighted_values(q, k, vc), vc[:q.shape[0]], atol=1e-12)


def test_rv_orthogonal_and_diagonalises_cs(orc):
    q, k, v = _calibration(2)
    r32, r64, ev = orc.build_rv(q, k, v)
    assert np.abs(r64 @ r64.T - np.eye(D)).max() < 1e-12
    assert np.abs(r32.astype(np.float64) @ r32.T.astype(np.float64) - np.eye(D)).max() < 1e-6
    c = orc.value_covariance(q, k, v)
    ref = scipy.linalg.eigh(c, eigvals_only=True)[::-1]
    assert np.allclose(ev, ref, rtol=1e-9, atol=1e-12)
    assert (np.diff(ev) <= 1e-15).all()
    # undo the Hadamard / bit reversal: the remaining basis U_S diagonalises C_S
    pbr = np.zeros((D, D))
    pbr[np.arange(D), [orc.bitrev7(i) for i in range(D)]] = 1.0
    u = r64 @ np.linalg.inv(orc.hadamard128() @ pbr)
    d = u.T @ c @ u
    assert np.abs(d - np.diag(np.diag(d))).max() < 1e-9 * np.abs(ev).max()
    assert np.allclose(np.diag(d), ev, rtol=1e-9, atol=1e-12)


def test_rk_builder_on_score_weighted_samples_gives_rv(orc):
    # R_K's builder takes samples and forms (1/n) sum y^T y: fed rows of S V it targets C_S
    q, k, v = _calibration(3)
    y = orc.score_weighted_values(q, k, v).astype(np.float32)
    _, r64_samples, ev_samples = orc.build_rk(y)
    _, r64_def, ev_def = orc.build_rv(q, k, v)
    assert np.allclose(ev_samples, ev_def, rtol=1e-5, atol=1e-9)     # fp32 samples vs fp64 C_S
    for r in (r64_samples, r64_def):
        assert np.abs(r @ r.T - np.eye(D)).max() < 1e-12


def test_absorption_into_value_and_output_projections(orc):
    # V' = X W_V R_V and W_O' = R_V^T W_O leave attention's output unchanged
    rng = np.random.default_rng(4)
    d_model, t = 256, 200
    x = rng.standard_normal((t, d_model))
    w_k = rng.standard_normal((d_model, D)) / np.sqrt(d_model)
    w_v = rng.standard_normal((d_model, D)) / np.sqrt(d_model)
    w_o = rng.standard_normal((D, d_model)) / np.sqrt(D)
    q_cal = rng.standard_normal((64, D))
    _, r_v, _ = orc.build_rv(q_cal, x @ w_k, x @ w_v)
    q = rng.standard_normal((5, D))
    out = orc.score_weighted_values(q, x @ w_k, x @ w_v) @ w_o
    out_rot = orc.score_weighted_values(q, x @ w_k, x @ (w_v @ r_v)) @ (r_v.T @ w_o)
    assert np.allclose(out, out_rot, rtol=1e-10, atol=1e-12)
    # the rotated values are what a cache would store; they differ from the plain ones
    assert not np.allclose(x @ w_v, x @ (w_v @ r_v))

"""Pins of the OptR calibration oracle (oracle/optr.py), CPU only.

* the backward pass (straight-through quantiser, softmax, KL, post-W_O error,
  rotation, matrix-exponential adjoint) against central finite differences of
  the same objectives with the clip surrogate, whose exact derivative equals
  the straight-through derivative of the INT2 quantiser;
* the adjoint of the Frechet derivative of exp against finite differences;
* the INT2 quantiser forward against the C oracle's quantiser (an independent
  implementation of the library's fp32/fp16 quantiser);
* Adam against torch.optim.Adam; the causal softmax against a loop;
* special cases: an exact quantiser gives zero loss and zero gradient; R stays
  orthogonal; a short calibration lowers both losses.
"""
import numpy as np
import pytest

import oracle
from oracle import optr


def _orth(rng, d):
    q, r = np.linalg.qr(rng.standard_normal((d, d)))
    return q * np.sign(np.diag(r))[None, :]


def _case(seed=0, T=40, Nq=6, G=2, D=8, Dm=12):
    rng = np.random.default_rng(seed)
    K = rng.standard_normal((T, D)) + rng.standard_normal(D)[None, :] * 2
    V = rng.standard_normal((T, D))
    Q = rng.standard_normal((Nq, G, D)) * 1.5
    W = rng.standard_normal((G, Dm, D)) / np.sqrt(G * D)
    mu = K.mean(axis=0)
    R0 = _orth(rng, D)
    A = rng.standard_normal((D, D)) * 0.05
    return K, V, Q, W, mu, R0, A


def _fd(f, A, eps=1e-6, picks=None, rng=None):
    """Central differences of f at A in random directions (returns pairs of
    (directional derivative, <grad, dir>))."""
    out = []
    rng = rng or np.random.default_rng(5)
    for _ in range(picks or 6):
        H = rng.standard_normal(A.shape)
        out.append((f(A + eps * H) - f(A - eps * H)) / (2 * eps))
    return out


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_key_gradient_matches_finite_differences(seed):
    K, V, Q, W, mu, R0, A = _case(seed)
    f = lambda X: optr.key_loss(X, R0, K, V, Q, W, mu, 0.9, lam=0.7, mode="clip")[0]
    L, g, aux = optr.key_loss(A, R0, K, V, Q, W, mu, 0.9, lam=0.7, mode="clip")
    assert aux["kl"] > 0 and aux["err"] > 0
    rng = np.random.default_rng(11 + seed)
    for _ in range(6):
        H = rng.standard_normal(A.shape)
        fd = (f(A + 1e-6 * H) - f(A - 1e-6 * H)) / 2e-6
        assert abs(fd - (g * H).sum()) <= 1e-6 * max(1.0, abs(fd)), (fd, (g * H).sum())


@pytest.mark.parametrize("seed", [0, 3])
def test_value_gradient_matches_finite_differences(seed):
    K, V, Q, W, mu, R0, A = _case(seed)
    pt = optr.causal_softmax(Q, K, 1 / np.sqrt(K.shape[1]))
    f = lambda X: optr.value_loss(X, R0, V, pt, W, 0.85, mode="clip")[0]
    L, g, _ = optr.value_loss(A, R0, V, pt, W, 0.85, mode="clip")
    assert L > 0
    rng = np.random.default_rng(21 + seed)
    for _ in range(6):
        H = rng.standard_normal(A.shape)
        fd = (f(A + 1e-6 * H) - f(A - 1e-6 * H)) / 2e-6
        assert abs(fd - (g * H).sum()) <= 1e-6 * max(1.0, abs(fd))


def test_expm_adjoint_is_the_transpose_frechet():
    import scipy.linalg
    rng = np.random.default_rng(7)
    S = optr.skew(rng.standard_normal((6, 6)) * 0.4)
    Gb = rng.standard_normal((6, 6))
    adj = optr.expm_adjoint(S, Gb)
    for _ in range(5):
        H = rng.standard_normal((6, 6))
        fd = ((Gb * (scipy.linalg.expm(S + 1e-6 * H) - scipy.linalg.expm(S - 1e-6 * H))).sum()
              / 2e-6)
        assert abs(fd - (adj * H).sum()) <= 1e-7 * max(1.0, abs(fd))


def test_int2_quantiser_matches_the_c_oracle():
    """With R = I the C oracle's fmaf chain returns r = x exactly, so both
    quantisers see the same fp32 vector."""
    rng = np.random.default_rng(3)
    I = np.eye(128, dtype=np.float32)
    for i in range(40):
        x = (rng.standard_normal(128) * (0.5 + i)).astype(np.float32)
        bits = ((x.view(np.uint32) + 0x7FFF + ((x.view(np.uint32) >> 16) & 1)) >> 16)
        bits = bits.astype(np.uint16)                     # bf16, round to nearest even
        xr = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        code, s16, z16, r, t = oracle.quantize(bits, I, 0.92)
        s = np.float16(np.frombuffer(np.uint16(s16).tobytes(), np.float16)[0]).astype(np.float32)
        z = np.float16(np.frombuffer(np.uint16(z16).tobytes(), np.float16)[0]).astype(np.float32)
        want = code.astype(np.float32) * s + z
        got, _ = optr.quantise(xr[None, :], 0.92, "int2")
        assert np.array_equal(got[0].astype(np.float32), want), i


def test_adam_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(4)
    A = rng.standard_normal((5, 5))
    target = rng.standard_normal((5, 5))
    p = torch.nn.Parameter(torch.tensor(A.copy()))
    opt = torch.optim.Adam([p], lr=0.01)
    m = np.zeros_like(A)
    v = np.zeros_like(A)
    for t in range(1, 8):
        g = 2 * (A - target) + np.sin(A)
        A, m, v = optr.adam_step(A, g, m, v, t, 0.01)
        opt.zero_grad()
        loss = ((p - torch.tensor(target)) ** 2).sum() - torch.cos(p).sum()
        loss.backward()
        opt.step()
        assert np.allclose(A, p.detach().numpy(), rtol=0, atol=1e-12)


def test_causal_softmax_against_a_loop():
    rng = np.random.default_rng(9)
    T, Nq, G, D = 13, 4, 2, 5
    Q = rng.standard_normal((Nq, G, D))
    K = rng.standard_normal((T, D))
    p = optr.causal_softmax(Q, K, 0.3)
    for i in range(Nq):
        pos = T - Nq + i
        for h in range(G):
            l = np.array([0.3 * Q[i, h] @ K[s] for s in range(pos + 1)])
            w = np.exp(l - l.max())
            w /= w.sum()
            assert np.allclose(p[i, h, :pos + 1], w, rtol=0, atol=1e-14)
            assert not p[i, h, pos + 1:].any()


def test_exact_quantiser_gives_zero_loss_and_gradient():
    K, V, Q, W, mu, R0, A = _case(4)
    L, g, _ = optr.key_loss(A, R0, K, V, Q, W, mu, 1.0, mode="clip")
    assert abs(L) < 1e-12 and np.abs(g).max() < 1e-10
    pt = optr.causal_softmax(Q, K, 0.35)
    L, g, _ = optr.value_loss(A, R0, V, pt, W, 1.0, mode="clip")
    assert abs(L) < 1e-20 and np.abs(g).max() < 1e-10


def test_rotation_stays_orthogonal_and_calibration_lowers_the_losses():
    rng = np.random.default_rng(6)
    T, Nq, G, D, Dm = 256, 32, 4, 128, 256
    K = rng.standard_normal((T, D)) + rng.normal(0, 2, D)[None, :]
    K[:, :4] = rng.standard_t(3, size=(T, 4)) * 8
    V = rng.standard_normal((T, D))
    Q = rng.standard_normal((Nq, G, D))
    W = rng.standard_normal((G, Dm, D)) / np.sqrt(G * D)
    mu = K.mean(axis=0)
    R0K, R0V = _orth(rng, D), _orth(rng, D)
    RK, RV, h = optr.calibrate(R0K, R0V, K, V, Q, W, mu, 0.96, 0.92, lr=2e-3, steps=12)
    for R in (RK, RV):
        assert np.abs(R.T @ R - np.eye(D)).max() < 1e-12
    assert h["key"][-1] < h["key"][0] and h["value"][-1] < h["value"][0]


def _attend(Q, Kx, Vx, W, scale):
    """Post-W_O outputs y [Nq, Dm] of causal attention, by explicit loops:
    y_q = sum_h (sum_t p_qht v_t) W[h]^T."""
    T = Kx.shape[0]
    Nq, G, _ = Q.shape
    y = np.zeros((Nq, W.shape[1]))
    P = np.zeros((Nq, G, T))
    for i in range(Nq):
        pos = T - Nq + i
        for h in range(G):
            logit = np.array([scale * (Q[i, h] @ Kx[t]) for t in range(pos + 1)])
            w = np.exp(logit - logit.max())
            w /= w.sum()
            P[i, h, :pos + 1] = w
            o = sum(w[t] * Vx[t] for t in range(pos + 1))
            y[i] += W[h] @ o
    return y, P


@pytest.mark.parametrize("seed", [0, 1])
def test_objectives_follow_the_post_wo_error_decomposition(seed):
    """Eq. 8 ("What carries the argument"): with k~, v~ the dequantised keys and
    values, y~ - y = (sum_t (p~_t - p_t) v_t) W_O^T + (sum_t p~_t (v~_t - v_t)) W_O^T.
    The two error vectors the objectives use are checked against y~ - y built
    from attention computed by loops, which pins their signs, which attention
    each term is taken at and the normalisation of both losses and of the KL."""
    import scipy.linalg
    K, V, Q, W, mu, R0, A = _case(seed, G=3)
    rng = np.random.default_rng(40 + seed)
    R0v = _orth(rng, K.shape[1])
    B = rng.standard_normal(A.shape) * 0.05
    clip_k, clip_v, lam = 0.96, 0.92, 0.7
    D = K.shape[1]
    scale = 1.0 / np.sqrt(D)
    Nq = Q.shape[0]
    Lk, _, ak = optr.key_loss(A, R0, K, V, Q, W, mu, clip_k, lam=lam)
    Lv, _, av = optr.value_loss(B, R0v, V, ak["pt"], W, clip_v)
    # dequantised keys and values, rotations built here from their definition
    RK = R0 @ scipy.linalg.expm(A - A.T)
    RV = R0v @ scipy.linalg.expm(B - B.T)
    kt = optr.quantise((K - mu) @ RK, clip_k)[0] @ RK.T + mu
    vt = optr.quantise(V @ RV, clip_v)[0] @ RV.T
    y, p = _attend(Q, K, V, W, scale)
    y_k, pt = _attend(Q, kt, V, W, scale)          # keys quantised, values exact
    y_kv, _ = _attend(Q, kt, vt, W, scale)         # both quantised
    dy = y_kv - y
    tol = 1e-12 * np.linalg.norm(dy)
    assert np.linalg.norm(pt - ak["pt"]) <= 1e-12 * np.linalg.norm(pt)
    assert np.linalg.norm(ak["e"] - (y_k - y)) <= tol          # key-induced term
    assert np.linalg.norm(av["e"] - (y_kv - y_k)) <= tol       # value-induced term
    assert np.linalg.norm(ak["e"] + av["e"] - dy) <= tol
    # the same split with the attention of exact keys and an explicit cross term
    y_v, _ = _attend(Q, K, vt, W, scale)
    cross = dy - (y_k - y) - (y_v - y)
    assert np.linalg.norm((y_k - y) + (y_v - y) + cross - dy) <= tol
    assert np.linalg.norm(cross) > 1e-6 * np.linalg.norm(dy)   # the cross term is not zero
    # normalisation: mean over queries of squared norms; KL summed over heads
    err_k = (np.linalg.norm(y_k - y, axis=1) ** 2).mean()
    err_v = (np.linalg.norm(y_kv - y_k, axis=1) ** 2).mean()
    kl = sum(p[i, h, t] * np.log(p[i, h, t] / pt[i, h, t])
             for i in range(Nq) for h in range(Q.shape[1]) for t in range(K.shape[0])
             if p[i, h, t] > 0) / Nq
    assert abs(ak["err"] - err_k) <= 1e-12 * err_k
    assert abs(ak["kl"] - kl) <= 1e-10 * kl
    assert abs(Lk - (kl + lam * err_k)) <= 1e-10 * Lk
    assert abs(Lv - err_v) <= 1e-12 * err_v

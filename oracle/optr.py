"""Oracle of OptR rotation calibration (float64 numpy).

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``: only ``tests/`` and the
CPU legs of ``bench.py`` may import it; the product never does.

What it restates ("Output-Aware Rotation for INT2 KV-Cache Quantization",
pith.science review of arXiv 2608.02691):
  * "What carries the argument", mechanism (1): a per-head correction of a base
    rotation, R = R0 exp(S) with S = A - A^T skew-symmetric, so R stays
    orthogonal;
  * mechanism (2): keys are centred, k -> k - mu, before rotation;
  * mechanism (3): the loss is taken through the whole quantised path (rotate,
    clip, group, round, dequantise, inverse-rotate) with a straight-through
    estimator for the rounding;
  * "What carries the argument" (the post-W_O error decomposition, Eq. 8) and
    the referee report on Eqs. (14) and (16): key calibration minimises a KL
    term plus lambda_K times the key-induced post-W_O error with values in
    BF16; value calibration then minimises the value-induced post-W_O error
    with the quantised-key attention held fixed;
  * "Assumptions & free parameters": lambda_K = 1, Adam, 80 steps per head,
    keys before values; the objective is taken over the last 64 query
    positions of a calibration chunk (causal attention).

Readings where the pages are silent:
  * KL(p || p~) with p the attention of the unquantised keys (teacher);
  * the losses are averaged over the calibration queries; the KL is summed
    over the G query heads of the KV head, and the post-W_O error of a query is
    the squared norm of the sum of its G heads' contributions;
  * A starts at 0; Adam with beta1 0.9, beta2 0.999, eps 1e-8;
  * the quantiser is the library's INT2 quantiser (fp32 arithmetic, fp16 scale
    and zero, round half to even); STE: the rounding is replaced by the
    identity in the backward pass, clipping and the max/min that set the scale
    are differentiated exactly.  That derivative is exactly the derivative of
    clip(r, c min r, c max r), which ``quantise(..., mode="clip")`` computes so
    that finite differences can pin the backward pass.

Shapes for one KV head: keys K, values V [T, D]; queries Q [Nq, G, D] at
positions T - Nq .. T - 1; W_O slice W [G, Dm, D] (head h's output is o_h W[h]^T).
"""
from __future__ import annotations

import numpy as np
import scipy.linalg


def skew(A):
    return A - A.T


def rotation(R0, A):
    """R = R0 exp(A - A^T)."""
    return R0 @ scipy.linalg.expm(skew(A))


# ---- the quantiser and its straight-through backward --------------------------

def quantise(r, clip, mode="int2"):
    """Rows of r (float64) through the INT2 quantiser.  mode "int2": the
    library's fp32/fp16 quantiser (codes from rint); mode "clip": the
    piecewise-linear function clip(r, c min r, c max r) whose exact derivative
    is the straight-through derivative of the INT2 quantiser.  Returns
    (r_tilde float64, info) where info holds what the backward pass needs."""
    r = np.asarray(r, np.float64)
    c32 = np.float32(clip)
    if mode == "int2":
        r32 = r.astype(np.float32)
        mx = r32.max(axis=1, keepdims=True)
        mn = r32.min(axis=1, keepdims=True)
        mxc, mnc = c32 * mx, c32 * mn                       # fp32 products
        s32 = (mxc - mnc) / np.float32(3.0)
        s = s32.astype(np.float16).astype(np.float32)
        z = mnc.astype(np.float16).astype(np.float32)
        with np.errstate(divide="ignore", invalid="ignore"):
            t = (r32 - z) / s
        code = np.where(s != 0, np.clip(np.rint(t), 0, 3), 0).astype(np.float32)
        rt = (code * s + z).astype(np.float64)
        # elements whose code sits at a clamp because the pre-rounding value was
        # outside [0, 3]: their value follows c*max (high) or c*min (low)
        high = (s != 0) & (t > 3)
        low = (s == 0) | (t < 0)
    else:
        mx = r.max(axis=1, keepdims=True)
        mn = r.min(axis=1, keepdims=True)
        hi, lo = float(c32) * mx, float(c32) * mn
        rt = np.clip(r, lo, hi)
        high = r > hi
        low = r < lo
    info = {"argmax": r.argmax(axis=1), "argmin": r.argmin(axis=1), "high": high, "low": low,
            "clip": float(c32)}
    return rt, info


def quantise_backward(g, info):
    """d loss / d r from d loss / d r_tilde (straight-through)."""
    g = np.asarray(g, np.float64)
    out = np.where(info["high"] | info["low"], 0.0, g)
    c = info["clip"]
    rows = np.arange(g.shape[0])
    np.add.at(out, (rows, info["argmax"]), c * np.where(info["high"], g, 0.0).sum(axis=1))
    np.add.at(out, (rows, info["argmin"]), c * np.where(info["low"], g, 0.0).sum(axis=1))
    return out


def expm_adjoint(S, Gbar):
    """Gradient with respect to S of <Gbar, exp(S)>: the adjoint of the Frechet
    derivative of exp at S applied to Gbar, which is L_exp(S^T, Gbar)."""
    return scipy.linalg.expm_frechet(S.T, Gbar, compute_expm=False)


# ---- attention pieces ------------------------------------------------------------

def causal_softmax(Q, Kt, scale):
    """p [Nq, G, T] for queries at positions T - Nq .. T - 1 over keys Kt [T, D]."""
    T = Kt.shape[0]
    Nq = Q.shape[0]
    logits = np.einsum("qgd,td->qgt", Q, Kt) * scale
    pos = T - Nq + np.arange(Nq)
    mask = np.arange(T)[None, :] > pos[:, None]                      # [Nq, T]
    logits = np.where(mask[:, None, :], -np.inf, logits)
    logits -= logits.max(axis=2, keepdims=True)
    e = np.exp(logits)
    return e / e.sum(axis=2, keepdims=True)


def post_wo(D_att, W):
    """Per-query post-W_O vectors: e_q = sum_h D_att[q, h] W[h]^T  ([Nq, Dm])."""
    return np.einsum("qhd,hmd->qm", D_att, W)


# ---- the two objectives with their gradients --------------------------------------

def key_loss(A, R0, K, V, Q, W, mu, clip, lam=1.0, scale=None, mode="int2"):
    """L_K and dL_K/dA for one KV head (values unquantised)."""
    K, V, Q, W = (np.asarray(x, np.float64) for x in (K, V, Q, W))
    D = K.shape[1]
    Nq = Q.shape[0]
    scale = 1.0 / np.sqrt(D) if scale is None else scale
    S = skew(A)
    E = scipy.linalg.expm(S)
    R = R0 @ E
    kc = K - mu[None, :]
    r = kc @ R
    rt, info = quantise(r, clip, mode)
    kt = rt @ R.T + mu[None, :]
    p = causal_softmax(Q, K, scale)
    pt = causal_softmax(Q, kt, scale)
    with np.errstate(divide="ignore", invalid="ignore"):
        kl_terms = np.where(p > 0, p * (np.log(p) - np.log(pt)), 0.0)
    kl = kl_terms.sum() / Nq
    dA_att = np.einsum("qht,td->qhd", pt - p, V)                     # sum_s dp_s v_s
    e = post_wo(dA_att, W)
    err = (e * e).sum() / Nq
    L = kl + lam * err
    # backward
    g_e = 2.0 * lam * e / Nq                                         # [Nq, Dm]
    g_att = np.einsum("qm,hmd->qhd", g_e, W)                         # dL/d(dA_att)
    g_pt = np.einsum("qhd,td->qht", g_att, V)                        # from the error term
    g_logit = pt * (g_pt - (pt * g_pt).sum(axis=2, keepdims=True))
    g_logit += (pt - p) / Nq                                         # from the KL term
    g_kt = np.einsum("qht,qhd->td", g_logit, Q) * scale              # dL/d k~
    g_rt = g_kt @ R
    g_R = g_kt.T @ rt
    g_r = quantise_backward(g_rt, info)
    g_R += kc.T @ g_r
    g_S = expm_adjoint(S, R0.T @ g_R)
    return L, g_S - g_S.T, {"kl": kl, "err": err, "pt": pt, "R": R, "e": e}


def value_loss(A, R0, V, pt, W, clip, mode="int2"):
    """L_V and dL_V/dA for one KV head, the attention pt [Nq, G, T] fixed."""
    V, pt, W = (np.asarray(x, np.float64) for x in (V, pt, W))
    Nq = pt.shape[0]
    S = skew(A)
    E = scipy.linalg.expm(S)
    R = R0 @ E
    r = V @ R
    rt, info = quantise(r, clip, mode)
    vt = rt @ R.T
    dB = np.einsum("qht,td->qhd", pt, vt - V)                        # sum_s p~_s dv_s
    e = post_wo(dB, W)
    L = (e * e).sum() / Nq
    g_B = np.einsum("qm,hmd->qhd", 2.0 * e / Nq, W)
    g_vt = np.einsum("qht,qhd->td", pt, g_B)
    g_rt = g_vt @ R
    g_R = g_vt.T @ rt
    g_r = quantise_backward(g_rt, info)
    g_R += V.T @ g_r
    g_S = expm_adjoint(S, R0.T @ g_R)
    return L, g_S - g_S.T, {"R": R, "e": e}


# ---- Adam and the calibration loop ----------------------------------------------

def adam_step(A, g, m, v, t, lr, b1=0.9, b2=0.999, eps=1e-8):
    """One Adam update (t counts from 1); returns (A, m, v)."""
    m = b1 * m + (1.0 - b1) * g
    v = b2 * v + (1.0 - b2) * g * g
    mh = m / (1.0 - b1 ** t)
    vh = v / (1.0 - b2 ** t)
    return A - lr * mh / (np.sqrt(vh) + eps), m, v


def calibrate(R0K, R0V, K, V, Q, W, mu, clip_k, clip_v, lam=1.0, lr=1e-3, steps=80):
    """Keys, then values, for one KV head.  Returns (R_K, R_V, history) where
    history holds the losses before each step and after the last one."""
    D = K.shape[1]
    A = np.zeros((D, D))
    m = np.zeros_like(A)
    v = np.zeros_like(A)
    hist_k, hist_v = [], []
    for t in range(1, steps + 1):
        L, g, _ = key_loss(A, R0K, K, V, Q, W, mu, clip_k, lam)
        hist_k.append(L)
        A, m, v = adam_step(A, g, m, v, t, lr)
    L, _, aux = key_loss(A, R0K, K, V, Q, W, mu, clip_k, lam)
    hist_k.append(L)
    RK, pt = aux["R"], aux["pt"]
    B = np.zeros((D, D))
    m = np.zeros_like(B)
    v = np.zeros_like(B)
    for t in range(1, steps + 1):
        L, g, _ = value_loss(B, R0V, V, pt, W, clip_v)
        hist_v.append(L)
        B, m, v = adam_step(B, g, m, v, t, lr)
    L, _, aux = value_loss(B, R0V, V, pt, W, clip_v)
    hist_v.append(L)
    return RK, aux["R"], {"key": np.array(hist_k), "value": np.array(hist_v), "A_K": A, "A_V": B}

"""GPU parity of OptR rotation calibration (kvq_optr_loss_grad, kvq_optr_calibrate)
against the float64 oracle (oracle/optr.py) on synthetic calibration traces.

* the key and value objectives and their straight-through gradients at A = 0
  and at random generators (small ones, and one large enough for the matrix
  exponentials to need squarings), also at sizes off the GEMM tiles: losses
  within 1e-3 and gradients within 2e-3 relative (L2) of the oracle;
* a short calibration: the loss history within 1e-2 of the oracle's (Adam's
  first steps follow the gradient's signs, so entries whose gradient is near
  zero may step differently), the calibrated rotations orthogonal to 1e-5;
* a longer calibration lowers both objectives of every head.
"""
import numpy as np
import pytest
import torch

from oracle import optr
from rotated_int2_kv_kvq_gb300 import kvq as K
from rotated_int2_kv_kvq_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _setup(heads=(0, 1), T=256, Nq=32, Dm=256, layer=0):
    wl = W.WORKLOADS["qwen3_8b_32k"]
    Kb, Vb, Qb, Wo = W.calibration_traces(wl, layer, T, Nq, Dm, heads)
    R0 = W.rotations(wl, layer)[:, list(heads)].copy()
    mu = W.key_mean(wl, layer)[list(heads)].copy()
    dev16 = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()
    gpu = dict(K=dev16(Kb), V=dev16(Vb), Q=dev16(Qb), W_O=torch.from_numpy(Wo).cuda(),
               R0=torch.from_numpy(R0).cuda(), mu=torch.from_numpy(mu).cuda())
    f = lambda b: W.bf16_bits_to_float(b).astype(np.float64)
    Hs, G = Qb.shape[0], Qb.shape[2]
    # the ABI's W_O [Hs, Dm, G*D] as the oracle's per-head slices [Hs, G, Dm, D]
    Wh = Wo.reshape(Hs, Dm, G, 128).transpose(0, 2, 1, 3).astype(np.float64)
    host = dict(K=f(Kb), V=f(Vb), Q=f(Qb), W=Wh, R0=R0.astype(np.float64),
                mu=mu.astype(np.float64))
    return wl, gpu, host


def _rel(a, b):
    return float(np.linalg.norm(np.asarray(a) - np.asarray(b)) / max(np.linalg.norm(b), 1e-30))


@pytest.mark.parametrize("scale,shape", [(0.0, (256, 32, 256)), (0.02, (256, 32, 256)),
                                         (0.02, (200, 20, 200)), (0.3, (256, 32, 256))])
def test_objectives_and_gradients_match_the_oracle(scale, shape):
    """(200, 20, 200): T, Nq * G and d_model off every GEMM tile (the guarded
    GEMM); scale 0.3: a generator large enough that the exponentials need
    squarings."""
    T, Nq, Dm = shape
    wl, gpu, host = _setup(T=T, Nq=Nq, Dm=Dm)
    H = host["K"].shape[0]
    rng = np.random.default_rng(17)
    A_k = (rng.standard_normal((H, 128, 128)) * scale).astype(np.float32)
    A_v = (rng.standard_normal((H, 128, 128)) * scale).astype(np.float32)
    lk, gk = K.kvq_optr_loss_grad(gpu["K"], gpu["V"], gpu["Q"], gpu["W_O"], gpu["R0"], gpu["mu"],
                                  wl.clip_k, wl.clip_v, torch.from_numpy(A_k).cuda(), which=0)
    lv, gv = K.kvq_optr_loss_grad(gpu["K"], gpu["V"], gpu["Q"], gpu["W_O"], gpu["R0"], gpu["mu"],
                                  wl.clip_k, wl.clip_v, torch.from_numpy(A_k).cuda(),
                                  torch.from_numpy(A_v).cuda(), which=1)
    lk, gk, lv, gv = (x.cpu().numpy() for x in (lk, gk, lv, gv))
    for h in range(H):
        Lk, Gk, aux = optr.key_loss(A_k[h].astype(np.float64), host["R0"][0, h], host["K"][h],
                                    host["V"][h], host["Q"][h], host["W"][h], host["mu"][h],
                                    wl.clip_k)
        Lv, Gv, _ = optr.value_loss(A_v[h].astype(np.float64), host["R0"][1, h], host["V"][h],
                                    aux["pt"], host["W"][h], wl.clip_v)
        assert abs(lk[h] - Lk) <= 1e-3 * abs(Lk), (h, lk[h], Lk)
        assert abs(lv[h] - Lv) <= 1e-3 * abs(Lv), (h, lv[h], Lv)
        assert _rel(gk[h], Gk) <= 2e-3, (h, _rel(gk[h], Gk))
        assert _rel(gv[h], Gv) <= 2e-3, (h, _rel(gv[h], Gv))
        # the gradient is skew-symmetric (it is taken through A - A^T)
        assert np.abs(gk[h] + gk[h].T).max() <= 1e-6 * np.abs(gk[h]).max()


def test_short_calibration_matches_the_oracle():
    wl, gpu, host = _setup()
    H = host["K"].shape[0]
    steps = 5
    R, hist = K.kvq_optr_calibrate(gpu["K"], gpu["V"], gpu["Q"], gpu["W_O"], gpu["R0"], gpu["mu"],
                                   wl.clip_k, wl.clip_v, lr=1e-3, steps=steps)
    R, hist = R.cpu().numpy().astype(np.float64), hist.cpu().numpy()
    for h in range(H):
        RK, RV, oh = optr.calibrate(host["R0"][0, h], host["R0"][1, h], host["K"][h], host["V"][h],
                                    host["Q"][h], host["W"][h], host["mu"][h], wl.clip_k,
                                    wl.clip_v, lr=1e-3, steps=steps)
        assert _rel(hist[0, :, h], oh["key"]) <= 1e-2, (hist[0, :, h], oh["key"])
        assert _rel(hist[1, :, h], oh["value"]) <= 1e-2, (hist[1, :, h], oh["value"])
        assert abs(hist[0, 0, h] - oh["key"][0]) <= 1e-3 * oh["key"][0]
        for which, Ro in ((0, RK), (1, RV)):
            Rg = R[which, h]
            assert np.abs(Rg.T @ Rg - np.eye(128)).max() <= 1e-5
            assert np.abs(Rg - Ro).max() <= 2e-2


def test_calibration_lowers_both_objectives():
    wl, gpu, host = _setup(heads=(0, 1, 2, 3), T=1024, Nq=64, Dm=512)
    R, hist = K.kvq_optr_calibrate(gpu["K"], gpu["V"], gpu["Q"], gpu["W_O"], gpu["R0"], gpu["mu"],
                                   wl.clip_k, wl.clip_v, lr=1e-3, steps=40)
    hist = hist.cpu().numpy()
    assert np.all(hist[0, -1] < 0.8 * hist[0, 0]), hist[0]
    # every head ends below its start (the float64 oracle on these traces ends
    # at 0.53-0.78 of the start: no head is near the bound)
    assert np.all(hist[1, -1] < hist[1, 0]), hist[1]
    Rn = R.cpu().numpy().astype(np.float64)
    for which in range(2):
        for h in range(4):
            assert np.abs(Rn[which, h].T @ Rn[which, h] - np.eye(128)).max() <= 1e-5

"""Pins of the CPU oracle against what the method's description and plain
mathematics fix — not against the oracle itself.

Each test names the property it checks and where that property comes from.
Sources: "Output-Aware Rotation for INT2 KV-Cache Quantization" (pith.science
review of arXiv 2608.02691), cited by section; IEEE 754 for number formats;
library routines (numpy float16 casts, torch bfloat16 casts, scipy softmax) as
independent references.
"""
import math

import numpy as np
import pytest

from conftest import read_golden
from rotated_int2_kv_kvq_gb300 import workloads as W

D = 128


def _bf16(x):
    return W.to_bf16_bits(np.asarray(x, np.float32))


def _f16(h):
    return float(np.array([h], np.uint16).view(np.float16)[0])


# ---------------------------------------------------------------------------
# Number formats: the oracle's binary16 rounding against numpy's cast.
# ---------------------------------------------------------------------------

def test_f32_to_f16_matches_numpy_cast(orc):
    g = np.random.default_rng(0)
    xs = np.concatenate([
        g.standard_normal(20000).astype(np.float32) * np.float32(10.0) ** g.integers(-9, 6, 20000),
        np.array([0.0, -0.0, 1.0, 65504.0, 65519.99, 65520.0, 70000.0, -1e9, 2.0 ** -24,
                  2.0 ** -25, 1.5 * 2.0 ** -24, 2.0 ** -14, 2.0 ** -14 - 2.0 ** -25,
                  np.inf, -np.inf], np.float32),
    ]).astype(np.float32)
    # ties: midpoints between consecutive fp16 values, exactly representable in fp32
    h = np.arange(0, 0x7bff, 37, dtype=np.uint16)
    a = h.view(np.float16).astype(np.float32)
    b = (h + 1).view(np.float16).astype(np.float32)
    xs = np.concatenate([xs, (a + b) / np.float32(2), -(a + b) / np.float32(2)]).astype(np.float32)
    want = xs.astype(np.float16).view(np.uint16)
    got = np.array([orc.f32_to_f16_bits(x) for x in xs], np.uint16)
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(float(xs[i]), hex(got[i]), hex(want[i])) for i in bad[:5]]


def test_f16_to_f32_exact(orc):
    for h in list(range(0, 0x7c00, 13)) + [0x7c00, 0x8001, 0xfbff, 0x0001, 0x03ff, 0x0400]:
        assert orc.f16_bits_to_f32(h) == float(np.array([h], np.uint16).view(np.float16)[0])


def test_bf16_generator_matches_torch_cast(orc):
    torch = pytest.importorskip("torch")
    g = np.random.default_rng(1)
    x = (g.standard_normal(50000) * 10.0 ** g.integers(-6, 6, 50000)).astype(np.float32)
    ours = W.to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    # and the oracle's bf16 -> f32 is the top-half reinterpretation
    for b in ours[:200]:
        assert orc.bf16_bits_to_f32(b) == float(W.bf16_bits_to_float(np.array([b]))[0])


# ---------------------------------------------------------------------------
# Quantiser: worked examples derived by hand (tests/golden) and closed forms.
# ---------------------------------------------------------------------------

def _golden_quant(name):
    rows = {r[0]: r[1:] for r in read_golden(name)}
    pattern = [float(v) for v in rows["pattern"]]
    x = np.array(pattern * (D // len(pattern)), np.float32)
    return (float(rows["clip"][0]), x, int(rows["s16"][0], 16), int(rows["z16"][0], 16),
            [int(c) for c in rows["codes"]] * (D // len(pattern)),
            float(rows["key_offset"][0]) if "key_offset" in rows else None)


@pytest.mark.parametrize("name", ["quant_grid.txt", "quant_clip.txt"])
def test_quantiser_worked_examples(orc, name):
    clip, x, s16, z16, codes, key_offset = _golden_quant(name)
    eye = np.eye(D, dtype=np.float32)
    c, s, z, r, t = orc.quantize(_bf16(x), eye, clip)
    assert (s, z) == (s16, z16)
    assert c.tolist() == codes
    if key_offset is not None:
        mu = np.full(D, key_offset, np.float32)
        c2, s2, z2, _, _ = orc.quantize(_bf16(x + key_offset), eye, clip, mu=mu)
        assert (s2, z2) == (s16, z16) and c2.tolist() == codes
        # centring with the wrong sign would not reproduce the example
        c3, s3, z3, _, _ = orc.quantize(_bf16(x + key_offset), eye, clip, mu=-mu)
        assert (s3, z3) != (s16, z16)


def test_quantiser_grid_roundtrip_exact(orc):
    """Values already on a grid z + k*s with fp16-exact s, z and clip = 1 come
    back exactly (the quantise/dequantise pair is the identity on its grid)."""
    g = np.random.default_rng(2)
    for trial in range(50):
        s = float(np.float16(2.0 ** g.integers(-6, 4)))
        z = float(np.float16(g.integers(-40, 40) * s / 4))
        k = g.integers(0, 4, D)
        k[:2] = [0, 3]                      # make min and max attained
        x = np.float32(z) + k.astype(np.float32) * np.float32(s)
        xb = _bf16(x)
        assert np.array_equal(W.bf16_bits_to_float(xb), x), "set-up must be bf16-exact"
        c, s16, z16, r, t = orc.quantize(xb, np.eye(D, dtype=np.float32), 1.0)
        assert np.array_equal(c, k)
        assert _f16(s16) == s and _f16(z16) == z


def test_quantiser_degenerate_group(orc):
    """All elements equal: max == min, the scale is 0, every code is 0 and the
    group dequantises to z = fp16(clip * x)."""
    for v in [0.0, 1.0, -3.5, 1000.0]:
        x = _bf16(np.full(D, v, np.float32))
        c, s16, z16, r, t = orc.quantize(x, np.eye(D, dtype=np.float32), 0.96)
        assert s16 in (0x0000, 0x8000) and not c.any()
        assert z16 == int(np.float16(np.float32(0.96) * np.float32(v)).view(np.uint16))


def test_quantiser_brute_force_and_error_bound(orc):
    """Against brute force: each code is the grid level nearest to the rotated
    value (argmin over 4 levels, ties to even), inside the clip range the
    round-trip error is at most s/2, and outside it the code is the end level."""
    g = np.random.default_rng(3)
    Rs = W.rotations(W.WORKLOADS["qwen3_8b_32k"])[:, :2]
    near_tie = 0
    for trial in range(300):
        R = Rs[trial % 2, (trial // 2) % 2]
        x = _bf16(g.standard_normal(D) * g.uniform(0.1, 30))
        clip = [1.0, 0.96, 0.92, 0.5][trial % 4]
        c, s16, z16, r, t = orc.quantize(x, R, clip)
        s, z = _f16(s16), _f16(z16)
        assert s > 0
        lv = z + np.arange(4)[None, :] * s                      # float64 grid levels
        dist = np.abs(r.astype(np.float64)[:, None] - lv)
        best = dist.argmin(axis=1)
        # ties (equal distance to two levels) resolve to the even level
        second = np.sort(dist, axis=1)[:, 1]
        tie = np.isclose(dist.min(axis=1), second, rtol=0, atol=1e-12 * s)
        best[tie] = np.where(best[tie] % 2 == 0, best[tie], best[tie] + 1)
        mism = np.nonzero(best != c)[0]
        for i in mism:
            # allowed only where fp32 (r - z)/s sits within 2 ulp of a half-integer
            frac = abs(float(t[i]) - math.floor(float(t[i])) - 0.5)
            assert frac <= 2 * np.spacing(np.float32(t[i])), (i, t[i], best[i], c[i])
            near_tie += 1
        inside = (r >= z) & (r <= z + 3 * s)
        deq = z + c.astype(np.float64) * s
        assert np.all(np.abs(deq - r)[inside] <= s / 2 * (1 + 2.0 ** -20))
        assert np.all(c[r < z - s / 2] == 0) and np.all(c[r > z + 3 * s + s / 2] == 3)
    assert near_tie <= 3


def test_clip_shrinks_range(orc):
    """A smaller clip ratio gives a smaller scale (clipping narrows the grid)."""
    g = np.random.default_rng(4)
    x = _bf16(g.standard_normal(D) * 3)
    eye = np.eye(D, dtype=np.float32)
    s = [_f16(orc.quantize(x, eye, cl)[1]) for cl in (1.0, 0.96, 0.92, 0.8)]
    assert s[0] > s[1] > s[2] > s[3]


# ---------------------------------------------------------------------------
# Rotation: orthogonality and the row-vector convention.
# ---------------------------------------------------------------------------

def test_generated_rotations_are_orthogonal():
    R = W.rotations(W.WORKLOADS["qwen3_8b_32k"]).astype(np.float64)
    for m in R.reshape(-1, D, D):
        assert np.abs(m.T @ m - np.eye(D)).max() <= 1e-6


def test_rotation_index_convention(orc):
    """r_i = sum_j c_j R[j][i]: with a permutation matrix P[j][perm[j]] = 1 the
    rotated vector is r[perm[j]] = c[j] (a transposed R would give the inverse
    permutation); with a diagonal +-1 matrix r is a sign flip, exactly."""
    g = np.random.default_rng(5)
    perm = g.permutation(D)
    P = np.zeros((D, D), np.float32)
    P[np.arange(D), perm] = 1.0
    x = _bf16(g.standard_normal(D))
    xf = W.bf16_bits_to_float(x)
    _, _, _, r, _ = orc.quantize(x, P, 1.0)
    want = np.empty(D, np.float32)
    want[perm] = xf
    assert np.array_equal(r, want)
    S = np.diag(np.where(g.random(D) < 0.5, -1.0, 1.0)).astype(np.float32)
    _, _, _, r2, _ = orc.quantize(x, S, 1.0)
    assert np.array_equal(r2, xf * np.diag(S))
    # float64 rotation routines: same convention, and transpose-rotation inverts
    y = orc.rotate_f64(xf, P)
    assert np.array_equal(y, want.astype(np.float64))
    assert np.array_equal(orc.rotate_t_f64(y, P), xf.astype(np.float64))


def test_fma_chain_within_dot_product_bound(orc):
    """The fp32 chain differs from the exact (float64) product by at most the
    classical bound gamma_D * sum |c_j R_ji| for a length-D dot product."""
    wl = W.WORKLOADS["qwen3_8b_32k"]
    R = W.rotations(wl)[0, 0]
    mu = W.key_mean(wl)[0]
    g = np.random.default_rng(6)
    gamma = D * 2.0 ** -24 / (1 - D * 2.0 ** -24)
    for _ in range(20):
        x = W.token_at(wl, 0, int(g.integers(0, 16)), 0, int(g.integers(0, 32768)))[0]
        _, _, _, r, _ = orc.quantize(x, R, 0.96, mu=mu)
        c = (W.bf16_bits_to_float(x) - mu).astype(np.float32).astype(np.float64)
        exact = c @ R.astype(np.float64)
        bound = gamma * (np.abs(c)[:, None] * np.abs(R.astype(np.float64))).sum(axis=0)
        assert np.all(np.abs(r - exact) <= bound)


def test_orthogonal_invariance_of_logits(orc):
    """An orthogonal R applied to q and k leaves q.k unchanged ("What carries the
    argument": R stays in O(d)), checked in float64 to 1e-10 relative."""
    R = W.rotations(W.WORKLOADS["qwen3_8b_32k"])[0, 3]
    g = np.random.default_rng(7)
    # orthogonalise the fp32 matrix in float64 so the identity is exact up to rounding
    Rq = np.linalg.qr(R.astype(np.float64))[0]
    Rq = Rq * np.sign(np.diag(np.linalg.qr(R.astype(np.float64))[1]))[None, :]
    for _ in range(20):
        q, k = g.standard_normal(D), g.standard_normal(D) * 5
        lhs = float(q @ k)
        rhs = float((q @ Rq) @ (k @ Rq))
        assert abs(lhs - rhs) <= 1e-10 * np.linalg.norm(q) * np.linalg.norm(k)
    # with the stored fp32 R the identity holds to its orthogonality error
    q, k = g.standard_normal(D), g.standard_normal(D)
    qr_, kr_ = orc.rotate_f64(q, R), orc.rotate_f64(k, R)
    assert abs(q @ k - qr_ @ kr_) <= 1e-5 * np.linalg.norm(q) * np.linalg.norm(k)


# ---------------------------------------------------------------------------
# Page layout: hand-derived positions and bijectivity.
# ---------------------------------------------------------------------------

def test_layout_hand_derived_positions(orc):
    for row in read_golden("layout_int2.txt"):
        kind = row[0]
        vals = [int(v) for v in row[1:]]
        if kind == "code":
            which, tau, d, byte, shift = vals
            assert orc.int2_locate(which, tau, d) == (byte, shift), row
        elif kind == "meta":
            which, tau, off = vals
            assert orc.int2_meta_offset(which, tau) == off, row
        elif kind == "bf16":
            which, tau, d, off = vals
            assert orc.bf16_locate(which, tau, d) == off, row


def test_int2_layout_is_a_bijection(orc):
    seen = np.zeros(1024 * 4, np.int32)            # one slot per 2-bit field
    for which in range(2):
        for tau in range(16):
            for d in range(D):
                b, s = orc.int2_locate(which, tau, d)
                assert 0 <= b < 1024 and s % 2 == 0
                assert (b < 512) == (which == 0)
                seen[b * 4 + s // 2] += 1
    assert np.all(seen == 1)
    meta = set()
    for which in range(2):
        for tau in range(16):
            o = orc.int2_meta_offset(which, tau)
            assert 1024 <= o and o + 4 <= 1152
            meta.update(range(o, o + 4))
    assert meta == set(range(1024, 1152))


def test_bf16_layout_is_a_bijection(orc):
    seen = np.zeros(4096, np.int32)
    for which in range(2):
        for tau in range(16):
            for d in range(D):
                o = orc.bf16_locate(which, tau, d)
                assert o % 2 == 0 and (o < 4096) == (which == 0)
                seen[o // 2] += 1
    assert np.all(seen == 1)


def test_int2_store_load_and_known_bytes(orc):
    rec = np.zeros(1152, np.uint8)
    ones = np.ones(D, np.uint8)
    orc.int2_store(rec, 0, 0, ones, 0x1234, 0xabcd)
    # token 0, keys: lanes 0..3, words 0 and 1 -> bytes 16t..16t+7, every field = 01
    want = np.zeros(1152, np.uint8)
    for t in range(4):
        want[16 * t:16 * t + 8] = 0x55
    want[1024:1028] = [0x34, 0x12, 0xcd, 0xab]
    assert np.array_equal(rec, want)
    orc.int2_store(rec, 1, 1, ones * 3, 0, 0)
    # token 1, values: t=0, e=1 (high halves), lanes 4g, words 0 and 1
    for g_ in range(8):
        for dh in range(2):
            o = 512 + 64 * g_ + 4 * dh + 2
            want[o:o + 2] = 0xff
    assert np.array_equal(rec, want)
    g = np.random.default_rng(8)
    codes = g.integers(0, 4, (2, 16, D)).astype(np.uint8)
    sz = g.integers(0, 65536, (2, 16, 2))
    rec = np.full(1152, 0xa5, np.uint8)
    for which in range(2):
        for tau in range(16):
            orc.int2_store(rec, which, tau, codes[which, tau], *sz[which, tau])
    for which in range(2):
        for tau in range(16):
            c, s, z = orc.int2_load(rec, which, tau)
            assert np.array_equal(c, codes[which, tau]) and (s, z) == tuple(sz[which, tau])


# ---------------------------------------------------------------------------
# Attention
# ---------------------------------------------------------------------------

def _naive_attention(q, keys, values, scale):
    """Pure-Python float64 softmax attention, written independently."""
    logits = [scale * sum(qi * ki for qi, ki in zip(q, k)) for k in keys]
    m = max(logits)
    w = [math.exp(l - m) for l in logits]
    tot = sum(w)
    return [sum(w[t] * values[t][d] for t in range(len(keys))) / tot for d in range(len(q))]


def test_attention_brute_force_tiny(orc):
    scipy_special = pytest.importorskip("scipy.special")
    g = np.random.default_rng(9)
    for T, Dt in [(1, 8), (3, 8), (17, 8), (40, 128)]:
        q, k, v = g.standard_normal(Dt), g.standard_normal((T, Dt)) * 3, g.standard_normal((T, Dt))
        out = orc.attend_f64(q, k, v, 0.37)
        ref = _naive_attention(q.tolist(), k.tolist(), v.tolist(), 0.37)
        assert np.allclose(out, ref, rtol=1e-12, atol=1e-12)
        p = scipy_special.softmax(0.37 * (k @ q))
        assert np.allclose(out, p @ v, rtol=1e-12, atol=1e-12)
    assert np.array_equal(orc.attend_f64(np.ones(8), np.zeros((0, 8)), np.zeros((0, 8)), 1.0),
                          np.zeros(8))


def test_key_centring_leaves_softmax_unchanged(orc):
    """"What carries the argument", mechanism (2): subtracting one mean from
    every key adds a per-query constant to the logits; in full precision the
    attention output is unchanged."""
    wl = W.WORKLOADS["qwen3_8b_32k"]
    mu = W.key_mean(wl)[2].astype(np.float64)
    k = W.bf16_bits_to_float(W.tokens(wl, 0, 1, 0, 100, 300)[:, 2]).astype(np.float64)
    v = W.bf16_bits_to_float(W.tokens(wl, 0, 1, 1, 100, 300)[:, 2]).astype(np.float64)
    g = np.random.default_rng(10)
    for _ in range(5):
        q = g.standard_normal(D)
        a = orc.attend_f64(q, k, v, 1 / math.sqrt(D))
        b = orc.attend_f64(q, k - mu, v, 1 / math.sqrt(D))
        assert np.abs(a - b).max() <= 1e-12 * max(1.0, np.abs(a).max())


def test_error_decomposition_identity(orc):
    """Eq. 8 of the paper ("What carries the argument"): with W_O = I,
    y~ - y = sum_s (p~_s - p_s) v_s + sum_s p~_s (v~_s - v_s), in float64."""
    g = np.random.default_rng(11)
    T = 50
    q = g.standard_normal(D)
    k, v = g.standard_normal((T, D)), g.standard_normal((T, D))
    kq, vq = k + 0.1 * g.standard_normal((T, D)), v + 0.1 * g.standard_normal((T, D))
    sc = 1 / math.sqrt(D)
    y, yq = orc.attend_f64(q, k, v, sc), orc.attend_f64(q, kq, vq, sc)
    p = np.exp(sc * k @ q - (sc * k @ q).max()); p /= p.sum()
    pq = np.exp(sc * kq @ q - (sc * kq @ q).max()); pq /= pq.sum()
    assert np.allclose(yq - y, (pq - p) @ v + pq @ (vq - v), rtol=0, atol=1e-12)


def _small_int2_cache(orc, wl, ctx, seed=12):
    """Append ctx tokens of sequence 0 into a shuffled pool with the oracle."""
    pt, npool = W.page_table(wl)
    pt = pt[:1, :(ctx + 15) // 16]
    pool = np.zeros(npool * wl.num_kv_heads * 1152, np.uint8)
    K = W.tokens(wl, 0, 0, 0, 0, ctx)
    V = W.tokens(wl, 0, 0, 1, 0, ctx)
    R = W.rotations(wl)
    mu = W.key_mean(wl)
    sk = orc.append_int2(pool, npool, wl.num_kv_heads, K, V, np.zeros(ctx, np.int32),
                         np.arange(ctx, dtype=np.int32), pt, R, mu, wl.clip_k, wl.clip_v)
    assert sk == 0
    return pool, npool, pt, K, V, R, mu


def test_append_places_quantised_tokens(orc):
    """Each appended token's codes and s/z sit in the record of
    page_table[position // 16], slot position % 16, and equal the quantiser's."""
    wl = W.WORKLOADS["tiny_1k"]
    pool, npool, pt, K, V, R, mu = _small_int2_cache(orc, wl, 70)
    recs = pool.reshape(npool, 1, 1152)
    for p in [0, 1, 15, 16, 31, 47, 69]:
        rec = recs[pt[0, p // 16], 0]
        for which, X, Rm, m, cl in [(0, K, R[0, 0], mu[0], wl.clip_k), (1, V, R[1, 0], None, wl.clip_v)]:
            c, s, z, _, _ = orc.quantize(X[p, 0], Rm, cl, mu=m)
            c2, s2, z2 = orc.int2_load(rec, which, p % 16)
            assert np.array_equal(c, c2) and (s, z) == (s2, z2)
    # a bad page id is skipped, not written
    bad = pt.copy()
    bad[0, 0] = npool + 5
    pool2 = np.zeros_like(pool)
    sk = orc.append_int2(pool2, npool, 1, K[:3], V[:3], np.zeros(3, np.int32),
                         np.arange(3, dtype=np.int32), bad, R, mu, wl.clip_k, wl.clip_v)
    assert sk == 3 and not pool2.any()


def test_decode_matches_dequantised_attention(orc):
    """The oracle's paged decode equals softmax attention computed here in numpy
    from the oracle's dequantised cache (q rotated by R_K, output rotated back
    by R_V^T), and the rotated-output flag skips only the last rotation."""
    wl = W.WORKLOADS["tiny_1k"]
    ctx = 83
    pool, npool, pt, K, V, R, mu = _small_int2_cache(orc, wl, ctx)
    q = W.queries(wl)
    Kd, Vd = orc.dequant_int2(pool, npool, 1, pt, 0, 0, ctx)
    pairs = np.array([[0, h] for h in range(4)])
    out = orc.decode_pairs("int2", pool, npool, 4, 1, q, pt, np.array([ctx]), pairs, R=R)
    outr = orc.decode_pairs("int2", pool, npool, 4, 1, q, pt, np.array([ctx]), pairs, R=R,
                            out_rotated=True)
    for h in range(4):
        qf = W.bf16_bits_to_float(q[0, h]).astype(np.float64)
        qrot = qf @ R[0, 0].astype(np.float64)
        lg = (Kd[:, 0].astype(np.float64) @ qrot) / math.sqrt(D)
        p = np.exp(lg - lg.max()); p /= p.sum()
        orot = p @ Vd[:, 0].astype(np.float64)
        assert np.allclose(outr[h], orot, rtol=1e-9, atol=1e-9)
        assert np.allclose(out[h], orot @ R[1, 0].astype(np.float64).T, rtol=1e-9, atol=1e-9)


def test_decode_special_cases(orc):
    """One token: the output is that token's dequantised value rotated back.
    Empty context: zero."""
    wl = W.WORKLOADS["tiny_1k"]
    pool, npool, pt, K, V, R, mu = _small_int2_cache(orc, wl, 1)
    q = W.queries(wl)
    out = orc.decode_pairs("int2", pool, npool, 4, 1, q, pt, np.array([1]), [[0, 2]], R=R)
    _, Vd = orc.dequant_int2(pool, npool, 1, pt, 0, 0, 1)
    assert np.allclose(out[0], Vd[0, 0].astype(np.float64) @ R[1, 0].astype(np.float64).T,
                       rtol=1e-12, atol=1e-12)
    z = orc.decode_pairs("int2", pool, npool, 4, 1, q, pt, np.array([0]), [[0, 1]], R=R)
    assert not z.any()


def test_identical_keys_give_mean_of_values(orc):
    g = np.random.default_rng(13)
    k = np.tile(g.standard_normal(D), (9, 1))
    v = g.standard_normal((9, D))
    assert np.allclose(orc.attend_f64(g.standard_normal(D), k, v, 0.5), v.mean(axis=0),
                       rtol=1e-12, atol=1e-12)


def test_bf16_append_and_decode(orc):
    wl = W.WORKLOADS["tiny_1k"]
    ctx = 40
    pt, npool = W.page_table(wl)
    pool = np.zeros(npool * 8192, np.uint8)
    K, V = W.tokens(wl, 0, 0, 0, 0, ctx), W.tokens(wl, 0, 0, 1, 0, ctx)
    assert orc.append_bf16(pool, npool, 1, K, V, np.zeros(ctx, np.int32),
                           np.arange(ctx, dtype=np.int32), pt) == 0
    q = W.queries(wl)
    out = orc.decode_pairs("bf16", pool, npool, 4, 1, q, pt, np.array([ctx]), [[0, 3]])
    ref = _naive_attention(W.bf16_bits_to_float(q[0, 3]).astype(np.float64).tolist(),
                           W.bf16_bits_to_float(K[:, 0]).astype(np.float64).tolist(),
                           W.bf16_bits_to_float(V[:, 0]).astype(np.float64).tolist(),
                           1 / math.sqrt(D))
    assert np.allclose(out[0], ref, rtol=1e-11, atol=1e-11)


# ---------------------------------------------------------------------------
# BF16 sink + recent window ("Assumptions & free parameters": 64 sink and 256
# recent tokens kept in BF16).
# ---------------------------------------------------------------------------

def _window_fixture(orc, ctx=150):
    wl = W.WORKLOADS["tiny_1k"]
    pool, npool, pt, K, V, R, mu = _small_int2_cache(orc, wl, ctx)
    bpool = np.zeros(npool * 8192, np.uint8)
    assert orc.append_bf16(bpool, npool, 1, K, V, np.zeros(ctx), np.arange(ctx), pt) == 0
    return wl, pool, npool, pt, bpool, K, V, R, mu


def test_window_reduces_to_the_plain_paths(orc):
    wl, pool, npool, pt, bpool, K, V, R, mu = _window_fixture(orc)
    q = W.queries(wl, 0, 3)
    pairs = [[0, h] for h in range(4)]
    for L in (1, 37, 150):
        # empty window: the INT2 path (the added q.mu is one constant per query)
        w0 = orc.decode_window_pairs(pool, npool, bpool, npool, pt, 4, 1, q, pt, [L], pairs, 0, 0,
                                     R, mu)
        i2 = orc.decode_pairs("int2", pool, npool, 4, 1, q, pt, [L], pairs, R=R)
        assert np.allclose(w0, i2, rtol=0, atol=1e-12 * max(1.0, np.abs(i2).max()))
        # window covering the whole context: plain BF16 attention
        wa = orc.decode_window_pairs(pool, npool, bpool, npool, pt, 4, 1, q, pt, [L], pairs, 64,
                                     256, R, mu)
        bf = orc.decode_pairs("bf16", bpool, npool, 4, 1, q, pt, [L], pairs)
        assert np.allclose(wa, bf, rtol=0, atol=1e-12 * max(1.0, np.abs(bf).max()))


def test_window_mixed_context_matches_direct_formula(orc):
    wl, pool, npool, pt, bpool, K, V, R, mu = _window_fixture(orc)
    q = W.queries(wl, 0, 4)
    L, sink, recent = 150, 16, 40
    Kd, Vd = orc.dequant_int2(pool, npool, 1, pt, 0, 0, L)
    RK, RV = R[0, 0].astype(np.float64), R[1, 0].astype(np.float64)
    out = orc.decode_window_pairs(pool, npool, bpool, npool, pt, 4, 1, q, pt, [L],
                                  [[0, h] for h in range(4)], sink, recent, R, mu)
    outr = orc.decode_window_pairs(pool, npool, bpool, npool, pt, 4, 1, q, pt, [L],
                                   [[0, h] for h in range(4)], sink, recent, R, mu,
                                   out_rotated=True)
    for h in range(4):
        qf = W.bf16_bits_to_float(q[0, h]).astype(np.float64)
        lg, vals = [], []
        for p in range(L):
            if p < sink or p >= L - recent:
                lg.append(qf @ W.bf16_bits_to_float(K[p, 0]).astype(np.float64))
                vals.append(W.bf16_bits_to_float(V[p, 0]).astype(np.float64))
            else:
                lg.append((qf @ RK) @ Kd[p, 0].astype(np.float64) + qf @ mu[0].astype(np.float64))
                vals.append(Vd[p, 0].astype(np.float64) @ RV.T)
        lg = np.array(lg) / math.sqrt(D)
        w = np.exp(lg - lg.max())
        want = (w / w.sum()) @ np.array(vals)
        assert np.allclose(out[h], want, rtol=1e-6, atol=1e-6)
        assert np.allclose(outr[h], want @ RV, rtol=1e-6, atol=1e-6)

"""Pins of the oracle's dropout (inverted dropout of P with a Philox4x32-10
keep rule; the summary fuses dropout into the kernel, "Kernel Fusion", and
benchmarks with it, section 4.4).  Each pin checks the oracle against
something other than itself: published generator outputs, closed forms,
statistics of the keep rule, finite differences, and the expectation over
seeds."""
import json
import os

import numpy as np
import pytest

import oracle

HERE = os.path.dirname(os.path.abspath(__file__))


def _kat():
    with open(os.path.join(HERE, "golden", "philox4x32_10_kat.json")) as f:
        return [{k: [int(x, 16) for x in v[k]] for k in ("counter", "key", "out")}
                for v in json.load(f)["vectors"]]


def _le_bytes(words):
    return np.array([(w >> (8 * b)) & 0xFF for w in words for b in range(4)], dtype=np.uint8)


def test_philox_known_answers():
    for v in _kat():
        assert list(oracle.philox4x32_10(v["counter"], v["key"])) == v["out"]


def test_dropout_bytes_follow_the_counter_layout():
    """Element (b*H+h, i, j) draws byte j mod 16 (little-endian words) of
    Philox(counter = (j / 16, i, b*H+h, offset), key = (seed lo, seed hi)):
    every known-answer vector reappears as 16 consecutive element bytes."""
    for v in _kat():
        c, k = v["counter"], v["key"]
        seed = k[0] | (k[1] << 32)
        got = oracle.dropout_bytes(seed, c[3], c[2], c[1], 16 * c[0], 16)
        assert np.array_equal(got, _le_bytes(v["out"]))


def test_keep_rate_and_byte_uniformity():
    N = 256
    z_bytes = np.concatenate([oracle.dropout_bytes(7, 3, bh, i, 0, N)
                              for bh in range(2) for i in range(N)])
    n = z_bytes.size
    counts = np.bincount(z_bytes, minlength=256)
    chi2 = float(((counts - n / 256) ** 2 / (n / 256)).sum())
    assert chi2 < 255 + 6 * np.sqrt(2 * 255), chi2       # df = 255
    for p in (0.1, 0.5, 0.9):
        z = oracle.dropout_keep(7, 3, p, 1, 2, N)
        q = (256 - oracle.dropout_threshold(p)) / 256
        sigma = np.sqrt(q * (1 - q) / z.size)
        assert abs(z.mean() - q) < 6 * sigma, (p, z.mean(), q)


def test_threshold_rounding():
    assert oracle.dropout_threshold(0.0) == 0
    assert oracle.dropout_threshold(0.1) == 26            # 25.6 -> 26
    assert oracle.dropout_threshold(0.5) == 128
    assert oracle.dropout_threshold(220 / 256) == 220


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


@pytest.mark.parametrize("causal", [False, True])
def test_p_zero_is_the_undropped_oracle(causal):
    q, k, v, do = (_rand((2, 3, 40, 8), s) for s in range(4))
    o0, l0 = oracle.forward(q, k, v, 0.3, causal=causal)
    o1, l1 = oracle.forward(q, k, v, 0.3, causal=causal, dropout=(0.0, 123, 4))
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1)
    g0 = oracle.backward(q, k, v, do, 0.3, causal=causal)
    g1 = oracle.backward(q, k, v, do, 0.3, causal=causal, dropout=(0.0, 123, 4))
    for a, b in zip(g0, g1):
        assert np.array_equal(a, b)


def test_closed_form_two_keys():
    """One query, two keys, seed 0, offset 0, batch 0, head 0, row 0: the
    element bytes are those of the first known-answer vector, 0xd5 = 213 for
    key 0 and 0xe8 = 232 for key 1.  With t = 220 key 0 is dropped and key 1
    kept (scale 256/36); with t = 200 both are kept (scale 256/56)."""
    d = 4
    qv = np.array([0.5, -1.0, 0.25, 2.0])
    kv = np.array([[1.0, 0.0, -1.0, 0.5], [-0.5, 1.5, 0.0, 1.0]])
    vv = np.array([[1.0, 2.0, 3.0, 4.0], [-2.0, 0.5, 1.0, -1.0]])
    scale = 0.7
    s = scale * kv @ qv
    P = np.exp(s - s.max()) / np.exp(s - s.max()).sum()
    lse = s.max() + np.log(np.exp(s - s.max()).sum())
    q = qv.reshape(1, 1, 1, d)
    k = kv.reshape(1, 1, 2, d)
    v = vv.reshape(1, 1, 2, d)
    # the query row is row 0 of a 2-row problem (row 1 only pads the shape)
    q2 = np.concatenate([q, q], axis=2)
    for t, z in ((220, (0, 1)), (200, (1, 1))):
        o, l = oracle.forward(q2, k, v, scale, dropout=(t / 256, 0, 0))
        want = (256 / (256 - t)) * (z[0] * P[0] * vv[0] + z[1] * P[1] * vv[1])
        assert np.allclose(o[0, 0, 0], want, rtol=1e-13, atol=1e-13), t
        assert abs(l[0, 0, 0] - lse) < 1e-13


@pytest.mark.parametrize("causal", [False, True])
def test_finite_differences_with_dropout(causal):
    B, H, N, d = 1, 2, 12, 4
    q, k, v, do = (_rand((B, H, N, d), 10 + s) for s in range(4))
    drop = (0.3, 99, 5)
    scale = 0.6
    dq, dk, dv = oracle.backward(q, k, v, do, scale, causal=causal, dropout=drop)

    def f(q_, k_, v_):
        o, _ = oracle.forward(q_, k_, v_, scale, causal=causal, dropout=drop)
        return float((o * do).sum())

    eps = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = {"q": (xp, k, v), "k": (q, xp, v), "v": (q, k, xp)}[name]
            args_m = {"q": (xm, k, v), "k": (q, xm, v), "v": (q, k, xm)}[name]
            num[idx] = (f(*args_p) - f(*args_m)) / (2 * eps)
        assert np.abs(num - g).max() <= 1e-6 * max(1.0, np.abs(g).max()), name


def test_mean_over_seeds_is_the_undropped_output():
    """Inverted dropout is unbiased: E_z[O] = O (the 1/(1-p') scaling)."""
    q, k, v = (_rand((1, 1, 8, 4), 20 + s) for s in range(3))
    o_ref, _ = oracle.forward(q, k, v, 0.5)
    samples = np.stack([oracle.forward(q, k, v, 0.5, dropout=(0.5, s, 0))[0]
                        for s in range(600)])
    mean, sd = samples.mean(0), samples.std(0)
    assert np.all(np.abs(mean - o_ref) <= 5 * sd / np.sqrt(len(samples)) + 1e-12)
    # a missing 1/(1-p) would halve the mean
    assert np.abs(mean - o_ref).max() < 0.25 * np.abs(o_ref).max()


def test_forward_uses_the_keep_indicator():
    """Q = 0 and V = I (N = d): O_ic = z_ic / (1-p') / N, which exposes the
    keep indicator the forward applied element by element."""
    B, H, N = 2, 2, 16
    q = np.zeros((B, H, N, N))
    k = _rand((B, H, N, N), 30)
    v = np.broadcast_to(np.eye(N), (B, H, N, N)).copy()
    p = 0.25
    o, _ = oracle.forward(q, k, v, 1.0, dropout=(p, 11, 2))
    t = oracle.dropout_threshold(p)
    z = oracle.dropout_keep(11, 2, p, B, H, N)
    assert np.allclose(o, z * (256 / (256 - t)) / N, atol=1e-14)


def test_varlen_dropout_equals_equal_length_batch():
    """A packed batch of equal-length sequences draws the same keep
    indicator as the [B, H, N, d] batch (sequence b is batch b)."""
    B, H, N, d = 3, 2, 20, 4
    q, k, v, do = (_rand((B, H, N, d), 40 + s) for s in range(4))
    drop = (0.2, 5, 9)
    o, l = oracle.forward(q, k, v, 0.5, causal=True, dropout=drop)
    pk = lambda x: np.ascontiguousarray(x.transpose(1, 0, 2, 3).reshape(H, B * N, d))
    cu = np.arange(B + 1) * N
    ov, lv = oracle.forward_varlen(pk(q), pk(k), pk(v), cu, 0.5, causal=True, dropout=drop)
    assert np.allclose(ov, pk(o), atol=1e-13)
    g = oracle.backward(q, k, v, do, 0.5, causal=True, dropout=drop)
    gv = oracle.backward_varlen(pk(q), pk(k), pk(v), pk(do), cu, 0.5, causal=True, dropout=drop)
    for a, b in zip(g, gv):
        assert np.allclose(b, pk(a), atol=1e-13)

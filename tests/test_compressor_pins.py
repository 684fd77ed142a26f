"""Pins for the oracle's indexer compressor (CPU only).

[HiSA issue] = "feat(deepseek-v4): implement HiSA hierarchical sparse attention",
sections "The pooled stream and positions" and "Configuration": gated pooling of r-token
windows (the overlap variant also draws on the previous window, output width 2 D_i),
RMSNorm, and RoPE with base 160000 on the interleaved pairs of dims 64..127 at the pooled
row's position p r. Each test ties oracle.compress_rows / rope_interleaved / rms_norm to a
closed form or an invariant, not to a restatement of the same formula.
"""
import math

import numpy as np
import pytest

from oracle import hisa_oracle as O

D, R = 128, 4


def unit_rms(v):
    return v / np.sqrt(np.mean(v * v))


def test_one_hot_gate_picks_one_token_of_the_current_window():
    """Row 0 has no previous window; a gate logit far above the rest puts all weight on
    one token per output dim, so the pooled row is that token's value (channels D..2D-1),
    unit RMS, at position 0 (no rotation)."""
    rng = np.random.default_rng(1)
    kv = rng.standard_normal((R, 2 * D))
    v = unit_rms(rng.standard_normal(D))
    winner = rng.integers(0, R, D)                 # the token that wins dim d
    for d in range(D):
        kv[winner[d], D + d] = v[d]
    gate = np.zeros((R, 2 * D))
    gate[winner, D + np.arange(D)] = 1e3
    out = O.compress_rows(kv, gate, np.zeros((R, 2 * D)), np.ones(D), [0], R)[0]
    np.testing.assert_allclose(out, v / math.sqrt(1 + O.RMS_EPS), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("which", ["previous", "current"])
def test_overlap_draws_first_half_from_previous_window(which):
    """Row p > 0 weighs 2r entries: channels 0..D-1 of the previous window's tokens and
    channels D..2D-1 of its own window's tokens. A one-hot gate on either side returns
    that token's half, rotated at position p r."""
    rng = np.random.default_rng(2)
    p = 3
    T = (p + 1) * R
    kv = rng.standard_normal((T, 2 * D))
    v = unit_rms(rng.standard_normal(D))
    gate = np.zeros((T, 2 * D))
    if which == "previous":
        t = (p - 1) * R + 2
        kv[t, :D] = v
        gate[t, :D] = 1e3
    else:
        t = p * R + 1
        kv[t, D:] = v
        gate[t, D:] = 1e3
    out = O.compress_rows(kv, gate, np.zeros((R, 2 * D)), np.ones(D), [p], R)[0]
    want = O.rope_interleaved(v / math.sqrt(1 + O.RMS_EPS), p * R)
    np.testing.assert_allclose(out, want, rtol=1e-12, atol=1e-12)
    # and position p r rotates pair 32 (the first rotated pair, 1 rad per position) by 12 rad
    a, b = v[64] / math.sqrt(1 + O.RMS_EPS), v[65] / math.sqrt(1 + O.RMS_EPS)
    ang = p * R * 1.0
    assert out[64] == pytest.approx(a * math.cos(ang) - b * math.sin(ang), abs=1e-12)
    assert out[65] == pytest.approx(a * math.sin(ang) + b * math.cos(ang), abs=1e-12)


def test_uniform_gate_is_the_mean_of_the_entries():
    """Equal gate logits (gate + ape constant per dim) weigh every entry 1/(2r): the pooled
    row before the norm is the mean of the 2r entries; with a unit-RMS mean and no rotated
    dims (rope_dims = 0) the output is that mean / sqrt(1 + eps)."""
    rng = np.random.default_rng(3)
    p = 2
    T = (p + 1) * R
    kv = rng.standard_normal((T, 2 * D))
    ape = rng.standard_normal((R, 2 * D))
    gate = np.tile(-ape, (p + 1, 1)) + 0.25       # gate + ape = 0.25 everywhere
    prev = kv[(p - 1) * R:p * R, :D]
    cur = kv[p * R:(p + 1) * R, D:]
    m = (prev.sum(axis=0) + cur.sum(axis=0)) / (2 * R)
    s = 1.0 / np.sqrt(np.mean(m * m))
    out = O.compress_rows(kv * s, gate, ape, np.ones(D), [p], R, rope_dims=0)[0]
    np.testing.assert_allclose(out, m * s / math.sqrt(1 + O.RMS_EPS), rtol=1e-11, atol=1e-12)
    # row 0: the r entries of its own window only
    m0 = kv[:R, D:].mean(axis=0)
    s0 = 1.0 / np.sqrt(np.mean(m0 * m0))
    out0 = O.compress_rows(kv * s0, gate, ape, np.ones(D), [0], R, rope_dims=0)[0]
    np.testing.assert_allclose(out0, m0 * s0 / math.sqrt(1 + O.RMS_EPS), rtol=1e-11, atol=1e-12)
    # without the overlap variant, r entries of width D
    kv1 = kv[:, :D]
    m1 = kv1[p * R:(p + 1) * R].mean(axis=0)
    s1 = 1.0 / np.sqrt(np.mean(m1 * m1))
    out1 = O.compress_rows(kv1 * s1, np.zeros((T, D)), np.zeros((R, D)), np.ones(D), [p], R,
                           overlap=False, rope_dims=0)[0]
    np.testing.assert_allclose(out1, m1 * s1 / math.sqrt(1 + O.RMS_EPS), rtol=1e-11, atol=1e-12)


def test_pooled_row_depends_only_on_its_two_windows():
    """Pooled row p is anchored at [p r, p r + r - 1] and, with overlap, the window before."""
    rng = np.random.default_rng(4)
    T = 6 * R
    kv, gate = rng.standard_normal((T, 2 * D)), rng.standard_normal((T, 2 * D))
    ape, w = rng.standard_normal((R, 2 * D)), rng.standard_normal(D)
    p = 3
    base = O.compress_rows(kv, gate, ape, w, [p], R)[0]
    for t in range(T):
        kv2 = kv.copy()
        kv2[t] += 1.0
        moved = not np.allclose(O.compress_rows(kv2, gate, ape, w, [p], R)[0], base,
                                rtol=0, atol=1e-12)
        assert moved == ((p - 1) * R <= t < (p + 1) * R), t


def test_rms_norm_unit_weight_and_scale_invariance():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((3, D)) * 5.0
    y = O.rms_norm(x, np.ones(D))
    ms = np.mean(x * x, axis=-1)
    np.testing.assert_allclose(np.mean(y * y, axis=-1), ms / (ms + O.RMS_EPS), rtol=1e-13)
    cos = np.sum(y * x, axis=-1) / np.linalg.norm(y, axis=-1) / np.linalg.norm(x, axis=-1)
    np.testing.assert_allclose(cos, 1.0, rtol=1e-13)
    w = rng.standard_normal(D)
    np.testing.assert_allclose(O.rms_norm(x, w), O.rms_norm(x, np.ones(D)) * w, rtol=1e-13)


def test_rope_frequencies_closed_forms():
    """theta = 160000 over a 64-dim subspace: the first rotated pair turns 1 rad per
    position, pair 16 turns theta^(-1/2) = 1/400 rad, and consecutive pairs differ by
    the constant ratio theta^(-1/32); dims 0..63 never move."""
    rng = np.random.default_rng(6)
    x = rng.standard_normal(D)
    pos = 7
    y = O.rope_interleaved(x, pos)
    np.testing.assert_array_equal(y[:64], x[:64])

    def angle(i):
        m = 32 + i
        a = math.atan2(x[2 * m] * y[2 * m + 1] - x[2 * m + 1] * y[2 * m],
                       x[2 * m] * y[2 * m] + x[2 * m + 1] * y[2 * m + 1])
        return a

    assert angle(0) == pytest.approx(pos - 2 * math.pi, abs=1e-12)          # 7 rad
    assert angle(16) == pytest.approx(pos / 400.0, abs=1e-14)
    ratio = [(angle(i + 1) / angle(i)) for i in range(8, 31)]
    np.testing.assert_allclose(ratio, 160000.0 ** (-1 / 32), rtol=1e-9)
    # each pair keeps its length
    n_x = x[64:].reshape(32, 2)
    n_y = y[64:].reshape(32, 2)
    np.testing.assert_allclose(np.linalg.norm(n_y, axis=1), np.linalg.norm(n_x, axis=1), rtol=1e-13)


def test_rope_composition_and_relative_position():
    rng = np.random.default_rng(7)
    q, k = rng.standard_normal(D), rng.standard_normal(D)
    np.testing.assert_allclose(O.rope_interleaved(q, 0), q, rtol=0, atol=0)
    np.testing.assert_allclose(O.rope_interleaved(O.rope_interleaved(q, 100), 23),
                               O.rope_interleaved(q, 123), rtol=1e-12, atol=1e-12)
    d1 = O.rope_interleaved(q, 5000) @ O.rope_interleaved(k, 4000)
    d2 = O.rope_interleaved(q, 1003) @ O.rope_interleaved(k, 3)
    assert d1 == pytest.approx(d2, rel=1e-9)

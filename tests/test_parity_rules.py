"""The comparison rules of oracle/parity.py can fail: planted mistakes are rejected,
the rounding the kernels are designed to do is accepted (CPU only).

Mistakes are planted in the oracle's own outputs and arguments: an all-zero output,
a random selection, a dropped sink, a missing sliding-window mask, a re-mask off by
one row, and indexer scores from a query split into two bf16 planes instead of three.
The accepted side simulates, in f64, exactly the roundings the kernels make: softmax
weights rounded to bf16 before the value product, and f32 evaluation of the scores.
Page cited: "feat(deepseek-v4): implement HiSA hierarchical sparse attention"
("Consuming the selection: sparse combine", "Conventions").
"""
import numpy as np
import pytest

from deepseek_sparse_attention_hisa_gb300 import inputs
from oracle import hisa_oracle as O
from oracle import parity as P


def bf16_round(x):
    """f64 -> f32 -> bf16 (nearest even) -> f64."""
    return O.to_f64(inputs.f32_to_bf16_bits(np.asarray(x, dtype=np.float32)))


def bf16_trunc(x):
    """f32 -> bf16 by dropping the low 16 bits (toward zero)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32) & np.uint32(0xFFFF0000)
    return u.view(np.float32)


def weights_and_values(data, b, j, I_row):
    """The oracle's normalised softmax weights of row (b, j) over [local rows; selected
    rows] and those rows' values (test-side restatement, for the rounding simulation)."""
    wl = data["wl"]
    s = P.seq(data, b)
    o, n = O.sparse_combine(data["q_attn"][b, j:j + 1], s["local_kv"], s["local_pos0"],
                            s["pooled_kv"], None if I_row is None else np.asarray(I_row)[None],
                            data["sinks"], s["t0"] + j, wl.r, wl.window, causal=wl.L > 1,
                            return_lse=True)
    q = O.to_f64(data["q_attn"][b, j]) * wl.Dh ** -0.5
    loc = O.to_f64(s["local_kv"])
    t = s["t0"] + j
    spos = s["local_pos0"] + np.arange(loc.shape[0])
    lvis = (t - spos >= 0) & (t - spos < wl.window)
    ids = np.asarray(I_row, dtype=np.int64)
    pvis = ids >= 0
    if wl.L > 1:
        pvis &= ids < O.visible_len(t, wl.r, s["Np"])
    pooled = O.to_f64(s["pooled_kv"])[np.where(ids >= 0, ids, 0)]
    V = np.concatenate([loc, pooled])
    vis = np.concatenate([lvis, pvis])
    S = q @ V.T
    Wt = np.where(vis[None, :], np.exp(np.where(vis[None, :], S, 0.0) - n[0][:, None]), 0.0)
    return Wt, V, o[0]


@pytest.fixture(scope="module")
def decode_case():
    """V4-Flash decode (Np = 32768) with the oracle's own HiSA selection."""
    data = inputs.generate("v4flash_decode")
    s = P.seq(data, 0)
    sel = O.hisa_select_decode(data["q_idx"][0, 0], data["w"][0, 0], s["keys"], 64, 16, 512)
    return data, sel


@pytest.fixture(scope="module")
def peaked_decode_case():
    data = inputs.generate(inputs.peaked(inputs.WORKLOADS["v4flash_decode"]))
    s = P.seq(data, 0)
    sel = O.hisa_select_decode(data["q_idx"][0, 0], data["w"][0, 0], s["keys"], 64, 16, 512)
    return data, sel


def rejects(data, b, j, I_row, bad):
    """True when the attention check rejects output `bad` for row (b, j)."""
    o = P.combine_row(data, b, j, I_row)
    E = P.combine_row(data, b, j, I_row, magnitude=True)
    dt = P._dtype_name(data["pooled_kv"])
    err, _, n_bad = P.attention_violations(bad, o, E, dt)
    return err > P.ATTN_TOL[dt] or n_bad > 0


def test_magnitude_bounds_the_output_and_equals_it_for_positive_values():
    data = inputs.generate(inputs.small_workload(seed=3, kv_dtype="f32"))
    I = np.arange(32)
    o = P.combine_row(data, 0, 0, I)
    E = P.combine_row(data, 0, 0, I, magnitude=True)
    assert np.all(E >= np.abs(o) - 1e-15) and np.all(E > 0)
    data["local_kv"] = np.abs(data["local_kv"])
    data["pooled_kv"] = np.abs(data["pooled_kv"])
    o = P.combine_row(data, 0, 0, I)
    E = P.combine_row(data, 0, 0, I, magnitude=True)
    assert np.allclose(o, E, rtol=1e-14, atol=0)


@pytest.mark.parametrize("case", ["decode_case", "peaked_decode_case"])
def test_bf16_weight_rounding_is_accepted(case, request):
    data, sel = request.getfixturevalue(case)
    Wt, V, o = weights_and_values(data, 0, 0, sel["I"])
    sim = bf16_round(Wt) @ V                       # the kernel's rounding of P, in f64
    assert np.abs(sim - o).max() > 0
    o_ref = P.combine_row(data, 0, 0, sel["I"])
    assert np.allclose(o, o_ref, rtol=1e-12, atol=1e-15)
    E = P.combine_row(data, 0, 0, sel["I"], magnitude=True)
    err, r, n_bad = P.attention_violations(sim, o_ref, E, "bf16")
    assert n_bad == 0 and err <= 1e-2, (err, r)
    assert r > 0.05 * P.ATTN_EPS["bf16"]            # the bound is not vacuous for this rounding


def test_decode_mistakes_are_rejected(decode_case):
    """The pages' V4-Flash decode distributions: outputs are about 1e-3, below the
    absolute tolerance, so only the element-wise bound can see these mistakes."""
    data, sel = decode_case
    I = sel["I"]
    o = P.combine_row(data, 0, 0, I)
    assert np.abs(o).max() < P.ATTN_TOL["bf16"]     # why the absolute bound alone is blind
    assert rejects(data, 0, 0, I, np.zeros_like(o))
    rnd = np.random.default_rng(5).choice(32768, 512, replace=False)
    assert rejects(data, 0, 0, I, P.combine_row(data, 0, 0, rnd))
    one_off = np.array(I)
    one_off[0] = (one_off[0] + 1) % 32768 if one_off[0] + 1 not in set(I.tolist()) else \
        (one_off[0] + 2) % 32768
    assert rejects(data, 0, 0, I, P.combine_row(data, 0, 0, one_off))   # one row swapped
    half = np.array(I)
    half[256:] = -1
    assert rejects(data, 0, 0, I, P.combine_row(data, 0, 0, half))      # half the rows dropped


def test_peaked_decode_mistakes_are_rejected(peaked_decode_case):
    data, sel = peaked_decode_case
    I = sel["I"]
    o = P.combine_row(data, 0, 0, I)
    assert np.abs(o).max() > 10 * P.ATTN_TOL["bf16"]  # outputs of order one
    assert rejects(data, 0, 0, I, np.zeros_like(o))
    rnd = np.random.default_rng(6).choice(32768, 512, replace=False)
    assert rejects(data, 0, 0, I, P.combine_row(data, 0, 0, rnd))
    no_sink = dict(data, sinks=np.full_like(data["sinks"], -np.inf))
    assert rejects(data, 0, 0, I, P.combine_row(no_sink, 0, 0, I))      # sink dropped
    sink_twice = dict(data, sinks=data["sinks"] + np.float32(np.log(2.0)))
    assert rejects(data, 0, 0, I, P.combine_row(sink_twice, 0, 0, I))   # sink counted twice
    unscaled = P.combine_row(data, 0, 0, I, scale=1.0 / 16.0)           # 1/16 for Dh^-1/2
    assert rejects(data, 0, 0, I, unscaled)


@pytest.fixture(scope="module")
def prefill_rows_case():
    """Prefill-shaped rows (V4 attention shape, L = 40 rows from t0 = 3000, Np = 2048) with
    random selections that include ids past V(t): the re-mask and the window both matter."""
    wl = inputs.small_workload(name="rows", seed=13, L=40, H_i=64, D_i=128, index_block=64,
                               index_keep=16, index_topk=512, H=64, Dh=512, window=128,
                               q_idx_dtype="f32", key_dtype="bf16", kv_dtype="bf16",
                               Np=(2048,), t0=3000)
    out = {}
    for name, w in (("pages", wl), ("peaked", inputs.peaked(wl))):
        data = inputs.generate(w)
        rng = np.random.default_rng(1)
        I = np.stack([rng.choice(2048, 512, replace=False) for _ in range(40)])
        for j in range(40):                         # every row holds the id V(t) itself
            V = O.visible_len(3000 + j, 4, 2048)
            if V not in set(I[j].tolist()):
                I[j, 0] = V
        out[name] = (data, I)
    return out


@pytest.mark.parametrize("dist", ["pages", "peaked"])
def test_prefill_row_mistakes_are_rejected(prefill_rows_case, dist, monkeypatch):
    data, I = prefill_rows_case[dist]
    rows = [0, 17, 39]
    for j in rows:
        Wt, V, o = weights_and_values(data, 0, j, I[j])
        E = P.combine_row(data, 0, j, I[j], magnitude=True)
        _, _, n_bad = P.attention_violations(bf16_round(Wt) @ V, o, E, "bf16")
        assert n_bad == 0
        assert rejects(data, 0, j, I[j], np.zeros_like(o))
        # no sliding-window mask: every cached local row visible (row 0's window already
        # holds every local row at or before it)
        if j > 0:
            assert rejects(data, 0, j, I[j], P.combine_row(data, 0, j, I[j], window=10 ** 9))
        # no causal re-mask of pooled ids past V(t)
        assert rejects(data, 0, j, I[j], P.combine_row(data, 0, j, I[j], causal=False))
    # the re-mask one row late: the id V(t) itself counted as visible
    real = O.visible_len
    late = {j: None for j in rows}
    for j in rows:
        monkeypatch.setattr(O, "visible_len", lambda t, r, Np: real(t, r, Np) + 1)
        late[j] = P.combine_row(data, 0, j, I[j])
        monkeypatch.setattr(O, "visible_len", real)
    assert any(rejects(data, 0, j, I[j], late[j]) for j in rows)
    # the window edge one row wide (0 <= t - s <= window)
    assert any(rejects(data, 0, j, I[j], P.combine_row(data, 0, j, I[j], window=129))
               for j in rows)


def test_prefill_workload_rows_reject_a_missing_window_mask():
    """The prefill workload itself (L = 4096 rows from t0 = 61440, 128 cached + 4096 new
    local rows): the window mask keeps 128 of them per row."""
    data = inputs.generate("prefill")
    s = P.seq(data, 0)
    for j in (0, 2000, 4095):
        V = O.visible_len(61440 + j, 4, 16384)
        sel = O.hisa_select_batched(data["q_idx"][0, j:j + 1], data["w"][0, j:j + 1], s["keys"],
                                    61440 + j, 4, 64, 16, 512)
        I = sel["I"][0]
        assert np.all(I < V)
        o = P.combine_row(data, 0, j, I)
        assert rejects(data, 0, j, I, np.zeros_like(o))
        assert rejects(data, 0, j, I, P.combine_row(data, 0, j, I, window=10 ** 9))


# ----------------------------------------------------------------------------
# indexer scores: f32 precision
# ----------------------------------------------------------------------------
def _fine_inputs(decode_case):
    data, sel = decode_case
    s = P.seq(data, 0)
    q, w = data["q_idx"][0, 0], data["w"][0, 0]
    pos = np.sort(sel["pos"])
    rows = np.asarray(s["keys"])[pos]
    return q, w, rows


def f32_scores(q, w, rows):
    """Scores evaluated in f32 arithmetic (f32 products and sums, f32 head weights)."""
    q32 = np.asarray(O.to_f64(q), dtype=np.float32)
    r32 = np.asarray(O.to_f64(rows), dtype=np.float32)
    H_i, D_i = q32.shape
    wp = (np.asarray(w, np.float32) * np.float32(O.head_scale(H_i, D_i))).astype(np.float32)
    dots = np.maximum(q32 @ r32.T, np.float32(0))
    return (wp @ dots).astype(np.float64)


def test_f32_score_evaluation_is_accepted(decode_case):
    q, w, rows = _fine_inputs(decode_case)
    o = O.combined_scores(q, w, rows)
    g = f32_scores(q, w, rows)
    assert np.abs(g - o).max() > 0
    P.check_scores(g, o, P.score_scale(q, w, rows), what="f32 evaluation")


def test_two_plane_query_split_is_rejected(decode_case):
    """A query split into two truncated bf16 planes (16 significant bits) instead of three
    (all 24 of f32): exact products of the truncated query fail the f32 bound while they
    still pass the looser target tolerance."""
    q, w, rows = _fine_inputs(decode_case)
    q32 = np.asarray(O.to_f64(q), dtype=np.float32)
    hi = bf16_trunc(q32)
    lo = bf16_trunc(q32 - hi)
    mid_lo = q32 - hi - lo
    assert np.array_equal(hi.astype(np.float64) + lo + bf16_trunc(mid_lo), q32)   # 3 planes exact
    q2 = hi.astype(np.float64) + lo.astype(np.float64)
    o = O.combined_scores(q, w, rows)
    g = O.combined_scores(q2, w, rows)
    A = P.score_scale(q, w, rows)
    P.check_scores(g, o, A, f32_tol=None, what="two planes, target only")
    with pytest.raises(AssertionError, match="f32 bound"):
        P.check_scores(g, o, A, what="two planes")


def test_score_scale_skips_heads_that_relu_zeroes():
    """A' counts a head only where its dot product can pass the relu."""
    q = np.array([[1.0, 0.0], [1.0, 0.0]])
    w = np.array([1.0, 1.0])
    rows = np.array([[2.0, 0.0], [-2.0, 0.0]])
    A = P.score_scale(q, w, rows)
    c = O.head_scale(2, 2)
    assert A[0] == pytest.approx(4.0 * c) and A[1] == 0.0
    q = np.array([[1.0, 0.0], [-1.0, 0.0]])
    A = P.score_scale(q, w, rows)
    assert A[0] == pytest.approx(2.0 * c) and A[1] == pytest.approx(2.0 * c)


@pytest.mark.parametrize("kv", ["f32", "bf16"])
def test_bf16_output_rounding_is_accepted_and_mistakes_are_not(kv):
    """A bf16 output (hisa_attn_desc.out_dtype) is the result rounded to nearest once: the
    oracle's own output rounded so passes the widened check. With f32 KV the plain f32 check
    (eps = 2^-13) rejects that rounding, so the widening is what admits it; zeros and a sign
    flip of one head stay rejected."""
    data = inputs.generate(inputs.peaked(inputs.WORKLOADS["v4flash_decode"]) if kv == "bf16"
                           else inputs.small_workload(seed=5, kv_dtype="f32"))
    Np = int(data["Np"][0])
    k = int(data["wl"].index_topk)
    I = np.arange(min(k, Np))
    o = P.combine_row(data, 0, 0, I)
    E = P.combine_row(data, 0, 0, I, magnitude=True)
    r = inputs.f32_to_bf16_bits(o.astype(np.float32))
    err, _, n_bad = P.attention_violations(r, o, E, kv, out_bf16=True)
    assert n_bad == 0 and err <= P.ATTN_TOL[kv] + P.OUT_BF16_U * np.abs(o).max()
    if kv == "f32":
        _, _, n_plain = P.attention_violations(O.to_f64(r), o, E, kv)
        assert n_plain > 0
    for bad in (np.zeros_like(o), np.where(np.arange(o.shape[0])[:, None] == 3, -o, o)):
        b16 = inputs.f32_to_bf16_bits(bad.astype(np.float32))
        _, _, nb = P.attention_violations(b16, o, E, kv, out_bf16=True)
        assert nb > 0

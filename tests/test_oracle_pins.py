"""Pins for the CPU oracle: checks against what the pages and the mathematics fix.

Each test ties an oracle function to something other than itself: values the
pages print (tests/golden/), closed forms, brute-force enumeration on tiny
inputs, invariants the page states, and a textbook-softmax restatement of the
combine. Page cited: "feat(deepseek-v4): implement HiSA hierarchical sparse
attention" ([HiSA issue]).
"""
import itertools
import math
import os

import numpy as np
import pytest
from scipy.special import softmax as sp_softmax

from deepseek_sparse_attention_hisa_gb300 import inputs
from oracle import hisa_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------
# helpers independent of the oracle
# --------------------------------------------------------------------------
def _beats(sa, ia, sb, ib):
    """Total order of the selection: higher score first, equal scores by lower id."""
    return sa > sb or (sa == sb and ia < ib)


def brute_topk_set(scores, k, ids=None):
    """The unique k-subset whose every member beats every non-member (enumeration)."""
    n = len(scores)
    ids = list(range(n)) if ids is None else list(ids)
    found = []
    for S in itertools.combinations(range(n), k):
        inside = set(S)
        if all(_beats(scores[a], ids[a], scores[b], ids[b])
               for a in S for b in range(n) if b not in inside):
            found.append(S)
    assert len(found) == 1
    return {ids[i] for i in found[0]}


def loop_score(q, w, row):
    """score of one row by plain Python loops (f64)."""
    H_i, D_i = len(q), len(q[0])
    c = 1.0 / math.sqrt(H_i * D_i)
    tot = 0.0
    for h in range(H_i):
        dot = 0.0
        for d in range(D_i):
            dot += float(q[h][d]) * float(row[d])
        tot += float(w[h]) * c * max(dot, 0.0)
    return tot


def rand_case(rng, H_i=4, D_i=8, Np=40, L=1):
    q = rng.standard_normal((L, H_i, D_i))
    w = rng.standard_normal((L, H_i))
    keys = rng.standard_normal((Np, D_i))
    return q, w, keys


# --------------------------------------------------------------------------
# widening of bf16 inputs: the bf16 format definition
# --------------------------------------------------------------------------
def test_bf16_widening_closed_form():
    bits = np.array([0x3F80, 0xC000, 0x3F81, 0x0001, 0x7F7F, 0x8000, 0x4049], dtype=np.uint16)
    want = [1.0, -2.0, 1.0 + 2.0 ** -7, 2.0 ** -133, (2 - 2.0 ** -7) * 2.0 ** 127, -0.0,
            3.140625]
    got = O.to_f64(bits)
    assert list(got) == want
    assert math.copysign(1.0, got[5]) == -1.0


def test_generator_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(7)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32),
                        np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -1.0 - 2 ** -8, 0.0, -0.0],
                                 dtype=np.float32)])
    mine = inputs.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(mine, ref)


# --------------------------------------------------------------------------
# positions: V(t)  ([HiSA issue] "The pooled stream and positions")
# --------------------------------------------------------------------------
def test_visible_len_matches_window_rule():
    # pooled row p covers tokens [p*r, p*r + r - 1]; it is complete (visible) at t iff
    # its last token p*r + r - 1 <= t, i.e. r*(p+1) <= t+1. Count by enumeration.
    for r in (1, 4, 128):
        for Np in (0, 1, 7, 64):
            for t in range(0, 300, 7):
                count = sum(1 for p in range(Np) if p * r + r - 1 <= t)
                assert O.visible_len(t, r, Np) == count


def test_prefill_visibility_values():
    # t0 = 61440, L = 4096, r = 4, Np = 16384: first row sees 61441 // 4 = 15360 rows,
    # the last row (t = 65535) sees all 16384.
    assert O.visible_len(61440, 4, 16384) == 15360
    assert O.visible_len(61440 + 4095, 4, 16384) == 16384
    assert O.visible_len(61440 + 4094, 4, 16384) == 16383


# --------------------------------------------------------------------------
# top-k as a set: brute-force enumeration
# --------------------------------------------------------------------------
@pytest.mark.parametrize("seed", range(6))
def test_top_k_equals_bruteforce_with_ties(seed):
    rng = np.random.default_rng(seed)
    n = 9
    s = rng.integers(-3, 4, n).astype(np.float64)   # many exact ties
    s[rng.integers(0, n)] = -0.0                      # -0.0 ties with +0.0
    for k in range(0, n + 1):
        assert set(O.top_k(s, k).tolist()) == brute_topk_set(list(s), k)


def test_top_k_custom_ids_break_ties_by_id():
    s = np.array([1.0, 2.0, 1.0, 1.0])
    ids = np.array([30, 10, 5, 20])
    assert set(O.top_k(s, 2, ids).tolist()) == {10, 5}
    assert set(O.top_k(s, 3, ids).tolist()) == brute_topk_set(list(s), 3, list(ids))


# --------------------------------------------------------------------------
# scores: closed forms and a loop definition
# --------------------------------------------------------------------------
def test_scores_closed_form_one_hot():
    # H_i = 4, D_i = 16 gives scale H_i^-1/2 * D_i^-1/2 = 1/8 exactly. With
    # q_h = a_h e_{d_h}, key_p = b_p e_{e_p} and w_h = 8 m_h, every score is the
    # integer sum_h m_h * max(0, a_h b_p [d_h == e_p]).
    H_i, D_i, Np = 4, 16, 24
    rng = np.random.default_rng(3)
    a = rng.integers(-3, 4, H_i)
    dh = rng.integers(0, 4, H_i)
    m = rng.integers(-5, 6, H_i)
    bp = rng.integers(-3, 4, Np)
    ep = rng.integers(0, 4, Np)
    q = np.zeros((H_i, D_i))
    q[np.arange(H_i), dh] = a
    keys = np.zeros((Np, D_i))
    keys[np.arange(Np), ep] = bp
    w = 8.0 * m
    want = [sum(int(m[h]) * max(0, int(a[h]) * int(bp[p]) * int(dh[h] == ep[p]))
                for h in range(H_i)) for p in range(Np)]
    got = O.combined_scores(q, w, keys)
    assert got.tolist() == [float(x) for x in want]
    # the same through bf16 inputs (small integers are exact in bf16)
    qb = inputs.f32_to_bf16_bits(q.astype(np.float32))
    kb = inputs.f32_to_bf16_bits(keys.astype(np.float32))
    assert O.combined_scores(qb, w, kb).tolist() == [float(x) for x in want]


def test_scores_match_loop_definition():
    rng = np.random.default_rng(11)
    q, w, keys = rand_case(rng, H_i=3, D_i=5, Np=6)
    got = O.combined_scores(q[0], w[0], keys)
    want = [loop_score(q[0], w[0], keys[p]) for p in range(6)]
    np.testing.assert_allclose(got, want, rtol=1e-13, atol=1e-15)


def test_flat_mask_only_beyond_visible_prefix():
    rng = np.random.default_rng(5)
    L, Np, r, t0 = 6, 30, 4, 100          # V runs 25, 25, 25, 26, 26, 26
    q, w, keys = rand_case(rng, Np=Np, L=L)
    s = O.flat_scores(q, w, keys, t0, r)
    for j in range(L):
        V = (t0 + j + 1) // r
        assert np.all(s[j, V:] == -1e30)
        np.testing.assert_allclose(s[j, :V], O.combined_scores(q[j], w[j], keys)[:V], rtol=0)
    # L == 1 skips the mask
    s1 = O.flat_scores(q[:1], w[:1], keys, 0, r)
    assert np.all(s1 > -1e29)


def test_flat_selection_bruteforce_with_cutoff():
    rng = np.random.default_rng(9)
    L, Np, r, k = 5, 9, 1, 3
    t0 = 3                                   # V = 4, 5, 6, 7, 8 with r = 1
    q, w, keys = rand_case(rng, H_i=2, D_i=3, Np=Np, L=L)
    I = O.flat_top_indices(q, w, keys, t0, r, k)
    for j in range(L):
        V = t0 + j + 1
        sc = [loop_score(q[j], w[j], keys[p]) if p < V else -1e30 for p in range(Np)]
        assert set(I[j].tolist()) == brute_topk_set(sc, k)
        assert all(i < V for i in I[j])


def test_flat_k_clamped_to_Np():
    rng = np.random.default_rng(1)
    q, w, keys = rand_case(rng, Np=5)
    I = O.flat_top_indices(q, w, keys, 100, 4, 32)
    assert I.shape == (1, 5) and set(I[0].tolist()) == set(range(5))


# --------------------------------------------------------------------------
# HiSA  ([HiSA issue] "HiSA decode path", "HiSA batched path")
# --------------------------------------------------------------------------
def test_block_means_closed_form():
    b, nb, tail = 4, 5, 3
    Np = nb * b + tail
    keys = np.repeat(np.arange(Np, dtype=np.float64)[:, None], 3, axis=1)
    keys[:, 1] *= -2.0
    rep = O.block_means(keys, b)
    assert rep.shape == (nb, 3)
    for beta in range(nb):
        mean_p = beta * b + (b - 1) / 2.0     # mean of b consecutive integers
        assert rep[beta].tolist() == [mean_p, -2.0 * mean_p, mean_p]


@pytest.mark.parametrize("seed", range(4))
def test_hisa_equals_flat_when_every_block_kept(seed):
    # keep = nb and Np = nb * b: the candidate table is every pooled row, so the
    # fine stage rescans exactly the flat scores.
    rng = np.random.default_rng(seed)
    b, nb, k = 8, 6, 10
    Np = nb * b
    q, w, keys = rand_case(rng, Np=Np, L=3)
    d = O.hisa_select_decode(q[0], w[0], keys, b, nb, k)
    flat = O.flat_top_indices(q[:1], w[:1], keys, 4 * Np - 1, 4, k)[0]
    assert set(d["I"].tolist()) == set(flat.tolist())
    t0 = 4 * (Np - 20)                          # some rows see fewer than Np rows
    bt = O.hisa_select_batched(q, w, keys, t0, 4, b, nb, k)
    fl = O.flat_top_indices(q, w, keys, t0, 4, k)
    for j in range(3):
        assert set(bt["I"][j].tolist()) == set(fl[j].tolist())


def test_hisa_planted_equivalence():
    # Plant score mass so the true top-k rows lie inside Kb blocks whose means also
    # score highest; then the hierarchy returns the flat top-k set.
    rng = np.random.default_rng(21)
    H_i, D_i, b, nb, keep, k = 4, 16, 16, 32, 4, 24
    Np = nb * b + 5
    u = rng.standard_normal(D_i)
    u /= np.linalg.norm(u)
    q = (u[None, :] * 2.0 + 0.05 * rng.standard_normal((H_i, D_i)))
    w = np.abs(rng.standard_normal(H_i)) + 0.5
    keys = rng.standard_normal((Np, D_i))
    keys -= np.outer(keys @ u, u)               # no component along u ...
    keys -= 0.5 * u                             # ... and a negative one everywhere
    planted = rng.choice(nb, keep, replace=False)
    for beta in planted:
        keys[beta * b:(beta + 1) * b] += 4.0 * u + 0.3 * rng.standard_normal((b, D_i))
    flat = O.flat_top_indices(q[None], w[None], keys, 4 * Np - 1, 4, k)[0]
    assert set(flat // b) <= set(planted)       # precondition of the construction
    d = O.hisa_select_decode(q, w, keys, b, keep, k)
    assert set(d["top_blk"].tolist()) == set(planted.tolist())
    assert set(d["I"].tolist()) == set(flat.tolist())
    bt = O.hisa_select_batched(np.stack([q, q]), np.stack([w, w]), keys, 4 * Np - 2, 4, b,
                               keep, k)
    assert set(bt["I"][1].tolist()) == set(flat.tolist())


def test_head_permutation_and_tied_head_invariance():
    rng = np.random.default_rng(4)
    H_i, D_i, Np, b, keep, k = 6, 8, 96, 8, 3, 12
    q, w, keys = rand_case(rng, H_i=H_i, D_i=D_i, Np=Np)
    q, w = q[0], w[0]
    base = O.hisa_select_decode(q, w, keys, b, keep, k)
    perm = rng.permutation(H_i)
    p = O.hisa_select_decode(q[perm], w[perm], keys, b, keep, k)
    np.testing.assert_allclose(p["fscore"], base["fscore"], rtol=1e-12, atol=1e-14)
    assert set(p["I"].tolist()) == set(base["I"].tolist())
    # two identical heads with weights w1, w2 act as one head of weight w1 + w2;
    # merging changes H_i, so every weight carries the ratio of the two scales.
    q2 = np.concatenate([q, q[:1]])
    w2 = np.concatenate([w, [0.7]])
    tied = O.hisa_select_decode(q2, w2, keys, b, keep, k)
    merged_w = w * math.sqrt(H_i / (H_i + 1))   # every head: scale of H_i+1 heads
    merged_w[0] = (w[0] + 0.7) * math.sqrt(H_i / (H_i + 1))
    merged = O.hisa_select_decode(q, merged_w, keys, b, keep, k)
    np.testing.assert_allclose(tied["fscore"], merged["fscore"], rtol=1e-12, atol=1e-14)
    assert set(tied["I"].tolist()) == set(merged["I"].tolist())


def test_positive_homogeneity():
    # relu is positively homogeneous: q -> 2q, w -> 4w scales every score by 8 exactly.
    rng = np.random.default_rng(8)
    q, w, keys = rand_case(rng, Np=64)
    s = O.combined_scores(q[0], w[0], keys)
    s2 = O.combined_scores(2 * q[0], 4 * w[0], keys)
    assert np.array_equal(s2, 8 * s)
    a = O.hisa_select_decode(q[0], w[0], keys, 8, 3, 10)
    c = O.hisa_select_decode(2 * q[0], 4 * w[0], keys, 8, 3, 10)
    assert set(a["I"].tolist()) == set(c["I"].tolist())


def test_coarse_sums_select_same_blocks_as_means():
    rng = np.random.default_rng(6)
    b = 8
    q, w, keys = rand_case(rng, Np=8 * 20)
    rep = O.block_means(keys, b)
    _, tb_mean = O.hisa_coarse(q[0], w[0], rep, 5, b)
    _, tb_sum = O.hisa_coarse(q[0], w[0], rep * b, 5, b)   # b is a power of 2: exact
    assert set(tb_mean.tolist()) == set(tb_sum.tolist())


def test_tail_exclusion():
    rng = np.random.default_rng(12)
    b, nb, tail, keep, k = 8, 10, 6, 4, 8
    Np = nb * b + tail
    q, w, keys = rand_case(rng, Np=Np)
    w = np.abs(w)
    keys[nb * b:] = 10.0 * np.sign(q[0].sum(axis=0))     # the best rows sit in the tail
    flat = O.flat_top_indices(q, w, keys, 4 * Np - 1, 4, k)[0]
    assert any(i >= nb * b for i in flat)
    d = O.hisa_select_decode(q[0], w[0], keys, b, keep, k)
    assert all(i < nb * b for i in d["I"])
    bt = O.hisa_select_batched(np.repeat(q, 2, 0), np.repeat(w, 2, 0), keys, 4 * Np - 2, 4, b,
                               keep, k)
    assert np.all(bt["I"] < nb * b)


def test_batched_causality_and_eligibility():
    rng = np.random.default_rng(13)
    b, nb, keep, k, r = 4, 16, 4, 8, 4
    Np = nb * b
    L = 40
    t0 = 4                                   # V(t) grows from 1 to 11
    q, w, keys = rand_case(rng, Np=Np, L=L)
    bt = O.hisa_select_batched(q, w, keys, t0, r, b, keep, k)
    for j in range(L):
        V = bt["valid_len"][j]
        assert V == min(Np, (t0 + j + 1) // r)
        eligible = [beta for beta in range(nb) if beta * b < V]
        # coarse: all eligible blocks come first; ineligible ones only by lowest id
        if len(eligible) >= keep:
            assert set(bt["top_blk"][j].tolist()) <= set(eligible)
        else:
            assert set(eligible) <= set(bt["top_blk"][j].tolist())
        if V >= k and len(eligible) >= keep:
            cand_vis = [p for p in bt["pos"][j] if p < V]
            if len(cand_vis) >= k:
                assert np.all(bt["I"][j] < V)


def test_coarse_eligibility_boundary():
    # A block whose first row equals valid_len is ineligible even if it scores best;
    # the block just before it (first row valid_len - b) is eligible.
    rng = np.random.default_rng(15)
    b, nb, keep, k, r = 4, 12, 2, 4, 1
    Np = nb * b
    q, w, keys = rand_case(rng, Np=Np, L=1)
    w = np.abs(w)
    V = 5 * b                                    # rows 0..19 visible: blocks 0..4 eligible
    keys[V:V + b] = 50.0 * np.sign(q[0].sum(axis=0))   # block 5 starts exactly at V
    keys[V - b:V] = 20.0 * np.sign(q[0].sum(axis=0))   # block 4 ends at V - 1
    t0 = V - 1                                   # r = 1: V(t0) = t0 + 1
    bt = O.hisa_select_batched(np.repeat(q, 2, 0), np.repeat(w, 2, 0), keys, t0, r, b, keep, k)
    assert bt["valid_len"][0] == V
    assert 5 not in bt["top_blk"][0] and 4 in bt["top_blk"][0]
    assert 5 in bt["top_blk"][1]                 # next row: V + 1 > 5 * b, block 5 eligible


def _tiny_hisa_decode_bruteforce(q, w, keys, b, keep, k):
    """HiSA decode by plain loops and enumeration of every block and row subset."""
    Np, D_i = len(keys), len(keys[0])
    nb = Np // b
    rep = [[sum(keys[beta * b + i][d] for i in range(b)) / b for d in range(D_i)]
           for beta in range(nb)]
    cs = [loop_score(q, w, rep[beta]) for beta in range(nb)]
    blocks = brute_topk_set(cs, min(keep, nb))
    cand = [beta * b + i for beta in sorted(blocks) for i in range(b)]
    fs = [loop_score(q, w, keys[p]) for p in cand]
    return blocks, brute_topk_set(fs, k, ids=cand)


@pytest.mark.parametrize("seed", range(5))
def test_hisa_decode_bruteforce_tiny(seed):
    rng = np.random.default_rng(100 + seed)
    b, keep, k = 4, 2, 4
    Np = 4 * 6 + (seed % 3)                   # with and without a tail
    q, w, keys = rand_case(rng, H_i=2, D_i=4, Np=Np)
    blocks, sel = _tiny_hisa_decode_bruteforce(q[0].tolist(), w[0].tolist(), keys.tolist(),
                                               b, keep, k)
    d = O.hisa_select_decode(q[0], w[0], keys, b, keep, k)
    assert set(d["top_blk"].tolist()) == blocks
    assert set(d["I"].tolist()) == sel


def test_fine_result_independent_of_block_order():
    rng = np.random.default_rng(14)
    q, w, keys = rand_case(rng, Np=64)
    q, w = q[0], w[0]
    w[:] = 0.0                                  # every fine score ties at 0
    _, _, a = O.hisa_fine(q, w, keys, [5, 1, 3], 8, 6)
    _, _, c = O.hisa_fine(q, w, keys, [3, 5, 1], 8, 6)
    assert set(a.tolist()) == set(c.tolist()) == set(range(8, 14))


# --------------------------------------------------------------------------
# gates and thresholds: the page's printed table
# --------------------------------------------------------------------------
def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


def test_engagement_thresholds_golden():
    for Np, L, path, branch in _golden_rows("engagement_thresholds.txt"):
        Np, L = int(Np), int(L)
        assert O.selection_path(L, Np, 64, 16, 512) == path, (Np, L)
        assert O.attention_branch(Np, 512) == branch, Np


def test_gate_fallbacks():
    assert not O.hisa_gate(1, 100000, 0, 16, 512)        # index_block == 0: flat only
    assert not O.hisa_gate(1, 1023, 64, 16, 512)         # Np < b * keep
    assert not O.hisa_gate(1, 100000, 16, 16, 512)       # b * keep < k
    assert O.hisa_gate(1, 1024, 64, 16, 512)


def test_v4flash_workload_matches_config_table():
    cfg = dict((a, int(b)) for a, b in _golden_rows("v4flash_config.txt"))
    for name in ("v4flash_decode", "ragged_decode", "prefill", "long_context"):
        wl = inputs.WORKLOADS[name]
        assert (wl.index_topk, wl.H_i, wl.D_i, wl.window, wl.index_block, wl.index_keep) == (
            cfg["index_topk"], cfg["index_n_heads"], cfg["index_head_dim"],
            cfg["sliding_window"], cfg["index_block"], cfg["index_keep"])


# --------------------------------------------------------------------------
# sparse combine  ([HiSA issue] "Consuming the selection: sparse combine")
# --------------------------------------------------------------------------
def _attn_case(rng, L=3, H=4, Dh=8, W=10, Np=20, k=6, t0=60, window=6):
    q = rng.standard_normal((L, H, Dh))
    local = rng.standard_normal((W, Dh)) / math.sqrt(Dh)
    pos0 = t0 + L - W
    pooled = rng.standard_normal((Np, Dh)) / math.sqrt(Dh)
    I = np.stack([rng.choice(Np, k, replace=False) for _ in range(L)])
    sinks = rng.standard_normal(H)
    return q, local, pos0, pooled, I, sinks


def _textbook(q, local, pos0, pooled, I, sinks, t0, r, window, causal, with_sink=True):
    """Plain softmax over the concatenated visible keys plus a sink column of value 0."""
    L, H, Dh = q.shape
    out = np.zeros((L, H, Dh))
    for j in range(L):
        t = t0 + j
        rows = [local[i] for i in range(len(local)) if t - window < pos0 + i <= t]
        Vt = min(len(pooled), (t + 1) // r) if causal else len(pooled)
        ids = range(len(pooled)) if I is None else I[j]
        rows += [pooled[p] for p in ids if 0 <= p < Vt]
        K = np.array(rows).reshape(-1, Dh)
        for h in range(H):
            logits = K @ q[j, h] / math.sqrt(Dh)
            if with_sink:
                wts = sp_softmax(np.append(logits, sinks[h]))[:-1]
            else:
                wts = sp_softmax(logits)
            out[j, h] = wts @ K
    return out


def test_combine_equals_textbook_softmax():
    rng = np.random.default_rng(30)
    q, local, pos0, pooled, I, sinks = _attn_case(rng)
    I[1, 2] = -1                                  # padding is skipped
    I[0, 0] = 19                                  # 19 >= V(60) = 15: re-masked in prefill
    I[2, 1] = 15                                  # exactly V(62) = 15: the first invisible id
    I[1, 3] = 14                                  # V(61) - 1 = 14: the last visible id
    got = O.sparse_combine(q, local, pos0, pooled, I, sinks, 60, 4, 6)
    want = _textbook(q, local, pos0, pooled, I, sinks, 60, 4, 6, causal=True)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-14)
    got1 = O.sparse_combine(q[:1], local, pos0, pooled, I[:1], sinks, 60, 4, 6)  # L == 1
    want1 = _textbook(q[:1], local, pos0, pooled, I[:1], sinks, 60, 4, 6, causal=False)
    np.testing.assert_allclose(got1, want1, rtol=1e-12, atol=1e-14)


def test_sparse_with_every_row_equals_dense():
    # k == Np: every pooled row selected, in any order; the combine reduces to dense.
    rng = np.random.default_rng(31)
    q, local, pos0, pooled, _, sinks = _attn_case(rng, Np=12, k=12, t0=200)
    I = np.stack([rng.permutation(12) for _ in range(3)])
    a = O.sparse_combine(q, local, pos0, pooled, I, sinks, 200, 4, 6)
    d = O.dense_combine(q, local, pos0, pooled, sinks, 200, 4, 6)
    np.testing.assert_allclose(a, d, rtol=1e-12, atol=1e-14)
    # Np < k: the selection pads with -1 and still equals dense
    Ipad = np.concatenate([I, -np.ones((3, 4), dtype=np.int64)], axis=1)
    np.testing.assert_allclose(O.sparse_combine(q, local, pos0, pooled, Ipad, sinks, 200, 4, 6),
                               d, rtol=1e-12, atol=1e-14)


def test_sink_limits_and_normaliser():
    rng = np.random.default_rng(32)
    q, local, pos0, pooled, I, sinks = _attn_case(rng, t0=300)
    # sink -> -inf: plain softmax attention without a sink
    lo = O.sparse_combine(q, local, pos0, pooled, I, np.full(4, -1e300), 300, 4, 6)
    want = _textbook(q, local, pos0, pooled, I, sinks, 300, 4, 6, causal=True, with_sink=False)
    np.testing.assert_allclose(lo, want, rtol=1e-12, atol=1e-14)
    # sink -> +inf: all mass goes to the sink, which carries no value
    hi = O.sparse_combine(q, local, pos0, pooled, I, np.full(4, 1e4), 300, 4, 6)
    assert np.max(np.abs(hi)) < 1e-300
    # weights plus the sink's share sum to one
    out, n = O.sparse_combine(q, local, pos0, pooled, I, sinks, 300, 4, 6, return_lse=True)
    for j in range(3):
        t = 300 + j
        for h in range(4):
            lg = [local[i] @ q[j, h] / math.sqrt(8) for i in range(len(local))
                  if 0 <= t - (pos0 + i) < 6]
            lg += [pooled[p] @ q[j, h] / math.sqrt(8) for p in I[j] if p < (t + 1) // 4]
            tot = sum(math.exp(x - n[j, h]) for x in lg) + math.exp(sinks[h] - n[j, h])
            assert abs(tot - 1.0) < 1e-12


def test_local_only_and_window_edge():
    rng = np.random.default_rng(33)
    q, local, pos0, pooled, I, sinks = _attn_case(rng, W=12, window=5)
    empty = np.zeros((0, 8))
    a = O.sparse_combine(q, local, pos0, empty, None, sinks, 60, 4, 5)
    want = _textbook(q, local, pos0, empty, None, sinks, 60, 4, 5, causal=True)
    np.testing.assert_allclose(a, want, rtol=1e-12, atol=1e-14)

"""Comparison rules between the CUDA path and the oracle (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and bench's CPU legs use this module.

Indexer scores ([HiSA issue] "Conventions": all selection scoring in f32).
  A'[p] = sum over the heads h whose oracle dot product q_h . row_p is not clearly
  negative (>= -1e-5 * sum_d |q_hd row_pd|) of |w'_h| * sum_d |q_hd row_pd|, with
  w'_h = w_h * H_i^-1/2 * D_i^-1/2: the size of every product that reaches score[p]
  through a relu that can pass it. A head whose dot product is clearly negative adds
  exactly zero on both sides, so it cannot add error. Two bounds are asserted:
  * target:    |g - o| <= 1e-5 * max(|o|, A')
  * f32 check: |g - o| <= SCORE_F32 * A', SCORE_F32 = 8 u = 4.8e-7 (u = 2^-24).
    With f32 operands split exactly into bf16 planes every product is exact, and a
    D_i = 128 dot product reaches its f32 accumulator in D_i / 16 = 8 steps of 16
    products (one tensor-core MMA each); each step rounds the running sum once, by u
    of its magnitude on average (at most the head's sum_d |q_hd row_d|), so 8 u per
    head, and the f32 head sum adds far less. A sequential f32 evaluation stays near
    0.3 u. Splitting an f32 operand into two bf16 planes instead of three leaves each
    product off by up to 2^-16 relative (about 15 u A' on the V4-Flash inputs) and
    fails this bound.
  Masked entries must be exactly -1e30.

Selections (unordered sets): equal, except ids whose oracle score lies within
1e-5 * max(|s_k|, A'_k, A'_id) of the k-th oracle score s_k (a near-tie that f32
rounding may order either way); at most NEAR_TIES_MAX such ids per row.

Attention outputs ([HiSA issue] "Consuming the selection: sparse combine"):
  * target:  max |g - o| <= 1e-2 for bf16 KV, 1e-4 for f32 KV.
  * element: |g - o| <= eps * E element by element, E = sum_j weight_j |v_j| (the
    oracle's softmax weights applied to |V|). The tensor-core combine rounds each
    softmax weight to bf16 (relative error <= 2^-8) before the value product; the
    rest is f32 with errors of order 1e-6 relative to E. So eps = 2^-8 * 9/8 for bf16
    KV (an eighth of margin for the f32 products, sums and the exp2 approximation).
    The f32 combine keeps the weights in f32: eps = 2^-13 (n u for n up to 2^11
    rows, u = 2^-24, times two for the exp and the normalisation).
  Zeros, a dropped row, a missing sink or a wrong mask move outputs by a sizeable
  fraction of E, which this bound catches where the absolute one cannot.
  * a bf16 output (hisa_attn_desc.out_dtype) is the f32 result rounded to nearest once,
    which adds at most u |g32| with u = 2^-8 (8 significand bits; |g32| <= |o| + eps E,
    |o| <= E): both bounds widen, to eps E (1 + u) + u |o| and target + u max|o|.

Every check records its worst ratios in STATS, printed at the end of a pytest run.
"""
from __future__ import annotations

import os

import numpy as np

from . import hisa_oracle as O

SCORE_RTOL = 1e-5
SCORE_F32 = 8 * 2.0 ** -24
NEAR_TIES_MAX = 4
ATTN_TOL = {"bf16": 1e-2, "f32": 1e-4}
ATTN_EPS = {"bf16": 2.0 ** -8 * 9 / 8, "f32": 2.0 ** -13}
OUT_BF16_U = 2.0 ** -8

STATS: dict = {}


def _record(kind, **vals):
    test = os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0].split("::")[-1] or "-"
    ent = STATS.setdefault((test, kind), {"checks": 0})
    ent["checks"] += 1
    for k, v in vals.items():
        if k.startswith("sum_"):
            ent[k] = ent.get(k, 0) + v
        else:
            ent[k] = max(ent.get(k, 0.0), v)


def format_stats() -> str:
    lines = []
    for (test, kind), ent in sorted(STATS.items()):
        vals = ", ".join(f"{k}={v:.3g}" if isinstance(v, float) else f"{k}={v}"
                         for k, v in ent.items())
        lines.append(f"{test} [{kind}]: {vals}")
    return "\n".join(lines)


def score_scale(q, w, rows) -> np.ndarray:
    """A'[p]: the magnitude of the products that reach score[p] through heads whose
    oracle dot product is not clearly negative (see the module docstring)."""
    q = O.to_f64(q)
    w = O.to_f64(w)
    rows = O.to_f64(rows)
    H_i, D_i = q.shape
    dots = q @ rows.T                      # (H_i, n)
    mags = np.abs(q) @ np.abs(rows).T      # (H_i, n)
    live = dots >= -SCORE_RTOL * mags
    return (np.abs(w * O.head_scale(H_i, D_i))[:, None] * np.where(live, mags, 0.0)).sum(axis=0)


def check_scores(gpu, ora, A, rtol=SCORE_RTOL, f32_tol=SCORE_F32, what="scores"):
    gpu = np.asarray(gpu, dtype=np.float64)
    ora = np.asarray(ora, dtype=np.float64)
    A = np.asarray(A, dtype=np.float64)
    masked = ora <= -1e29
    assert np.all(gpu[masked] == np.float64(np.float32(-1e30))), f"{what}: masked entries differ"
    free = ~masked
    err = np.abs(gpu[free] - ora[free])
    o, a = np.abs(ora[free]), A[free]
    bound = rtol * np.maximum(o, a)
    bad = err > bound
    assert not np.any(bad), (f"{what}: {int(bad.sum())} of {bad.size} outside the target "
                             f"tolerance; worst err {err[bad].max():.3e}")
    if err.size:
        with np.errstate(divide="ignore", invalid="ignore"):
            r_a = np.where(a > 0, err / a, np.where(err > 0, np.inf, 0.0))
            big = o > 1e-3 * a
            r_o = float((err[big] / o[big]).max()) if np.any(big) else 0.0
        _record("scores", err_over_A=float(r_a.max()), err_over_o=r_o)
        if f32_tol is not None:
            bad = err > f32_tol * a
            assert not np.any(bad), (
                f"{what}: {int(bad.sum())} of {bad.size} beyond the f32 bound {f32_tol:.2e} A'; "
                f"worst err/A' {float(r_a.max()):.3e}")
        return float(r_a.max())
    return 0.0


def check_selection(gpu_ids, ids, score, A, k, rtol=SCORE_RTOL, what="selection",
                    max_ties=NEAR_TIES_MAX):
    """gpu_ids: the CUDA path's selection (may hold -1 padding).
    ids/score/A: the oracle's candidate universe with f64 scores and error scales.
    Returns the number of ids exempted as near-ties (asserted <= max_ties)."""
    gpu = [int(x) for x in np.asarray(gpu_ids).ravel() if int(x) >= 0]
    assert len(gpu) == len(set(gpu)), f"{what}: duplicate ids"
    ids = np.asarray(ids, dtype=np.int64)
    score = np.asarray(score, dtype=np.float64)
    A = np.asarray(A, dtype=np.float64)
    k = min(k, ids.shape[0])
    assert len(gpu) == k, f"{what}: {len(gpu)} ids, want {k}"
    pos_of = {int(i): n for n, i in enumerate(ids)}
    assert all(g in pos_of for g in gpu), f"{what}: id outside the candidate set"
    ora = O.top_k(score, k, ids)
    if k == 0:
        return 0
    kth = pos_of[int(ora[-1])]
    s_k, A_k = score[kth], A[kth]
    diff = set(gpu) ^ set(int(x) for x in ora)
    for i in diff:
        n = pos_of[i]
        tol = rtol * max(abs(s_k), A_k, A[n])
        assert abs(score[n] - s_k) <= tol, (
            f"{what}: id {i} differs (score {score[n]:.9g}, k-th {s_k:.9g}, tol {tol:.3g})")
    _record("selection", near_ties_max=len(diff), sum_near_ties=len(diff), sum_rows=1)
    assert len(diff) <= max_ties, f"{what}: {len(diff)} near-tie ids exempted (> {max_ties})"
    return len(diff)


def attention_violations(gpu, ora, E, dtype, out_bf16=False):
    """(max abs error, worst err/E, elements beyond the element-wise bound) of one output
    block: eps*E, or eps*E*(1 + u) + u*|o| for a bf16 output."""
    g = np.asarray(O.to_f64(gpu) if out_bf16 else gpu, np.float64)
    o = np.asarray(ora, np.float64)
    E = np.asarray(E, np.float64)
    err = np.abs(g - o)
    eps = ATTN_EPS[dtype]
    bound = eps * E * (1 + OUT_BF16_U) + OUT_BF16_U * np.abs(o) if out_bf16 else eps * E
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(E > 0, err / E, np.where(err > 0, np.inf, 0.0))
    return float(err.max()) if err.size else 0.0, float(r.max()) if r.size else 0.0, \
        int(np.sum(err > bound))


def check_attention(gpu, ora, E, dtype, what="attention", out_bf16=False):
    err, r, n_bad = attention_violations(gpu, ora, E, dtype, out_bf16)
    max_o = float(np.max(np.abs(ora))) if np.size(ora) else 0.0
    _record(f"attention {dtype}" + (" -> bf16 out" if out_bf16 else ""), max_abs_err=err,
            err_over_E=r, max_abs_out=max_o)
    tol = ATTN_TOL[dtype] + (OUT_BF16_U * max_o if out_bf16 else 0.0)
    assert err <= tol, f"{what}: max abs err {err:.3e} > {tol}"
    assert n_bad == 0, (f"{what}: {n_bad} elements beyond the element-wise bound "
                        f"(worst err/E {r:.3e})")
    return err


def check_pooled(gpu, ora, dtype, what="pooled rows"):
    """Compressor output rows ([HiSA issue] "The pooled stream and positions"). The kernel
    evaluates each row in f32 (softmax weights, weighted sum, RMS, rotation of an angle
    reduced modulo 2 pi in f64): error e <= 4e-6 of the row's largest |value|. bf16 rows
    are then rounded to nearest: |g - o| <= 2^-8 |o| + 1.01 e."""
    g = np.asarray(O.to_f64(gpu), np.float64)
    o = np.asarray(ora, np.float64)
    e = 4e-6 * np.max(np.abs(o), axis=-1, keepdims=True)
    tol = (2.0 ** -8 * np.abs(o) + 1.01 * e) if dtype == "bf16" else e
    err = np.abs(g - o)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = float(np.max(np.where(tol > 0, err / tol, np.where(err > 0, np.inf, 0.0))))
    _record(f"pooled {dtype}", err_over_tol=r)
    bad = err > tol
    assert not np.any(bad), f"{what}: {int(bad.sum())} values beyond tolerance (worst {r:.3g} x)"
    return r


# ----------------------------------------------------------------------------
# per-row checks of every stage of one generated problem (numpy in, asserts out)
# ----------------------------------------------------------------------------
def seq(data, b):
    """Sequence b's slices of the packed arrays."""
    k0, k1 = int(data["key_off"][b]), int(data["key_off"][b + 1])
    s = dict(keys=data["keys"][k0:k1], Np=k1 - k0, t0=int(data["t0"][b]))
    if "pooled_kv" in data:
        s["pooled_kv"] = data["pooled_kv"][k0:k1]
        s["local_kv"] = data["local_kv"][b, : int(data["local_len"][b])]
        s["local_pos0"] = int(data["local_pos0"][b])
    return s


def _dtype_name(a):
    return "bf16" if np.asarray(a).dtype == np.uint16 else "f32"


def check_block_means(data, gpu_means, means_off, b_blk):
    for b in range(len(data["Np"])):
        s = seq(data, b)
        rep = O.block_means(s["keys"], b_blk)
        m0 = int(means_off[b])
        g = np.asarray(gpu_means[m0:m0 + rep.shape[0]], dtype=np.float64)
        scale = np.abs(O.to_f64(s["keys"])).max() if s["Np"] else 1.0
        assert np.max(np.abs(g - rep), initial=0.0) <= 1e-6 * scale, f"block means of seq {b}"


def check_coarse(data, b, j, gpu_top_blk, gpu_cscores, b_blk, keep, gpu_means=None):
    """Coarse scores (when given) and the kept block set of row (b, j)."""
    wl = data["wl"]
    s = seq(data, b)
    q, w = data["q_idx"][b, j], data["w"][b, j]
    rep = O.block_means(s["keys"], b_blk)
    V = O.visible_len(s["t0"] + j, wl.r, s["Np"]) if wl.L > 1 else None
    cs, _ = O.hisa_coarse(q, w, rep, min(keep, rep.shape[0]), b_blk, V)
    A = score_scale(q, w, rep)
    if gpu_cscores is not None:
        check_scores(gpu_cscores[: rep.shape[0]], cs, A, what=f"cscore[{b},{j}]")
    return check_selection(gpu_top_blk, np.arange(rep.shape[0]), cs, A, min(keep, rep.shape[0]),
                           what=f"top_blk[{b},{j}]")


def check_fine(data, b, j, gpu_top_blk, gpu_I, gpu_fscores, b_blk, k):
    """Fine stage of row (b, j) re-run by the oracle on the CUDA path's kept blocks."""
    wl = data["wl"]
    s = seq(data, b)
    q, w = data["q_idx"][b, j], data["w"][b, j]
    tb = np.sort(np.asarray(gpu_top_blk, dtype=np.int64))
    V = O.visible_len(s["t0"] + j, wl.r, s["Np"]) if wl.L > 1 else None
    pos, fs, _ = O.hisa_fine(q, w, s["keys"], tb, b_blk, k, V)
    A = score_scale(q, w, np.asarray(s["keys"])[pos])
    if gpu_fscores is not None:
        check_scores(gpu_fscores, fs, A, what=f"fscore[{b},{j}]")
    return check_selection(gpu_I, pos, fs, A, k, what=f"I[{b},{j}]")


def check_flat(data, b, j, gpu_I, k, gpu_scores=None):
    wl = data["wl"]
    s = seq(data, b)
    q, w = data["q_idx"][b, j], data["w"][b, j]
    sc = O.flat_scores(q[None], w[None], s["keys"], s["t0"] + j, wl.r, causal=wl.L > 1)[0]
    A = score_scale(q, w, s["keys"])
    if gpu_scores is not None:
        check_scores(gpu_scores[: s["Np"]], sc, A, what=f"flat score[{b},{j}]")
    return check_selection(gpu_I, np.arange(s["Np"]), sc, A, min(k, s["Np"]),
                           what=f"flat I[{b},{j}]")


def combine_row(data, b, j, I_row, magnitude=False, **kw):
    """The oracle combine of row (b, j) over the given selection (None = dense branch)."""
    wl = data["wl"]
    s = seq(data, b)
    args = dict(window=wl.window, causal=wl.L > 1)
    args.update(kw)
    return O.sparse_combine(data["q_attn"][b, j:j + 1], s["local_kv"], s["local_pos0"],
                            s["pooled_kv"], None if I_row is None else np.asarray(I_row)[None],
                            data["sinks"], s["t0"] + j, wl.r, magnitude=magnitude, **args)[0]


def check_attend(data, b, j, gpu_out, I_row, out_bf16=False):
    """The combine of row (b, j) over the given selection (None = dense branch); gpu_out as
    bf16 bit patterns (uint16) when out_bf16."""
    o = combine_row(data, b, j, I_row)
    E = combine_row(data, b, j, I_row, magnitude=True)
    return check_attention(gpu_out, o, E, _dtype_name(data["pooled_kv"]), what=f"out[{b},{j}]",
                           out_bf16=out_bf16)

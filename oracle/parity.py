"""Comparison rules between the CUDA path and the oracle (test infrastructure only).

Tolerances (the numbers are those fixed for this path; the arithmetic behind them):
  * scores: |g - o| <= 1e-5 * max(|o|, A), A = sum_h |w_h * scale| * sum_d |q_hd row_d|:
    an f32 evaluation of the nested sums is rounded against the magnitude of its terms,
    not against |o|, which can cancel (w has both signs, and a head's dot product can
    sit near zero). Masked entries must be exactly -1e30.
  * selections (unordered sets): equal, except that an id may differ between the two
    sides when its oracle score lies within 1e-5 * max(|s_k|, A_k, A_id) of the k-th
    oracle score s_k (a near-tie that f32 rounding may order either way).
  * attention outputs: max |g - o| <= 1e-2 for bf16 KV, 1e-4 for f32.
"""
from __future__ import annotations

import numpy as np

from . import hisa_oracle as O

SCORE_RTOL = 1e-5
ATTN_TOL = {"bf16": 1e-2, "f32": 1e-4}


def check_scores(gpu, ora, A, rtol=SCORE_RTOL, what="scores"):
    gpu = np.asarray(gpu, dtype=np.float64)
    ora = np.asarray(ora, dtype=np.float64)
    A = np.asarray(A, dtype=np.float64)
    masked = ora <= -1e29
    assert np.all(gpu[masked] == np.float64(np.float32(-1e30))), f"{what}: masked entries differ"
    free = ~masked
    err = np.abs(gpu[free] - ora[free])
    bound = rtol * np.maximum(np.abs(ora[free]), A[free])
    bad = err > bound
    assert not np.any(bad), (f"{what}: {int(bad.sum())} of {bad.size} outside tolerance; worst "
                             f"err {err[bad].max():.3e} vs bound {bound[bad][np.argmax(err[bad])]:.3e}")
    rel = err / np.maximum(bound / rtol, 1e-300)
    return float(rel.max()) if rel.size else 0.0


def check_selection(gpu_ids, ids, score, A, k, rtol=SCORE_RTOL, what="selection"):
    """gpu_ids: the CUDA path's selection (may hold -1 padding).
    ids/score/A: the oracle's candidate universe with f64 scores and error scales.
    Returns the number of ids exempted as near-ties."""
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
    return len(diff)


def check_attention(gpu, ora, dtype, what="attention"):
    err = float(np.max(np.abs(np.asarray(gpu, np.float64) - np.asarray(ora, np.float64))))
    tol = ATTN_TOL[dtype]
    assert err <= tol, f"{what}: max abs err {err:.3e} > {tol}"
    return err


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
    cs = O.combined_scores(q, w, rep)
    if wl.L > 1:
        V = O.visible_len(s["t0"] + j, wl.r, s["Np"])
        cs = np.where(np.arange(rep.shape[0]) * b_blk >= V, O.NEG, cs)
    A = O.error_scale(q, w, rep)
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
    A = O.error_scale(q, w, np.asarray(s["keys"])[pos])
    if gpu_fscores is not None:
        check_scores(gpu_fscores, fs, A, what=f"fscore[{b},{j}]")
    return check_selection(gpu_I, pos, fs, A, k, what=f"I[{b},{j}]")


def check_flat(data, b, j, gpu_I, k, gpu_scores=None):
    wl = data["wl"]
    s = seq(data, b)
    q, w = data["q_idx"][b, j], data["w"][b, j]
    sc = O.flat_scores(q[None], w[None], s["keys"], s["t0"] + j, wl.r, causal=wl.L > 1)[0]
    A = O.error_scale(q, w, s["keys"])
    if gpu_scores is not None:
        check_scores(gpu_scores[: s["Np"]], sc, A, what=f"flat score[{b},{j}]")
    return check_selection(gpu_I, np.arange(s["Np"]), sc, A, min(k, s["Np"]),
                           what=f"flat I[{b},{j}]")


def check_attend(data, b, j, gpu_out, I_row):
    """The combine of row (b, j) over the given selection (None = dense branch)."""
    wl = data["wl"]
    s = seq(data, b)
    o = O.sparse_combine(data["q_attn"][b, j:j + 1], s["local_kv"], s["local_pos0"],
                         s["pooled_kv"], None if I_row is None else np.asarray(I_row)[None],
                         data["sinks"], s["t0"] + j, wl.r, wl.window, causal=wl.L > 1)[0]
    return check_attention(gpu_out, o, _dtype_name(data["pooled_kv"]), what=f"out[{b},{j}]")

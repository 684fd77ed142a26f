"""Plain, slow f64 CPU oracle of the HiSA sparse-attention step.

TEST INFRASTRUCTURE ONLY. Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import or call this module. The CUDA
library never uses it, and this module imports nothing from the CUDA side.

Every function follows the page "feat(deepseek-v4): implement HiSA
hierarchical sparse attention" (cited below as [HiSA issue], with its section)
in the page's order and notation: q, w, pooled, rep, cs/cscore, top_blk, pos,
cand, fs/fscore, sel, I, valid_len, NEG. Arithmetic is numpy float64; bf16
inputs arrive as uint16 bit patterns and are widened exactly. Top-k uses a full
sort instead of argpartition.

Readings where the page leaves a step open (each is also pinned by a test):
  * Top-k is a set (argpartition is unordered, [HiSA issue] "Conventions"). To
    make it unique, equal scores are ordered by ascending absolute id (pooled
    row id, or block id in the coarse stage); -0.0 and +0.0 compare equal.
  * NEG = -1e30 for every selection mask ([HiSA issue] "Flat selection" and
    "HiSA batched path"); the attention re-mask uses -inf.
  * The causal pooled mask is applied when ``causal`` is set; by default that
    is L > 1, since the page skips it for L == 1 ("Flat selection", "HiSA
    decode path") and calls the attention re-mask "prefill only".
  * Local-window visibility: key at absolute position s is visible to the
    query at position t iff 0 <= t - s < window.
  * Head weights arrive raw (weights_proj(x)); the oracle applies
    H_i^-1/2 * D_i^-1/2 once per head ([HiSA issue] "The indexer query and
    per-head weights").
  * An id of -1 in a selection is padding and is skipped by the combine.

Parity status: every function here is pinned by tests/test_oracle_pins.py
(closed forms, brute force on tiny inputs, invariants the page states, and a
textbook softmax formulation of the combine).
"""
from __future__ import annotations

import numpy as np

NEG = -1e30


# ----------------------------------------------------------------------------
# inputs
# ----------------------------------------------------------------------------
def to_f64(a) -> np.ndarray:
    """Widen an input tensor to float64. uint16 arrays are bf16 bit patterns."""
    a = np.asarray(a)
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


# ----------------------------------------------------------------------------
# positions  ([HiSA issue] "The pooled stream and positions")
# ----------------------------------------------------------------------------
def visible_len(t: int, r: int, Np: int) -> int:
    """V(t) = min(Np, floor((t + 1) / r)): the visible pooled prefix of token t."""
    return min(int(Np), (int(t) + 1) // int(r))


# ----------------------------------------------------------------------------
# top-k  ([HiSA issue] "Conventions": argpartition returns an unordered set)
# ----------------------------------------------------------------------------
def top_k(score: np.ndarray, k: int, ids: np.ndarray | None = None) -> np.ndarray:
    """The k entries with the largest score; equal scores by ascending id.

    Returns the selected ids ordered by (score desc, id asc); callers treat the
    result as a set.
    """
    score = np.asarray(score, dtype=np.float64)
    if ids is None:
        ids = np.arange(score.shape[0], dtype=np.int64)
    order = np.lexsort((ids, -score))  # primary: -score ascending; secondary: id ascending
    return ids[order[:k]]


# ----------------------------------------------------------------------------
# head-combined relu scores
# ([HiSA issue] "The indexer query and per-head weights", "Flat selection")
# ----------------------------------------------------------------------------
def head_scale(H_i: int, D_i: int) -> float:
    return H_i ** -0.5 * D_i ** -0.5


def combined_scores(q: np.ndarray, w: np.ndarray, rows: np.ndarray) -> np.ndarray:
    """score[p] = sum_h relu(q_h . rows_p) * scale * w_h * H_i^-1/2, in f64.

    q: (H_i, D_i); w: (H_i,) raw weights; rows: (n, D_i). Returns (n,).
    """
    q = to_f64(q)
    w = to_f64(w)
    rows = to_f64(rows)
    H_i, D_i = q.shape
    s = np.maximum(q @ rows.T, 0.0)            # (H_i, n): relu(sum_d q[h,d] * row[p,d])
    return (w * head_scale(H_i, D_i)) @ s      # sum over h


def error_scale(q: np.ndarray, w: np.ndarray, rows: np.ndarray) -> np.ndarray:
    """A[p] = sum_h |w_h * scale| * sum_d |q_hd * rows_pd|: the magnitude of every
    product that enters score[p], which is what an f32 evaluation of the two nested
    sums is rounded against (a head's dot product can cancel to near zero while its
    terms stay large). Used for tolerances only."""
    q = to_f64(q)
    w = to_f64(w)
    rows = to_f64(rows)
    H_i, D_i = q.shape
    return np.abs(w * head_scale(H_i, D_i)) @ (np.abs(q) @ np.abs(rows).T)


# ----------------------------------------------------------------------------
# flat selection  ([HiSA issue] "Flat selection (baseline path)")
# ----------------------------------------------------------------------------
def flat_scores(q_rows, w_rows, pooled, t0: int, r: int, causal: bool | None = None) -> np.ndarray:
    """score[j, p] for one sequence; NEG where p >= V(t0 + j) when causal.

    q_rows: (L, H_i, D_i); w_rows: (L, H_i); pooled: (Np, D_i). Returns (L, Np).
    """
    q_rows = to_f64(q_rows)
    L = q_rows.shape[0]
    Np = np.asarray(pooled).shape[0]
    if causal is None:
        causal = L > 1
    out = np.empty((L, Np), dtype=np.float64)
    for j in range(L):
        out[j] = combined_scores(q_rows[j], w_rows[j], pooled)
        if causal:
            out[j, visible_len(t0 + j, r, Np):] = NEG
    return out


def flat_top_indices(q_rows, w_rows, pooled, t0: int, r: int, index_topk: int,
                     causal: bool | None = None) -> np.ndarray:
    """I (L, k), k = min(index_topk, Np): flat top-k of the (masked) scores."""
    score = flat_scores(q_rows, w_rows, pooled, t0, r, causal)
    k = min(index_topk, score.shape[1])
    return np.stack([top_k(score[j], k) for j in range(score.shape[0])]) if score.shape[0] else \
        np.zeros((0, k), dtype=np.int64)


# ----------------------------------------------------------------------------
# HiSA  ([HiSA issue] "HiSA decode path", "HiSA batched path")
# ----------------------------------------------------------------------------
def block_means(pooled, b: int) -> np.ndarray:
    """rep[beta] = mean of pooled rows [beta*b, (beta+1)*b); the tail is dropped."""
    pooled = to_f64(pooled)
    nb = pooled.shape[0] // b
    return pooled[: nb * b].reshape(nb, b, pooled.shape[1]).mean(axis=1)


def hisa_coarse(q, w, rep, Kb: int, b: int, valid_len: int | None = None):
    """Coarse stage for one query row: cscore over block means and the top Kb blocks.

    With valid_len (batched path) a block is eligible iff its first row is
    visible: cscore = NEG when beta * b >= valid_len.
    Returns (cscore (nb,), top_blk (Kb,)).
    """
    cscore = combined_scores(q, w, rep)
    if valid_len is not None:
        first_row = np.arange(cscore.shape[0]) * b
        cscore = np.where(first_row >= valid_len, NEG, cscore)
    return cscore, top_k(cscore, Kb)


def hisa_fine(q, w, pooled, top_blk, b: int, k: int, valid_len: int | None = None):
    """Fine stage for one query row: candidate table, exact rescoring, top k.

    pos[c] = top_blk[c // b] * b + c % b; cand = pooled[pos]; with valid_len the
    candidates at pos >= valid_len are NEG. Returns (pos (C,), fscore (C,), I (k,)).
    """
    top_blk = np.asarray(top_blk, dtype=np.int64)
    C = top_blk.shape[0] * b
    c = np.arange(C)
    pos = top_blk[c // b] * b + (c % b)
    cand = np.asarray(pooled)[pos]
    fscore = combined_scores(q, w, cand)
    if valid_len is not None:
        fscore = np.where(pos >= valid_len, NEG, fscore)
    sel_ids = top_k(fscore, k, ids=pos)  # sel mapped through pos: I = pos[sel]
    return pos, fscore, sel_ids


def hisa_select_decode(q, w, pooled, b: int, keep: int, index_topk: int, rep=None) -> dict:
    """HiSA decode path (L == 1): coarse over block means, fine over kept blocks."""
    Np = np.asarray(pooled).shape[0]
    nb = Np // b
    Kb = min(keep, nb)
    k = min(index_topk, Np)
    if rep is None:
        rep = block_means(pooled, b)
    cscore, top_blk = hisa_coarse(q, w, rep, Kb, b)
    pos, fscore, I = hisa_fine(q, w, pooled, top_blk, b, k)
    return dict(rep=rep, cscore=cscore, top_blk=top_blk, pos=pos, fscore=fscore, I=I)


def hisa_select_batched(q_rows, w_rows, pooled, t0: int, r: int, b: int, keep: int,
                        index_topk: int, rep=None) -> dict:
    """HiSA batched path (L > 1): per-row coarse eligibility and fine re-mask.

    The page tiles the fine stage over query chunks of 512 rows to bound a
    gather's memory; the result does not depend on the chunking, so the oracle
    runs one row at a time.
    """
    Np = np.asarray(pooled).shape[0]
    nb = Np // b
    Kb = min(keep, nb)
    k = min(index_topk, Np)
    if rep is None:
        rep = block_means(pooled, b)
    L = np.asarray(q_rows).shape[0]
    valid_len = np.array([visible_len(t0 + j, r, Np) for j in range(L)], dtype=np.int64)
    top_blk = np.zeros((L, Kb), dtype=np.int64)
    cscore = np.zeros((L, nb))
    fscore = np.zeros((L, Kb * b))
    pos = np.zeros((L, Kb * b), dtype=np.int64)
    I = np.zeros((L, k), dtype=np.int64)
    for j in range(L):
        cscore[j], top_blk[j] = hisa_coarse(q_rows[j], w_rows[j], rep, Kb, b, valid_len[j])
        pos[j], fscore[j], I[j] = hisa_fine(q_rows[j], w_rows[j], pooled, top_blk[j], b, k,
                                            valid_len[j])
    return dict(rep=rep, valid_len=valid_len, cscore=cscore, top_blk=top_blk, pos=pos,
                fscore=fscore, I=I)


# ----------------------------------------------------------------------------
# gates and thresholds
# ([HiSA issue] "HiSA decode path", "HiSA batched path", "Engagement thresholds",
#  "Consuming the selection: sparse combine")
# ----------------------------------------------------------------------------
def hisa_gate(L: int, Np: int, index_block: int, index_keep: int, index_topk: int) -> bool:
    """Both HiSA gates: index_block > 0, Np >= b*keep, b*keep >= k (L picks the variant)."""
    b, keep = index_block, index_keep
    return L >= 1 and b > 0 and Np >= b * keep and b * keep >= index_topk


def attention_branch(Np: int, index_topk: int) -> str:
    """Three-way branch on the attention-side pooled length."""
    if Np == 0:
        return "local"
    if Np <= index_topk:
        return "dense"
    return "sparse"


def selection_path(L: int, Np: int, index_block: int, index_keep: int, index_topk: int) -> str:
    """Which selector runs: 'none' (dense branch), 'hisa_decode', 'hisa_batched' or 'flat'."""
    if attention_branch(Np, index_topk) != "sparse":
        return "none"
    if hisa_gate(L, Np, index_block, index_keep, index_topk):
        return "hisa_decode" if L == 1 else "hisa_batched"
    return "flat"


# ----------------------------------------------------------------------------
# sparse combine  ([HiSA issue] "Consuming the selection: sparse combine")
# ----------------------------------------------------------------------------
def _logsumexp(x: np.ndarray) -> np.ndarray:
    m = np.max(x, axis=-1, keepdims=True) if x.shape[-1] else np.full(x.shape[:-1] + (1,), -np.inf)
    safe = np.where(np.isfinite(m), m, 0.0)
    with np.errstate(divide="ignore"):
        out = np.log(np.sum(np.exp(x - safe), axis=-1)) + safe[..., 0]
    return np.where(np.isfinite(m[..., 0]), out, -np.inf)


def _logaddexp(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    return np.logaddexp(a, b)


def sparse_combine(q_rows, local_kv, local_pos0: int, pooled_kv, I, sinks, t0: int, r: int,
                   window: int, scale: float | None = None, causal: bool | None = None,
                   return_lse: bool = False):
    """One split softmax over the local stream, the gathered pooled rows and the sink.

    q_rows: (L, H, Dh), already roped. local_kv: (W, Dh), row i at absolute
    position local_pos0 + i. pooled_kv: (Np, Dh); K = V in both streams.
    I: (L, k) pooled ids or None for the dense branch (all Np rows). sinks: (H,).
    Returns out (L, H, Dh) [and the normaliser n (L, H)].
    """
    q_rows = to_f64(q_rows)
    local_kv = to_f64(local_kv)
    pooled_kv = to_f64(pooled_kv)
    sinks = to_f64(sinks)
    L, H, Dh = q_rows.shape
    Np = pooled_kv.shape[0]
    if scale is None:
        scale = Dh ** -0.5
    if causal is None:
        causal = L > 1
    W = local_kv.shape[0]
    out = np.zeros((L, H, Dh))
    lse = np.zeros((L, H))
    s_pos = local_pos0 + np.arange(W)
    for j in range(L):
        t = t0 + j
        q_s = q_rows[j] * scale                                    # (H, Dh)
        # local stream with the sliding-window causal mask
        local_scores = q_s @ local_kv.T                            # (H, W)
        local_vis = (t - s_pos >= 0) & (t - s_pos < window)
        local_scores = np.where(local_vis[None, :], local_scores, -np.inf)
        # gathered pooled rows P = pooled_kv[I]
        ids = np.arange(Np) if I is None else np.asarray(I[j], dtype=np.int64)
        if np.any(ids >= Np):
            raise ValueError("selected id out of range")
        present = ids >= 0
        P = pooled_kv[np.where(present, ids, 0)] if Np else np.zeros((ids.shape[0], Dh))
        pooled_scores = q_s @ P.T                                  # (H, k)
        vis = present.copy()
        if causal:
            vis &= ids < visible_len(t, r, Np)                     # re-mask invisible rows
        pooled_scores = np.where(vis[None, :], pooled_scores, -np.inf)
        n = _logaddexp(_logsumexp(local_scores), _logsumexp(pooled_scores))
        n = _logaddexp(n, sinks)                                   # the sink joins the normaliser
        with np.errstate(invalid="ignore"):
            w_local = np.exp(local_scores - n[:, None])
            w_pooled = np.exp(pooled_scores - n[:, None])
        w_local = np.where(np.isfinite(local_scores), w_local, 0.0)
        w_pooled = np.where(np.isfinite(pooled_scores), w_pooled, 0.0)
        out[j] = w_local @ local_kv + w_pooled @ P                 # the sink adds no value
        lse[j] = n
    return (out, lse) if return_lse else out


def dense_combine(q_rows, local_kv, local_pos0, pooled_kv, sinks, t0, r, window, scale=None,
                  causal=None, return_lse=False):
    """Branch 2 of the three-way branch: local + all pooled rows (no selection)."""
    return sparse_combine(q_rows, local_kv, local_pos0, pooled_kv, None, sinks, t0, r, window,
                          scale, causal, return_lse)

"""Plain, slow f64 CPU oracle of the HiSA sparse-attention step.

TEST INFRASTRUCTURE ONLY. Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import or call this module. The CUDA
library never uses it, and this module imports nothing from the CUDA side.

Every function follows the page "feat(deepseek-v4): implement HiSA
hierarchical sparse attention" (cited below as [HiSA issue], with its section)
in the page's order and notation: q, w, pooled, rep, cscore, top_blk, pos,
fscore, I, valid_len, NEG. Arithmetic is numpy float64; bf16
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
# the indexer's compressor  ([HiSA issue] "The pooled stream and positions",
# "Configuration": compressor.{wkv, wgate, ape, norm}, compress_rope_theta,
# qk_rope_head_dim)
# ----------------------------------------------------------------------------
ROPE_THETA = 160000.0
RMS_EPS = 1e-6


def rms_norm(x, weight, eps: float = RMS_EPS) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * weight over the last axis."""
    x = to_f64(x)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * to_f64(weight)


def rope_interleaved(x, pos, theta: float = ROPE_THETA, rope_dims: int = 64) -> np.ndarray:
    """Rotate the last rope_dims dims of x (pairs (2m, 2m+1)) by the angles pos * f_i,
    f_i = theta^(-2i / rope_dims) for the i-th rotated pair; the leading dims pass
    through. x: (..., D); pos: an integer or an array broadcastable to x[..., 0]."""
    x = to_f64(x).copy()
    D = x.shape[-1]
    first = (D - rope_dims) // 2                 # index of the first rotated pair
    pos = np.asarray(pos, dtype=np.float64)[..., None]
    for i in range(rope_dims // 2):
        m = first + i
        ang = pos[..., 0] * theta ** (-2.0 * i / rope_dims)
        c, s = np.cos(ang), np.sin(ang)
        a, b = x[..., 2 * m].copy(), x[..., 2 * m + 1].copy()
        x[..., 2 * m] = a * c - b * s
        x[..., 2 * m + 1] = a * s + b * c
    return x


def compress_rows(kv, gate, ape, norm_w, p_rows, r: int, tok0: int = 0, overlap: bool = True,
                  theta: float = ROPE_THETA, rope_dims: int = 64, eps: float = RMS_EPS):
    """Pooled indexer keys p in p_rows from the projected token rows of one sequence.

    kv, gate: (T, 2 D) = wkv(x), wgate(x) of tokens tok0 .. tok0 + T - 1 (absolute
    positions). ape: (r, 2 D), added to the gate logit of the token at offset i of its
    window. Pooled row p is anchored at the window [p r, p r + r - 1]; with the overlap
    variant it also draws on the previous window [(p - 1) r, p r - 1]: channels D .. 2D - 1
    of the current window's tokens and channels 0 .. D - 1 of the previous window's
    tokens, all 2r of them weighted by one softmax over their gate logits per output dim
    (p = 0 has no previous window: r entries). Without overlap (2 D = the head dim) a
    softmax over the current window's r tokens per dim. Then RMSNorm with norm_w and the
    interleaved RoPE of the last rope_dims dims at position p r. Returns (len(p_rows), D).
    """
    kv, gate, ape = to_f64(kv), to_f64(gate), to_f64(ape)
    C = kv.shape[1]
    D = C // 2 if overlap else C
    out = np.zeros((len(p_rows), D))
    for n, p in enumerate(p_rows):
        vals, logits = [], []
        if overlap and p > 0:
            for i in range(r):
                t = (p - 1) * r + i - tok0
                vals.append(kv[t, :D])
                logits.append(gate[t, :D] + ape[i, :D])
        for i in range(r):
            t = p * r + i - tok0
            vals.append(kv[t, D:] if overlap else kv[t])
            logits.append(gate[t, D:] + ape[i, D:] if overlap else gate[t] + ape[i])
        vals, logits = np.array(vals), np.array(logits)          # (entries, D)
        wts = np.exp(logits - logits.max(axis=0))
        wts /= wts.sum(axis=0)
        out[n] = (wts * vals).sum(axis=0)
    out = rms_norm(out, norm_w, eps)
    return rope_interleaved(out, np.asarray(p_rows) * r, theta, rope_dims)


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
    """Coarse stage for one query row: block-level scores and the Kb best blocks.

    Each block is scored through its mean row exactly as a pooled row is scored.
    With valid_len (batched path) a block whose first pooled row is not visible
    cannot be kept: its score is NEG. Returns (cscore (nb,), top_blk (Kb,)).
    """
    cscore = combined_scores(q, w, rep)
    if valid_len is not None:
        for beta in range(cscore.shape[0]):
            if beta * b >= valid_len:
                cscore[beta] = NEG
    return cscore, top_k(cscore, Kb)


def hisa_fine(q, w, pooled, top_blk, b: int, k: int, valid_len: int | None = None):
    """Fine stage for one query row: every pooled row of the kept blocks is scored
    again exactly, and the k best rows are kept.

    The candidates are the b rows of each kept block, block after block in the
    order given. With valid_len, candidates at or past valid_len score NEG.
    Returns (pos (C,) candidate pooled ids, fscore (C,), I (k,) selected ids).
    """
    blocks = [int(beta) for beta in np.asarray(top_blk).ravel()]
    pos = np.array([beta * b + i for beta in blocks for i in range(b)], dtype=np.int64)
    fscore = combined_scores(q, w, np.asarray(pooled)[pos]) if pos.size else np.zeros(0)
    if valid_len is not None:
        fscore[pos >= valid_len] = NEG
    return pos, fscore, top_k(fscore, k, ids=pos)


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
                   return_lse: bool = False, magnitude: bool = False):
    """One split softmax over the local stream, the gathered pooled rows and the sink.

    q_rows: (L, H, Dh), already roped. local_kv: (W, Dh), row i at absolute
    position local_pos0 + i. pooled_kv: (Np, Dh); K = V in both streams.
    I: (L, k) pooled ids or None for the dense branch (all Np rows). sinks: (H,).
    Returns out (L, H, Dh) [and the normaliser n (L, H)].

    magnitude=True returns instead E = sum_j weight_j * |v_j| (the same softmax
    weights applied to the absolute values): the scale against which a rounding
    of the weights perturbs each output element (used for tolerances only).
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
        if magnitude:
            out[j] = w_local @ np.abs(local_kv) + w_pooled @ np.abs(P)
        else:
            out[j] = w_local @ local_kv + w_pooled @ P             # the sink adds no value
        lse[j] = n
    return (out, lse) if return_lse else out


def dense_combine(q_rows, local_kv, local_pos0, pooled_kv, sinks, t0, r, window, scale=None,
                  causal=None, return_lse=False):
    """Branch 2 of the three-way branch: local + all pooled rows (no selection)."""
    return sparse_combine(q_rows, local_kv, local_pos0, pooled_kv, None, sinks, t0, r, window,
                          scale, causal, return_lse)

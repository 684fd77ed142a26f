"""Seeded synthetic inputs for the HiSA sparse-attention step.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic. Both the CUDA path (tests, bench) and the CPU oracle
(tests only) consume the arrays it returns.

Workloads follow the shapes of the DeepSeek-V4-Flash ratio-4 layers described
on the page "feat(deepseek-v4): implement HiSA hierarchical sparse attention"
(sections "Configuration" and "Consuming the selection: sparse combine"):

  tiny_decode      B=1  L=1    H_i=4  D_i=32  Np=512     b=16 keep=4  k=32  H=8  Dh=64  W=16  all f32
  v4flash_decode   B=1  L=1    H_i=64 D_i=128 Np=32768   b=64 keep=16 k=512 H=64 Dh=512 W=128
  ragged_decode    B=32 L=1    as v4flash, Np_b ~ U[4096, 65536] per sequence
  prefill          B=1  L=4096 as v4flash, t0=61440, Np=16384, indexer q and keys bf16
  long_context     B=1  L=1    H_i=64 D_i=128 Np=262144, 1% of keys planted +3 sigma along q

Draw order per workload (numpy default_rng(seed)): [Np_b for ragged], indexer q,
head weights w, indexer keys, [plant positions], attention q, local KV, pooled
KV, sinks. Normal draws are f32; tensors stored as bf16 are rounded to nearest
even and kept as raw uint16 bit patterns.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

_CHUNK = 1 << 24  # values per draw, bounds host memory for the large caches


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    B: int
    L: int
    r: int
    H_i: int
    D_i: int
    index_block: int
    index_keep: int
    index_topk: int
    H: int
    Dh: int
    window: int
    q_idx_dtype: str  # "f32" | "bf16"
    key_dtype: str
    kv_dtype: str
    Np: tuple | None = None      # fixed pooled rows per sequence (None: ragged draw)
    Np_range: tuple | None = None
    t0: int | None = None        # None: decode position 4*Np_b - 1 per sequence
    local_prefix: int = 0        # cached local rows before t0 (prefill)
    plant_frac: float = 0.0
    with_attention: bool = True
    kv_std: float | None = None  # local / pooled KV std (None: Dh^-1/2)
    q_attn_std: float = 1.0      # attention q std
    sink_mean: float = 0.0       # sinks ~ N(sink_mean, 1)

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "tiny_decode": Workload(
        "tiny_decode", 0, B=1, L=1, r=4, H_i=4, D_i=32, index_block=16, index_keep=4,
        index_topk=32, H=8, Dh=64, window=16, q_idx_dtype="f32", key_dtype="f32",
        kv_dtype="f32", Np=(512,), t0=2047),
    "v4flash_decode": Workload(
        "v4flash_decode", 1, B=1, L=1, r=4, H_i=64, D_i=128, index_block=64, index_keep=16,
        index_topk=512, H=64, Dh=512, window=128, q_idx_dtype="f32", key_dtype="bf16",
        kv_dtype="bf16", Np=(32768,)),
    "ragged_decode": Workload(
        "ragged_decode", 2, B=32, L=1, r=4, H_i=64, D_i=128, index_block=64, index_keep=16,
        index_topk=512, H=64, Dh=512, window=128, q_idx_dtype="f32", key_dtype="bf16",
        kv_dtype="bf16", Np_range=(4096, 65536)),
    "prefill": Workload(
        "prefill", 3, B=1, L=4096, r=4, H_i=64, D_i=128, index_block=64, index_keep=16,
        index_topk=512, H=64, Dh=512, window=128, q_idx_dtype="bf16", key_dtype="bf16",
        kv_dtype="bf16", Np=(16384,), t0=61440, local_prefix=128),
    "long_context": Workload(
        "long_context", 4, B=1, L=1, r=4, H_i=64, D_i=128, index_block=64, index_keep=16,
        index_topk=512, H=64, Dh=512, window=128, q_idx_dtype="f32", key_dtype="bf16",
        kv_dtype="bf16", Np=(262144,), plant_frac=0.01, with_attention=False),
}


def peaked(wl: Workload) -> Workload:
    """The same workload with attention inputs drawn so that a wrong combine is visible
    at bf16 precision: KV ~ N(0, 1) (outputs of order one), q ~ N(0, 9) (logits of std 3,
    so a few rows dominate each head's softmax) and sinks ~ N(9, 1), about the largest
    logit of 640 rows, so each sink holds a sizeable share of its head's normaliser.
    The indexer inputs are the same draws as the plain workload's."""
    return wl.replace(kv_std=1.0, q_attn_std=3.0, sink_mean=9.0)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round f32 to bf16 (nearest, ties to even); returns the uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    return ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)


def _normal(rng, shape, dtype: str, std: float = 1.0, mean: float = 0.0) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.uint16 if dtype == "bf16" else np.float32)
    s = np.float32(std)
    for lo in range(0, n, _CHUNK):
        hi = min(n, lo + _CHUNK)
        z = rng.standard_normal(hi - lo, dtype=np.float32)
        if std != 1.0:
            z *= s
        if mean != 0.0:
            z += np.float32(mean)
        out[lo:hi] = f32_to_bf16_bits(z) if dtype == "bf16" else z
    return out.reshape(shape)


def generate(wl: Workload | str, seed: int | None = None) -> dict:
    """Draw every input of one workload. Returns a dict of numpy arrays + metadata.

    Keys: q_idx (B,L,H_i,D_i), w (B,L,H_i) f32, keys (sum Np_b, D_i), key_off (B+1) i64,
    t0 (B) i32, Np (B) i64; with attention also q_attn (B,L,H,Dh), local_kv (B,Wmax,Dh),
    local_len (B) i32, local_pos0 (B) i32, pooled_kv (sum Np_b, Dh), sinks (H) f32.
    bf16 tensors are uint16 bit patterns.
    """
    if isinstance(wl, str):
        wl = WORKLOADS[wl]
    rng = np.random.default_rng(wl.seed if seed is None else seed)
    if wl.Np is not None:
        Np = np.array(wl.Np if len(wl.Np) == wl.B else wl.Np * wl.B, dtype=np.int64)
    else:
        lo, hi = wl.Np_range
        Np = rng.integers(lo, hi, endpoint=True, size=wl.B).astype(np.int64)
    key_off = np.zeros(wl.B + 1, dtype=np.int64)
    key_off[1:] = np.cumsum(Np)
    total = int(key_off[-1])
    if wl.t0 is not None:
        t0 = np.full(wl.B, wl.t0, dtype=np.int32)
    else:
        t0 = (wl.r * Np - 1).astype(np.int32)

    out = dict(wl=wl, Np=Np, key_off=key_off, t0=t0)
    out["q_idx"] = _normal(rng, (wl.B, wl.L, wl.H_i, wl.D_i), wl.q_idx_dtype)
    out["w"] = _normal(rng, (wl.B, wl.L, wl.H_i), "f32")
    if wl.plant_frac > 0.0:
        # Keys are drawn in f32, a fraction of them shifted by +3 along the unit
        # direction of the weighted query sum, then rounded to bf16.
        keys = _normal(rng, (total, wl.D_i), "f32")
        q = out["q_idx"].astype(np.float32)
        for b in range(wl.B):
            n_plant = int(math.floor(wl.plant_frac * int(Np[b])))
            pos = rng.choice(int(Np[b]), size=n_plant, replace=False)
            u = np.einsum("h,hd->d", out["w"][b, 0].astype(np.float64), q[b, 0].astype(np.float64))
            u = (u / np.linalg.norm(u)).astype(np.float32)
            keys[key_off[b] + pos] += np.float32(3.0) * u
        out["plant_pos"] = pos
        out["keys"] = f32_to_bf16_bits(keys) if wl.key_dtype == "bf16" else keys
    else:
        out["keys"] = _normal(rng, (total, wl.D_i), wl.key_dtype)
    if wl.with_attention:
        W_rows = wl.window + (wl.L - 1) if wl.local_prefix == 0 else wl.local_prefix + wl.L
        W_rows = max(W_rows, 1)
        kv_std = wl.Dh ** -0.5 if wl.kv_std is None else wl.kv_std
        out["q_attn"] = _normal(rng, (wl.B, wl.L, wl.H, wl.Dh), wl.kv_dtype, std=wl.q_attn_std)
        out["local_kv"] = _normal(rng, (wl.B, W_rows, wl.Dh), wl.kv_dtype, std=kv_std)
        if wl.local_prefix:
            pos0 = t0.astype(np.int64) - wl.local_prefix
        else:
            # the last W rows ending at the current token (decode)
            pos0 = t0.astype(np.int64) + (wl.L - 1) - (W_rows - 1)
        out["local_len"] = np.full(wl.B, W_rows, dtype=np.int32)
        out["local_pos0"] = pos0.astype(np.int32)
        out["pooled_kv"] = _normal(rng, (total, wl.Dh), wl.kv_dtype, std=kv_std)
        out["sinks"] = _normal(rng, (wl.H,), "f32", mean=wl.sink_mean)
    return out


def compressor_inputs(seed: int, p_first, n_new, D: int = 128, r: int = 4, overlap: bool = True,
                      key_dtype: str = "bf16", capacity=None) -> dict:
    """Synthetic inputs of the indexer's compressor for B sequences ([HiSA issue]
    "Configuration": compressor.{wkv, wgate, ape, norm}). The projections wkv(x), wgate(x)
    stand for x ~ N(0, 1) through weights ~ N(0, 1 / hidden), so they are drawn directly as
    N(0, 1) rows; ape ~ N(0, 1); norm weight ~ 1 + N(0, 0.1^2). Sequence b holds
    (n_new[b] + 1) * r token rows (the window before its first new pooled row, then the new
    rows' windows) and a pooled key cache of capacity[b] rows (default p_first + n_new),
    whose rows below p_first[b] are drawn as earlier pooled keys ~ N(0, 1).
    Draw order: kv, gate, ape, norm weight, earlier keys."""
    rng = np.random.default_rng(seed)
    p_first = np.asarray(p_first, dtype=np.int32)
    n_new = np.asarray(n_new, dtype=np.int32)
    B = len(p_first)
    C = 2 * D if overlap else D
    T = (n_new.astype(np.int64) + 1) * r
    tok_off = np.zeros(B + 1, dtype=np.int64)
    tok_off[1:] = np.cumsum(T)
    cap = (p_first.astype(np.int64) + n_new) if capacity is None else np.asarray(capacity, np.int64)
    key_off = np.zeros(B + 1, dtype=np.int64)
    key_off[1:] = np.cumsum(cap)
    out = dict(B=B, D=D, r=r, C=C, overlap=overlap, p_first=p_first, n_new=n_new,
               tok_off=tok_off, key_off=key_off)
    out["kv"] = _normal(rng, (int(tok_off[-1]), C), "f32")
    out["gate"] = _normal(rng, (int(tok_off[-1]), C), "f32")
    out["ape"] = _normal(rng, (r, C), "f32")
    out["norm_w"] = _normal(rng, (D,), "f32", std=0.1, mean=1.0)
    keys = _normal(rng, (int(key_off[-1]), D), key_dtype)
    out["keys"] = keys
    return out


def small_workload(**kw) -> Workload:
    """A custom small workload (edge cases, several tiles, ragged tails)."""
    base = dict(name="custom", seed=1234, B=1, L=1, r=4, H_i=4, D_i=32, index_block=16,
                index_keep=4, index_topk=32, H=8, Dh=64, window=16, q_idx_dtype="f32",
                key_dtype="f32", kv_dtype="f32", Np=(512,))
    base.update(kw)
    return Workload(**base)


def generate_device(wl: Workload, device="cuda", seed: int | None = None) -> dict:
    """Like generate(), but drawn on the device with torch's generator (for batches too
    large to draw on the host). Same shapes, distributions and layout; different random
    stream, so results are only comparable with the oracle on host copies of the draws.
    Every sequence has wl.Np[0] pooled rows, or, for a ragged workload (wl.Np None), the
    per-sequence counts generate() draws (the same numpy draw, first from default_rng(seed));
    returns torch tensors (bf16 as torch.bfloat16).
    """
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(wl.seed if seed is None else seed)
    B = wl.B
    if wl.Np is None:
        lo, hi = wl.Np_range
        rng = np.random.default_rng(wl.seed if seed is None else seed)
        npb = rng.integers(lo, hi, endpoint=True, size=B).astype(np.int64)
    else:
        npb = np.full(B, int(wl.Np[0]), dtype=np.int64)
    key_off = np.zeros(B + 1, dtype=np.int64)
    key_off[1:] = np.cumsum(npb)
    t0 = (wl.r * npb - 1).astype(np.int32) if wl.t0 is None else np.full(B, wl.t0, np.int32)
    tdt = {"f32": torch.float32, "bf16": torch.bfloat16}

    def normal(shape, dtype, std=1.0, rows_per_draw=None, mean=0.0):
        out = torch.empty(shape, dtype=tdt[dtype], device=device)
        flat = out.view(shape[0], -1)
        step = rows_per_draw or shape[0]
        for lo in range(0, shape[0], step):
            hi = min(shape[0], lo + step)
            z = torch.randn((hi - lo, flat.shape[1]), generator=g, device=device,
                            dtype=torch.float32)
            if std != 1.0:
                z *= std
            if mean != 0.0:
                z += mean
            flat[lo:hi] = z.to(tdt[dtype])
        return out

    total = int(key_off[-1])
    out = dict(wl=wl, Np=npb, key_off=key_off, t0=t0)
    out["q_idx"] = normal((B, wl.L, wl.H_i, wl.D_i), wl.q_idx_dtype)
    out["w"] = normal((B, wl.L, wl.H_i), "f32")
    out["keys"] = normal((total, wl.D_i), wl.key_dtype, rows_per_draw=1 << 20)
    if wl.with_attention:
        W_rows = wl.window + (wl.L - 1) if wl.local_prefix == 0 else wl.local_prefix + wl.L
        kv_std = wl.Dh ** -0.5 if wl.kv_std is None else wl.kv_std
        out["q_attn"] = normal((B, wl.L, wl.H, wl.Dh), wl.kv_dtype, std=wl.q_attn_std)
        out["local_kv"] = normal((B, W_rows, wl.Dh), wl.kv_dtype, std=kv_std)
        out["local_len"] = np.full(B, W_rows, dtype=np.int32)
        if wl.local_prefix:
            pos0 = t0.astype(np.int64) - wl.local_prefix
        else:
            pos0 = t0.astype(np.int64) + (wl.L - 1) - (W_rows - 1)
        out["local_pos0"] = pos0.astype(np.int32)
        out["pooled_kv"] = normal((total, wl.Dh), wl.kv_dtype, std=kv_std,
                                  rows_per_draw=1 << 17)
        out["sinks"] = normal((wl.H,), "f32", mean=wl.sink_mean)
    return out

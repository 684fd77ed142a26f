"""Device-resident state of one HiSA problem and the calls of the step, in order.

Marshalling only: torch allocates the tensors and owns the stream; every stage is
one libhisa entry point (include/hisa.h). Stages follow the page "feat(deepseek-v4):
implement HiSA hierarchical sparse attention": block means -> coarse filter ->
fine top-k (or the flat top-k) -> sparse combine.
"""
from __future__ import annotations

import numpy as np

from . import binding as hb


def _i64(a, device):
    import torch
    return torch.as_tensor(np.asarray(a, dtype=np.int64), device=device)


def _i32(a, device):
    import torch
    if isinstance(a, torch.Tensor):                  # no copy when it already is (graph capture)
        return a.to(device=device, dtype=torch.int32)
    return torch.as_tensor(np.asarray(a, dtype=np.int32), device=device)


class Problem:
    """One batch of B sequences x L query rows, resident in device memory.

    `data` is the dict returned by inputs.generate (numpy arrays; uint16 = bf16 bits).
    """

    def __init__(self, data: dict, device="cuda", index_keep: int | None = None, out_dtype="f32"):
        import torch
        wl = data["wl"]
        self.wl = wl
        self.device = device
        self.B, self.L = wl.B, wl.L
        self.b = wl.index_block
        self.keep = wl.index_keep if index_keep is None else index_keep
        self.k = wl.index_topk
        Np = np.asarray(data["Np"], dtype=np.int64)
        self.Np = Np
        self.Np_max = int(Np.max()) if Np.size else 0
        dev = device
        self.q_idx = hb.to_device(data["q_idx"], dev)
        self.w = hb.to_device(data["w"], dev)
        self.keys = hb.to_device(data["keys"], dev)
        self.key_off = _i64(data["key_off"], dev)
        self.t0 = _i32(data["t0"], dev)
        self.idesc = hb.IndexDesc(
            B=wl.B, L=wl.L, H_i=wl.H_i, D_i=wl.D_i, r=wl.r, index_topk=wl.index_topk,
            index_block=self.b, index_keep=self.keep, Np_max=self.Np_max,
            keys_rows=int(self.keys.shape[0]), means_rows=0,
            q_dtype=hb.dtype_code(self.q_idx), k_dtype=hb.dtype_code(self.keys))
        nb = Np // self.b if self.b > 0 else np.zeros_like(Np)
        self.nb = nb
        means_off = np.zeros(wl.B + 1, dtype=np.int64)
        means_off[1:] = np.cumsum(nb)
        self.means_off = _i64(means_off, dev)
        self.means = torch.zeros((max(int(means_off[-1]), 1), wl.D_i), dtype=torch.float32,
                                 device=dev)
        self.idesc.means_rows = int(self.means.shape[0])
        rows = wl.B * wl.L
        self.top_blk = torch.full((rows, max(self.keep, 1)), -7, dtype=torch.int32, device=dev)
        self.I = torch.full((rows, self.k), -7, dtype=torch.int32, device=dev)
        ops = [hb.OP_INDEX_SCORES, hb.OP_BLOCK_MEANS, hb.OP_FLAT_TOPK]
        if self.b > 0 and self.keep > 0 and self.b * self.keep >= self.k:
            ops += [hb.OP_BLOCK_FILTER, hb.OP_SELECT_TOPK]
        need = max(hb.workspace_bytes(op, self.idesc) for op in ops)
        self.has_attention = "q_attn" in data
        if self.has_attention:
            self.q_attn = hb.to_device(data["q_attn"], dev)
            self.local_kv = hb.to_device(data["local_kv"], dev)
            self.local_len = _i32(data["local_len"], dev)
            self.local_pos0 = _i32(data["local_pos0"], dev)
            self.pooled_kv = hb.to_device(data["pooled_kv"], dev)
            self.sinks = hb.to_device(data["sinks"], dev)
            self.adesc = hb.AttnDesc(
                B=wl.B, L=wl.L, H=wl.H, Dh=wl.Dh, window=wl.window,
                W_max=int(data["local_kv"].shape[1]), r=wl.r, k=self.k, Np_max=self.Np_max,
                kv_rows=int(self.pooled_kv.shape[0]), scale=0.0, q_dtype=hb.dtype_code(self.q_attn),
                kv_dtype=hb.dtype_code(self.pooled_kv),
                out_dtype=hb.HISA_BF16 if out_dtype == "bf16" else hb.HISA_F32)
            self.out = torch.empty((rows, wl.H, wl.Dh), device=dev,
                                   dtype=torch.bfloat16 if out_dtype == "bf16" else torch.float32)
            need = max(need, hb.workspace_bytes(hb.OP_SPARSE_ATTEND, self.adesc))
        if need == 0:
            raise ValueError("descriptor rejected by hisa_workspace_bytes")
        self.ws_bytes = need
        self.ws = hb.alloc_workspace(need, dev)
        # the same descriptors with HISA_FLAG_CHAINED: for calls that directly follow the
        # previous libhisa call of the step on the stream
        self.idesc_chained = hb.IndexDesc.from_buffer_copy(self.idesc)
        self.idesc_chained.flags = hb.FLAG_CHAINED
        if self.has_attention:
            self.adesc_chained = hb.AttnDesc.from_buffer_copy(self.adesc)
            self.adesc_chained.flags = hb.FLAG_CHAINED

    def with_out(self, out_dtype: str):
        """The same problem (inputs, caches, selections, workspace) with the combine writing
        an output of another dtype ("f32" or "bf16") into a buffer of its own."""
        import copy
        import torch
        c = copy.copy(self)
        code = hb.HISA_BF16 if out_dtype == "bf16" else hb.HISA_F32
        c.adesc = hb.AttnDesc.from_buffer_copy(self.adesc)
        c.adesc.out_dtype = code
        c.adesc_chained = hb.AttnDesc.from_buffer_copy(self.adesc_chained)
        c.adesc_chained.out_dtype = code
        c.out = torch.empty(self.out.shape, device=self.out.device,
                            dtype=torch.bfloat16 if out_dtype == "bf16" else torch.float32)
        return c

    def io_clone(self):
        """A second set of the per-step buffers (query inputs, selections, output, workspace)
        sharing this problem's keys, block-mean cache and KV, so that one step's inputs can be
        copied in (or its results copied out) while another step computes."""
        import copy
        import torch
        c = copy.copy(self)
        c.q_idx = self.q_idx.clone()
        c.w = self.w.clone()
        c.top_blk = torch.empty_like(self.top_blk)
        c.I = torch.empty_like(self.I)
        if self.has_attention:
            c.q_attn = self.q_attn.clone()
            c.out = torch.empty_like(self.out)
        c.ws = hb.alloc_workspace(self.ws_bytes, self.device)
        return c

    # ---- stages -------------------------------------------------------------
    def block_means(self, first_block=None, stream=None):
        fb = None if first_block is None else _i32(first_block, self.device)
        hb.block_means(self.idesc, self.keys, self.key_off, self.means_off, fb, self.means,
                       self.ws, stream)

    def block_filter(self, cscores=None, stream=None):
        ld = 0 if cscores is None else cscores.shape[1]
        hb.block_filter(self.idesc, self.q_idx, self.w, self.means, self.means_off, self.key_off,
                        self.t0, self.top_blk, self.ws, cscores, ld, stream)

    def block_filter_append(self, first_block=None, cscores=None, stream=None):
        """Append the means of blocks [first_block[b], nb_b), then the coarse filter."""
        ld = 0 if cscores is None else cscores.shape[1]
        hb.block_filter_append(self.idesc, self.q_idx, self.w, self.keys, self.key_off, self.means,
                               self.means_off, first_block, self.t0, self.top_blk, self.ws,
                               cscores, ld, stream)

    def select_topk(self, fscores=None, top_blk=None, stream=None, chained=False):
        tb = self.top_blk if top_blk is None else top_blk
        d = self.idesc_chained if chained else self.idesc
        hb.select_topk(d, self.q_idx, self.w, self.keys, self.key_off, self.t0, tb, self.I,
                       self.ws, fscores, stream)

    def flat_topk(self, I=None, stream=None):
        hb.flat_topk(self.idesc, self.q_idx, self.w, self.keys, self.key_off, self.t0,
                     self.I if I is None else I, self.ws, stream)

    def index_scores(self, scores, stream=None):
        hb.index_scores(self.idesc, self.q_idx, self.w, self.keys, self.key_off, self.t0, scores,
                        scores.shape[1], self.ws, stream)

    def attend(self, I="selected", out=None, stream=None, chained=False):
        """I: 'selected' (self.I), None (dense branch over all pooled rows) or a tensor."""
        sel = self.I if isinstance(I, str) else I
        d = self.adesc_chained if chained else self.adesc
        hb.sparse_attend(d, self.q_attn, self.local_kv, self.local_len, self.local_pos0,
                         self.pooled_kv, self.key_off, sel, self.sinks, self.t0,
                         self.out if out is None else out, self.ws, stream)

    def hisa_step(self, first_block=None, stream=None):
        """The HiSA step: newest block means, coarse filter, fine top-k, sparse combine; the
        fine top-k and the combine are chained to the call before them."""
        if first_block is not None:
            self.block_means(first_block, stream)
        self.block_filter(stream=stream)
        self.select_topk(stream=stream, chained=True)
        if self.has_attention:
            self.attend(stream=stream, chained=True)

    def status(self, stream=None) -> int:
        return hb.device_status(self.ws, stream)

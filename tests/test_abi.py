"""The C ABI without a GPU: the library loads, exports every function include/hisa.h
declares, the ctypes binding matches the prototypes and struct layouts, and host-side
validation rejects bad arguments before anything reaches the device."""
import ctypes
import os
import re
import shutil
import subprocess
import tempfile

import pytest

from deepseek_sparse_attention_hisa_gb300 import binding as hb
from deepseek_sparse_attention_hisa_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "hisa.h")


@pytest.fixture(scope="module")
def lib():
    build.build_library()
    return hb.lib()


def prototypes():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    out = {}
    for m in re.finditer(r"HISA_API\s+([\w\s\*]+?)\b(hisa_\w+)\s*\(([^)]*)\)\s*;", text):
        params = [p.strip() for p in m.group(3).split(",") if p.strip()]
        out[m.group(2)] = (m.group(1).strip(), params)
    return out


def _ctype_of(param):
    if "*" in param or "hisa_stream_t" in param:
        return "ptr"
    if "int64_t" in param:
        return "i64"
    if "int32_t" in param:
        return "i32"
    if "size_t" in param:
        return "size"
    raise AssertionError(param)


def _kind(ct):
    if ct is ctypes.c_void_p or (isinstance(ct, type) and issubclass(ct, ctypes._Pointer)):
        return "ptr"
    return {ctypes.c_int64: "i64", ctypes.c_int32: "i32", ctypes.c_size_t: "size"}[ct]


def test_header_declares_the_step():
    names = set(prototypes())
    assert {"hisa_index_scores", "hisa_block_means", "hisa_block_filter", "hisa_select_topk",
            "hisa_flat_topk", "hisa_sparse_attend", "hisa_workspace_bytes",
            "hisa_workspace_init", "hisa_device_status", "hisa_status_string"} <= names


def test_every_declared_symbol_is_exported(lib):
    for name in prototypes():
        assert hasattr(lib, name), name


def test_binding_signatures_match_header(lib):
    protos = prototypes()
    assert set(hb._SIG) == set(protos)
    for name, (_, params) in protos.items():
        _, args = hb._SIG[name]
        assert [_ctype_of(p) for p in params] == [_kind(a) for a in args], name


def test_struct_layout_matches_c():
    gcc = shutil.which("gcc") or shutil.which("cc")
    if gcc is None:
        pytest.skip("no C compiler")
    src = r"""
#include <stdio.h>
#include <stddef.h>
#include "hisa.h"
int main(void) {
  printf("%zu %zu %zu %zu %zu %zu %zu\n", sizeof(hisa_index_desc), offsetof(hisa_index_desc, Np_max),
         offsetof(hisa_index_desc, keys_rows), offsetof(hisa_index_desc, means_rows),
         offsetof(hisa_index_desc, q_dtype), offsetof(hisa_index_desc, k_dtype),
         offsetof(hisa_index_desc, flags));
  printf("%zu %zu %zu %zu %zu %zu %zu %zu\n", sizeof(hisa_attn_desc), offsetof(hisa_attn_desc, Np_max),
         offsetof(hisa_attn_desc, kv_rows), offsetof(hisa_attn_desc, scale),
         offsetof(hisa_attn_desc, q_dtype), offsetof(hisa_attn_desc, kv_dtype),
         offsetof(hisa_attn_desc, flags), offsetof(hisa_attn_desc, out_dtype));
  printf("%zu %zu %zu %zu %zu %zu %zu\n", sizeof(hisa_compress_desc),
         offsetof(hisa_compress_desc, rope_theta), offsetof(hisa_compress_desc, eps),
         offsetof(hisa_compress_desc, tok_rows), offsetof(hisa_compress_desc, keys_rows),
         offsetof(hisa_compress_desc, means_rows), offsetof(hisa_compress_desc, flags));
  return 0;
}
"""
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "probe.c")
        exe = os.path.join(d, "probe")
        open(c, "w").write(src)
        subprocess.run([gcc, "-I", os.path.join(ROOT, "include"), c, "-o", exe], check=True)
        lines = subprocess.run([exe], capture_output=True, text=True, check=True).stdout.split("\n")
    i = [int(x) for x in lines[0].split()]
    a = [int(x) for x in lines[1].split()]
    c = [int(x) for x in lines[2].split()]
    C = hb.CompressDesc
    assert c == [ctypes.sizeof(C), C.rope_theta.offset, C.eps.offset, C.tok_rows.offset,
                 C.keys_rows.offset, C.means_rows.offset, C.flags.offset]
    assert i == [ctypes.sizeof(hb.IndexDesc), hb.IndexDesc.Np_max.offset,
                 hb.IndexDesc.keys_rows.offset, hb.IndexDesc.means_rows.offset,
                 hb.IndexDesc.q_dtype.offset, hb.IndexDesc.k_dtype.offset, hb.IndexDesc.flags.offset]
    assert a == [ctypes.sizeof(hb.AttnDesc), hb.AttnDesc.Np_max.offset, hb.AttnDesc.kv_rows.offset,
                 hb.AttnDesc.scale.offset, hb.AttnDesc.q_dtype.offset, hb.AttnDesc.kv_dtype.offset,
                 hb.AttnDesc.flags.offset, hb.AttnDesc.out_dtype.offset]


def v4_index_desc(**kw):
    d = dict(B=1, L=1, H_i=64, D_i=128, r=4, index_topk=512, index_block=64, index_keep=16,
             Np_max=32768, keys_rows=32768, means_rows=512, q_dtype=hb.HISA_F32,
             k_dtype=hb.HISA_BF16)
    d.update(kw)
    return hb.IndexDesc(**d)


def v4_attn_desc(**kw):
    d = dict(B=1, L=1, H=64, Dh=512, window=128, W_max=128, r=4, k=512, Np_max=32768,
             kv_rows=32768, scale=0.0,
             q_dtype=hb.HISA_BF16, kv_dtype=hb.HISA_BF16)
    d.update(kw)
    return hb.AttnDesc(**d)


def test_workspace_bytes_host_arithmetic(lib):
    assert hb.workspace_bytes(hb.OP_INDEX_SCORES, v4_index_desc()) == 256
    assert hb.workspace_bytes(hb.OP_FLAT_TOPK, v4_index_desc(Np_max=262144)) == 256 + 262144 * 4
    assert hb.workspace_bytes(hb.OP_BLOCK_FILTER, v4_index_desc()) == 256 + 512 * 4
    assert hb.workspace_bytes(hb.OP_SELECT_TOPK, v4_index_desc(B=3)) == 256 + 3 * 1024 * 4
    assert hb.workspace_bytes(hb.OP_SPARSE_ATTEND, v4_attn_desc()) >= 256
    # invalid descriptors size to 0
    assert hb.workspace_bytes(hb.OP_FLAT_TOPK, v4_index_desc(D_i=48)) == 0
    assert hb.workspace_bytes(hb.OP_BLOCK_FILTER, v4_index_desc(index_block=0)) == 0
    assert hb.workspace_bytes(hb.OP_BLOCK_FILTER, v4_index_desc(index_keep=4)) == 0  # b*keep < k
    assert hb.workspace_bytes(hb.OP_SPARSE_ATTEND, v4_attn_desc(H=7)) == 0
    assert hb.workspace_bytes(99, v4_index_desc()) == 0


def test_host_validation_rejects_before_launch(lib):
    P = ctypes.c_void_p
    fake = P(1 << 20)          # never dereferenced: validation fails first
    d = v4_index_desc()
    # NULL tensors
    assert lib.hisa_flat_topk(ctypes.byref(d), None, fake, fake, fake, fake, fake, fake, 1 << 30,
                              None) == hb.HISA_EINVAL
    # unsupported head dim
    bad = v4_index_desc(D_i=96)
    assert lib.hisa_index_scores(ctypes.byref(bad), fake, fake, fake, fake, fake, fake, 32768,
                                 fake, 1 << 30, None) == hb.HISA_EDTYPE
    # gate checks the host can see
    g = v4_index_desc(index_block=0)
    assert lib.hisa_block_filter(ctypes.byref(g), fake, fake, fake, fake, fake, fake, fake, None,
                                 0, fake, 1 << 30, None) == hb.HISA_EINVAL
    g = v4_index_desc(index_keep=4)
    assert lib.hisa_select_topk(ctypes.byref(g), fake, fake, fake, fake, fake, fake, fake, None,
                                fake, 1 << 30, None) == hb.HISA_EINVAL
    # misaligned q
    assert lib.hisa_flat_topk(ctypes.byref(d), P((1 << 20) + 4), fake, fake, fake, fake, fake,
                              fake, 1 << 30, None) == hb.HISA_EINVAL
    # workspace missing / too small / misaligned
    assert lib.hisa_flat_topk(ctypes.byref(d), fake, fake, fake, fake, fake, fake, None, 1 << 30,
                              None) == hb.HISA_EWORKSPACE
    assert lib.hisa_flat_topk(ctypes.byref(d), fake, fake, fake, fake, fake, fake, fake, 100,
                              None) == hb.HISA_EWORKSPACE
    assert lib.hisa_flat_topk(ctypes.byref(d), fake, fake, fake, fake, fake, fake,
                              P((1 << 20) + 16), 1 << 30, None) == hb.HISA_EWORKSPACE
    # ld_scores below Np_max
    assert lib.hisa_index_scores(ctypes.byref(d), fake, fake, fake, fake, fake, fake, 100, fake,
                                 1 << 30, None) == hb.HISA_EINVAL
    # attention: mixed dtypes, unsupported heads, I with k == 0
    a = v4_attn_desc(q_dtype=hb.HISA_F32)
    args = [fake] * 11 + [1 << 30, None]    # q .. out, ws; ws_bytes; stream
    assert lib.hisa_sparse_attend(ctypes.byref(a), *args) == hb.HISA_EDTYPE
    a = v4_attn_desc(H=32)
    assert lib.hisa_sparse_attend(ctypes.byref(a), *args) == hb.HISA_EDTYPE
    a = v4_attn_desc(k=0)
    assert lib.hisa_sparse_attend(ctypes.byref(a), *args) == hb.HISA_EINVAL
    # flag bits other than HISA_FLAG_CHAINED
    a = v4_attn_desc(flags=0x2)
    assert lib.hisa_sparse_attend(ctypes.byref(a), *args) == hb.HISA_EINVAL
    # output dtype: f32 (0) or bf16 (1)
    a = v4_attn_desc(out_dtype=2)
    assert lib.hisa_sparse_attend(ctypes.byref(a), *args) == hb.HISA_EDTYPE
    assert hb.workspace_bytes(hb.OP_SPARSE_ATTEND, v4_attn_desc(out_dtype=hb.HISA_BF16)) >= 256
    assert hb.workspace_bytes(hb.OP_SPARSE_ATTEND, v4_attn_desc(flags=hb.FLAG_CHAINED)) >= 256
    g = v4_index_desc(flags=0x4)
    assert lib.hisa_flat_topk(ctypes.byref(g), fake, fake, fake, fake, fake, fake, fake, 1 << 30,
                              None) == hb.HISA_EINVAL
    assert hb.workspace_bytes(hb.OP_FLAT_TOPK, v4_index_desc(flags=0x4)) == 0
    # status helpers
    assert lib.hisa_device_status(None, None, None) == hb.HISA_EINVAL
    assert lib.hisa_workspace_init(None, 0, None) == hb.HISA_EWORKSPACE


def v4_compress_desc(**kw):
    d = dict(B=2, D_i=128, r=4, overlap=1, rope_dims=64, index_block=64, n_new_max=16,
             k_dtype=hb.HISA_BF16, rope_theta=160000.0, eps=1e-6, tok_rows=1 << 20,
             keys_rows=1 << 20, means_rows=1 << 14)
    d.update(kw)
    return hb.CompressDesc(**d)


def test_compress_host_validation(lib):
    P = ctypes.c_void_p
    fake = P(1 << 20)
    args = [fake] * 11 + [fake, 1 << 30, None]     # kv .. means_off, ws; ws_bytes; stream
    assert hb.workspace_bytes(hb.OP_COMPRESS, v4_compress_desc()) == 256
    for bad, code in ((dict(D_i=96), hb.HISA_EDTYPE), (dict(r=0), hb.HISA_EINVAL),
                      (dict(rope_dims=65), hb.HISA_EINVAL), (dict(rope_dims=256), hb.HISA_EINVAL),
                      (dict(overlap=2), hb.HISA_EINVAL), (dict(eps=0.0), hb.HISA_EINVAL),
                      (dict(rope_theta=1.0), hb.HISA_EINVAL), (dict(n_new_max=-1), hb.HISA_EINVAL),
                      (dict(flags=0x8), hb.HISA_EINVAL), (dict(k_dtype=7), hb.HISA_EDTYPE)):
        d = v4_compress_desc(**bad)
        assert lib.hisa_compress_append(ctypes.byref(d), *args) == code, bad
        assert hb.workspace_bytes(hb.OP_COMPRESS, d) == 0, bad
    d = v4_compress_desc()
    assert lib.hisa_compress_append(ctypes.byref(d), None, *args[1:]) == hb.HISA_EINVAL
    # means without their offsets
    a2 = list(args)
    a2[10] = None
    assert lib.hisa_compress_append(ctypes.byref(d), *a2) == hb.HISA_EINVAL
    # misaligned f32 input
    a3 = list(args)
    a3[0] = P((1 << 20) + 2)
    assert lib.hisa_compress_append(ctypes.byref(d), *a3) == hb.HISA_EINVAL
    a4 = list(args)
    a4[11] = None
    assert lib.hisa_compress_append(ctypes.byref(d), *a4) == hb.HISA_EWORKSPACE


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5):
        assert hb.status_string(code).startswith("HISA_")
    assert "unknown" in hb.status_string(42)

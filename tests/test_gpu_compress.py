"""GPU parity of the indexer compressor (hisa_compress_append) against the oracle.

[HiSA issue] "The pooled stream and positions" / "Configuration": gated pooling of r-token
windows (overlap variant: also the previous window), RMSNorm, interleaved RoPE of the
trailing 64 dims at position p r with base 160000; new pooled rows appended to the key
cache and the block means they complete appended to the block-mean cache, with the bits
hisa_block_means writes. Tolerances: oracle/parity.py check_pooled.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from deepseek_sparse_attention_hisa_gb300 import binding as hb  # noqa: E402
from deepseek_sparse_attention_hisa_gb300 import inputs  # noqa: E402
from oracle import hisa_oracle as O  # noqa: E402
from oracle import parity as P  # noqa: E402

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from deepseek_sparse_attention_hisa_gb300 import build
    build.build_library()
    hb.lib()


def dev(a):
    return hb.to_device(a, "cuda")


def run(data, b_blk=64, rope_dims=64, keys_rows=None, means=True, p_first=None, n_new=None):
    """One hisa_compress_append call on `data`; returns (keys, means, means_off, status)."""
    B, D = data["B"], data["D"]
    pf = data["p_first"] if p_first is None else p_first
    nn = data["n_new"] if n_new is None else n_new
    keys = dev(data["keys"])
    cap = np.diff(data["key_off"])
    nb = cap // b_blk if b_blk > 0 else np.zeros_like(cap)
    means_off = np.zeros(B + 1, dtype=np.int64)
    means_off[1:] = np.cumsum(nb)
    m = torch.full((max(int(means_off[-1]), 1), D), 7.0, device="cuda") if means else None
    desc = hb.CompressDesc(B=B, D_i=D, r=data["r"], overlap=int(data["overlap"]),
                           rope_dims=rope_dims, index_block=b_blk,
                           n_new_max=int(np.max(nn)), k_dtype=hb.dtype_code(keys),
                           rope_theta=O.ROPE_THETA, eps=O.RMS_EPS,
                           tok_rows=int(data["tok_off"][-1]),
                           keys_rows=int(keys.shape[0]) if keys_rows is None else keys_rows,
                           means_rows=int(m.shape[0]) if means else 0)
    ws = hb.alloc_workspace(hb.workspace_bytes(hb.OP_COMPRESS, desc))
    hb.compress_append(desc, dev(data["kv"]), dev(data["gate"]), dev(data["tok_off"]),
                       dev(np.asarray(pf, np.int32)), dev(np.asarray(nn, np.int32)),
                       dev(data["ape"]), dev(data["norm_w"]), keys, dev(data["key_off"]),
                       m, dev(means_off) if means else None, ws)
    torch.cuda.synchronize()
    st = hb.device_status(ws)
    return keys, m, means_off, st


def host(t):
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def check_rows(data, keys_out, rope_dims=64):
    kd = "bf16" if np.asarray(data["keys"]).dtype == np.uint16 else "f32"
    g = host(keys_out)
    for b in range(data["B"]):
        p0, nn = int(data["p_first"][b]), int(data["n_new"][b])
        k0 = int(data["key_off"][b])
        t0, t1 = int(data["tok_off"][b]), int(data["tok_off"][b + 1])
        # token rows start at the window before p0: absolute position (p0 - 1) r
        tok0 = (p0 - 1) * data["r"]
        o = O.compress_rows(data["kv"][t0:t1], data["gate"][t0:t1], data["ape"], data["norm_w"],
                            list(range(p0, p0 + nn)), data["r"], tok0=tok0,
                            overlap=data["overlap"], rope_dims=rope_dims)
        P.check_pooled(g[k0 + p0:k0 + p0 + nn], o, kd, what=f"pooled rows of seq {b}")
        # rows before p0 and past p0 + nn are untouched
        np.testing.assert_array_equal(g[k0:k0 + p0], data["keys"][k0:k0 + p0])
        k1 = int(data["key_off"][b + 1])
        np.testing.assert_array_equal(g[k0 + p0 + nn:k1], data["keys"][k0 + p0 + nn:k1])
    return g


def check_means(data, keys_out, m, means_off, b_blk=64):
    """Means of every block the new rows complete: the bits of hisa_block_means on the same
    keys, and the oracle's block means within 1e-6 of the largest |key|; others untouched."""
    B, D = data["B"], data["D"]
    cap = np.diff(data["key_off"])
    idesc = hb.IndexDesc(B=B, L=1, H_i=64, D_i=D, r=data["r"], index_topk=512,
                         index_block=b_blk, index_keep=16, Np_max=int(cap.max()),
                         keys_rows=int(keys_out.shape[0]), means_rows=int(m.shape[0]),
                         q_dtype=hb.HISA_F32, k_dtype=hb.dtype_code(keys_out))
    ref = torch.full_like(m, 7.0)
    ws = hb.alloc_workspace(256)
    hb.block_means(idesc, keys_out, dev(data["key_off"]), dev(means_off), None, ref, ws)
    torch.cuda.synchronize()
    assert hb.device_status(ws) == 0
    g, r = host(m), host(ref)
    kh = host(keys_out)
    done = 0
    for b in range(B):
        p0, nn = int(data["p_first"][b]), int(data["n_new"][b])
        k0 = int(data["key_off"][b])
        for beta in range(int(cap[b]) // b_blk):
            row = int(means_off[b]) + beta
            complete_now = beta * b_blk + b_blk - 1 >= p0 and (beta + 1) * b_blk <= p0 + nn
            if complete_now:
                np.testing.assert_array_equal(g[row], r[row])
                blk = O.to_f64(kh[k0 + beta * b_blk:k0 + (beta + 1) * b_blk])
                scale = max(np.abs(blk).max(), 1e-30)
                assert np.max(np.abs(g[row] - blk.mean(axis=0))) <= 1e-6 * scale
                done += 1
            else:
                assert np.all(g[row] == 7.0), (b, beta)
    return done


def test_decode_and_prefill_appends_v4_shape():
    """D_i = 128, r = 4, overlap, bf16 cache: a decode append that completes block 0 from
    63 cached rows, a prefill of 200 rows from row 0 (blocks 0-2 complete, 3 partial), an
    append starting inside block 2 that completes blocks 2 and 3, and one that completes
    nothing."""
    data = inputs.compressor_inputs(101, p_first=[63, 0, 150, 70], n_new=[1, 200, 106, 5],
                                    capacity=[64, 256, 300, 80])
    keys, m, moff, st = run(data)
    assert st == 0
    check_rows(data, keys)
    assert check_means(data, keys, m, moff) == 1 + 3 + 2


def test_prefill_sized_append_and_a_long_context_position():
    """One sequence appending 1024 pooled rows (4096 prompt tokens, 16 blocks), and one at
    pooled row 262100 (token position 1,048,400), where the first rotated pair turns by
    about 10^6 rad."""
    data = inputs.compressor_inputs(102, p_first=[0, 262100], n_new=[1024, 44],
                                    capacity=[1024, 262144])
    keys, m, moff, st = run(data)
    assert st == 0
    check_rows(data, keys)
    assert check_means(data, keys, m, moff) == 16 + 1


@pytest.mark.parametrize("D,r,overlap,rope,kd", [(64, 8, False, 32, "f32"), (32, 4, True, 16, "bf16"),
                                                 (128, 128, False, 64, "f32")])
def test_other_shapes(D, r, overlap, rope, kd):
    """The plain variant (a softmax over the window's r tokens only), other head dims and
    ratios (r = 128 as on the other compressed layers), f32 caches, no block means."""
    data = inputs.compressor_inputs(103 + D + r, p_first=[0, 5, 17], n_new=[9, 3, 40], D=D, r=r,
                                    overlap=overlap, key_dtype=kd)
    keys, m, moff, st = run(data, b_blk=0, rope_dims=rope, means=False)
    assert st == 0
    check_rows(data, keys, rope_dims=rope)


def test_rows_past_the_cache_are_flagged_not_written():
    """A sequence whose new rows would pass its cache capacity (key_off[b+1]) or the
    allocation (keys_rows) is skipped and flagged; the others are written."""
    data = inputs.compressor_inputs(104, p_first=[10, 20], n_new=[5, 50], capacity=[64, 64])
    keys, m, moff, st = run(data)
    assert st & hb.DEV_BAD_OFFSETS
    g = host(keys)
    np.testing.assert_array_equal(g[64:], data["keys"][64:])          # sequence 1 untouched
    one = dict(data, B=1, p_first=data["p_first"][:1], n_new=data["n_new"][:1],
               tok_off=data["tok_off"][:2], key_off=data["key_off"][:2])
    check_rows(one, keys[:64])
    # the same call with keys_rows one row short for sequence 0
    data2 = inputs.compressor_inputs(105, p_first=[10], n_new=[5], capacity=[15])
    keys2, _, _, st2 = run(data2, keys_rows=14)
    assert st2 & hb.DEV_BAD_OFFSETS
    np.testing.assert_array_equal(host(keys2), data2["keys"])


@pytest.mark.parametrize("B", [100, 200])
def test_many_sequences_appending_a_row_or_two(B):
    """Decode and two-token appends for many sequences at once: one or two new pooled rows
    each, some completing a block (from 62, 63 or 127 cached rows), some inside one. With
    up to two touched blocks per sequence the call runs 2 B CTAs: 200 take the compressor's
    four-row-lane form (two CTAs per SM), 400 its one-lane form."""
    rng = np.random.default_rng(200 + B)
    p_first = rng.choice([62, 63, 127, 30, 95], size=B)
    n_new = rng.integers(1, 3, size=B)
    data = inputs.compressor_inputs(300 + B, p_first=p_first.tolist(), n_new=n_new.tolist(),
                                    capacity=[192] * B)
    keys, m, moff, st = run(data)
    assert st == 0
    check_rows(data, keys)
    done = check_means(data, keys, m, moff)
    want = sum(1 for p, n in zip(p_first, n_new) for beta in range(3)
               if beta * 64 + 63 >= p and (beta + 1) * 64 <= p + n)
    assert done == want and done > 0

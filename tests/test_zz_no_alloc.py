"""The allocation-free flat selection (hisa_flat_topk_noalloc) against hisa_flat_topk.

Collected last on purpose: it must give the same selections whether it runs alone in a
fresh process or after every other test has used the device. All calls go through the
C ABI. Selections are integer results, so the comparison is exact.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from deepseek_sparse_attention_hisa_gb300 import binding as hb  # noqa: E402
from deepseek_sparse_attention_hisa_gb300 import inputs  # noqa: E402
from deepseek_sparse_attention_hisa_gb300.problem import Problem  # noqa: E402


@pytest.fixture(scope="module")
def lib():
    from deepseek_sparse_attention_hisa_gb300 import build
    build.build_library()
    return hb.lib()


def _desc(B, Np_max, D_i=128):
    return hb.IndexDesc(B=B, L=1, H_i=64, D_i=D_i, r=4, index_topk=512, index_block=64,
                        index_keep=16, Np_max=Np_max, keys_rows=B * Np_max, q_dtype=hb.HISA_F32,
                        k_dtype=hb.HISA_BF16)


def test_noalloc_rejects_before_launch(lib):
    """Host checks only: no pointer is dereferenced and nothing reaches a device."""
    fake = [16 * (i + 1) for i in range(6)]  # q .. I: aligned, never dereferenced
    # One score more than the fixed array holds.
    over = _desc(B=128, Np_max=32768 + 1)
    assert lib.hisa_flat_topk_noalloc(hb.ctypes.byref(over), *fake, None, None) == \
        hb.HISA_EWORKSPACE
    # Exactly at the limit the size passes and the missing pointers are reported.
    at = _desc(B=128, Np_max=32768)
    assert 128 * 32768 == hb.FLAT_NOALLOC_MAX_SCORES
    assert lib.hisa_flat_topk_noalloc(hb.ctypes.byref(at), None, *fake[1:], None, None) == \
        hb.HISA_EINVAL
    # An invalid descriptor gives hisa_flat_topk's own verdict.
    bad = _desc(B=1, Np_max=1024, D_i=48)
    assert lib.hisa_flat_topk_noalloc(hb.ctypes.byref(bad), *fake, None, None) == hb.HISA_EDTYPE
    assert lib.hisa_flat_topk_noalloc(None, *fake, None, None) == hb.HISA_EINVAL


def _problems():
    v4 = inputs.WORKLOADS["v4flash_decode"].replace(with_attention=False)
    ragged = inputs.small_workload(name="ragged_causal", seed=77, B=3, L=3, Np=(700, 37, 1000),
                                   t0=2000, with_attention=False)
    return [("v4flash_decode", inputs.generate(v4)), ("ragged_causal_f32", inputs.generate(ragged))]


def _existing(prob):
    I = torch.full((prob.B * prob.L, prob.k), -7, dtype=torch.int32, device="cuda")
    hb.workspace_init(prob.ws)
    hb.flat_topk(prob.idesc, prob.q_idx, prob.w, prob.keys, prob.key_off, prob.t0, I, prob.ws)
    torch.cuda.synchronize()
    assert prob.status() == 0
    return I.cpu().numpy()


def _noalloc(prob, st):
    I = torch.full((prob.B * prob.L, prob.k), -7, dtype=torch.int32, device="cuda")
    st.fill_(0x7fff)
    hb.flat_topk_noalloc(prob.idesc, prob.q_idx, prob.w, prob.keys, prob.key_off, prob.t0, I, st)
    torch.cuda.synchronize()
    return I.cpu().numpy(), int(st.item())


@pytest.mark.gpu
@pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")
def test_noalloc_matches_flat_topk_on_consecutive_calls(lib):
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    # The larger problem runs first, so the second one finds stale scores in the array.
    for name, data in _problems():
        prob = Problem(data, device="cuda")
        ref = _existing(prob)
        for call in range(2):
            got, status = _noalloc(prob, st)
            assert status == 0, (name, call, status)
            np.testing.assert_array_equal(np.sort(got, axis=1), np.sort(ref, axis=1),
                                          err_msg=f"{name}, call {call}")
            assert np.array_equal(got, ref), (name, call)


@pytest.mark.gpu
@pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")
def test_noalloc_status_is_per_call(lib):
    """A call whose offsets run past the keys flags HISA_DEV_BAD_OFFSETS; the next, clean
    call reports a clear status, because every call starts from a cleared status word."""
    data = inputs.generate(inputs.small_workload(name="offsets", seed=5, B=2, Np=(300, 400),
                                                 with_attention=False))
    prob = Problem(data, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    ref = _existing(prob)
    good_off = prob.key_off.clone()
    prob.key_off[2] = prob.idesc.keys_rows + 64      # sequence 1 ends past the allocation
    got, status = _noalloc(prob, st)
    assert status & hb.DEV_BAD_OFFSETS
    assert (got[1] == -1).all()
    np.testing.assert_array_equal(got[0], ref[0])
    prob.key_off.copy_(good_off)
    got, status = _noalloc(prob, st)
    assert status == 0
    np.testing.assert_array_equal(got, ref)

"""GPU parity: every stage of the CUDA path against the oracle on seeded inputs.

All calls go through the C ABI (libhisa.so via the ctypes binding). Comparison rules
are those of oracle/parity.py: scores within 1e-5 * max(|o|, A') and within the f32
bound 4.8e-7 * A', selections equal as sets up to a few near-ties of the k-th oracle
score, attention max-abs 1e-2 (bf16 KV) / 1e-4 (f32) and element-wise within
eps * E (E the softmax-weighted |V|). V4-shape combine tests also run on the "peaked"
attention inputs (KV ~ N(0, 1), logits of std 3, sinks near the largest logit), where
outputs are of order one and each sink holds a visible share of its normaliser.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from deepseek_sparse_attention_hisa_gb300 import binding as hb  # noqa: E402
from deepseek_sparse_attention_hisa_gb300 import inputs  # noqa: E402
from deepseek_sparse_attention_hisa_gb300.problem import Problem  # noqa: E402
from oracle import hisa_oracle as O  # noqa: E402
from oracle import parity as P  # noqa: E402

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from deepseek_sparse_attention_hisa_gb300 import build
    build.build_library()
    hb.lib()


_CACHE = {}


def gen(name, dist="pages"):
    key = (name, dist)
    if key not in _CACHE:
        _CACHE.clear()
        wl = inputs.WORKLOADS[name]
        _CACHE[key] = inputs.generate(inputs.peaked(wl) if dist == "peaked" else wl)
    return _CACHE[key]


def np_(t):
    return t.detach().cpu().numpy()


def run_hisa(prob, with_scores=True):
    """block means -> coarse -> fine -> combine; returns host copies of each stage."""
    rows = prob.B * prob.L
    nb_max = max(int(prob.nb.max()), 1)
    cs = torch.full((rows, nb_max), 7.0, device="cuda") if with_scores else None
    fs = torch.full((rows, prob.b * prob.keep), 7.0, device="cuda") if with_scores else None
    prob.block_means()
    prob.block_filter(cscores=cs)
    prob.select_topk(fscores=fs)
    if prob.has_attention:
        prob.attend()
    torch.cuda.synchronize()
    assert prob.status() == 0
    return dict(means=np_(prob.means), top_blk=np_(prob.top_blk), I=np_(prob.I),
                cs=None if cs is None else np_(cs), fs=None if fs is None else np_(fs),
                out=np_(prob.out) if prob.has_attention else None)


def check_rows(data, prob, res, rows):
    wl = data["wl"]
    P.check_block_means(data, res["means"], np_(prob.means_off), wl.index_block)
    for b, j in rows:
        r = b * wl.L + j
        P.check_coarse(data, b, j, res["top_blk"][r],
                       None if res["cs"] is None else res["cs"][r], wl.index_block, prob.keep)
        P.check_fine(data, b, j, res["top_blk"][r], res["I"][r],
                     None if res["fs"] is None else res["fs"][r], wl.index_block, wl.index_topk)
        if res["out"] is not None:
            P.check_attend(data, b, j, res["out"][r], res["I"][r])


def run_flat(prob, with_scores=True):
    rows = prob.B * prob.L
    sc = torch.full((rows, max(prob.Np_max, 1)), 7.0, device="cuda") if with_scores else None
    if with_scores:
        prob.index_scores(sc)
    I = torch.full((rows, prob.k), -7, dtype=torch.int32, device="cuda")
    prob.flat_topk(I=I)
    torch.cuda.synchronize()
    assert prob.status() == 0
    return np_(I), None if sc is None else np_(sc)


# ----------------------------------------------------------------------------
# the five workloads
# ----------------------------------------------------------------------------
def test_tiny_decode_every_stage():
    data = gen("tiny_decode")
    prob = Problem(data)
    res = run_hisa(prob)
    check_rows(data, prob, res, [(0, 0)])
    I, sc = run_flat(prob)
    P.check_flat(data, 0, 0, I[0], 32, sc[0])
    prob.attend(I=None)                        # dense branch over all 512 pooled rows
    P.check_attend(data, 0, 0, np_(prob.out)[0], None)


@pytest.mark.parametrize("dist", ["pages", "peaked"])
def test_v4flash_decode_every_stage(dist):
    data = gen("v4flash_decode", dist)
    prob = Problem(data)
    res = run_hisa(prob)
    check_rows(data, prob, res, [(0, 0)])
    I, sc = run_flat(prob)
    P.check_flat(data, 0, 0, I[0], 512, sc[0])
    # the flat selection feeds the same combine
    prob.attend(I=torch.as_tensor(I, device="cuda"))
    P.check_attend(data, 0, 0, np_(prob.out)[0], I[0])


@pytest.mark.parametrize("dist", ["pages", "peaked"])
def test_ragged_decode_all_sequences(dist):
    data = gen("ragged_decode", dist)
    prob = Problem(data)
    res = run_hisa(prob)
    check_rows(data, prob, res, [(b, 0) for b in range(data["wl"].B)])
    if dist == "peaked":
        return
    I, _ = run_flat(prob, with_scores=False)
    for b in (0, 7, 31):
        P.check_flat(data, b, 0, I[b], 512)


@pytest.mark.parametrize("dist", ["pages", "peaked"])
def test_prefill_sampled_rows(dist):
    data = gen("prefill", dist)
    prob = Problem(data)
    res = run_hisa(prob, with_scores=True)
    L = data["wl"].L
    rng = np.random.default_rng(0)
    rows = sorted({0, 1, 2, 255, 256, 511, 512, 2047, L - 2, L - 1} |
                  set(rng.integers(0, L, 6).tolist()))
    check_rows(data, prob, res, [(0, j) for j in rows])
    if dist == "peaked":        # the indexer inputs are the same draws: scored above
        return
    # the dense L x Np x (H_i * D_i) contraction, sampled rows
    sc = torch.empty((L, prob.Np_max), device="cuda")
    prob.index_scores(sc)
    torch.cuda.synchronize()
    sc = np_(sc)
    for j in rows[:6]:
        q, w = data["q_idx"][0, j], data["w"][0, j]
        o = O.flat_scores(q[None], w[None], data["keys"], int(data["t0"][0]) + j, 4, causal=True)[0]
        P.check_scores(sc[j], o, P.score_scale(q, w, data["keys"]), what=f"prefill score row {j}")
    # the flat selection over those scores
    I = torch.full((L, prob.k), -7, dtype=torch.int32, device="cuda")
    prob.flat_topk(I)
    torch.cuda.synchronize()
    I = np_(I)
    for j in rows[:4]:
        P.check_flat(data, 0, j, I[j], prob.k)


@pytest.mark.parametrize("keep", [16, 64])
def test_long_context_flat_and_hisa(keep):
    data = gen("long_context")
    prob = Problem(data, index_keep=keep)
    res = run_hisa(prob, with_scores=True)
    check_rows(data, prob, res, [(0, 0)])
    I, sc = run_flat(prob)
    P.check_flat(data, 0, 0, I[0], 512, sc[0])
    recall = len(set(res["I"][0].tolist()) & set(I[0].tolist())) / 512
    print(f"long context keep={keep}: recall vs flat = {recall:.3f}")
    assert recall > 0.0


# ----------------------------------------------------------------------------
# edge cases: several tiles, ragged tails, short sequences, L > 1 causality
# ----------------------------------------------------------------------------
def small(**kw):
    return inputs.generate(inputs.small_workload(**kw))


def test_ragged_tails_and_tiles():
    # Np not a multiple of b, several 256-row score tiles, f32 and bf16 keys
    for kd in ("f32", "bf16"):
        data = small(B=3, Np=(700, 1000, 1333), key_dtype=kd, kv_dtype=kd, seed=5)
        data["t0"][:] = 4 * data["Np"] - 1
        prob = Problem(data)
        res = run_hisa(prob)
        check_rows(data, prob, res, [(b, 0) for b in range(3)])
        for b in range(3):
            assert np.all(res["I"][b] < (data["Np"][b] // 16) * 16)   # tail exclusion
        I, sc = run_flat(prob)
        for b in range(3):
            P.check_flat(data, b, 0, I[b], 32, sc[b])


def test_flat_pads_when_Np_below_k_and_dense_branch():
    data = small(Np=(20,), seed=6)
    prob = Problem(data)
    I, sc = run_flat(prob)
    assert np.all(I[0, 20:] == -1)
    P.check_flat(data, 0, 0, I[0], 32, sc[0])
    prob.attend(I=None)
    P.check_attend(data, 0, 0, np_(prob.out)[0], None)
    prob.attend(I=torch.as_tensor(I, device="cuda"))      # -1 padding is skipped
    P.check_attend(data, 0, 0, np_(prob.out)[0], I[0])


def test_local_only_attention():
    data = small(Np=(0,), seed=7)
    prob = Problem(data)
    prob.attend(I=None)
    torch.cuda.synchronize()
    P.check_attend(data, 0, 0, np_(prob.out)[0], None)


@pytest.mark.parametrize("t0", [60, 1900])
def test_batched_rows_with_few_visible(t0):
    # L > 1. With t0 = 60 every row sees fewer than k = 32 pooled rows and fewer than
    # keep eligible blocks (masked ids are selected, then re-masked by the combine);
    # with t0 = 1900 rows see partially visible blocks at the edge of V(t).
    data = small(L=48, Np=(512,), seed=8, t0=t0)
    prob = Problem(data)
    res = run_hisa(prob)
    check_rows(data, prob, res, [(0, j) for j in range(48)])
    I, sc = run_flat(prob)
    for j in range(0, 48, 5):
        P.check_flat(data, 0, j, I[j], 32, sc[j])


def test_device_gate_and_bad_ids_are_flagged_not_faulted():
    data = small(B=2, Np=(512, 40), seed=9)   # sequence 1 fails Np >= b * keep = 64
    prob = Problem(data)
    prob.block_means()
    prob.block_filter()
    prob.select_topk()
    torch.cuda.synchronize()
    assert prob.status() & hb.DEV_GATE
    assert np.all(np_(prob.top_blk)[1] == -1) and np.all(np_(prob.I)[1] == -1)
    hb.workspace_init(prob.ws)
    # out-of-range ids in I are skipped and flagged; in-range ones still attend
    I = torch.as_tensor(np.array([[3, 5, 10 ** 6, -5] + [-1] * 28] * 2, dtype=np.int32),
                        device="cuda")
    prob.attend(I=I)
    torch.cuda.synchronize()
    assert prob.status() & hb.DEV_BAD_ID
    clean = np.array([3, 5, -1, -1] + [-1] * 28)
    P.check_attend(data, 0, 0, np_(prob.out)[0], clean)
    hb.workspace_init(prob.ws)
    tb = torch.as_tensor(np.array([[0, 1, 2, 99], [0, 1, 2, 3]], dtype=np.int32), device="cuda")
    prob.select_topk(top_blk=tb)
    torch.cuda.synchronize()
    st = prob.status()
    assert st & hb.DEV_BAD_BLOCK and np.all(np_(prob.I)[0] == -1)


def test_host_validation_raises():
    data = small(seed=10)
    prob = Problem(data)
    bad = hb.IndexDesc.from_buffer_copy(prob.idesc)
    bad.D_i = 48
    with pytest.raises(hb.HisaError) as e:
        hb.flat_topk(bad, prob.q_idx, prob.w, prob.keys, prob.key_off, prob.t0, prob.I, prob.ws)
    assert e.value.status == hb.HISA_EDTYPE
    small_ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(hb.HisaError) as e:
        hb.flat_topk(prob.idesc, prob.q_idx, prob.w, prob.keys, prob.key_off, prob.t0, prob.I,
                     small_ws)
    assert e.value.status == hb.HISA_EWORKSPACE


def test_graph_capture_replays_the_step():
    data = small(B=4, Np=(512, 600, 700, 1024), key_dtype="bf16", kv_dtype="bf16", seed=11)
    data["t0"][:] = 4 * data["Np"] - 1
    prob = Problem(data)
    prob.block_means()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        prob.hisa_step(stream=s)                 # warm-up (sets kernel attributes)
    torch.cuda.synchronize()
    eager_I, eager_out = np_(prob.I).copy(), np_(prob.out).copy()
    prob.I.fill_(-7)
    prob.out.fill_(0)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        prob.hisa_step(stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(np_(prob.I), eager_I)
    assert np.array_equal(np_(prob.out), eager_out)


def v4_small(dist="pages", **kw):
    base = dict(H_i=64, D_i=128, index_block=64, index_keep=16, index_topk=512, H=64, Dh=512,
                window=128, q_idx_dtype="f32", key_dtype="bf16", kv_dtype="bf16")
    base.update(kw)
    wl = inputs.small_workload(**base)
    return inputs.generate(inputs.peaked(wl) if dist == "peaked" else wl)


@pytest.mark.parametrize("dist", ["pages", "peaked"])
def test_v4_combine_edges(dist):
    # the tensor-core combine (64 heads x 512, bf16): -1 padding (Np < k), local only
    # (Np = 0), and the dense branch over 3000 rows split across many CTAs
    data = v4_small(dist, B=3, Np=(100, 0, 3000), seed=12)
    data["t0"][:] = np.maximum(4 * data["Np"] - 1, 200)
    data["local_pos0"][:] = data["t0"] - 127
    prob = Problem(data)
    I = np.full((3, 512), -1, dtype=np.int32)
    I[0, :100] = np.arange(100)[::-1]
    I[2] = np.random.default_rng(0).choice(3000, 512, replace=False)
    prob.attend(I=torch.as_tensor(I, device="cuda"))
    torch.cuda.synchronize()
    assert prob.status() == 0
    out = np_(prob.out)
    for b in range(3):
        P.check_attend(data, b, 0, out[b], I[b])
    prob.attend(I=None)
    torch.cuda.synchronize()
    out = np_(prob.out)
    for b in range(3):
        P.check_attend(data, b, 0, out[b], None)


@pytest.mark.parametrize("dist", ["pages", "peaked"])
def test_v4_combine_prefill_rows(dist):
    # L > 1 with the V4 shape: local window per row, causal re-mask of pooled ids (every
    # row's selection holds the id V(t) itself, the first one the re-mask hides)
    data = v4_small(dist, L=40, Np=(2048,), seed=13, t0=3000, kv_dtype="bf16")
    prob = Problem(data)
    rng = np.random.default_rng(1)
    I = np.stack([rng.choice(2048, 512, replace=False) for _ in range(40)]).astype(np.int32)
    for j in range(40):
        V = O.visible_len(3000 + j, 4, 2048)
        if V not in set(I[j].tolist()):
            I[j, 0] = V
    prob.attend(I=torch.as_tensor(I, device="cuda"))
    torch.cuda.synchronize()
    assert prob.status() == 0
    out = np_(prob.out)
    for j in range(40):
        P.check_attend(data, 0, j, out[j], I[j])


def test_offsets_past_the_allocation_are_skipped():
    # keys_rows / kv_rows bound every read: a sequence whose rows end past them is
    # skipped (-1 rows, zero output) and flagged, and the others are unaffected.
    data = v4_small(B=2, Np=(2048, 2048), seed=14)
    prob = Problem(data)
    prob.block_means()
    torch.cuda.synchronize()
    short = hb.IndexDesc.from_buffer_copy(prob.idesc)
    short.keys_rows = 3000
    I = torch.full_like(prob.I, -7)
    hb.flat_topk(short, prob.q_idx, prob.w, prob.keys, prob.key_off, prob.t0, I, prob.ws)
    hb.select_topk(short, prob.q_idx, prob.w, prob.keys, prob.key_off, prob.t0, prob.top_blk,
                   prob.I, prob.ws)
    torch.cuda.synchronize()
    assert prob.status() & hb.DEV_BAD_OFFSETS
    assert np.all(np_(I)[1] == -1) and np.all(np_(prob.I)[1] == -1)
    P.check_flat(data, 0, 0, np_(I)[0], 512)
    hb.workspace_init(prob.ws)
    a = hb.AttnDesc.from_buffer_copy(prob.adesc)
    a.kv_rows = 3000
    out = torch.full_like(prob.out, 5.0)
    hb.sparse_attend(a, prob.q_attn, prob.local_kv, prob.local_len, prob.local_pos0,
                     prob.pooled_kv, prob.key_off, None, prob.sinks, prob.t0, out, prob.ws)
    torch.cuda.synchronize()
    assert prob.status() & hb.DEV_BAD_OFFSETS
    P.check_attend(data, 0, 0, np_(out)[0], None)


def test_many_queries_per_sm_with_invalid_rows_between():
    """More query rows than SMs, so each persistent scoring CTA walks several; rows that
    fail the gate or carry a bad kept block sit between valid ones and must not disturb
    the rows after them."""
    B = 330
    rng = np.random.default_rng(21)
    Np = rng.integers(1024, 3000, size=B)
    Np[[5, 157, 158, 310]] = 700                  # below index_block * index_keep = 1024
    wl = inputs.small_workload(name="many_rows", seed=21, B=B, H_i=64, D_i=128, index_block=64,
                               index_keep=16, index_topk=512, q_idx_dtype="f32", key_dtype="bf16",
                               Np=tuple(int(x) for x in Np), with_attention=False)
    data = inputs.generate(wl)
    prob = Problem(data)
    rows_cs = torch.full((B, int(prob.nb.max())), 7.0, device="cuda")
    rows_fs = torch.full((B, 1024), 7.0, device="cuda")
    prob.block_means()
    prob.block_filter(cscores=rows_cs)
    torch.cuda.synchronize()
    assert prob.status() == hb.DEV_GATE
    tb = np_(prob.top_blk)
    bad = [5, 157, 158, 310]
    assert np.all(tb[bad] == -1)
    tb_bad = tb.copy()
    tb_bad[200, 3] = 10 ** 6                      # one row with an out-of-range kept block
    hb.workspace_init(prob.ws)
    prob.select_topk(top_blk=torch.as_tensor(tb_bad, device="cuda"), fscores=rows_fs)
    torch.cuda.synchronize()
    assert prob.status() == (hb.DEV_GATE | hb.DEV_BAD_BLOCK)
    I = np_(prob.I)
    assert np.all(I[bad] == -1) and np.all(I[200] == -1)
    cs, fs = np_(rows_cs), np_(rows_fs)
    for b in (0, 1, 4, 6, 151, 152, 153, 156, 159, 199, 201, 303, 304, 309, 311, 329):
        P.check_coarse(data, b, 0, tb[b], cs[b], wl.index_block, wl.index_keep)
        P.check_fine(data, b, 0, tb[b], I[b], fs[b], wl.index_block, wl.index_topk)


@pytest.mark.parametrize("t0,qd", [(2000, "f32"), (7000, "bf16")])
def test_v4_shape_batched_rows_with_few_visible(t0, qd):
    """The tensor-core pipeline with L > 1 at the V4 indexer shape: at t0 = 2000 every row
    sees fewer than keep eligible blocks and fewer than k visible candidates (masked ids
    fill the selection); at t0 = 7000 the visibility edge falls inside the kept blocks."""
    wl = inputs.small_workload(name="v4_few_visible", seed=31, L=48, H_i=64, D_i=128,
                               index_block=64, index_keep=16, index_topk=512, q_idx_dtype=qd,
                               key_dtype="bf16", Np=(2048,), t0=t0, with_attention=False)
    data = inputs.generate(wl)
    prob = Problem(data)
    res = run_hisa(prob)
    check_rows(data, prob, res, [(0, j) for j in range(0, 48, 3)] + [(0, 47)])


def test_dense_scoring_partial_units_and_ragged_sequences():
    """The dense scoring of many bf16 query rows per sequence (four rows per tensor-core
    unit): L = 6 leaves a partial unit, three sequences of different Np, and the causal
    edge V(t0 + j) falls inside the key tiles of the first two."""
    wl = inputs.small_workload(name="dense_rows", seed=41, B=3, L=6, H_i=64, D_i=128,
                               index_block=64, index_keep=16, index_topk=512, q_idx_dtype="bf16",
                               key_dtype="bf16", Np=(700, 1500, 300), t0=2200, with_attention=False)
    data = inputs.generate(wl)
    prob = Problem(data)
    sc = torch.full((wl.B * wl.L, prob.Np_max), 7.0, device="cuda")
    prob.index_scores(sc)
    I = torch.full((wl.B * wl.L, wl.index_topk), -7, dtype=torch.int32, device="cuda")
    prob.flat_topk(I)
    torch.cuda.synchronize()
    assert prob.status() == 0
    sc, I = np_(sc), np_(I)
    for b in range(wl.B):
        s = P.seq(data, b)
        for j in range(wl.L):
            r = b * wl.L + j
            q, w = data["q_idx"][b, j], data["w"][b, j]
            o = O.flat_scores(q[None], w[None], s["keys"], s["t0"] + j, wl.r, causal=True)[0]
            P.check_scores(sc[r, : s["Np"]], o, P.score_scale(q, w, s["keys"]),
                           what=f"dense score row {b},{j}")
            assert np.all(sc[r, s["Np"]:] == 7.0)        # columns past Np are not written
            P.check_flat(data, b, j, I[r], wl.index_topk)


def test_block_filter_append_matches_means_then_filter():
    """hisa_block_filter_append (means of the new blocks computed inside the coarse kernel
    for decode) gives the bits of hisa_block_means followed by hisa_block_filter: zero,
    one, three and all blocks new, across ragged sequences."""
    B = 6
    wl = inputs.small_workload(name="append", seed=51, B=B, H_i=64, D_i=128, index_block=64,
                               index_keep=16, index_topk=512, q_idx_dtype="f32", key_dtype="bf16",
                               Np=(2048, 4100, 8192, 1024, 3000, 6400), with_attention=False)
    data = inputs.generate(wl)
    ref, fus = Problem(data), Problem(data)
    nb = np.asarray(data["Np"]) // 64
    fb = np.array([nb[0] - 1, nb[1], nb[2] - 3, 0, nb[4] - 1, nb[5] - 2], dtype=np.int32)
    fb_t = torch.as_tensor(fb, device="cuda")
    # both start from a cache whose new blocks hold garbage
    ref.block_means()
    fus.means.copy_(ref.means)
    for b in range(B):
        m0 = int(np_(ref.means_off)[b])
        ref.means[m0 + int(fb[b]):m0 + int(nb[b])] = 123.0
        fus.means[m0 + int(fb[b]):m0 + int(nb[b])] = -77.0
    cs_ref = torch.full((B, int(nb.max())), 7.0, device="cuda")
    cs_fus = torch.full((B, int(nb.max())), 7.0, device="cuda")
    hb.block_means(ref.idesc, ref.keys, ref.key_off, ref.means_off, fb_t, ref.means, ref.ws)
    ref.block_filter(cscores=cs_ref)
    fus.block_filter_append(first_block=fb_t, cscores=cs_fus)
    torch.cuda.synchronize()
    assert ref.status() == 0 and fus.status() == 0
    assert torch.equal(ref.means, fus.means)
    assert torch.equal(cs_ref, cs_fus)
    assert np.array_equal(np.sort(np_(ref.top_blk), axis=1), np.sort(np_(fus.top_blk), axis=1))
    P.check_block_means(data, np_(fus.means), np_(fus.means_off), 64)
    for b in range(B):
        P.check_coarse(data, b, 0, np_(fus.top_blk)[b], np_(cs_fus)[b], 64, 16)


def test_block_filter_append_two_call_path():
    """Shapes the fused kernel does not take (f32 keys, or L > 1) run the two calls."""
    for kw in (dict(seed=52, B=2, Np=(700, 1000)), dict(seed=53, L=6, Np=(512,), t0=1900)):
        data = small(**kw)
        prob = Problem(data)
        fb = torch.zeros(data["wl"].B, dtype=torch.int32, device="cuda")
        prob.block_filter_append(first_block=fb)
        torch.cuda.synchronize()
        assert prob.status() == 0
        P.check_block_means(data, np_(prob.means), np_(prob.means_off), data["wl"].index_block)
        for b in range(data["wl"].B):
            for j in range(data["wl"].L):
                P.check_coarse(data, b, j, np_(prob.top_blk)[b * data["wl"].L + j], None,
                               data["wl"].index_block, data["wl"].index_keep)


def test_selection_ties_equal_means_and_outliers():
    """Selections where value bins cannot separate the scores. Sequences built from a few
    distinct key rows give groups of bit-identical fine scores (64 equal ones with the k-th
    at a group's edge, and 208 equal ones, more than a value bin resolves itself) and, with
    16 distinct rows, block means that are all equal; a sequence whose blocks repeat with
    period 7 ties both stages inside a group (10 blocks and 6 of 9; 6 of 10 equal fine
    scores); one sequence holds a block of keys 1000 times larger than the rest, so the
    other scores share a few bins. Equal scores are taken by ascending id, and the sets
    equal the oracle's exactly (no near-ties here besides the exact ones). With 310 query
    rows the first five are selected beside the next row's scoring and the last five by
    the whole CTA, the two forms of the pipeline's select."""
    B, Np = 310, 4096
    special = [0, 1, 2, 3, 4, 304, 305, 306, 307, 308]
    sizes = tuple(Np if b in special else 1024 for b in range(B))
    wl = inputs.small_workload(name="ties", seed=61, B=B, H_i=64, D_i=128, index_block=64,
                               index_keep=16, index_topk=512, q_idx_dtype="f32",
                               key_dtype="bf16", Np=sizes, with_attention=False)
    data = inputs.generate(wl)
    keys = data["keys"]
    r = np.arange(Np)
    for b in special:
        k0, kind = int(data["key_off"][b]), b % 304
        if kind in (0, 1):
            keys[k0:k0 + Np] = keys[k0 + r % (16 if kind == 0 else 5)]
        elif kind == 2:
            big = O.to_f64(keys[k0 + 7 * 64:k0 + 8 * 64]) * 1000.0
            keys[k0 + 7 * 64:k0 + 8 * 64] = inputs.f32_to_bf16_bits(big.astype(np.float32))
        elif kind == 3:                               # block beta is a copy of block beta % 7
            keys[k0:k0 + Np] = keys[k0 + (r // 64 % 7) * 64 + r % 64]
    prob = Problem(data)
    cs = torch.full((B, Np // 64), 7.0, device="cuda")
    fs = torch.full((B, 1024), 7.0, device="cuda")
    prob.block_means()
    prob.block_filter(cscores=cs)
    prob.select_topk(fscores=fs)
    torch.cuda.synchronize()
    assert prob.status() == 0
    tb, I, cs, fs = np_(prob.top_blk), np_(prob.I), np_(cs), np_(fs)
    for b in (0, 304):                                # equal means: the first 16 blocks
        assert np.all(cs[b, :64] == cs[b, 0])
        assert np.array_equal(np.sort(tb[b]), np.arange(16))
    for b in special + [5, 151, 152, 153, 303, 309]:
        P.check_coarse(data, b, 0, tb[b], cs[b], 64, 16)
        P.check_fine(data, b, 0, tb[b], I[b], fs[b], 64, 512)
        s = P.seq(data, b)
        q, w = data["q_idx"][b, 0], data["w"][b, 0]
        if b % 304 != 1:     # rotated copies of rows round their block sums differently
            _, c_top = O.hisa_coarse(q, w, O.block_means(s["keys"], 64), 16, 64)
            assert set(tb[b].tolist()) == set(c_top.tolist()), f"top_blk[{b}]"
        _, _, f_top = O.hisa_fine(q, w, s["keys"], np.sort(tb[b]), 64, 512)
        assert set(I[b].tolist()) == set(f_top.tolist()), f"I[{b}]"
        assert np.all(np.diff(I[b]) > 0)              # ascending ids


def test_long_rows_split_scoring_and_chunked_flat_select():
    """Few long rows: coarse and fine scoring split over CTAs with a separate select (nb and
    keep * b of 2048 and more), and flat rows longer than 8192 selected chunk by chunk (last
    chunks shorter and longer than 2k, and exact ties across chunks: keys repeat every 5000
    rows in sequence 1, so equal scores straddle chunk edges and must go by ascending id)."""
    B = 3
    Np = (131072 + 700, 140000, 8192 * 2 + 3000)
    wl = inputs.small_workload(name="long_rows", seed=71, B=B, H_i=64, D_i=128, index_block=64,
                               index_keep=32, index_topk=512, q_idx_dtype="f32", key_dtype="bf16",
                               Np=Np, with_attention=False)
    data = inputs.generate(wl)
    k0 = int(data["key_off"][1])
    r = np.arange(Np[1])
    data["keys"][k0:k0 + Np[1]] = data["keys"][k0 + r % 5000]
    prob = Problem(data)
    res = run_hisa(prob)
    for b in range(B):
        P.check_coarse(data, b, 0, res["top_blk"][b], res["cs"][b], 64, 32)
        P.check_fine(data, b, 0, res["top_blk"][b], res["I"][b], res["fs"][b], 64, 512)
    I, sc = run_flat(prob)
    for b in range(B):
        P.check_flat(data, b, 0, I[b], 512, sc[b])
    # sequence 1: every score repeats every 5000 rows; the selection is exactly the oracle's
    s = P.seq(data, 1)
    o = O.flat_scores(data["q_idx"][1, :1], data["w"][1, :1], s["keys"], s["t0"], wl.r)[0]
    assert set(I[1].tolist()) == set(O.top_k(o, 512).tolist())
    assert np.all(np.diff(I[1]) > 0)


@pytest.mark.parametrize("L,t0", [(1, None), (4, 3000)])
def test_per_token_indexer_r1(L, t0):
    """The per-token indexer variant (every token is a key, r = 1): flat scoring and top-k,
    and the HiSA stages, on the V4 indexer shape. Decode (L = 1, V = Np) and a four-token
    verify block whose causal edge V(t0 + j) = t0 + j + 1 falls inside the keys."""
    wl = inputs.small_workload(name="r1", seed=81, B=2, L=L, r=1, H_i=64, D_i=128, index_block=64,
                               index_keep=16, index_topk=512, q_idx_dtype="f32",
                               key_dtype="bf16", Np=(4096, 3500), t0=t0, with_attention=False)
    data = inputs.generate(wl)
    prob = Problem(data)
    I, sc = run_flat(prob)
    res = run_hisa(prob)
    for b in range(wl.B):
        for j in range(L):
            r_ = b * L + j
            P.check_flat(data, b, j, I[r_], 512, sc[r_])
    check_rows(data, prob, res, [(b, j) for b in range(wl.B) for j in range(L)])


@pytest.mark.parametrize("L", [2, 4, 8])
def test_multi_token_verify_end_to_end(L):
    """Multi-token verify on the HiSA batched path ([HiSA issue] "HiSA batched path"):
    L draft tokens per sequence at positions t0 .. t0 + L - 1, the pooled cache holding
    every window those tokens complete (Np = floor((t0 + L) / 4)), so the first rows see
    one or two pooled rows fewer than the last ones. The last complete block holds twice
    the keys of row 0's best block, so row 0 keeps it while its last rows sit past V(t):
    the causal edge inside a kept block. Block filter, fine top-k and the combine (pages
    and peaked attention inputs) against the oracle, row by row."""
    B = 4
    t0 = np.array([16379, 16381, 8190, 12001], dtype=np.int64)
    Np = (t0 + L) // 4
    wl = inputs.small_workload(name="verify", seed=90 + L, B=B, L=L, H_i=64, D_i=128,
                               index_block=64, index_keep=16, index_topk=512, H=64, Dh=512,
                               window=128, q_idx_dtype="f32", key_dtype="bf16",
                               kv_dtype="bf16", Np=tuple(int(x) for x in Np), t0=0)
    edge_rows = 0
    for dist in ("pages", "peaked"):
        data = inputs.generate(inputs.peaked(wl) if dist == "peaked" else wl)
        data["t0"][:] = t0
        data["local_pos0"][:] = t0 + (L - 1) - (data["local_kv"].shape[1] - 1)
        for b in range(B):
            s = P.seq(data, b)
            nb = int(Np[b]) // 64
            _, top = O.hisa_coarse(data["q_idx"][b, 0], data["w"][b, 0],
                                   O.block_means(s["keys"], 64), 1, 64)
            k0 = int(data["key_off"][b])
            src = O.to_f64(data["keys"][k0 + int(top[0]) * 64:k0 + int(top[0]) * 64 + 64])
            data["keys"][k0 + (nb - 1) * 64:k0 + nb * 64] = \
                inputs.f32_to_bf16_bits((2.0 * src).astype(np.float32))
        prob = Problem(data)
        res = run_hisa(prob)
        check_rows(data, prob, res, [(b, j) for b in range(B) for j in range(L)])
        for b in range(B):
            nb = int(Np[b]) // 64
            for j in range(L):
                V = O.visible_len(int(t0[b]) + j, 4, int(Np[b]))
                if V < nb * 64 and (nb - 1) in set(res["top_blk"][b * L + j].tolist()):
                    edge_rows += 1
    assert edge_rows > 0


def test_inputs_written_by_the_kernel_just_before_a_call():
    """Calls without HISA_FLAG_CHAINED start after the previous kernel on the stream has
    completed, so inputs a caller's own kernel writes just before them are seen: q and w
    of the fine stage and q of the combine are overwritten by torch kernels right before
    each call, and the results follow the new values."""
    data = v4_small("peaked", B=2, Np=(4096, 3000), seed=15)
    prob = Problem(data)
    prob.block_means()
    prob.block_filter()
    torch.cuda.synchronize()
    fresh = v4_small("peaked", B=2, Np=(4096, 3000), seed=16)
    q_new = hb.to_device(fresh["q_idx"], "cuda")
    w_new = hb.to_device(fresh["w"], "cuda")
    qa_new = hb.to_device(fresh["q_attn"], "cuda")
    for _ in range(3):
        prob.q_idx.zero_()
        prob.w.zero_()
        prob.q_attn.zero_()
        torch.cuda.synchronize()
        prob.q_idx.copy_(q_new)                    # a torch kernel writes q ...
        prob.w.copy_(w_new)
        prob.select_topk()                         # ... and the call comes right after it
        prob.q_attn.copy_(qa_new)
        prob.attend()
        torch.cuda.synchronize()
        assert prob.status() == 0
        mixed = dict(data, q_idx=fresh["q_idx"], w=fresh["w"], q_attn=fresh["q_attn"])
        tb, I, out = np_(prob.top_blk), np_(prob.I), np_(prob.out)
        for b in range(2):
            P.check_fine(mixed, b, 0, tb[b], I[b], None, 64, 512)
            P.check_attend(mixed, b, 0, out[b], I[b])


def test_prefill_coarse_contraction_ragged_rows():
    """The coarse stage of many bf16 query rows runs as one dense contraction over the block
    means split into three bf16 planes: three sequences of 100 rows each (block counts 32, 78
    and 17, none a multiple of the 128-block tile), rows whose visible prefix ends inside a
    block, and rows that see fewer than keep eligible blocks. Coarse scores element by
    element (f32 bound included) and the kept sets against the oracle, then the fine stage."""
    L = 100
    wl = inputs.small_workload(name="coarse_rows", seed=77, B=3, L=L, H_i=64, D_i=128,
                               index_block=64, index_keep=16, index_topk=512, q_idx_dtype="bf16",
                               key_dtype="bf16", Np=(2048, 5000, 1100), t0=0, with_attention=False)
    data = inputs.generate(wl)
    data["t0"][:] = np.array([4 * 2048 - 4 * L - 50, 4 * 5000 - 7000, 3780], dtype=np.int32)
    prob = Problem(data)
    res = run_hisa(prob)
    rows = [(b, j) for b in range(3) for j in (0, 1, 2, 17, 50, 63, 64, 98, 99)]
    check_rows(data, prob, res, rows)


def test_combine_writes_to_page_locked_host_memory():
    """The combine's output may be page-locked host memory (its device address): the kernels
    then write the results straight to the host (over NVLink-C2C on GB300). The host copy
    equals, bit for bit, the output written to device memory; the split path (few rows,
    partials in the workspace, then the merge kernel) and the single-pass path both."""
    data = v4_small("peaked", B=3, Np=(2048, 3000, 1500), seed=17)
    prob = Problem(data)
    rng = np.random.default_rng(3)
    I = np.stack([rng.choice(int(n), 512, replace=False) for n in (2048, 3000, 1500)]).astype(np.int32)
    It = torch.as_tensor(I, device="cuda")
    prob.attend(I=It)
    torch.cuda.synchronize()
    ref = prob.out.cpu()
    host_out = torch.full(tuple(prob.out.shape), 5.0, dtype=torch.float32).pin_memory()
    dptr = hb.device_pointer_of_pinned(host_out)
    prob.attend(I=It, out=hb.DevicePointer(dptr, host_out.numel()))
    torch.cuda.synchronize()
    assert prob.status() == 0
    assert torch.equal(host_out, ref)
    for b in range(3):
        P.check_attend(data, b, 0, host_out[b].numpy(), I[b])


def test_many_long_coarse_rows_in_chunks():
    """Coarse rows of more than 1024 blocks (Np over 65536 pooled rows) with more rows than a
    few: the coarse pipeline scores each row as chunks of 1024 blocks (the newest blocks' means
    appended by the chunk that holds them), each chunk selects its top blocks with their scores,
    and a merge picks the row's top blocks; a 262144-row sequence takes four chunks, two short
    sequences leave their second chunk empty. The fine stage follows as usual."""
    B = 24
    rng = np.random.default_rng(91)
    Np = [int(x) for x in rng.integers(65600, 70000, size=B)]
    Np[3], Np[11], Np[19] = 5000, 1100, 262144
    Np = tuple(Np)
    wl = inputs.small_workload(name="past_pipe", seed=91, B=B, H_i=64, D_i=128, index_block=64,
                               index_keep=16, index_topk=512, q_idx_dtype="f32", key_dtype="bf16",
                               Np=Np, with_attention=False)
    data = inputs.generate(wl)
    prob = Problem(data)
    nb = np.asarray(Np) // 64
    cs = torch.full((B, int(nb.max())), 7.0, device="cuda")
    fs = torch.full((B, 1024), 7.0, device="cuda")
    prob.block_means(first_block=np.zeros(B, np.int32))
    prob.block_filter_append(first_block=torch.as_tensor((nb - 2).astype(np.int32), device="cuda"),
                             cscores=cs)
    prob.select_topk(fscores=fs)
    torch.cuda.synchronize()
    assert prob.status() == 0
    tb, I, cs, fs = np_(prob.top_blk), np_(prob.I), np_(cs), np_(fs)
    P.check_block_means(data, np_(prob.means), np_(prob.means_off), 64)
    for b in (0, 3, 7, 11, 19, 23):
        P.check_coarse(data, b, 0, tb[b], cs[b], 64, 16)
        P.check_fine(data, b, 0, tb[b], I[b], fs[b], 64, 512)


@pytest.mark.parametrize("Np", [(41034, 5000, 65536), (30000,)], ids=["B3", "B1"])
def test_few_sequences_append_filter_select(Np):
    """A batch of a few sequences (one scoring CTA per row, most SMs idle): a 1024-block
    row, a ragged 641-block row, a short row and a single query, with the newest two blocks'
    means appended by the coarse call itself; block means, coarse and fine against the oracle,
    and a repeated coarse call on the same workspace gives the same kept blocks."""
    B = len(Np)
    wl = inputs.small_workload(name="few_sequences", seed=93, B=B, H_i=64, D_i=128,
                               index_block=64, index_keep=16, index_topk=512, q_idx_dtype="f32",
                               key_dtype="bf16", Np=Np, with_attention=False)
    data = inputs.generate(wl)
    prob = Problem(data)
    nb = np.asarray(Np) // 64
    cs = torch.full((B, int(nb.max())), 7.0, device="cuda")
    fs = torch.full((B, 1024), 7.0, device="cuda")
    prob.block_means(first_block=np.zeros(B, np.int32))
    prob.block_filter_append(first_block=torch.as_tensor((nb - 2).astype(np.int32), device="cuda"),
                             cscores=cs)
    prob.select_topk(fscores=fs)
    torch.cuda.synchronize()
    assert prob.status() == 0
    tb, I, cs, fs = np_(prob.top_blk), np_(prob.I), np_(cs), np_(fs)
    P.check_block_means(data, np_(prob.means), np_(prob.means_off), 64)
    for b in range(B):
        P.check_coarse(data, b, 0, tb[b], cs[b], 64, 16)
        P.check_fine(data, b, 0, tb[b], I[b], fs[b], 64, 512)
    prob.top_blk.fill_(-7)
    prob.block_filter()
    torch.cuda.synchronize()
    assert prob.status() == 0
    assert np.array_equal(np_(prob.top_blk), tb)


@pytest.mark.parametrize("B,L,Np", [(3, 4, (65536, 40000, 65536)), (2, 3, (40000, 38000))],
                         ids=["1024_blocks", "625_blocks"])
def test_few_long_coarse_rows_ties_and_masked_tails(B, L, Np):
    """A few long coarse rows, L = 3 or 4 query rows per sequence (one scoring CTA per row).
    Sequence 0's blocks from 120 on repeat with period 7, so groups of bit-equal block means
    run across the whole row and the lowest ids must win; sequence 1 sees all of its blocks;
    the other rows see about 312 of their blocks, so most of each row is masked. The newest
    two blocks' means are appended by the coarse call, and a repeated call gives the same
    kept blocks."""
    wl = inputs.small_workload(name="few_long_rows", seed=95, B=B, L=L, H_i=64, D_i=128, index_block=64,
                               index_keep=16, index_topk=512, q_idx_dtype="f32", key_dtype="bf16",
                               Np=Np, t0=80000, with_attention=False)
    data = inputs.generate(wl)
    data["t0"][1] = 4 * Np[1]                         # every block of sequence 1 visible
    keys, k0 = data["keys"], int(data["key_off"][0])
    r = np.arange(120 * 64, Np[0])
    keys[k0 + r] = keys[k0 + 120 * 64 + ((r // 64 - 120) % 7) * 64 + r % 64]
    prob = Problem(data)
    nb = np.asarray(Np) // 64
    cs = torch.full((B * L, int(nb.max())), 7.0, device="cuda")
    fs = torch.full((B * L, 1024), 7.0, device="cuda")
    prob.block_means(first_block=np.zeros(B, np.int32))
    prob.block_filter_append(first_block=torch.as_tensor((nb - 2).astype(np.int32), device="cuda"),
                             cscores=cs)
    prob.select_topk(fscores=fs)
    torch.cuda.synchronize()
    assert prob.status() == 0
    tb, I, cs, fs = np_(prob.top_blk), np_(prob.I), np_(cs), np_(fs)
    P.check_block_means(data, np_(prob.means), np_(prob.means_off), 64)
    for b in range(B):
        s = P.seq(data, b)
        for j in range(L):
            row = b * L + j
            P.check_coarse(data, b, j, tb[row], cs[row], 64, 16)
            P.check_fine(data, b, j, tb[row], I[row], fs[row], 64, 512)
            if b == 0:                                # exact ties: the oracle's set itself
                V = O.visible_len(s["t0"] + j, wl.r, s["Np"])
                _, c_top = O.hisa_coarse(data["q_idx"][b, j], data["w"][b, j],
                                         O.block_means(s["keys"], 64), 16, 64, V)
                assert set(tb[row].tolist()) == set(c_top.tolist()), f"top_blk[{row}]"
    prob.top_blk.fill_(-7)
    prob.block_filter()
    torch.cuda.synchronize()
    assert prob.status() == 0
    assert np.array_equal(np_(prob.top_blk), tb)


@pytest.mark.parametrize("case", ["tc_rows", "tc_split", "simt"])
def test_bf16_output_is_the_f32_output_rounded_once(case):
    """hisa_attn_desc.out_dtype = HISA_BF16: the combine's f32 result rounded to nearest even
    once (bit for bit the f32 output of the same call rounded), within the widened bound of
    the oracle. tc_rows: 160 V4-shape rows, one item per row (the tensor-core epilogue);
    tc_split: 3 rows split over CTAs (the merge kernel writes out); simt: f32 KV on the CUDA
    cores."""
    if case == "simt":
        data = small(B=2, Np=(300, 700), seed=17, kv_dtype="f32", key_dtype="f32")
        k = 32
    else:
        B = 160 if case == "tc_rows" else 3
        rng = np.random.default_rng(18)
        Np = tuple(int(x) for x in rng.integers(600, 1500, size=B))
        data = v4_small("peaked", B=B, Np=Np, seed=18)
        k = 512
    B = data["wl"].B
    f32 = Problem(data)
    b16 = Problem(data, out_dtype="bf16")
    rng = np.random.default_rng(19)
    I = np.stack([rng.choice(int(n), min(k, int(n)), replace=False).tolist() + [-1] * (k - min(k, int(n)))
                  for n in data["Np"]]).astype(np.int32)
    It = torch.as_tensor(I, device="cuda")
    f32.attend(I=It)
    b16.attend(I=It)
    torch.cuda.synchronize()
    assert f32.status() == 0 and b16.status() == 0
    assert b16.out.dtype == torch.bfloat16
    want = f32.out.to(torch.bfloat16)                     # round to nearest even
    assert torch.equal(b16.out.view(torch.int16), want.view(torch.int16))
    got = b16.out.view(torch.int16).cpu().numpy().view(np.uint16)
    for b in sorted({0, 1, B - 1}):
        P.check_attend(data, b, 0, got[b], I[b], out_bf16=True)

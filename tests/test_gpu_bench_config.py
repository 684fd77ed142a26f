"""GPU parity in the launch configuration the benchmark times: 304 V4-Flash-shaped decode
sequences per batch (Np = 32768 pooled rows each, bf16 keys and KV, f32 indexer q), drawn on
the device exactly as the benchmark draws them, the step (newest block means appended inside
the coarse filter, fine top-k and combine chained to the call before them) captured as one
graph for batch A then batch B, replayed twice. Two rows per scoring CTA; sampled rows of
batch A (the first and last CTAs' two rows each, and rows in between) are checked against the
oracle on host copies of their sequences, and the two replays must agree bit for bit.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from deepseek_sparse_attention_hisa_gb300 import binding as hb  # noqa: E402
from deepseek_sparse_attention_hisa_gb300 import inputs  # noqa: E402
from deepseek_sparse_attention_hisa_gb300.problem import Problem  # noqa: E402
from oracle import parity as P  # noqa: E402

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")]

R, NP = 304, 32768
SAMPLED = (0, 1, 150, 151, 152, 153, 250, 302, 303)


@pytest.fixture(scope="module", autouse=True)
def _built():
    from deepseek_sparse_attention_hisa_gb300 import build
    build.build_library()
    hb.lib()


def _host(t):
    """A device tensor as the oracle's numpy form (bf16 as uint16 bit patterns)."""
    t = t.detach().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def _host_subset(data, bwl, rows):
    """The sampled sequences of a device-drawn batch as a host data dict of their own."""
    key_off = np.asarray(data["key_off"], dtype=np.int64)
    sl = [slice(int(key_off[b]), int(key_off[b + 1])) for b in rows]
    Np = np.array([s.stop - s.start for s in sl], dtype=np.int64)
    off = np.zeros(len(rows) + 1, dtype=np.int64)
    off[1:] = np.cumsum(Np)
    idx = torch.as_tensor(list(rows), device=data["q_idx"].device)
    sub = dict(wl=bwl.replace(B=len(rows)), Np=Np, key_off=off,
               t0=np.asarray(data["t0"])[list(rows)])
    sub["keys"] = np.concatenate([_host(data["keys"][s]) for s in sl])
    sub["pooled_kv"] = np.concatenate([_host(data["pooled_kv"][s]) for s in sl])
    for name in ("q_idx", "w", "q_attn", "local_kv"):
        sub[name] = _host(data[name].index_select(0, idx))
    sub["local_len"] = np.asarray(data["local_len"])[list(rows)]
    sub["local_pos0"] = np.asarray(data["local_pos0"])[list(rows)]
    sub["sinks"] = _host(data["sinks"])
    return sub


def test_bench_step_sampled_rows_against_the_oracle():
    dev = "cuda:0"
    bwl = inputs.WORKLOADS["v4flash_decode"].replace(B=R, Np=(NP,))
    data = inputs.generate_device(bwl, device=dev, seed=1000)
    prob = Problem(data, device=dev)
    prob_b = Problem(inputs.generate_device(bwl, device=dev, seed=1100), device=dev)
    nb = int(prob.nb[0])
    newest = torch.as_tensor(np.full(R, nb - 1, dtype=np.int32), device=dev)
    prob.block_means()
    prob_b.block_means()
    torch.cuda.synchronize()

    def step(pr, s):
        pr.block_filter_append(first_block=newest, stream=s)
        pr.select_topk(stream=s, chained=True)
        pr.attend(stream=s, chained=True)

    s = torch.cuda.Stream(device=dev)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step(prob, s)                                # eager warm-up: attributes, lazy init
        step(prob_b, s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step(prob, s)
        step(prob_b, s)
    outs = []
    for _ in range(2):
        prob.top_blk.fill_(-7)
        prob.I.fill_(-7)
        prob.out.fill_(0.0)
        with torch.cuda.stream(s):
            g.replay()
        s.synchronize()
        assert prob.status() == 0 and prob_b.status() == 0
        outs.append((prob.top_blk.cpu().numpy().copy(), prob.I.cpu().numpy().copy(),
                     prob.out.cpu().numpy().copy()))
    for a, b in zip(outs[0], outs[1]):
        assert np.array_equal(a, b), "replays differ"
    tb, I, out = outs[0]
    assert np.all(np.diff(np.sort(I, axis=1), axis=1) > 0)     # distinct ids in every row

    sub = _host_subset(data, bwl, SAMPLED)
    m_off = np.asarray(prob.means_off.cpu().numpy(), dtype=np.int64)
    gm = prob.means.cpu().numpy()
    sub_means = np.concatenate([gm[m_off[b]:m_off[b + 1]] for b in SAMPLED])
    sub_off = np.zeros(len(SAMPLED) + 1, dtype=np.int64)
    sub_off[1:] = np.cumsum([m_off[b + 1] - m_off[b] for b in SAMPLED])
    P.check_block_means(sub, sub_means, sub_off, 64)
    for i, b in enumerate(SAMPLED):
        P.check_coarse(sub, i, 0, tb[b], None, 64, 16)
        P.check_fine(sub, i, 0, tb[b], I[b], None, 64, 512)
        P.check_attend(sub, i, 0, out[b], I[b])

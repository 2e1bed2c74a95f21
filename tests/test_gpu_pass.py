"""The whole verify pass of the benchmark against the oracle.

bench.py times one CUDA graph per pass: the 129 activation kernels and GEMMs
of the 9B-class decoder (q/k/v and gate/up fused, programmatic dependent
launch between kernels) and the acceptance of the 16-node draft tree from the
LM head's logits.  Here the same graph is captured and replayed once, then
for every GEMM a seeded sample of 64 output channels (plus the first and last
channel of every fused part) is recomputed by the oracle from the same inputs
and weights, and the acceptance outputs are recomputed from the GPU's logits.
"""
import numpy as np
import pytest
import torch

import bench
import oracle
from quantized_speculative_verify_gb300 import hq, synth
from tolerance import assert_close, strict_fraction

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def replayed_pass():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    hq.load()
    vp = bench.VerifyPass(torch, hq, synth, torch.device(DEV), fuse_qkv=True, pdl=True)
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        vp.launch()  # eager warm-up (launch set-up happens before capture)
    stream.synchronize()
    for y in vp.ys:
        y.fill_(float("nan"))  # every output must be written by the replay
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        vp.launch()
    for y in vp.ys:
        y.fill_(float("nan"))
    graph.replay()
    torch.cuda.synchronize()
    assert hq.hq_workspace_status(vp.ws) == hq.HQ_OK
    yield vp
    del vp
    torch.cuda.empty_cache()


def test_every_gemm_output_of_the_pass(replayed_pass):
    vp = replayed_pass
    rng = np.random.default_rng(7)
    fractions = []
    for ii, li in vp.plan:
        name, K, parts = vp.gemms[li]
        X = vp.inputs[ii][2].cpu().numpy()
        s_host = vp.inputs[ii][6]
        Y = vp.ys[li].cpu().numpy()
        assert not np.isnan(Y).any(), name
        Ws = vp.part_weights(li, DEV)
        off = 0
        for (pname, n, _), W in zip(parts, Ws):
            idx = np.unique(np.concatenate([rng.choice(n, size=min(64, n), replace=False), [0, n - 1]]))
            rows = W[torch.from_numpy(idx).to(DEV)].cpu().numpy()
            ref = oracle.verify_linear(X, rows, vp.G, vp.fmt, s_host)
            fractions.append(assert_close(Y[:, off + idx], ref))
            off += n
        del Ws
    print(f"pass: {len(fractions)} parts checked; elementwise 1e-6 + 1e-5|Y| met by "
          f"{min(fractions):.5f} (worst part) .. {np.mean(fractions):.5f} (mean) of the sampled outputs")


def test_acceptance_of_the_pass(replayed_pass):
    vp = replayed_pass
    logits = vp.ys[-1].cpu().numpy()
    g_ref = oracle.argmax_rows(logits)
    parent = vp.parent.cpu().numpy()
    tokens = vp.tokens.cpu().numpy()
    path_ref, n_ref, bonus_ref = oracle.tree_accept(g_ref, parent, tokens)
    assert np.array_equal(vp.greedy.cpu().numpy(), g_ref)
    out = vp.accept_out.cpu().numpy()
    assert int(out[0]) == n_ref and int(out[1]) == bonus_ref
    assert np.array_equal(vp.path.cpu().numpy()[:n_ref], path_ref)

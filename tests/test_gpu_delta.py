"""Rollback-free DeltaNet tree pass and its commit on the GPU, against the
CPU oracle.

Page "Karpathy's Trick for Faster Local LLMs Finally Has Proper Tooling",
section "Verifying a draft tree without restoring model state" (the gated
delta rule is the published one).  Tolerance, from the fp32 arithmetic: a
node with a root path of n steps goes through n warp dot products of 128
terms (7 levels of pairwise sums over 4-term partials) and 2 rounded vector
operations each, then one 128-term product with the committed state (16
sequential terms and 3 levels); with unit keys, alpha <= 1 and beta <= 1 every
step is a contraction, so |error| <= (11 n + 20) * 2^-24 * scale with
scale = max_r ||S_c[r]||_1 * ||q||_2 + sum_path beta ||q||_2 max|v|.  The
commit applies n + 1 such steps to every state row: |error| <= (n + 2) * 16 *
2^-24 * (max_r ||S_c[r]||_2 + sum_steps beta max|v|).
"""
import numpy as np
import pytest
import torch

import oracle
from quantized_speculative_verify_gb300 import hq

pytestmark = pytest.mark.gpu
DEV = "cuda"
U = 2.0 ** -24
D = hq.HQ_DELTA_HEAD_DIM


def _inputs(seed, M, H, sscale=0.3):
    rng = np.random.default_rng(seed)
    st = (rng.standard_normal((H, D, D)) * sscale).astype(np.float32)
    q = rng.standard_normal((M, H, D)).astype(np.float32)
    k = rng.standard_normal((M, H, D))
    k = (k / np.linalg.norm(k, axis=2, keepdims=True)).astype(np.float32)
    v = rng.standard_normal((M, H, D)).astype(np.float32)
    al = rng.uniform(0.6, 1.0, (M, H)).astype(np.float32)
    be = rng.uniform(0.0, 1.0, (M, H)).astype(np.float32)
    return st, q, k, v, al, be


def _tree(seed, M, width=3):
    rng = np.random.default_rng(seed)
    par = np.zeros(M, dtype=np.int32)
    for i in range(1, M):
        par[i] = rng.integers(max(0, i - width), i)
    return par


def _path(parent, i):
    chain = [i]
    while chain[-1] > 0 and 0 <= parent[chain[-1]] < chain[-1]:
        chain.append(int(parent[chain[-1]]))
    return chain


def _dev(*xs):
    return [torch.from_numpy(np.ascontiguousarray(x)).to(DEV) for x in xs]


def _check_tree(st, q, k, v, al, be, parent, got):
    ref = oracle.delta_tree(st, q, k, v, al, be, parent, openmp=True)
    srow = np.abs(st.astype(np.float64)).sum(axis=2).max(axis=1)  # [H]
    for i in range(q.shape[0]):
        chain = _path(parent, i)
        qn = np.linalg.norm(q[i].astype(np.float64), axis=1)      # [H]
        vmax = np.abs(v[chain].astype(np.float64)).max(axis=(0, 2))
        bsum = be[chain].astype(np.float64).sum(axis=0)
        scale = srow * qn + bsum * qn * vmax
        tol = (11 * len(chain) + 20) * U * scale
        err = np.abs(got[i] - ref[i]).max(axis=1)
        assert (err <= tol).all(), f"node {i}: err {err.max():.3e} tol {tol.min():.3e}"
    return ref


CASES = [(1, 1), (2, 4), (7, 3), (16, 32), (31, 8), (64, 2), (128, 1)]


@pytest.mark.parametrize("M,H", CASES)
def test_delta_tree_matches_oracle(M, H):
    st, q, k, v, al, be = _inputs(M * 10 + H, M, H)
    parent = _tree(M + H, M)
    args = _dev(st, q, k, v, al, be, parent)
    out = hq.delta_tree(*args)
    torch.cuda.synchronize()
    _check_tree(st, q, k, v, al, be, parent, out.cpu().numpy().astype(np.float64))


def test_delta_tree_deep_chain_and_star():
    for parent in (np.maximum(np.arange(128, dtype=np.int32) - 1, 0), np.zeros(40, dtype=np.int32)):
        M = parent.shape[0]
        st, q, k, v, al, be = _inputs(M, M, 2)
        out = hq.delta_tree(*_dev(st, q, k, v, al, be, parent), flags=hq.HQ_LAUNCH_PDL)
        torch.cuda.synchronize()
        _check_tree(st, q, k, v, al, be, parent, out.cpu().numpy().astype(np.float64))


def test_delta_tree_invalid_parent_starts_from_the_committed_state():
    st, q, k, v, al, be = _inputs(3, 6, 4)
    parent = np.array([0, 0, 4, 2, -1, 3], dtype=np.int32)
    out = hq.delta_tree(*_dev(st, q, k, v, al, be, parent))
    torch.cuda.synchronize()
    _check_tree(st, q, k, v, al, be, parent, out.cpu().numpy().astype(np.float64))


def test_delta_tree_leaves_the_committed_state_untouched():
    st, q, k, v, al, be = _inputs(4, 16, 8)
    parent = _tree(4, 16)
    args = _dev(st, q, k, v, al, be, parent)
    hq.delta_tree(*args)
    torch.cuda.synchronize()
    assert np.array_equal(args[0].cpu().numpy(), st)


def test_delta_tree_full_size_layer():
    """The 9B-class DeltaNet layer of the benchmark: 16 tree nodes, 32 heads
    of 128; every output against the oracle."""
    M, H = 16, 32
    st, q, k, v, al, be = _inputs(5, M, H)
    parent = np.array([0, 0, 1, 2, 3, 0, 5, 6, 1, 8, 2, 10, 11, 0, 13, 14], dtype=np.int32)
    out = hq.delta_tree(*_dev(st, q, k, v, al, be, parent), flags=hq.HQ_LAUNCH_PDL)
    torch.cuda.synchronize()
    _check_tree(st, q, k, v, al, be, parent, out.cpu().numpy().astype(np.float64))


@pytest.mark.parametrize("n", [3, 0, -1, 15])
def test_delta_commit_matches_oracle(n):
    M, H = 16, 8
    st, q, k, v, al, be = _inputs(50 + n, M, H)
    path = np.full(M, -1, dtype=np.int32)
    chain = {3: [2, 6, 9], 15: list(range(1, 16))}.get(n, [])
    path[: len(chain)] = chain
    std, kd, vd, ald, bed, pd = _dev(st, k, v, al, be, path)
    hq.delta_commit(std, kd, vd, ald, bed, pd, torch.tensor([n], dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    got = std.cpu().numpy().astype(np.float64)
    ref = oracle.delta_commit(st, k, v, al, be, path[: max(n, 0)], n)
    if n < 0:
        assert np.array_equal(got, st.astype(np.float64))
        return
    steps = [0] + chain[:n]
    scale = np.linalg.norm(st.astype(np.float64), axis=2).max() + \
        (be[steps].astype(np.float64) * np.abs(v[steps]).max(axis=2)).sum(axis=0).max()
    assert np.abs(got - ref).max() <= (n + 2) * 16 * U * scale


def test_accept_then_commit_then_continue():
    """One verify step end to end: tree outputs, acceptance from logits, state
    commit; the committed state answers the accepted node's query as the tree
    pass did."""
    M, H, V = 8, 4, 50
    st, q, k, v, al, be = _inputs(60, M, H)
    parent = np.array([0, 0, 1, 2, 0, 4, 2, 6], dtype=np.int32)
    rng = np.random.default_rng(61)
    logits = rng.standard_normal((M, V)).astype(np.float32)
    g = logits.argmax(axis=1).astype(np.int32)
    tokens = np.array([0] + [g[parent[i]] if i in (1, 2, 3) else (g[parent[i]] + 1) % V for i in range(1, M)],
                      dtype=np.int32)
    std, qd, kd, vd, ald, bed, pard = _dev(st, q, k, v, al, be, parent)
    out = hq.delta_tree(std, qd, kd, vd, ald, bed, pard)
    _, pathd, acc = hq.tree_accept(torch.from_numpy(logits).to(DEV), pard, torch.from_numpy(tokens).to(DEV))
    hq.delta_commit(std, kd, vd, ald, bed, pathd, acc[0:1])
    torch.cuda.synchronize()
    rpath, rn, _ = oracle.tree_accept(g, parent, tokens)
    assert int(acc[0]) == rn == 3 and list(rpath) == [1, 2, 3]
    S = std.cpu().numpy().astype(np.float64)
    again = np.einsum("hrc,hc->hr", S, q[3].astype(np.float64))
    np.testing.assert_allclose(again, out.cpu().numpy()[3], rtol=0, atol=1e-4)

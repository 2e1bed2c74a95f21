"""Tree-masked verify attention and the accepted-path KV commit on the GPU,
against the CPU oracle.

Page "Karpathy's Trick for Faster Local LLMs Finally Has Proper Tooling",
section "Verifying a draft tree without restoring model state".  Tolerance:
the kernel rounds the softmax probabilities to fp16 for the product with V,
which perturbs each weight by at most 2^-11 relative, so
|out - exact| <= 2^-11 * max|v|; fp32 score, exp2 and merge rounding add far
less (bounded here by 1e-4 * max|v|).  The commit is a copy: bit-exact.
"""
import numpy as np
import pytest
import torch

import oracle
from quantized_speculative_verify_gb300 import hq

pytestmark = pytest.mark.gpu
DEV = "cuda"
TOL = 2.0 ** -11 + 1e-4


def _inputs(seed, M, Hq, Hkv, L, extra=0, qscale=1.0):
    rng = np.random.default_rng(seed)
    D = hq.HQ_ATTN_HEAD_DIM
    q = (rng.standard_normal((M, Hq, D)) * qscale).astype(np.float16)
    k = rng.standard_normal((Hkv, L + M + extra, D)).astype(np.float16)
    v = rng.standard_normal((Hkv, L + M + extra, D)).astype(np.float16)
    return q, k, v


def _random_tree(seed, M, width=3):
    rng = np.random.default_rng(seed)
    par = np.zeros(M, dtype=np.int32)
    for i in range(1, M):
        par[i] = rng.integers(max(0, i - width), i)
    return par


def _gpu(q, k, v, L, parent, scale, flags=0):
    qd, kd, vd = (torch.from_numpy(x).to(DEV) for x in (q, k, v))
    pd = torch.from_numpy(parent).to(DEV)
    ws = torch.zeros(hq.hq_tree_attention_workspace_bytes(k.shape[0]), dtype=torch.uint8, device=DEV)
    out = hq.tree_attention(qd, kd, vd, L, pd, scale, workspace=ws, flags=flags)
    torch.cuda.synchronize()
    assert hq.hq_workspace_status(ws) == hq.HQ_OK
    return out.cpu().numpy().astype(np.float64)


def _check(got, ref, v):
    vmax = float(np.abs(v.astype(np.float64)).max())
    err = np.abs(got - ref)
    assert np.isfinite(got).all()
    assert err.max() <= TOL * vmax, f"max err {err.max():.3e} > {TOL * vmax:.3e}"
    return err


CASES = [  # M, Hq, Hkv, L
    (1, 8, 8, 0), (1, 32, 8, 1), (2, 4, 1, 0), (5, 8, 2, 63), (16, 32, 8, 64), (16, 32, 8, 65),
    (16, 32, 8, 1000), (31, 16, 4, 300), (64, 8, 8, 129), (128, 32, 8, 40), (128, 16, 1, 7), (17, 64, 4, 200),
    (3, 32, 32, 5000), (5, 64, 2, 100), (3, 64, 1, 300), (16, 32, 8, 56), (9, 16, 8, 8),
]


@pytest.mark.parametrize("M,Hq,Hkv,L", CASES)
def test_tree_attention_matches_oracle(M, Hq, Hkv, L):
    seed = M * 1000 + Hq * 10 + L
    q, k, v = _inputs(seed, M, Hq, Hkv, L, extra=M % 3)
    parent = _random_tree(seed, M)
    scale = 1.0 / np.sqrt(hq.HQ_ATTN_HEAD_DIM)
    got = _gpu(q, k, v, L, parent, scale)
    ref = oracle.tree_attention(q, k, v, L, parent, scale, openmp=True)
    _check(got, ref, v)


def test_tree_attention_peaked_softmax_and_shapes():
    """Large scores (one key dominates) and the degenerate trees: chain and star."""
    M, Hq, Hkv, L = 24, 16, 4, 333
    q, k, v = _inputs(5, M, Hq, Hkv, L, qscale=4.0)
    for parent in (np.maximum(np.arange(M, dtype=np.int32) - 1, 0), np.zeros(M, dtype=np.int32)):
        got = _gpu(q, k, v, L, parent, 0.3)
        _check(got, oracle.tree_attention(q, k, v, L, parent, 0.3, openmp=True), v)


def test_tree_attention_invalid_parent_ends_the_walk():
    M, Hq, Hkv, L = 6, 8, 2, 70
    q, k, v = _inputs(6, M, Hq, Hkv, L)
    parent = np.array([0, 0, 5, 2, -3, 4], dtype=np.int32)
    got = _gpu(q, k, v, L, parent, 0.1)
    _check(got, oracle.tree_attention(q, k, v, L, parent, 0.1), v)


def test_tree_attention_single_visible_key_is_exact():
    """L = 0, M = 1: the root sees only itself, the output is its value row."""
    q, k, v = _inputs(7, 1, 8, 2, 0)
    got = _gpu(q, k, v, 0, np.zeros(1, dtype=np.int32), 0.2)
    ref = np.repeat(v[:, 0].astype(np.float64), 4, axis=0)[None]
    assert np.array_equal(got, ref)


def test_tree_attention_full_size_decoder_layer():
    """The 9B-class attention layer the benchmark times: 16 tree nodes, 32
    query heads over 8 key/value heads, 8192 committed positions; every
    output against the oracle, with programmatic dependent launch on."""
    M, Hq, Hkv, L = 16, 32, 8, 8192
    q, k, v = _inputs(8, M, Hq, Hkv, L, extra=16)
    parent = np.array([0, 0, 1, 2, 3, 0, 5, 6, 1, 8, 2, 10, 11, 0, 13, 14], dtype=np.int32)
    scale = 1.0 / np.sqrt(hq.HQ_ATTN_HEAD_DIM)
    got = _gpu(q, k, v, L, parent, scale, flags=hq.HQ_LAUNCH_PDL)
    ref = oracle.tree_attention(q, k, v, L, parent, scale, openmp=True)
    err = _check(got, ref, v)
    assert np.median(err) < 1e-4


def test_tree_attention_repeated_calls_share_a_workspace():
    ws = torch.zeros(hq.hq_tree_attention_workspace_bytes(4), dtype=torch.uint8, device=DEV)
    for i, (M, Hq, L) in enumerate([(16, 16, 500), (3, 8, 0), (40, 32, 2000)]):
        q, k, v = _inputs(20 + i, M, Hq, 4, L)
        parent = _random_tree(i, M)
        out = hq.tree_attention(torch.from_numpy(q).to(DEV), torch.from_numpy(k).to(DEV),
                                torch.from_numpy(v).to(DEV), L, torch.from_numpy(parent).to(DEV), 0.125,
                                workspace=ws)
        torch.cuda.synchronize()
        _check(out.cpu().numpy().astype(np.float64), oracle.tree_attention(q, k, v, L, parent, 0.125), v)
    assert hq.hq_workspace_status(ws) == hq.HQ_OK


@pytest.mark.parametrize("n", [3, 0, -1, 1, 15])
def test_tree_commit_kv_matches_oracle(n):
    rng = np.random.default_rng(30 + n)
    Hkv, L, M, D = 8, 100, 16, hq.HQ_ATTN_HEAD_DIM
    cap = L + M + 4
    k = rng.standard_normal((Hkv, cap, D)).astype(np.float16)
    v = rng.standard_normal((Hkv, cap, D)).astype(np.float16)
    path = np.full(M, -1, dtype=np.int32)
    chain = {3: [2, 6, 9], 1: [5], 15: list(range(1, 16))}.get(n, [])
    path[: len(chain)] = chain
    kd, vd = torch.from_numpy(k).to(DEV), torch.from_numpy(v).to(DEV)
    hq.tree_commit_kv(kd, vd, L, M, torch.from_numpy(path).to(DEV),
                      torch.tensor([n], dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    rk, rv = oracle.tree_commit_kv(k, v, L, path[: max(n, 0)], n)
    assert np.array_equal(kd.cpu().numpy().view(np.uint16), rk.view(np.uint16))
    assert np.array_equal(vd.cpu().numpy().view(np.uint16), rv.view(np.uint16))


def test_accept_then_commit_then_attend_again():
    """One verify step end to end on the GPU: attention over the tree, greedy
    acceptance from logits, commit of the accepted path; the next step's root
    then attends to the committed prefix exactly as if the accepted tokens had
    been decoded one by one (checked against the oracle with a chain)."""
    M, Hq, Hkv, L, V = 8, 16, 4, 50, 64
    D = hq.HQ_ATTN_HEAD_DIM
    cap = L + 2 * M
    q, k, v = _inputs(40, M, Hq, Hkv, L, extra=M)
    parent = np.array([0, 0, 1, 2, 0, 4, 2, 6], dtype=np.int32)
    rng = np.random.default_rng(41)
    logits = rng.standard_normal((M, V)).astype(np.float32)
    g = logits.argmax(axis=1).astype(np.int32)
    tokens = np.zeros(M, dtype=np.int32)
    for i in range(1, M):
        tokens[i] = g[parent[i]] if i in (1, 2, 6, 7) else (g[parent[i]] + 1) % V
    kd, vd = torch.from_numpy(k).to(DEV), torch.from_numpy(v).to(DEV)
    _, pathd, out2 = hq.tree_accept(torch.from_numpy(logits).to(DEV), torch.from_numpy(parent).to(DEV),
                                    torch.from_numpy(tokens).to(DEV))
    hq.tree_commit_kv(kd, vd, L, M, pathd, out2[0:1])
    torch.cuda.synchronize()
    rpath, rn, _ = oracle.tree_accept(g, parent, tokens)
    assert int(out2[0]) == rn == 4 and list(rpath) == [1, 2, 6, 7]
    rk, rv = oracle.tree_commit_kv(k, v, L, rpath, rn)
    assert np.array_equal(kd.cpu().numpy().view(np.uint16), rk.view(np.uint16))
    # the accepted prefix now sits at [L, L + 1 + rn): a fresh root there sees it as committed cache
    L2 = L + 1 + rn
    q2, _, _ = _inputs(42, 1, Hq, Hkv, 0)
    k3, v3 = rk.copy(), rv.copy()
    got = _gpu(q2, k3, v3, L2, np.zeros(1, dtype=np.int32), 0.09)
    _check(got, oracle.tree_attention(q2, k3, v3, L2, np.zeros(1, dtype=np.int32), 0.09), v3[:, : L2 + 1])

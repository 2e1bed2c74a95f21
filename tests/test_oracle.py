"""Pins of the CPU oracle against facts that do not come from the oracle.

Each test checks one oracle function against something fixed independently:
a library routine (scipy's Hadamard matrix, numpy int64 matmul), a closed
form, a hand-derived worked example under tests/golden/, or an error bound
that follows from the arithmetic.  Method source: page "Karpathy's Trick for
Faster Local LLMs Finally Has Proper Tooling", section "How Uzu optimizes
bytes and tokens per pass".
"""
import os
import struct

import numpy as np
import pytest
import scipy.linalg

import oracle
from quantized_speculative_verify_gb300 import synth

C_BITS = 0x3E3504F3
C = np.float32(struct.unpack("<f", struct.pack("<I", C_BITS))[0])
EPS32 = 2.0 ** -24


def f32_bits(x) -> int:
    return struct.unpack("<I", struct.pack("<f", float(x)))[0]


def sylvester(n=32):
    i = np.arange(n)
    pc = np.vectorize(lambda v: bin(int(v)).count("1"))(i[:, None] & i[None, :])
    return np.where(pc % 2 == 0, 1, -1).astype(np.int64)


# ---------------------------------------------------------------- signs ---
def test_splitmix64_published_vector(golden_dir):
    lines = [l.split() for l in open(os.path.join(golden_dir, "splitmix64.txt")) if l.strip() and l[0] != "#"]
    seed = int(lines[0][1])
    expect = [int(l[0]) for l in lines[1:]]
    got = [int(v) for v in oracle.splitmix64(seed, len(expect))]
    assert got == expect


def test_sign_packing_follows_top_bits():
    K = 256
    raw = oracle.splitmix64(77, K)
    signs = oracle.make_signs(77, K)
    for i in range(K):
        bit = (int(signs[i // 32]) >> (i % 32)) & 1
        assert bit == int(raw[i]) >> 63
    # roughly half the signs are negative
    assert 0.35 < np.mean(oracle.signs_to_pm1(signs, K) < 0) < 0.65


def test_make_signs_rejects_bad_K():
    with pytest.raises(ValueError):
        oracle.make_signs(1, 48)


# ------------------------------------------------------------- Hadamard ---
def oracle_hadamard_matrix():
    """Column j of the butterfly applied to unit vector e_j, as an int matrix."""
    H = np.zeros((32, 32), dtype=np.int64)
    for j in range(32):
        e = np.zeros(32, dtype=np.float32)
        e[j] = 1.0
        H[j] = oracle.fwht32(e).astype(np.int64)
    return H


def test_butterfly_is_sylvester_hadamard():
    H = oracle_hadamard_matrix()
    assert np.array_equal(H, scipy.linalg.hadamard(32).astype(np.int64))
    assert np.array_equal(H, sylvester(32))
    assert set(np.unique(H)) == {-1, 1}


def test_hadamard_orthogonal():
    H = oracle_hadamard_matrix()
    assert np.array_equal(H @ H.T, 32 * np.eye(32, dtype=np.int64))


def test_butterfly_equals_matrix_product_on_integers():
    rng = np.random.default_rng(5)
    H = scipy.linalg.hadamard(32).astype(np.int64)
    for _ in range(50):
        v = rng.integers(-(2 ** 18), 2 ** 18, size=32)
        got = oracle.fwht32(v.astype(np.float32))
        assert np.array_equal(got.astype(np.int64), v @ H)


def test_butterfly_twice_is_32_identity():
    rng = np.random.default_rng(6)
    for _ in range(20):
        v = rng.integers(-(2 ** 12), 2 ** 12, size=32).astype(np.float32)
        assert np.array_equal(oracle.fwht32(oracle.fwht32(v)), 32 * v)


def fp64_rotation(V, signs):
    """(V o s) blockdiag(H) / sqrt(32) in fp64 with scipy's Hadamard matrix."""
    V = np.atleast_2d(np.asarray(V, dtype=np.float64))
    R_, K = V.shape
    s = oracle.signs_to_pm1(signs, K)
    H = scipy.linalg.hadamard(32).astype(np.float64)
    return ((V * s).reshape(R_, K // 32, 32) @ H / np.sqrt(32.0)).reshape(R_, K)


def test_rotation_matches_fp64_definition():
    K = 512
    signs = oracle.make_signs(11, K)
    X = synth.activations(8, K, seed=3, outlier_channels=2).numpy()
    got = oracle.rotate(X, signs).astype(np.float64)
    ref = fp64_rotation(X, signs)
    l1 = np.abs(X.astype(np.float64)).reshape(8, K // 32, 32).sum(-1)
    bound = (6 * EPS32 * l1 + 1e-30)[:, :, None] * np.ones((1, 1, 32))
    assert np.all(np.abs(got - ref).reshape(8, K // 32, 32) <= bound)


def test_rotation_inverse_roundtrip():
    K = 1024
    signs = oracle.make_signs(12, K)
    W = synth.weights(16, K, seed=4).numpy()
    back = oracle.rotate_inverse(oracle.rotate(W, signs), signs).astype(np.float64)
    l1 = np.abs(W.astype(np.float64)).reshape(16, K // 32, 32).sum(-1)[:, :, None]
    err = np.abs(back - W).reshape(16, K // 32, 32)
    assert np.all(err <= 14 * EPS32 * l1)
    # the inverse undoes the signs too: without them it would not round-trip
    assert np.max(err) < 1e-6


def test_rotation_preserves_product():
    K = 2048
    signs = oracle.make_signs(13, K)
    X = synth.activations(16, K, seed=5, outlier_channels=2).numpy()
    W = synth.weights(64, K, seed=6).numpy()
    ref = X.astype(np.float64) @ W.astype(np.float64).T
    rot = oracle.rotate(X, signs).astype(np.float64) @ oracle.rotate(W, signs).astype(np.float64).T
    assert np.linalg.norm(rot - ref) / np.linalg.norm(ref) <= 1e-5


def test_outlier_spreading_golden(golden_dir):
    cases = [l.split() for l in open(os.path.join(golden_dir, "outlier_spread.txt")) if l.startswith("case")]
    assert len(cases) == 3
    for _, K, j, t, sbit, mag_hex, pattern in cases:
        K, j, t, sbit, mag = int(K), int(j), float(t), int(sbit), int(mag_hex, 16)
        signs = np.zeros(K // 32, dtype=np.uint32)
        if sbit:
            signs[j // 32] |= np.uint32(1 << (j % 32))
        v = np.zeros(K, dtype=np.float32)
        v[j] = t
        u = oracle.rotate(v, signs)[0]
        b = j // 32
        block = u[b * 32:(b + 1) * 32]
        for i in range(32):
            assert f32_bits(abs(block[i])) == mag
            assert (block[i] > 0) == (pattern[i] == "+")
        rest = np.concatenate([u[: b * 32], u[(b + 1) * 32:]])
        assert np.all(rest == 0.0)
        # the outlier's magnitude is spread: every entry is |t| / sqrt(32)
        assert np.allclose(np.abs(block), abs(t) / np.sqrt(32.0), rtol=1e-7)


# ----------------------------------------------------------- quantizers ---
def parse_quant_golden(golden_dir):
    out = []
    for line in open(os.path.join(golden_dir, "quant_groups.txt")):
        if not line.strip() or line.startswith("#"):
            continue
        kind, rest = line.split(None, 1)
        parts = [p.split() for p in rest.split("|")]
        out.append((kind, parts))
    return out


def test_quantizers_golden(golden_dir):
    cases = parse_quant_golden(golden_dir)
    kinds = {k for k, _ in cases}
    assert kinds == {"asym4", "sym8", "act"}
    for kind, parts in cases:
        w = np.array([float(v) for v in parts[0]], dtype=np.float32)
        if kind == "asym4":
            q, s, z = oracle.quant_group_asym4(w)
            assert f32_bits(s) == f32_bits(np.float32(parts[1][0])), (w, s)
            assert z == int(parts[1][1]), (w, z)
            assert q.tolist() == [int(v) for v in parts[2]], (w, q)
        elif kind == "sym8":
            q, s = oracle.quant_group_sym8(w)
            assert f32_bits(s) == f32_bits(np.float32(parts[1][0])), (w, s)
            assert q.tolist() == [int(v) for v in parts[2]], (w, q)
        else:
            q, s = oracle.quant_row_act(w)
            assert f32_bits(s) == f32_bits(np.float32(parts[1][0])), (w, s)
            assert q.tolist() == [int(v) for v in parts[2]], (w, q)


def test_act_quant_error_bound_and_extremes():
    rng = np.random.default_rng(7)
    for trial in range(40):
        K = 32 * int(rng.integers(1, 20))
        u = (rng.standard_normal(K) * 10.0 ** rng.uniform(-6, 3)).astype(np.float32)
        if trial % 5 == 0:
            u[rng.integers(K)] *= 50
        q, s = oracle.quant_row_act(u)
        assert s > 0 and np.all(np.abs(q.astype(int)) <= 127)
        err = np.abs(u.astype(np.float64) - q.astype(np.float64) * np.float64(s))
        assert np.all(err <= np.float64(s) * (0.5 + 2.0 ** -16))
        amax = int(np.argmax(np.abs(u)))
        assert abs(int(q[amax])) == 127 and np.sign(q[amax]) == np.sign(u[amax])
        assert np.float64(s) == pytest.approx(np.max(np.abs(u)) / 127.0, rel=1e-7)


def test_w4_group_error_bound():
    rng = np.random.default_rng(8)
    for trial in range(200):
        n = int(rng.choice([16, 32, 64, 128, 256]))
        w = (rng.standard_normal(n) * 0.02).astype(np.float32)
        if trial % 3 == 0:
            w[rng.integers(n)] *= 20
        if trial % 7 == 0:
            w = np.abs(w)
        if trial % 11 == 0:
            w = -np.abs(w)
        q, s, z = oracle.quant_group_asym4(w)
        assert 0 <= z <= 15 and np.all(q <= 15)
        deq = np.float64(s) * (q.astype(np.float64) - z)
        assert np.all(np.abs(w - deq) <= np.float64(s) * (0.5 + 2.0 ** -16))
        # zero is represented exactly by the code z
        q0, _, _ = oracle.quant_group_asym4(np.concatenate([w, [0.0]]).astype(np.float32))
        assert q0[-1] == oracle.quant_group_asym4(np.concatenate([w, [0.0]]).astype(np.float32))[2]


def test_w8_group_error_bound():
    rng = np.random.default_rng(9)
    for trial in range(200):
        n = int(rng.choice([32, 64, 128]))
        w = (rng.standard_normal(n) * 0.02).astype(np.float32)
        if trial % 3 == 0:
            w[rng.integers(n)] *= 20
        q, s = oracle.quant_group_sym8(w)
        assert np.all(np.abs(q.astype(int)) <= 127)
        err = np.abs(w.astype(np.float64) - np.float64(s) * q.astype(np.float64))
        assert np.all(err <= np.float64(s) * (0.5 + 2.0 ** -16))
        amax = int(np.argmax(np.abs(w)))
        assert abs(int(q[amax])) == 127


def test_quant_act_composes_rotation_row_quant_and_group_sums():
    K, G, M = 256, 64, 5
    signs = oracle.make_signs(21, K)
    X = synth.activations(M, K, seed=8, outlier_channels=2).numpy()
    X[3] = 0.0
    qx, sx, gsum = oracle.quant_act(X, G, signs)
    U = oracle.rotate(X, signs)
    for m in range(M):
        q, s = oracle.quant_row_act(U[m])
        assert np.array_equal(q, qx[m]) and f32_bits(s) == f32_bits(sx[m])
    assert np.array_equal(gsum, qx.astype(np.int64).reshape(M, K // G, G).sum(-1))
    assert sx[3] == 0.0 and not qx[3].any() and not gsum[3].any()


def test_quant_weights_compose_rotation_and_group_quant():
    K, G, N = 256, 32, 6
    signs = oracle.make_signs(22, K)
    W = synth.weights(N, K, seed=9).numpy()
    W[2, 64:96] = 0.0
    codes, scales, zeros = oracle.quant_w4(W, G, signs)
    c8, s8 = oracle.quant_w8(W, G, signs)
    U = oracle.rotate(W, signs)
    for n in range(N):
        for g in range(K // G):
            q, s, z = oracle.quant_group_asym4(U[n, g * G:(g + 1) * G])
            assert np.array_equal(q, codes[n, g * G:(g + 1) * G]) and s == scales[n, g] and z == zeros[n, g]
            q8, s_8 = oracle.quant_group_sym8(U[n, g * G:(g + 1) * G])
            assert np.array_equal(q8, c8[n, g * G:(g + 1) * G]) and s_8 == s8[n, g]
    # rotating a zero block gives zeros: that group quantizes to scale 0
    assert scales[2, 2] == 0.0 and zeros[2, 2] == 0 and not codes[2, 64:96].any()


# ------------------------------------------------------- integer GEMM ---
def brute_partials(qx, codes, zeros, G):
    M, K = qx.shape
    N = codes.shape[0]
    a = qx.astype(np.int64).reshape(M, K // G, G)
    w = codes.astype(np.int64).reshape(N, K // G, G)
    if zeros is not None:
        w = w - zeros.astype(np.int64)[:, :, None]
    return np.einsum("mgk,ngk->mng", a, w)


@pytest.mark.parametrize("fmt,G,K,N,M", [("w4", 32, 32, 3, 2), ("w4", 16, 64, 8, 4), ("w4", 64, 128, 5, 3),
                                         ("w8", 32, 64, 8, 4), ("w8", 128, 256, 4, 1), ("w4", 128, 256, 7, 3)])
def test_partials_brute_force(fmt, G, K, N, M):
    rng = np.random.default_rng(K + N + M)
    qx = rng.integers(-127, 128, size=(M, K)).astype(np.int8)
    if fmt == "w4":
        codes = rng.integers(0, 16, size=(N, K)).astype(np.uint8)
        zeros = rng.integers(0, 16, size=(N, K // G)).astype(np.uint8)
    else:
        codes = rng.integers(-127, 128, size=(N, K)).astype(np.int8)
        zeros = None
    P = oracle.partials(qx, codes, zeros, G)
    assert np.array_equal(P.astype(np.int64), brute_partials(qx, codes, zeros, G))


def test_partials_zero_point_identity():
    K, G, N, M = 256, 64, 6, 3
    signs = oracle.make_signs(31, K)
    r = oracle.verify_linear(synth.activations(M, K, seed=10).numpy(), synth.weights(N, K, seed=11).numpy(), G,
                             "w4", signs)
    raw = np.einsum("mgk,ngk->mng", r["qx"].astype(np.int64).reshape(M, K // G, G),
                    r["codes"].astype(np.int64).reshape(N, K // G, G))
    corr = r["zeros"].astype(np.int64)[None, :, :] * r["gsum"].astype(np.int64)[:, None, :]
    assert np.array_equal(r["P"].astype(np.int64), raw - corr)


def test_partials_int32_headroom_extremes():
    for fmt, G in (("w4", 256), ("w8", 256), ("w4", 128), ("w8", 128)):
        K, N, M = 2 * G, 2, 2
        qx = np.full((M, K), 127, dtype=np.int8)
        qx[1] = -127
        if fmt == "w4":
            codes = np.full((N, K), 15, dtype=np.uint8)
            zeros = np.zeros((N, K // G), dtype=np.uint8)
            codes[1] = 0
            zeros[1] = 15
            top = 127 * 15 * G
        else:
            codes = np.full((N, K), 127, dtype=np.int8)
            codes[1] = -127
            zeros = None
            top = 127 * 127 * G
        P = oracle.partials(qx, codes, zeros, G)
        assert P[0, 0, 0] == top and P[1, 0, 0] == -top and P[0, 1, 0] == -top and P[1, 1, 0] == top


def test_epilogue_matches_fp64_within_rounding():
    rng = np.random.default_rng(14)
    M, N, NG = 4, 9, 64
    P = rng.integers(-(2 ** 20), 2 ** 20, size=(M, N, NG)).astype(np.int32)
    sx = (rng.random(M) * 0.1).astype(np.float32)
    scales = (rng.random((N, NG)) * 0.01).astype(np.float32)
    Y = oracle.output(P, sx, scales).astype(np.float64)
    terms = scales.astype(np.float64)[None] * P.astype(np.float64)
    exact = sx.astype(np.float64)[:, None] * terms.sum(-1)
    bound = (NG + 2) * EPS32 * sx.astype(np.float64)[:, None] * np.abs(terms).sum(-1)
    assert np.all(np.abs(Y - exact) <= bound)
    # the order is g ascending: recompute sequentially in fp32 and match bit for bit
    for m in range(M):
        for n in range(N):
            acc = np.float32(0.0)
            for g in range(NG):
                acc = np.float32(acc + np.float32(scales[n, g] * np.float32(P[m, n, g])))
            assert np.float32(sx[m] * acc) == np.float32(Y[m, n])


def layer_error_bound(X, W, G, fmt, signs, r):
    """|Y - x' w'^T| bound from the quantization steps and the fp32 epilogue (fp64)."""
    Xr = oracle.rotate(X, signs).astype(np.float64)
    Wr = oracle.rotate(W, signs).astype(np.float64)
    M, K = Xr.shape
    N = Wr.shape[0]
    ex = r["sx"].astype(np.float64) * (0.5 + 2.0 ** -16)                  # [M]
    ew = np.repeat(r["scales"].astype(np.float64), G, axis=1) * (0.5 + 2.0 ** -16)  # [N][K]
    bound = np.abs(Xr) @ ew.T + ex[:, None] * np.abs(Wr).sum(1)[None, :] + ex[:, None] * ew.sum(1)[None, :]
    terms = np.abs(r["scales"].astype(np.float64)[None] * r["P"].astype(np.float64)).sum(-1)
    bound += (K // G + 2) * EPS32 * r["sx"].astype(np.float64)[:, None] * terms
    return Xr @ Wr.T, bound


@pytest.mark.parametrize("fmt,G", [("w4", 32), ("w4", 64), ("w4", 16), ("w8", 128), ("w8", 32)])
def test_layer_output_within_quantization_error_bound(fmt, G):
    K, N, M = 512, 48, 5
    signs = oracle.make_signs(40 + G, K)
    X = synth.activations(M, K, seed=12, outlier_channels=2).numpy()
    W = synth.weights(N, K, seed=13).numpy()
    r = oracle.verify_linear(X, W, G, fmt, signs)
    exact, bound = layer_error_bound(X, W, G, fmt, signs, r)
    err = r["Y"].astype(np.float64) - exact
    assert np.all(np.abs(err) <= bound)
    # The bound above is worst case (all rounding errors aligned).  Rounding to
    # nearest makes each error roughly uniform on +-step/2, so the output error
    # variance is about sum_k (x'_k^2 sw_k^2 + w'_k^2 sx^2) / 12: a wrong sign,
    # a dropped zero point or a misplaced scale shows up as far more than that.
    Xr = oracle.rotate(X, signs).astype(np.float64)
    Wr = oracle.rotate(W, signs).astype(np.float64)
    sw2 = np.repeat(r["scales"].astype(np.float64), G, axis=1) ** 2
    var = (Xr ** 2) @ sw2.T / 12 + (r["sx"].astype(np.float64) ** 2)[:, None] * (Wr ** 2).sum(1)[None, :] / 12
    assert np.mean(err ** 2) <= 4.0 * np.mean(var)
    assert np.mean(err ** 2) >= 0.05 * np.mean(var)


def test_layer_plausible_against_unquantized_product():
    K, N, M = 1024, 64, 16
    signs = oracle.make_signs(50, K)
    X = synth.activations(M, K, seed=14, outlier_channels=2).numpy()
    W = synth.weights(N, K, seed=15).numpy()
    ref = X.astype(np.float64) @ W.astype(np.float64).T
    for fmt, G, tol in (("w4", 64, 0.15), ("w8", 128, 0.02)):
        Y = oracle.verify_linear(X, W, G, fmt, signs)["Y"].astype(np.float64)
        assert np.linalg.norm(Y - ref) / np.linalg.norm(ref) < tol


def test_rotation_lowers_4bit_error_on_outlier_weights():
    K, N, G = 256, 256, 32
    W = synth.weights(N, K, seed=0, outlier_frac=0.005).numpy()
    signs = oracle.make_signs(0, K)
    no_rot = np.zeros(K // 32, dtype=np.uint32)

    def mse(rotated: bool):
        s = signs if rotated else no_rot
        Wr = oracle.rotate(W, s) if rotated else W
        codes, scales, zeros = oracle.quant_w4(W, G, s) if rotated else _quant_w4_unrotated(W, G)
        deq = np.repeat(scales, G, 1) * (codes.astype(np.float32) - np.repeat(zeros, G, 1).astype(np.float32))
        return float(np.mean((deq - Wr) ** 2))

    assert mse(True) < 0.8 * mse(False)


def _quant_w4_unrotated(W, G):
    N, K = W.shape
    codes = np.empty((N, K), np.uint8)
    scales = np.empty((N, K // G), np.float32)
    zeros = np.empty((N, K // G), np.uint8)
    for n in range(N):
        for g in range(K // G):
            codes[n, g * G:(g + 1) * G], scales[n, g], zeros[n, g] = oracle.quant_group_asym4(W[n, g * G:(g + 1) * G])
    return codes, scales, zeros


def test_fused_gemm_equals_partials_then_output():
    K, N, M, G = 256, 40, 7, 64
    signs = oracle.make_signs(60, K)
    for fmt in ("w4", "w8"):
        r = oracle.verify_linear(synth.activations(M, K, seed=16).numpy(), synth.weights(N, K, seed=17).numpy(), G,
                                 fmt, signs)
        Y2 = oracle.verify_gemm(r["qx"], r["sx"], r["codes"], r["scales"], r["zeros"], G)
        assert np.array_equal(Y2.view(np.uint32), r["Y"].view(np.uint32))


def test_openmp_build_matches_single_thread():
    K, N, M, G = 256, 64, 4, 32
    signs = oracle.make_signs(61, K)
    X = synth.activations(M, K, seed=18).numpy()
    W = synth.weights(N, K, seed=19).numpy()
    a = oracle.quant_w4(W, G, signs)
    b = oracle.quant_w4(W, G, signs, openmp=True)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    qx, sx, _ = oracle.quant_act(X, G, signs)
    y1 = oracle.verify_gemm(qx, sx, a[0], a[1], a[2], G)
    y2 = oracle.verify_gemm(qx, sx, a[0], a[1], a[2], G, openmp=True)
    assert np.array_equal(y1.view(np.uint32), y2.view(np.uint32))
    assert oracle.num_threads(False) == 1 and oracle.num_threads(True) >= 1


# ---------------------------------------------------- tree acceptance ---
def parse_tree_golden(golden_dir):
    out = []
    for line in open(os.path.join(golden_dir, "tree_accept.txt")):
        if not line.startswith("case"):
            continue
        f = [x.strip() for x in line[len("case"):].split("|")]
        name, par, tok, g, path, adv = f[0], *[np.array(x.split(), dtype=np.int64) for x in f[1:5]], int(f[5])
        out.append((name, par, tok, g, path, adv))
    return out


def test_tree_accept_golden(golden_dir):
    cases = parse_tree_golden(golden_dir)
    assert len(cases) >= 6
    for name, par, tok, g, path, adv in cases:
        p, n, bonus = oracle.tree_accept(g, par, tok)
        assert list(p) == list(path), name
        assert n + 1 == adv, name
        last = path[-1] if len(path) else 0
        assert bonus == g[last], name


def test_argmax_rows_matches_numpy_first_index():
    # numpy.argmax returns the first index of the maximum (and the first NaN)
    rng = np.random.default_rng(5)
    L = rng.integers(-3, 4, size=(40, 301)).astype(np.float32)  # many ties
    L[7, 100] = np.nan
    L[9, 0] = np.nan
    L[11] = -np.inf
    L[12, 200] = np.inf
    assert np.array_equal(oracle.argmax_rows(L), np.argmax(L, axis=1))


def brute_force_accept(g, parent, tokens):
    """Every root-to-node path checked edge by edge; deepest valid, lowest index."""
    best, best_path = 0, []
    for i in range(1, len(parent)):
        path, j, ok = [], i, True
        while j != 0:
            ok &= tokens[j] == g[parent[j]]
            path.append(j)
            j = parent[j]
        if ok and len(path) > len(best_path):
            best, best_path = i, path[::-1]
    return best_path, g[best]


def test_tree_accept_brute_force_random_trees():
    rng = np.random.default_rng(6)
    for trial in range(300):
        M = int(rng.integers(1, 40))
        parent = np.array([-1] + [int(rng.integers(0, i)) for i in range(1, M)], dtype=np.int32)
        g = rng.integers(0, 4, size=M).astype(np.int32)
        tokens = rng.integers(0, 4, size=M).astype(np.int32)
        path, n, bonus = oracle.tree_accept(g, parent, tokens)
        bp, bb = brute_force_accept(g, parent, tokens)
        assert list(path) == bp and n == len(bp) and bonus == bb, trial


def test_tree_accept_rejects_bad_parents():
    g = np.zeros(3, dtype=np.int32)
    for parent in ([-1, 1, 0], [-1, 0, 2], [-1, -1, 0]):
        with pytest.raises(ValueError):
            oracle.tree_accept(g, np.array(parent, dtype=np.int32), np.zeros(3, dtype=np.int32))


# ------------------------------------------------------ tree attention ---
# Page "Karpathy's Trick for Faster Local LLMs Finally Has Proper Tooling",
# section "Verifying a draft tree without restoring model state": the main
# model checks every branch of the draft tree in one pass; an attention layer
# reads its cache of past tokens.  Reading: a node sees the committed cache,
# its ancestors and itself.

def _attn_inputs(rng, M, Hq, Hkv, D, L, extra=0, vscale=1.0):
    q = (rng.standard_normal((M, Hq, D)) * 0.5).astype(np.float16)
    k = (rng.standard_normal((Hkv, L + M + extra, D)) * 0.5).astype(np.float16)
    v = (rng.standard_normal((Hkv, L + M + extra, D)) * vscale).astype(np.float16)
    return q, k, v


def _random_tree(rng, M):
    par = np.zeros(M, dtype=np.int32)
    for i in range(1, M):
        par[i] = rng.integers(0, i)
    return par


def _dense_reference(q, k, v, L, parent, scale):
    """Masked softmax attention with the tree mask from a boolean transitive
    closure (repeated squaring of the parent relation), numpy fp64 einsum."""
    M, Hq, D = q.shape
    Hkv = k.shape[0]
    G = Hq // Hkv
    A = np.zeros((M, M), dtype=bool)  # A[i, j]: j is the parent of i
    for i in range(1, M):
        if 0 <= parent[i] < i:
            A[i, parent[i]] = True
    R = A | np.eye(M, dtype=bool)
    for _ in range(int(np.ceil(np.log2(max(M, 2)))) + 1):
        R = R | ((R.astype(np.int64) @ R.astype(np.int64)) > 0)
    mask = np.concatenate([np.ones((M, L), dtype=bool), R], axis=1)  # [M][L + M]
    qd, kd, vd = q.astype(np.float64), k[:, : L + M].astype(np.float64), v[:, : L + M].astype(np.float64)
    kh = np.repeat(kd, G, axis=0)  # [Hq][L+M][D]
    vh = np.repeat(vd, G, axis=0)
    s = scale * np.einsum("ihd,htd->iht", qd, kh)
    s = np.where(mask[:, None, :], s, -np.inf)
    s = s - s.max(axis=2, keepdims=True)
    p = np.exp(s)
    p = p / p.sum(axis=2, keepdims=True)
    return np.einsum("iht,htd->ihd", p, vh)


def test_half_decoding_matches_numpy_for_every_bit_pattern():
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    for b in bits:
        got = oracle.half_to_double(int(b))
        r = ref[int(b)]
        assert (np.isnan(got) and np.isnan(r)) or got == r, hex(int(b))


@pytest.mark.parametrize("L,M", [(0, 1), (0, 6), (5, 4), (33, 9)])
def test_tree_attention_chain_is_causal_attention(L, M):
    """A chain (node i's parent is i-1) is ordinary causal decoding of L + M
    tokens: torch's scaled_dot_product_attention (fp64, CPU) with a causal
    mask offset by L."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(L * 31 + M)
    Hq = Hkv = 2
    D = 16
    q, k, v = _attn_inputs(rng, M, Hq, Hkv, D, L)
    parent = np.maximum(np.arange(M, dtype=np.int32) - 1, 0)
    scale = 1.0 / np.sqrt(D)
    got = oracle.tree_attention(q, k, v, L, parent, scale)
    Q = torch.from_numpy(q.astype(np.float64)).permute(1, 0, 2)        # [H][M][D]
    K = torch.from_numpy(k[:, : L + M].astype(np.float64))              # [H][L+M][D]
    V = torch.from_numpy(v[:, : L + M].astype(np.float64))
    mask = torch.ones(M, L + M, dtype=torch.bool).tril(diagonal=L)
    ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=mask, scale=scale)
    np.testing.assert_allclose(got, ref.permute(1, 0, 2).numpy(), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("seed", range(4))
def test_tree_attention_matches_dense_closure_reference(seed):
    rng = np.random.default_rng(100 + seed)
    M, Hq, Hkv, D, L = int(rng.integers(2, 20)), 8, 2, 12, int(rng.integers(0, 40))
    q, k, v = _attn_inputs(rng, M, Hq, Hkv, D, L, extra=3)
    parent = _random_tree(rng, M)
    got = oracle.tree_attention(q, k, v, L, parent, 0.37)
    np.testing.assert_allclose(got, _dense_reference(q, k, v, L, parent, 0.37), rtol=1e-12, atol=1e-12)


def test_tree_attention_star_tree_sees_root_and_itself():
    """Every drafted node a child of the root: node i sees the cache, the root
    and itself, never its siblings (closed form for L = 0: a two-key softmax)."""
    rng = np.random.default_rng(7)
    M, H, D = 6, 1, 4
    q, k, v = _attn_inputs(rng, M, H, H, D, 0)
    parent = np.zeros(M, dtype=np.int32)
    got = oracle.tree_attention(q, k, v, 0, parent, 1.0)
    qd, kd, vd = q.astype(np.float64)[:, 0], k.astype(np.float64)[0], v.astype(np.float64)[0]
    assert np.array_equal(got[0, 0], vd[0])  # the root sees only itself
    for i in range(1, M):
        s0, si = qd[i] @ kd[0], qd[i] @ kd[i]
        w0 = 1.0 / (1.0 + np.exp(si - s0))
        np.testing.assert_allclose(got[i, 0], w0 * vd[0] + (1 - w0) * vd[i], rtol=1e-13, atol=1e-14)


def test_tree_attention_zero_scale_is_the_mean_of_visible_values():
    rng = np.random.default_rng(8)
    M, Hq, Hkv, D, L = 7, 4, 4, 5, 3
    q, k, v = _attn_inputs(rng, M, Hq, Hkv, D, L)
    parent = np.array([0, 0, 1, 2, 0, 4, 2], dtype=np.int32)
    got = oracle.tree_attention(q, k, v, L, parent, 0.0)
    anc = {0: [0], 1: [0, 1], 2: [0, 1, 2], 3: [0, 1, 2, 3], 4: [0, 4], 5: [0, 4, 5], 6: [0, 1, 2, 6]}
    for i in range(M):
        cols = list(range(L)) + [L + j for j in anc[i]]
        np.testing.assert_allclose(got[i], v[:, cols].astype(np.float64).mean(axis=1), rtol=1e-14, atol=1e-15)


def test_tree_attention_grouped_heads_equal_repeated_kv_heads():
    rng = np.random.default_rng(9)
    M, Hq, Hkv, D, L = 5, 8, 2, 6, 11
    q, k, v = _attn_inputs(rng, M, Hq, Hkv, D, L)
    parent = np.array([0, 0, 1, 1, 3], dtype=np.int32)
    got = oracle.tree_attention(q, k, v, L, parent, 0.5)
    rep = oracle.tree_attention(q, np.repeat(k, Hq // Hkv, axis=0), np.repeat(v, Hq // Hkv, axis=0), L, parent, 0.5)
    np.testing.assert_allclose(got, rep, rtol=0, atol=0)


def test_tree_attention_ignores_the_order_of_committed_positions():
    rng = np.random.default_rng(10)
    M, Hq, Hkv, D, L = 4, 2, 1, 8, 9
    q, k, v = _attn_inputs(rng, M, Hq, Hkv, D, L)
    parent = np.array([0, 0, 1, 0], dtype=np.int32)
    perm = np.concatenate([rng.permutation(L), np.arange(L, L + M)])
    a = oracle.tree_attention(q, k, v, L, parent, 0.7)
    b = oracle.tree_attention(q, k[:, perm], v[:, perm], L, parent, 0.7)
    np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-14)


def test_tree_attention_invalid_parent_ends_the_ancestor_walk():
    rng = np.random.default_rng(11)
    M, H, D, L = 4, 1, 4, 2
    q, k, v = _attn_inputs(rng, M, H, H, D, L)
    parent = np.array([0, 0, 3, 2], dtype=np.int32)  # node 2's parent is not before it
    got = oracle.tree_attention(q, k, v, L, parent, 1.0)
    # node 2 sees the cache and itself; node 3 sees the cache, node 2 and itself
    ref = _dense_reference(q, k, v, L, np.array([0, 0, -1, 2], dtype=np.int32), 1.0)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_tree_commit_kv_moves_the_accepted_path_next_to_the_root():
    rng = np.random.default_rng(12)
    Hkv, L, M, D = 3, 5, 8, 4
    cap = L + M + 2
    k = rng.standard_normal((Hkv, cap, D)).astype(np.float16)
    v = rng.standard_normal((Hkv, cap, D)).astype(np.float16)
    path = np.array([2, 5, 7], dtype=np.int32)  # node 2 at depth 1, 5 at depth 2, 7 at depth 3
    k2, v2 = oracle.tree_commit_kv(k, v, L, path, 3)
    for d, node in enumerate(path):
        assert np.array_equal(k2[:, L + 1 + d], k[:, L + node]) and np.array_equal(v2[:, L + 1 + d], v[:, L + node])
    untouched = [t for t in range(cap) if not (L + 1 <= t < L + 4)]
    assert np.array_equal(k2[:, untouched], k[:, untouched]) and np.array_equal(v2[:, untouched], v[:, untouched])
    # a chain path is already in place; no accepted node or a bad tree moves nothing
    kc, vc = oracle.tree_commit_kv(k, v, L, np.array([1, 2, 3], dtype=np.int32), 3)
    assert np.array_equal(kc, k) and np.array_equal(vc, v)
    for n in (0, -1):
        kn, vn = oracle.tree_commit_kv(k, v, L, path, n)
        assert np.array_equal(kn, k) and np.array_equal(vn, v)


# ------------------------------------------------------ DeltaNet tree pass ---
# Page "Karpathy's Trick for Faster Local LLMs Finally Has Proper Tooling",
# section "Verifying a draft tree without restoring model state" (the state of
# a Gated DeltaNet layer changes with every accepted token; verification must
# not change it).  Recurrence: the published gated delta rule,
# S_t = alpha_t S_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T, o_t = S_t q_t.

def _delta_inputs(rng, M, H, D, unit_keys=True):
    st = rng.standard_normal((H, D, D)).astype(np.float32) * 0.3
    q = rng.standard_normal((M, H, D)).astype(np.float32)
    k = rng.standard_normal((M, H, D)).astype(np.float32)
    if unit_keys:
        k = (k / np.linalg.norm(k, axis=2, keepdims=True)).astype(np.float32)
    v = rng.standard_normal((M, H, D)).astype(np.float32)
    al = rng.uniform(0.6, 1.0, (M, H)).astype(np.float32)
    be = rng.uniform(0.0, 1.0, (M, H)).astype(np.float32)
    return st, q, k, v, al, be


def _unrolled_chain(st, k, v, al, be, nodes, h):
    """S after the nodes in order, as the unrolled sum of transition-matrix
    products: S_c T_1 ... T_n + sum_j beta_j v_j k_j^T T_{j+1} ... T_n with
    T_j = alpha_j (I - beta_j k_j k_j^T) (numpy fp64 matrix products)."""
    D = st.shape[1]
    I = np.eye(D)
    kd, vd = k.astype(np.float64), v.astype(np.float64)
    T = [float(al[j, h]) * (I - float(be[j, h]) * np.outer(kd[j, h], kd[j, h])) for j in nodes]
    def tail(a):
        P = I.copy()
        for Tm in T[a:]:
            P = P @ Tm
        return P
    S = st[h].astype(np.float64) @ tail(0)
    for a, j in enumerate(nodes):
        S = S + float(be[j, h]) * np.outer(vd[j, h], kd[j, h]) @ tail(a + 1)
    return S


def _root_path(parent, i):
    chain = [i]
    while chain[-1] > 0 and 0 <= parent[chain[-1]] < chain[-1]:
        chain.append(int(parent[chain[-1]]))
    return chain[::-1]


@pytest.mark.parametrize("seed", range(3))
def test_delta_tree_matches_unrolled_products_on_every_root_path(seed):
    rng = np.random.default_rng(200 + seed)
    M, H, D = 9, 2, 12
    st, q, k, v, al, be = _delta_inputs(rng, M, H, D)
    parent = np.array([0, 0, 1, 1, 0, 4, 2, 6, 3], dtype=np.int32)
    got = oracle.delta_tree(st, q, k, v, al, be, parent)
    for i in range(M):
        for h in range(H):
            S = _unrolled_chain(st, k, v, al, be, _root_path(parent, i), h)
            np.testing.assert_allclose(got[i, h], S @ q[i, h].astype(np.float64), rtol=1e-11, atol=1e-11)


def test_delta_tree_without_writes_only_decays_the_state():
    rng = np.random.default_rng(210)
    M, H, D = 6, 3, 8
    st, q, k, v, al, be = _delta_inputs(rng, M, H, D)
    be[:] = 0.0
    parent = np.array([0, 0, 1, 2, 0, 4], dtype=np.int32)
    got = oracle.delta_tree(st, q, k, v, al, be, parent)
    for i in range(M):
        decay = np.prod([al[j].astype(np.float64) for j in _root_path(parent, i)], axis=0)  # [H]
        ref = decay[:, None] * np.einsum("hrc,hc->hr", st.astype(np.float64), q[i].astype(np.float64))
        np.testing.assert_allclose(got[i], ref, rtol=1e-12, atol=1e-12)


def test_delta_rule_overwrites_the_value_stored_under_a_unit_key():
    """alpha = beta = 1 and |k| = 1: after the step, S k = v exactly (the
    delta rule replaces what the key retrieves); querying with the node's own
    key returns its value."""
    rng = np.random.default_rng(211)
    M, H, D = 5, 2, 16
    st, q, k, v, al, be = _delta_inputs(rng, M, H, D)
    al[:] = 1.0
    be[:] = 1.0
    q = k.copy()
    got = oracle.delta_tree(st, q, k, v, al, be, np.array([0, 0, 1, 2, 1], dtype=np.int32))
    np.testing.assert_allclose(got, v.astype(np.float64), rtol=0, atol=1e-6)


def test_delta_rule_with_orthonormal_keys_replaces_columns():
    """Keys e_0, e_1, ... along a chain with alpha = beta = 1: the state is the
    committed one with column j replaced by v_j for every node j on the path."""
    rng = np.random.default_rng(212)
    M, H, D = 4, 1, 6
    st, q, k, v, al, be = _delta_inputs(rng, M, H, D)
    k[:] = 0.0
    for j in range(M):
        k[j, 0, j] = 1.0
    al[:] = 1.0
    be[:] = 1.0
    parent = np.array([0, 0, 1, 2], dtype=np.int32)
    got = oracle.delta_tree(st, q, k, v, al, be, parent)
    for i in range(M):
        S = st[0].astype(np.float64).copy()
        for j in range(i + 1):
            S[:, j] = v[j, 0]
        np.testing.assert_allclose(got[i, 0], S @ q[i, 0].astype(np.float64), rtol=1e-12, atol=1e-12)


def test_delta_tree_node_ignores_other_branches():
    rng = np.random.default_rng(213)
    M, H, D = 7, 2, 8
    st, q, k, v, al, be = _delta_inputs(rng, M, H, D)
    parent = np.array([0, 0, 0, 1, 2, 3, 2], dtype=np.int32)
    a = oracle.delta_tree(st, q, k, v, al, be, parent)
    k2, v2 = k.copy(), v.copy()
    k2[[2, 4, 6]] = rng.standard_normal((3, H, D)).astype(np.float32)  # the other branch of node 5
    v2[[2, 4, 6]] = rng.standard_normal((3, H, D)).astype(np.float32)
    b = oracle.delta_tree(st, q, k2, v2, al, be, parent)
    for i in (0, 1, 3, 5):
        assert np.array_equal(a[i], b[i])


def test_delta_commit_is_the_accepted_nodes_state():
    rng = np.random.default_rng(214)
    M, H, D = 8, 2, 8
    st, q, k, v, al, be = _delta_inputs(rng, M, H, D)
    parent = np.array([0, 0, 1, 2, 0, 4, 5, 2], dtype=np.int32)
    path = np.array([4, 5, 6], dtype=np.int32)  # root -> 4 -> 5 -> 6
    S = oracle.delta_commit(st, k, v, al, be, path, 3)
    for h in range(H):
        np.testing.assert_allclose(S[h], _unrolled_chain(st, k, v, al, be, [0, 4, 5, 6], h), rtol=1e-11, atol=1e-11)
    # the new committed state answers node 6's query as the tree pass did
    got = oracle.delta_tree(st, q, k, v, al, be, parent)
    np.testing.assert_allclose(np.einsum("hrc,hc->hr", S, q[6].astype(np.float64)), got[6], rtol=1e-12, atol=1e-12)
    # no drafted token accepted: only the root advances; a malformed tree changes nothing
    S0 = oracle.delta_commit(st, k, v, al, be, path, 0)
    for h in range(H):
        np.testing.assert_allclose(S0[h], _unrolled_chain(st, k, v, al, be, [0], h), rtol=1e-12, atol=1e-12)
    assert np.array_equal(oracle.delta_commit(st, k, v, al, be, path, -1), st.astype(np.float64))

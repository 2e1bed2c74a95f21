"""CPU oracle of the quantized speculative-verify linear layer.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline of ``bench.py`` may import this package; the product path
(``quantized_speculative_verify_gb300``) never does, and shares no code with
it.  The arithmetic lives in ``hq_oracle.c`` (plain scalar C99, compiled with
``-O2 -ffp-contract=off``); this module only compiles it with gcc and marshals
numpy arrays through ctypes.

Source of the method: "Karpathy's Trick for Faster Local LLMs Finally Has
Proper Tooling", section "How Uzu optimizes bytes and tokens per pass" (4-bit
asymmetric / 8-bit symmetric weights, 8-bit activations on the fly, 32-block
randomized Hadamard transform before quantization, transform block and
quantization group independent).  The readings of that prose are listed at the
top of ``hq_oracle.c``.

Every function here is pinned by ``tests/test_oracle.py`` against facts that
do not come from the oracle itself (library Hadamard matrix, closed forms,
hand-derived golden examples under ``tests/golden/``, int64 brute force,
error bounds).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "hq_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_CFLAGS = ["-std=c99", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]

_libs: dict = {}
_lock = threading.Lock()


def _so_path(openmp: bool) -> str:
    return os.path.join(_BUILD, "liboracle_omp.so" if openmp else "liboracle.so")


def build(force: bool = False) -> None:
    """Compile the single-thread and the OpenMP build of the oracle."""
    os.makedirs(_BUILD, exist_ok=True)
    for openmp in (False, True):
        out = _so_path(openmp)
        if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
            continue
        cmd = ["gcc", *_CFLAGS, *(["-fopenmp"] if openmp else []), _SRC, "-o", out + ".tmp", "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(out + ".tmp", out)


_P = ctypes.c_void_p
_I = ctypes.c_int


def _load(openmp: bool = False) -> ctypes.CDLL:
    with _lock:
        if openmp in _libs:
            return _libs[openmp]
        # A test that plants a mistake in a copy of the oracle points this
        # variable at the copy's build; nothing else sets it.
        override = os.environ.get("HQ_ORACLE_TEST_LIB")
        if override:
            lib = ctypes.CDLL(override)
        else:
            build()
            lib = ctypes.CDLL(_so_path(openmp))
        lib.or_splitmix64_next.restype = ctypes.c_uint64
        lib.or_splitmix64_next.argtypes = [ctypes.POINTER(ctypes.c_uint64)]
        lib.or_make_signs.argtypes = [ctypes.c_uint64, _I, _P]
        lib.or_fwht32.argtypes = [_P]
        lib.or_fwht32.restype = None
        lib.or_rotate_vec.argtypes = [_P, _I, _P, _P]
        lib.or_rotate_vec.restype = None
        lib.or_rotate_inverse_vec.argtypes = [_P, _I, _P, _P]
        lib.or_rotate_inverse_vec.restype = None
        lib.or_rotate_rows.argtypes = [_P, _I, _I, _P, _P]
        lib.or_rotate_rows.restype = None
        lib.or_quant_row_act.argtypes = [_P, _I, _P, _P]
        lib.or_quant_row_act.restype = None
        lib.or_quant_group_asym4.argtypes = [_P, _I, _P, _P, _P]
        lib.or_quant_group_asym4.restype = None
        lib.or_quant_group_sym8.argtypes = [_P, _I, _P, _P]
        lib.or_quant_group_sym8.restype = None
        lib.or_quant_act.argtypes = [_P, _I, _I, _I, _P, _P, _P, _P]
        lib.or_quant_w4.argtypes = [_P, _I, _I, _I, _P, _P, _P, _P]
        lib.or_quant_w8.argtypes = [_P, _I, _I, _I, _P, _P, _P]
        lib.or_partials.argtypes = [_P, _I, _P, _P, _I, _I, _I, _I, _P]
        lib.or_output.argtypes = [_P, _P, _P, _I, _I, _I, _P]
        lib.or_verify_gemm.argtypes = [_P, _P, _I, _P, _P, _P, _I, _I, _I, _I, _P]
        lib.or_num_threads.argtypes = []
        lib.or_argmax_rows.argtypes = [_P, _I, _I, _P]
        lib.or_tree_accept.argtypes = [_P, _P, _P, _I, _P, _P, _P]
        lib.or_half_to_double.argtypes = [ctypes.c_uint16]
        lib.or_half_to_double.restype = ctypes.c_double
        lib.or_tree_attention.argtypes = [_P, _P, _P, _I, _I, _I, _I, _I, _I, _P, ctypes.c_double, _P]
        lib.or_tree_commit_kv.argtypes = [_P, _P, _I, _I, _I, _I, _P, _I]
        lib.or_delta_tree.argtypes = [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _P]
        lib.or_delta_commit.argtypes = [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I]
        _libs[openmp] = lib
        return lib


def _c(a: np.ndarray, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise ValueError(f"oracle {what} failed with code {rc}")


# ---------------------------------------------------------------- signs ---
def splitmix64(seed: int, count: int) -> np.ndarray:
    """The first `count` outputs of SplitMix64 started at `seed`."""
    lib = _load()
    st = ctypes.c_uint64(seed & (2**64 - 1))
    return np.array([lib.or_splitmix64_next(ctypes.byref(st)) for _ in range(count)], dtype=np.uint64)


def make_signs(seed: int, K: int) -> np.ndarray:
    """Bit-packed sign vector uint32[K/32]; bit set => the feature is negated."""
    out = np.zeros(K // 32, dtype=np.uint32)
    _check(_load().or_make_signs(ctypes.c_uint64(seed & (2**64 - 1)), K, _ptr(out)), "make_signs")
    return out


def signs_to_pm1(signs: np.ndarray, K: int) -> np.ndarray:
    """Unpack the bit-packed signs to a +-1 float64 vector (a plain view)."""
    k = np.arange(K)
    bits = (signs[k // 32] >> (k % 32).astype(np.uint32)) & 1
    return np.where(bits == 1, -1.0, 1.0)


# ------------------------------------------------------------- rotation ---
def fwht32(u: np.ndarray) -> np.ndarray:
    """Unnormalized butterfly (strides 1..16, fp32) on a copy of 32 values."""
    a = _c(u, np.float32).copy()
    assert a.shape == (32,)
    _load().or_fwht32(_ptr(a))
    return a


def rotate(V: np.ndarray, signs: np.ndarray) -> np.ndarray:
    """Rows of V [R][K] -> V R, R = blockdiag(D_b H_32 / sqrt(32))."""
    V = _c(np.atleast_2d(V), np.float32)
    out = np.empty_like(V)
    _load().or_rotate_rows(_ptr(V), V.shape[0], V.shape[1], _ptr(_c(signs, np.uint32)), _ptr(out))
    return out


def rotate_inverse(U: np.ndarray, signs: np.ndarray) -> np.ndarray:
    U = _c(np.atleast_2d(U), np.float32)
    out = np.empty_like(U)
    s = _c(signs, np.uint32)
    lib = _load()
    for r in range(U.shape[0]):
        row = np.ascontiguousarray(U[r])
        o = np.empty_like(row)
        lib.or_rotate_inverse_vec(_ptr(row), U.shape[1], _ptr(s), _ptr(o))
        out[r] = o
    return out


# ----------------------------------------------------------- quantizers ---
def quant_row_act(u: np.ndarray):
    """One already-rotated activation row -> (int8 codes, fp32 scale)."""
    u = _c(u, np.float32)
    q = np.empty(u.shape[0], dtype=np.int8)
    s = np.zeros(1, dtype=np.float32)
    _load().or_quant_row_act(_ptr(u), u.shape[0], _ptr(q), _ptr(s))
    return q, np.float32(s[0])


def quant_group_asym4(w: np.ndarray):
    """One group of rotated weights -> (uint8 codes 0..15, fp32 scale, zero point)."""
    w = _c(w, np.float32)
    q = np.empty(w.shape[0], dtype=np.uint8)
    s = np.zeros(1, dtype=np.float32)
    z = np.zeros(1, dtype=np.uint8)
    _load().or_quant_group_asym4(_ptr(w), w.shape[0], _ptr(q), _ptr(s), _ptr(z))
    return q, np.float32(s[0]), int(z[0])


def quant_group_sym8(w: np.ndarray):
    w = _c(w, np.float32)
    q = np.empty(w.shape[0], dtype=np.int8)
    s = np.zeros(1, dtype=np.float32)
    _load().or_quant_group_sym8(_ptr(w), w.shape[0], _ptr(q), _ptr(s))
    return q, np.float32(s[0])


def quant_act(X: np.ndarray, G: int, signs: np.ndarray):
    """X [M][K] fp32 -> qx int8 [M][K], sx fp32 [M], gsum int32 [M][K/G]."""
    X = _c(np.atleast_2d(X), np.float32)
    M, K = X.shape
    qx = np.empty((M, K), dtype=np.int8)
    sx = np.empty(M, dtype=np.float32)
    gsum = np.empty((M, K // G), dtype=np.int32)
    _check(_load().or_quant_act(_ptr(X), M, K, G, _ptr(_c(signs, np.uint32)), _ptr(qx), _ptr(sx), _ptr(gsum)),
           "quant_act")
    return qx, sx, gsum


def quant_w4(W: np.ndarray, G: int, signs: np.ndarray, openmp: bool = False):
    """W [N][K] fp32 -> codes uint8 [N][K] (0..15), scales fp32 [N][K/G], zeros uint8 [N][K/G]."""
    W = _c(W, np.float32)
    N, K = W.shape
    codes = np.empty((N, K), dtype=np.uint8)
    scales = np.empty((N, K // G), dtype=np.float32)
    zeros = np.empty((N, K // G), dtype=np.uint8)
    _check(_load(openmp).or_quant_w4(_ptr(W), N, K, G, _ptr(_c(signs, np.uint32)), _ptr(codes), _ptr(scales),
                                     _ptr(zeros)), "quant_w4")
    return codes, scales, zeros


def quant_w8(W: np.ndarray, G: int, signs: np.ndarray, openmp: bool = False):
    """W [N][K] fp32 -> codes int8 [N][K], scales fp32 [N][K/G]."""
    W = _c(W, np.float32)
    N, K = W.shape
    codes = np.empty((N, K), dtype=np.int8)
    scales = np.empty((N, K // G), dtype=np.float32)
    _check(_load(openmp).or_quant_w8(_ptr(W), N, K, G, _ptr(_c(signs, np.uint32)), _ptr(codes), _ptr(scales)),
           "quant_w8")
    return codes, scales


def partials(qx: np.ndarray, codes: np.ndarray, zeros, G: int, openmp: bool = False) -> np.ndarray:
    """Per-group int32 partial sums P [M][N][K/G]; `zeros` is None for the 8-bit format."""
    qx = _c(qx, np.int8)
    M, K = qx.shape
    N = codes.shape[0]
    is_w4 = zeros is not None
    cd = _c(codes, np.uint8 if is_w4 else np.int8)
    zz = _c(zeros, np.uint8) if is_w4 else np.zeros(1, dtype=np.uint8)
    P = np.empty((M, N, K // G), dtype=np.int32)
    _check(_load(openmp).or_partials(_ptr(qx), M, _ptr(cd), _ptr(zz), N, K, G, int(is_w4), _ptr(P)), "partials")
    return P


def output(P: np.ndarray, sx: np.ndarray, scales: np.ndarray, openmp: bool = False) -> np.ndarray:
    """fp32 epilogue: Y[m][n] = sx[m] * sum_g (scales[n][g] * P[m][n][g]), g ascending."""
    P = _c(P, np.int32)
    M, N, NG = P.shape
    Y = np.empty((M, N), dtype=np.float32)
    _check(_load(openmp).or_output(_ptr(P), _ptr(_c(sx, np.float32)), _ptr(_c(scales, np.float32)), M, N, NG,
                                   _ptr(Y)), "output")
    return Y


def verify_gemm(qx, sx, codes, scales, zeros, G: int, openmp: bool = False) -> np.ndarray:
    """Integer GEMM + epilogue without materializing P (same arithmetic)."""
    qx = _c(qx, np.int8)
    M, K = qx.shape
    N = codes.shape[0]
    is_w4 = zeros is not None
    cd = _c(codes, np.uint8 if is_w4 else np.int8)
    zz = _c(zeros, np.uint8) if is_w4 else np.zeros(1, dtype=np.uint8)
    Y = np.empty((M, N), dtype=np.float32)
    _check(_load(openmp).or_verify_gemm(_ptr(qx), _ptr(_c(sx, np.float32)), M, _ptr(cd),
                                        _ptr(_c(scales, np.float32)), _ptr(zz), N, K, G, int(is_w4), _ptr(Y)),
           "verify_gemm")
    return Y


def num_threads(openmp: bool) -> int:
    return int(_load(openmp).or_num_threads())


def verify_linear(X: np.ndarray, W: np.ndarray, G: int, fmt: str, signs: np.ndarray):
    """The whole layer: returns a dict with every intermediate of the path."""
    qx, sx, gsum = quant_act(X, G, signs)
    if fmt == "w4":
        codes, scales, zeros = quant_w4(W, G, signs)
    elif fmt == "w8":
        (codes, scales), zeros = quant_w8(W, G, signs), None
    else:
        raise ValueError(fmt)
    P = partials(qx, codes, zeros, G)
    Y = output(P, sx, scales)
    return dict(qx=qx, sx=sx, gsum=gsum, codes=codes, scales=scales, zeros=zeros, P=P, Y=Y)


def argmax_rows(logits: np.ndarray) -> np.ndarray:
    """Greedy token per row: lowest index among equal maxima; the first NaN wins."""
    L = _c(np.atleast_2d(logits), np.float32)
    M, V = L.shape
    g = np.empty(M, dtype=np.int32)
    _check(_load().or_argmax_rows(_ptr(L), M, V, _ptr(g)), "argmax_rows")
    return g


def tree_accept(g: np.ndarray, parent: np.ndarray, tokens: np.ndarray):
    """(path of accepted drafted nodes, number accepted, bonus token) for a draft tree."""
    g, parent, tokens = _c(g, np.int32), _c(parent, np.int32), _c(tokens, np.int32)
    M = g.shape[0]
    path = np.full(M, -1, dtype=np.int32)
    n = np.zeros(1, dtype=np.int32)
    bonus = np.zeros(1, dtype=np.int32)
    _check(_load().or_tree_accept(_ptr(g), _ptr(parent), _ptr(tokens), M, _ptr(path), _ptr(n), _ptr(bonus)),
           "tree_accept")
    return path[: int(n[0])], int(n[0]), int(bonus[0])


def half_to_double(bits: int) -> float:
    """Value of an IEEE binary16 bit pattern."""
    return float(_load().or_half_to_double(int(bits) & 0xFFFF))


def tree_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, L: int, parent: np.ndarray, scale: float,
                   openmp: bool = False) -> np.ndarray:
    """Tree-masked attention of the M tree nodes (fp64).

    q float16 [M][Hq][D]; k, v float16 [Hkv][cap][D] with the committed
    positions [0, L) and the tree nodes at [L, L + M); parent int32 [M].
    Returns float64 [M][Hq][D]."""
    q16 = _c(q, np.float16)
    k16, v16 = _c(k, np.float16), _c(v, np.float16)
    M, Hq, D = q16.shape
    Hkv, cap, D2 = k16.shape
    if D2 != D or v16.shape != k16.shape:
        raise ValueError("shape mismatch")
    par = _c(parent, np.int32)
    out = np.empty((M, Hq, D), dtype=np.float64)
    _check(_load(openmp).or_tree_attention(_ptr(q16.view(np.uint16)), _ptr(k16.view(np.uint16)),
                                           _ptr(v16.view(np.uint16)), cap, L, M, Hq, Hkv, D, _ptr(par),
                                           float(scale), _ptr(out)), "tree_attention")
    return out


def tree_commit_kv(k: np.ndarray, v: np.ndarray, L: int, path: np.ndarray, n_accept: int):
    """Copies of k and v [Hkv][cap][D] after moving the accepted path next to the root."""
    k16, v16 = np.array(k, dtype=np.float16, order="C"), np.array(v, dtype=np.float16, order="C")
    Hkv, cap, D = k16.shape
    p = _c(np.asarray(path).reshape(-1), np.int32)
    if p.size == 0:
        p = np.zeros(1, dtype=np.int32)
    _check(_load().or_tree_commit_kv(_ptr(k16.view(np.uint16)), _ptr(v16.view(np.uint16)), cap, L, Hkv, D,
                                     _ptr(p), int(n_accept)), "tree_commit_kv")
    return k16, v16


def delta_tree(state: np.ndarray, q: np.ndarray, k: np.ndarray, v: np.ndarray, alpha: np.ndarray, beta: np.ndarray,
               parent: np.ndarray, openmp: bool = False) -> np.ndarray:
    """Outputs of every tree node of a gated delta-rule layer (fp64).

    state float32 [H][D][D] (committed, read only); q, k, v float32 [M][H][D];
    alpha, beta float32 [M][H]; parent int32 [M].  Returns float64 [M][H][D]."""
    st = _c(state, np.float32)
    q, k, v = _c(q, np.float32), _c(k, np.float32), _c(v, np.float32)
    al, be, par = _c(alpha, np.float32), _c(beta, np.float32), _c(parent, np.int32)
    M, H, D = q.shape
    out = np.empty((M, H, D), dtype=np.float64)
    _check(_load(openmp).or_delta_tree(_ptr(st), _ptr(q), _ptr(k), _ptr(v), _ptr(al), _ptr(be), _ptr(par), M, H, D,
                                       _ptr(out)), "delta_tree")
    return out


def delta_commit(state: np.ndarray, k: np.ndarray, v: np.ndarray, alpha: np.ndarray, beta: np.ndarray,
                 path: np.ndarray, n_accept: int) -> np.ndarray:
    """The committed state after accepting the root and path[:n_accept] (fp64 copy)."""
    st = np.array(state, dtype=np.float64, order="C")
    k, v = _c(k, np.float32), _c(v, np.float32)
    al, be = _c(alpha, np.float32), _c(beta, np.float32)
    M, H, D = k.shape
    p = _c(np.asarray(path).reshape(-1), np.int32)
    if p.size == 0:
        p = np.zeros(1, dtype=np.int32)
    _check(_load().or_delta_commit(_ptr(st), _ptr(k), _ptr(v), _ptr(al), _ptr(be), _ptr(p), int(n_accept), M, H, D),
           "delta_commit")
    return st

"""Python binding of libhq.so (include/hq.h): argument marshalling only.

Every step of the verify-pass linear layer runs in the library's CUDA kernels.
This module converts torch tensors to raw device pointers, passes the current
CUDA stream, and turns status codes into exceptions.  There is no fallback: if
libhq.so is missing or cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import numpy as np
import torch

from . import build as _build

HQ_OK = 0
HQ_ERR_INVALID_ARG = 1
HQ_ERR_UNSUPPORTED = 2
HQ_ERR_CUDA = 3
HQ_ERR_TIMEOUT = 4
HQ_W4_ASYM = 0
HQ_W8_SYM = 1
HQ_LAUNCH_DEFAULT = 0
HQ_LAUNCH_PDL = 1
HQ_LAUNCH_DETERMINISTIC = 2
HQ_LAUNCH_EXACT_ORDER = 4
HQ_MAX_M = 128

FORMATS = {"w4": HQ_W4_ASYM, "w8": HQ_W8_SYM}

# Every symbol include/hq.h declares.
EXPORTS = ("hq_tree_accept_workspace_bytes", "hq_tree_accept", "hq_status_string", "hq_version", "hq_packed_bytes", "hq_workspace_bytes", "hq_act_operand_bytes",
           "hq_make_signs",
           "hq_pack_weights", "hq_pack_weights_at", "hq_rotate_quant_act", "hq_verify_gemm", "hq_workspace_q8_bytes",
           "hq_verify_gemm_q8", "hq_unpack_codes", "hq_workspace_status",
           "hq_selftest_wait_timeout", "hq_selftest_gemm_wait_timeout", "hq_verify_gemm_noalloc", "hq_noalloc_status",
           "hq_tree_attention_workspace_bytes",
           "hq_tree_attention", "hq_tree_commit_kv", "hq_delta_tree", "hq_delta_commit")

HQ_ATTN_HEAD_DIM = 128
HQ_DELTA_HEAD_DIM = 128


class HQError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)}")


class hq_layer_desc(ctypes.Structure):
    _fields_ = [("K", ctypes.c_int32), ("N", ctypes.c_int32), ("group", ctypes.c_int32), ("format", ctypes.c_int32)]


_lib = None


def library_path() -> str:
    return _build.LIB


def load() -> ctypes.CDLL:
    """Load libhq.so (building it first if the sources are newer)."""
    global _lib
    if _lib is not None:
        return _lib
    if not _build.up_to_date():
        _build.build()
    if not os.path.exists(_build.LIB):
        raise HQError(HQ_ERR_CUDA, f"libhq.so not found at {_build.LIB}")
    lib = ctypes.CDLL(_build.LIB)
    P, I32, U32, U64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint32, ctypes.c_uint64, ctypes.c_size_t
    D = ctypes.POINTER(hq_layer_desc)
    sig = {
        "hq_status_string": (ctypes.c_char_p, [ctypes.c_int]),
        "hq_version": (I32, []),
        "hq_packed_bytes": (SZ, [D]),
        "hq_workspace_bytes": (SZ, [D, I32]),
        "hq_act_operand_bytes": (SZ, [D, I32]),
        "hq_make_signs": (ctypes.c_int, [U64, I32, P]),
        "hq_pack_weights": (ctypes.c_int, [D, P, P, P, P]),
        "hq_pack_weights_at": (ctypes.c_int, [D, I32, I32, P, P, P, P]),
        "hq_rotate_quant_act": (ctypes.c_int, [D, P, I32, P, P, P, P, P, U32, P]),
        "hq_verify_gemm": (ctypes.c_int, [D, P, P, P, I32, P, P, P, U32, P]),
        "hq_workspace_q8_bytes": (SZ, [D, I32]),
        "hq_verify_gemm_q8": (ctypes.c_int, [D, P, P, P, P, I32, P, P, P, U32, P]),
        "hq_unpack_codes": (ctypes.c_int, [D, P, P, P, P, P]),
        "hq_workspace_status": (ctypes.c_int, [P, P]),
        "hq_selftest_wait_timeout": (ctypes.c_int, [P, ctypes.c_int64, P]),
        "hq_selftest_gemm_wait_timeout": (ctypes.c_int, [D, P, P, P, I32, P, P, ctypes.c_int64, P]),
        "hq_verify_gemm_noalloc": (ctypes.c_int, [D, P, P, P, I32, P, P, U32, P]),
        "hq_noalloc_status": (ctypes.c_int, [P]),
        "hq_tree_accept_workspace_bytes": (SZ, [I32, I32]),
        "hq_tree_accept": (ctypes.c_int, [P, I32, I32, P, P, P, P, P, P, P, U32, P]),
        "hq_tree_attention_workspace_bytes": (SZ, [I32]),
        "hq_tree_attention": (ctypes.c_int, [P, P, P, I32, I32, I32, I32, I32, I32, P, ctypes.c_float, P, P, U32, P]),
        "hq_tree_commit_kv": (ctypes.c_int, [P, P, I32, I32, I32, I32, I32, P, P, U32, P]),
        "hq_delta_tree": (ctypes.c_int, [P, P, P, P, P, P, P, I32, I32, I32, P, U32, P]),
        "hq_delta_commit": (ctypes.c_int, [P, P, P, P, P, P, P, I32, I32, I32, U32, P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().hq_status_string(int(status)).decode()


def _check(rc: int, what: str) -> None:
    if rc != HQ_OK:
        raise HQError(rc, what)


def _ptr(t) -> int | None:
    """A device-pointer argument: None, a raw address (int), or a CUDA tensor
    (which must live on the current device: the library launches there; not
    checked per pointer, to keep eager launches cheap).  Host tensors and numpy
    arrays are refused: the kernels read and write device memory, and on a
    system whose GPU can reach host memory a host buffer would not fault but
    run silently on host memory."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if isinstance(t, torch.Tensor):
        if not t.is_cuda:
            raise TypeError("device memory expected, got a CPU tensor (move it to the GPU first)")
        return t.data_ptr()
    raise TypeError(f"device memory expected, cannot pass {type(t).__name__} as a device pointer")


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def make_desc(K: int, N: int, group: int, fmt) -> hq_layer_desc:
    return hq_layer_desc(int(K), int(N), int(group), FORMATS.get(fmt, fmt) if isinstance(fmt, str) else int(fmt))


# ------------------------------------------------------------ C-ABI calls ---
def hq_version() -> int:
    return int(load().hq_version())


def hq_packed_bytes(desc: hq_layer_desc) -> int:
    return int(load().hq_packed_bytes(ctypes.byref(desc)))


def hq_workspace_bytes(desc: hq_layer_desc, M: int) -> int:
    return int(load().hq_workspace_bytes(ctypes.byref(desc), int(M)))


def hq_act_operand_bytes(desc: hq_layer_desc, M: int) -> int:
    return int(load().hq_act_operand_bytes(ctypes.byref(desc), int(M)))


def hq_make_signs(seed: int, K: int) -> np.ndarray:
    out = np.zeros(max(K // 32, 1), dtype=np.uint32)
    _check(load().hq_make_signs(ctypes.c_uint64(seed & (2 ** 64 - 1)), int(K), out.ctypes.data), "hq_make_signs")
    return out[: K // 32]


def hq_pack_weights(desc, W, signs, blob, stream=None) -> None:
    _check(load().hq_pack_weights(ctypes.byref(desc), _ptr(W), _ptr(signs), _ptr(blob), _stream(stream)),
           "hq_pack_weights")


def hq_pack_weights_at(desc, n0: int, rows: int, W, signs, blob, stream=None) -> None:
    _check(load().hq_pack_weights_at(ctypes.byref(desc), int(n0), int(rows), _ptr(W), _ptr(signs), _ptr(blob),
                                     _stream(stream)), "hq_pack_weights_at")


def hq_rotate_quant_act(desc, X, M: int, signs, qx, gsum, qop, sx, flags: int = 0, stream=None) -> None:
    _check(load().hq_rotate_quant_act(ctypes.byref(desc), _ptr(X), int(M), _ptr(signs), _ptr(qx), _ptr(gsum),
                                      _ptr(qop), _ptr(sx), int(flags), _stream(stream)), "hq_rotate_quant_act")


def hq_verify_gemm(desc, blob, qop, sx, M: int, Y, partials, workspace, flags: int = 0, stream=None) -> None:
    _check(load().hq_verify_gemm(ctypes.byref(desc), _ptr(blob), _ptr(qop), _ptr(sx), int(M), _ptr(Y),
                                 _ptr(partials), _ptr(workspace), int(flags), _stream(stream)), "hq_verify_gemm")


def hq_workspace_q8_bytes(desc: hq_layer_desc, M: int) -> int:
    return int(load().hq_workspace_q8_bytes(ctypes.byref(desc), int(M)))


def hq_verify_gemm_q8(desc, blob, qx, sx, gsum, M: int, Y, partials, workspace, flags: int = 0, stream=None) -> None:
    _check(load().hq_verify_gemm_q8(ctypes.byref(desc), _ptr(blob), _ptr(qx), _ptr(sx), _ptr(gsum), int(M), _ptr(Y),
                                    _ptr(partials), _ptr(workspace), int(flags), _stream(stream)), "hq_verify_gemm_q8")


def hq_unpack_codes(desc, blob, codes, scales, zeros, stream=None) -> None:
    _check(load().hq_unpack_codes(ctypes.byref(desc), _ptr(blob), _ptr(codes), _ptr(scales), _ptr(zeros),
                                  _stream(stream)), "hq_unpack_codes")


def hq_workspace_status(workspace, stream=None) -> int:
    return int(load().hq_workspace_status(_ptr(workspace), _stream(stream)))


def hq_selftest_wait_timeout(workspace, limit_ns: int, stream=None) -> None:
    _check(load().hq_selftest_wait_timeout(_ptr(workspace), int(limit_ns), _stream(stream)),
           "hq_selftest_wait_timeout")


def hq_selftest_gemm_wait_timeout(desc, blob, qop, sx, M: int, Y, workspace, limit_ns: int, stream=None) -> None:
    _check(load().hq_selftest_gemm_wait_timeout(ctypes.byref(desc), _ptr(blob), _ptr(qop), _ptr(sx), int(M), _ptr(Y),
                                                _ptr(workspace), int(limit_ns), _stream(stream)),
           "hq_selftest_gemm_wait_timeout")


HQ_NOALLOC_SCRATCH_BYTES = 60 * 1024 * 1024 + 128 * 1024


def hq_verify_gemm_noalloc(desc, blob, qop, sx, M: int, Y, partials=None, flags: int = 0, stream=None) -> None:
    """hq_verify_gemm with the library's fixed device scratch array instead of a workspace."""
    rc = load().hq_verify_gemm_noalloc(ctypes.byref(desc), _ptr(blob), _ptr(qop), _ptr(sx), int(M), _ptr(Y),
                                       _ptr(partials), int(flags), _stream(stream))
    if rc == HQ_ERR_UNSUPPORTED:
        need = hq_workspace_bytes(desc, M)
        raise HQError(rc, f"hq_verify_gemm_noalloc: this call needs {need} bytes of scratch, more than the "
                          f"library's fixed {HQ_NOALLOC_SCRATCH_BYTES}-byte array")
    _check(rc, "hq_verify_gemm_noalloc")


def hq_noalloc_status(stream=None) -> int:
    """HQ_ERR_TIMEOUT if an allocation-free call on the current device timed out since the last status call."""
    return int(load().hq_noalloc_status(_stream(stream)))


# ------------------------------------------------------- tensor helpers ---
@dataclass
class PackedLayer:
    """A packed layer on the device: its descriptor, blob and device signs."""
    desc: hq_layer_desc
    blob: torch.Tensor
    signs: torch.Tensor

    @property
    def K(self) -> int:
        return self.desc.K

    @property
    def N(self) -> int:
        return self.desc.N

    @property
    def group(self) -> int:
        return self.desc.group

    @property
    def fmt(self) -> int:
        return self.desc.format


def pack_layer(W: torch.Tensor, group: int, fmt, signs_host: np.ndarray, stream=None) -> PackedLayer:
    """Rotate + quantize + pack W [N][K] (fp32, on the device)."""
    N, K = W.shape
    desc = make_desc(K, N, group, fmt)
    nbytes = hq_packed_bytes(desc)
    if nbytes == 0:
        raise HQError(HQ_ERR_INVALID_ARG, "hq_packed_bytes")
    blob = torch.empty(nbytes, dtype=torch.uint8, device=W.device)
    signs = torch.from_numpy(signs_host.astype(np.int32, copy=False).view(np.int32)).to(W.device)
    hq_pack_weights(desc, W.contiguous(), signs, blob, stream)
    return PackedLayer(desc, blob, signs)


@dataclass
class FusedLayer:
    """Several layers that read the same activations, packed into one blob:
    one GEMM computes all of them; `split(Y)` gives each part's outputs as
    views of Y's columns."""
    layer: PackedLayer
    widths: list
    offsets: list

    def split(self, Y: torch.Tensor) -> list:
        return [Y[:, o:o + w] for o, w in zip(self.offsets, self.widths)]


def pack_fused(Ws: list, group: int, fmt, signs_host: np.ndarray, stream=None) -> FusedLayer:
    """Pack the parts Ws (fp32 [N_i][K] on the device, same K) into one blob;
    every part but the last must have a multiple of 128 rows."""
    K = Ws[0].shape[1]
    widths = [int(w.shape[0]) for w in Ws]
    if any(w.shape[1] != K for w in Ws) or any(n % 128 for n in widths[:-1]):
        raise HQError(HQ_ERR_INVALID_ARG, "pack_fused: parts need the same K and widths that are multiples of 128")
    offsets = [sum(widths[:i]) for i in range(len(widths))]
    desc = make_desc(K, sum(widths), group, fmt)
    nbytes = hq_packed_bytes(desc)
    if nbytes == 0:
        raise HQError(HQ_ERR_INVALID_ARG, "hq_packed_bytes")
    dev = Ws[0].device
    blob = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    signs = torch.from_numpy(signs_host.astype(np.int32, copy=False).view(np.int32)).to(dev)
    for W, o in zip(Ws, offsets):
        hq_pack_weights_at(desc, o, W.shape[0], W.contiguous(), signs, blob, stream)
    return FusedLayer(PackedLayer(desc, blob, signs), widths, offsets)


def act_buffers(desc: hq_layer_desc, M: int, device, int8_codes: bool = True, group_sums: bool = False) -> tuple:
    """Buffers of hq_rotate_quant_act for M rows of the activations of layers like `desc`:
    (qx int8 [M][K] or None, gsum int32 [M][K/group] or None, GEMM activation operand (opaque bytes), sx fp32 [M])."""
    K, group = desc.K, desc.group
    qx = torch.empty((M, K), dtype=torch.int8, device=device) if int8_codes else None
    gsum = torch.empty((M, K // group), dtype=torch.int32, device=device) if group_sums else None
    qop = torch.empty(hq_act_operand_bytes(desc, M), dtype=torch.uint8, device=device)
    sx = torch.empty(M, dtype=torch.float32, device=device)
    return qx, gsum, qop, sx


def workspace(desc: hq_layer_desc, M: int, device) -> torch.Tensor:
    n = hq_workspace_bytes(desc, M)
    if n == 0:
        raise HQError(HQ_ERR_INVALID_ARG, "hq_workspace_bytes")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def unpack(layer: PackedLayer, stream=None):
    N, K, G = layer.N, layer.K, layer.group
    dev = layer.blob.device
    codes = torch.empty((N, K), dtype=torch.uint8, device=dev)
    scales = torch.empty((N, K // G), dtype=torch.float32, device=dev)
    zeros = torch.empty((N, K // G), dtype=torch.uint8, device=dev) if layer.fmt == HQ_W4_ASYM else None
    hq_unpack_codes(layer.desc, layer.blob, codes, scales, zeros, stream)
    return codes, scales, zeros


def verify_linear(layer: PackedLayer, X: torch.Tensor, ws: torch.Tensor, Y: torch.Tensor | None = None,
                  bufs=None, flags: int = 0, partials: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Y = dequant(int GEMM(quant(rotate(X)), packed W)): the two kernels in sequence."""
    M, K = X.shape
    if bufs is None:
        bufs = act_buffers(layer.desc, M, X.device, int8_codes=False)
    qx, gsum, qop, sx = bufs
    if Y is None:
        Y = torch.empty((M, layer.N), dtype=torch.float32, device=X.device)
    hq_rotate_quant_act(layer.desc, X, M, layer.signs, qx, gsum, qop, sx, flags & HQ_LAUNCH_PDL, stream)
    hq_verify_gemm(layer.desc, layer.blob, qop, sx, M, Y, partials, ws, flags, stream)
    return Y


def hq_tree_accept_workspace_bytes(M: int, V: int) -> int:
    return int(load().hq_tree_accept_workspace_bytes(int(M), int(V)))


def hq_tree_accept(logits, M: int, V: int, parent, tokens, greedy, path, n_accept, bonus, workspace, flags: int = 0,
                   stream=None) -> None:
    _check(load().hq_tree_accept(_ptr(logits), M, V, _ptr(parent), _ptr(tokens), _ptr(greedy), _ptr(path),
                                 _ptr(n_accept), _ptr(bonus), _ptr(workspace), flags, _stream(stream)),
           "hq_tree_accept")


def tree_accept(logits: torch.Tensor, parent: torch.Tensor, tokens: torch.Tensor, flags: int = 0, stream=None):
    """Greedy tokens, accepted path, number accepted and bonus token of a draft tree (device tensors)."""
    M, V = logits.shape
    dev = logits.device
    greedy = torch.empty(M, dtype=torch.int32, device=dev)
    path = torch.empty(M, dtype=torch.int32, device=dev)
    out = torch.empty(2, dtype=torch.int32, device=dev)
    ws = torch.empty(hq_tree_accept_workspace_bytes(M, V), dtype=torch.uint8, device=dev)
    hq_tree_accept(logits, M, V, parent, tokens, greedy, path, out[0:1], out[1:2], ws, flags, stream)
    return greedy, path, out


def hq_tree_attention_workspace_bytes(Hkv: int) -> int:
    return int(load().hq_tree_attention_workspace_bytes(int(Hkv)))


def hq_tree_attention(q, k_cache, v_cache, cap: int, L: int, M: int, Hq: int, Hkv: int, D: int, parent, scale: float,
                      out, workspace, flags: int = 0, stream=None) -> None:
    _check(load().hq_tree_attention(_ptr(q), _ptr(k_cache), _ptr(v_cache), cap, L, M, Hq, Hkv, D, _ptr(parent),
                                    float(scale), _ptr(out), _ptr(workspace), flags, _stream(stream)),
           "hq_tree_attention")


def hq_tree_commit_kv(k_cache, v_cache, cap: int, L: int, M: int, Hkv: int, D: int, path, n_accept, flags: int = 0,
                      stream=None) -> None:
    _check(load().hq_tree_commit_kv(_ptr(k_cache), _ptr(v_cache), cap, L, M, Hkv, D, _ptr(path), _ptr(n_accept),
                                    flags, _stream(stream)),
           "hq_tree_commit_kv")


def tree_attention(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, L: int, parent: torch.Tensor,
                   scale: float, out: torch.Tensor = None, workspace: torch.Tensor = None, flags: int = 0,
                   stream=None) -> torch.Tensor:
    """Tree-masked attention of the M tree nodes.  q fp16 [M][Hq][D]; k_cache,
    v_cache fp16 [Hkv][cap][D] with the tree nodes at positions [L, L + M);
    parent int32 [M] (device).  Returns fp32 [M][Hq][D]."""
    M, Hq, D = q.shape
    Hkv, cap, _ = k_cache.shape
    if out is None:
        out = torch.empty((M, Hq, D), dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = torch.zeros(hq_tree_attention_workspace_bytes(Hkv), dtype=torch.uint8, device=q.device)
    hq_tree_attention(q, k_cache, v_cache, cap, L, M, Hq, Hkv, D, parent, scale, out, workspace, flags, stream)
    return out


def tree_commit_kv(k_cache: torch.Tensor, v_cache: torch.Tensor, L: int, M: int, path: torch.Tensor,
                   n_accept: torch.Tensor, flags: int = 0, stream=None) -> None:
    """Moves the accepted path next to the root in both caches (in place)."""
    Hkv, cap, D = k_cache.shape
    hq_tree_commit_kv(k_cache, v_cache, cap, L, M, Hkv, D, path, n_accept, flags, stream)


def hq_delta_tree(state, q, k, v, alpha, beta, parent, M: int, H: int, D: int, out, flags: int = 0,
                  stream=None) -> None:
    _check(load().hq_delta_tree(_ptr(state), _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(parent), M, H,
                                D, _ptr(out), flags, _stream(stream)), "hq_delta_tree")


def hq_delta_commit(state, k, v, alpha, beta, path, n_accept, M: int, H: int, D: int, flags: int = 0,
                    stream=None) -> None:
    _check(load().hq_delta_commit(_ptr(state), _ptr(k), _ptr(v), _ptr(alpha), _ptr(beta), _ptr(path),
                                  _ptr(n_accept), M, H, D, flags, _stream(stream)), "hq_delta_commit")


def delta_tree(state: torch.Tensor, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, alpha: torch.Tensor,
               beta: torch.Tensor, parent: torch.Tensor, out: torch.Tensor = None, flags: int = 0,
               stream=None) -> torch.Tensor:
    """Outputs of every tree node of a gated delta-rule layer; the committed
    state [H][D][D] is only read.  q, k, v fp32 [M][H][D]; alpha, beta [M][H]."""
    M, H, D = q.shape
    if out is None:
        out = torch.empty((M, H, D), dtype=torch.float32, device=q.device)
    hq_delta_tree(state, q, k, v, alpha, beta, parent, M, H, D, out, flags, stream)
    return out


def delta_commit(state: torch.Tensor, k: torch.Tensor, v: torch.Tensor, alpha: torch.Tensor, beta: torch.Tensor,
                 path: torch.Tensor, n_accept: torch.Tensor, flags: int = 0, stream=None) -> None:
    """Advances the state (in place) along the root and the accepted path."""
    M, H, D = k.shape
    hq_delta_commit(state, k, v, alpha, beta, path, n_accept, M, H, D, flags, stream)

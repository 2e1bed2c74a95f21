"""The C-ABI library on the host, without a GPU: it loads, exports every
symbol include/hq.h declares, computes sizes, draws the same signs as the
oracle, and rejects invalid arguments before launching anything."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

import oracle
from quantized_speculative_verify_gb300 import hq

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "hq.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(hq_[a-z0-9_]+)\s*\(", src)))


def test_header_and_binding_agree():
    assert declared_functions() == sorted(hq.EXPORTS)


def test_library_exports_every_declared_symbol():
    lib = hq.load()
    out = subprocess.run(["nm", "-D", "--defined-only", hq.library_path()], capture_output=True, text=True,
                         check=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if l.strip()}
    for name in declared_functions():
        assert name in exported, name
        assert getattr(lib, name) is not None


def test_header_compiles_as_c():
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-fsyntax-only", "-x", "c", HEADER],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_status_strings_and_version():
    assert hq.status_string(hq.HQ_OK) == "HQ_OK"
    assert hq.status_string(hq.HQ_ERR_TIMEOUT) == "HQ_ERR_TIMEOUT"
    assert hq.status_string(99) == "HQ_ERR_UNKNOWN"
    assert hq.hq_version() >> 16 == 2  # 2.x: opaque activation operand with group sums, one GEMM launch up to 128 rows


@pytest.mark.parametrize("seed,K", [(0, 32), (1, 4096), (2, 12288), (1234567, 256), (2 ** 63 + 5, 8192)])
def test_make_signs_matches_oracle(seed, K):
    assert np.array_equal(hq.hq_make_signs(seed, K), oracle.make_signs(seed, K))


def test_make_signs_rejects_bad_K():
    lib = hq.load()
    buf = np.zeros(4, dtype=np.uint32)
    for K in (0, -32, 48):
        assert lib.hq_make_signs(1, K, buf.ctypes.data) == hq.HQ_ERR_INVALID_ARG
    assert lib.hq_make_signs(1, 64, None) == hq.HQ_ERR_INVALID_ARG


@pytest.mark.parametrize("K,N,G,fmt", [(256, 256, 32, "w4"), (4096, 4096, 64, "w4"), (4096, 24576, 128, "w8"),
                                       (8192, 8192, 64, "w4"), (8192, 8192, 128, "w8"), (12288, 4096, 64, "w4"),
                                       (4096, 151552, 64, "w4"), (4096, 1024, 256, "w4"), (4096, 1024, 16, "w8")])
def test_packed_bytes_equal_algorithmic_bytes(K, N, G, fmt):
    d = hq.make_desc(K, N, G, fmt)
    per_weight = (0.5 + 4.5 / G) if fmt == "w4" else (1.0 + 4.0 / G)
    assert hq.hq_packed_bytes(d) == int(round(N * K * per_weight))
    assert hq.hq_packed_bytes(d) % 16 == 0


def test_packed_bytes_pad_ragged_shapes():
    # N and K are padded to whole 128 x 128 tiles
    d = hq.make_desc(96, 200, 32, "w4")
    assert hq.hq_packed_bytes(d) == 2 * 1 * (128 * 128 // 2 + 4 * 128 * 4 + 4 * 64)


@pytest.mark.parametrize("K,N,G,fmt", [(0, 8, 32, 0), (48, 8, 16, 0), (64, 8, 48, 0), (96, 8, 64, 0), (64, 0, 32, 0),
                                       (64, 8, 32, 2), (64, 8, 512, 1), (64, -1, 32, 1)])
def test_invalid_desc_has_no_size(K, N, G, fmt):
    d = hq.hq_layer_desc(K, N, G, fmt)
    assert hq.hq_packed_bytes(d) == 0
    assert hq.hq_workspace_bytes(d, 16) == 0


def test_tile_count_bound():
    # the kernels index tiles with ints: at most 2^30 tiles (128 channels x 128 features each) per layer
    at_bound = hq.hq_layer_desc(1 << 16, 1 << 28, 64, hq.HQ_W4_ASYM)  # 2^21 x 2^9 tiles
    assert hq.hq_packed_bytes(at_bound) == (1 << 30) * (128 * 128 // 2 + 2 * 128 * 4 + 2 * 128 // 2)
    beyond = hq.hq_layer_desc(1 << 16, (1 << 28) + 128, 64, hq.HQ_W4_ASYM)
    assert hq.hq_packed_bytes(beyond) == 0 and hq.hq_workspace_bytes(beyond, 16) == 0
    lib = hq.load()
    fake = 0x10000  # never dereferenced: the descriptor is rejected first
    assert lib.hq_verify_gemm(ctypes.byref(beyond), fake, fake, fake, 16, fake, None, fake, 0, None) == \
        hq.HQ_ERR_INVALID_ARG
    assert lib.hq_pack_weights(ctypes.byref(beyond), fake, fake, fake, None) == hq.HQ_ERR_INVALID_ARG


@pytest.mark.parametrize("K", [65536 + 64, 1 << 24, 2 ** 31 - 64])
def test_K_above_the_activation_limit_is_invalid(K):
    # K is bounded by what one activation row may hold (65536), far below
    # where the tile arithmetic (K + 127 in int) could overflow
    d = hq.hq_layer_desc(K, 128, 64, hq.HQ_W4_ASYM)
    assert hq.hq_packed_bytes(d) == 0 and hq.hq_workspace_bytes(d, 16) == 0
    ok = hq.hq_layer_desc(65536, 128, 64, hq.HQ_W4_ASYM)
    assert hq.hq_packed_bytes(ok) > 0
    lib = hq.load()
    fake = 0x10000
    assert lib.hq_verify_gemm(ctypes.byref(d), fake, fake, fake, 16, fake, None, fake, 0, None) == \
        hq.HQ_ERR_INVALID_ARG


def test_q8_workspace_and_argument_checks():
    d = hq.make_desc(4096, 384, 64, "w4")
    for M in (1, 16, 40, 128):
        assert hq.hq_workspace_q8_bytes(d, M) >= hq.hq_workspace_bytes(d, M) + hq.hq_act_operand_bytes(d, M)
        assert hq.hq_workspace_q8_bytes(d, M) % 16 == 0
    assert hq.hq_workspace_q8_bytes(d, 129) == 0 and hq.hq_workspace_q8_bytes(d, -1) == 0
    lib = hq.load()
    FAKE = ctypes.c_void_p(0x10000)
    E = hq.HQ_ERR_INVALID_ARG
    D = ctypes.byref(d)
    # null pointers, bad M, unknown flags, misaligned workspace: refused before any launch
    assert lib.hq_verify_gemm_q8(D, None, FAKE, FAKE, None, 4, FAKE, None, FAKE, 0, None) == E
    assert lib.hq_verify_gemm_q8(D, FAKE, None, FAKE, None, 4, FAKE, None, FAKE, 0, None) == E
    assert lib.hq_verify_gemm_q8(D, FAKE, FAKE, FAKE, None, 129, FAKE, None, FAKE, 0, None) == E
    assert lib.hq_verify_gemm_q8(D, FAKE, FAKE, FAKE, None, 4, FAKE, None, FAKE, 1 << 9, None) == E
    assert lib.hq_verify_gemm_q8(D, FAKE, FAKE, FAKE, None, 4, FAKE, None, ctypes.c_void_p(0x10008), 0, None) == E
    assert lib.hq_verify_gemm_q8(D, FAKE, FAKE, FAKE, None, 0, FAKE, None, FAKE, 0, None) == hq.HQ_OK


def test_act_operand_bytes():
    # opaque, but its size follows from the rows padded to the MMA's N (16, 32,
    # 64, 128), 128-feature blocks of 2 bytes per code (fp16, or two e4m3
    # digits; rows of 272 bytes for the register-resident GEMM up to 32
    # rows), and one fp32 sum per group and row where the
    # GEMM applies a 4-bit zero point through them (above 32 rows)
    def size(M, K, G, fmt="w4"):
        return hq.hq_act_operand_bytes(hq.make_desc(K, 128, G, fmt), M)
    assert size(16, 4096, 64) == 32 * 16 * 272  # the zero point is applied to the weights
    assert size(16, 4096, 64, "w8") == 32 * 16 * 272
    assert size(33, 4096, 64, "w8") == 32 * 64 * 256  # the tensor-memory GEMM's encoding
    assert size(3, 96, 32) == 1 * 16 * 272  # one padded block
    assert size(32, 4096, 256) == 32 * 32 * 272
    assert size(33, 512, 256) == 4 * 64 * 256 + 2 * 64 * 4  # group sums for the 4-bit zero point
    assert size(33, 512, 256, "w8") == 4 * 64 * 256  # symmetric: no zero point
    assert size(128, 4096, 16) == 32 * 128 * 256 + 256 * 128 * 4
    assert size(0, 4096, 64) == 0 and size(129, 4096, 64) == 0
    for bad in (hq.hq_layer_desc(100, 128, 32, 0), hq.hq_layer_desc(96, 128, 64, 0), hq.hq_layer_desc(256, 128, 48, 0)):
        assert hq.hq_act_operand_bytes(bad, 4) == 0


def test_workspace_bytes():
    d = hq.make_desc(4096, 4096, 64, "w4")
    assert hq.hq_workspace_bytes(d, 16) == hq.hq_workspace_bytes(d, 1) > 20 * 1024 * 1024
    assert hq.hq_workspace_bytes(d, 129) == 0 and hq.hq_workspace_bytes(d, -1) == 0
    assert hq.hq_workspace_bytes(d, 128) == hq.hq_workspace_bytes(d, 1)  # one launch for every M
    assert hq.hq_workspace_bytes(d, 16) % 16 == 0
    # a wider layer needs more counters, at the same offsets: a workspace sized
    # for the widest layer serves every layer
    wide = hq.make_desc(4096, 24576, 64, "w4")
    assert hq.hq_workspace_bytes(wide, 16) - hq.hq_workspace_bytes(d, 16) == (192 - 32) * 8


FAKE = 0x10000  # a 16-byte aligned non-NULL value; never dereferenced: every call below fails validation


def test_invalid_arguments_are_rejected_before_launch():
    lib = hq.load()
    d = hq.make_desc(256, 256, 32, "w4")
    D = ctypes.byref(d)
    bad = hq.hq_layer_desc(100, 256, 32, 0)
    E = hq.HQ_ERR_INVALID_ARG
    # pack
    assert lib.hq_pack_weights(None, FAKE, FAKE, FAKE, None) == E
    assert lib.hq_pack_weights(ctypes.byref(bad), FAKE, FAKE, FAKE, None) == E
    assert lib.hq_pack_weights(D, None, FAKE, FAKE, None) == E
    assert lib.hq_pack_weights(D, FAKE, FAKE, FAKE + 8, None) == E  # blob must be 16-byte aligned
    # activations: (desc, X, M, signs, qx, gsum, qop, sx, flags, stream)
    assert lib.hq_rotate_quant_act(D, FAKE, 129, FAKE, FAKE, None, FAKE, FAKE, 0, None) == E
    assert lib.hq_rotate_quant_act(D, FAKE, -1, FAKE, FAKE, None, FAKE, FAKE, 0, None) == E
    assert lib.hq_rotate_quant_act(ctypes.byref(bad), FAKE, 4, FAKE, FAKE, None, FAKE, FAKE, 0, None) == E
    assert lib.hq_rotate_quant_act(None, FAKE, 4, FAKE, FAKE, None, FAKE, FAKE, 0, None) == E
    assert lib.hq_rotate_quant_act(D, None, 4, FAKE, FAKE, None, FAKE, FAKE, 0, None) == E
    assert lib.hq_rotate_quant_act(D, FAKE, 4, FAKE, None, None, None, FAKE, 0, None) == E  # no output
    assert lib.hq_rotate_quant_act(D, FAKE + 4, 4, FAKE, FAKE, None, FAKE, FAKE, 0, None) == E
    assert lib.hq_rotate_quant_act(D, FAKE, 4, FAKE, FAKE, None, FAKE + 8, FAKE, 0, None) == E  # operand
    assert lib.hq_rotate_quant_act(D, FAKE, 4, FAKE, FAKE, FAKE + 2, FAKE, FAKE, 0, None) == E  # gsum
    assert lib.hq_rotate_quant_act(D, FAKE, 4, FAKE, FAKE, None, FAKE, FAKE, 2, None) == E
    # gemm
    assert lib.hq_verify_gemm(D, FAKE, FAKE, FAKE, 129, FAKE, None, FAKE, 0, None) == E
    assert lib.hq_verify_gemm(D, None, FAKE, FAKE, 4, FAKE, None, FAKE, 0, None) == E
    assert lib.hq_verify_gemm(D, FAKE, None, FAKE, 4, FAKE, None, FAKE, 0, None) == E
    assert lib.hq_verify_gemm(D, FAKE, FAKE, FAKE, 4, FAKE, None, None, 0, None) == E  # workspace
    assert lib.hq_verify_gemm(D, FAKE + 8, FAKE, FAKE, 4, FAKE, None, FAKE, 0, None) == E
    assert lib.hq_verify_gemm(D, FAKE, FAKE + 8, FAKE, 4, FAKE, None, FAKE, 0, None) == E
    assert lib.hq_verify_gemm(D, FAKE, FAKE, FAKE, 4, FAKE, None, FAKE, 8, None) == E
    assert lib.hq_verify_gemm(D, FAKE, FAKE, FAKE, 4, FAKE, None, FAKE, 16, None) == E  # unknown flag bit
    assert lib.hq_verify_gemm(ctypes.byref(bad), FAKE, FAKE, FAKE, 4, FAKE, None, FAKE, 0, None) == E
    # unpack / status / self-test
    assert lib.hq_unpack_codes(D, FAKE, FAKE, FAKE, None, None) == E  # W4 needs zeros
    assert lib.hq_workspace_status(None, None) == E
    assert lib.hq_selftest_wait_timeout(FAKE, 10, None) == E
    assert lib.hq_selftest_wait_timeout(None, 10 ** 6, None) == E
    assert lib.hq_selftest_gemm_wait_timeout(D, FAKE, FAKE, FAKE, 4, FAKE, FAKE, 10, None) == E
    assert lib.hq_selftest_gemm_wait_timeout(D, FAKE, FAKE, FAKE, 0, FAKE, FAKE, 10 ** 6, None) == E
    assert lib.hq_selftest_gemm_wait_timeout(D, FAKE, FAKE, FAKE, 4, FAKE, None, 10 ** 6, None) == E


def test_empty_batch_is_a_no_op():
    lib = hq.load()
    d = hq.make_desc(256, 256, 32, "w4")
    # M = 0: nothing to do, nothing launched, pointers never touched
    assert lib.hq_rotate_quant_act(ctypes.byref(d), None, 0, None, None, None, None, None, 0, None) == hq.HQ_OK
    assert lib.hq_verify_gemm(ctypes.byref(d), None, None, None, 0, None, None, None, 0, None) == hq.HQ_OK


def test_tree_accept_sizes_and_validation():
    lib = hq.load()
    assert hq.hq_tree_accept_workspace_bytes(16, 151552) == 16 * 19 * 8
    assert hq.hq_tree_accept_workspace_bytes(0, 100) == 0 and hq.hq_tree_accept_workspace_bytes(129, 100) == 0
    assert hq.hq_tree_accept_workspace_bytes(4, 0) == 0
    E = hq.HQ_ERR_INVALID_ARG
    args = [FAKE, 4, 100, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, None]
    assert lib.hq_tree_accept(*args[:1], 0, *args[2:]) == E          # M = 0
    assert lib.hq_tree_accept(*args[:1], 129, *args[2:]) == E        # M > HQ_MAX_M
    assert lib.hq_tree_accept(*args[:2], 0, *args[3:]) == E          # V = 0
    assert lib.hq_tree_accept(None, *args[1:]) == E
    assert lib.hq_tree_accept(*args[:9], FAKE + 8, 0, None) == E     # workspace alignment
    assert lib.hq_tree_accept(*args[:10], 2, None) == E              # unknown flag


def test_tree_attention_arguments_are_checked_before_launch():
    lib = hq.load()
    E, U = hq.HQ_ERR_INVALID_ARG, hq.HQ_ERR_UNSUPPORTED
    D = hq.HQ_ATTN_HEAD_DIM
    ok = dict(q=FAKE, k=FAKE, v=FAKE, cap=100, L=50, M=16, Hq=32, Hkv=8, D=D, parent=FAKE, scale=0.1, out=FAKE,
              ws=FAKE, flags=0)

    def call(**kw):
        a = dict(ok, **kw)
        return lib.hq_tree_attention(a["q"], a["k"], a["v"], a["cap"], a["L"], a["M"], a["Hq"], a["Hkv"], a["D"],
                                     a["parent"], a["scale"], a["out"], a["ws"], a["flags"], None)
    assert call(M=0) == E and call(M=129) == E and call(L=-1) == E
    assert call(cap=65) == E                      # L + M > cap
    assert call(Hq=30) == E and call(Hkv=0) == E  # Hq not a multiple of Hkv
    assert call(q=None) == E and call(ws=None) == E and call(parent=None) == E
    assert call(k=FAKE + 8) == E and call(out=FAKE + 4) == E
    assert call(flags=2) == E and call(scale=float("nan")) == E and call(scale=float("inf")) == E
    assert call(D=64) == U                        # head dimension other than 128
    assert call(Hq=96, Hkv=1) == U                # 64 not a multiple of Hq / Hkv
    assert hq.hq_tree_attention_workspace_bytes(8) == 16 + 8 * 4096 * (D + 2) * 4
    assert hq.hq_tree_attention_workspace_bytes(0) == 0
    # commit
    c = lib.hq_tree_commit_kv
    assert c(FAKE, FAKE, 60, 50, 16, 8, D, FAKE, FAKE, 0, None) == E   # L + M > cap
    assert c(None, FAKE, 100, 50, 16, 8, D, FAKE, FAKE, 0, None) == E
    assert c(FAKE, FAKE, 100, 50, 16, 8, D, None, FAKE, 0, None) == E
    assert c(FAKE, FAKE, 100, 50, 0, 8, D, FAKE, FAKE, 0, None) == E
    assert c(FAKE, FAKE, 100, 50, 16, 8, 64, FAKE, FAKE, 0, None) == U
    assert c(FAKE, FAKE, 100, 50, 16, 8, D, FAKE, FAKE, 4, None) == E


def test_delta_arguments_are_checked_before_launch():
    lib = hq.load()
    E, U = hq.HQ_ERR_INVALID_ARG, hq.HQ_ERR_UNSUPPORTED
    D = hq.HQ_DELTA_HEAD_DIM
    t = lib.hq_delta_tree
    assert t(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, 4, D, FAKE, 0, None) == E    # M = 0
    assert t(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 129, 4, D, FAKE, 0, None) == E  # M > 128
    assert t(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 16, 0, D, FAKE, 0, None) == E   # no head
    assert t(None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 16, 4, D, FAKE, 0, None) == E
    assert t(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 16, 4, D, None, 0, None) == E
    assert t(FAKE, FAKE + 4, FAKE, FAKE, FAKE, FAKE, FAKE, 16, 4, D, FAKE, 0, None) == E  # q not 16-byte aligned
    assert t(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 16, 4, D, FAKE, 2, None) == E
    assert t(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 16, 4, 64, FAKE, 0, None) == U
    c = lib.hq_delta_commit
    assert c(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 0, 4, D, 0, None) == E
    assert c(FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, 16, 4, D, 0, None) == E
    assert c(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, 16, 4, D, 0, None) == E
    assert c(FAKE + 8, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 16, 4, D, 0, None) == E
    assert c(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 16, 4, 256, 0, None) == U


def test_binding_refuses_host_buffers_as_device_pointers():
    # the kernels read and write device memory; a host buffer is refused
    # before the library is called (no GPU needed to see it)
    import torch
    d = hq.make_desc(256, 256, 32, "w4")
    with pytest.raises(TypeError, match="CPU tensor"):
        hq.hq_rotate_quant_act(d, torch.zeros((1, 256)), 1, None, None, None, None, None)
    with pytest.raises(TypeError, match="ndarray"):
        hq.hq_verify_gemm(d, np.zeros(16, dtype=np.uint8), None, None, 1, None, None, None)
    with pytest.raises(TypeError, match="CPU tensor"):
        hq.tree_attention(torch.zeros((1, 8, hq.HQ_ATTN_HEAD_DIM), dtype=torch.float16),
                          torch.zeros((1, 4, hq.HQ_ATTN_HEAD_DIM), dtype=torch.float16),
                          torch.zeros((1, 4, hq.HQ_ATTN_HEAD_DIM), dtype=torch.float16), 3,
                          torch.zeros(1, dtype=torch.int32), 0.1)

"""hq_verify_gemm_noalloc: the verify GEMM for callers that cannot allocate.

Some callers cannot call cudaMalloc where they run the verify GEMM: a plugin
whose host process owns every device allocation, a memory-capped serving
process whose allocator refuses new blocks, or code on a latency-critical
path where an allocation would synchronize the device.  For them the library
exports one more entry point that takes no workspace and allocates nothing:
its scratch is a fixed file-scope device array inside the library.  These
tests check that it gives the same outputs as hq_verify_gemm with a caller
workspace, on two calls in a row (the array keeps the previous call's
contents), and that calls needing more scratch than the array are refused.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from quantized_speculative_verify_gb300 import hq, synth

ATOL, RTOL = 1e-6, 1e-5


def test_noalloc_refuses_calls_larger_than_its_array():
    lib = hq.load()
    d = hq.make_desc(4096, 4096, 64, "w4")
    fake = 0x10000  # never dereferenced: the size check comes first
    # every M fits (the GEMM runs at most 32 rows per launch); a huge N does not
    assert hq.hq_workspace_bytes(d, 128) <= hq.HQ_NOALLOC_SCRATCH_BYTES
    wide = hq.make_desc(4096, 128 * 20000, 64, "w4")
    assert hq.hq_workspace_bytes(wide, 32) > hq.HQ_NOALLOC_SCRATCH_BYTES
    rc = lib.hq_verify_gemm_noalloc(ctypes.byref(wide), fake, fake, fake, 32, fake, None, 0, None)
    assert rc == hq.HQ_ERR_UNSUPPORTED
    rc = lib.hq_verify_gemm_noalloc(ctypes.byref(d), None, fake, fake, 16, fake, None, 0, None)
    assert rc == hq.HQ_ERR_INVALID_ARG
    assert lib.hq_verify_gemm_noalloc(ctypes.byref(d), None, None, None, 0, None, None, 0, None) == hq.HQ_OK


def test_noalloc_rejects_descriptors_beyond_the_kernel_limits():
    lib = hq.load()
    fake = 0x10000  # never dereferenced: the descriptor is rejected first
    for d in (hq.hq_layer_desc(65536, (1 << 28) + 128, 64, hq.HQ_W4_ASYM),  # one n-block past 2^30 tiles
              hq.hq_layer_desc(65536 + 64, 128, 64, hq.HQ_W4_ASYM),         # K past the activation limit
              hq.hq_layer_desc(2 ** 31 - 64, 128, 64, hq.HQ_W4_ASYM)):      # K near the int range
        rc = lib.hq_verify_gemm_noalloc(ctypes.byref(d), fake, fake, fake, 16, fake, None, 0, None)
        assert rc == hq.HQ_ERR_INVALID_ARG


def _layer(fmt, M, K, N, G, dev):
    X = synth.activations(M, K, seed=M + 3, outlier_channels=2).to(dev)
    W = synth.weights(N, K, seed=N + 5).to(dev)
    signs = hq.hq_make_signs(17, K)
    layer = hq.pack_layer(W, G, fmt, signs)
    _, _, qop, sx = hq.act_buffers(layer.desc, M, dev, int8_codes=False)
    hq.hq_rotate_quant_act(layer.desc, X, M, layer.signs, None, None, qop, sx)
    return layer, qop, sx


@pytest.mark.gpu
@pytest.mark.parametrize("fmt,M,K,N,G", [("w4", 16, 4096, 1024, 64), ("w8", 32, 4096, 384, 128),
                                         ("w4", 5, 512, 200, 32), ("w4", 70, 1024, 256, 64)])
def test_noalloc_matches_workspace_entry_point_twice(fmt, M, K, N, G):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = "cuda"
    layer, qop, sx = _layer(fmt, M, K, N, G, dev)
    ws = hq.workspace(layer.desc, M, dev)
    det = hq.HQ_LAUNCH_DETERMINISTIC
    y_ref = torch.empty((M, N), dtype=torch.float32, device=dev)
    hq.hq_verify_gemm(layer.desc, layer.blob, qop, sx, M, y_ref, None, ws, det)
    assert hq.hq_workspace_status(ws) == hq.HQ_OK
    ref = y_ref.cpu().numpy()
    # fixed summation order: the two entry points agree bit for bit, with and
    # without programmatic dependent launch
    for call, flags in enumerate((det, det, det | hq.HQ_LAUNCH_PDL)):
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device=dev)
        hq.hq_verify_gemm_noalloc(layer.desc, layer.blob, qop, sx, M, y, flags=flags)
        torch.cuda.synchronize()
        assert np.array_equal(y.cpu().numpy().view(np.uint32), ref.view(np.uint32)), f"call {call + 1} differs"
        assert hq.hq_noalloc_status() == hq.HQ_OK
    # accumulating mode: every output written, within 1e-5 of the row's largest output
    y = torch.full((M, N), float("nan"), dtype=torch.float32, device=dev)
    hq.hq_verify_gemm_noalloc(layer.desc, layer.blob, qop, sx, M, y)
    torch.cuda.synchronize()
    assert hq.hq_noalloc_status() == hq.HQ_OK
    got = y.cpu().numpy().astype(np.float64)
    r64 = ref.astype(np.float64)
    assert np.all(np.abs(got - r64) <= ATOL + RTOL * np.abs(r64).max(axis=1, keepdims=True))


@pytest.mark.gpu
def test_noalloc_check_mode_partials_match_bit_for_bit():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = "cuda"
    M, K, N, G = 16, 2048, 640, 64
    layer, qop, sx = _layer("w4", M, K, N, G, dev)
    ws = hq.workspace(layer.desc, M, dev)
    p_ref = torch.empty((M, N, K // G), dtype=torch.int32, device=dev)
    y_ref = torch.empty((M, N), dtype=torch.float32, device=dev)
    hq.hq_verify_gemm(layer.desc, layer.blob, qop, sx, M, y_ref, p_ref, ws, hq.HQ_LAUNCH_DETERMINISTIC)
    for _ in range(2):
        p = torch.full((M, N, K // G), -1, dtype=torch.int32, device=dev)
        y = torch.full((M, N), float("nan"), dtype=torch.float32, device=dev)
        hq.hq_verify_gemm_noalloc(layer.desc, layer.blob, qop, sx, M, y, p, flags=hq.HQ_LAUNCH_DETERMINISTIC)
        torch.cuda.synchronize()
        assert torch.equal(p, p_ref)
        assert np.array_equal(y.cpu().numpy().view(np.uint32), y_ref.cpu().numpy().view(np.uint32))
    assert hq.hq_noalloc_status() == hq.HQ_OK


@pytest.mark.gpu
def test_noalloc_wide_call_then_narrow_call():
    # a wide layer's counters must not leak into the next, narrower call
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    dev = "cuda"
    wide = _layer("w4", 16, 4096, 8192, 64, dev)
    narrow = _layer("w4", 16, 4096, 384, 64, dev)
    refs = []
    for layer, qop, sx in (wide, narrow):
        ws = hq.workspace(layer.desc, 16, dev)
        y = torch.empty((16, layer.N), dtype=torch.float32, device=dev)
        hq.hq_verify_gemm(layer.desc, layer.blob, qop, sx, 16, y, None, ws, hq.HQ_LAUNCH_DETERMINISTIC)
        refs.append(y.cpu().numpy())
    for rep in range(2):
        for (layer, qop, sx), ref in zip((wide, narrow), refs):
            y = torch.full((16, layer.N), float("nan"), dtype=torch.float32, device=dev)
            hq.hq_verify_gemm_noalloc(layer.desc, layer.blob, qop, sx, 16, y, flags=hq.HQ_LAUNCH_DETERMINISTIC)
            torch.cuda.synchronize()
            assert np.array_equal(y.cpu().numpy().view(np.uint32), ref.view(np.uint32)), (rep, layer.N)
    assert hq.hq_noalloc_status() == hq.HQ_OK

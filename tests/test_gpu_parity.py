"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Integer stages (int8 activations, row scales, group sums, packed codes,
scales, zero points, per-group int32 partial sums) must match bit for bit;
fp32 outputs within |dY| <= 1e-6 + 1e-5 |Y_oracle|.  Inputs are seeded and
synthetic (quantized_speculative_verify_gb300.synth); the oracle and the GPU
receive the same arrays.  Large shapes compare a seeded sample of output
channels: each channel depends only on its own weight row, so the oracle
quantizes just the sampled rows.
"""
import numpy as np
import pytest
import torch

import oracle
from quantized_speculative_verify_gb300 import hq, synth
from guard import Guarded
from tolerance import ATOL, RTOL, assert_close, strict_fraction  # noqa: F401

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    hq.load()


def gpu_act(X, signs_dev, G, fmt="w4"):
    M, K = X.shape
    desc = hq.make_desc(K, 128, G, fmt)
    qx = Guarded((M, K), torch.int8, DEV)
    gsum = Guarded((M, K // G), torch.int32, DEV)
    qop = Guarded((hq.hq_act_operand_bytes(desc, M),), torch.uint8, DEV, fill=0xFF)  # padding must be written
    sx = Guarded((M,), torch.float32, DEV)
    hq.hq_rotate_quant_act(desc, X, M, signs_dev, qx.t, gsum.t, qop.t, sx.t)
    torch.cuda.synchronize()
    for name, g in (("qx", qx), ("gsum", gsum), ("operand", qop), ("sx", sx)):
        g.check(name)
    return qx.t, gsum.t, qop.t, sx.t


def check_act(qx, gsum, sx, rq, rs, rg):
    assert np.array_equal(qx.cpu().numpy(), rq)
    assert np.array_equal(gsum.cpu().numpy(), rg)
    assert np.array_equal(sx.cpu().numpy().view(np.uint32), rs.view(np.uint32))


def signs_pair(seed, K):
    s = hq.hq_make_signs(seed, K)
    return s, torch.from_numpy(s.view(np.int32)).to(DEV)


# ------------------------------------------------------- activations ---
ACT_CASES = [(1, 32, 32), (3, 64, 16), (16, 256, 32), (17, 256, 64), (16, 4096, 64), (32, 4096, 128),
             (7, 4096, 256), (16, 12288, 64), (128, 4096, 16), (64, 8192, 128), (5, 96, 32), (2, 40960, 256),
             (4, 2048, 64), (3, 16384, 128), (2, 32768, 256), (9, 1024, 32)]


@pytest.mark.parametrize("M,K,G", ACT_CASES)
def test_rotate_quant_act_bit_exact(M, K, G):
    X = synth.activations(M, K, seed=M * 7 + K, outlier_channels=min(2, K), heavy_frac=0.01)
    s_host, s_dev = signs_pair(M + K, K)
    rq, rs, rg = oracle.quant_act(X.numpy(), G, s_host)
    for fmt in ("w4", "w8"):  # the two operand encodings
        qx, gsum, qop, sx = gpu_act(X.to(DEV), s_dev, G, fmt)
        check_act(qx, gsum, sx, rq, rs, rg)


def test_rotate_quant_act_degenerate_rows():
    M, K, G = 6, 256, 32
    X = synth.activations(M, K, seed=3)
    X[1] = 0.0                       # all-zero row -> scale 0, codes 0
    X[2] = 0.0
    X[2, 37] = -5.0                  # one outlier -> spread over its block
    X[3] = 1e-30                     # tiny values (subnormal products)
    X[4, :32] = 3.0                  # constant block
    X[5] = 1e30                      # huge values
    s_host, s_dev = signs_pair(9, K)
    qx, gsum, qop, sx = gpu_act(X.to(DEV), s_dev, G)
    rq, rs, rg = oracle.quant_act(X.numpy(), G, s_host)
    check_act(qx, gsum, sx, rq, rs, rg)
    assert sx[1].item() == 0.0 and not qx[1].any()


def test_rotate_quant_act_nan_does_not_crash():
    M, K, G = 2, 64, 32
    X = synth.activations(M, K, seed=4)
    X[0, 3] = float("nan")
    X[1, 9] = float("inf")
    _, s_dev = signs_pair(1, K)
    gpu_act(X.to(DEV), s_dev, G)  # values unspecified; it must return


# ----------------------------------------------------------- packing ---
PACK_CASES = [("w4", 256, 256, 32), ("w4", 4096, 4096, 64), ("w8", 4096, 1024, 128), ("w4", 32, 200, 32),
              ("w4", 96, 130, 16), ("w8", 64, 1, 32), ("w4", 12288, 256, 64), ("w8", 512, 384, 256),
              ("w4", 1024, 136, 128), ("w4", 512, 128, 256), ("w8", 256, 256, 16)]


def gpu_pack(W, G, fmt, s_host):
    layer = hq.pack_layer(W.to(DEV), G, fmt, s_host)
    codes, scales, zeros = hq.unpack(layer)
    torch.cuda.synchronize()
    return layer, codes, scales, zeros


@pytest.mark.parametrize("fmt,K,N,G", PACK_CASES)
def test_pack_bit_exact(fmt, K, N, G):
    W = synth.weights(N, K, seed=K + N, outlier_frac=0.005)
    if N > 3:
        W[2, :] = 0.0             # all-zero channel
        W[3, : min(K, 64)] = 0.25  # constant stretch
    s_host, _ = signs_pair(K * 3 + G, K)
    _, codes, scales, zeros = gpu_pack(W, G, fmt, s_host)
    if fmt == "w4":
        rc, rs, rz = oracle.quant_w4(W.numpy(), G, s_host, openmp=True)
        assert np.array_equal(zeros.cpu().numpy(), rz)
    else:
        rc, rs = oracle.quant_w8(W.numpy(), G, s_host, openmp=True)
        rc = rc.view(np.uint8)
    assert np.array_equal(codes.cpu().numpy(), rc)
    assert np.array_equal(scales.cpu().numpy().view(np.uint32), rs.view(np.uint32))


# ---------------------------------------------------------------- GEMM ---
# workspace: 16-byte error word, 480 blocks x 2 slots x 128 x 128 fp32 partial sums, counters
COUNTER_OFFSET = 16 + 480 * 2 * 128 * 128 * 4


def run_layer(X, W, G, fmt, s_host, check=False, flags=0, layer=None):
    M, K = X.shape
    if layer is None:
        layer = hq.pack_layer(W.to(DEV), G, fmt, s_host)
    ws = hq.workspace(layer.desc, M, DEV)
    bufs = hq.act_buffers(layer.desc, M, DEV)
    P = Guarded((M, layer.N, K // G), torch.int32, DEV) if check else None
    # Y starts as NaN: an output the kernel fails to write (or to zero before
    # accumulating into it) stays NaN and fails the comparison; both live
    # between guard bands
    Y = Guarded((M, layer.N), torch.float32, DEV, fill=float("nan"))
    hq.verify_linear(layer, X.to(DEV), ws, Y=Y.t, bufs=bufs, partials=None if P is None else P.t, flags=flags)
    assert hq.hq_workspace_status(ws) == hq.HQ_OK
    torch.cuda.synchronize()
    Y.check("Y")
    if P is not None:
        P.check("partials")
    # every call leaves the error word and the n-block counters (after the
    # partial-sum slots) at zero
    assert not ws[:16].any() and not ws[COUNTER_OFFSET:].any()
    return dict(Y=Y.t.cpu().numpy(), P=None if P is None else P.t.cpu().numpy(), layer=layer, ws=ws)


GEMM_CASES = [("w4", 1, 256, 256, 32), ("w4", 16, 256, 256, 32), ("w4", 3, 512, 200, 64), ("w8", 17, 384, 136, 128),
              ("w4", 32, 1024, 1024, 16), ("w8", 8, 1024, 512, 32), ("w4", 64, 512, 256, 64), ("w8", 128, 256, 384, 128),
              ("w4", 128, 256, 128, 256), ("w4", 16, 32, 136, 32), ("w8", 24, 96, 64, 32), ("w4", 5, 12288, 128, 64),
              ("w8", 1, 4096, 256, 256), ("w4", 40, 2048, 1000, 128)]


@pytest.mark.parametrize("flags", [hq.HQ_LAUNCH_DEFAULT, hq.HQ_LAUNCH_DETERMINISTIC])
@pytest.mark.parametrize("fmt,M,K,N,G", GEMM_CASES)
def test_gemm_partials_bit_exact_and_output_close(fmt, M, K, N, G, flags):
    X = synth.activations(M, K, seed=M + K, outlier_channels=2)
    W = synth.weights(N, K, seed=N + K + 1, outlier_frac=0.005)
    s_host, _ = signs_pair(M * N + K, K)
    r = run_layer(X, W, G, fmt, s_host, check=True, flags=flags)
    ref = oracle.verify_linear(X.numpy(), W.numpy(), G, fmt, s_host)
    assert np.array_equal(r["P"], ref["P"])
    assert_close(r["Y"], ref)


@pytest.mark.parametrize("flags", [hq.HQ_LAUNCH_DEFAULT, hq.HQ_LAUNCH_DETERMINISTIC | hq.HQ_LAUNCH_PDL])
@pytest.mark.parametrize("fmt,M,K,N,G", GEMM_CASES)
def test_gemm_default_mode_output_close(fmt, M, K, N, G, flags):
    # without check mode the kernel folds each group with one fused
    # multiply-add (the instance the verify pass runs)
    X = synth.activations(M, K, seed=M + K + 7, outlier_channels=2)
    W = synth.weights(N, K, seed=N + K + 8, outlier_frac=0.005)
    s_host, _ = signs_pair(M * N + K + 9, K)
    r = run_layer(X, W, G, fmt, s_host, flags=flags)
    ref = oracle.verify_linear(X.numpy(), W.numpy(), G, fmt, s_host)
    assert_close(r["Y"], ref)


@pytest.mark.parametrize("fmt,M,K,N,G", GEMM_CASES)
def test_gemm_exact_order_is_bit_exact(fmt, M, K, N, G):
    # HQ_LAUNCH_EXACT_ORDER: every output summed over its groups in ascending
    # order by one thread block -> the oracle's sequential fp32 sum, bit for bit
    X = synth.activations(M, K, seed=M + K, outlier_channels=2)
    W = synth.weights(N, K, seed=N + K + 1, outlier_frac=0.005)
    s_host, _ = signs_pair(M * N + K, K)
    r = run_layer(X, W, G, fmt, s_host, check=True, flags=hq.HQ_LAUNCH_EXACT_ORDER | hq.HQ_LAUNCH_PDL)
    ref = oracle.verify_linear(X.numpy(), W.numpy(), G, fmt, s_host)
    assert np.array_equal(r["P"], ref["P"])
    assert np.array_equal(r["Y"].view(np.uint32), ref["Y"].view(np.uint32))


Q8_CASES = [("w4", 16, 4096, 384, 64), ("w4", 1, 256, 256, 32), ("w4", 40, 2048, 1000, 128), ("w4", 100, 512, 256, 64),
            ("w8", 16, 1024, 512, 128), ("w4", 32, 1024, 1024, 16), ("w4", 7, 4096, 256, 256)]


@pytest.mark.parametrize("flags", [hq.HQ_LAUNCH_EXACT_ORDER, hq.HQ_LAUNCH_DEFAULT])
@pytest.mark.parametrize("fmt,M,K,N,G", Q8_CASES)
def test_gemm_on_int8_codes(fmt, M, K, N, G, flags):
    # the boundary's int8 form: the oracle's own codes qx and scales sx go in
    # (hq_verify_gemm_q8 converts them inside its workspace); the outputs are
    # the oracle's (bit for bit in exact-order mode), the partials exact
    X = synth.activations(M, K, seed=M + K + 21, outlier_channels=2)
    W = synth.weights(N, K, seed=N + K + 22, outlier_frac=0.005)
    s_host, _ = signs_pair(M * N + K + 23, K)
    ref = oracle.verify_linear(X.numpy(), W.numpy(), G, fmt, s_host)
    layer = hq.pack_layer(W.to(DEV), G, fmt, s_host)
    ws = torch.zeros(hq.hq_workspace_q8_bytes(layer.desc, M), dtype=torch.uint8, device=DEV)
    assert ws.numel() > hq.hq_workspace_bytes(layer.desc, M) + hq.hq_act_operand_bytes(layer.desc, M) - 256
    qx = torch.from_numpy(ref["qx"]).to(DEV)
    sx = torch.from_numpy(ref["sx"]).to(DEV)
    Y = Guarded((M, N), torch.float32, DEV, fill=float("nan"))
    P = Guarded((M, N, K // G), torch.int32, DEV)
    hq.hq_verify_gemm_q8(layer.desc, layer.blob, qx, sx, None, M, Y.t, P.t, ws, flags | hq.HQ_LAUNCH_PDL)
    assert hq.hq_workspace_status(ws) == hq.HQ_OK
    torch.cuda.synchronize()
    Y.check("Y")
    P.check("partials")
    assert np.array_equal(P.t.cpu().numpy(), ref["P"])
    y = Y.t.cpu().numpy()
    if flags & hq.HQ_LAUNCH_EXACT_ORDER:
        assert np.array_equal(y.view(np.uint32), ref["Y"].view(np.uint32))
    else:
        assert_close(y, ref)
    # the same codes through the two-call path give the same outputs
    r = run_layer(X, None, G, fmt, s_host, flags=hq.HQ_LAUNCH_EXACT_ORDER, layer=layer)
    if flags & hq.HQ_LAUNCH_EXACT_ORDER:
        assert np.array_equal(r["Y"].view(np.uint32), y.view(np.uint32))


def test_gemm_wait_timeout_selftest_reports_error_and_recovers():
    # a GEMM whose waits between thread blocks ask for one arrival too many:
    # each runs out after 1 ms, the call reports HQ_ERR_TIMEOUT, no hang
    M, K, N, G = 16, 4096, 1024, 64  # 256 tiles over at most 152 blocks: split outputs
    X = synth.activations(M, K, seed=41, outlier_channels=2)
    W = synth.weights(N, K, seed=42)
    s_host, s_dev = signs_pair(43, K)
    layer = hq.pack_layer(W.to(DEV), G, "w4", s_host)
    _, _, qop, sx = hq.act_buffers(layer.desc, M, DEV, int8_codes=False)
    hq.hq_rotate_quant_act(layer.desc, X.to(DEV), M, layer.signs, None, None, qop, sx)
    ws = hq.workspace(layer.desc, M, DEV)
    Y = torch.empty((M, N), dtype=torch.float32, device=DEV)
    hq.hq_selftest_gemm_wait_timeout(layer.desc, layer.blob, qop, sx, M, Y, ws, 1_000_000)
    assert hq.hq_workspace_status(ws) == hq.HQ_ERR_TIMEOUT
    # the context is still usable and a clean workspace gives the right outputs
    ws.zero_()
    hq.hq_verify_gemm(layer.desc, layer.blob, qop, sx, M, Y, None, ws, hq.HQ_LAUNCH_EXACT_ORDER)
    assert hq.hq_workspace_status(ws) == hq.HQ_OK
    ref = oracle.verify_linear(X.numpy(), W.numpy(), G, "w4", s_host)
    assert np.array_equal(Y.cpu().numpy().view(np.uint32), ref["Y"].view(np.uint32))


def test_gemm_unsplit_blocks_default_mode_rounds_once_per_group():
    # K = 128: every 128-channel block is one tile, handled by one thread
    # block from its first to its last group.  The exact-order mode repeats the
    # oracle's separately rounded multiply and add bit for bit; the default
    # and deterministic modes fold each group with one fused multiply-add (one
    # rounding instead of two), so they meet the elementwise tolerance on every
    # output without being bit-identical.
    M, K, N, G = 16, 128, 1024, 32
    X = synth.activations(M, K, seed=1, outlier_channels=2)
    W = synth.weights(N, K, seed=2)
    s_host, _ = signs_pair(5, K)
    for fmt in ("w4", "w8"):
        ref = oracle.verify_linear(X.numpy(), W.numpy(), G, fmt, s_host)
        r = run_layer(X, W, G, fmt, s_host, flags=hq.HQ_LAUNCH_EXACT_ORDER)
        assert np.array_equal(r["Y"].view(np.uint32), ref["Y"].view(np.uint32))
        for flags in (hq.HQ_LAUNCH_DEFAULT, hq.HQ_LAUNCH_DETERMINISTIC):
            r = run_layer(X, W, G, fmt, s_host, flags=flags, layer=r["layer"])
            assert strict_fraction(r["Y"], ref) == 1.0
            assert_close(r["Y"], ref)


def test_gemm_deterministic_flag_repeats_bit_for_bit():
    # every n-block of this layer is split between thread blocks
    M, K, N, G = 16, 4096, 1024, 64
    X = synth.activations(M, K, seed=11, outlier_channels=2)
    W = synth.weights(N, K, seed=12)
    s_host, _ = signs_pair(13, K)
    det = hq.HQ_LAUNCH_DETERMINISTIC
    r0 = run_layer(X, W, G, "w4", s_host, flags=det)
    r1 = run_layer(X, W, G, "w4", s_host, flags=det | hq.HQ_LAUNCH_PDL, layer=r0["layer"])
    r2 = run_layer(X, W, G, "w4", s_host, flags=det | hq.HQ_LAUNCH_PDL, layer=r0["layer"])
    assert np.array_equal(r0["Y"].view(np.uint32), r1["Y"].view(np.uint32))
    assert np.array_equal(r1["Y"].view(np.uint32), r2["Y"].view(np.uint32))
    # the accumulating mode, repeated on the same layer, stays within the
    # oracle's tolerance every time
    ref = oracle.verify_linear(X.numpy(), W.numpy(), G, "w4", s_host)
    assert_close(r0["Y"], ref)
    for _ in range(3):
        r = run_layer(X, W, G, "w4", s_host, flags=hq.HQ_LAUNCH_PDL, layer=r0["layer"])
        assert_close(r["Y"], ref)


def test_shared_workspace_across_layers_and_batches():
    # one workspace, sized for the widest layer, serves layers of different
    # width, depth and batch in a PDL chain; every output equals the one
    # computed with a fresh workspace, bit for bit
    shapes = [(2048, 3072, 16), (2048, 2048, 16), (2048, 12288, 16), (6144, 2048, 16), (2048, 12288, 5),
              (2048, 640, 40), (2048, 12288, 16)]
    layers, inputs = [], []
    for i, (K, N, M) in enumerate(shapes):
        s_host, _ = signs_pair(100 + i, K)
        W = synth.weights(N, K, seed=200 + i)
        layers.append(hq.pack_layer(W.to(DEV), 64, "w4", s_host))
        inputs.append(synth.activations(M, K, seed=300 + i, outlier_channels=2).to(DEV))
    need = max(hq.hq_workspace_bytes(l.desc, x.shape[0]) for l, x in zip(layers, inputs))
    ws = torch.zeros(need, dtype=torch.uint8, device=DEV)
    det = hq.HQ_LAUNCH_DETERMINISTIC
    shared = [hq.verify_linear(l, x, ws, flags=hq.HQ_LAUNCH_PDL | det) for l, x in zip(layers, inputs)]
    # the accumulating mode in the same chain, alternating with the other mode
    accum = []
    for l, x in zip(layers, inputs):
        accum.append(hq.verify_linear(l, x, ws, flags=hq.HQ_LAUNCH_PDL))
        hq.verify_linear(l, x, ws, flags=hq.HQ_LAUNCH_PDL | det)
    torch.cuda.synchronize()
    assert hq.hq_workspace_status(ws) == hq.HQ_OK
    assert not ws[:16].any() and not ws[COUNTER_OFFSET:].any()
    for l, x, y, ya in zip(layers, inputs, shared, accum):
        fresh = hq.verify_linear(l, x, hq.workspace(l.desc, x.shape[0], DEV), flags=det)
        assert torch.equal(y.view(torch.int32), fresh.view(torch.int32))
        # same outputs up to the order of the fp32 adds of split outputs:
        # within 1e-5 of the largest output of the row
        d = (ya.double() - y.double()).abs()
        assert not torch.isnan(ya).any()
        assert (d <= ATOL + RTOL * y.double().abs().amax(dim=1, keepdim=True)).all()


def test_gemm_extreme_codes_int32_headroom():
    # activations whose rotated rows are +-a (all codes +-127) and weights whose
    # rotated groups are constant (all codes 15 with zero point 0 / all 127)
    M, K, N = 4, 512, 128
    s_host, _ = signs_pair(21, K)
    Xr = np.stack([np.full(K, (m + 1) * (1.0 if m % 2 == 0 else -1.0)) for m in range(M)]).astype(np.float32)
    X = torch.from_numpy(oracle.rotate_inverse(Xr, s_host))
    Wr = np.ones((N, K), dtype=np.float32) * 0.5
    Wr[1::2] *= -1.0
    W = torch.from_numpy(oracle.rotate_inverse(Wr, s_host))
    for fmt, G in (("w4", 256), ("w8", 256), ("w4", 64)):
        r = run_layer(X, W, G, fmt, s_host, check=True)
        ref = oracle.verify_linear(X.numpy(), W.numpy(), G, fmt, s_host)
        assert np.array_equal(r["P"], ref["P"])
        assert np.abs(ref["P"]).max() > 0.9 * 127 * (15 if fmt == "w4" else 127) * G
        assert_close(r["Y"], ref)


def test_gemm_zero_weights_and_zero_rows():
    M, K, N, G = 8, 512, 256, 64
    X = synth.activations(M, K, seed=31)
    X[2] = 0.0
    W = synth.weights(N, K, seed=32)
    W[:, :128] = 0.0
    W[7] = 0.0
    s_host, _ = signs_pair(33, K)
    for fmt in ("w4", "w8"):
        r = run_layer(X, W, G, fmt, s_host, check=True)
        ref = oracle.verify_linear(X.numpy(), W.numpy(), G, fmt, s_host)
        assert np.array_equal(r["P"], ref["P"])
        assert_close(r["Y"], ref)
        assert not r["Y"][2].any() and not r["Y"][:, 7].any()


def test_wait_timeout_selftest_reports_error_and_recovers():
    ws = torch.zeros(64, dtype=torch.uint8, device=DEV)
    hq.hq_selftest_wait_timeout(ws, 1_000_000)
    assert hq.hq_workspace_status(ws) == hq.HQ_ERR_TIMEOUT
    assert hq.hq_workspace_status(ws) == hq.HQ_OK  # the word was cleared
    # the context is still usable
    assert torch.ones(4, device=DEV).sum().item() == 4.0


# ------------------------------------------------ full-size workloads ---
def sampled_channels(N, count, seed):
    g = np.random.default_rng(seed)
    idx = set(g.choice(N, size=min(count, N), replace=False).tolist())
    idx.update([0, N - 1, min(127, N - 1), min(128, N - 1), N // 2])
    return np.array(sorted(idx))


def check_full_layer(K, N, G, fmt, M, seed, wcfg, xcfg, count=384, layer=None, W=None):
    """Full-size layer on the GPU; the oracle recomputes `count` sampled channels."""
    s_host, _ = signs_pair(seed, K)
    if W is None:
        W = synth.weights(N, K, seed=seed, device=DEV, **wcfg)
    X = synth.activations(M, K, seed=seed + 1, **xcfg)
    if layer is None:
        layer = hq.pack_layer(W, G, fmt, s_host)
    ws = hq.workspace(layer.desc, M, DEV)
    Y = hq.verify_linear(layer, X.to(DEV), ws, flags=hq.HQ_LAUNCH_PDL)
    assert hq.hq_workspace_status(ws) == hq.HQ_OK
    idx = sampled_channels(N, count, seed)
    Ws = W[torch.from_numpy(idx).to(DEV)].cpu().numpy()
    ref = oracle.verify_linear(X.numpy(), Ws, G, fmt, s_host)
    assert_close(Y.cpu().numpy()[:, idx], ref)
    return layer


@pytest.mark.parametrize("M", [1, 16])
def test_workload_tiny_256(M):
    c = synth.CONFIGS["tiny_256"]
    check_full_layer(c["K"], c["N"], c["G"], c["fmt"], M, c["seed"], c["w"], c["x"], count=256)


def test_workload_attn_4096():
    c = synth.CONFIGS["attn_4096"]
    check_full_layer(c["K"], c["N"], c["G"], c["fmt"], 16, c["seed"], c["w"], c["x"], count=4096)


def test_workload_gateup_w8():
    c = synth.CONFIGS["gateup_w8"]
    W = synth.weights(c["N"], c["K"], seed=c["seed"], device=DEV, **c["w"])
    layer = None
    for M in c["Ms"]:
        layer = check_full_layer(c["K"], c["N"], c["G"], c["fmt"], M, c["seed"], c["w"], c["x"], layer=layer, W=W)


@pytest.mark.parametrize("name", ["sweep_8192_w8", "sweep_8192_w4"])
def test_workload_sweep_8192(name):
    c = synth.CONFIGS[name]
    W = synth.weights(c["N"], c["K"], seed=c["seed"], device=DEV, **c["w"])
    layer = None
    for M in c["Ms"]:
        layer = check_full_layer(c["K"], c["N"], c["G"], c["fmt"], M, c["seed"], c["w"], c["x"], count=192,
                                 layer=layer, W=W)


def test_workload_decoder_9b_each_shape():
    cfg = synth.DECODER_9B
    shapes = {}
    for name, K, N in synth.decoder_linears(cfg):
        shapes.setdefault((K, N), name)
    assert len(shapes) == 5  # q and o, k and v, gate_up, down, lm_head
    for i, ((K, N), name) in enumerate(sorted(shapes.items())):
        check_full_layer(K, N, cfg["G"], cfg["fmt"], cfg["M"], synth.layer_seed(cfg["seed"], i), cfg["w"], cfg["x"],
                         count=256)
        torch.cuda.empty_cache()


# ----------------------------------------------------- tree acceptance ---
def random_tree(rng, M, branchy):
    if branchy:
        return np.array([-1] + [int(rng.integers(0, i)) for i in range(1, M)], dtype=np.int32)
    return np.arange(-1, M - 1, dtype=np.int32)  # a chain


def gpu_accept(L, parent, tokens, flags=0):
    greedy, path, out = hq.tree_accept(torch.from_numpy(L).to(DEV), torch.from_numpy(parent).to(DEV),
                                       torch.from_numpy(tokens).to(DEV), flags=flags)
    torch.cuda.synchronize()
    return greedy.cpu().numpy(), path.cpu().numpy(), int(out[0].item()), int(out[1].item())


@pytest.mark.parametrize("M,V,branchy", [(1, 1, False), (5, 7, False), (16, 151552, True), (16, 151552, False),
                                         (128, 8193, True), (33, 32003, True), (16, 8192, False)])
def test_tree_accept_matches_oracle(M, V, branchy):
    rng = np.random.default_rng(M * 1000 + V)
    # integer-valued logits: many ties, so the lowest-index rule is exercised
    L = rng.integers(-50, 50, size=(M, V)).astype(np.float32)
    L[:, int(rng.integers(0, V))] = 60.0
    if V > 10:
        L[0, 3] = np.nan if M > 1 else L[0, 3]
        L[min(1, M - 1), 5] = np.inf
        L[M - 1] = -0.0
        L[M - 1, V // 2] = 0.0
    parent = random_tree(rng, M, branchy)
    g_ref = oracle.argmax_rows(L)
    # drafts agree with the main model with probability 3/4
    tokens = np.where(rng.random(M) < 0.75, g_ref[np.maximum(parent, 0)], rng.integers(0, V, size=M)).astype(np.int32)
    path_ref, n_ref, bonus_ref = oracle.tree_accept(g_ref, parent, tokens)
    g, path, n, bonus = gpu_accept(L, parent, tokens, flags=hq.HQ_LAUNCH_PDL)
    assert np.array_equal(g, g_ref)
    assert n == n_ref and bonus == bonus_ref
    assert np.array_equal(path[:n], path_ref) and (path[n:] == -1).all()


def test_tree_accept_page_example():
    # five drafted tokens, the main model agrees with the first four: the pass advances five
    V = 64
    L = np.zeros((6, V), dtype=np.float32)
    for i, tok in enumerate([21, 22, 23, 24, 25, 26]):
        L[i, tok] = 1.0
    parent = np.arange(-1, 5, dtype=np.int32)
    tokens = np.array([11, 21, 22, 23, 24, 40], dtype=np.int32)
    g, path, n, bonus = gpu_accept(L, parent, tokens)
    assert list(path[:n]) == [1, 2, 3, 4] and n + 1 == 5 and bonus == 25


def test_tree_accept_reports_bad_parent():
    L = np.zeros((3, 10), dtype=np.float32)
    g, path, n, bonus = gpu_accept(L, np.array([-1, 2, 0], dtype=np.int32), np.zeros(3, dtype=np.int32))
    assert n == -1 and bonus == -1

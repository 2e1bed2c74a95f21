#!/usr/bin/env python
"""Throughput of the verify-pass quantized linear layers on GB300.

One step = one verify pass of a 9B-class decoder over M = 16 draft-tree
tokens: for each of 32 layers the q, k, v, o, fused gate+up and down
projections, then the LM head and the acceptance of the 16-node draft tree
from its logits -- every activation input runs the rotation +
int8 quantization kernel once and every linear the W4A8 GEMM kernel of
libhq.so (4-bit asymmetric weights, group 64).  q, k and v read the same
input; by default their weights are packed as one [6144][4096] matrix and
run as one GEMM (the same arithmetic, fewer launches; --no-fuse-qkv runs
three).  The pass streams 3.875 GB of packed weights,
far more than the 129 MB L2, so every pass reads its weights from HBM.

Reported (one JSON line on rank 0):
  value        weight GB/s of the whole pass (packed weight bytes / time)
  e2e          the same through host buffers: per step the activations are
               copied host->device and the logits device->host
  roofline     the GEMM kernel's weight bytes / its own time, vs measured HBM
  cpu_baseline the CPU oracle on a bounded sample (a 4096x4096 layer)
With torchrun (N > 1) every rank runs its own pass (independent verify
batches, weak scaling, no collective on the data path).
`--impl reference` times the CPU oracle instead (the slow reference arm).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "W4A8 verify-GEMM weight GB/s (% of HBM peak) and passes/s at M=16 rows"
WORKLOAD = "decoder_9b_verify_pass"
TAUS = (1.0, 8.39, 16.0)  # tokens per pass: plain decoding, the pages' measured 8.39, the 16-token tree budget
FALLBACK_HBM_GBS = 6800.0


def parse_args():
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=400)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=("gb300", "reference"), default="gb300")
    p.add_argument("--no-fuse-qkv", action="store_true",
                   help="run q, k and v as three GEMMs instead of one over their concatenated [6144][4096] weights")
    p.add_argument("--no-pdl", action="store_true", help="launch without programmatic dependent launch")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-attention", action="store_true", help="skip the tree-masked attention measurement")
    p.add_argument("--attn-context", type=int, default=8192, help="committed positions of the attention measurement")
    p.add_argument("--no-sweep", action="store_true",
                   help="skip the K=N=8192 arithmetic-intensity sweep and the single-layer timings")
    p.add_argument("--only-attention", action="store_true",
                   help="run only the tree-attention and DeltaNet measurements (for profiling their kernels)")
    p.add_argument("--summarize-ncu", metavar="CSV",
                   help="summarize an ncu --csv log of this program into profiles/ and exit")
    p.add_argument("--ncu-command", default="", help="the ncu command line that produced CSV (recorded)")
    p.add_argument("--ncu-name", default="decoder_9b", help="workload name used in the summary file names")
    p.add_argument("--one-gemm", metavar="K,N,G,FMT,M",
                   help="time one GEMM layer of this shape alone (K,N,G,w4|w8,M), print its JSON line and exit")
    return p.parse_args()


# ----------------------------------------------------------------- ranks ---
class Ranks:
    def __init__(self):
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.dist = None
        if self.world > 1:
            import torch.distributed as dist
            import torch
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            dist.init_process_group(backend=backend)
            self.dist = dist

    def barrier(self):
        if self.dist:
            self.dist.barrier()

    def max(self, x: float) -> float:
        if not self.dist:
            return x
        import torch
        dev = "cuda" if torch.cuda.is_available() else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.dist.all_reduce(t, op=self.dist.ReduceOp.MAX)
        return float(t.item())

    def sum(self, x: float) -> float:
        if not self.dist:
            return x
        import torch
        dev = "cuda" if torch.cuda.is_available() else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.dist.all_reduce(t, op=self.dist.ReduceOp.SUM)
        return float(t.item())

    def close(self):
        if self.dist:
            self.dist.destroy_process_group()


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# ---------------------------------------------------------------- clocks ---
class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int, period_ms: int = 20):
        self.samples = []
        self.proc = None
        self.t0 = self.t1 = None
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(device_index), "-lms", str(period_ms)],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except OSError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def mark_start(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def stop(self):
        if self.proc:
            time.sleep(0.05)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        if not self.proc or not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        win = [s for t, s in self.samples if self.t0 is not None and self.t0 <= t <= (self.t1 or t)]
        if not win:  # a very short timed region: take the samples nearest to it
            win = [s for _, s in self.samples][-3:]
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for s in win:
            f = [x.strip() for x in s.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for name, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# -------------------------------------------------------------- CPU side ---
def cpu_oracle_sample(target_s: float = 10.0):
    """Time the oracle (OpenMP build, as it stands) on one 4096x4096 W4 G64 layer at M = 16:
    activation rotation + quantization and the integer GEMM with its epilogue."""
    import oracle
    from quantized_speculative_verify_gb300 import synth
    K = N = 4096
    G, M, seed = 64, 16, 7
    W = synth.weights(N, K, seed=seed).numpy()
    X = synth.activations(M, K, seed=seed + 1, outlier_channels=2).numpy()
    signs = oracle.make_signs(seed, K)
    codes, scales, zeros = oracle.quant_w4(W, G, signs, openmp=True)
    wbytes = N * K * (0.5 + 4.5 / G)

    def one():
        qx, sx, _ = oracle.quant_act(X, G, signs)
        oracle.verify_gemm(qx, sx, codes, scales, zeros, G, openmp=True)

    t = time.perf_counter()
    one()
    first = time.perf_counter() - t
    reps = max(1, int(target_s / max(first, 1e-3)))
    t = time.perf_counter()
    for _ in range(reps):
        one()
    dt = time.perf_counter() - t
    # the single-thread build on the same layer, a few repetitions (bounded)
    t = time.perf_counter()
    qx, sx, _ = oracle.quant_act(X, G, signs)
    oracle.verify_gemm(qx, sx, codes, scales, zeros, G, openmp=False)
    dt1 = time.perf_counter() - t
    return dict(value=wbytes * reps / dt / 1e9, unit="GB/s", cores=oracle.num_threads(True), kind="oracle",
                sample=f"one 4096x4096 W4 G64 layer (q-projection shape of the pass), M=16, act-quant + GEMM, "
                       f"{reps} repetitions in {dt:.1f} s",
                single_thread={"value": wbytes / dt1 / 1e9, "unit": "GB/s", "cores": 1,
                               "sample": f"the same layer once, {dt1:.1f} s"}), dt / reps, wbytes


def run_reference(args, ranks: Ranks):
    """The reference arm: the CPU oracle, one bounded sample per step."""
    if ranks.rank != 0:
        return 0
    import oracle
    oracle.build()
    from quantized_speculative_verify_gb300 import synth
    K = N = 4096
    G, M, seed = 64, 16, 7
    W = synth.weights(N, K, seed=seed).numpy()
    X = synth.activations(M, K, seed=seed + 1, outlier_channels=2).numpy()
    signs = oracle.make_signs(seed, K)
    codes, scales, zeros = oracle.quant_w4(W, G, signs, openmp=True)
    wbytes = N * K * (0.5 + 4.5 / G)

    def step():
        qx, sx, _ = oracle.quant_act(X, G, signs)
        oracle.verify_gemm(qx, sx, codes, scales, zeros, G, openmp=True)

    for _ in range(args.warmup):
        step()
    t = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t
    value = wbytes * args.steps / dt / 1e9
    sample = "one 4096x4096 W4 G64 layer (q-projection shape of the pass) per step, M=16, act-quant + GEMM"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int8",
            "data": "synthetic", "config": {"workload": WORKLOAD, "M": 16, "format": "w4_asym", "group": 64,
                                            "sample": sample},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": oracle.num_threads(True), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# -------------------------------------------------------------- GPU side ---
def gemm_source_parts(csrc: str) -> list:
    """The sources that determine the GEMM's code and launch: its kernel
    header and instance files, the device helpers (everything before the
    launcher declarations) and the GEMM launcher of the API file."""
    def read(f):
        with open(os.path.join(csrc, f)) as fh:
            return fh.read()
    parts = [read("k_gemm.cuh"), read("k_gemm_w4.cu"), read("k_gemm_w8.cu"), read("gemm_common.cuh"),
             read("k_gemm_rs.cuh"), read("k_gemm_rs.cu"), read("k_gemm_rs_w8.cu")]
    internal = read("hq_internal.cuh")
    parts.append(internal.split("// Launchers (defined in the kernel translation units).")[0])
    api = read("hq_api.cu")
    i = api.index("cudaError_t launch_verify_gemm(")
    parts.append(api[i:api.index("\n}\n", i)])
    return parts


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for part in gemm_source_parts(os.path.join(ROOT, "quantized_speculative_verify_gb300", "csrc")):
        h.update(part.encode())
    return h.hexdigest()[:16]


def gemm_kernel_name(fmt: str, M: int) -> str:
    """The GEMM kernel the library runs for a format and row count: the
    register-resident kernel up to 32 rows, else the tensor-memory kernel."""
    return "k_verify_gemm_rs" if M <= 32 else "k_verify_gemm"


def gemm_traffic_record():
    """ncu DRAM bytes of the GEMM for this workload, if taken on the current kernel source."""
    path = os.path.join(ROOT, "profiles", "k_verify_gemm_decoder_9b_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    if d.get("kernel_source_hash") != kernel_source_hash():
        return None
    return d


class VerifyPass:
    """All packed weights, inputs and outputs of one decoder verify pass, resident on the device.

    Each activation input (a layer's attention input, read by q, k and v; the
    o input; the MLP input, read by gate and up; the down input; the LM head
    input) has its own sign vector, X, and quantized buffers; the layers that
    read an input are packed with that input's signs.  Layers that read the
    same input run as one GEMM over their weight matrices packed into one blob
    (hq_pack_weights_at): gate and up always, q, k and v unless
    --no-fuse-qkv."""

    def __init__(self, torch, hq, synth, device, fuse_qkv: bool, pdl: bool):
        cfg = synth.DECODER_9B
        self.torch, self.hq, self.synth = torch, hq, synth
        self.cfg = cfg
        self.M, self.G, self.fmt = cfg["M"], cfg["G"], cfg["fmt"]
        self.flags = hq.HQ_LAUNCH_PDL if pdl else hq.HQ_LAUNCH_DEFAULT
        self.gemms = synth.decoder_gemms(cfg, fuse_qkv=fuse_qkv)
        self.linears = [(name, K, sum(n for _, n, _ in parts)) for name, K, parts in self.gemms]
        self.layers, self.fused, self.ys, self.inputs, self.plan = [], [], [], [], []
        seed = cfg["seed"]
        ws_need = 0
        s_host = None
        for li, (name, K, parts) in enumerate(self.gemms):
            if not name.endswith((".k", ".v")):  # a new activation input
                s_host = hq.hq_make_signs(synth.layer_seed(seed, 500 + li), K)
                X = synth.activations(self.M, K, seed=synth.layer_seed(seed, 2000 + li), device=device, **cfg["x"])
                adesc = hq.make_desc(K, 128, self.G, self.fmt)  # the layers that read this input
                _, _, qop, sx = hq.act_buffers(adesc, self.M, device, int8_codes=False)
                self.inputs.append([name, K, X, qop, sx, None, s_host, adesc])
            Ws = [synth.weights(n, K, seed=synth.layer_seed(seed, wi), device=device, **cfg["w"])
                  for _, n, wi in parts]
            fused = hq.pack_fused(Ws, self.G, self.fmt, s_host)
            del Ws
            layer = fused.layer
            if self.inputs[-1][5] is None:
                self.inputs[-1][5] = layer.signs
            self.layers.append(layer)
            self.fused.append(fused)
            self.ys.append(torch.empty((self.M, layer.N), dtype=torch.float32, device=device))
            self.plan.append((len(self.inputs) - 1, li))
            ws_need = max(ws_need, hq.hq_workspace_bytes(layer.desc, self.M))
        self.ws = torch.zeros(ws_need, dtype=torch.uint8, device=device)
        # every activation input as a view into one device buffer, so that an
        # end-to-end step moves all of them from the host with one copy
        self.x_all = torch.empty(sum(inp[2].numel() for inp in self.inputs), dtype=torch.float32, device=device)
        off = 0
        for inp in self.inputs:
            n = inp[2].numel()
            view = self.x_all[off:off + n].view(inp[2].shape)
            view.copy_(inp[2])
            inp[2] = view
            off += n
        self.weight_bytes = sum(int(l.blob.numel()) for l in self.layers)
        self.algo_weight_bytes = sum(K * N * (0.5 + 4.5 / self.G) for _, K, N in self.linears)
        self.n_act = len(self.inputs)
        self.n_gemm = len(self.layers)
        # the draft tree verified by the pass: 16 nodes, the root and three
        # branches of depth 5 (parents listed first), drafted tokens seeded
        self.parent = torch.tensor([-1, 0, 1, 2, 3, 4, 0, 6, 7, 8, 9, 0, 11, 12, 13, 14], dtype=torch.int32,
                                   device=device)[: self.M]
        gen = torch.Generator(device="cpu").manual_seed(cfg["seed"] + 77)
        V = self.linears[-1][2]
        self.tokens = torch.randint(0, V, (self.M,), generator=gen, dtype=torch.int32).to(device)
        self.greedy = torch.empty(self.M, dtype=torch.int32, device=device)
        self.path = torch.empty(self.M, dtype=torch.int32, device=device)
        self.accept_out = torch.empty(2, dtype=torch.int32, device=device)
        self.accept_ws = torch.empty(hq.hq_tree_accept_workspace_bytes(self.M, V), dtype=torch.uint8, device=device)
        self.n_accept_kernels = 2

    def part_weights(self, li: int, device):
        """The fp32 weight matrices of GEMM li's parts, regenerated from their seeds (for checking)."""
        name, K, parts = self.gemms[li]
        return [self.synth.weights(n, K, seed=self.synth.layer_seed(self.cfg["seed"], wi), device=device,
                                   **self.cfg["w"]) for _, n, wi in parts]

    def launch(self, act=True, gemm=True):
        hq = self.hq
        done = set()
        for ii, li in self.plan:
            name, K, X, qop, sx, signs, _, adesc = self.inputs[ii]
            if act and ii not in done:
                hq.hq_rotate_quant_act(adesc, X, self.M, signs, None, None, qop, sx, self.flags)
                done.add(ii)
            if gemm:
                layer = self.layers[li]
                hq.hq_verify_gemm(layer.desc, layer.blob, qop, sx, self.M, self.ys[li], None, self.ws, self.flags)
        if act and gemm:
            # accept the draft tree from the LM head's logits
            V = self.linears[-1][2]
            hq.hq_tree_accept(self.ys[-1], self.M, V, self.parent, self.tokens, self.greedy, self.path,
                              self.accept_out[0:1], self.accept_out[1:2], self.accept_ws, self.flags)

    def point_inputs_at(self, buf):
        """Re-point every activation input at the same offsets of `buf` (a
        buffer shaped like x_all); returns the buffer previously used."""
        prev, off = self.x_all, 0
        for inp in self.inputs:
            n = inp[2].numel()
            inp[2] = buf[off:off + n].view(inp[2].shape)
            off += n
        self.x_all = buf
        return prev

    def h2d_bytes(self):
        return self.x_all.numel() * 4


def run_gpu(args, ranks: Ranks):
    import torch
    from quantized_speculative_verify_gb300 import hq, synth

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (the product path has no CPU fallback)")
    torch.cuda.set_device(ranks.local)
    device = torch.device("cuda", ranks.local)
    hq.load()
    peak, peak_kind = measured_peaks()

    vp = VerifyPass(torch, hq, synth, device, fuse_qkv=not args.no_fuse_qkv, pdl=not args.no_pdl)
    torch.cuda.synchronize()

    stream = torch.cuda.Stream(device=device)
    torch.cuda.set_stream(stream)
    # correctness of the run itself: one eager pass, no device-side time-out
    vp.launch()
    if hq.hq_workspace_status(vp.ws) != hq.HQ_OK:
        raise SystemExit("device-side wait timed out")

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        vp.launch()
    gemm_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gemm_graph, stream=stream):
        vp.launch(act=False)

    # ---- the timed region: K whole passes (the clock sampler starts first,
    # so the warm-up passes also bring the clocks back up after its start-up)
    clocks = ClockSampler(ranks.local)
    time.sleep(0.3)
    for _ in range(max(args.warmup, 3)):
        graph.replay()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    ranks.barrier()
    clocks.mark_start()
    ev0.record(stream)
    for _ in range(args.steps):
        graph.replay()
    ev1.record(stream)
    ev1.synchronize()
    clocks.mark_end()
    torch.cuda.synchronize()
    ranks.barrier()
    clocks.stop()
    ms = ev0.elapsed_time(ev1)
    ms_max = ranks.max(ms)
    if hq.hq_workspace_status(vp.ws) != hq.HQ_OK:
        raise SystemExit("device-side wait timed out during the timed region")
    total_bytes = ranks.sum(vp.algo_weight_bytes * args.steps)
    value = total_bytes / (ms_max / 1e3) / 1e9
    passes_per_s = args.steps * ranks.world / (ms_max / 1e3)

    # ---- the dominant kernel alone: the same GEMM launches without the activation kernels
    for _ in range(max(args.warmup, 3)):
        gemm_graph.replay()
    reps = max(20, args.steps // 2)
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    g0.record(stream)
    for _ in range(reps):
        gemm_graph.replay()
    g1.record(stream)
    g1.synchronize()
    gemm_ms_per_pass = g0.elapsed_time(g1) / reps
    gemm_achieved = vp.algo_weight_bytes / (gemm_ms_per_pass / 1e3) / 1e9
    traffic = gemm_traffic_record()
    roofline = {"bound": "hbm", "achieved": gemm_achieved, "peak": peak, "unit": "GB/s",
                "frac": gemm_achieved / peak, "peak_kind": f"{peak_kind} (HBM copy bandwidth)",
                "traffic": None if traffic is None else traffic["dram_bytes_per_launch"],
                "kernel": gemm_kernel_name(vp.fmt, vp.M), "launches_per_pass": vp.n_gemm,
                "avg_launch_us": gemm_ms_per_pass * 1e3 / vp.n_gemm,
                "algorithmic_bytes_per_launch": vp.algo_weight_bytes / vp.n_gemm}

    # ---- end to end through host buffers
    e2e = None
    if not args.no_e2e:
        # Two input buffers, one captured pass per buffer: step k's inputs are
        # copied on a copy stream while step k-1 computes (each step still
        # copies all of its inputs from pinned host memory, inside the timed
        # region); the logits come back on the compute stream after the pass.
        host_all = torch.empty_like(vp.x_all, device="cpu").pin_memory()
        host_all.copy_(vp.x_all.cpu())
        bufs = [vp.x_all, torch.empty_like(vp.x_all)]
        graphs = [graph, torch.cuda.CUDAGraph()]
        # the second graph reads the second input buffer and writes the second logits buffer
        logits_dev = [vp.ys[-1], torch.empty_like(vp.ys[-1])]
        vp.point_inputs_at(bufs[1])
        vp.ys[-1] = logits_dev[1]
        with torch.cuda.graph(graphs[1], stream=stream):
            vp.launch()
        vp.point_inputs_at(bufs[0])
        vp.ys[-1] = logits_dev[0]
        logits_host = [torch.empty_like(logits_dev[0], device="cpu").pin_memory() for _ in range(2)]
        h2d_stream = torch.cuda.Stream(device=device)
        d2h_stream = torch.cuda.Stream(device=device)
        e_steps = max(4, args.steps // 4)
        done = [torch.cuda.Event(), torch.cuda.Event()]     # the pass that used buffer pair b is complete
        copied = [torch.cuda.Event(), torch.cuda.Event()]   # input buffer b holds the step's inputs
        read = [torch.cuda.Event(), torch.cuda.Event()]     # logits buffer b was read back
        for b in range(2):
            done[b].record(stream)
            read[b].record(stream)

        def e2e_step(k):
            # step k's inputs go in on one copy stream while step k-1 runs, and
            # its logits come back on another while step k+1 runs; the two
            # buffer pairs alternate between steps
            b = k % 2
            h2d_stream.wait_event(done[b])
            with torch.cuda.stream(h2d_stream):
                bufs[b].copy_(host_all, non_blocking=True)
            copied[b].record(h2d_stream)
            stream.wait_event(copied[b])
            stream.wait_event(read[b])       # step k-2's logits are out before they are overwritten
            graphs[b].replay()
            done[b].record(stream)
            d2h_stream.wait_event(done[b])
            with torch.cuda.stream(d2h_stream):
                logits_host[b].copy_(logits_dev[b], non_blocking=True)
            read[b].record(d2h_stream)

        for k in range(4):
            e2e_step(k)
        torch.cuda.synchronize()
        ranks.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        h2d_stream.wait_event(e0)
        for k in range(e_steps):
            e2e_step(k)
        for b in range(2):
            stream.wait_event(read[b])       # every step's logits are on the host
        e1.record(stream)
        e1.synchronize()
        e_ms = ranks.max(e0.elapsed_time(e1))
        e2e = {"value": ranks.sum(vp.algo_weight_bytes * e_steps) / (e_ms / 1e3) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": vp.h2d_bytes(), "d2h_bytes_per_step": logits_dev[0].numel() * 4,
               "ms_per_step": e_ms / e_steps, "steps": e_steps}

    sweep = None if args.no_sweep else measure_sweep(torch, hq, synth, device, stream, args, peak)
    layers = None if args.no_sweep else measure_layers(torch, hq, synth, device, stream, peak)
    attn = delta = None
    if not args.no_attention:
        attn = measure_tree_attention(torch, hq, device, stream, args, peak)
        delta = measure_delta_tree(torch, hq, device, stream, args, peak)

    cpu = None
    if not args.no_cpu_baseline and ranks.rank == 0:
        cpu, _, _ = cpu_oracle_sample()

    if ranks.rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ranks.world, "steps": args.steps,
            "warmup": max(args.warmup, 3), "ms_per_step": ms_max / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "int8", "data": "synthetic",
            "config": {"workload": WORKLOAD, "M": vp.M, "format": "w4_asym", "group": vp.G, "layers": 32,
                       "linears_per_pass": vp.n_gemm, "activation_inputs_per_pass": vp.n_act,
                       "tree_accept": "16-node draft tree accepted from the LM head's logits each pass",
                       "qkv_fused": not args.no_fuse_qkv, "pdl": not args.no_pdl,
                       "weight_bytes_per_pass": vp.weight_bytes,
                       "l2": "inputs larger than L2: 3.875 GB of packed weights streamed per pass, L2 129 MB",
                       "parallelism": f"replicas x{ranks.world} (independent verify batches)"},
            "passes_per_s": passes_per_s,
            "pct_of_hbm_peak": 100.0 * value / (peak * ranks.world),
            "tokens_per_s_ceiling": {f"tau={t:g}": passes_per_s * t for t in TAUS},
            "roofline": roofline,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "clocks": clocks.summary(),
            "gpu_launches": args.steps * (vp.n_act + vp.n_gemm + vp.n_accept_kernels),
            "tree_attention": attn,
            "delta_tree": delta,
            "sweep": sweep,
            "layers": layers,
        }
        print(json.dumps(line))
    return 0


def measure_sweep(torch, hq, synth, device, stream, args, peak):
    """The arithmetic-intensity sweep: one K=N=8192 layer, W8 G128 and W4 G64,
    M in {1, ..., 128} rows (activation quantization + GEMM per call, the
    layer's hot path).  Four copies of the packed layer (153 / 276 MB, larger
    than L2) are cycled so every call streams its weights from HBM.  Per M:
    microseconds per call, weight GB/s, integer tera-ops/s (2*M*N*K) and the
    verify cost ratio t(M) / t(1).  Every M runs as one GEMM launch (the
    rows are the tensor-core MMA's N: 16, 32, 64 or 128)."""
    out = {}
    K = N = 8192
    copies = 4
    for name in ("sweep_8192_w8", "sweep_8192_w4"):
        c = synth.CONFIGS[name]
        signs = hq.hq_make_signs(c["seed"], K)
        W = synth.weights(N, K, seed=c["seed"], device=device)
        first = hq.pack_layer(W, c["G"], c["fmt"], signs)
        layers = [first] + [hq.PackedLayer(first.desc, first.blob.clone(), first.signs) for _ in range(copies - 1)]
        del W
        rows = []
        t1 = None
        for M in c["Ms"]:
            X = synth.activations(M, K, seed=c["seed"] + M, device=device)
            bufs = hq.act_buffers(layers[0].desc, M, device, int8_codes=False)
            Y = torch.empty((M, N), dtype=torch.float32, device=device)
            ws = hq.workspace(layers[0].desc, M, device)
            for i in range(copies * 2):
                hq.verify_linear(layers[i % copies], X, ws, bufs=bufs, Y=Y, stream=stream)
            reps = copies * 5
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            e0.record(stream)
            for i in range(reps):
                hq.verify_linear(layers[i % copies], X, ws, bufs=bufs, Y=Y, stream=stream)
            e1.record(stream)
            e1.synchronize()
            if hq.hq_workspace_status(ws) != hq.HQ_OK:
                raise SystemExit("device-side wait timed out in the sweep")
            us = e0.elapsed_time(e1) * 1e3 / reps
            t1 = us if t1 is None else t1
            wbytes = layers[0].blob.numel()
            rows.append({"M": M, "us": us, "weight_gbs": wbytes / us / 1e3, "frac_hbm": wbytes / us / 1e3 / peak,
                         "int_tops": 2.0 * M * N * K / us / 1e6, "cost_ratio": us / t1})
        out[name] = {"fmt": c["fmt"], "group": c["G"], "K": K, "N": N, "weight_bytes": layers[0].blob.numel(),
                     "copies": copies, "rows": rows}
        del layers
        torch.cuda.empty_cache()
    return out


def measure_layers(torch, hq, synth, device, stream, peak):
    """The single-layer workloads (tiny 256x256 W4 G32, the 4096x4096 W4 G64
    projection, the W8 G128 gate+up 4096 -> 2x12288), per M: `warm_us` over
    cycled copies of the packed layer (repeated calls, weights from HBM where
    the copies exceed L2), and `cold_us`, the median of 5 single calls each
    after writing a 512 MB buffer (L2 flushed).  Each call is activation
    quantization + GEMM, the layer's hot path."""
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=device)
    out = {}
    for name in ("tiny_256", "attn_4096", "gateup_w8"):
        c = synth.CONFIGS[name]
        K, N = c["K"], c["N"]
        signs = hq.hq_make_signs(c["seed"], K)
        W = synth.weights(N, K, seed=c["seed"], device=device, **c["w"])
        first = hq.pack_layer(W, c["G"], c["fmt"], signs)
        del W
        wbytes = first.blob.numel()
        copies = max(1, min(8, -(-256 * 1024 * 1024 // wbytes)))
        packed = [first] + [hq.PackedLayer(first.desc, first.blob.clone(), first.signs) for _ in range(copies - 1)]
        rows = []
        for M in c["Ms"]:
            X = synth.activations(M, K, seed=c["seed"] + 1, device=device, **c["x"])
            bufs = hq.act_buffers(first.desc, M, device, int8_codes=False)
            Y = torch.empty((M, N), dtype=torch.float32, device=device)
            ws = hq.workspace(first.desc, M, device)
            for i in range(2 * copies):
                hq.verify_linear(packed[i % copies], X, ws, bufs=bufs, Y=Y, stream=stream)
            reps = max(20, 2 * copies)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            e0.record(stream)
            for i in range(reps):
                hq.verify_linear(packed[i % copies], X, ws, bufs=bufs, Y=Y, stream=stream)
            e1.record(stream)
            e1.synchronize()
            warm = e0.elapsed_time(e1) * 1e3 / reps
            cold = []
            for _ in range(5):
                with torch.cuda.stream(stream):
                    flush.zero_()
                c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                c0.record(stream)
                hq.verify_linear(first, X, ws, bufs=bufs, Y=Y, stream=stream)
                c1.record(stream)
                c1.synchronize()
                cold.append(c0.elapsed_time(c1) * 1e3)
            if hq.hq_workspace_status(ws) != hq.HQ_OK:
                raise SystemExit("device-side wait timed out in the single-layer timings")
            cold_us = sorted(cold)[2]
            rows.append({"M": M, "warm_us": warm, "warm_weight_gbs": wbytes / warm / 1e3, "cold_us": cold_us,
                         "cold_weight_gbs": wbytes / cold_us / 1e3, "warm_frac_hbm": wbytes / warm / 1e3 / peak})
        out[name] = {"K": K, "N": N, "fmt": c["fmt"], "group": c["G"], "weight_bytes": wbytes, "copies": copies,
                     "rows": rows}
        del packed, first
        torch.cuda.empty_cache()
    del flush
    return out


def measure_tree_attention(torch, hq, device, stream, args, peak):
    """Tree-masked verify attention of the 9B-class decoder: its 8 attention
    layers (the other 24 are DeltaNet layers), 16 tree nodes, 32 query heads
    over 8 key/value heads of 128, fp16 caches of L committed positions each
    (8 x 33.6 MB at L = 8192: larger than L2, so each pass streams them from
    HBM).  One step = the 8 layers' attention calls, replayed from a CUDA graph
    with programmatic dependent launch.  Algorithmic bytes = the K and V rows
    read (committed + tree positions) plus q in and out."""
    layers, M, Hq, Hkv, D, L = 8, 16, 32, 8, hq.HQ_ATTN_HEAD_DIM, args.attn_context
    cap = L + M
    gen = torch.Generator(device=device)
    gen.manual_seed(1234)
    caches = [(torch.randn((Hkv, cap, D), generator=gen, device=device, dtype=torch.float16),
               torch.randn((Hkv, cap, D), generator=gen, device=device, dtype=torch.float16)) for _ in range(layers)]
    qs = [torch.randn((M, Hq, D), generator=gen, device=device, dtype=torch.float16) for _ in range(layers)]
    parent = torch.tensor([0, 0, 1, 2, 3, 0, 5, 6, 1, 8, 2, 10, 11, 0, 13, 14], dtype=torch.int32, device=device)
    outs = [torch.empty((M, Hq, D), dtype=torch.float32, device=device) for _ in range(layers)]
    ws = torch.zeros(hq.hq_tree_attention_workspace_bytes(Hkv), dtype=torch.uint8, device=device)
    scale = 1.0 / D ** 0.5

    def step():
        for i in range(layers):
            hq.hq_tree_attention(qs[i], caches[i][0], caches[i][1], cap, L, M, Hq, Hkv, D, parent, scale, outs[i],
                                 ws, hq.HQ_LAUNCH_PDL, stream)

    step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        step()
    for _ in range(max(args.warmup, 3)):
        g.replay()
    reps = max(20, args.steps // 4)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(reps):
        g.replay()
    e1.record(stream)
    e1.synchronize()
    ms = e0.elapsed_time(e1) / reps
    if hq.hq_workspace_status(ws) != hq.HQ_OK:
        raise SystemExit("device-side wait timed out in the attention measurement")
    kv_bytes = layers * 2 * Hkv * (L + M) * D * 2
    io_bytes = layers * (M * Hq * D * 2 + M * Hq * D * 4)
    gbs = (kv_bytes + io_bytes) / (ms / 1e3) / 1e9
    return {"workload": f"9B-class tree verify attention: {layers} layers, M={M} tree nodes, Hq={Hq}, Hkv={Hkv}, "
                        f"D={D}, L={L} committed positions, fp16 caches",
            "value": gbs, "unit": "GB/s", "us_per_layer": ms * 1e3 / layers, "ms_per_step": ms,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                         "algorithmic_bytes_per_layer": (kv_bytes + io_bytes) / layers},
            "kernels": ["k_tree_attn_split", "k_tree_attn_merge"], "launches_per_step": 2 * layers,
            "steps": reps}


def measure_delta_tree(torch, hq, device, stream, args, peak):
    """Rollback-free DeltaNet tree pass of the 9B-class decoder: its 24 Gated
    DeltaNet layers, 16 tree nodes, 32 heads with 128 x 128 fp32 states
    (2 MB per layer).  Three copies of every layer's state (144 MB, larger
    than L2) are cycled so each step reads its states from HBM, as inside a
    pass that streams 3.9 GB of weights.  One step = the 24 layers' tree
    passes from a CUDA graph with programmatic dependent launch.  Algorithmic
    bytes = the committed states read plus q, k, v, gates in and outputs out."""
    layers, copies, M, H, D = 24, 3, 16, 32, hq.HQ_DELTA_HEAD_DIM
    gen = torch.Generator(device=device)
    gen.manual_seed(4321)
    states = [torch.randn((H, D, D), generator=gen, device=device) * 0.05 for _ in range(layers * copies)]

    def unit(x):
        return x / x.norm(dim=-1, keepdim=True)
    qkv = [(torch.randn((M, H, D), generator=gen, device=device),
            unit(torch.randn((M, H, D), generator=gen, device=device)),
            torch.randn((M, H, D), generator=gen, device=device),
            torch.rand((M, H), generator=gen, device=device) * 0.4 + 0.6,
            torch.rand((M, H), generator=gen, device=device)) for _ in range(layers)]
    parent = torch.tensor([0, 0, 1, 2, 3, 0, 5, 6, 1, 8, 2, 10, 11, 0, 13, 14], dtype=torch.int32, device=device)
    outs = [torch.empty((M, H, D), dtype=torch.float32, device=device) for _ in range(layers)]
    graphs = []
    for c in range(copies):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for i in range(layers):
                q, k, v, al, be = qkv[i]
                hq.hq_delta_tree(states[c * layers + i], q, k, v, al, be, parent, M, H, D, outs[i],
                                 hq.HQ_LAUNCH_PDL, stream)
        graphs.append(g)
    for r in range(max(args.warmup, 3) * copies):
        graphs[r % copies].replay()
    reps = max(21, args.steps // 4) // copies * copies
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for r in range(reps):
        graphs[r % copies].replay()
    e1.record(stream)
    e1.synchronize()
    ms = e0.elapsed_time(e1) / reps
    state_bytes = layers * H * D * D * 4
    io_bytes = layers * (M * H * D * 4 * 4 + M * H * 4 * 2)
    gbs = (state_bytes + io_bytes) / (ms / 1e3) / 1e9
    return {"workload": f"9B-class DeltaNet tree pass: {layers} layers, M={M} tree nodes, H={H} heads, "
                        f"{D}x{D} fp32 states, {copies} copies cycled (inputs larger than L2)",
            "value": gbs, "unit": "GB/s", "us_per_layer": ms * 1e3 / layers, "ms_per_step": ms,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s", "frac": gbs / peak,
                         "algorithmic_bytes_per_layer": (state_bytes + io_bytes) / layers},
            "kernels": ["k_delta_tree"], "launches_per_step": layers, "steps": reps}


def summarize_ncu(args) -> int:
    """Per-kernel launches, time and share from an ncu --csv log; with DRAM
    byte metrics present, also the GEMM's traffic record read by the bench."""
    import collections
    import csv
    rows = list(csv.reader(open(args.summarize_ncu)))
    hi = next(i for i, r in enumerate(rows) if r and r[0] == "ID")
    hdr = rows[hi]
    ix = {h: i for i, h in enumerate(hdr)}
    scale = {"nsecond": 1e-3, "ns": 1e-3, "usecond": 1.0, "us": 1.0, "msecond": 1e3, "ms": 1e3,
             "byte": 1.0, "Kbyte": 1e3, "Mbyte": 1e6, "Gbyte": 1e9}
    per = collections.defaultdict(lambda: collections.defaultdict(float))
    launches = collections.defaultdict(set)
    for r in rows[hi + 1:]:
        if len(r) < len(hdr):
            continue
        name = r[ix["Kernel Name"]].replace("(anonymous namespace)::", "").replace("void ", "").split("(")[0]
        name = name.replace("unnamed>::", "")
        metric, unit = r[ix["Metric Name"]], r[ix["Metric Unit"]]
        val = float(r[ix["Metric Value"]].replace(",", "")) * scale.get(unit, 1.0)
        per[name][metric] += val
        launches[name].add(r[ix["ID"]])
    tot_us = sum(d.get("gpu__time_duration.sum", 0.0) for d in per.values())
    out = [f"# ncu launch list: {args.ncu_name}", "",
           f"Command: `{args.ncu_command}`" if args.ncu_command else "", "",
           "Per kernel over the captured launches (ncu serializes launches and runs them with cold caches, so",
           "compare the shares, not the absolute times, with the bench's CUDA-event timings).", "",
           "| kernel | launches | total time (us) | share | DRAM read (MB) | DRAM write (MB) |",
           "|---|---|---|---|---|---|"]
    for name, d in sorted(per.items(), key=lambda kv: -kv[1].get("gpu__time_duration.sum", 0.0)):
        t = d.get("gpu__time_duration.sum", 0.0)
        out.append(f"| `{name}` | {len(launches[name])} | {t:.1f} | {100 * t / tot_us if tot_us else 0:.1f}% | "
                   f"{d.get('dram__bytes_read.sum', 0) / 1e6:.1f} | {d.get('dram__bytes_write.sum', 0) / 1e6:.1f} |")
    md = os.path.join(ROOT, "profiles", f"launches_{args.ncu_name}.md")
    with open(md, "w") as f:
        f.write("\n".join(out) + "\n")
    print(md)
    gemm = [n for n in per if n.startswith("k_verify_gemm")]
    if gemm and any("dram__bytes_read.sum" in per[n] for n in gemm):
        n_l = sum(len(launches[n]) for n in gemm)
        dram = sum(per[n].get("dram__bytes_read.sum", 0) + per[n].get("dram__bytes_write.sum", 0) for n in gemm)
        rec = {"kernel": ", ".join(sorted(gemm)), "workload": args.ncu_name, "launches": n_l,
               "dram_bytes_total": dram, "dram_bytes_per_launch": dram / n_l,
               "kernel_source_hash": kernel_source_hash(), "command": args.ncu_command}
        js = os.path.join(ROOT, "profiles", f"k_verify_gemm_{args.ncu_name}_traffic.json")
        with open(js, "w") as f:
            json.dump(rec, f, indent=1)
        print(js)
    return 0


def run_only_attention(args) -> int:
    """The tree-attention and DeltaNet measurements alone (one line of JSON), for profiling."""
    import torch
    from quantized_speculative_verify_gb300 import hq
    device = torch.device("cuda", 0)
    hq.load()
    peak, _ = measured_peaks()
    stream = torch.cuda.Stream(device=device)
    torch.cuda.set_stream(stream)
    print(json.dumps({"tree_attention": measure_tree_attention(torch, hq, device, stream, args, peak),
                      "delta_tree": measure_delta_tree(torch, hq, device, stream, args, peak)}))
    return 0


def run_one_gemm(args) -> int:
    """One layer of the given shape: rotate/quantize once, then --steps timed GEMM launches
    (CUDA events, after --warmup launches); the weights are larger than L2 for the 9B shapes."""
    import torch
    from quantized_speculative_verify_gb300 import hq, synth

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (the product path has no CPU fallback)")
    K, N, G, fmt, M = args.one_gemm.split(",")
    K, N, G, M = int(K), int(N), int(G), int(M)
    dev = torch.device("cuda", 0)
    W = synth.weights(N, K, seed=1, device=dev)
    layer = hq.pack_layer(W, G, fmt, hq.hq_make_signs(3, K))
    del W
    X = synth.activations(M, K, seed=2, device=dev)
    _, _, qop, sx = hq.act_buffers(layer.desc, M, dev, int8_codes=False)
    hq.hq_rotate_quant_act(layer.desc, X, M, layer.signs, None, None, qop, sx)
    ws = hq.workspace(layer.desc, M, dev)
    Y = torch.empty((M, N), dtype=torch.float32, device=dev)
    for _ in range(max(args.warmup, 1)):
        hq.hq_verify_gemm(layer.desc, layer.blob, qop, sx, M, Y, None, ws)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record()
    for _ in range(args.steps):
        hq.hq_verify_gemm(layer.desc, layer.blob, qop, sx, M, Y, None, ws)
    e1.record()
    e1.synchronize()
    if hq.hq_workspace_status(ws) != hq.HQ_OK:
        raise SystemExit("device-side wait timed out")
    us = e0.elapsed_time(e1) * 1e3 / args.steps
    print(json.dumps({"gemm": {"K": K, "N": N, "group": G, "format": fmt, "M": M}, "us_per_launch": us,
                      "weight_bytes": int(layer.blob.numel()), "GB_per_s": layer.blob.numel() / us / 1e3}))
    return 0


def main():
    args = parse_args()
    if args.summarize_ncu:
        return summarize_ncu(args)
    if args.one_gemm:
        return run_one_gemm(args)
    if args.only_attention:
        return run_only_attention(args)
    ranks = Ranks()
    try:
        if args.impl == "reference":
            return run_reference(args, ranks)
        return run_gpu(args, ranks)
    finally:
        ranks.close()


if __name__ == "__main__":
    sys.exit(main())

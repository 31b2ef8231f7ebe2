#!/usr/bin/env python3
"""Benchmark of the N:M structured-sparsity hot path on GB300.

One step is one training pass over the GPT-neo-125M-shaped linears (12
layers of QKV 768->2304, O 768->768, FC1 768->3072, FC2 3072->768, 16384
tokens, bf16, synthetic): for every weight a run-time transposable 2:4 prune
and compression (W and W^T, tensor-core metadata, bit mask), the sparse
forward Y = X W^T, the sparse backward dX = dY W (through the compressed
W^T) and the masked weight gradient dW = mask * (dY^T X).  The step is
captured once as a CUDA graph and replayed.

``value`` is the step's dense-equivalent throughput: the 144 products' 2*M*N*K
over the step time (prune included).  ``rows`` reports every hot-path row on
its own: each product class against the 2:4-sparse or dense tensor peak,
cuBLAS on the same shapes, prune/compress/decompress/check and the N:M GEMV
in GB/s against HBM bandwidth.  ``cpu_baseline`` times the CPU oracle on a
bounded sample of the same step.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]
"""
from __future__ import annotations

import argparse
import datetime as _dt
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "2:4 SpMM dense-equiv TFLOPS & % of sparse TC peak; prune+compress GB/s"
UNIT = "TFLOPS (dense-equivalent)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
SPARSE_RATIO = 2.0  # nominal 2:4-sparse / dense tensor rate for 16-bit inputs
WORKLOAD = ("gptneo125m_train_linears: 12 layers x {qkv 2304x768, o 768x768, fc1 3072x768, fc2 768x3072}, "
            "16384 tokens (8x2048), bf16, run-time transposable 2:4 prune+compress, Y=X W^T, dX=dY W, "
            "dW=mask*(dY^T X)")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.txt")
KERNEL_SOURCES = {
    "spmm_tc_sparse": "structured_sparse_gemm_nm_gb300/csrc/nm_spmm_tc.cu",
    "spmm_tc_dense_masked": "structured_sparse_gemm_nm_gb300/csrc/nm_spmm_tc.cu",
    "transposable": "structured_sparse_gemm_nm_gb300/csrc/nm_transposable.cu",
}


# ------------------------------------------------------------------ helpers
def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {k: float(d.get(k, FALLBACK_PEAKS[k])) for k in FALLBACK_PEAKS}, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def source_hash(rel: str) -> str:
    return hashlib.sha256(open(os.path.join(ROOT, rel), "rb").read()).hexdigest()[:16]


def recorded_traffic(kernel: str):
    """Per-launch DRAM bytes from the committed ncu summary, if taken on the current kernel source."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    want = source_hash(KERNEL_SOURCES[kernel])
    for line in open(TRAFFIC_FILE):
        parts = line.split()
        if len(parts) >= 4 and parts[0] == kernel and parts[1] == want:
            return {"bytes_per_launch": float(parts[2]), "workload": " ".join(parts[3:])}
    return None


class ClockSampler:
    """nvidia-smi samples taken while the timed regions run."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.windows = []

    def start(self):
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(self.index), "-lms", "50"], stdout=self.out,
                                         stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.5)

    def mark(self, t0: float, t1: float):
        self.windows.append((t0, t1))

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.2)
        self.proc.terminate()
        self.proc.wait()
        self.out.flush()
        rows = []
        for line in open(self.out.name):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                ts = _dt.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(f[2]), float(f[3]), f[5:9]))
            except ValueError:
                continue
        os.unlink(self.out.name)
        inside = [r for r in rows if any(a - 0.06 <= r[0] <= b + 0.06 for a, b in self.windows)] or rows
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        reasons = sorted({names[i] for r in inside for i in range(4) if r[3][i].lower().startswith("active")})
        return {"sm_mhz": statistics.median([r[1] for r in inside]) if inside else None,
                "sm_max_mhz": max([r[2] for r in inside]) if inside else None,
                "reasons": reasons, "samples": len(inside)}


# ------------------------------------------------------------------ workload
class GptNeoTrain:
    """Device buffers, plans and launch sequence of one training step."""

    def __init__(self, torch, nb, inputs, dev, layers: int, tokens: int):
        self.torch, self.nb = torch, nb
        self.T = T = tokens
        self.dtype = "bf16"
        tdt = torch.bfloat16
        TC = nb.NM_META_TC
        self.linears = inputs.GPTNEO_LINEARS
        self.layers = []
        for l in range(layers):
            lay = []
            for j, (_, out_f, in_f) in enumerate(self.linears):
                vb, mb = nb.nm_compressed_size(out_f, in_f, "bf16", 2, 4, TC)
                vbT, mbT = nb.nm_compressed_size(in_f, out_f, "bf16", 2, 4, TC)
                lay.append(dict(
                    out=out_f, inp=in_f,
                    W=inputs.normal((out_f, in_f), 0.02, inputs.gptneo_seed(l, j, 0), "bf16", device=dev),
                    X=inputs.normal((T, in_f), 1.0, inputs.gptneo_seed(l, j, 1), "bf16", device=dev),
                    dY=inputs.normal((T, out_f), 1.0, inputs.gptneo_seed(l, j, 2), "bf16", device=dev),
                    vals=torch.empty(vb, dtype=torch.uint8, device=dev), meta=torch.empty(mb, dtype=torch.uint8, device=dev),
                    valsT=torch.empty(vbT, dtype=torch.uint8, device=dev),
                    metaT=torch.empty(mbT, dtype=torch.uint8, device=dev),
                    mask=torch.empty(out_f * ((in_f + 31) // 32), dtype=torch.int32, device=dev),
                    dW=torch.empty((out_f, in_f), dtype=tdt, device=dev),
                    # outputs of the linear's own: work on different linears may overlap
                    Y=torch.empty((T, out_f), dtype=tdt, device=dev),
                    dX=torch.empty((T, in_f), dtype=tdt, device=dev),
                    prune_bytes=out_f * in_f * 2 + vb + mb + vbT + mbT + out_f * ((in_f + 31) // 32) * 4,
                ))
            self.layers.append(lay)
        self.s_prune = torch.cuda.Stream(device=dev)
        self.s_dw = torch.cuda.Stream(device=dev)
        self.p_fwd, self.p_dx, self.p_dw, self.ws = [], [], [], []
        for (_, o, i) in self.linears:
            self.p_fwd.append(nb.nm_spmm_plan(nb.make_desc(M=o, N=T, K=i, ab_type="bf16", cd_type="bf16", ldb=i, ldd=o)))
            self.p_dx.append(nb.nm_spmm_plan(nb.make_desc(M=i, N=T, K=o, ab_type="bf16", cd_type="bf16", ldb=o, ldd=i)))
            pdw = nb.nm_spmm_plan(nb.make_desc(M=o, N=i, K=T, mode=nb.NM_SPMM_DENSE_MASKED, ab_type="bf16",
                                               cd_type="bf16", order_a=nb.NM_COL, order_b=nb.NM_ROW,
                                               order_cd=nb.NM_ROW, lda=o, ldb=i, ldd=i,
                                               meta_layout=nb.NM_META_CANONICAL))
            self.p_dw.append(pdw)
            wsb = nb.nm_spmm_plan_workspace(pdw)
            self.ws.append((torch.empty(max(wsb, 16), dtype=torch.uint8, device=dev), wsb))
        self.algos = {}

    def search_plans(self):
        """Plan-time algorithm search for every product shape of the step, on layer 0's buffers
        (outside any timed region); records the kernel each plan keeps."""
        names = {self.nb.NM_ALGO_PAIRED: "paired", self.nb.NM_ALGO_SINGLE: "single", 0: "default"}
        for j, (name, _, _) in enumerate(self.linears):
            L = self.layers[0][j]
            ws, wsb = self.ws[j]
            a = self.nb.nm_spmm_search(self.p_fwd[j], 1.0, L["vals"], L["meta"], L["X"], 0.0, None, L["Y"])
            b = self.nb.nm_spmm_search(self.p_dx[j], 1.0, L["valsT"], L["metaT"], L["dY"], 0.0, None, L["dX"])
            c = self.nb.nm_spmm_search(self.p_dw[j], 1.0, L["dY"], L["mask"], L["X"], 0.0, None, L["dW"],
                                       ws if wsb else None, wsb)
            self.algos[name] = {"fwd": names.get(a, a), "dx": names.get(b, b), "dw": names.get(c, c),
                                "dw_split_k": self.nb.nm_spmm_plan_split_k(self.p_dw[j])}

    def gemm_flops(self, j: int) -> float:
        _, o, i = self.linears[j]
        return 2.0 * o * i * self.T

    def flops_per_step(self) -> float:
        return 3.0 * sum(self.gemm_flops(j) for j in range(len(self.linears))) * len(self.layers)

    # one library call each; the return value is the number of kernels it launches
    def prune_one(self, l: int, j: int) -> int:
        nb, L = self.nb, self.layers[l][j]
        o, i = L["out"], L["inp"]
        nb.nm_prune_transposable(L["W"], o, i, i, "bf16", None, 0, L["mask"], L["vals"], L["meta"], L["valsT"],
                                 L["metaT"], nb.NM_META_TC)
        return 1

    def fwd_one(self, l: int, j: int) -> int:
        L = self.layers[l][j]
        self.nb.nm_spmm(self.p_fwd[j], 1.0, L["vals"], L["meta"], L["X"], 0.0, None, L["Y"])
        return 1

    def dx_one(self, l: int, j: int) -> int:
        L = self.layers[l][j]
        self.nb.nm_spmm(self.p_dx[j], 1.0, L["valsT"], L["metaT"], L["dY"], 0.0, None, L["dX"])
        return 1

    def dw_one(self, l: int, j: int) -> int:
        L = self.layers[l][j]
        ws, wsb = self.ws[j]
        self.nb.nm_spmm(self.p_dw[j], 1.0, L["dY"], L["mask"], L["X"], 0.0, None, L["dW"], ws if wsb else None, wsb)
        # the product, and the finalize when a K split is not summed inside the product
        return self.nb.nm_spmm_plan_launches(self.p_dw[j])

    def enqueue_one(self, l: int, j: int) -> int:
        """Launch one linear's work (layer l, linear j) on the current stream; returns the launch count."""
        return self.prune_one(l, j) + self.fwd_one(l, j) + self.dx_one(l, j) + self.dw_one(l, j)

    def enqueue_training_step(self) -> int:
        """One training step on three streams, with the ordering a real one has: the
        weights' run-time prune runs ahead on its own stream; the forward products run in
        layer order, each after its weight's prune; the dX products run in reverse order
        after them, and each linear's masked dW runs on a third stream once its dX has
        been issued (its dY is known by then), beside the rest of the dX chain.  The
        split-K workspace of a linear shape is shared by its dW launches, which stay in
        order on their stream.  Returns the number of kernels launched."""
        torch = self.torch
        main = torch.cuda.current_stream()
        self.s_prune.wait_stream(main)
        self.s_dw.wait_stream(main)
        n = 0
        pruned = {}
        with torch.cuda.stream(self.s_prune):
            for l, lay in enumerate(self.layers):
                for j in range(len(lay)):
                    n += self.prune_one(l, j)
                    e = torch.cuda.Event()
                    e.record(self.s_prune)
                    pruned[(l, j)] = e
        for l, lay in enumerate(self.layers):
            for j in range(len(lay)):
                main.wait_event(pruned[(l, j)])
                n += self.fwd_one(l, j)
        for l in reversed(range(len(self.layers))):
            for j in reversed(range(len(self.layers[l]))):
                n += self.dx_one(l, j)
                e = torch.cuda.Event()
                e.record(main)
                self.s_dw.wait_event(e)
                with torch.cuda.stream(self.s_dw):
                    n += self.dw_one(l, j)
        main.wait_stream(self.s_prune)
        main.wait_stream(self.s_dw)
        return n

    def enqueue(self, parts=("prune", "fwd", "dx", "dw"), only=None) -> int:
        """Launch the step's work on the current stream; returns the number of kernels launched."""
        nb = self.nb
        n = 0
        for l, lay in enumerate(self.layers):
            for j, L in enumerate(lay):
                if only is not None and j != only:
                    continue
                if "prune" in parts:
                    n += self.prune_one(l, j)
                if "fwd" in parts:
                    n += self.fwd_one(l, j)
                if "dx" in parts:
                    n += self.dx_one(l, j)
                if "dw" in parts:
                    n += self.dw_one(l, j)
        return n


def capture(torch, fn):
    """CUDA graph of fn's launches (fn runs once untimed first)."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def time_replays(torch, g, reps: int, barrier=None) -> float:
    """Milliseconds for `reps` back-to-back replays, events on the replay stream."""
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    if barrier:
        barrier()
    a.record()
    for _ in range(reps):
        g.replay()
    b.record()
    torch.cuda.synchronize()
    if barrier:
        barrier()
    return a.elapsed_time(b)


class Flusher:
    """Evicts L2 between timed launches: writes a buffer larger than L2, then reads
    it back, so the dirty lines of the write are written back to HBM before the
    timed launch starts instead of during it."""

    def __init__(self, torch, dev, mib=512):
        self.buf = torch.empty(mib << 19, dtype=torch.int16, device=dev)

    def __call__(self):
        self.buf.fill_(1)
        self.buf.max()


def time_launch(torch, fn, flush, reps=10, warm=3):
    """Median milliseconds of one launch of fn, L2 flushed before each."""
    for _ in range(warm):
        fn()
    ts = []
    for _ in range(reps):
        flush()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    return statistics.median(ts)


L2_BYTES = 132_000_000  # 126 MiB of L2 on GB300


def cusparselt_ms(torch, nb, A, B_t, flush, dt="bf16"):
    """cuSPARSELt's own 2:4 product (torch's private binding, run as a black box) of the 2:4-pruned
    A (M x K, pruned here by this library's nm_prune) and B_t (N x K, so B = B_t^T), D written N x M
    as this library's plans write it; the library's best algorithm id from its own search.  Returns
    (ms, note), ms None where the installed build has no cuSPARSELt."""
    try:
        if not torch.backends.cusparselt.is_available():
            return None, "cuSPARSELt not available in this torch build"
        M, K = A.shape
        Ap = torch.empty_like(A)
        nb.nm_prune(A, M, K, K, dt, 2, 4, Ap, K)
        Ac = torch._cslt_compress(Ap)
        try:
            alg = int(torch._cslt_sparse_mm_search(Ac, B_t.t(), transpose_result=True))
        except Exception:
            alg = 0
        fn = lambda: torch._cslt_sparse_mm(Ac, B_t.t(), transpose_result=True, alg_id=alg)  # noqa: E731
        fn()
        torch.cuda.synchronize()
        return time_launch(torch, fn, flush), f"torch._cslt_sparse_mm, cuSPARSELt {torch.backends.cusparselt.version()}, alg {alg}"
    except Exception as e:  # a comparator only: the row keeps its own measurement
        return None, f"cuSPARSELt failed: {type(e).__name__}: {str(e)[:120]}"


def copies_for(bytes_per_launch: int) -> int:
    """Independent problem copies whose inputs and outputs together exceed twice the L2."""
    return max(4, min(32, -(-2 * L2_BYTES // max(1, bytes_per_launch))))


def time_stream(torch, fns, reps=5):
    """Median milliseconds per launch of `fns` run back to back on the stream.

    Every function works on its own buffers and the buffers of all of them
    together exceed twice the L2, so each launch reads its inputs from HBM,
    as it does inside a longer sequence of work.  The launches are captured
    once in a CUDA graph and the graph is replayed, as the training step is:
    the host's per-call work (argument checks, marshalling) then does not
    stand between the kernels, and launch latency overlaps the previous one."""
    g = capture(torch, lambda: [f() for f in fns])
    g.replay()
    torch.cuda.synchronize()
    ts = [time_replays(torch, g, 1) / len(fns) for _ in range(reps)]
    return statistics.median(ts)


def hbm_row(torch, make, byt, hbm, flush, **extra):
    """Row of an HBM-bound kernel: `make(r)` builds copy r's launch; `byt` = algorithmic bytes per launch."""
    fns = [make(r) for r in range(copies_for(byt))]
    t = time_stream(torch, fns)
    t1 = time_launch(torch, fns[0], flush)
    row = {"ms": t, "bytes": byt, "gbs": byt / t / 1e6, "frac_hbm": byt / t / 1e6 / hbm, "copies": len(fns),
           "ms_single": t1, "gbs_single": byt / t1 / 1e6}
    row.update(extra)
    return row


# ------------------------------------------------------------------ next rows
def time_steps(torch, fn, reps=10, warm=3, trials=3):
    """Milliseconds per call of fn in a training loop: `reps` calls back to back between two CUDA
    events on the current stream (the host enqueues ahead of the GPU as a loop does; no L2
    flush), the median over `trials` such loops."""
    for _ in range(warm):
        fn()
    torch.cuda.synchronize()
    ts = []
    for _ in range(trials):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            fn()
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b) / reps)
    return statistics.median(ts)


def time_graph(torch, fn, reps=10, warm=3, trials=3):
    """Milliseconds per replay of fn captured once in a CUDA graph (warmed up on the capture
    stream first): the step's GPU time without the host's per-call work."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(warm):
            fn()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fn()
    return time_steps(torch, g.replay, reps=reps, warm=1, trials=trials)


def layer_rows(torch, nb, inputs, dev, flush, sparse_peak):
    """The built next rows: the 2:4 training layer (forward, backward and the SGD step fused
    into the transposable re-prune), the activation-sparse layer, and the int8 and fp32
    outputs of the products, each beside dense PyTorch (cuBLAS) doing the same work."""
    from structured_sparse_gemm_nm_gb300.sparse_activation import SparseActivationLinear
    from structured_sparse_gemm_nm_gb300.sparse_linear import SemiStructuredSparseLinear

    F = torch.nn.functional
    rows = {}
    tdt = {"f16": torch.float16, "bf16": torch.bfloat16}
    lr = 1e-3
    # N1: the MLP workload (512 -> 256, 4096 post-ReLU tokens, fp16) and a GPT-neo FC1 layer (bf16)
    for name, (T, in_f, out_f, dt) in (("mlp", (4096, 512, 256, "f16")), ("gptneo_fc1", (16384, 768, 3072, "bf16"))):
        W = inputs.normal((out_f, in_f), 0.05 if name == "mlp" else 0.02, inputs.SEED_W, dt, device=dev)
        X = (inputs.relu_normal((T, in_f), inputs.SEED_X, dt) if name == "mlp" else
             inputs.normal((T, in_f), 1.0, inputs.SEED_X, dt)).to(dev).requires_grad_(True)
        dY = inputs.normal((T, out_f), 0.01 if name == "mlp" else 1.0, inputs.SEED_DY, dt, device=dev)
        layer = SemiStructuredSparseLinear(in_f, out_f, tdt[dt], dev, weight=W)

        def step(layer=layer, X=X, dY=dY):
            layer.weight.grad = None
            X.grad = None
            layer(X).backward(dY)
            layer.sgd_step_(lr)
        t = time_steps(torch, step)
        Wd = torch.nn.Parameter(W.clone())

        def dense_step(Wd=Wd, X=X, dY=dY):
            Wd.grad = None
            X.grad = None
            F.linear(X, Wd).backward(dY)
            with torch.no_grad():
                Wd.add_(Wd.grad, alpha=-lr)
        td = time_steps(torch, dense_step)
        tg, tdg = time_graph(torch, step), time_graph(torch, dense_step)
        f = 3 * 2.0 * T * in_f * out_f
        rows[f"N1_layer_{name}"] = {
            "shape_T_in_out": [T, in_f, out_f], "ms": t, "tflops": f / t / 1e9, "dense_torch_ms": td,
            "speedup_vs_dense": td / t, "ms_graph": tg, "tflops_graph": f / tg / 1e9, "dense_torch_ms_graph": tdg,
            "speedup_vs_dense_graph": tdg / tg,
            "note": "SemiStructuredSparseLinear forward, backward (2:4 dX, masked dW) and sgd_step_ (SGD write fused "
                    "with the transposable re-prune and both compressions), eager, steps back to back on the current "
                    "stream, and the same step captured once in a CUDA graph (_graph keys); dense: F.linear forward, "
                    "backward and an in-place SGD update, timed the same two ways"}
        del layer, X, dY, Wd
    # N2: activation-sparse GPT-neo FC2 (3072 -> 768, 16384 post-ReLU tokens, bf16)
    T, in_f, out_f = 16384, 3072, 768
    W = inputs.normal((out_f, in_f), 0.02, inputs.SEED_W, "bf16", device=dev)
    X = inputs.relu_normal((T, in_f), inputs.SEED_X, "bf16").to(dev).requires_grad_(True)
    dY = inputs.normal((T, out_f), 1.0, inputs.SEED_DY, "bf16", device=dev)
    layer = SparseActivationLinear(in_f, out_f, torch.bfloat16, dev, weight=W)

    def act_step():
        layer.weight.grad = None
        X.grad = None
        layer(X).backward(dY)
    t = time_steps(torch, act_step)
    Wd = torch.nn.Parameter(W.clone())

    def act_dense():
        Wd.grad = None
        X.grad = None
        F.linear(X, Wd).backward(dY)
    td = time_steps(torch, act_dense)
    tg, tdg = time_graph(torch, act_step), time_graph(torch, act_dense)
    f = 3 * 2.0 * T * in_f * out_f
    rows["N2_activation_gptneo_fc2"] = {
        "shape_T_in_out": [T, in_f, out_f], "ms": t, "tflops": f / t / 1e9, "dense_torch_ms": td,
        "speedup_vs_dense": td / t, "ms_graph": tg, "tflops_graph": f / tg / 1e9, "dense_torch_ms_graph": tdg,
        "speedup_vs_dense_graph": tdg / tg,
        "note": "SparseActivationLinear forward (one-pass 2:4 prune+compress of X, X as the sparse operand) and "
                "backward (masked dX, dW on the pruned X), eager and captured in a CUDA graph (_graph keys); "
                "dense: F.linear forward and backward, timed the same two ways"}
    del layer, X, dY, Wd
    # N4: the int8 output of the int8 2:4 product and the fp32 output of the 16-bit one
    M, N, K = 4096, 4096, 1024
    Wi = inputs.uniform_int8((M, K), inputs.SEED_W + M).to(dev)
    Xi = inputs.uniform_int8((N, K), inputs.SEED_X + N).to(dev)
    vb, mb = nb.nm_compressed_size(M, K, "i8", 2, 4, nb.NM_META_CANONICAL)
    vals = torch.empty(vb, dtype=torch.uint8, device=dev)
    meta = torch.empty(mb, dtype=torch.uint8, device=dev)
    nb.nm_compress(Wi, M, K, K, "i8", 2, 4, 0, nb.NM_META_CANONICAL, vals, meta)
    Di = torch.empty((N, M), dtype=torch.int8, device=dev)
    plan = nb.nm_spmm_plan(nb.make_desc(M=M, N=N, K=K, ab_type="i8", cd_type="i8", ldb=K, ldd=M,
                                        meta_layout=nb.NM_META_CANONICAL))
    t = time_launch(torch, lambda: nb.nm_spmm(plan, 0.01, vals, meta, Xi, 0.0, None, Di), flush)
    rows["N4_int8_out_4096x4096x1024"] = {"ms": t, "tops": 2.0 * M * N * K / t / 1e9,
                                          "note": "int8 in, int8 out: saturate(rne(alpha * acc)), one launch after an "
                                                  "L2 flush"}
    plan.destroy()
    M, N, K = 3072, 16384, 768
    W = inputs.normal((M, K), 0.02, inputs.SEED_W, "bf16", device=dev)
    Xb = inputs.normal((N, K), 1.0, inputs.SEED_X, "bf16", device=dev)
    vb, mb = nb.nm_compressed_size(M, K, "bf16", 2, 4, nb.NM_META_TC)
    vals = torch.empty(vb, dtype=torch.uint8, device=dev)
    meta = torch.empty(mb, dtype=torch.uint8, device=dev)
    nb.nm_compress(W, M, K, K, "bf16", 2, 4, 0, nb.NM_META_TC, vals, meta)
    D32 = torch.empty((N, M), dtype=torch.float32, device=dev)
    plan = nb.nm_spmm_plan(nb.make_desc(M=M, N=N, K=K, ab_type="bf16", cd_type="f32", ldb=K, ldd=M))
    t = time_launch(torch, lambda: nb.nm_spmm(plan, 1.0, vals, meta, Xb, 0.0, None, D32), flush)
    f = 2.0 * M * N * K
    rows["N4_f32_out_gptneo_fc1_fwd"] = {"shape_MNK": [M, N, K], "ms": t, "tflops": f / t / 1e9,
                                         "frac_sparse_peak": f / t / 1e9 / sparse_peak,
                                         "note": "bf16 in, fp32 D (201 MB written), one launch after an L2 flush"}
    plan.destroy()
    torch.cuda.empty_cache()
    return rows


# ------------------------------------------------------------------ rows
def measure_rows(torch, nb, inputs, dev, wl: GptNeoTrain, peaks):
    flush = Flusher(torch, dev)
    hbm = peaks["hbm_gbs"]
    dense_peak = peaks["bf16_tflops"]
    sparse_peak = dense_peak * SPARSE_RATIO
    rows = {}

    # S5/S6/S7 per GPT-neo shape, one layer's weights, with cuBLAS on the dense pruned weight
    L0 = wl.layers[0]
    for j, (name, o, i) in enumerate(wl.linears):
        L = L0[j]
        f = wl.gemm_flops(j)
        t_fwd = time_launch(torch, lambda: nb.nm_spmm(wl.p_fwd[j], 1.0, L["vals"], L["meta"], L["X"], 0.0, None, L["Y"]), flush)
        t_dx = time_launch(torch, lambda: nb.nm_spmm(wl.p_dx[j], 1.0, L["valsT"], L["metaT"], L["dY"], 0.0, None, L["dX"]), flush)
        ws, wsb = wl.ws[j]
        t_dw = time_launch(torch, lambda: nb.nm_spmm(wl.p_dw[j], 1.0, L["dY"], L["mask"], L["X"], 0.0, None, L["dW"],
                                                     ws if wsb else None, wsb), flush)
        Wd = L["W"]
        t_cub = time_launch(torch, lambda: torch.matmul(L["X"], Wd.t()), flush)
        t_cub_dx = time_launch(torch, lambda: torch.matmul(L["dY"], Wd), flush)
        rows[f"S5_fwd_{name}"] = {"shape_MNK": [o, wl.T, i], "ms": t_fwd, "tflops": f / t_fwd / 1e9,
                                  "frac_sparse_peak": f / t_fwd / 1e9 / sparse_peak,
                                  "cublas_dense_tflops": f / t_cub / 1e9, "speedup_vs_cublas": t_cub / t_fwd}
        rows[f"S6_dx_{name}"] = {"shape_MNK": [i, wl.T, o], "ms": t_dx, "tflops": f / t_dx / 1e9,
                                 "frac_sparse_peak": f / t_dx / 1e9 / sparse_peak,
                                 "cublas_dense_tflops": f / t_cub_dx / 1e9, "speedup_vs_cublas": t_cub_dx / t_dx}
        for key, A, Bt, t_own in ((f"S5_fwd_{name}", Wd, L["X"], t_fwd),
                                  (f"S6_dx_{name}", Wd.t().contiguous(), L["dY"], t_dx)):
            t_sl, note = cusparselt_ms(torch, nb, A, Bt, flush)
            rows[key]["cusparselt_tflops"] = f / t_sl / 1e9 if t_sl else None
            rows[key]["speedup_vs_cusparselt"] = t_sl / t_own if t_sl else None
            rows[key]["cusparselt_note"] = note
        t_cub_dw = time_launch(torch, lambda: torch.matmul(L["dY"].t(), L["X"]), flush)
        rows[f"S7_dw_{name}"] = {"shape_MNK": [o, i, wl.T], "ms": t_dw, "tflops": f / t_dw / 1e9,
                                 "frac_dense_peak": f / t_dw / 1e9 / dense_peak,
                                 "cublas_dense_tflops": f / t_cub_dw / 1e9, "speedup_vs_cublas": t_cub_dw / t_dw,
                                 "cublas_note": "torch.matmul(dY^T, X) without the mask multiply"}
        # the forward product with each tensor-core kernel fixed (the step's plan keeps the searched one)
        for algo, aname in ((nb.NM_ALGO_PAIRED, "paired"), (nb.NM_ALGO_SINGLE, "single")):
            pp = nb.nm_spmm_plan(nb.make_desc(M=o, N=wl.T, K=i, ab_type="bf16", cd_type="bf16", ldb=i, ldd=o,
                                              algo=algo))
            t_a = time_launch(torch, lambda: nb.nm_spmm(pp, 1.0, L["vals"], L["meta"], L["X"], 0.0, None, L["Y"]),
                              flush)
            rows[f"S5_fwd_{name}_{aname}"] = {"shape_MNK": [o, wl.T, i], "ms": t_a, "tflops": f / t_a / 1e9,
                                              "frac_sparse_peak": f / t_a / 1e9 / sparse_peak}
            pp.destroy()

    # HBM-bound rows: `ms` is the per-launch time of back-to-back launches over
    # copies whose buffers exceed the L2 (see time_stream); `ms_single` is one
    # launch after an L2 flush, launch latency included.
    def empty(nbytes):
        return torch.empty(max(16, nbytes), dtype=torch.uint8, device=dev)

    # S3: transposable prune + dual compress (+ mask) of each GPT-neo weight shape, bf16
    for j, (name, o, i) in enumerate(wl.linears):
        vb, mb = nb.nm_compressed_size(o, i, "bf16", 2, 4, nb.NM_META_TC)
        vbT, mbT = nb.nm_compressed_size(i, o, "bf16", 2, 4, nb.NM_META_TC)
        byt = o * i * 2 + vb + mb + vbT + mbT + o * i // 8

        def make(r, o=o, i=i, vb=vb, mb=mb, vbT=vbT, mbT=mbT):
            Wr = inputs.normal((o, i), 0.02, 500 + r, "bf16", device=dev)
            bufs = [empty(o * i // 8), empty(vb), empty(mb), empty(vbT), empty(mbT)]
            return lambda: nb.nm_prune_transposable(Wr, o, i, i, "bf16", None, 0, bufs[0], bufs[1], bufs[2], bufs[3],
                                                    bufs[4], nb.NM_META_TC)
        rows[f"S3_transposable_{name}"] = hbm_row(torch, make, byt, hbm, flush, shape=[o, i])

    # S1 / S2 / S4 / S8 on 4096 x 4096 f16 weights
    M = K = 4096

    def weight(r):
        return inputs.normal((M, K), 0.02, inputs.SEED_W + 100 * r, "f16", device=dev)

    for layout, lname in ((nb.NM_META_CANONICAL, "canonical"), (nb.NM_META_TC, "tensor_core")):
        vb, mb = nb.nm_compressed_size(M, K, "f16", 2, 4, layout)

        def make(r, vb=vb, mb=mb, layout=layout):
            Wr, v, m = weight(r), empty(vb), empty(mb)
            return lambda: nb.nm_compress(Wr, M, K, K, "f16", 2, 4, 0, layout, v, m)
        rows[f"S1_prune_compress_24_{lname}"] = hbm_row(torch, make, M * K * 2 + vb + mb, hbm, flush, shape=[M, K])

        def make(r, vb=vb, mb=mb, layout=layout):
            Wr, v, m = weight(r), empty(vb), empty(mb)
            nb.nm_compress(Wr, M, K, K, "f16", 2, 4, 0, layout, v, m)
            return lambda: nb.nm_decompress(v, m, M, K, "f16", 2, 4, layout, Wr, K)
        rows[f"S4_decompress_24_{lname}"] = hbm_row(torch, make, vb + mb + M * K * 2, hbm, flush)

    def make(r):
        Wr, cnt = weight(r), torch.zeros(4, dtype=torch.int32, device=dev)
        return lambda: nb.nm_check(Wr, M, K, K, "f16", 2, 4, 1, cnt)
    rows["S4_check_24_transposable"] = hbm_row(torch, make, M * K * 2, hbm, flush)

    def make(r):
        Wr, mask = weight(r), empty(M * K // 8)
        return lambda: nb.nm_prune(Wr, M, K, K, "f16", 2, 4, Wr, K, mask)
    rows["S1_prune_inplace_24_mask"] = hbm_row(torch, make, M * K * 4 + M * K // 8, hbm, flush)

    for n in (4, 8, 16):
        vb, mb = nb.nm_compressed_size(M, K, "f16", n, 32)

        def make(r, n=n, vb=vb, mb=mb):
            Wr, v, m = weight(r), empty(vb), empty(mb)
            return lambda: nb.nm_compress(Wr, M, K, K, "f16", n, 32, 0, nb.NM_META_CANONICAL, v, m)
        rows[f"S2_prune_compress_{n}of32"] = hbm_row(torch, make, M * K * 2 + vb + mb, hbm, flush)
        for b in (1, 8):
            plan = nb.nm_spmm_plan(nb.make_desc(M=M, N=b, K=K, n=n, m=32, ab_type="f16", cd_type="f16", ldb=K, ldd=M,
                                                meta_layout=nb.NM_META_CANONICAL))

            def make(r, n=n, vb=vb, mb=mb, b=b, plan=plan):
                Wr, v, m = weight(r % 4), empty(vb), empty(mb)
                nb.nm_compress(Wr, M, K, K, "f16", n, 32, 0, nb.NM_META_CANONICAL, v, m)
                x = inputs.normal((b, K), 1.0, inputs.SEED_VEC + r, "f16", device=dev)
                y = torch.empty((b, M), dtype=torch.float16, device=dev)
                return lambda: nb.nm_spmm(plan, 1.0, v, m, x, 0.0, None, y)
            byt = vb + mb + b * K * 2 + b * M * 2
            row = hbm_row(torch, make, byt, hbm, flush)
            row["gflops"] = 2.0 * M * (K // 32) * n * b / row["ms"] / 1e6
            rows[f"S8_gemv_{n}of32_b{b}"] = row
            plan.destroy()

    # S9: vector-wise (1 x 32) and block-wise (32 x 32) selection at density 0.25, then the product
    for bh, uname in ((1, "vector_wise"), (32, "block_wise")):
        keep = (M // bh) * (K // 32) // 4
        wsb = nb.nm_prune_units_workspace(M, K, bh, 32)
        csr_b, vals_b = (M // bh + 1 + keep) * 4, keep * bh * 32 * 2

        def make(r, bh=bh, keep=keep, wsb=wsb, csr_b=csr_b, vals_b=vals_b):
            Wr, ws, csr, vals = weight(r), empty(wsb), empty(csr_b), empty(vals_b)
            if bh == 1:
                return lambda: nb.nm_prune_vector_wise(Wr, M, K, K, "f16", 32, keep, nb.NM_SCORE_ABS_OF_SUM, csr=csr,
                                                       vals=vals, workspace=ws, workspace_bytes=wsb)
            return lambda: nb.nm_prune_block_wise(Wr, M, K, K, "f16", 32, 32, keep, csr=csr, vals=vals, workspace=ws,
                                                  workspace_bytes=wsb)
        rows[f"S9_{uname}_select_compress"] = hbm_row(torch, make, M * K * 2 + csr_b + vals_b, hbm, flush,
                                                      kept_units=keep)
        for b in (1, 8):
            plan = nb.nm_spmm_plan(nb.make_desc(M=M, N=b, K=K, mode=nb.NM_SPMM_BLOCK_SPARSE_A, n=bh, m=32,
                                                ab_type="f16", cd_type="f16", ldb=K, ldd=M,
                                                meta_layout=nb.NM_META_CANONICAL))

            def make(r, bh=bh, keep=keep, wsb=wsb, csr_b=csr_b, vals_b=vals_b, b=b, plan=plan):
                Wr, ws, csr, vals = weight(r % 4), empty(wsb), empty(csr_b), empty(vals_b)
                if bh == 1:
                    nb.nm_prune_vector_wise(Wr, M, K, K, "f16", 32, keep, nb.NM_SCORE_ABS_OF_SUM, csr=csr, vals=vals,
                                            workspace=ws, workspace_bytes=wsb)
                else:
                    nb.nm_prune_block_wise(Wr, M, K, K, "f16", 32, 32, keep, csr=csr, vals=vals, workspace=ws,
                                           workspace_bytes=wsb)
                x = inputs.normal((b, K), 1.0, inputs.SEED_VEC + r, "f16", device=dev)
                y = torch.empty((b, M), dtype=torch.float16, device=dev)
                return lambda: nb.nm_spmm(plan, 1.0, vals, csr, x, 0.0, None, y)
            byt = vals_b + csr_b + b * K * 2 + b * M * 2
            row = hbm_row(torch, make, byt, hbm, flush)
            row["gflops"] = 2.0 * keep * bh * 32 * b / row["ms"] / 1e6
            rows[f"S9_{uname}_gemv_b{b}"] = row
            plan.destroy()
        torch.cuda.empty_cache()

    # BERT-Large-shaped sparse products (f16) with cuBLAS on the same shapes
    for (Mb, Nb, Kb) in inputs.BERT_SHAPES:
        Wb = inputs.normal((Mb, Kb), 0.02, inputs.SEED_W, "f16", device=dev)
        Xb = inputs.normal((Nb, Kb), 1.0, inputs.SEED_X, "f16", device=dev)
        vb, mb = nb.nm_compressed_size(Mb, Kb, "f16", 2, 4, nb.NM_META_TC)
        vals = torch.empty(vb, dtype=torch.uint8, device=dev)
        meta = torch.empty(mb, dtype=torch.uint8, device=dev)
        nb.nm_compress(Wb, Mb, Kb, Kb, "f16", 2, 4, 0, nb.NM_META_TC, vals, meta)
        D = torch.empty((Nb, Mb), dtype=torch.float16, device=dev)
        plan = nb.nm_spmm_plan(nb.make_desc(M=Mb, N=Nb, K=Kb, ab_type="f16", cd_type="f16", ldb=Kb, ldd=Mb))
        t = time_launch(torch, lambda: nb.nm_spmm(plan, 1.0, vals, meta, Xb, 0.0, None, D), flush)
        tc = time_launch(torch, lambda: torch.matmul(Xb, Wb.t()), flush)
        f = 2.0 * Mb * Nb * Kb
        rows[f"S5_bert_{Mb}x{Nb}x{Kb}_f16"] = {"ms": t, "tflops": f / t / 1e9, "frac_sparse_peak": f / t / 1e9 / sparse_peak,
                                                "cublas_dense_tflops": f / tc / 1e9, "speedup_vs_cublas": tc / t}
        plan.destroy()
    # the BERT-Large layers of the cuSPARSELt blog's Table 1 (fp16, the same TN layout; the
    # page's numbers are A100 context: dense / sparse TFLOPS 188/263, 183/242, 196/270, 211/339)
    for lname, (Mb, Nb, Kb) in (("qkv", (3072, 16384, 1024)), ("proj", (1024, 16384, 1024)),
                                ("fc1", (4096, 16384, 1024)), ("fc2", (1024, 16384, 4096))):
        Wb = inputs.normal((Mb, Kb), 0.02, inputs.SEED_W, "f16", device=dev)
        Xb = inputs.normal((Nb, Kb), 1.0, inputs.SEED_X, "f16", device=dev)
        vb, mb = nb.nm_compressed_size(Mb, Kb, "f16", 2, 4, nb.NM_META_TC)
        vals = torch.empty(vb, dtype=torch.uint8, device=dev)
        meta = torch.empty(mb, dtype=torch.uint8, device=dev)
        nb.nm_compress(Wb, Mb, Kb, Kb, "f16", 2, 4, 0, nb.NM_META_TC, vals, meta)
        D = torch.empty((Nb, Mb), dtype=torch.float16, device=dev)
        plan = nb.nm_spmm_plan(nb.make_desc(M=Mb, N=Nb, K=Kb, ab_type="f16", cd_type="f16", ldb=Kb, ldd=Mb))
        t = time_launch(torch, lambda: nb.nm_spmm(plan, 1.0, vals, meta, Xb, 0.0, None, D), flush)
        tc = time_launch(torch, lambda: torch.matmul(Xb, Wb.t()), flush)
        f = 2.0 * Mb * Nb * Kb
        t_sl, note = cusparselt_ms(torch, nb, Wb, Xb, flush, "f16")
        rows[f"S5_bert_large_{lname}_{Mb}x{Nb}x{Kb}_f16"] = {
            "ms": t, "tflops": f / t / 1e9, "frac_sparse_peak": f / t / 1e9 / sparse_peak,
            "cublas_dense_tflops": f / tc / 1e9, "speedup_vs_cublas": tc / t,
            "cusparselt_tflops": f / t_sl / 1e9 if t_sl else None,
            "speedup_vs_cusparselt": t_sl / t if t_sl else None, "cusparselt_note": note}
        plan.destroy()
    # the same shapes in int8 (INT32 accumulation), against torch's int8 matmul of the dense
    # pruned weight where the installed build has one, and against the rate of the warp-level
    # sparse int8 MMA itself, measured now by the library's rate probe (no published figure)
    i8_peak = nb.nm_test_i8_sparse_mma_rate(20000)
    for (Mb, Nb, Kb) in inputs.BERT_SHAPES:
        Wi = inputs.uniform_int8((Mb, Kb), inputs.SEED_W + Mb).to(dev)
        Xi = inputs.uniform_int8((Nb, Kb), inputs.SEED_X + Nb).to(dev)
        vb, mb = nb.nm_compressed_size(Mb, Kb, "i8", 2, 4, nb.NM_META_CANONICAL)
        vals = torch.empty(vb, dtype=torch.uint8, device=dev)
        meta = torch.empty(mb, dtype=torch.uint8, device=dev)
        nb.nm_compress(Wi, Mb, Kb, Kb, "i8", 2, 4, 0, nb.NM_META_CANONICAL, vals, meta)
        Di = torch.empty((Nb, Mb), dtype=torch.int32, device=dev)
        plan = nb.nm_spmm_plan(nb.make_desc(M=Mb, N=Nb, K=Kb, ab_type="i8", cd_type="i32", ldb=Kb, ldd=Mb,
                                            meta_layout=nb.NM_META_CANONICAL))
        t = time_launch(torch, lambda: nb.nm_spmm(plan, 1, vals, meta, Xi, 0, None, Di), flush)
        f = 2.0 * Mb * Nb * Kb
        row = {"ms": t, "tops": f / t / 1e9, "kernel": "spmm_i8_kernel (warp-level mma.sp m16n8k64)",
               "frac_i8_sparse_mma_peak": f / t / 1e9 / i8_peak}
        try:
            WiT = Wi.t().contiguous()
            tq = time_launch(torch, lambda: torch._int_mm(Xi, WiT), flush)
            row["torch_int8_dense_tops"] = f / tq / 1e9
            row["speedup_vs_dense_int8"] = tq / t
        except Exception as e:  # no int8 matmul in this build
            row["torch_int8_dense"] = f"unavailable: {type(e).__name__}"
        rows[f"S5_bert_{Mb}x{Nb}x{Kb}_i8"] = row
        plan.destroy()
    rows.update(layer_rows(torch, nb, inputs, dev, flush, sparse_peak))
    rows["_peaks"] = {"sparse_tflops": sparse_peak, "dense_tflops": dense_peak, "hbm_gbs": hbm,
                      "i8_sparse_mma_tops": i8_peak,
                      "i8_note": "nm_test_i8_sparse_mma_rate: mma.sp m16n8k64 s8 on register operands, 8 warps x "
                                 "4 chains per SM, all SMs, dense-equivalent TOPS",
                      "note": "tensor rows: one launch after an L2 flush, burst peaks; HBM rows: back-to-back "
                              "launches over copies larger than L2 (ms), and one flushed launch (ms_single)"}
    return rows


# ------------------------------------------------------------------ CPU oracle
def oracle_sample_step(inputs, layers: int, tokens: int, seed_base: int = 0):
    """One bounded sample of the step on the CPU oracle; returns (seconds, dense-equivalent flops)."""
    import numpy as np

    import oracle as o

    flops = 0.0
    data = []
    for l in range(layers):
        for j, (_, out_f, in_f) in enumerate(inputs.GPTNEO_LINEARS):
            W = inputs.as_numpy_bits(inputs.normal((out_f, in_f), 0.02, inputs.gptneo_seed(l, j, 0) + seed_base, "bf16"))
            X = inputs.as_numpy_bits(inputs.normal((tokens, in_f), 1.0, inputs.gptneo_seed(l, j, 1) + seed_base, "bf16"))
            dY = inputs.as_numpy_bits(inputs.normal((tokens, out_f), 1.0, inputs.gptneo_seed(l, j, 2) + seed_base, "bf16"))
            data.append((W, X, dY, out_f, in_f))
    t0 = time.perf_counter()
    for (W, X, dY, out_f, in_f) in data:
        pruned, mask, (v, m), (vT, mT) = o.nm_prune_transposable(W, "bf16")
        o.meta_to_tc_layout(m, out_f, in_f)
        o.meta_to_tc_layout(mT, in_f, out_f)
        Xd, dYd = o.decode(X, "bf16"), o.decode(dY, "bf16")
        A = o.decode(o.nm_decompress(v, m, out_f, in_f, 2, 4), "bf16")
        AT = o.decode(o.nm_decompress(vT, mT, in_f, out_f, 2, 4), "bf16")
        o.spmm(1.0, A, Xd.T)       # Y^T
        o.spmm(1.0, AT, dYd.T)     # dX^T
        o.masked_weight_grad(dYd, Xd, mask)
        flops += 3 * 2.0 * out_f * in_f * tokens
    return time.perf_counter() - t0, flops


def cpu_threads() -> int:
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var])
    return os.cpu_count() or 1


ORACLE_SAMPLE = (1, 8192)  # layers, tokens per sample step


def cpu_model() -> str:
    """The host CPU's model name (lscpu), else the machine type."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform

    return platform.machine()


SINGLE_THREAD_SAMPLE = (1, 1024)  # layers, tokens


def single_thread_oracle():
    """The same oracle sample on one host thread (BLAS threads are fixed when numpy loads, so this runs
    in a child process with one thread)."""
    layers, tokens = SINGLE_THREAD_SAMPLE
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1", MKL_NUM_THREADS="1")
    code = ("import json, sys; sys.path.insert(0, %r); import bench; from structured_sparse_gemm_nm_gb300 import inputs; "
            "s, f = bench.oracle_sample_step(inputs, %d, %d); print(json.dumps([s, f]))" % (ROOT, layers, tokens))
    try:
        r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=300)
        secs, flops = json.loads(r.stdout.strip().splitlines()[-1])
    except (OSError, subprocess.SubprocessError, ValueError, IndexError):
        return None
    return {"value": flops / secs / 1e12, "unit": UNIT, "cores": 1,
            "sample": f"{layers} layer(s) x 4 linears, {tokens} of 16384 tokens, {secs:.1f} s"}


def cpu_baseline(inputs):
    layers, tokens = ORACLE_SAMPLE
    secs, flops = oracle_sample_step(inputs, layers, tokens)
    return {"value": flops / secs / 1e12, "unit": UNIT, "cores": cpu_threads(), "kind": "oracle",
            "cpu_model": cpu_model(), "single_thread": single_thread_oracle(),
            "sample": f"{layers} layer(s) x 4 linears, {tokens} of 16384 tokens (fwd, dX, masked dW in float64 "
                      f"numpy/BLAS; transposable prune, compress, decompress), {secs:.1f} s"}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    from structured_sparse_gemm_nm_gb300 import inputs

    layers, tokens = ORACLE_SAMPLE
    for _ in range(args.warmup):
        oracle_sample_step(inputs, layers, tokens)
    secs, flops = 0.0, 0.0
    for k in range(args.steps):
        s, f = oracle_sample_step(inputs, layers, tokens, seed_base=k)
        secs += s
        flops += f
    value = flops / secs / 1e12
    sample = f"{layers} layer(s) x 4 linears, {tokens} of 16384 tokens per step"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "sample": sample},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_threads(), "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ native arm
def host_link_gbs(torch, dev, nbytes=1 << 30):
    """Host-device copy bandwidth of this machine, measured in the same run: pinned 1 GiB copies each way."""
    h = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    d = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    out = {}
    for name, fn in (("h2d", lambda: d.copy_(h, non_blocking=True)), ("d2h", lambda: h.copy_(d, non_blocking=True))):
        fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(3):
            fn()
        b.record()
        torch.cuda.synchronize()
        out[name] = 3 * nbytes / (a.elapsed_time(b) * 1e-3) / 1e9
    del h, d
    return out


def aggregate_over_ranks(torch, dist, elapsed_ms: float) -> float:
    """Max of a per-rank elapsed time over all ranks (plain value when not distributed)."""
    if dist is None:
        return elapsed_ms
    t = torch.tensor([elapsed_ms], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_native(args):
    import torch

    from structured_sparse_gemm_nm_gb300 import binding as nb
    from structured_sparse_gemm_nm_gb300 import inputs

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist_mod

        torch.cuda.set_device(local)
        dist_mod.init_process_group("nccl")
        dist = dist_mod
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    barrier = dist.barrier if dist else None
    peaks, peak_kind = load_peaks()
    nb.lib()

    wl = GptNeoTrain(torch, nb, inputs, dev, inputs.GPTNEO_LAYERS, inputs.GPTNEO_TOKENS)
    # the native arm's algorithm search (its tensor-core products keep whichever of the paired and
    # single-CTA kernels measured faster on each shape, the dW products also the fastest of the
    # K splits near the planned one); --no-search keeps the library's default
    # (paired CTAs where M spans an even number of 128-row blocks), e.g. for profiler runs, where
    # the search would time its candidates through the profiler
    if args.no_search:
        wl.algos = {name: {"fwd": "default", "dx": "default", "dw": "default",
                           "dw_split_k": nb.nm_spmm_plan_split_k(wl.p_dw[j])} for j, (name, _, _) in enumerate(wl.linears)}
    else:
        wl.search_plans()
    torch.cuda.synchronize()
    launches_per_step = [0]

    def step():
        launches_per_step[0] = wl.enqueue_training_step()

    g_step = capture(torch, step)
    sampler = ClockSampler(local)
    sampler.start()
    for _ in range(args.warmup):
        g_step.replay()
    torch.cuda.synchronize()
    t0 = time.time()
    ms = time_replays(torch, g_step, args.steps, barrier)
    sampler.mark(t0, time.time())
    ms = aggregate_over_ranks(torch, dist, ms)
    ms_step = ms / args.steps
    flops = wl.flops_per_step()
    value = flops * world / (ms_step * 1e-3) / 1e12

    # per-class graphs: the roofline of the dominant kernel and the split of the step
    classes = {}
    for cls, parts in (("spmm_tc_sparse", ("fwd", "dx")), ("spmm_tc_dense_masked", ("dw",)),
                       ("transposable", ("prune",))):
        cnt = [0]

        def f(parts=parts, cnt=cnt):
            cnt[0] = wl.enqueue(parts)

        g = capture(torch, f)
        t0 = time.time()
        cms = time_replays(torch, g, args.steps, barrier)
        sampler.mark(t0, time.time())
        classes[cls] = {"ms_per_step": cms / args.steps, "launches_per_step": cnt[0]}
        del g
    sparse_flops = 2 * sum(wl.gemm_flops(j) for j in range(4)) * len(wl.layers)
    dense_flops = sum(wl.gemm_flops(j) for j in range(4)) * len(wl.layers)
    prune_bytes = sum(L["prune_bytes"] for lay in wl.layers for L in lay)
    classes["spmm_tc_sparse"]["tflops"] = sparse_flops / classes["spmm_tc_sparse"]["ms_per_step"] / 1e9
    classes["spmm_tc_dense_masked"]["tflops"] = dense_flops / classes["spmm_tc_dense_masked"]["ms_per_step"] / 1e9
    classes["transposable"]["gbs"] = prune_bytes / classes["transposable"]["ms_per_step"] / 1e6
    dominant = max(classes, key=lambda c: classes[c]["ms_per_step"])
    c = classes[dominant]
    # Each class is timed alone as its own graph of a few tens of milliseconds: the burst peak
    # applies (the sustained one is for a kernel timed inside a seconds-long region).
    burst = peaks["bf16_tflops"]
    if dominant == "transposable":
        achieved, peak, unit, bound = c["gbs"], peaks["hbm_gbs"], "GB/s", "hbm"
        per_launch_alg = prune_bytes / c["launches_per_step"]
        pnote = f"HBM copy bandwidth ({peak_kind})"
    else:
        achieved = c["tflops"]
        sparse = dominant == "spmm_tc_sparse"
        peak = burst * (SPARSE_RATIO if sparse else 1.0)
        unit, bound = "TFLOP/s", "tensor"
        per_launch_alg = (sparse_flops if sparse else dense_flops) / c["launches_per_step"]
        pnote = (f"{peak_kind} burst bf16 dense" + (" x 2 (nominal 2:4 sparse ratio)" if sparse else "") +
                 "; the class is timed alone as its own CUDA graph")
    tr = recorded_traffic(dominant)
    roofline = {"kernel": dominant, "bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                "frac": achieved / peak, "traffic": tr["bytes_per_launch"] if tr else None,
                "algorithmic_per_launch": per_launch_alg, "peak_source": pnote,
                "traffic_source": tr["workload"] if tr else "no ncu capture of the current kernel source"}

    # end to end: inputs from pinned host memory, dW back to the host, every step
    e2e = None
    if not args.no_e2e:
        host_in, host_out = [], []
        for lay in wl.layers:
            for L in lay:
                for key in ("W", "X", "dY"):
                    h = torch.empty(L[key].shape, dtype=L[key].dtype, pin_memory=True)
                    h.copy_(L[key])
                    host_in.append((h, L[key]))
                host_out.append((torch.empty(L["dW"].shape, dtype=L["dW"].dtype, pin_memory=True), L["dW"]))
        h2d = sum(h.numel() * h.element_size() for h, _ in host_in)
        d2h = sum(h.numel() * h.element_size() for h, _ in host_out)

        # Pipelined: each linear's inputs are copied on one of two copy streams, its work runs on
        # the compute stream as soon as they have landed, and its dW goes back on a third stream
        # as soon as it is written.  Across steps, a copy into a buffer waits for the previous
        # step's reads of it (compute reading W, X, dY; the copy-out reading dW).
        n_lin = len(host_out)
        s_c = torch.cuda.current_stream()
        s_in = [torch.cuda.Stream(), torch.cuda.Stream()]
        s_out = torch.cuda.Stream()
        e_in = [torch.cuda.Event() for _ in range(n_lin)]
        e_done = [torch.cuda.Event() for _ in range(n_lin)]
        e_out = [torch.cuda.Event() for _ in range(n_lin)]
        seen = [False]

        def e2e_step():
            for st in s_in + [s_out]:
                st.wait_stream(s_c)
            k = 0
            for l, lay in enumerate(wl.layers):
                for j, L in enumerate(lay):
                    si = s_in[k % 2]
                    with torch.cuda.stream(si):
                        if seen[0]:
                            si.wait_event(e_done[k])
                        for h, d in host_in[3 * k:3 * k + 3]:
                            d.copy_(h, non_blocking=True)
                        e_in[k].record(si)
                    s_c.wait_event(e_in[k])
                    if seen[0]:
                        s_c.wait_event(e_out[k])
                    wl.enqueue_one(l, j)
                    e_done[k].record(s_c)
                    with torch.cuda.stream(s_out):
                        s_out.wait_event(e_done[k])
                        h, d = host_out[k]
                        h.copy_(d, non_blocking=True)
                        e_out[k].record(s_out)
                    k += 1
            seen[0] = True
            for st in s_in + [s_out]:
                s_c.wait_stream(st)

        e2e_step()
        torch.cuda.synchronize()
        reps = max(1, args.steps)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if barrier:
            barrier()
        t0 = time.time()
        a.record()
        for _ in range(reps):
            e2e_step()
        b.record()
        torch.cuda.synchronize()
        sampler.mark(t0, time.time())
        ems = aggregate_over_ranks(torch, dist, a.elapsed_time(b)) / reps
        link = host_link_gbs(torch, dev)
        e2e = {"value": flops * world / (ems * 1e-3) / 1e12, "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": ems, "host_link_gbs": link,
               "link_bound_ms_per_step": h2d / (link["h2d"] * 1e6),
               "path": "pinned host -> device copies of W, X, dY of every linear on two copy streams; each "
                       "linear's prune, forward, dX and dW through the C ABI on the compute stream once its "
                       "inputs have landed; each dW back to pinned host memory on a third stream once written"}
        del host_in, host_out
    clocks = sampler.stop()

    rows = None
    if rank == 0 and not args.no_rows:
        rows = measure_rows(torch, nb, inputs, dev, wl, peaks)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = cpu_baseline(inputs)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": WORKLOAD, "global_tokens": inputs.GPTNEO_TOKENS * world,
                       "l2": "inputs larger than L2: 4.8 GB of distinct per-linear activations per step",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "graph": "one CUDA graph per step on three streams: run-time prune ahead, forward chain "
                                "then dX chain, each dW beside the dX chain",
                       "algos": wl.algos},
            "roofline": roofline, "cpu_baseline": cpu, "clocks": clocks, "e2e": e2e,
            "gpu_launches": launches_per_step[0] * args.steps,
            "step_split_ms": {k: v["ms_per_step"] for k, v in classes.items()},
            "classes": classes, "rows": rows,
        }
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()
    return 0


# ------------------------------------------------------------------ single-kernel cases (ncu captures)
LINEARS = {"qkv": (2304, 768), "o": (768, 768), "fc1": (3072, 768), "fc2": (768, 3072)}  # out x in
SPARSE_CASES = tuple(f"sparse_{lin}_{d}" for lin in LINEARS for d in ("fwd", "dx"))
KERNEL_CASES = SPARSE_CASES + ("dense_fc1_dw", "dense_o_dw", "transposable_fc1", "prune24_4096",
                               "prune_8of32_4096", "gemv_8of32_b8", "vector_wise_4096", "check24_4096")


def run_kernel_case(name: str, reps: int = 3):
    """Runs one kernel of the hot path `reps` times on inputs larger than L2 (for profiler captures)."""
    import torch

    from structured_sparse_gemm_nm_gb300 import binding as nb
    from structured_sparse_gemm_nm_gb300 import inputs

    dev = torch.device("cuda", 0)
    nb.lib()
    T = inputs.GPTNEO_TOKENS
    if name in SPARSE_CASES:
        # the step's sparse product of one linear: forward (M = out, K = in) or dX (M = in, K = out)
        _, lin, d = name.split("_")
        o, i = LINEARS[lin]
        M, K = (o, i) if d == "fwd" else (i, o)
        W = inputs.normal((M, K), 0.02, 1, "bf16", device=dev)
        vb, mb = nb.nm_compressed_size(M, K, "bf16", 2, 4, nb.NM_META_TC)
        vals, meta = (torch.empty(vb, dtype=torch.uint8, device=dev), torch.empty(mb, dtype=torch.uint8, device=dev))
        nb.nm_compress(W, M, K, K, "bf16", 2, 4, 0, nb.NM_META_TC, vals, meta)
        X = inputs.normal((T, K), 1.0, 2, "bf16", device=dev)
        Y = torch.empty((T, M), dtype=torch.bfloat16, device=dev)
        plan = nb.nm_spmm_plan(nb.make_desc(M=M, N=T, K=K, ab_type="bf16", cd_type="bf16", ldb=K, ldd=M))
        fn = [lambda: nb.nm_spmm(plan, 1.0, vals, meta, X, 0.0, None, Y)]
    elif name in ("dense_fc1_dw", "dense_o_dw", "transposable_fc1"):
        # FC1 weight (out x in; FC2 dX has the same M, K), or the O weight, whose dW sums seven
        # K splits in the separate finalize
        o, i = (768, 768) if name == "dense_o_dw" else (3072, 768)
        W = inputs.normal((o, i), 0.02, 1, "bf16", device=dev)
        vb, mb = nb.nm_compressed_size(o, i, "bf16", 2, 4, nb.NM_META_TC)
        vals, meta = (torch.empty(vb, dtype=torch.uint8, device=dev), torch.empty(mb, dtype=torch.uint8, device=dev))
        mask = torch.empty(o * i // 32, dtype=torch.int32, device=dev)
        nb.nm_prune_transposable(W, o, i, i, "bf16", None, 0, mask, vals, meta, None, None, nb.NM_META_TC)
        if name == "transposable_fc1":
            Ws = [inputs.normal((o, i), 0.02, 10 + r, "bf16", device=dev) for r in range(reps)]
            vbT, mbT = nb.nm_compressed_size(i, o, "bf16", 2, 4, nb.NM_META_TC)
            valsT, metaT = (torch.empty(vbT, dtype=torch.uint8, device=dev), torch.empty(mbT, dtype=torch.uint8, device=dev))
            fn = [lambda Wr=Wr: nb.nm_prune_transposable(Wr, o, i, i, "bf16", None, 0, mask, vals, meta, valsT, metaT,
                                                         nb.NM_META_TC) for Wr in Ws]
        else:
            dY = inputs.normal((T, o), 1.0, 2, "bf16", device=dev)
            X = inputs.normal((T, i), 1.0, 3, "bf16", device=dev)
            dW = torch.empty((o, i), dtype=torch.bfloat16, device=dev)
            plan = nb.nm_spmm_plan(nb.make_desc(M=o, N=i, K=T, mode=nb.NM_SPMM_DENSE_MASKED, ab_type="bf16",
                                                cd_type="bf16", order_a=nb.NM_COL, order_b=nb.NM_ROW, order_cd=nb.NM_ROW,
                                                lda=o, ldb=i, ldd=i, meta_layout=nb.NM_META_CANONICAL))
            wsb = nb.nm_spmm_plan_workspace(plan)
            ws = torch.empty(max(16, wsb), dtype=torch.uint8, device=dev)
            fn = [lambda: nb.nm_spmm(plan, 1.0, dY, mask, X, 0.0, None, dW, ws if wsb else None, wsb)]
    elif name in ("prune24_4096", "prune_8of32_4096", "gemv_8of32_b8"):
        M = K = 4096
        n, m = (2, 4) if name == "prune24_4096" else (8, 32)
        layout = nb.NM_META_TC if m == 4 else nb.NM_META_CANONICAL
        Ws = [inputs.normal((M, K), 0.02, 20 + r, "f16", device=dev) for r in range(max(reps, 5))]
        vb, mb = nb.nm_compressed_size(M, K, "f16", n, m, layout)
        vals, meta = (torch.empty(vb, dtype=torch.uint8, device=dev), torch.empty(mb, dtype=torch.uint8, device=dev))
        if name == "gemv_8of32_b8":
            nb.nm_compress(Ws[0], M, K, K, "f16", n, m, 0, layout, vals, meta)
            x = inputs.normal((8, K), 1.0, 4, "f16", device=dev)
            y = torch.empty((8, M), dtype=torch.float16, device=dev)
            plan = nb.nm_spmm_plan(nb.make_desc(M=M, N=8, K=K, n=n, m=m, ab_type="f16", cd_type="f16", ldb=K, ldd=M,
                                                meta_layout=nb.NM_META_CANONICAL))
            fn = [lambda: nb.nm_spmm(plan, 1.0, vals, meta, x, 0.0, None, y)]
        else:
            fn = [lambda Wr=Wr: nb.nm_compress(Wr, M, K, K, "f16", n, m, 0, layout, vals, meta) for Wr in Ws]
    elif name == "check24_4096":
        M = K = 4096
        Ws = [inputs.normal((M, K), 0.02, 40 + r, "f16", device=dev) for r in range(max(reps, 5))]
        cnt = torch.zeros(1, dtype=torch.int32, device=dev)
        fn = [lambda Wr=Wr: nb.nm_check(Wr, M, K, K, "f16", 2, 4, 1, cnt) for Wr in Ws]
    elif name == "vector_wise_4096":
        M = K = 4096
        keep = M * (K // 32) // 4
        Ws = [inputs.normal((M, K), 0.02, 30 + r, "f16", device=dev) for r in range(max(reps, 5))]
        wsb = nb.nm_prune_units_workspace(M, K, 1, 32)
        ws = torch.empty(wsb, dtype=torch.uint8, device=dev)
        csr = torch.empty((M + 1 + keep) * 4, dtype=torch.uint8, device=dev)
        vals = torch.empty(keep * 64, dtype=torch.uint8, device=dev)
        fn = [lambda Wr=Wr: nb.nm_prune_vector_wise(Wr, M, K, K, "f16", 32, keep, nb.NM_SCORE_ABS_OF_SUM, csr=csr,
                                                     vals=vals, workspace=ws, workspace_bytes=wsb) for Wr in Ws]
    else:
        raise SystemExit(f"unknown kernel case {name}; one of {KERNEL_CASES}")
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for r in range(reps):
        fn[r % len(fn)]()
    b.record()
    torch.cuda.synchronize()
    print(json.dumps({"kernel_case": name, "reps": reps, "ms_per_launch": a.elapsed_time(b) / reps}), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("native", "reference"), default="native")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-rows", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-search", action="store_true", help="keep each plan's default kernel (no plan-time search)")
    ap.add_argument("--kernel-case", choices=KERNEL_CASES, help="run one kernel a few times (profiler captures)")
    ap.add_argument("--reps", type=int, default=3)
    args = ap.parse_args(argv)
    if args.kernel_case:
        return run_kernel_case(args.kernel_case, args.reps)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_native(args)


if __name__ == "__main__":
    sys.exit(main())

"""Benchmark of the factorized-linear decode path on one GB300 (or N replicas).

A step is one decode step of the whole path over one batch: remap_compact of
the batch's active rows out of a paged pool, a 32-layer LLaMA-7B-shaped
decomposed stack (q/k/v/o + SiLU-GLU MLP, every projection a rank-r factor
pair at 40 % parameter reduction), and remap_scatter of the results, replayed
as one CUDA graph.  Inputs are seeded synthetic data (7.75 GB of bf16 factors,
far larger than L2, so every step streams them from HBM).

Prints one JSON line.  ``--impl reference`` times the fp64 CPU oracle on a
bounded sample of the same workload instead.
"""

from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

RHO = 0.4
BLOCK_ROWS = 16


class Model:
    """Block dimensions of a decomposed stack (mlp: "swiglu" or the non-GLU "relu")."""

    def __init__(self, name, d, dff, nh, nkv, hd, layers, mlp="swiglu"):
        self.name, self.d, self.dff, self.nh, self.nkv, self.hd, self.layers = name, d, dff, nh, nkv, hd, layers
        self.mlp = mlp


MODELS = {
    "llama7b": Model("llama7b", 4096, 11008, 32, 32, 128, 32),
    "llama70b": Model("llama70b", 8192, 28672, 64, 8, 128, 80),   # GQA, 8 kv heads
    "opt30b": Model("opt30b", 7168, 28672, 56, 56, 128, 48, mlp="relu"),
}
LLAMA7B = MODELS["llama7b"]
LLAMA70B = MODELS["llama70b"]
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def rank_for(d_in, d_out, rho):
    """r = (1 - rho) d_in d_out / (d_in + d_out) rounded to the nearest multiple of 64."""
    from fractions import Fraction
    exact = (1 - Fraction(str(rho))) * d_in * d_out / (d_in + d_out)
    return int(64 * max((exact / 64 + Fraction(1, 2)).__floor__(), 1))


def shapes(rho=RHO, m=LLAMA7B):
    """(d_in, d_out, r) of the 7 projections; None for the gate of a non-GLU MLP."""
    d, dff, dq, dkv = m.d, m.dff, m.nh * m.hd, m.nkv * m.hd
    io = [(d, dq), (d, dkv), (d, dkv), (dq, d), (d, dff), (d, dff), (dff, d)]
    return [None if (p == 4 and m.mlp == "relu") else (a, b, rank_for(a, b, rho))
            for p, (a, b) in enumerate(io)]


def linear_bytes(M, d_in, d_out, r):
    """Algorithmic HBM bytes of one factorized linear: both factors plus x in and y out (bf16)."""
    return 2 * r * (d_in + d_out) + 2 * M * (d_in + d_out)


def step_bytes(M, n_layers, rho=RHO, m=LLAMA7B):
    return n_layers * sum(linear_bytes(M, *sh) for sh in shapes(rho, m) if sh is not None)


def decode_traffic():
    """Per-launch DRAM traffic of the decode kernel from profiles/, or None.

    The profile records a hash of the kernel source it was taken on; a
    changed kernel makes the figure stale, and then None is reported.
    """
    import hashlib
    prof = os.path.join(ROOT, "profiles", "decode_kernel_traffic.txt")
    src = os.path.join(ROOT, "rank_decomposed_gb300", "csrc", "lr_decode.cu")
    if not (os.path.exists(prof) and os.path.exists(src)):
        return None
    kv = {}
    for line in open(prof):
        if "=" in line and not line.startswith("#"):
            k, v = line.strip().split("=", 1)
            kv[k.strip()] = v.strip()
    digest = hashlib.sha256(open(src, "rb").read()).hexdigest()
    if kv.get("source_sha256") != digest:
        return None
    try:
        return float(kv["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        hbm = p.get("hbm_gbs")
        # the prefill leg times a few milliseconds of GEMMs at a time: the burst figure
        tf = p.get("bf16_tflops") or p.get("bf16_tflops_sustained")
        if hbm and tf:
            return float(hbm), float(tf), "measured"
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


# ------------------------------------------------------------------ inputs
def batch(seed, n_seq, cap):
    """Paged decode batch: lengths U{128..4096}, 16-row blocks, last row of each sequence."""
    L, table, total = synth.paged_batch(seed, n_seq, 128, 4096, BLOCK_ROWS)
    order = synth.permutation(seed, synth.make_tag(0, 2, synth.KIND_PERM), n_seq)
    return L[order], table[order], total * BLOCK_ROWS


class Clocks:
    """nvidia-smi sampler run during the timed region."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index, uuid=None):
        # nvidia-smi ignores CUDA_VISIBLE_DEVICES: select the GPU by its UUID
        # when torch reports one, so the samples come from the GPU in use
        self.index = index
        self.select = uuid if uuid else str(index)
        self.proc = None
        # the raw samples go to a temporary file; LR_CLOCKS_CSV keeps them at a chosen path
        self.keep = os.environ.get("LR_CLOCKS_CSV")
        self.path = None

    def start(self):
        try:
            import tempfile
            if self.keep:
                self.path = self.keep
            else:
                fd, self.path = tempfile.mkstemp(prefix="clocks_%d_" % self.index, suffix=".csv")
                os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", self.select, "--query-gpu=" + self.QUERY,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
            if getattr(self, "f", None) is not None:
                self.f.close()
            if self.path and not self.keep and os.path.exists(self.path):
                os.remove(self.path)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        self.proc.terminate()
        self.proc.wait()
        self.f.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not self.keep:
            os.remove(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(smax)),
                "reasons": sorted(reasons), "samples": len(sm), "gpu": self.select}


# -------------------------------------------------------------- our arm
class Workload:
    def __init__(self, torch, lr, M, n_layers, seed=0, rho=RHO, n_seq=None, mode=0, model=LLAMA7B,
                 layers=None):
        self.torch, self.lr = torch, lr
        self.M, self.n_layers, self.rho, self.model = M, n_layers, rho, model
        m = model
        D = m.d
        dev = "cuda"
        self.layers = [] if layers is None else layers
        cs_cache = {}
        for l in range(0 if layers is not None else n_layers):
            fs = []
            for p, sh in enumerate(shapes(rho, m)):
                if sh is None:
                    fs.append(None)
                    continue
                a, b, r = sh
                sa, sg = synth.factor_stds(a, r)
                At = torch.empty((r, a), dtype=torch.bfloat16, device=dev)
                Bt = torch.empty((b, r), dtype=torch.bfloat16, device=dev)
                if r not in cs_cache:
                    cs_cache[r] = torch.from_numpy(synth.sigma_scale(r)).to(dev)
                synth.fill_bf16_normal_device(At.data_ptr(), r, a, seed, synth.make_tag(l, p, synth.KIND_A), sa)
                synth.fill_bf16_normal_device(Bt.data_ptr(), b, r, seed, synth.make_tag(l, p, synth.KIND_B), sg,
                                              cs_cache[r].data_ptr())
                fs.append(lr.FactorPair(At, Bt))
            self.layers.append(lr.Block(m.d, m.dff, m.nh, m.nkv, m.hd, fs,
                                        mlp=lr.MLP_RELU if m.mlp == "relu" else lr.MLP_SWIGLU))
        torch.cuda.synchronize()
        n_seq = M if n_seq is None else n_seq
        self.lengths, self.table, pool_rows = batch(seed, n_seq, M)
        pool = torch.empty((pool_rows, D), dtype=torch.bfloat16, device=dev)
        synth.fill_bf16_normal_device(pool.data_ptr(), pool_rows, D, seed,
                                      synth.make_tag(0, 0, synth.KIND_POOL), 1.0)
        remap, n_active, self.n_runs = lr.remap_build(self.lengths, self.table, BLOCK_ROWS, 1, M)
        self.stack = lr.Stack(
            self.layers, pool, torch.empty_like(pool), torch.from_numpy(remap).to(dev),
            torch.tensor([n_active], dtype=torch.int32, device=dev),
            torch.zeros(M, D, dtype=torch.bfloat16, device=dev),
            torch.zeros(M, D, dtype=torch.float32, device=dev),
            torch.zeros(M, D, dtype=torch.bfloat16, device=dev),
            torch.zeros(lr.Stack.scratch_bytes(M, self.layers, mode), dtype=torch.uint8, device=dev),
            torch.zeros(1, dtype=torch.int32, device=dev), mode=mode)
        self.n_active = n_active

    def free(self):
        self.stack.destroy()
        self.stack = None


def time_graph(torch, stack, steps, warmup, clocks=None, barrier=None):
    for _ in range(warmup):
        stack.replay()
    torch.cuda.synchronize()
    if barrier:
        barrier()
    if clocks:
        clocks.start()
        time.sleep(0.3)
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(s)
    for _ in range(steps):
        stack.replay(s)
    e1.record(s)
    torch.cuda.synchronize()
    ck = clocks.stop() if clocks else None
    if barrier:
        barrier()
    return e0.elapsed_time(e1) / steps, ck


def time_eager(torch, stack, steps, warmup):
    for _ in range(warmup):
        stack.forward()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        stack.forward()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def time_e2e(torch, lr, w, steps, warmup):
    """Host-driven steps through the public API, as a serving loop runs them.

    Every step copies its remap table and n_active from pinned host memory to
    the device, replays the graph and reads the step's output rows back to the
    host; the host then waits for them.  The host remap scan of the next step
    runs while the GPU executes the current one (double-buffered pinned
    tables), which is where a serving loop schedules its next batch.
    """
    st = w.stack
    cap = w.M
    remap_h = [torch.empty(cap, dtype=torch.int32, pin_memory=True) for _ in range(2)]
    nact_h = [torch.empty(1, dtype=torch.int32, pin_memory=True) for _ in range(2)]
    out_h = torch.empty((cap, w.model.d), dtype=torch.bfloat16, pin_memory=True)
    stream = torch.cuda.current_stream()

    def prepare(b):
        remap, n, _ = lr.remap_build(w.lengths, w.table, BLOCK_ROWS, 1, cap)
        remap_h[b].numpy()[:] = remap
        nact_h[b].numpy()[0] = n

    def run(total):
        prepare(0)
        for i in range(total):
            b = i & 1
            st.remap.copy_(remap_h[b], non_blocking=True)
            st.n_active.copy_(nact_h[b], non_blocking=True)
            st.replay()
            out_h.copy_(st.ybuf, non_blocking=True)
            if i + 1 < total:
                prepare(b ^ 1)       # overlaps the GPU work of step i
            stream.synchronize()     # step i's rows are on the host

    run(warmup)
    t0 = time.perf_counter()
    run(steps)
    dt = (time.perf_counter() - t0) / steps
    return dt, remap_h[0].numel() * 4 + 4, out_h.numel() * 2


def time_linears(torch, lr, w, reps=3):
    """Decode GEMM kernel timing over every linear of the stack (down + up launch each).

    Two measurements on the stack's own shapes and factors:
    * chained: all linears' launches back to back in one CUDA graph, as in the
      step (programmatic dependent launch between them), timed with events
      around the graph: the kernel's average launch duration in steady state;
    * isolated: an event pair around every linear, with the stream pre-queued
      behind a fixed-length GPU sleep so no host time is counted; each linear
      then pays its own launch and ramp.
    Returns a dict with bytes, times, launch count and per-projection GB/s.
    """
    M, DFF = w.M, w.model.dff
    x = torch.empty((M, DFF), dtype=torch.bfloat16, device="cuda")
    synth.fill_bf16_normal_device(x.data_ptr(), M, DFF, 1, synth.make_tag(0, 0, synth.KIND_X), 1.0)
    y = torch.empty((M, DFF), dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(max(lr.linear_workspace_bytes(M, f) for f in w.layers[0].factors if f is not None),
                     dtype=torch.uint8, device="cuda")
    calls = [(p, f) for b in w.layers for p, f in enumerate(b.factors) if f is not None]
    n = len(calls)
    nbytes = [linear_bytes(M, f.d_in, f.d_out, f.r) for _, f in calls]
    for p, f in calls[:7]:
        lr.linear_forward(x[:, : f.d_in], f, y[:, : f.d_out], ws, None)
    torch.cuda.synchronize()
    # chained: one graph of all launches
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for p, f in calls:
                lr.linear_forward(x[:, : f.d_in], f, y[:, : f.d_out], ws, None, stream=s)
    g.replay()
    torch.cuda.synchronize()
    chained = None
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        t = e0.elapsed_time(e1) * 1e-3
        chained = t if chained is None else min(chained, t)
    del g
    # isolated: an event pair around every linear
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n + 1)]
    best = None
    for _ in range(reps):
        torch.cuda._sleep(100_000_000)          # ~50 ms of GPU time while the host queues
        for i, (p, f) in enumerate(calls):
            evs[i].record()
            lr.linear_forward(x[:, : f.d_in], f, y[:, : f.d_out], ws, None)
        evs[n].record()
        torch.cuda.synchronize()
        times = [evs[i].elapsed_time(evs[i + 1]) * 1e-3 for i in range(n)]
        if best is None or sum(times) < sum(best):
            best = times
    per_proj = {}
    for (p, f), t, bb in zip(calls, best, nbytes):
        k = synth.PROJ_NAMES[p]
        a, c = per_proj.get(k, (0.0, 0.0))
        per_proj[k] = (a + bb, c + t)
    return {"bytes": float(sum(nbytes)), "chained_s": float(chained), "isolated_s": float(sum(best)),
            "launches": 2 * n,
            "isolated_per_projection_gbs": {k: round(v[0] / v[1] / 1e9, 1) for k, v in per_proj.items()}}


def time_prefill(torch, lr, M=16384, rhos=(0.2, 0.4, 0.6), reps=3, m=LLAMA7B):
    """Prefill: the 7 projections of one layer at M rows, per rank sweep."""
    out = {}
    DFF = m.dff
    x = torch.empty((M, DFF), dtype=torch.bfloat16, device="cuda")
    synth.fill_bf16_normal_device(x.data_ptr(), M, DFF, 2, synth.make_tag(0, 0, synth.KIND_X), 1.0)
    y = torch.empty((M, DFF), dtype=torch.bfloat16, device="cuda")
    for rho in rhos:
        fs = []
        for p, sh in enumerate(shapes(rho, m)):
            if sh is None:
                continue
            a, b, r = sh
            sa, sg = synth.factor_stds(a, r)
            At = torch.empty((r, a), dtype=torch.bfloat16, device="cuda")
            Bt = torch.empty((b, r), dtype=torch.bfloat16, device="cuda")
            cs = torch.from_numpy(synth.sigma_scale(r)).cuda()
            synth.fill_bf16_normal_device(At.data_ptr(), r, a, 3, synth.make_tag(0, p, synth.KIND_A), sa)
            synth.fill_bf16_normal_device(Bt.data_ptr(), b, r, 3, synth.make_tag(0, p, synth.KIND_B), sg, cs.data_ptr())
            fs.append(lr.FactorPair(At, Bt))
        ws = torch.zeros(max(lr.linear_workspace_bytes(M, f) for f in fs), dtype=torch.uint8, device="cuda")
        flops = sum(2.0 * M * f.r * (f.d_in + f.d_out) for f in fs)
        for f in fs:
            lr.linear_forward(x[:, : f.d_in], f, y[:, : f.d_out], ws, None)
        torch.cuda.synchronize()
        best = None
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for f in fs:
                lr.linear_forward(x[:, : f.d_in], f, y[:, : f.d_out], ws, None)
            e1.record()
            torch.cuda.synchronize()
            t = e0.elapsed_time(e1) * 1e-3
            best = t if best is None else min(best, t)
        out[str(rho)] = {"ranks": [f.r for f in fs], "ms_per_layer": round(best * 1e3, 3),
                         "tokens_per_s_%d_layers" % m.layers: round(M / (best * m.layers), 1),
                         "tflops": round(flops / best / 1e12, 1)}
        del fs, ws
        torch.cuda.empty_cache()
    return out


def time_kv_reconstruct(torch, lr, m=LLAMA7B, n_seq=64, reps=5, hbm=None, tf=None):
    """Low-rank KV reconstruction of a whole decode batch's context.

    Every position of 64 sequences (lengths U{128..4096}) is rebuilt from its
    k latent (r columns) by one fixed-size GEMM with B_k, as in the pages'
    graph-replay stage, two ways: row-level (remap_build lists every position,
    remap_compact copies the latents into a [cap, r] buffer, then the GEMM),
    and block-level (remap_build_blocks lists the paged blocks and the GEMM
    reads them straight from the pool: one launch, no buffer).  Reported for
    the model's k projection and for the LLaMA-70B-GQA k shape (576 -> 1024).
    """
    shapes_kv = [("%s_k" % m.name, rank_for(m.d, m.nkv * m.hd, RHO), m.nkv * m.hd)]
    if m.name != "llama70b":
        shapes_kv.append(("llama70b_k", rank_for(LLAMA70B.d, LLAMA70B.nkv * LLAMA70B.hd, RHO),
                          LLAMA70B.nkv * LLAMA70B.hd))
    L, table, pool_rows = batch(7, n_seq, n_seq)
    cap = int(L.sum())
    remap, n, runs = lr.remap_build(L, table, BLOCK_ROWS, 0, cap)
    cap_b = int(sum((int(x) + BLOCK_ROWS - 1) // BLOCK_ROWS for x in L))
    blocks, nb, bruns = lr.remap_build_blocks(L, table, BLOCK_ROWS, cap_b)
    res = {"rows": cap, "blocks": nb, "remap_runs": runs, "block_runs": bruns, "shapes": []}

    def best_of(fn):
        fn()
        torch.cuda.synchronize()
        best = None
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            t = e0.elapsed_time(e1) * 1e-3
            best = t if best is None else min(best, t)
        return best

    for name, r, d_kv in shapes_kv:
        pool = torch.empty((pool_rows, r), dtype=torch.bfloat16, device="cuda")
        synth.fill_bf16_normal_device(pool.data_ptr(), pool_rows, r, 7, synth.make_tag(0, 1, synth.KIND_POOL), 1.0)
        _, sg = synth.factor_stds(m.d, r)
        Bt = torch.empty((d_kv, r), dtype=torch.bfloat16, device="cuda")
        cs = torch.from_numpy(synth.sigma_scale(r)).cuda()
        synth.fill_bf16_normal_device(Bt.data_ptr(), d_kv, r, 7, synth.make_tag(0, synth.PROJ_K, synth.KIND_B), sg,
                                      cs.data_ptr())
        buf = torch.empty((cap, r), dtype=torch.bfloat16, device="cuda")
        out = torch.empty((cap, d_kv), dtype=torch.bfloat16, device="cuda")
        out_b = torch.empty((cap_b * BLOCK_ROWS, d_kv), dtype=torch.bfloat16, device="cuda")
        d_remap = torch.from_numpy(remap).cuda()
        d_n = torch.tensor([n], dtype=torch.int32, device="cuda")
        d_blocks = torch.from_numpy(blocks).cuda()
        d_nb = torch.tensor([nb], dtype=torch.int32, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        t_row = best_of(lambda: lr.kv_reconstruct(pool, d_remap, d_n, buf, Bt, out, st))
        t_blk = best_of(lambda: lr.kv_reconstruct_paged(pool, d_blocks, d_nb, Bt, out_b, st))
        if int(st.item()) != 0:
            raise SystemExit("kv_reconstruct status %d" % int(st.item()))
        rows_b = cap_b * BLOCK_ROWS
        flops = 2.0 * rows_b * r * d_kv
        # algorithmic bytes: the latent rows read once, B_k, the reconstructed rows written
        nbytes_b = 2.0 * rows_b * r + 2.0 * d_kv * r + 2.0 * rows_b * d_kv
        nbytes_r = 2.0 * cap * r * 2 + 2.0 * d_kv * r + 2.0 * cap * d_kv     # + the buffer written and read
        entry = {"shape": name, "r": r, "d_kv": d_kv,
                 "row_level": {"ms": round(t_row * 1e3, 4), "rows_per_s": round(cap / t_row, 1),
                               "gbs": round(nbytes_r / t_row / 1e9, 1)},
                 "paged": {"ms": round(t_blk * 1e3, 4), "rows_per_s": round(cap / t_blk, 1),
                           "gbs": round(nbytes_b / t_blk / 1e9, 1), "tflops": round(flops / t_blk / 1e12, 1),
                           "algorithmic_bytes": nbytes_b, "rows_computed": rows_b}}
        if hbm:
            entry["paged"]["frac_of_hbm"] = round(nbytes_b / t_blk / 1e9 / hbm, 4)
        if tf:
            entry["paged"]["frac_of_bf16_peak"] = round(flops / t_blk / 1e12 / tf, 4)
        res["shapes"].append(entry)
        del pool, Bt, buf, out, out_b
        torch.cuda.empty_cache()
    return res


def rank_sharding(torch, lr, M=64, Gs=(2, 4, 8), rho=RHO, m=None, reps=20):
    """The low-rank communication scheme of the pages, simulated on this GPU.

    Per layer of the LLaMA-70B-shaped stack (the model the pages analyse), the
    collective bytes that the busiest of G processes receives: the rank-space
    all-gather of every down-projection output t, against the all-reduce of
    every full-width output y that a naive split of the two factors needs.
    Then the gate projection run as G simulated processes on this GPU (their
    launches one after another, the all-gather as device copies) against the
    plain two-launch linear.
    """
    m = LLAMA70B if m is None else m
    names = ["q", "k", "v", "o", "gate", "up", "down"]
    sh = shapes(rho, m)
    acct = {}
    for G in Gs:
        tot_r = tot_f = 0
        per = {}
        for name, s_ in zip(names, sh):
            if s_ is None:
                continue
            _, d_out, r = s_
            if 64 * G > min(r, d_out):
                per[name] = None
                continue
            rs, fs = lr.rank_shard_comm_bytes(M, d_out, r, G, 2)
            per[name] = {"rank_space_bytes": rs, "full_space_bytes": fs}
            tot_r += rs
            tot_f += fs
        acct[str(G)] = {"rank_space_bytes": tot_r, "full_space_bytes": tot_f,
                        "reduction": round(1.0 - tot_r / tot_f, 4), "per_linear": per}
    d_in, d_out, r = sh[4]
    sa, sg = synth.factor_stds(d_in, r)
    At = torch.empty((r, d_in), dtype=torch.bfloat16, device="cuda")
    Bt = torch.empty((d_out, r), dtype=torch.bfloat16, device="cuda")
    cs = torch.from_numpy(synth.sigma_scale(r)).cuda()
    synth.fill_bf16_normal_device(At.data_ptr(), r, d_in, 3, synth.make_tag(0, 4, synth.KIND_A), sa)
    synth.fill_bf16_normal_device(Bt.data_ptr(), d_out, r, 3, synth.make_tag(0, 4, synth.KIND_B), sg, cs.data_ptr())
    x = torch.empty((M, d_in), dtype=torch.bfloat16, device="cuda")
    synth.fill_bf16_normal_device(x.data_ptr(), M, d_in, 3, synth.make_tag(0, 0, synth.KIND_X), 1.0)
    f = lr.FactorPair(At, Bt)
    y = torch.empty((M, d_out), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")

    def timeit(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps

    ws = torch.zeros(lr.linear_workspace_bytes(M, f), dtype=torch.uint8, device="cuda")
    plain_ms = timeit(lambda: lr.linear_forward(x, f, y, ws, st))
    sim = {}
    for G in Gs:
        wsg = torch.zeros(lr.rank_sharded_workspace_bytes(M, f, G), dtype=torch.uint8, device="cuda")
        ms = timeit(lambda: lr.linear_forward_rank_sharded(x, f, G, y, wsg, st))
        sim[str(G)] = {"ms_all_processes": round(ms, 4), "ms_per_process": round(ms / G, 4),
                       "gather_copy_bytes": M * r * 2}
    if int(st.item()) != 0:
        raise SystemExit("rank_sharding status %d" % int(st.item()))
    return {"model": m.name, "M": M, "rho": rho, "elem_bytes": 2,
            "collective_bytes_per_layer_busiest_process": acct,
            "simulated_gate": {"shape": [d_in, d_out, r], "plain_ms": round(plain_ms, 4),
                               "sharded": sim,
                               "note": "all G processes run on this one GPU in turn; per-process time is "
                                       "their average, not a multi-GPU measurement"}}


def decode_sweep(torch, lr, model, n_layers, layers, Ms, steps):
    """Graph-replayed step time at each decode batch size, the same factors."""
    out = []
    for M in Ms:
        ww = Workload(torch, lr, M, n_layers, seed=0, model=model, layers=layers)
        ww.stack.capture()
        t, _ = time_graph(torch, ww.stack, steps, 3)
        sb = step_bytes(M, n_layers, m=model)
        out.append({"M": M, "ms_per_step": round(t, 4), "tokens_per_s": round(M / (t * 1e-3), 1),
                    "step_hbm_gbs": round(sb / (t * 1e-3) / 1e9, 1)})
        ww.free()
        del ww
        torch.cuda.empty_cache()
    return out


def prefill_summary(res, model, M, tf):
    """Prefill results with named keys: the rho = 0.4 figures at the top, the sweep as a list."""
    sweep = []
    for rho, v in sorted(res.items()):
        v = dict(v)
        v["rho"] = float(rho)
        v["frac_of_bf16_peak"] = round(v["tflops"] / tf, 4)
        sweep.append(v)
    main = next(v for v in sweep if abs(v["rho"] - 0.4) < 1e-9)
    return {"workload": "%s-shaped projections of one layer (q,k,v,o,gate,up,down), M=%d rows" % (model.name, M),
            "M": M, "rho": 0.4, "tflops": main["tflops"], "frac_of_bf16_peak": main["frac_of_bf16_peak"],
            "ms_per_layer": main["ms_per_layer"],
            "tokens_per_s_all_layers": main["tokens_per_s_%d_layers" % model.layers],
            "peak_tflops": tf,
            "kernel": "prefill_pair_kernel: tcgen05 cta_group::2 256x256 tiles on SM pairs; a linear under "
                      "1.5e12 flops as one launch (down tiles, then up tiles), larger ones as two",
            "timed": "CUDA events around the seven linears back to back, best of the repetitions",
            "sweep": sweep}


def config4(torch, lr, tf, steps):
    """The LLaMA-70B-GQA-shaped stack (80 layers, rho 0.4): decode sweep and one prefill."""
    m = LLAMA70B
    layers = None
    sweep = []
    for M in (1, 16, 64, 256):
        ww = Workload(torch, lr, M, m.layers, seed=0, model=m, layers=layers)
        layers = ww.layers
        ww.stack.capture()
        t, _ = time_graph(torch, ww.stack, steps, 3)
        sb = step_bytes(M, m.layers, m=m)
        sweep.append({"M": M, "ms_per_step": round(t, 4), "tokens_per_s": round(M / (t * 1e-3), 1),
                      "step_hbm_gbs": round(sb / (t * 1e-3) / 1e9, 1)})
        ww.free()
        del ww
        torch.cuda.empty_cache()
    del layers
    torch.cuda.empty_cache()
    pm = 8 * 4096
    pre = prefill_summary(time_prefill(torch, lr, M=pm, m=m, rhos=(0.4,), reps=2), m, pm, tf)
    return {"workload": "LLaMA-70B-GQA-shaped 80-layer stack (d 8192, ffn 28672, 8 kv heads, rho 0.4), "
                        "graph-replayed decode steps; prefill of 8 x 4096 rows through one layer's projections",
            "layers": m.layers, "decode": sweep, "prefill": pre}


def oracle_sample(M, layers_sample, seed=0, rho=RHO, m=LLAMA7B):
    """Time the fp64 oracle on M rows through `layers_sample` layers (factor generation untimed)."""
    import oracle
    D, NH, NKV, HD = m.d, m.nh, m.nkv, m.hd
    L, table, pool_rows = batch(seed, M, M)
    remap, n, _ = oracle.remap_build(L, table, BLOCK_ROWS, 1, M)
    # the active rows of the pool, regenerated element-exactly from their stream offsets
    key = synth.stream_key(seed, synth.make_tag(0, 0, synth.KIND_POOL))
    x = np.stack([synth.f64_to_bf16_bits(synth.normal_f64(key, D, start=int(j) * D)) for j in remap[:n]])
    h = oracle.widen_bf16(x)
    total = 0.0
    for l in range(layers_sample):
        fac = {}
        for p, sh in enumerate(shapes(rho, m)):
            if sh is None:
                fac[synth.PROJ_NAMES[p]] = None
                continue
            At, Bt = synth.factor_pair(seed, l, p, *sh)
            fac[synth.PROJ_NAMES[p]] = oracle.factor_from_stored(At, Bt)
        t0 = time.perf_counter()
        h = oracle.block_forward(h, fac, NH, NKV, HD, mlp=m.mlp)
        total += time.perf_counter() - t0
    return total, n


def gpu_uuid(torch):
    """'GPU-<uuid>' of the current device as nvidia-smi names it, or None."""
    try:
        u = str(torch.cuda.get_device_properties(torch.cuda.current_device()).uuid)
    except Exception:
        return None
    if not u:
        return None
    return u if u.startswith("GPU-") else "GPU-" + u


def cpu_threads():
    try:
        import threadpoolctl
        info = threadpoolctl.threadpool_info()
        n = max((i.get("num_threads", 0) for i in info), default=0)
        if n:
            return int(n)
    except Exception:
        pass
    return os.cpu_count()


def aggregate(dist, ms, tokens):
    """Whole-job step time and tokens over the ranks of a replica run.

    Every rank runs its own batch (no collective on the data path); the job's
    step takes as long as the slowest rank, and the job's tokens are the sum.
    """
    if dist is None:
        return float(ms), float(tokens)
    import torch
    dev = "cuda" if torch.cuda.is_available() and dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(ms)], dtype=torch.float64, device=dev)
    n = torch.tensor([float(tokens)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(n, op=dist.ReduceOp.SUM)
    return float(t.item()), float(n.item())


# ------------------------------------------------------------------ main
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="llama7b", choices=sorted(MODELS))
    ap.add_argument("--M", type=int, default=64)
    ap.add_argument("--layers", type=int, default=0, help="0: the model's layer count")
    ap.add_argument("--no-extras", action="store_true", help="skip the M sweep, eager and prefill legs")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline leg")
    ap.add_argument("--no-config4", action="store_true", help="skip the LLaMA-70B-shaped legs")
    ap.add_argument("--only", choices=["roofline", "prefill", "kv"],
                    help="run one leg alone (for profiling): the event-timed decode linears, or "
                         "the prefill projections at rho=0.4")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    model = MODELS[args.config]
    if args.layers <= 0:
        args.layers = model.layers
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    rk = shapes(RHO, model)
    label = {"llama7b": "LLaMA-7B", "llama70b": "LLaMA-70B (GQA)", "opt30b": "OPT-30B (ReLU MLP)"}[model.name]
    workload = ("%s-shaped %d-layer decomposed stack (rho=0.4; ranks q %d, k/v %d, o %d, mlp %d), "
                "decode M=%d rows compacted by remap from a paged pool, CUDA-graph replay"
                % (label, args.layers, rk[0][2], rk[1][2], rk[3][2], rk[5][2], args.M))

    if args.impl == "reference":
        if rank != 0:
            return
        run_reference(args, workload)
        return

    import torch
    import rank_decomposed_gb300 as lr

    dist = None
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    else:
        torch.cuda.set_device(0)
    barrier = (lambda: dist.barrier()) if dist else None

    if args.only == "kv":
        hbm, tf, _ = load_peaks()
        print(json.dumps({"leg": "kv_reconstruct", "config": model.name,
                          "result": time_kv_reconstruct(torch, lr, m=model, hbm=hbm, tf=tf)}))
        return
    if args.only == "prefill":
        M = 8 * 4096 if model.name == "llama70b" else 16384
        print(json.dumps({"leg": "prefill", "config": model.name, "M": M,
                          "result": time_prefill(torch, lr, M=M, rhos=(0.4,), m=model, reps=2)}))
        return
    w = Workload(torch, lr, args.M, args.layers, seed=rank, model=model)
    if args.only == "roofline":
        r = time_linears(torch, lr, w, reps=1)
        print(json.dumps({"leg": "roofline", "config": model.name, "M": args.M, "layers": args.layers,
                          "launches": r["launches"], "algorithmic_bytes_per_launch": r["bytes"] / r["launches"],
                          "chained_gbs": r["bytes"] / r["chained_s"] / 1e9,
                          "isolated_gbs": r["bytes"] / r["isolated_s"] / 1e9}))
        return
    w.stack.capture()
    clocks = Clocks(torch.cuda.current_device() if world == 1 else local, gpu_uuid(torch))
    ms, ck = time_graph(torch, w.stack, args.steps, args.warmup, clocks, barrier)
    ms, tokens = aggregate(dist, ms, args.M)
    if int(w.stack.status.item()) != 0:
        raise SystemExit("device status %d" % int(w.stack.status.item()))
    # The same graph serves any batch that fits: only the remap contents and
    # n_active change (a real step writes them before each replay).
    n_active_check = {}
    for n in sorted({args.M, max(1, (args.M * 37) // 64), 1}, reverse=True):
        w.stack.n_active.fill_(n)
        t_n, _ = time_graph(torch, w.stack, 5, 3)
        n_active_check[str(n)] = round(t_n, 4)
    w.stack.n_active.fill_(w.n_active)
    torch.cuda.synchronize()
    if int(w.stack.status.item()) != 0:
        raise SystemExit("device status %d after n_active replays" % int(w.stack.status.item()))
    value = tokens / (ms * 1e-3)
    launches = w.stack.launch_count() * args.steps

    hbm, tf, peak_kind = load_peaks()
    line = {
        "metric": "factorized-linear tokens/s (decode)",
        "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": workload, "model": "%s-shaped factorized stack (random factors)" % model.name,
                   "global_batch": int(tokens), "seq_len": 1, "rows_per_gpu": args.M,
                   "layers": args.layers, "rho": RHO, "parallelism": "replicas" if world > 1 else "single",
                   "l2": "inputs larger than L2: %.2f GB of factors and activations streamed per step" % (step_bytes(args.M, args.layers, m=model) / 1e9),
                   "remap_runs": w.n_runs},
        "clocks": ck, "gpu_launches": launches, "graph_ms_by_n_active": n_active_check,
        "step_hbm_gbs": round(step_bytes(args.M, args.layers, m=model) / (ms * 1e-3) / 1e9, 1),
    }
    if rank == 0:
        e2e_s, bi, bo = time_e2e(torch, lr, w, max(5, args.steps // 2), 3)
        line["e2e"] = {"value": round(tokens / e2e_s, 1), "unit": "tokens/s",
                       "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
                       "ms_per_step": round(e2e_s * 1e3, 4),
                       "path": "per step: pinned H2D of remap/n_active, graph replay, D2H of the step's rows, host wait; the host remap_build of the next step overlaps the GPU work"}
        # Roofline of the step as it runs: the graph's own launches, timed by
        # the CUDA events of the timed region above.  The algorithmic bytes are
        # the factors plus every linear's x in and y out; the glue kernels'
        # time is included, so this is a lower bound for the GEMM kernel alone.
        per_step = w.stack.launch_count()
        sb = step_bytes(args.M, args.layers, m=model)
        achieved = sb / (ms * 1e-3) / 1e9
        # DRAM bytes of the decode kernel per step: the profiled per-launch traffic
        # of the per-linear launches (7 projections x down/up, 2 layers) times the
        # 14 such launches of every layer; the step's grouped launches move the
        # same bytes.  Glue kernels are not counted.
        per_launch = decode_traffic() if model.name == "llama7b" and args.M == 64 else None
        traffic = None if per_launch is None else round(per_launch * 14 * args.layers)
        line["roofline"] = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                            "frac": round(achieved / hbm, 4), "traffic": traffic, "peak_source": peak_kind,
                            "traffic_note": "per step: DRAM read+write bytes of the decode kernel (ncu, "
                                            "profiles/decode_kernel_traffic.txt) scaled from 2 layers; null "
                                            "when the kernel source changed since the capture",
                            "kernel": "decode_kernel (tcgen05 swap-AB down/up projections) with the step's "
                                      "glue kernels, as replayed in the step's CUDA graph",
                            "timed": "CUDA events around the timed replays on the replay stream",
                            "launches_timed": per_step * args.steps,
                            "avg_launch_us": round(ms * 1e3 / per_step, 3),
                            "algorithmic_bytes_per_step": sb,
                            "algorithmic_bytes_per_launch": round(sb / per_step)}
        if not args.no_extras:
            r = time_linears(torch, lr, w)
            line["roofline"]["isolated_linears"] = {
                "achieved": round(r["bytes"] / r["isolated_s"] / 1e9, 1),
                "avg_launch_us": round(r["isolated_s"] / r["launches"] * 1e6, 2),
                "note": "each linear of the stack (down + up launch) timed alone with an event pair",
                "per_projection_gbs": r["isolated_per_projection_gbs"]}
            # the analogue of the pages' CUDA-graph ablation: the same step
            # replayed as a graph and enqueued eagerly
            eager_ms = time_eager(torch, w.stack, 5, 3)
            cmp = {"graph_ms": round(ms, 4), "eager_ms": round(eager_ms, 4),
                   "launches_per_step": w.stack.launch_count()}
            line["graph_vs_eager"] = cmp
        layers = w.layers
        w.free()
        del w
        torch.cuda.empty_cache()
        if not args.no_extras:
            line["decode_sweep"] = decode_sweep(torch, lr, model, args.layers, layers,
                                                (1, 8, 32, 64) if model.name != "llama70b" else (1, 16, 64, 256),
                                                max(10, args.steps // 2))
            del layers
            torch.cuda.empty_cache()
            pm = 8 * 4096 if model.name == "llama70b" else 16384
            line["prefill"] = prefill_summary(time_prefill(torch, lr, M=pm, m=model,
                                                           rhos=(0.2, 0.4, 0.6) if model.name == "llama7b" else (0.4,)),
                                              model, pm, tf)
            line["kv_reconstruct"] = time_kv_reconstruct(torch, lr, m=model, hbm=hbm, tf=tf)
            line["rank_sharding"] = rank_sharding(torch, lr)
            if model.name == "llama7b" and not args.no_config4:
                line["config4"] = config4(torch, lr, tf, max(10, args.steps // 2))
        else:
            del layers
        if not args.no_cpu:
            sample_layers = oracle_sample_layers(args.layers)
            tcpu, n = oracle_sample(args.M, sample_layers, m=model)
            v = n / (tcpu * args.layers / sample_layers)
            line["cpu_baseline"] = {"value": round(v, 3), "unit": "tokens/s", "cores": cpu_threads(),
                                    "kind": "oracle",
                                    "sample": "fp64 oracle over the same %d rows through %d of %d layers (%.1f s)%s"
                                              % (n, sample_layers, args.layers, tcpu,
                                                 "" if sample_layers == args.layers
                                                 else ", scaled linearly to the full stack")}
        print(json.dumps(line), flush=True)
    if dist:
        dist.barrier()
        dist.destroy_process_group()


def oracle_sample_layers(n_layers):
    """Layers of the stack the oracle runs per timed sample (the same in both arms).

    The whole stack when it has at most 32 layers (the 7B and OPT shapes'
    step, about a second on 16 cores); otherwise 8 layers, whose time is
    scaled to the full stack (rows are independent and every layer has the
    same shapes, so the time is linear in the layer count).
    """
    return n_layers if n_layers <= 32 else 8


def run_reference(args, workload):
    """The oracle as it stands, on the host cores: each step is the oracle on M rows
    through oracle_sample_layers(L) layers of the stack."""
    import oracle  # noqa: F401
    model = MODELS[args.config]
    ls = oracle_sample_layers(args.layers)
    for _ in range(args.warmup):
        oracle_sample(args.M, ls, m=model)
    tot, n = 0.0, 0
    for _ in range(args.steps):
        t, n = oracle_sample(args.M, ls, m=model)
        tot += t
    per_step = tot / args.steps                       # measured: what each step ran
    full = per_step * args.layers / ls                # the whole stack (= per_step when ls == layers)
    value = n / full
    sample = ("each step: the fp64 oracle on %d rows through %d of %d layers" % (n, ls, args.layers)
              + ("" if ls == args.layers else ", time scaled linearly to the full stack"))
    line = {"impl": "reference", "metric": "factorized-linear tokens/s (decode)", "value": round(value, 3),
            "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(per_step * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload, "rows": n, "layers": args.layers, "layers_per_step": ls,
                       "rho": RHO},
            "cpu_baseline": {"value": round(value, 3), "unit": "tokens/s", "cores": cpu_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": round(value, 3), "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    if ls != args.layers:
        line["ms_full_stack_extrapolated"] = round(full * 1e3, 3)
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()

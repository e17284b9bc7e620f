"""Throughput of the MultiTowerDIN sparse forward (EmbeddingBag pooling +
padding-free DIN target attention) on synthetic Taobao-shaped batches.

One step = one din_sparse_fwd call (KJT offsets, pooled gather over 16 tables,
query, jagged sequence gather, attention MLP on tensor cores, masked softmax,
weighted sum) over one batch of B=8192 samples already resident in HBM.
Between timed steps L2 is flushed by writing a buffer larger than L2; each
step is timed by its own pair of CUDA events, so the flush is not counted.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

N>1 runs independent replicas, one per rank (launched by torch.distributed.run);
the path has no cross-sample exchange, so there is no collective in a step.
The reference arm (--impl reference) is the CPU oracle, timed on the host
cores on a bounded sample of the same workload.

The K timed steps run inside a window of about a second of identical steps,
over which the SM clocks are sampled; the line reports the K-step mean (the
headline), the per-step median and spread, and the window's statistics.

Side legs, reported under their own keys of the same JSON line: the forward
on every workload at full size (configs: tiny, taobao, long_multihot,
gather_stress, wide_bf16, each with its roofline), the forward over a stream
of distinct batches without L2 flushes, the pooling stage alone (taobao, and
the B=65536 gather-stress workload), the forward over hashed tables, the
dense towers and one training step; and on the host, the oracle on all cores
(cpu_baseline), on one core, and the padded flow on one core.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "taobao"
METRIC = "samples/sec for sparse fwd (EmbBag+jagged DIN) at B=8192; % of HBM/tensor roofline"
UNIT = "samples/s"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
L2_FLUSH_BYTES = 512 << 20
E2E_GRAPH = 20    # pipelined end-to-end steps per captured graph
CLOCK_WINDOW_S = 1.2  # steps run around the timed ones while the clocks are sampled
KERNEL_SOURCES = ["fwd_kernel.cuh", "ptx.cuh", "hash.cuh", "launch.cuh", "fwd_attn_tc.cu"]


def workload_desc(B):
    return ("taobao-shaped MultiTowerDIN sparse fwd: B=%d, 16 fp32 dim-16 tables "
            "(201 MB, page-1 bucket sizes), Zipf(1.1) ids, 1 id/feature, seq len geometric "
            "mean 5 cap 100, attn MLP 192-256-64-1 bf16 tensor cores" % B)


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x, ws, device=None):
    """The largest of every rank's x (a float), through torch.distributed's
    MAX all-reduce on whatever backend the group uses; x itself when ws == 1."""
    if ws == 1:
        return float(x)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_rate(units_per_rank, slowest_ms, ws):
    """Whole-job throughput of ws replicas that each processed units_per_rank
    units, over the slowest rank's time."""
    return units_per_rank * ws / (slowest_ms / 1e3)


def peaks():
    """Measured HBM GB/s and bf16 TFLOP/s (burst, sustained) or the fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            flat = {}

            def walk(x, pre=""):
                if isinstance(x, dict):
                    for k, v in x.items():
                        walk(v, pre + k.lower() + ".")
                elif isinstance(x, (int, float)):
                    flat[pre[:-1]] = float(x)
            walk(d)
            hbm = next((v for k, v in flat.items() if "hbm" in k and "gb" in k), None)
            tfs = next((v for k, v in flat.items() if "bf16" in k and "tflop" in k
                        and "sustain" not in k), None)
            tfs_s = next((v for k, v in flat.items() if "bf16" in k and "sustain" in k), None)
            if hbm and tfs:
                return hbm, tfs, tfs_s or tfs, "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


def step_stats(us):
    """Per-step times (us): mean, median and spread."""
    a = np.asarray(us, dtype=np.float64)
    if a.size == 0:
        return None
    return {"mean": float(a.mean()), "median": float(np.median(a)), "p10": float(np.percentile(a, 10)),
            "p90": float(np.percentile(a, 90)), "min": float(a.min()), "max": float(a.max()), "n": int(a.size)}


def time_flushed(run, flush, steps, stream):
    """Per-step us of run() on stream, each step bracketed by its own pair of
    CUDA events, with L2 flushed (a 512 MB write) before each step, outside
    the events."""
    import torch
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    with torch.cuda.stream(stream):
        for i in range(steps):
            flush.fill_(float(i & 7))
            ev[i][0].record(stream)
            run()
            ev[i][1].record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(b) * 1e3 for a, b in ev]


def roofline(nbytes, flops, us):
    """HBM and tensor fractions of one launch of a kernel timed alone (the
    burst tensor peak), the binding one first."""
    hbm, tfs, _, src = peaks()
    t = us * 1e-6
    ach_gbs, ach_tfs = nbytes / t / 1e9, flops / t / 1e12
    t_hbm, t_tc = nbytes / (hbm * 1e9), flops / (tfs * 1e12)
    bound = "hbm" if t_hbm >= t_tc else "tensor"
    return {"bound": bound, "achieved": ach_gbs if bound == "hbm" else ach_tfs,
            "peak": hbm if bound == "hbm" else tfs, "unit": "GB/s" if bound == "hbm" else "TFLOP/s",
            "frac": ach_gbs / hbm if bound == "hbm" else ach_tfs / tfs,
            "hbm_frac": ach_gbs / hbm, "tensor_achieved_tflops": ach_tfs, "tensor_frac": ach_tfs / tfs,
            "combined_frac": max(t_hbm, t_tc) / t, "algorithmic_bytes_per_launch": nbytes,
            "flops_per_launch": flops, "peak_source": src, "tensor_peak_kind": "burst (kernel timed alone)"}


def pool_bytes(batch):
    """Algorithmic bytes of the pooling stage alone (rows a1-a2): 8 B per id +
    4 B per bag length + one table row per id + the pooled output row."""
    es = 2 if batch.wl.dtype == "bf16" else 4
    n_ids = int(batch.values.size)
    return 8 * n_ids + 4 * batch.F * batch.B + batch.D * es * n_ids + 4 * batch.F * batch.D * batch.B


def time_pool_only(binding, db, wsp, flush, steps, batch, ws, workload="taobao B=8192", also_unflushed=False):
    """emb_bag_pool alone (the KJT offsets scan and the pooled gather), graph
    replays with L2 flushed between steps, against the HBM peak; with
    also_unflushed, the same steps back to back without the flush as well (for
    a workload whose tables are far larger than L2)."""
    import torch
    B, F, D = db.B, db.F, db.D
    pooled = torch.empty(B, F * D, device=flush.device)
    status = torch.zeros(1, dtype=torch.int32, device=flush.device)
    stream = torch.cuda.Stream(device=flush.device)

    def step():
        binding.emb_bag_pool(db.tables, db.values, db.lengths, B, pooled, wsp, status=status, stream=stream)
    with torch.cuda.stream(stream):
        for _ in range(5):
            step()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step()
    stream.synchronize()
    per = time_flushed(g.replay, flush, steps, stream)
    per_nf = None
    if also_unflushed:
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
        with torch.cuda.stream(stream):
            for a, b in ev:
                a.record(stream)
                g.replay()
                b.record(stream)
        torch.cuda.synchronize()
        per_nf = [a.elapsed_time(b) * 1e3 for a, b in ev]
    if int(status.item()):
        raise RuntimeError("pool-only status 0x%x" % int(status.item()))
    total_ms = max_over_ranks(sum(per) / 1e3, ws, flush.device)
    us = total_ms * 1e3 / steps
    nbytes = pool_bytes(batch)
    hbm, _, _, src = peaks()
    ach = nbytes / (us * 1e-6) / 1e9
    out = {"what": "emb_bag_pool: KJT offsets and the pooled gather of all 16 tables (rows a1-a2)",
            "workload": workload, "us_per_step": us, "us_stats": step_stats(per),
            "samples_per_s": weak_rate(B * steps, total_ms, ws),
            "roofline": {"bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s", "frac": ach / hbm,
                         "algorithmic_bytes_per_launch": nbytes, "peak_source": src}}
    if per_nf is not None:
        st = step_stats(per_nf)
        a_nf = nbytes / (st["mean"] * 1e-6) / 1e9
        out["unflushed"] = {"what": "the same launches back to back, L2 not flushed: the tables (%.2f GB) "
                                    "are far larger than L2, ids uniform" % (sum(int(t.numel()) * t.element_size()
                                                                                for t in db.tables.tables) / 1e9),
                            "us_stats": st, "roofline": {"bound": "hbm", "achieved": a_nf, "peak": hbm,
                                                         "unit": "GB/s", "frac": a_nf / hbm}}
    return out


def time_steady_state(binding, synth, db, mlp, wsp, status, dev, n_batches, reps):
    """din_sparse_fwd over a stream of n_batches distinct batches (the same
    tables; ids, bag and sequence lengths drawn with other seeds), replayed back
    to back without an L2 flush. The tables (201 MB) are larger than L2 and each
    step reads another batch, so between steps L2 keeps only what the batches
    share: the Zipf-hot rows, as a stream of real batches would."""
    import torch
    B = db.B
    kb = []
    for i in range(n_batches):
        b = synth.generate(WORKLOAD, seed=1000 + i, ids_only=True)
        kb.append([torch.from_numpy(np.ascontiguousarray(x, dt)).to(dev)
                   for x, dt in ((b.values, np.int64), (b.lengths, np.int32),
                                 (b.seq_values, np.int64), (b.seq_lengths, np.int32))])
    pooled = torch.empty(B, db.F * db.D, device=dev)
    din = torch.empty(B, 3 * db.D, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def run_all():
        for v, ln, sv, sl in kb:
            binding.din_sparse_fwd(db.tables, v, ln, sv, sl, db.max_len, db.q_feat, db.seq_table, B, mlp,
                                   pooled, din, wsp, status=status, stream=stream)
    with torch.cuda.stream(stream):
        for _ in range(2):
            run_all()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            run_all()
        g.replay()
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
    if int(status.item()):
        raise RuntimeError("steady-state status 0x%x" % int(status.item()))
    us = e0.elapsed_time(e1) * 1e3 / (reps * n_batches)
    return {"what": "din_sparse_fwd over %d distinct batches (same tables), back to back, no L2 flush "
                    "(tables 201 MB > 129 MB L2)" % n_batches,
            "us_per_step": us, "samples_per_s": B / (us * 1e-6), "steps_timed": reps * n_batches}


def algorithmic_work(batch):
    """Bytes and FLOPs the method must move / do for one batch (fp32 D=16):
    deep: 8 B per id + 4 B per bag length + 64 B per row + 1024 B output row;
    DIN: 24 B of ids + 192 B of rows per valid position, 4 B length, 192 B output;
    MLP: 2*(192*256 + 256*64 + 64) FLOPs per valid position. Padded positions
    the method avoids are not counted; MLP weights (131 KB) are not counted."""
    D = batch.D
    es = 2 if batch.wl.dtype == "bf16" else 4
    n_ids = int(batch.values.size)
    F, B = batch.F, batch.B
    L = np.minimum(np.maximum(batch.seq_lengths, 0), batch.max_len).astype(np.int64)
    P = int(L.sum())
    deep = 8 * n_ids + 4 * F * B + D * es * n_ids + 4 * F * D * B
    din = 24 * P + 3 * D * es * P + 4 * B + 4 * 3 * D * B
    K1 = 12 * D
    flops = 2 * (K1 * 256 + 256 * 64 + 64) * P
    return deep + din, flops, P


CONFIG_STEPS = {"tiny": 400, "long_multihot": 200, "gather_stress": 20, "wide_bf16": 60}


def time_configs(binding, synth, dev, mode, flush, scale, headline):
    """din_sparse_fwd, captured in a CUDA graph, on every workload at its full
    size (taobao: the headline's figures): per-step times with L2 flushed
    between steps, and each one's roofline from its algorithmic bytes and
    FLOPs."""
    import torch
    from recsys_sparse_embedding_gb300.device_batch import to_device
    out = {}
    for name in synth.WORKLOAD_ORDER:
        if name == WORKLOAD:
            out[name] = headline
            continue
        b = synth.generate(name, seed=0)
        db = to_device(b, dev)
        B, D, F = db.B, db.D, db.F
        mlp = db.mlp(mode)
        wsp = binding.Workspace(B, D, device=dev)
        wsp.prepare(mlp)
        pooled = torch.empty(B, F * D, device=dev)
        din = torch.empty(B, 3 * D, device=dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)
        stream = torch.cuda.Stream(device=dev)

        def step():
            binding.din_sparse_fwd(db.tables, db.values, db.lengths, db.seq_values, db.seq_lengths,
                                   db.max_len, db.q_feat, db.seq_table, B, mlp, pooled, din, wsp,
                                   status=status, stream=stream)
        with torch.cuda.stream(stream):
            for _ in range(3):
                step()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                step()
        stream.synchronize()
        us = time_flushed(g.replay, flush, max(3, int(CONFIG_STEPS[name] * scale)), stream)
        st = int(status.item())
        if st & ~binding.FLAG_SEQ_TRUNC:
            raise RuntimeError("%s: status 0x%x" % (name, st))
        nbytes, flops, P = algorithmic_work(b)
        stats = step_stats(us)
        out[name] = {"B": B, "D": D, "dtype": b.wl.dtype, "valid_positions": P, "us_per_step": stats,
                     "samples_per_s": B / (stats["mean"] * 1e-6),
                     "roofline": roofline(nbytes, flops, stats["mean"])}
        del g, db, wsp, pooled, din, b
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    return out


def hashed_lookups(batch):
    """Lookups served by the hash table in one batch: the deep ids of the
    hashed features and the sequence ids of hashed sub-features."""
    hk = getattr(batch, "hash_keys", None) or {}
    F, B = batch.F, batch.B
    lengths = np.maximum(np.asarray(batch.lengths).reshape(F, B), 0)
    L = np.minimum(np.maximum(batch.seq_lengths, 0), batch.max_len).astype(np.int64)
    n = int(sum(int(lengths[f].sum()) for f in hk))
    n += int(L.sum()) * sum(1 for t in batch.seq_table if t in hk)
    return n


def traffic_record():
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    try:
        rec = json.load(open(path))
        if rec.get("kernel_hash") != kernel_hash():
            return None
        return float(rec["dram_bytes_per_launch"])
    except Exception:
        return None


def kernel_hash():
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "recsys_sparse_embedding_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        self.t0 = time.perf_counter()
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.seconds = time.perf_counter() - self.t0
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in getattr(self, "lines", []):
            parts = [x.strip() for x in l.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def time_dynamic_emb(binding, synth, batch, dev, mode, flush, steps, ws):
    """The same step with the five large tables served by one hash table
    (300K admitted keys each, the Zipf-hot ids; colder ids unseen): graph
    replays, L2 flushed between steps, CUDA events on the launching stream,
    max over ranks. Algorithmic bytes add one 64-byte bucket per hashed
    lookup to the plain step's."""
    import torch
    from recsys_sparse_embedding_gb300.device_batch import to_device
    hb = synth.dynamic_emb(batch, seed=0)
    db = to_device(hb, dev)
    B, D, F = db.B, db.D, db.F
    mlp = db.mlp(mode)
    wsp = binding.Workspace(B, D, device=dev)
    wsp.prepare(mlp)
    pooled = torch.empty(B, F * D, device=dev)
    din = torch.empty(B, 3 * D, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def step():
        binding.din_sparse_fwd(db.tables, db.values, db.lengths, db.seq_values, db.seq_lengths,
                               db.max_len, db.q_feat, db.seq_table, B, mlp, pooled, din, wsp,
                               status=status, stream=stream)
    with torch.cuda.stream(stream):
        for _ in range(5):
            step()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            step()
    stream.synchronize()
    per = time_flushed(g.replay, flush, steps, stream)
    if int(status.item()):
        raise RuntimeError("hashed step status 0x%x" % int(status.item()))
    total_ms = max_over_ranks(sum(per) / 1e3, ws, dev)
    us = total_ms * 1e3 / steps
    nbytes, flops, _ = algorithmic_work(hb)
    nh = hashed_lookups(hb)
    nbytes += 64 * nh
    hbm, _, _, src = peaks()
    ht = db.tables.hash
    return {"what": "din_sparse_fwd with user_id, adgroup_id, campaign_id, brand, customer in one "
                    "hash table (raw 56-bit keys, 300K admitted per table, unseen keys read zero)",
            "us_per_step": us, "us_stats": step_stats(per), "samples_per_s": weak_rate(B * steps, total_ms, ws),
            "hashed_lookups_per_step": nh, "hash_workspace_bytes": ht.nbytes,
            "hash_capacity": int(ht.c.capacity),
            "roofline": {"bound": "hbm", "achieved": nbytes / (us * 1e-6) / 1e9, "peak": hbm,
                         "unit": "GB/s", "frac": nbytes / (us * 1e-6) / 1e9 / hbm,
                         "algorithmic_bytes_per_launch": nbytes, "peak_source": src}}


BWD_FLOPS_PER_POSITION_D16 = 2 * (192 * 256 + 256 * 64 + 64 * 256 + 256 * 192 + 256 * 192 + 64 * 256)


def time_train_step(binding, db, mlp, wsp, pooled, din, status, flush, steps, batch):
    """One training step of the sparse path per iteration: din_sparse_fwd,
    din_sparse_bwd on fixed synthetic upstream gradients, and sparse AdaGrad
    (lr 1e-3) on the touched rows; L2 flushed between steps, CUDA events on
    the launching stream around each part. The tables are updated in place
    (a copy of the batch's tables, so the forward leg above is unaffected)."""
    import torch
    dev = pooled.device
    B, F, D = db.B, db.F, db.D
    tabs = binding.EmbeddingTables([t.clone() for t in db.tables.tables], db.tables.pooling, db.tables.hash)
    n_seq = int(db.seq_values.shape[-1])
    grads = binding.MlpGrads(D, device=dev)
    state = binding.SparseState(tabs, int(db.values.numel()) + 3 * n_seq, device=dev)
    bws = binding.BwdWorkspace(B, int(db.values.numel()), n_seq, D, device=dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(0)
    dpooled = torch.randn(B, F * D, device=dev, generator=gen)
    ddin = torch.randn(B, 3 * D, device=dev, generator=gen)
    stream = torch.cuda.Stream(device=dev)

    def fwd():
        binding.din_sparse_fwd(tabs, db.values, db.lengths, db.seq_values, db.seq_lengths, db.max_len, db.q_feat,
                               db.seq_table, B, mlp, pooled, din, wsp, status=status, stream=stream)

    def bwd():
        binding.din_sparse_bwd(tabs, db.values, db.lengths, db.seq_values, db.seq_lengths, db.max_len, db.q_feat,
                               db.seq_table, B, mlp, pooled, dpooled, ddin, grads, state, bws, status=status,
                               stream=stream)

    def upd():
        binding.emb_adagrad_update(tabs, state, 1e-3, 1e-10, status=status, stream=stream)
    with torch.cuda.stream(stream):
        for _ in range(3):
            fwd(); bwd(); upd()
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
        stream.synchronize()
        for i in range(steps):
            flush.fill_(float(i & 7))
            e = ev[i]
            e[0].record(stream); fwd(); e[1].record(stream); bwd(); e[2].record(stream); upd(); e[3].record(stream)
        torch.cuda.synchronize()
    if int(status.item()):
        raise RuntimeError("train step status 0x%x" % int(status.item()))
    f_l = [e[0].elapsed_time(e[1]) * 1e3 for e in ev]
    b_l = [e[1].elapsed_time(e[2]) * 1e3 for e in ev]
    u_l = [e[2].elapsed_time(e[3]) * 1e3 for e in ev]
    f_us, b_us, u_us = (sum(x) / steps for x in (f_l, b_l, u_l))
    step_us = f_us + b_us + u_us
    _, _, P = algorithmic_work(batch)
    flops = BWD_FLOPS_PER_POSITION_D16 * P if D == 16 else None
    _, tfs, _, src = peaks()
    out = {"what": "din_sparse_fwd + din_sparse_bwd (upstream gradients dpooled, ddin) + emb_adagrad_update",
           "us_per_step": step_us, "fwd_us": f_us, "bwd_us": b_us, "adagrad_us": u_us,
           "fwd_stats": step_stats(f_l), "bwd_stats": step_stats(b_l), "adagrad_stats": step_stats(u_l),
           "samples_per_s": B / (step_us * 1e-6)}
    if flops:
        ach = flops / (b_us * 1e-6) / 1e12
        out["bwd_roofline"] = {"bound": "tensor", "achieved": ach, "peak": tfs, "unit": "TFLOP/s",
                               "frac": ach / tfs, "flops_per_launch": flops, "peak_source": src,
                               "note": "the six MLP GEMMs of the backward over the valid positions"}
    return out


TOWER_FLOPS_PER_SAMPLE = 2 * (256 * 512 + 512 * 256 + 256 * 128 + 176 * 64)


def time_towers(binding, synth, pooled, din, B, dev, flush, steps):
    """The dense towers (deep 256-512-256-128, final cat[deep, din] 176-64-1)
    on the timed step's own outputs: one ctr_towers_fwd launch per step, L2
    flushed between steps, CUDA events on the launching stream. Reported beside
    the sparse forward, not inside its timed step."""
    import torch
    tw = binding.Towers([torch.from_numpy(w) for w in synth.tower_weights(0)], device=dev)
    stream = torch.cuda.Stream(device=dev)
    logit = torch.empty(B, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    with torch.cuda.stream(stream):
        tw.prepare(stream)
        for _ in range(5):
            binding.ctr_towers_fwd(pooled, din, B, tw, logit, status=st, stream=stream)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(steps)]
        stream.synchronize()
        for i in range(steps):
            flush.fill_(float(i & 7))
            ev[i][0].record(stream)
            binding.ctr_towers_fwd(pooled, din, B, tw, logit, status=st, stream=stream)
            ev[i][1].record(stream)
        torch.cuda.synchronize()
    if int(st.item()):
        raise RuntimeError("towers status 0x%x" % int(st.item()))
    us = sorted(a.elapsed_time(b) * 1e3 for a, b in ev)
    mean_us = sum(us) / len(us)
    flops = TOWER_FLOPS_PER_SAMPLE * B
    _, tfs, _, src = peaks()
    ach = flops / (mean_us * 1e-6) / 1e12
    return {"what": "ctr_towers_fwd on this step's pooled [B,256] and din [B,48] -> logit [B]",
            "B": B, "launches": steps, "us_per_launch": mean_us, "us_median": us[len(us) // 2],
            "samples_per_s": B / (mean_us * 1e-6),
            "roofline": {"bound": "tensor", "achieved": ach, "peak": tfs, "unit": "TFLOP/s",
                         "frac": ach / tfs, "flops_per_launch": flops, "peak_source": src,
                         "peak_kind": "burst (kernel timed alone)"}}


def cpu_oracle_rate(batch, samples_per_pass, passes, threads):
    """The oracle as it stands, split over host threads by sample chunks."""
    import concurrent.futures as cf
    import oracle
    chunks = np.array_split(np.arange(samples_per_pass, dtype=np.int32) % batch.B, threads)
    oracle.lib()

    def work(ch):
        if ch.size:
            oracle.pool_batch(batch, ch)
            oracle.din_batch(batch, ch)
    t0, c0 = time.perf_counter(), time.process_time()
    with cf.ThreadPoolExecutor(max_workers=threads) as ex:
        for _ in range(passes):
            list(ex.map(work, chunks))
    dt = time.perf_counter() - t0
    cpu_s = time.process_time() - c0  # all threads of this process
    return samples_per_pass * passes / dt, dt, cpu_s


def cpu_oracle_rate_padded(batch, samples_per_pass, passes):
    """The pages' padded flow as the oracle states it (every sequence padded
    to max_len, the MLP run on every padded position, masked before the
    softmax), single-threaded."""
    import oracle
    samples = np.arange(samples_per_pass, dtype=np.int32) % batch.B
    oracle.lib()
    t0 = time.perf_counter()
    for _ in range(passes):
        oracle.pool_batch(batch, samples)
        oracle.din_batch(batch, samples, padded=True)
    dt = time.perf_counter() - t0
    return samples_per_pass * passes / dt, dt


def cpu_baselines(synth, batch, single_samples, padded_samples):
    """The oracle on one host thread, and the padded flow on one thread for
    the tiny and taobao workloads."""
    rate1, dt1, _ = cpu_oracle_rate(batch, single_samples, 1, 1)
    out = {"oracle_1thread": {"value": rate1, "unit": UNIT, "cores": 1, "kind": "oracle",
                              "sample": "%d samples of the B=%d batch (%.1f s)" % (single_samples, batch.B, dt1)},
           "padded_flow_1thread": {}}
    for name, n in (("tiny", 64 * 8), (WORKLOAD, padded_samples)):
        b = batch if name == WORKLOAD else synth.generate(name, seed=0)
        per = min(n, b.B)
        rate, dt = cpu_oracle_rate_padded(b, per, max(1, n // per))
        out["padded_flow_1thread"][name] = {
            "value": rate, "unit": UNIT, "cores": 1, "kind": "oracle, padded flow",
            "sample": "%d samples of the B=%d batch, sequences padded to %d (%.1f s)"
                      % (per * max(1, n // per), b.B, b.max_len, dt)}
    return out


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    from recsys_sparse_embedding_gb300 import synth
    batch = synth.generate(WORKLOAD, seed=0)
    threads = os.cpu_count() or 1
    per_step = 1024
    for _ in range(args.warmup):
        cpu_oracle_rate(batch, 64, 1, threads)
    rate, dt, cpu_s = cpu_oracle_rate(batch, per_step, args.steps, threads)
    line = {
        "impl": "reference", "metric": METRIC, "value": rate, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": workload_desc(batch.B), "B": batch.B,
                   "reference": "CPU oracle (plain C, fp64 attention), %d host threads" % threads},
        "cpu_baseline": {"value": rate, "unit": UNIT, "cores": threads, "kind": "oracle",
                         "sample": "%d samples of the B=%d batch per step; %d steps took %.1f s wall, "
                                   "%.1f s of CPU time" % (per_step, batch.B, args.steps, dt, cpu_s)},
        "e2e": {"value": rate, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--mode", default="bf16", choices=["bf16", "fp32"])
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--cpu-sample", type=int, default=8192)
    ap.add_argument("--cpu-passes", type=int, default=8)
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--skip-towers", action="store_true")
    ap.add_argument("--skip-dynemb", action="store_true")
    ap.add_argument("--skip-pool", action="store_true")
    ap.add_argument("--pool-steps", type=int, default=500)
    ap.add_argument("--skip-pool-stress", action="store_true")
    ap.add_argument("--skip-steady", action="store_true")
    ap.add_argument("--steady-reps", type=int, default=100)
    ap.add_argument("--pool-stress-steps", type=int, default=200)
    ap.add_argument("--skip-train", action="store_true")
    ap.add_argument("--train-steps", type=int, default=100)
    ap.add_argument("--dynemb-steps", type=int, default=500)
    ap.add_argument("--towers-steps", type=int, default=300)
    ap.add_argument("--skip-configs", action="store_true")
    ap.add_argument("--config-scale", type=float, default=1.0)
    ap.add_argument("--cpu-single-sample", type=int, default=4096)
    ap.add_argument("--cpu-padded-sample", type=int, default=512)
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.impl == "reference":
        return run_reference(args)

    import torch
    import torch.distributed as dist
    from recsys_sparse_embedding_gb300 import binding, synth
    from recsys_sparse_embedding_gb300.device_batch import to_device

    ws, rank, local = dist_env()
    if ws > 1:
        dist.init_process_group("nccl", init_method="env://")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    batch = synth.generate(WORKLOAD, seed=rank)
    db = to_device(batch, dev)
    B, D, F = db.B, db.D, db.F
    mode = binding.DSF_MODE_BF16_TC if args.mode == "bf16" else binding.DSF_MODE_FP32
    mlp = db.mlp(mode)
    wsp = binding.Workspace(B, D, device=dev)
    wsp.prepare(mlp)
    pooled = torch.empty(B, F * D, device=dev)
    din = torch.empty(B, 3 * D, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def step():
        binding.din_sparse_fwd(db.tables, db.values, db.lengths, db.seq_values, db.seq_lengths,
                               db.max_len, db.q_feat, db.seq_table, B, mlp, pooled, din, wsp,
                               status=status, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            step()
        stream.synchronize()
        st = int(status.item())
        if st:
            raise RuntimeError("device status 0x%x during warm-up" % st)
        graph = None
        if not args.no_graph:
            try:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    step()
                g.replay()
                stream.synchronize()
                graph = g
            except Exception as e:  # capture unsupported: time direct launches
                print("graph capture unavailable: %s" % e, file=sys.stderr)
                graph = None
                torch.cuda.synchronize()
        run = graph.replay if graph is not None else step

        # The K timed steps sit inside a window of at least CLOCK_WINDOW_S of
        # identical steps, over which nvidia-smi samples the clocks (a short
        # timed region alone would end before its first sample).
        K = args.steps
        window_us = []
        with ClockSampler(local) as clk:
            t_end = time.perf_counter() + CLOCK_WINDOW_S / 2
            while time.perf_counter() < t_end:
                window_us += time_flushed(run, flush, 100, stream)
            if ws > 1:
                dist.barrier()
            torch.cuda.synchronize()
            times_us = time_flushed(run, flush, K, stream)
            if ws > 1:
                dist.barrier()
            t_end = time.perf_counter() + CLOCK_WINDOW_S / 2
            while time.perf_counter() < t_end:
                window_us += time_flushed(run, flush, 100, stream)
        window_s = clk.seconds
        st = int(status.item())
        total_ms = max_over_ranks(sum(times_us) / 1e3, ws, dev)
        value = weak_rate(B * K, total_ms, ws)
        ms_step = total_ms / K

        # End to end: every step copies its inputs from pinned host memory to the
        # device, calls the C ABI, and copies both outputs back to pinned host
        # memory. Steps are pipelined over two buffer slots: the copies of one
        # step run on their own streams (copy engines) while the kernel of the
        # next runs; events order each slot's reuse. E2E_GRAPH steps are
        # captured into one CUDA graph (host enqueue of ~15 calls per step would
        # otherwise bound the rate) and the graph is replayed.
        h_in = [x.cpu().pin_memory() for x in (db.values, db.lengths, db.seq_values, db.seq_lengths)]
        d_in = [[torch.empty_like(x, device=dev) for x in h_in] for _ in range(2)]
        d_out = [(torch.empty_like(pooled), torch.empty_like(din)) for _ in range(2)]
        h_out = [[torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in d_out[0]] for _ in range(2)]
        h2d = sum(x.numel() * x.element_size() for x in h_in)
        d2h = sum(t.numel() * t.element_size() for t in d_out[0])
        s_h2d = torch.cuda.Stream(device=dev)
        s_d2h = torch.cuda.Stream(device=dev)

        def e2e_steps(n):
            ev_run, ev_out = [None, None], [None, None]
            for i in range(n):
                j = i & 1
                if ev_run[j] is not None:
                    s_h2d.wait_event(ev_run[j])      # the kernel that read slot j is done
                with torch.cuda.stream(s_h2d):
                    for h, d in zip(h_in, d_in[j]):
                        d.copy_(h, non_blocking=True)
                ev_in = torch.cuda.Event()
                ev_in.record(s_h2d)
                stream.wait_event(ev_in)
                if ev_out[j] is not None:
                    stream.wait_event(ev_out[j])     # slot j's previous outputs are on the host
                binding.din_sparse_fwd(db.tables, d_in[j][0], d_in[j][1], d_in[j][2], d_in[j][3],
                                       db.max_len, db.q_feat, db.seq_table, B, mlp, d_out[j][0],
                                       d_out[j][1], wsp, status=status, stream=stream)
                ev_run[j] = torch.cuda.Event()
                ev_run[j].record(stream)
                s_d2h.wait_event(ev_run[j])
                with torch.cuda.stream(s_d2h):
                    for d, h in zip(d_out[j], h_out[j]):
                        h.copy_(d, non_blocking=True)
                ev_out[j] = torch.cuda.Event()
                ev_out[j].record(s_d2h)

        G = E2E_GRAPH
        E = max(G, (args.e2e_steps // G) * G)
        graph_e2e = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph_e2e, stream=stream):
            s_h2d.wait_stream(stream)
            s_d2h.wait_stream(stream)
            e2e_steps(G)
            stream.wait_stream(s_h2d)
            stream.wait_stream(s_d2h)
        for _ in range(2):
            graph_e2e.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(E // G):
            graph_e2e.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(e0.elapsed_time(e1), ws, dev)
        e2e_value = weak_rate(B * E, e2e_ms, ws)
        # the last step's results, read back, match the device-timed outputs
        if not (torch.equal(h_out[(G - 1) & 1][1], din.cpu()) and
                torch.equal(h_out[(G - 1) & 1][0], pooled.cpu())):
            raise RuntimeError("end-to-end outputs differ from the device-timed run")

    steady = None
    if not args.skip_steady:
        steady = time_steady_state(binding, synth, db, mlp, wsp, status, dev, 8, args.steady_reps)

    pool_only = None
    if not args.skip_pool:
        pool_only = time_pool_only(binding, db, wsp, flush, args.pool_steps, batch, ws)

    # the pooling stage where bandwidth, not the launch, dominates: B=65536,
    # 1.92 GB of tables (five of 2M-10M rows), uniform ids
    pool_stress = None
    if not args.skip_pool_stress:
        sb = synth.generate("gather_stress", seed=0)
        sdb = to_device(sb, dev)
        swsp = binding.Workspace(sb.B, sb.D, device=dev)
        pool_stress = time_pool_only(binding, sdb, swsp, flush, args.pool_stress_steps, sb, ws,
                                     workload="gather_stress B=65536, 1.92 GB fp32 tables, uniform ids",
                                     also_unflushed=True)
        del sdb, swsp, sb

    dynemb = None
    if not args.skip_dynemb:
        dynemb = time_dynamic_emb(binding, synth, batch, dev, mode, flush, args.dynemb_steps, ws)

    train = None
    if rank == 0 and not args.skip_train:
        train = time_train_step(binding, db, mlp, wsp, pooled, din, status, flush, args.train_steps, batch)

    towers = None
    if rank == 0 and not args.skip_towers:
        towers = time_towers(binding, synth, pooled, din, B, dev, flush, args.towers_steps)

    # roofline of the fused kernel (the only kernel of a step), timed alone:
    # the burst tensor peak
    nbytes, flops, P = algorithmic_work(batch)
    roof = roofline(nbytes, flops, ms_step * 1e3)
    roof["traffic"] = traffic_record()
    roof["valid_positions"] = P
    headline = {"B": B, "D": D, "dtype": batch.wl.dtype, "valid_positions": P,
                "us_per_step": step_stats(times_us), "samples_per_s": value, "roofline": roof}
    configs = None
    if rank == 0 and not args.skip_configs:
        configs = time_configs(binding, synth, dev, mode, flush, args.config_scale, headline)

    cpu = None
    if rank == 0 and ws == 1 and not args.skip_cpu:
        threads = os.cpu_count() or 1
        rate, dt, cpu_s = cpu_oracle_rate(batch, args.cpu_sample, args.cpu_passes, threads)
        cpu = {"value": rate, "unit": UNIT, "cores": threads, "kind": "oracle",
               "sample": "%d passes over %d samples of the B=%d batch (%.1f s wall, %.1f s of CPU time)"
               % (args.cpu_passes, args.cpu_sample, B, dt, cpu_s)}
        cpu.update(cpu_baselines(synth, batch, args.cpu_single_sample, args.cpu_padded_sample))

    clocks = clk.summary()
    if clocks.get("sm_mhz"):
        clocks["us_x_mhz_median"] = step_stats(times_us)["median"] * clocks["sm_mhz"]
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "fp32+bf16", "data": "synthetic",
            "config": {"workload": workload_desc(B), "B": B, "mode": args.mode,
                       "l2": "flushed between steps (512 MB write, not timed)",
                       "graph": graph is not None, "parallelism": "replicas" if ws > 1 else "1gpu"},
            "roofline": roof,
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h,
                    "method": "pinned host inputs -> device, din_sparse_fwd, both outputs -> "
                              "pinned host, every step; two buffer slots, copies on their own "
                              "streams overlap the next step's kernel; %d steps per captured CUDA "
                              "graph, %d steps timed; no L2 flush (tables 201 MB > 129 MB L2)"
                              % (E2E_GRAPH, E)},
            "gpu_launches": args.steps,
            "clocks": clocks,
            "us_per_step": step_stats(times_us),
            "clock_window": {"seconds": window_s, "steps": len(window_us) + K,
                             "us_per_step": step_stats(window_us + times_us),
                             "what": "the K timed steps and identical flushed steps around them, "
                                     "run while nvidia-smi samples the clocks every 100 ms"},
            "configs": configs,
            "status": st,
            "towers": towers,
            "steady_state": steady,
            "pool_only": pool_only,
            "pool_only_gather_stress": pool_stress,
            "dynamic_emb": dynemb,
            "train_step": train,
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())

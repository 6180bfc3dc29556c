"""Benchmark of one decode step of the library on a named workload.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--config NAME]

A step is one pass of the hot path over one batch: for every layer of the
workload, kv_append of the new token and the layer's decode (the sparse
workload runs its Full / Reuse / Reindex schedule). The headline workload
is the Llama-3.1-70B-shaped GQA decode (B=32, ragged lengths around 4.5K, 80
layers of 64 query / 8 kv heads of 128, bf16); every other workload is a
sub-record of the same line under `configs` (--sub-configs).

Prints ONE JSON line (rank 0). `value` is KV-read GB/s over all ranks:
algorithmic cache bytes read per step (every visible K and V element once)
divided by the device time of a step, inputs resident in HBM. Each layer has
its own cache, so a step's working set (45 GB for the headline, 2.1 GB for
the Llama-2-7B shape) is far larger than L2 and no flush is needed between
steps. `e2e` is the same metric when every
step also copies its inputs (q, k_new, v_new of all layers) from pinned host
memory and reads the outputs back. `roofline` times the dominant kernel
(the decode kernel) per launch with CUDA events on its stream.
`cpu_baseline` times the fp64 oracle on the host cores on a bounded sample.

--impl reference times that oracle alone as the reference arm.
Multi-GPU: independent replicas (the decode of a batch does not shard
across GPUs here), one process per GPU under torchrun, no collective on the
data path; the step time is the max over ranks.
"""
import argparse
import hashlib
import json
import multiprocessing as mp
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from kv_cache_decode_gqa_gb300 import inputs as I  # noqa: E402
from kv_cache_decode_gqa_gb300 import workloads as W  # noqa: E402

METRIC = ("decode attn: KV-read HBM GB/s (% of GB300 peak) and decode "
          "tokens/s per layer")
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0      # GB300 HBM3e, nominal (context beside the measured peak)
FALLBACK_BF16_TFLOPS = 1900.0


# ---------------------------------------------------------------------------
# algorithmic accounting
# ---------------------------------------------------------------------------
def kv_bytes_layer(shape, layer=0):
    """Cache bytes one layer's decode reads: every visible K and V element
    once (K-only rows for the latent cache; for the sparse schedule, the
    indexer keys of Full / Reindex layers plus the selected K and V rows)."""
    s = shape
    if s.kind == "gqa":
        seen = [min(L, s.window) if s.window else L for L in s.seq_lens]
        return sum(seen) * s.n_kv * 2 * s.head_dim * s.elem_bytes
    if s.kind == "mla":
        return sum(s.seq_lens) * s.head_dim * 2
    sel = s.batch * min(layer_topk(s, layer), min(s.seq_lens)) * 2 * \
        s.head_dim * 2
    if s.modes[layer] == "reindex" and s.pool_k:
        # a pooled Reindex layer scores only the pool's candidates (8 per
        # pool block, counted on the device after the warm-up)
        cands = getattr(s, "pool_cands", None)
        if cands is None:
            cands = sum(min(L, 16384) for L in s.seq_lens)
        sel += cands * s.idx_dim * 2
    elif s.modes[layer] in ("full", "reindex"):
        sel += sum(s.seq_lens) * s.idx_dim * 2
    return sel


def layer_topk(s, layer):
    """Positions the sparse schedule's layer attends to: its own
    selection's size, or the one it reuses."""
    k = s.topk
    for m in s.modes[:layer + 1]:
        if m == "full" or (m == "reindex" and not s.pool_k):
            k = s.topk
        elif m == "reindex":
            k = s.pool_k
    return k


def kv_bytes_step(shape):
    return sum(kv_bytes_layer(shape, l) for l in range(shape.n_layers))


def decode_launch_bytes(shape):
    """Algorithmic bytes of one decode call: cache read + q read + output
    written (GQA: the call also appends, so + the new rows read and
    written)."""
    s = shape
    if s.kind == "sparse":  # the average over the schedule's layers
        rows = sum(min(layer_topk(s, l), min(s.seq_lens))
                   for l in range(s.n_layers)) / s.n_layers
        b = int(s.batch * rows * 2 * s.head_dim * 2)
    else:
        b = kv_bytes_layer(s)
    b += s.batch * s.n_h * s.head_dim * 2 + s.batch * s.n_h * s.dv * 2
    if s.kind == "gqa":
        b += 2 * s.batch * s.n_kv * s.head_dim * (2 + s.elem_bytes)
    return b


def data_description(shape):
    """The bench line's `data`: what the seeded synthetic inputs are."""
    cache = {"fp8": "random E4M3 cache codes with per-head scales",
             "mxfp4": "random E2M1 cache codes with E4M3 group scales"}.get(
                 shape.dtype, "N(0,1) bf16 cache")
    return f"synthetic (seeded {cache}, N(0,1) bf16 queries)"


def measured_peaks(key="hbm_gbs"):
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d[key]), "measured"
    except Exception:
        return ({"hbm_gbs": FALLBACK_HBM_GBS}.get(key, FALLBACK_BF16_TFLOPS),
                "fallback")


# CTAs of a lane per 128-head tile in the tensor-core latent kernel (each
# holds 512 / LATENT_TC_PARTS of the output columns)
LATENT_TC_PARTS = 2


def latent_flops(shape):
    """Multiply-add work of one latent decode call, in FLOPs: useful (each
    head scores every cached row over 576 dims and sums 512 latent dims) and
    issued by the tensor-core kernel (each of a lane's LATENT_TC_PARTS
    value-part CTAs computes the full scores of its 128 heads)."""
    s = shape
    rows = sum(s.seq_lens)
    useful = 2 * rows * s.n_h * (s.head_dim + s.dv)
    issued = 2 * rows * s.n_h * (LATENT_TC_PARTS * s.head_dim + s.dv)
    return useful, issued


def profile_traffic(kernel_tag):
    """DRAM bytes per launch from an ncu capture of this kernel, if profiles/
    holds one ('traffic_bytes_per_launch: N') and the kernel's sources are
    unchanged since the capture (the file's 'kernel_sources_sha256:' matches
    a hash of the listed sources); otherwise None."""
    path = os.path.join(ROOT, "profiles", f"{kernel_tag}.txt")
    fields = {}
    try:
        with open(path) as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    fields[k.strip()] = v.strip()
    except OSError:
        return None
    v = fields.get("traffic_bytes_per_launch", "null")
    srcs = fields.get("kernel_sources", "").split()
    if v in ("", "null") or not srcs:
        return None
    h = hashlib.sha256()
    try:
        for name in srcs:
            with open(os.path.join(ROOT, "kv_cache_decode_gqa_gb300", "csrc",
                                   name), "rb") as f:
                h.update(f.read())
    except OSError:
        return None
    if h.hexdigest()[:16] != fields.get("kernel_sources_sha256"):
        return None  # the kernel changed after the counters were taken
    return float(v)


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,"
              "clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.lines = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100",
                 "-i", str(gpu_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for line in out.splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# distributed plumbing (replicas)
# ---------------------------------------------------------------------------
def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def dist_init(ws, backend):
    if ws <= 1:
        return None
    import torch.distributed as dist
    os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
    dist.init_process_group(backend)
    return dist


def max_over_ranks(dist, x, device=None):
    if dist is None:
        return x
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


# ---------------------------------------------------------------------------
# the oracle on the host cores (cpu_baseline and the reference arm)
# ---------------------------------------------------------------------------
def oracle_unit_inputs(name, layer, seqs):
    """Host inputs of one oracle unit: layer ``layer`` (every layer of the
    schedule for the sparse workloads) for sequences ``seqs`` (compact
    caches), with this step's append applied by the oracle's own
    kv_append."""
    import oracle
    s = W.config(name)
    pg = W.Paging(s)
    pos = [s.lengths[b] for b in seqs]
    lens = [s.seq_lens[b] for b in seqs]
    if s.kind == "sparse":
        kr, bt = W.host_cache_compact(s, pg, 0, W.T_K, seqs, n_kv=1)
        vr, _ = W.host_cache_compact(s, pg, 0, W.T_V, seqs, n_kv=1)
        ir, _ = W.host_cache_compact(s, pg, 0, W.T_IDXK, seqs,
                                     width=s.idx_dim, n_kv=1,
                                     table=I.normal_bf16_table())
        kn = W.host_bf16(s, 0, W.T_KNEW, (s.batch, 1, s.head_dim))[seqs]
        vn = W.host_bf16(s, 0, W.T_VNEW, (s.batch, 1, s.head_dim))[seqs]
        xn = W.host_bf16(s, 0, W.T_IDXKNEW, (s.batch, 1, s.idx_dim))[seqs]
        kr = oracle.kv_append(kr, bt, pos, kn, s.block_size)
        vr = oracle.kv_append(vr, bt, pos, vn, s.block_size)
        ir = oracle.kv_append(ir, bt, pos, xn, s.block_size)
        qs, qis, ws_ = {}, {}, {}
        for l in range(s.n_layers):
            qs[l] = oracle.bf16_bits_to_f64(
                W.host_bf16(s, l, W.T_Q, (s.batch, s.n_h, s.head_dim)))[seqs]
            if s.modes[l] != "reuse":
                qis[l] = oracle.bf16_bits_to_f64(
                    W.host_bf16(s, l, W.T_QIDX,
                                (s.batch, s.idx_heads, s.idx_dim)))[seqs]
                ws_[l] = W.host_weights(s, l)[seqs]
        return dict(kind="sparse", s=s, q=qs, q_idx=qis, w=ws_, kr=kr, vr=vr,
                    ir=ir, bt=bt, lens=lens, seqs=seqs, layer=layer)
    q = oracle.bf16_bits_to_f64(W.host_bf16(s, layer, W.T_Q,
                                            (s.batch, s.n_h, s.head_dim)))[seqs]
    knew = W.host_bf16(s, layer, W.T_KNEW, (s.batch, s.n_kv, s.head_dim))[seqs]
    kr, bt = W.host_cache_compact(s, pg, layer, W.T_K, seqs)
    kr = oracle.kv_append(kr, bt, pos, knew, s.block_size) \
        if s.dtype == "bf16" else kr
    vr = None
    if s.has_v:
        vnew = W.host_bf16(s, layer, W.T_VNEW,
                           (s.batch, s.n_kv, s.head_dim))[seqs]
        vr, _ = W.host_cache_compact(s, pg, layer, W.T_V, seqs)
        if s.dtype == "bf16":
            vr = oracle.kv_append(vr, bt, pos, vnew, s.block_size)
    d = dict(kind=s.kind, s=s, q=q, kr=kr, vr=vr, bt=bt, lens=lens,
             seqs=seqs, layer=layer)
    if s.dtype == "mxfp4":
        d["kr"] = oracle.kv_append(kr, bt, pos, knew, s.block_size, "mxfp4")
        d["vr"] = oracle.kv_append(vr, bt, pos, vnew, s.block_size, "mxfp4")
    if s.dtype == "fp8":
        ks, kinv = W.host_scales(s, layer, W.T_KSCALE)
        vs, vinv = W.host_scales(s, layer, W.T_VSCALE)
        d["kr"] = oracle.kv_append(kr, bt, pos, knew, s.block_size, "fp8", kinv)
        d["vr"] = oracle.kv_append(vr, bt, pos, vnew, s.block_size, "fp8", vinv)
        d["ks"], d["vs"] = ks, vs
    return d


def oracle_run_unit(d):
    """One oracle pass over a prepared unit. Returns (KV bytes read,
    sequence-layer decodes done): the metric's bytes, counted as for the GPU
    step, and the tokens of `tokens_per_s_per_layer`."""
    import oracle
    s = d["s"]
    n = len(d["seqs"])
    if d["kind"] == "gqa":
        if s.dtype == "fp8":
            oracle.gqa_decode(d["q"], d["kr"], d["vr"], d["bt"], d["lens"],
                              s.block_size, dtype="fp8", k_scale=d["ks"],
                              v_scale=d["vs"], window=s.window)
        else:
            oracle.gqa_decode(d["q"], d["kr"], d["vr"], d["bt"], d["lens"],
                              s.block_size, dtype=s.dtype, window=s.window)
        seen = [min(L, s.window) if s.window else L for L in d["lens"]]
        return sum(seen) * s.n_kv * 2 * s.head_dim * s.elem_bytes, n
    if d["kind"] == "mla":
        oracle.mla_decode(d["q"], d["kr"], d["bt"], d["lens"], s.block_size,
                          d_c=s.d_c)
        return sum(d["lens"]) * s.head_dim * 2, n
    # the sparse workloads: the whole Full / Reuse / Reindex schedule (its
    # bytes counted as for the GPU step, per sequence)
    L = range(s.n_layers)
    oracle.sparse_schedule(s.modes, [d["q"][l] for l in L],
                           [d["q_idx"].get(l) for l in L],
                           [d["w"].get(l) for l in L], d["kr"], d["vr"],
                           d["ir"], d["bt"], d["lens"], s.block_size, s.topk,
                           pool_k=s.pool_k)
    return kv_bytes_step(s) * n // s.batch, n * s.n_layers


def _oracle_worker_main(args):
    name, units, budget_s = args
    ds = [oracle_unit_inputs(name, layer, seqs) for layer, seqs in units]
    for d in ds:
        oracle_run_unit(d)                           # untimed first pass
    nbytes, toks, reps = 0, 0, 0
    t0 = time.perf_counter()
    while True:
        for d in ds:
            b, t = oracle_run_unit(d)
            nbytes += b
            toks += t
            reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return nbytes, toks, el, reps


def oracle_plan(shape, cores):
    """The oracle baseline's work, one list of (layer, sequences) units per
    worker (a worker takes its units in turn), and how it covers a step:
      Llama-2 shapes and tiny: every layer of the step, layers dealt out to
        the workers;
      Llama-3.1 shapes: one full layer (all 32 sequences dealt out to the
        workers), a step being 80 such layers;
      latent: a subset of the batch rows (one sequence a worker), scaled
        linearly in B;
      sparse: the whole 8-layer schedule, one sequence a worker."""
    s = shape
    if s.kind == "gqa" and s.n_layers <= 32:
        units = [(l, list(range(s.batch))) for l in range(s.n_layers)]
        n = min(cores, len(units))
        return [units[i::n] for i in range(n)], \
            f"every layer of the step ({s.n_layers} layers)"
    if s.kind == "gqa":
        n = min(cores, s.batch)
        return [[(0, list(range(s.batch))[i::n])] for i in range(n)], \
            f"one full layer (all {s.batch} sequences), x{s.n_layers} layers"
    if s.kind == "mla":
        n = min(cores, s.batch)
        return [[(0, [b])] for b in range(n)], \
            f"{n} of {s.batch} batch rows, scaled x{s.batch / n:g} in B"
    n = min(cores, s.batch)
    return [[(0, [b])] for b in range(n)], \
        f"the whole {s.n_layers}-layer schedule, one sequence a worker"


def cpu_baseline(name, budget_s=8.0, budget_1=3.0):
    """Time the oracle on the host cores, as it stands: one spawned
    single-threaded worker per core on its sampled unit for ~budget_s
    seconds (all cores), and one worker alone for ~budget_1 seconds (one
    thread). GB/s = bytes read / slowest worker's time; tokens/s per layer =
    sequence-layer decodes / that time."""
    s = W.config(name)
    cores = os.cpu_count() or 1
    plan, how = oracle_plan(s, cores)
    env_keys = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")
    saved = {k: os.environ.get(k) for k in env_keys}
    for k in env_keys:
        os.environ[k] = "1"
    try:
        ctx = mp.get_context("spawn")
        with ctx.Pool(1) as pool:
            one = pool.map(_oracle_worker_main,
                           [(name, plan[0], budget_1)])[0]
        with ctx.Pool(len(plan)) as pool:
            res = pool.map(_oracle_worker_main,
                           [(name, u, budget_s) for u in plan])
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    total = sum(r[0] for r in res)
    toks = sum(r[1] for r in res)
    wall = max(r[2] for r in res)
    reps = sum(r[3] for r in res)
    gbs = total / wall / 1e9
    step_bytes = kv_bytes_step(s)
    return {
        "value": round(gbs, 4), "unit": "GB/s", "cores": len(plan),
        "kind": "oracle",
        "value_1thread": round(one[0] / one[2] / 1e9, 4),
        "tokens_per_s_per_layer": round(toks / wall, 3),
        "tokens_per_s_per_layer_1thread": round(one[1] / one[2], 3),
        "ms_per_step": round(step_bytes / (gbs * 1e9) * 1e3, 2)
        if gbs > 0 else None,
        "sample": (f"{how}: {len(plan)} single-threaded processes, each "
                   f"repeating its units for ~{budget_s:g} s ({reps} oracle "
                   f"passes, {total / 1e9:.2f} GB of cache read); one thread:"
                   f" the first process's units alone for ~{budget_1:g} s"),
    }


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def build_step(K, wl, outs, wss, events=None):
    """The workload's step as a serving loop issues it. ``events`` (tag ->
    list of (start, end) event pairs to fill) brackets each call."""
    s = wl.shape

    def mark(tag, i):
        if events is not None:
            events.setdefault(tag, [])
            if len(events[tag]) <= i:
                import torch
                events[tag].append((torch.cuda.Event(enable_timing=True,
                                                     external=True),
                                    torch.cuda.Event(enable_timing=True,
                                                     external=True)))
            return events[tag][i]
        return None

    def timed(tag, i, fn):
        ev = mark(tag, i)
        if ev is not None:
            ev[0].record()
        fn()
        if ev is not None:
            ev[1].record()

    def step():
        if s.kind == "sparse":
            run_sparse_schedule(K, wl, outs, wss, timed)
            return
        for i, layer in enumerate(wl.layers):
            c = wl.caches[layer]
            if s.kind == "mla":
                timed("append", i, lambda: K.kv_append(
                    c, wl.block_table, wl.pos, wl.k_new[layer]))
                timed("decode", i, lambda: K.mla_decode(
                    c, wl.block_table, wl.seq_lens, wl.max_seq_len,
                    wl.q[layer], d_c=s.d_c, out=outs[layer],
                    workspace=wss[layer], want_lse=False))
            else:
                # the append rides in the decode's pass over the cache; the
                # lengths and block tables are set before the step, and the
                # rows before the newest were appended by earlier steps
                timed("decode", i, lambda: K.gqa_append_decode(
                    c, wl.block_table, wl.seq_lens, wl.max_seq_len, wl.pos,
                    wl.k_new[layer], wl.v_new[layer], wl.q[layer],
                    out=outs[layer], workspace=wss[layer], want_lse=False,
                    seqs_flags=K.SEQS_STABLE | K.SEQS_PREFIX_READY,
                    window=s.window))
    return step


def run_sparse_schedule(K, wl, outs, wss, timed=None):
    s = wl.shape
    if timed is None:
        def timed(tag, i, fn):
            fn()
    c = wl.caches[0]

    def appends():
        K.kv_append(c, wl.block_table, wl.pos, wl.k_new[0], wl.v_new[0])
        K.kv_append(wl.idx_cache, wl.block_table, wl.pos, wl.idx_k_new)
    timed("append", 0, appends)
    idx = None
    pooled = False
    n_sel = 0
    for layer in wl.layers:
        if s.modes[layer] == "reindex" and pooled:
            idx = wss["idx"][layer]
            timed("select", n_sel, lambda: K.indexer_topk_pool(
                wl.idx_cache, wl.block_table, wl.seq_lens, wl.max_seq_len,
                wl.q_idx[layer], wl.w[layer], wss["pool"], wss["pool_n"],
                s.pool_k, indices=wss["idx"][layer],
                workspace=wss["pooltopk"]))
            n_sel += 1
        elif s.modes[layer] != "reuse":
            idx = wss["idx"][layer]
            timed("select", n_sel, lambda: K.indexer_topk(
                wl.idx_cache, wl.block_table, wl.seq_lens, wl.max_seq_len,
                wl.q_idx[layer], wl.w[layer], s.topk,
                indices=wss["idx"][layer], workspace=wss["topk"],
                seqs_flags=K.SEQS_STABLE | K.SEQS_PREFIX_READY))
            n_sel += 1
            if s.modes[layer] == "full" and s.pool_k and not pooled:
                K.indexer_pool(wl.block_table, wl.seq_lens, wl.max_seq_len,
                               idx, pool=wss["pool"], pool_n=wss["pool_n"])
                pooled = True
        sel = idx
        timed("decode", layer, lambda: K.sparse_decode(
            c, wl.block_table, wl.seq_lens, wl.max_seq_len, sel,
            wl.q[layer], out=outs[layer], workspace=wss[layer],
            want_lse=False))


def pack_inputs(torch, wl):
    """Move every per-step input of every layer into one device buffer (and
    the tensors into views of it), so that the end-to-end step copies its
    inputs with one host-to-device transfer."""
    s = wl.shape
    tensors = []
    for layer in wl.layers:
        tensors.append(("q", layer))
        if s.kind != "sparse" or layer == 0:
            if layer in wl.k_new:
                tensors.append(("k_new", layer))
            if layer in wl.v_new:
                tensors.append(("v_new", layer))
        if s.kind == "sparse" and layer in wl.q_idx:
            tensors.append(("q_idx", layer))
    total = sum(getattr(wl, n)[l].numel() for n, l in tensors)
    if s.kind == "sparse":
        total += wl.idx_k_new.numel()
    buf = torch.empty(total, dtype=torch.bfloat16, device=wl.block_table.device)
    off = 0
    for n, l in tensors:
        t = getattr(wl, n)[l]
        view = buf[off:off + t.numel()].view(t.shape)
        view.copy_(t)
        getattr(wl, n)[l] = view
        off += t.numel()
    if s.kind == "sparse":
        t = wl.idx_k_new
        view = buf[off:off + t.numel()].view(t.shape)
        view.copy_(t)
        wl.idx_k_new = view
    return buf


def sparse_buffers(torch, K, wl, dev):
    """Index tensors of every layer and the selection workspaces of the
    sparse schedule (and the hierarchical indexer's pool)."""
    s = wl.shape
    b = {"idx": {l: torch.empty((s.batch, s.pool_k if s.pool_k and
                                 s.modes[l] == "reindex" else s.topk),
                                dtype=torch.int32, device=dev)
                 for l in wl.layers}}
    n = K.workspace_size(K.OP_INDEXER_TOPK, wl.idx_cache, wl.block_table,
                         wl.seq_lens, wl.max_seq_len, s.idx_heads, s.topk)
    b["topk"] = torch.zeros(max(n, 256), dtype=torch.uint8, device=dev)
    if s.pool_k:
        b["pool"] = torch.empty((s.batch, K.POOL_BLOCKS), dtype=torch.int32,
                                device=dev)
        b["pool_n"] = torch.empty((s.batch,), dtype=torch.int32, device=dev)
        n = K.workspace_size(K.OP_INDEXER_TOPK_POOL, wl.idx_cache,
                             wl.block_table, wl.seq_lens, wl.max_seq_len,
                             s.idx_heads, s.pool_k)
        b["pooltopk"] = torch.zeros(max(n, 256), dtype=torch.uint8,
                                    device=dev)
    return b


def config_dict(s, ws):
    """The bench line's `config`: the workload, by name and sizes (both
    arms print the same dict)."""
    return {"workload": s.name, "batch": s.batch,
            "cached_len": s.lengths[0] if len(set(s.lengths)) == 1
            else f"{min(s.lengths)}..{max(s.lengths)}",
            "layers": s.n_layers, "n_h": s.n_h, "n_kv": s.n_kv,
            "head_dim": s.head_dim, "block_size": s.block_size,
            "cache_dtype": s.dtype,
            **({"window": s.window} if s.window else {}),
            **({"topk": s.topk, "schedule": "/".join(s.modes)}
               if s.kind == "sparse" else {}),
            **({"pool_topk": s.pool_k} if s.pool_k else {}),
            "parallelism": f"replicas x{ws}",
            "l2": ("indexer keys (134 MB) and the selected rows read per "
                   "step exceed L2; Reuse layers re-read rows their Full "
                   "layer read; no flush" if s.kind == "sparse" else
                   "working set per step larger than L2 (distinct per-layer "
                   "caches, or one 2.4 GB latent cache); no flush")}


def kernel_tag(s):
    return {"gqa": "decode_simt" if s.n_h // s.n_kv <= 4 else "decode_mma",
            "mla": "decode_mla", "sparse": "decode_sparse"}[s.kind] + \
        "_" + s.name


def measure(K, torch, name, args, ws, dist, dev, local):
    """One workload: graph-captured steps, timed; end to end with host
    copies; each call bracketed by events. Returns its record (rank 0) with
    the step time as the max over ranks."""
    s = W.config(name)
    wl = W.DeviceWorkload(s, device=dev)
    outs = {l: torch.empty((s.batch, s.n_h, s.dv), dtype=torch.bfloat16,
                           device=dev) for l in wl.layers}
    wss = {}
    for l in wl.layers:
        if s.kind == "sparse":
            n = K.workspace_size(K.OP_SPARSE_DECODE, wl.caches[l],
                                 wl.block_table, wl.seq_lens, wl.max_seq_len,
                                 s.n_h, s.topk)
        elif s.kind == "mla":
            n = K.workspace_size(K.OP_MLA_DECODE, wl.caches[l], wl.block_table,
                                 wl.seq_lens, wl.max_seq_len, s.n_h)
        else:
            n = K.workspace_size(K.OP_GQA_DECODE, wl.caches[l], wl.block_table,
                                 wl.seq_lens, wl.max_seq_len, s.n_h)
        wss[l] = torch.zeros(max(n, 256), dtype=torch.uint8, device=dev)
    if s.kind == "sparse":
        wss.update(sparse_buffers(torch, K, wl, dev))
    in_buf = pack_inputs(torch, wl)
    out_views = [outs[l] for l in wl.layers]

    step = build_step(K, wl, outs, wss)
    step()                                   # eager once: validates, warms
    torch.cuda.synchronize()
    if K.device_error() != 0:
        raise RuntimeError(f"{name}: device error word set after a step")

    stream = torch.cuda.Stream(device=dev)
    graph = torch.cuda.CUDAGraph()
    n0 = K.launch_count()
    with torch.cuda.graph(graph, stream=stream):
        step()
    launches_per_step = K.launch_count() - n0
    torch.cuda.synchronize()

    clocks = ClockSampler(local)
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    if s.kind == "sparse" and s.pool_k:
        # the pooled Reindex layers' candidates (8 per pool block), for the
        # byte count; the pool is the same every step
        s.pool_cands = int(wss["pool_n"].sum().item()) * 8
    # keep replaying for a moment so the clock samples see the load
    t_end = time.perf_counter() + args.load_s
    while time.perf_counter() < t_end:
        for _ in range(10):
            graph.replay()
        torch.cuda.synchronize()

    # ---- timed region: K steps, inputs resident in HBM
    barrier(dist)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        graph.replay()
    e1.record()
    torch.cuda.synchronize()
    barrier(dist)
    clock_info = clocks.stop()
    ms = max_over_ranks(dist, e0.elapsed_time(e1) / args.steps, dev)

    # ---- end to end: host inputs in, outputs out, every step
    pinned_in = torch.empty(in_buf.numel(), dtype=torch.bfloat16,
                            pin_memory=True)
    pinned_in.copy_(in_buf)
    out_cat = torch.empty((len(out_views),) + tuple(out_views[0].shape),
                          dtype=torch.bfloat16, device=dev)
    pinned_out = torch.empty(out_cat.shape, dtype=torch.bfloat16,
                             pin_memory=True)

    def e2e_step():
        in_buf.copy_(pinned_in, non_blocking=True)
        graph.replay()
        torch.stack(out_views, out=out_cat)
        pinned_out.copy_(out_cat, non_blocking=True)

    for _ in range(max(args.warmup, 3)):
        e2e_step()
    torch.cuda.synchronize()
    barrier(dist)
    e2 = torch.cuda.Event(enable_timing=True)
    e3 = torch.cuda.Event(enable_timing=True)
    e2.record()
    for _ in range(args.steps):
        e2e_step()
    e3.record()
    torch.cuda.synchronize()
    barrier(dist)
    ms_e2e = max_over_ranks(dist, e2.elapsed_time(e3) / args.steps, dev)

    # ---- each call, CUDA events on its stream inside a captured step
    calls = time_calls(torch, K, wl, outs, wss, args)
    calls = {t: max_over_ranks(dist, v, dev) for t, v in calls.items()}
    del graph
    rec = None
    if dist is None or dist.get_rank() == 0:
        rec = record(s, ws, args, ms, ms_e2e, calls, clock_info,
                     launches_per_step, in_buf.numel() * 2,
                     out_cat.numel() * 2)
    del wl, outs, wss, in_buf, out_views, pinned_in, pinned_out, out_cat
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return rec


def time_calls(torch, K, wl, outs, wss, args):
    """Mean device time of each kind of call of a step (tag -> ms): the
    calls are bracketed by event nodes in a captured step, and the last of
    several replays is read."""
    evs = {}
    step = build_step(K, wl, outs, wss, events=evs)
    step()                      # creates the events (eager, untimed)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=torch.cuda.Stream()):
        step()
    for _ in range(max(args.warmup, 3) + args.steps):
        g.replay()
    torch.cuda.synchronize()
    res = {t: statistics.mean(a.elapsed_time(b) for a, b in pairs)
           for t, pairs in evs.items()}
    del g
    return res


def record(s, ws, args, ms, ms_e2e, calls, clock_info, launches_per_step,
           h2d, d2h):
    """The JSON record of one workload."""
    nbytes = kv_bytes_step(s)
    value = ws * nbytes / (ms / 1e3) / 1e9
    peak, peak_src = measured_peaks()
    launch_bytes = decode_launch_bytes(s)
    if s.kind == "gqa":
        # the step is this one call per layer, back to back: its average
        # duration inside the timed pipeline is the step time / layers (the
        # isolated, event-bracketed duration is reported beside it)
        call_ms = ms / s.n_layers
        timing = "timed step / layers (the step is this call per layer)"
    else:
        call_ms = calls["decode"]
        timing = "CUDA events around each call in a captured step"
    achieved = launch_bytes / (call_ms / 1e3) / 1e9
    tag = kernel_tag(s)
    rec = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": s.dtype,
        "data": data_description(s),
        "config": config_dict(s, ws),
        "pct_of_peak": round(100 * value / ws / peak, 1),
        "pct_of_nominal_hbm": round(100 * value / ws / NOMINAL_HBM_GBS, 1),
        "tokens_per_s_per_layer": round(s.batch * s.n_layers / (ms / 1e3), 1),
        "kv_bytes_per_step": nbytes,
        "e2e": {"value": round(ws * nbytes / (ms_e2e / 1e3) / 1e9, 1),
                "unit": "GB/s", "ms_per_step": round(ms_e2e, 4),
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": launches_per_step * args.steps,
        "gpu_launches_per_step": launches_per_step,
        "roofline": {"bound": "hbm", "kernel": tag,
                     "achieved": round(achieved, 1), "peak": peak,
                     "peak_source": peak_src, "unit": "GB/s",
                     "frac": round(achieved / peak, 4),
                     "bytes_per_launch": launch_bytes,
                     "launch_ms": round(call_ms, 5),
                     "launch_timing": timing,
                     "launch_ms_isolated": round(calls["decode"], 5),
                     "traffic": profile_traffic(tag)},
        "calls_ms": {t: round(v, 5) for t, v in calls.items()},
        "clocks": clock_info,
    }
    if s.kind == "mla":
        # the latent decode runs on the tensor cores: its tensor-side rate
        # against the measured bf16 peak (burst: the kernel is timed alone)
        useful, issued = latent_flops(s)
        kern_ms = calls["decode"]
        tpk, tsrc = measured_peaks("bf16_tflops")
        rec["roofline"]["tensor"] = {
            "useful_tflops": round(useful / (kern_ms / 1e3) / 1e12, 1),
            "issued_tflops": round(issued / (kern_ms / 1e3) / 1e12, 1),
            "peak": tpk, "peak_source": tsrc, "unit": "TFLOP/s",
            "frac_useful": round(useful / (kern_ms / 1e3) / 1e12 / tpk, 4),
            "frac_issued": round(issued / (kern_ms / 1e3) / 1e12 / tpk, 4),
            "flops_per_launch": {"useful": useful, "issued": issued}}
    if s.kind == "sparse" and "select" in calls:
        # the indexer + top-k call of a Full / Reindex layer, beside it
        sel_bytes = sum(s.seq_lens) * s.idx_dim * 2
        rec["select_call"] = {
            "ms": round(calls["select"], 5),
            "indexer_bytes_full_layer": sel_bytes,
            "note": "mean over the schedule's indexer + top-k calls (the "
                    "Full layer's reads every visible indexer key)"}
    return rec


def profile_run(args, local):
    """The workload's step, eagerly, warmup + steps times: a short program
    for profilers (no graph, no clock sampling, no oracle)."""
    import torch
    import kv_cache_decode_gqa_gb300 as K
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    s = W.config(args.config, **({"n_layers": args.layers}
                                 if args.layers else {}))
    wl = W.DeviceWorkload(s, device=dev)
    outs = {l: torch.empty((s.batch, s.n_h, s.dv), dtype=torch.bfloat16,
                           device=dev) for l in wl.layers}
    wss = {l: None for l in wl.layers}
    if s.kind == "sparse":
        wss.update(sparse_buffers(torch, K, wl, dev))
    step = build_step(K, wl, outs, wss)
    for _ in range(args.warmup + args.steps):
        step()
    torch.cuda.synchronize()
    print(json.dumps({"profile_run": s.name, "steps": args.warmup + args.steps,
                      "device_error": K.device_error()}))


# ---------------------------------------------------------------------------
# reference arm: the oracle on the host cores
# ---------------------------------------------------------------------------
def run_reference(args, ws, rank):
    if rank != 0:
        return None
    s = W.config(args.config)
    n = args.warmup + args.steps
    budget = max(1.0, min(8.0, 120.0 / max(n, 1)))
    vals, last = [], None
    for i in range(n):
        last = cpu_baseline(args.config, budget_s=budget,
                            budget_1=max(0.5, budget / 4))
        if i >= args.warmup:
            vals.append(last["value"])
    value = statistics.mean(vals) if vals else 0.0
    nbytes = kv_bytes_step(s)
    ms = nbytes / (value * 1e9) * 1e3 if value > 0 else None
    cpu = dict(last)
    cpu["value"] = round(value, 4)
    return {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 3) if ms else None,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": data_description(s),
        "config": config_dict(s, ws),
        "cpu_baseline": cpu,
        "e2e": {"value": round(value, 4), "unit": "GB/s",
                "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


HEADLINE = "llama31_70b_gqa"
SUB_CONFIGS = ["llama2_7b_mha", "llama31_70b_gqa_fp8", "mla", "sparse",
               "sparse_pool", "llama2_7b_mha_mxfp4",
               "llama31_70b_gqa_fp8_swa"]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default=HEADLINE, choices=W.CONFIGS,
                    help="the headline workload (top-level fields)")
    ap.add_argument("--sub-configs", default=",".join(SUB_CONFIGS),
                    help="comma-separated workloads reported under "
                         "`configs` in the same line ('' for none)")
    ap.add_argument("--no-cpu-baseline", action="store_true",
                    help="skip the oracle timing (for profiler runs)")
    ap.add_argument("--cpu-budget", type=float, default=4.0)
    ap.add_argument("--load-s", type=float, default=0.4,
                    help="seconds of untimed replays before each timed "
                         "region, so clock samples see the load")
    ap.add_argument("--profile-run", action="store_true",
                    help="only run warmup + steps eager steps (for ncu)")
    ap.add_argument("--layers", type=int, default=0,
                    help="with --profile-run: keep only this many layers of "
                         "the workload (same per-layer shape), so a profiler "
                         "capture holds a few GB")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    ws, rank, local = dist_setup()
    if args.profile_run:
        profile_run(args, local)
        return
    if args.impl == "reference":
        line = run_reference(args, ws, rank)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    subs = [c for c in args.sub_configs.split(",") if c and c != args.config]
    for c in subs:
        if c not in W.CONFIGS:
            ap.error(f"unknown workload {c}")
    names = [args.config] + subs
    # the oracle's process pools are spawned before this process touches
    # the GPU
    cpu = {}
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        for c in names:
            cpu[c] = cpu_baseline(c, args.cpu_budget,
                                  max(1.0, args.cpu_budget / 2.5))
    import torch
    import kv_cache_decode_gqa_gb300 as K
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = dist_init(ws, "nccl")
    recs = {}
    for c in names:
        recs[c] = measure(K, torch, c, args, ws, dist, dev, local)
    if dist is not None:
        dist.destroy_process_group()
    if rank != 0:
        return
    line = dict(recs[args.config])
    line["cpu_baseline"] = cpu.get(args.config)
    line["configs"] = {}
    for c in subs:
        r = dict(recs[c])
        r["cpu_baseline"] = cpu.get(c)
        line["configs"][c] = r
    # every launch of the line's timed regions, the sub-records' included
    line["gpu_launches_all_configs"] = sum(r["gpu_launches"]
                                           for r in recs.values())
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()

"""Benchmark of the NVFP4 block-sparse decode step on GB300.

One step = quantise-store of the step's new K / V / index-K rows + row map +
index score and block top-k (or the fused verify path) + block-sparse
attention, on one batch of a synthetic workload whose cache is already
resident in HBM. Default workload: the skewed decode batch (one 450K-token and
seven 150K-token requests, 16 q heads, 16 index heads, top-k 16).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...     # the fp64 CPU oracle arm

Prints one JSON line (rank 0). Under torchrun every rank runs its own replica
of the workload (the step shards by request; there is no exchange), so the
aggregate rows/s is weak-scaled.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("sparse-attn+index rows/s and achieved HBM GB/s vs ~8 TB/s peak, bs8 mixed ctx")
SM_SCALE = 1.0 / math.sqrt(128)
ROTARY_DIM = 64       # --write-path fused / staged: rotated dims per head
NORM_EPS = 1e-6       # and the RMSNorm epsilon
FALLBACK_BF16_TFLOPS = 1900.0
FALLBACK_HBM_GBS = 6800.0


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="skewed",
                    choices=["tiny", "decode", "verify", "skewed", "prefill"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-workload", action="store_true",
                    help="measure the headline workload only (default: all five, the others "
                         "reported under per_workload)")
    ap.add_argument("--topk-path", choices=["fused", "call", "pair"], default="fused",
                    help="decode rows: fused = m3s_index_attention (the scorer leaves per-CTA "
                         "candidates, the attention merges them: two launches); call = "
                         "m3s_index_score_topk then m3s_sparse_attention; pair = "
                         "m3s_index_block_scores, m3s_block_topk, m3s_sparse_attention. The scorer "
                         "and the attention are timed alone through the pair calls either way")
    ap.add_argument("--verify-path", choices=["call", "fused"], default="call",
                    help="verify and prefill rows: call = m3s_verify_score_topk then "
                         "m3s_sparse_attention (measured faster on the verify batch, equal on "
                         "prefill); fused = m3s_verify_index_attention (the verify scorer leaves "
                         "per-CTA candidates, the attention merges them: two launches)")
    ap.add_argument("--cache-format", choices=["nvfp4", "mxfp4"], default="nvfp4",
                    help="K / V / index-K record format")
    ap.add_argument("--write-path", choices=["store", "fused", "staged"], default="store",
                    help="store: the step's rows arrive normalised and are stored; fused: they "
                         "arrive before RMSNorm / RoPE and one quantise-at-write launch normalises, "
                         "rotates and stores them; staged: the same normalisation writes BF16 "
                         "staging rows that the batched store then quantises (the unfused path)")
    ap.add_argument("--oracle-leg", action="store_true", help=argparse.SUPPRESS)
    ap.add_argument("--oracle-reps", type=int, default=2, help=argparse.SUPPRESS)
    ap.add_argument("--oracle-procs", type=int, default=1, help=argparse.SUPPRESS)
    return ap.parse_args()


def peaks():
    """(HBM GB/s, dense bf16 TFLOP/s burst, source): the pool's measured figures,
    else the fallback ones. f16 tensor-core products run at the bf16 rate."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


# DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) per launch of the
# dominant kernel, from one ncu capture of this bench's workload (summary under
# profiles/). It is reported only while the kernel's sources hash to what was
# captured; after a change to the kernel it is null until the counters are
# taken again. (The hashes moved once without a new capture: the removal of
# device helpers no kernel called, with every kernel's registers, shared
# memory and stack as ptxas reported them before.)
NCU_TRAFFIC = {
    ("skewed", "score_decode_kernel"): {
        "bytes": 110_826_496 + 3_570_688,
        "sources": {"m3s_score_mma.cu": "e33f51210c0f3b77",
                    "m3s_score_common.cuh": "fd432d016e7fe20e",
                    "m3s_device.cuh": "8c6b356f0523f4a3"},
    },
    ("skewed-mxfp4", "score_decode_kernel"): {
        "bytes": 104_680_960 + 3_654_400,
        "sources": {"m3s_score_mma.cu": "e33f51210c0f3b77",
                    "m3s_score_common.cuh": "fd432d016e7fe20e",
                    "m3s_device.cuh": "8c6b356f0523f4a3"},
    },
    ("verify", "score_kernel"): {
        "bytes": 143_932_160 + 3_994_368,
        "sources": {"m3s_score.cu": "0e6af4207f397d38",
                    "m3s_score_common.cuh": "fd432d016e7fe20e",
                    "m3s_device.cuh": "8c6b356f0523f4a3"},
    },
}


def ncu_traffic(workload, kernel):
    import hashlib
    rec = NCU_TRAFFIC.get((workload, kernel))
    if rec is None:
        return None
    csrc = os.path.join(os.path.dirname(os.path.abspath(__file__)), "nvfp4_block_sparse_m3s_gb300",
                        "csrc")
    for name, digest in rec["sources"].items():
        try:
            with open(os.path.join(csrc, name), "rb") as f:
                if hashlib.sha256(f.read()).hexdigest()[:16] != digest:
                    return None
        except OSError:
            return None
    return rec["bytes"]


# --------------------------------------------------------------------------
# Multi-rank aggregation (one process per GPU; every rank runs its own copy of
# the workload, so per-rank work is fixed as ranks are added: weak scaling)
# --------------------------------------------------------------------------

def max_over_ranks(values, device="cpu"):
    """Each value's maximum over all ranks (unchanged without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def job_rows_per_s(world: int, rows_per_rank: int, ms: float) -> float:
    """Whole-job throughput: the rows every rank processed / the slowest rank's time."""
    return world * rows_per_rank / (ms * 1e-3)


#: the scorers' CTA bound: a score + top-k call with more query tiles than this
#: streams its top-k inside the scorer (one launch), else it launches the scorer
#: and then the top-k
MAX_GRID = 256

#: bytes per token and head of a K, V or index-K record
RECORD_BYTES = {"nvfp4": 72, "mxfp4": 68}


def workload_config(spec, ntok, fmt="nvfp4"):
    mx = fmt == "mxfp4"
    return {
        "workload": spec.description,
        "name": spec.name,
        "requests": spec.batch,
        "rows": spec.rows,
        "cached_tokens": ntok,
        "q_heads": spec.hq,
        "kv_heads": spec.hkv,
        "index_heads": spec.hi,
        "topk": spec.topk,
        "cache_format": ("MXFP4 (e2m1 + E8M0 per 32), 68 B per token and head" if mx else
                         "NVFP4 (e2m1 + E4M3 per 16), 72 B per token and head"),
        "arithmetic": ("MXFP4 index keys decoded exactly to f16 (per-key exponent normalisation), "
                       "f16 x f16 tensor-core products; K/V decoded exactly to bf16, bf16 x bf16 "
                       "products; f32 accumulation" if mx else
                       "NVFP4 decoded exactly to f16, f16 x f16 tensor-core products, f32 accumulation"),
        "l2": "flushed between timed steps: a 2 x L2 scratch written then read, outside the timed events",
    }


# --------------------------------------------------------------------------
# The CPU oracle arm (also the cpu_baseline samples)
# --------------------------------------------------------------------------

def _oracle_request(spec_name: str, fmt: str, b: int):
    """The oracle's resident cache of request b (setup, untimed): the pool's
    planes with the request's tokens stored, its source rows and step inputs."""
    import numpy as np

    from nvfp4_block_sparse_m3s_gb300 import workloads as W
    from oracle import m3s_oracle as O

    wl = W.make(spec_name, with_cache_src=False)
    s = wl.spec
    L = int(wl.seq_len[b])
    t0, t1 = int(wl.tok_off[b]), int(wl.tok_off[b + 1])
    qb = int(wl.cu_q[b + 1] - wl.cu_q[b])
    r0 = int(wl.cu_q[b])
    mx = fmt == "mxfp4"
    planes = {}
    srcs = {}
    for name, h in (("k", s.hkv), ("v", s.hkv), ("ik", 1)):
        c, sc = O.new_planes(wl.num_pages, h, mx=mx)
        src = W.bf16_tensor(s.seed, name, (wl.ntok, h, 128), s.n_out, s.out_factor, rows=(t0, t1))
        O.nvfp4_store(src, wl.slot_all[t0:t1], c, sc)          # the resident cache
        planes[name], srcs[name] = (c, sc), src
    new = wl.new_tok[(wl.new_tok >= t0) & (wl.new_tok < t1)] - t0   # this step's rows of b
    return {"wl": wl, "b": b, "L": L, "t0": t0, "qb": qb, "r0": r0, "planes": planes,
            "srcs": srcs, "new": new}


def _oracle_step(st, rows):
    """One timed oracle step of request ``st`` restricted to its local rows
    ``rows``: their new K / V / index-K rows stored, the request's row map,
    score + top-k and attention for those rows. Returns (seconds, causal keys)."""
    import numpy as np

    from oracle import m3s_oracle as O

    wl, b, qb, r0, t0 = st["wl"], st["b"], st["qb"], st["r0"], st["t0"]
    s = wl.spec
    (kc, ks), (vc, vs), (ic, is_) = st["planes"]["k"], st["planes"]["v"], st["planes"]["ik"]
    cu = np.array([0, qb], dtype=np.int32)
    seq = np.array([st["L"]], dtype=np.int32)
    bt = wl.block_table[b: b + 1]
    new = st["new"]
    new = new[np.array(rows)] if len(new) == qb else new
    q_idx, wgt, q = wl.q_idx[r0: r0 + qb], wl.w[r0: r0 + qb], wl.q[r0: r0 + qb]
    t = time.perf_counter()
    for name, (c, sc) in st["planes"].items():
        O.nvfp4_store(st["srcs"][name][new], wl.slot_all[t0 + new], c, sc)
    rr, rl = O.decode_rows(cu, seq, qb)
    ids, _, _ = O.index_score_topk(q_idx, wgt, ic, is_, bt, rr, rl, s.topk, rows=rows)
    O.sparse_attention(q, s.hkv, kc, ks, vc, vs, bt, rr, rl, ids, SM_SCALE, rows=rows)
    dt = time.perf_counter() - t
    return dt, int(sum(int(rl[r]) for r in rows))


def _spread(n_all: int, n: int):
    """At most n indices in [0, n_all), evenly spaced, the last one included."""
    n = max(1, min(n, n_all))
    return sorted({int(round(i * (n_all - 1) / max(1, n - 1))) for i in range(n)} | {n_all - 1})


def _batch_keys(spec_name: str) -> float:
    import numpy as np

    from nvfp4_block_sparse_m3s_gb300 import workloads as W
    from oracle import m3s_oracle as O

    wl = W.make(spec_name, with_cache_src=False)
    _, rl = O.decode_rows(wl.cu_q, wl.seq_len, wl.spec.rows)
    return float(np.sum(rl.astype(np.float64)))


def oracle_steps(spec_name: str, warm: int, steps: int, fmt: str = "nvfp4", cap_s: float = float("inf")):
    """Time the oracle's step for a bounded sample of the workload, on one core.

    The sample is the last request's step restricted to at most 8 of its
    rows, evenly spaced and always including its last row. The whole batch's
    step is extrapolated from it by the ratio of causal keys scored (scoring
    dominates the oracle's time). The request's resident cache is set up once
    (untimed); then ``warm`` untimed and ``steps`` timed sample steps run on it
    (storing a step's rows again writes the same bytes), the timed loop
    stopping early once ``cap_s`` seconds have passed.
    Returns (seconds of each timed sample step, description, rows in the
    batch, scale).
    """
    from nvfp4_block_sparse_m3s_gb300 import workloads as W

    spec = W.SPECS[spec_name]
    b = spec.batch - 1
    st = _oracle_request(spec_name, fmt, b)
    sample = _spread(st["qb"], 8)
    for _ in range(warm):
        _oracle_step(st, sample)
    times, keys = [], 0
    t0 = time.perf_counter()
    while len(times) < max(1, steps) and (not times or time.perf_counter() - t0 < cap_s):
        dt, keys = _oracle_step(st, sample)
        times.append(dt)
    scale = _batch_keys(spec_name) / keys
    desc = (f"oracle step of {len(sample)} of the {st['qb']} row(s) of request {b} ({st['L']} cached"
            f" tokens), scaled by causal keys x{scale:.2f} to the batch of {spec.rows} rows")
    return times, desc, spec.rows, scale


def oracle_sample(spec_name: str, reps: int, fmt: str = "nvfp4"):
    """The best of ``reps`` timed sample steps (``oracle_steps``)."""
    times, desc, rows, scale = oracle_steps(spec_name, 0, reps, fmt)
    return min(times), desc + f"; timed {len(times)}x (best)", rows, scale


def oracle_units(spec_name: str, n: int):
    """A sample of the workload cut into at most n units of work, one per
    process: one request per unit (up to 8 of its rows, evenly spaced) while the
    batch has at least n requests, else the last request's rows spread over
    the units (two rows each)."""
    from nvfp4_block_sparse_m3s_gb300 import workloads as W

    spec = W.SPECS[spec_name]
    B = spec.batch
    if B >= n or spec.q_rows[-1] < 2:
        return [(b, _spread(spec.q_rows[b], 8)) for b in range(max(0, B - n), B)]
    rows = _spread(spec.q_rows[-1], 2 * n)
    return [(B - 1, rows[i::n]) for i in range(n) if rows[i::n]]


def _oracle_unit_proc(spec_name, fmt, b, rows, barrier, out_q):
    """One process of the multi-core oracle leg: set up, wait for the others,
    time its unit."""
    st = _oracle_request(spec_name, fmt, b)
    barrier.wait(timeout=900)
    dt, keys = _oracle_step(st, rows)
    out_q.put((b, len(rows), dt, keys))


def oracle_multicore(spec_name: str, procs: int, fmt: str = "nvfp4"):
    """The oracle on several host cores: the units of ``oracle_units`` each in
    their own process (spawned, one BLAS thread each), set up in parallel, then
    timed together after a barrier. The parallel time is the slowest unit's; the
    batch is extrapolated from the sampled units by causal keys."""
    import multiprocessing as mp

    units = oracle_units(spec_name, procs)
    ctx = mp.get_context("spawn")
    barrier = ctx.Barrier(len(units))
    out_q = ctx.Queue()
    ps = [ctx.Process(target=_oracle_unit_proc, args=(spec_name, fmt, b, rows, barrier, out_q))
          for b, rows in units]
    for p in ps:
        p.start()
    res = [out_q.get(timeout=1800) for _ in ps]
    for p in ps:
        p.join()
    t_par = max(r[2] for r in res)
    keys = sum(r[3] for r in res)
    nrows = sum(r[1] for r in res)
    scale = _batch_keys(spec_name) / keys
    desc = (f"{len(units)} processes, one unit each ({nrows} sampled rows over "
            f"{len(set(r[0] for r in res))} request(s)), timed together after a barrier: the "
            f"slowest unit's time, scaled by causal keys x{scale:.2f} to the batch")
    return t_par, desc, len(units), scale


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_oracle_leg(args):
    from nvfp4_block_sparse_m3s_gb300 import workloads as W
    rows = W.SPECS[args.workload].rows
    if args.oracle_procs > 1:
        t, desc, cores, scale = oracle_multicore(args.workload, args.oracle_procs, args.cache_format)
    else:
        t, desc, _, scale = oracle_sample(args.workload, args.oracle_reps, args.cache_format)
        cores = 1
    print(json.dumps({"seconds_per_sample": t, "sample": desc, "rows": rows, "scale": scale,
                      "value": rows / (t * scale), "cores": cores}))


def cpu_baseline(workload: str, reps: int = 2, fmt: str = "nvfp4", procs: int = 1):
    """The oracle leg in a child process (one BLAS thread per process)."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-leg", "--workload",
                        workload, "--oracle-reps", str(reps), "--cache-format", fmt,
                        "--oracle-procs", str(procs)],
                       capture_output=True, text=True, env=env, timeout=1800)
    if r.returncode != 0:
        return {"error": r.stderr.strip().splitlines()[-1] if r.stderr.strip() else "failed"}
    d = json.loads(r.stdout.strip().splitlines()[-1])
    return {"value": d["value"], "unit": "rows/s", "cores": d["cores"], "kind": "oracle",
            "sample": d["sample"]}


def run_reference(args):
    """The oracle as it stands, timed on the host cores (rank 0 only)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    # one core, as the line states: numpy's BLAS pool is sized from these when
    # numpy is first imported, which happens below
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        os.environ[var] = "1"
    from nvfp4_block_sparse_m3s_gb300 import workloads as W
    spec = W.SPECS[args.workload]
    steps, warm = max(1, args.steps), max(0, args.warmup)
    # each step is one bounded sample (one request's step), extrapolated to the
    # batch: W untimed samples, then K timed ones (the timed loop stops after
    # two minutes; steps reports the samples taken), the median reported
    samples, desc, rows, scale = oracle_steps(args.workload, warm, steps, args.cache_format, cap_s=120.0)
    t_med = float(sorted(samples)[len(samples) // 2])
    value = rows / (t_med * scale)
    ms = t_med * scale * 1e3
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "rows/s",
            "n_gpus": args.gpus, "steps": len(samples), "warmup": warm, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": workload_config(spec, int(sum(spec.ctx)), args.cache_format),
            "cpu_baseline": {"value": value, "unit": "rows/s", "cores": 1, "kind": "oracle",
                             "sample": desc + f"; {len(samples)} timed samples, the median"},
            "e2e": {"value": value, "unit": "rows/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


# --------------------------------------------------------------------------
# Our arm
# --------------------------------------------------------------------------

class Clocks:
    """SM clock and clock-event reasons sampled through NVML (ctypes) in a thread
    every 2 ms while the timed region runs; nvidia-smi is the fallback."""

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, torch_device):
        import ctypes
        import threading
        self.ct = ctypes
        self.threading = threading
        self.samples = []
        self.max_mhz = None
        self.h = None
        self.err = None
        try:
            lib = ctypes.CDLL("libnvidia-ml.so.1")
            if lib.nvmlInit_v2() != 0:
                raise RuntimeError("nvmlInit failed")
            h = ctypes.c_void_p()
            import torch
            props = torch.cuda.get_device_properties(torch_device)
            ok = False
            uuid = getattr(props, "uuid", None)
            if uuid is not None:
                ok = lib.nvmlDeviceGetHandleByUUID(f"GPU-{uuid}".encode(), ctypes.byref(h)) == 0
            if not ok and hasattr(props, "pci_bus_id"):
                bus = f"{getattr(props, 'pci_domain_id', 0):08X}:{props.pci_bus_id:02X}:" \
                      f"{getattr(props, 'pci_device_id', 0):02X}.0"
                ok = lib.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)) == 0
            if not ok:
                ok = lib.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(h)) == 0
            if not ok:
                raise RuntimeError("no NVML handle")
            self.lib, self.h = lib, h
            m = ctypes.c_uint()
            if lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(m)) == 0:
                self.max_mhz = float(m.value)
            self.reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                lib.nvmlDeviceGetCurrentClocksThrottleReasons
        except Exception as e:  # no NVML on this machine
            self.err = str(e)

    def _run(self):
        ct = self.ct
        c = ct.c_uint()
        r = ct.c_ulonglong()
        while not self.stop_flag:
            if self.lib.nvmlDeviceGetClockInfo(self.h, 1, ct.byref(c)) == 0:
                rv = r.value if self.reasons_fn(self.h, ct.byref(r)) == 0 else 0
                self.samples.append((float(c.value), int(rv)))
            time.sleep(0.002)

    def start(self):
        self.stop_flag = False
        if self.h is not None:
            self.t = self.threading.Thread(target=self._run, daemon=True)
            self.t.start()

    def stop(self):
        self.stop_flag = True
        if self.h is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [f"NVML unavailable: {self.err}"]}
        self.t.join()
        sm = sorted(v for v, _ in self.samples)
        reasons = set()
        for _, bits in self.samples:
            for b, n in self.REASONS.items():
                if bits & b:
                    reasons.add(n)
        return {"sm_mhz": sm[len(sm) // 2] if sm else None, "sm_max_mhz": self.max_mhz,
                "reasons": sorted(reasons), "samples": len(sm),
                "source": "NVML, 2 ms sampling during the timed region"}


def measure_workload(name, args, dev, world):
    """One workload on this rank's GPU: its cache made resident by our store
    (untimed), then the step timed as one CUDA graph, the scorer and the
    attention timed from the same graph with event nodes around them, one graph
    per phase for the breakdown, and the step end to end from pinned host
    memory, both replayed as one graph and called eagerly through the C ABI.
    Returns the workload's figures; frees its device memory on return."""
    import numpy as np
    import torch

    from nvfp4_block_sparse_m3s_gb300 import binding as M
    from nvfp4_block_sparse_m3s_gb300 import workloads as W

    spec = W.SPECS[name]
    wl = W.make(spec)
    s = wl.spec
    R = s.rows
    fused = s.name in ("verify", "prefill")
    mx = args.cache_format == "mxfp4"
    rec_bytes = RECORD_BYTES[args.cache_format]

    def bf16(x):
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).to(dev).view(torch.bfloat16)

    # ---- resident cache: planes filled by our store (setup, untimed) ----
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    kc, ks = M.new_plane(wl.num_pages, s.hkv, dev, mx=mx)
    vc, vs = M.new_plane(wl.num_pages, s.hkv, dev, mx=mx)
    ic, is_ = M.new_plane(wl.num_pages, 1, dev, mx=mx)
    slot_all = torch.from_numpy(wl.slot_all).to(dev)
    for src, c, sc in ((wl.k_src, kc, ks), (wl.v_src, vc, vs), (wl.ik_src, ic, is_)):
        t = bf16(src)
        M.m3s_nvfp4_store(t, slot_all, c, sc, err)
        del t
    del slot_all
    torch.cuda.synchronize()
    new = wl.new_tok
    host_in = {
        "k_new": np.ascontiguousarray(wl.k_src[new]), "v_new": np.ascontiguousarray(wl.v_src[new]),
        "ik_new": np.ascontiguousarray(wl.ik_src[new]), "slots": wl.slot_all[new].copy(),
        "q": wl.q, "q_idx": wl.q_idx, "w": wl.w, "cu_q": wl.cu_q, "seq_len": wl.seq_len,
    }
    write_path = args.write_path
    if write_path != "store":
        # the same seeded rows taken as the pre-normalisation ones; RMSNorm weights
        # U(0.5, 1.5) per tensor, RoPE over the first ROTARY_DIM dims at each new
        # token's position (10000^(-i / (ROTARY_DIM / 2)) frequencies)
        wrng = np.random.default_rng(s.seed + 101)
        for k in ("wq", "wk", "wik"):
            host_in[k] = (wrng.random(128) + 0.5).astype(np.float32)
        pos = np.zeros(R, dtype=np.float64)   # row j of request b sits at seq_len - Q_b + j
        for b in range(len(wl.seq_len)):
            qb = int(wl.cu_q[b + 1] - wl.cu_q[b])
            pos[int(wl.cu_q[b]): int(wl.cu_q[b]) + qb] = int(wl.seq_len[b]) - qb + np.arange(qb)
        half = ROTARY_DIM // 2
        ang = pos[:, None] * (10000.0 ** (-np.arange(half) / half))[None, :]
        host_in["cos"] = np.cos(ang).astype(np.float32)
        host_in["sin"] = np.sin(ang).astype(np.float32)
    del wl.k_src, wl.v_src, wl.ik_src
    # The step's inputs live in one device buffer (each tensor at a 256-byte
    # aligned offset) mirrored by one pinned host buffer, so the end-to-end run
    # moves them with a single host-to-device copy; the outputs likewise.
    in_off, in_bytes = {}, 0
    for k, v in host_in.items():
        in_off[k] = in_bytes
        in_bytes += (v.nbytes + 255) // 256 * 256
    dev_in = torch.zeros(in_bytes, dtype=torch.uint8, device=dev)
    pin_in = torch.zeros(in_bytes, dtype=torch.uint8).pin_memory()
    d = {}
    for k, v in host_in.items():
        v = np.ascontiguousarray(v)
        pin_in[in_off[k]: in_off[k] + v.nbytes].copy_(torch.from_numpy(v.view(np.uint8).reshape(-1)))
        tdt = {np.dtype(np.uint16): torch.bfloat16, np.dtype(np.int32): torch.int32,
               np.dtype(np.int64): torch.int64, np.dtype(np.float32): torch.float32}[v.dtype]
        d[k] = dev_in[in_off[k]: in_off[k] + v.nbytes].view(tdt).view(v.shape)
    dev_in.copy_(pin_in)
    bt = torch.from_numpy(wl.block_table).to(dev)
    B, bt_stride = bt.shape
    row_req = torch.empty(R, dtype=torch.int32, device=dev)
    row_len = torch.empty(R, dtype=torch.int32, device=dev)
    out_shapes = {"out": ((R, s.hq, 128), torch.bfloat16, 2), "ids": ((R, s.topk), torch.int32, 4)}
    out_off, out_bytes = {}, 0
    for k, (shape, _, es) in out_shapes.items():
        out_off[k] = out_bytes
        out_bytes += (int(np.prod(shape)) * es + 255) // 256 * 256
    dev_out = torch.zeros(out_bytes, dtype=torch.uint8, device=dev)
    if write_path != "store":
        q_n = torch.empty_like(d["q"])            # the step's normalised, rotated queries
        qidx_n = torch.empty_like(d["q_idx"])
        staging = {k: torch.empty_like(d[k]) for k in ("k_new", "v_new", "ik_new")}

    def out_view(k):
        shape, dt, es = out_shapes[k]
        n = int(np.prod(shape)) * es
        return dev_out[out_off[k]: out_off[k] + n].view(dt).view(shape)
    ids = out_view("ids")
    out = out_view("out")
    bscores = torch.empty((R, bt_stride), dtype=torch.float32, device=dev)
    lse = torch.empty((R, s.hq), dtype=torch.float32, device=dev)
    # workspaces (zeroed once at allocation)
    ws_i = torch.zeros(max(16, M.m3s_workspace_bytes(M.OP_INDEX_SCORE_TOPK, R, B, bt_stride, 0, 0,
                                                     s.hi, s.topk, 1)),
                       dtype=torch.uint8, device=dev)
    ws_v = torch.zeros(max(16, M.m3s_workspace_bytes(M.OP_VERIFY_SCORE_TOPK, R, B, bt_stride, 0, 0,
                                                     s.hi, s.topk, max(s.q_rows))),
                       dtype=torch.uint8, device=dev)
    ws_a = torch.zeros(max(16, M.m3s_workspace_bytes(M.OP_SPARSE_ATTENTION, R, B, bt_stride, s.hq,
                                                     s.hkv, 0, s.topk)),
                       dtype=torch.uint8, device=dev)
    ws_ia = torch.zeros(max(16, M.m3s_workspace_bytes(M.OP_INDEX_ATTENTION, R, B, bt_stride, s.hq,
                                                      s.hkv, s.hi, s.topk)),
                        dtype=torch.uint8, device=dev)
    ws_via = torch.zeros(max(16, M.m3s_workspace_bytes(M.OP_VERIFY_INDEX_ATTENTION, R, B, bt_stride, s.hq,
                                                       s.hkv, s.hi, s.topk, max(s.q_rows))),
                         dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def pre():
        # the step's writes and its row map: the batched store with the row map
        # in the same launch, or the row map chained before the quantise-at-write
        # (a fork / join on two streams would cost a full graph edge)
        if write_path == "store":
            M.m3s_nvfp4_store_batch_rows([(d["k_new"], kc, ks), (d["v_new"], vc, vs),
                                          (d["ik_new"], ic, is_)], d["slots"], d["cu_q"], d["seq_len"], R,
                                         row_req, row_len, err)
        else:
            M.m3s_decode_rows(d["cu_q"], d["seq_len"], R, row_req, row_len)
            fused_w = write_path == "fused"
            dst = {"k_new": (kc, ks), "v_new": (vc, vs), "ik_new": (ic, is_)} if fused_w else staging
            M.m3s_qk_norm_rope_store(
                [(d["q"], d["wq"], True, q_n), (d["k_new"], d["wk"], True, dst["k_new"]),
                 (d["v_new"], None, False, dst["v_new"]), (d["q_idx"], None, True, qidx_n),
                 (d["ik_new"], d["wik"], True, dst["ik_new"])],
                d["slots"], d["cos"], d["sin"], ROTARY_DIM, NORM_EPS, err)
            if not fused_w:
                M.m3s_nvfp4_store_batch([(staging["k_new"], kc, ks), (staging["v_new"], vc, vs),
                                         (staging["ik_new"], ic, is_)], d["slots"], err)

    q_in = d["q"] if write_path == "store" else q_n
    qidx_in = d["q_idx"] if write_path == "store" else qidx_n
    path = getattr(args, "topk_path", "fused")
    vpath = getattr(args, "verify_path", "call")

    def score():   # the verify rows' fused score + top-k
        M.m3s_verify_score_topk(qidx_in, d["w"], ic, is_, bt, d["cu_q"], row_len,
                                max(s.q_rows), s.topk, ids, ws_v, err)

    def score_pair():
        M.m3s_index_block_scores(qidx_in, d["w"], ic, is_, bt, row_req, row_len, bscores, err)

    def score_call():
        M.m3s_index_score_topk(qidx_in, d["w"], ic, is_, bt, row_req, row_len, s.topk, ids,
                               None, ws_i, err)

    def index_attention():
        M.m3s_index_attention(qidx_in, d["w"], ic, is_, q_in, s.hkv, kc, ks, vc, vs, bt, row_req,
                              row_len, s.topk, SM_SCALE, ids, out, lse, ws_ia, err)

    def verify_index_attention():
        M.m3s_verify_index_attention(qidx_in, d["w"], ic, is_, q_in, s.hkv, kc, ks, vc, vs, bt, d["cu_q"],
                                     row_req, row_len, max(s.q_rows), s.topk, SM_SCALE, ids, out, lse,
                                     ws_via, err)

    def topk():
        M.m3s_block_topk(bscores, row_req, row_len, B, bt_stride, s.topk, ids)

    def attn():
        M.m3s_sparse_attention(q_in, s.hkv, kc, ks, vc, vs, bt, row_req, row_len, ids, SM_SCALE,
                               out, lse, ws_a, err)

    # eager warm-up (sets kernel attributes), then the whole step as one CUDA
    # graph (the timed step), and the same work as separate calls with
    # event-record nodes around the scorer and around the attention (an event
    # node between two kernels breaks their programmatic-launch overlap, so this
    # copy times those two kernels and not the step); one graph per separate
    # call for the breakdown
    if fused and vpath == "fused":
        phases = [pre, verify_index_attention]
        timing, score_fn = [pre, score, attn], score
    elif fused:
        phases = [pre, score, attn]
        timing, score_fn = phases, score
    elif path == "fused":
        phases = [pre, index_attention]
        timing, score_fn = [pre, score_pair, topk, attn], score_pair
    elif path == "pair":
        phases = [pre, score_pair, topk, attn]
        timing, score_fn = phases, score_pair
    else:
        phases = [pre, score_call, attn]
        timing, score_fn = phases, score_call
    for _ in range(2):
        for fn in phases + timing:
            fn()
    torch.cuda.synchronize()
    cap = torch.cuda.Stream(device=dev)
    graphs = []
    for fn in timing:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            fn()
        graphs.append(g)
    try:
        sev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(4)]
    except TypeError:   # a torch without event-record nodes in graphs
        sev = None
    whole = whole_ev = None
    if sev is not None:
        whole = torch.cuda.CUDAGraph()
        with torch.cuda.graph(whole, stream=cap):
            for fn in phases:
                fn()
        whole_ev = torch.cuda.CUDAGraph()
        with torch.cuda.graph(whole_ev, stream=cap):
            for fn in timing:
                if fn is score_fn:
                    sev[0].record()
                if fn is attn:
                    sev[2].record()
                fn()
                if fn is score_fn:
                    sev[1].record()
                if fn is attn:
                    sev[3].record()
    torch.cuda.synchronize()

    def step(phase_events=None):
        # phase_events: len(timing)+1 events bracketing each separate call's graph
        if whole is not None and phase_events is None:
            whole.replay()
            return
        for i, g in enumerate(graphs):
            if phase_events:
                phase_events[i].record(stream)
            g.replay()
        if phase_events:
            phase_events[-1].record(stream)

    # our kernels per step: store (or quantise-at-write; staged: + the store), row
    # map, then the scorer call's kernels and the attention (fused: the scorer and
    # the attention, no top-k launch)
    ntiles = B * ((max(s.q_rows) + 7) // 8) if fused else R
    streams = (fused or path == "call") and ntiles > MAX_GRID
    pre_launches = {"store": 1, "fused": 2, "staged": 3}[write_path]
    if (vpath if fused else path) == "fused":   # the scorer, then the attention merging its candidates
        launches_per_step = pre_launches + 2
    elif not fused and path == "pair":
        launches_per_step = pre_launches + 3
    else:
        launches_per_step = pre_launches + (1 if streams else 2) + 1

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush_buf = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)

    def flush():
        # evict the workload from L2: write a buffer larger than L2, then read it
        # back so the lines left in L2 are clean (no write-backs inside the timed step)
        flush_buf.fill_(1)
        flush_buf.max()

    warm = max(3, args.warmup)
    for _ in range(warm):
        step()
        flush()
    torch.cuda.synchronize()
    assert int(err.item()) == 0, f"device error bits {int(err.item())}"

    # algorithmic bytes (what the method must move)
    ids_h = ids.cpu().numpy()
    req_h = row_req.cpu().numpy()
    distinct = 0
    for b in range(B):
        sel = ids_h[req_h == b]
        distinct += len(set(int(x) for x in sel.ravel() if x >= 0))
    keys = int(np.sum(host_in["seq_len"].astype(np.int64)))
    rl = row_len.cpu().numpy().astype(np.int64)
    score_bytes = keys * rec_bytes + R * s.hi * (256 + 4) + R * s.topk * 4
    attn_bytes = distinct * 128 * 2 * rec_bytes * s.hkv + R * s.hq * 256 * 2
    store_bytes = R * (2 * s.hkv + 1) * (256 + rec_bytes)
    if write_path != "store":   # the queries read and written back normalised / rotated
        store_bytes += R * (s.hq + s.hi) * 256 * 2
    step_bytes = score_bytes + attn_bytes + store_bytes + R * 8

    # ---- timed region (device time, per step, L2 flushed between steps) ----
    import torch.distributed as dist
    clocks = Clocks(dev)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    pev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)]
           for _ in range(args.steps)]
    for i in range(args.steps):
        flush()
        pev[i][0].record(stream)
        step()
        pev[i][-1].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if world > 1:
        dist.barrier()
    ms = sum(e[0].elapsed_time(e[-1]) for e in pev) / args.steps
    # the scorer's and the attention's durations: the step graph with event
    # nodes; the in-graph events are re-recorded by every replay, so each step
    # is read back before the next one
    score_l, attn_l = [], []
    if whole_ev is not None:
        for i in range(args.steps):
            flush()
            whole_ev.replay()
            torch.cuda.synchronize()
            score_l.append(sev[0].elapsed_time(sev[1]))
            attn_l.append(sev[2].elapsed_time(sev[3]))
    # per-phase breakdown (one graph per phase, events between them; not the
    # headline: the graph boundaries add launch gaps the whole-step graph has not)
    ph_ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(timing) + 1)]
             for _ in range(args.steps)]
    for i in range(args.steps):
        flush()
        step(ph_ev[i])
    torch.cuda.synchronize()
    phase_ms = [sum(e[j].elapsed_time(e[j + 1]) for e in ph_ev) / args.steps
                for j in range(len(timing))]
    if not score_l:
        score_l = [phase_ms[timing.index(score_fn)]]
        attn_l = [phase_ms[timing.index(attn)]]
    score_ms = sum(score_l) / len(score_l)
    attn_ms = sum(attn_l) / len(attn_l)
    ms, score_ms, attn_ms = max_over_ranks([ms, score_ms, attn_ms], dev)
    assert int(err.item()) == 0, f"device error bits {int(err.item())}"

    # ---- end to end through the public API with host buffers ----
    # (every step's inputs from pinned host memory in one copy, its outputs back
    # in one copy; the bytes counted are the packed buffers, alignment included)
    pin_out = torch.empty(out_bytes, dtype=torch.uint8).pin_memory()
    h2d, d2h = in_bytes, out_bytes
    e2e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
    # (a) the copy in, the step and the copy out as one graph (one launch per
    # step, as a serving loop would replay it)
    e2e_graph = None
    if whole is not None:
        try:
            e2e_graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(e2e_graph, stream=cap):
                dev_in.copy_(pin_in, non_blocking=True)
                for fn in phases:
                    fn()
                pin_out.copy_(dev_out, non_blocking=True)
            for _ in range(warm):
                e2e_graph.replay()
            torch.cuda.synchronize()
        except RuntimeError:
            e2e_graph = None
            torch.cuda.synchronize()
    for i in range(args.steps):
        flush()
        e2e_ev[i][0].record(stream)
        if e2e_graph is not None:
            e2e_graph.replay()
        else:
            dev_in.copy_(pin_in, non_blocking=True)
            step()
            pin_out.copy_(dev_out, non_blocking=True)
        e2e_ev[i][1].record(stream)
    torch.cuda.synchronize()
    e2e_ms = sum(a.elapsed_time(b) for a, b in e2e_ev) / args.steps
    # (b) eager: every step calls the C-ABI entry points afresh through the
    # binding (host validation, tensor-map encode, launch), between the two
    # copies; the GPU is idle when the first event is recorded (host sync after
    # the flush), so the host's call overhead is inside the interval
    eager_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(args.steps)]
    for i in range(args.steps):
        flush()
        torch.cuda.synchronize()
        eager_ev[i][0].record(stream)
        dev_in.copy_(pin_in, non_blocking=True)
        for fn in phases:
            fn()
        pin_out.copy_(dev_out, non_blocking=True)
        eager_ev[i][1].record(stream)
        torch.cuda.synchronize()
    eager_ms = sum(a.elapsed_time(b) for a, b in eager_ev) / args.steps
    e2e_ms, eager_ms = max_over_ranks([e2e_ms, eager_ms], dev)
    assert int(err.item()) == 0, f"device error bits {int(err.item())}"

    hbm_peak, tc_peak, src = peaks()
    # the scorer's binding roofline: bytes at the HBM peak against f16 tensor-core
    # flops (every causal key x index head x 128-dim dot product) at the dense peak
    score_flops = float(np.sum(rl)) * s.hi * 128 * 2
    t_hbm = score_bytes / (hbm_peak * 1e9)
    t_tc = score_flops / (tc_peak * 1e12)
    if t_tc > t_hbm:
        bound, unit, peak = "tensor", "TFLOP/s", tc_peak
        achieved = score_flops / (score_ms * 1e-3) / 1e12
        peak_name = "bf16_tflops (f16 runs at the bf16 rate)"
    else:
        bound, unit, peak = "hbm", "GB/s", hbm_peak
        achieved = score_bytes / (score_ms * 1e-3) / 1e9
        peak_name = "hbm_gbs"
    psrc = (lambda nm: f"measured (MEASURED_PEAKS.json {nm})" if src == "measured" else "fallback")
    score_kernel = (("score_kernel<8> (m3s_verify_score_topk, top-k streamed inside)" if streams else
                     "score_kernel<8> + topk_kernel (m3s_verify_score_topk)") if fused else
                    ("score_decode_kernel (m3s_index_score_topk, top-k streamed inside)" if streams else
                     "score_decode_kernel + topk_kernel (m3s_index_score_topk)") if path == "call" else
                    "score_decode_kernel (timed alone through m3s_index_block_scores)")
    attn_gbs = attn_bytes / (attn_ms * 1e-3) / 1e9
    return {
        "name": s.name,
        "config": dict(workload_config(s, keys, args.cache_format), write_path=write_path),
        "rows": R,
        "ms_per_step": ms,
        "rows_per_s": job_rows_per_s(world, R, ms),
        "achieved_gbs_step": world * step_bytes / (ms * 1e-3) / 1e9,
        "algorithmic_bytes_per_step": step_bytes,
        "scorer": {"bound": bound, "achieved": achieved, "peak": peak, "unit": unit,
                   "frac": achieved / peak,
                   "traffic": ncu_traffic(s.name + ("-mxfp4" if mx else ""),
                                          "score_kernel" if fused else "score_decode_kernel"),
                   "kernel": score_kernel, "kernel_ms": score_ms, "bytes_per_launch": score_bytes,
                   "flops_per_launch": score_flops,
                   "hbm_gbs_achieved": score_bytes / (score_ms * 1e-3) / 1e9,
                   "peak_source": psrc(peak_name)},
        "attention": {"bound": "hbm", "achieved": attn_gbs, "peak": hbm_peak, "unit": "GB/s",
                      "frac": attn_gbs / hbm_peak, "kernel": "attention_kernel (m3s_sparse_attention)",
                      "kernel_ms": attn_ms, "bytes_per_launch": attn_bytes,
                      "peak_source": psrc("hbm_gbs")},
        "e2e": {"value": job_rows_per_s(world, R, e2e_ms), "unit": "rows/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "copies": ("pinned host <-> device, nodes of the step's graph" if e2e_graph is not None
                           else "pinned host <-> device, stream copies around the step graph")},
        "e2e_eager": {"value": job_rows_per_s(world, R, eager_ms), "unit": "rows/s",
                      "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                      "how": "every step calls the C-ABI entry points afresh between the pinned-host "
                             "copies; timed from an idle GPU, so host call overhead is included"},
        "gpu_launches": launches_per_step * args.steps,
        "step_graph": "one graph per step" if whole is not None else "one graph per phase",
        "phases_ms_separate_graphs": {fn.__name__: round(v, 5) for fn, v in zip(timing, phase_ms)},
        "clocks": clk,
        "warmup": warm,
    }


def run_ours(args):
    import torch
    import torch.distributed as dist

    from nvfp4_block_sparse_m3s_gb300 import binding as M

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    M.load()

    names = [args.workload]
    if not args.no_per_workload:
        names += [n for n in ("tiny", "decode", "verify", "skewed", "prefill") if n != args.workload]
    res = {}
    for n in names:
        res[n] = measure_workload(n, args, dev, world)
        torch.cuda.empty_cache()
    h = res[args.workload]
    mx = args.cache_format == "mxfp4"
    line = {
        "metric": METRIC,
        "value": h["rows_per_s"],
        "unit": "rows/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": h["warmup"],
        "ms_per_step": h["ms_per_step"],
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f16/bf16" if mx else "f16",
        "data": "synthetic",
        "config": h["config"],
        "achieved_gbs_step": h["achieved_gbs_step"],
        "algorithmic_bytes_per_step": h["algorithmic_bytes_per_step"],
        "roofline": h["scorer"],
        "attention_roofline": h["attention"],
        "e2e": h["e2e"],
        "e2e_eager": h["e2e_eager"],
        "gpu_launches": h["gpu_launches"],
        "step_graph": h["step_graph"],
        "phases_ms_separate_graphs": h["phases_ms_separate_graphs"],
        "clocks": h["clocks"],
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        procs = host_cores()
        for n in names:
            res[n]["cpu_baseline"] = cpu_baseline(n, fmt=args.cache_format)
            res[n]["cpu_baseline_multicore"] = cpu_baseline(n, reps=1, fmt=args.cache_format,
                                                            procs=procs)
        line["cpu_baseline"] = res[args.workload]["cpu_baseline"]
        line["cpu_baseline_multicore"] = res[args.workload]["cpu_baseline_multicore"]
    if len(names) > 1:
        keep = ("config", "rows", "ms_per_step", "rows_per_s", "achieved_gbs_step",
                "algorithmic_bytes_per_step", "scorer", "attention", "e2e", "e2e_eager",
                "phases_ms_separate_graphs", "clocks", "cpu_baseline", "cpu_baseline_multicore")
        line["per_workload"] = {n: {k: res[n][k] for k in keep if k in res[n]}
                                for n in names if n != args.workload}
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


def main():
    args = parse()
    if args.oracle_leg:
        run_oracle_leg(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()

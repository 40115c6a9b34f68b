#!/usr/bin/env python3
"""Benchmark of the batched speculative-sampling verify step.

Workload: B=256 sequences, K=8 draft positions, V=152064, bf16 logits, temperature 1, ragged
draft lengths uniform on 1..8, Zipf(1.1) log-prior + N(0,1) target logits, draft = target +
N(0, 0.5^2) (seeded, synthetic). One step = one verify call over the whole batch.

value     verified draft tokens per second (sum of draft lengths / verify time), whole job
          over all ranks, inputs resident in HBM, L2 flushed before each step (a 256 MiB write,
          then a 256 MiB read, so that no dirty line is left to write back).
e2e       the same metric through the host-buffer entry point spec_verify_host: host->device
          copy of the rows each sequence has, the verify call and the device->host copy of the
          outputs, all inside the timed region.
roofline  algorithmic bytes (the rows the outcome needs: target rows 0..a_b and draft rows
          0..min(a_b, L_b-1) of each sequence) per launch / mean kernel time, against the
          measured HBM peak.
cpu_baseline  the float64 oracle on the host cores over the same batch.

--impl reference times the oracle itself as the reference arm (rank 0 only).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verified draft tokens/sec and achieved HBM GB/s (% of roofline) at 1 GB300"
UNIT = "verified draft tokens/s"
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 256 << 20
L2_NOTE = ("flushed before each step (256 MiB write, then a 256 MiB read, outside the events: "
           "L2 starts cold and clean)")


class L2Flush:
    """Leaves L2 cold and clean before a timed step: a 256 MiB write evicts whatever the last
    step left, then a 256 MiB read of another buffer makes the write's dirty lines go back to HBM
    before the step starts (left dirty, their write-back ran inside the timed region and took
    HBM bandwidth from the step's reads: 154 against 146 us on the 256-sequence batch)."""

    def __init__(self):
        import torch
        from speculative_decoding_verification_33_gb300 import api
        self._api = api
        self.w = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device="cuda")
        self.r = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.int32, device="cuda")
        self.sink = torch.zeros(1, dtype=torch.int64, device="cuda")

    def __call__(self):
        self.w.zero_()
        self._api.hbm_read_probe(self.r, self.sink)


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cluster", type=int, default=0, help="CTAs per sequence (0 = library)")
    ap.add_argument("--workload", type=int, default=5, choices=[1, 2, 3, 4, 5],
                    help="synthetic workload (5 = B256 K8 V152064, the headline)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--l2-warm", action="store_true",
                    help="do not flush L2 between steps (small workloads then run from L2)")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--sample", type=int, default=16,
                    help="sequences per step of the reference arm")
    ap.add_argument("--kernel", choices=["verify", "draft_sample", "residual_topf", "lmhead",
                                         "verify_hidden"],
                    default="verify",
                    help="verify: the verify step (default); draft_sample / residual_topf: the "
                         "row kernels on the draft rows / draft positions of the same batch; "
                         "lmhead: the tensor-core LM head with its softmax statistics; "
                         "verify_hidden: the verify step from hidden states through that head")
    ap.add_argument("--head", default="head_B256_K8_V152064_d3584",
                    help="LM-head workload of --kernel lmhead")
    ap.add_argument("--no-legs", action="store_true",
                    help="default run: skip the row-kernel, LM-head and hidden-state legs that "
                         "are attached to the verify line")
    return ap.parse_args(argv)


def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


# ---------------------------------------------------------------------------------------------
# byte accounting
# ---------------------------------------------------------------------------------------------
def algorithmic_bytes(w, lens, acc) -> int:
    """Bytes of the rows the outcome needs: target rows 0..a_b, draft rows 0..min(a_b, L_b-1)
    (every draft row below L_b when top-F ids are requested), plus ids, lengths, uniforms and
    outputs."""
    rows = 0
    for L, a in zip(lens.tolist(), acc.tolist()):
        if a < 0:
            continue
        rows += a + 1
        if w.mode == "stochastic":
            rows += L if w.fanout else min(a, L - 1) + 1
    small = w.B * (4 * w.K + 4 + 4 * (w.K + 1) + 4 + 4 * (w.K + 1))
    return rows * w.V * w.elem_bytes + small


def top8_prepass(w) -> bool:
    """A bias set or top-F ids add the top-8 prepass over the draft rows before the verify
    kernel (the host entry point then stages the rows instead of reading them in place)."""
    return bool(w.mode == "stochastic" and (w.fanout or (w.beta < 1.0 and w.bias_k > 0)))


# the kernels of each route spec_verify can take (spec_verify_route), by build source key
ROUTE_NAMES = {0: "cluster walk", 1: "greedy rows", 2: "small batch, every row at once"}
ROUTE_SOURCES = {0: "verify", 1: "greedy", 2: "small"}


def input_bytes(w, lens) -> int:
    """Bytes of every row the sequences have (target 0..L_b, draft 0..L_b-1)."""
    rows = int(np.sum(lens + 1)) + (int(np.sum(lens)) if w.mode == "stochastic" else 0)
    return rows * w.V * w.elem_bytes


def host_copy_bytes(w, lens, acc=None, pinned=True):
    """Bytes spec_verify_host moves per call. With pinned rows and no top-8 prepass the kernel
    reads the rows in place: the rows the outcome needs (target 0..a_b, draft 0..min(a_b,
    L_b-1)) cross the host link once (the draw reads the decided position back from a device
    copy), plus the staged ids, lengths and uniforms. Otherwise it mirrors the per-sequence /
    whole-buffer staging."""
    B, K = w.B, w.K
    top8 = w.mode == "stochastic" and (w.fanout or (w.beta < 1.0 and w.bias_k > 0))
    if pinned and not top8 and acc is not None:
        rows = 0
        for L, a in zip(lens.tolist(), acc.tolist()):
            if a < 0:
                continue
            rows += a + 1 + (min(a, L - 1) + 1 if w.mode == "stochastic" else 0)
        h2d = rows * w.V * w.elem_bytes + B * K * 4 + B * 4
        if w.mode == "stochastic":
            h2d += B * (K + 1) * 4
        d2h = B * 4 + B * (K + 1) * 4
        return h2d, d2h
    need = int(np.sum(lens))
    per_seq = (2 * need + B) * 4 < 3 * B * (2 * K + 1)
    rows_t = int(np.sum(lens + 1)) if per_seq else B * (K + 1)
    rows_d = (need if per_seq else B * K) if w.mode == "stochastic" else 0
    h2d = (rows_t + rows_d) * w.V * w.elem_bytes + B * K * 4 + B * 4
    if w.mode == "stochastic":
        h2d += B * (K + 1) * 4
    d2h = B * 4 + B * (K + 1) * 4 + (B * K * max(w.fanout) * 4 if w.fanout else 0)
    return h2d, d2h


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, copy burst)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback (6.8 TB/s)"


def recorded_traffic(workload: str, digest: str):
    """DRAM bytes per launch from the committed ncu summary, if the kernel has not changed."""
    import glob
    for path in glob.glob(os.path.join(ROOT, "profiles", "*.md")):
        fields = {}
        with open(path) as f:
            for line in f:
                if ":" in line and line.startswith("- "):
                    k, v = line[2:].split(":", 1)
                    fields[k.strip()] = v.strip().strip("`")
        if fields.get("workload") == workload and fields.get("source_digest") == digest:
            try:
                return float(fields["dram_bytes_per_launch"]), os.path.basename(path)
            except (KeyError, ValueError):
                pass
    return None, None


# ---------------------------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------------------------
# multi-rank aggregation (weak scaling: every rank verifies its own batch)
# ---------------------------------------------------------------------------------------------
def aggregate(tokens: float, ms: float, group=None):
    """(sum of tokens over ranks, max of per-rank ms) -- plain values on a single rank."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return tokens, ms
    import torch
    dev = "cuda" if dist.get_backend(group) == "nccl" else "cpu"
    t = torch.tensor([tokens], dtype=torch.float64, device=dev)
    m = torch.tensor([ms], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM, group=group)
    dist.all_reduce(m, op=dist.ReduceOp.MAX, group=group)
    return float(t.item()), float(m.item())


def oracle_time(d, w, seqs):
    from oracle import verify as O
    t0 = time.perf_counter()
    res = O.verify_batch(d["target"], d["draft"] if w.mode == "stochastic" else None,
                         d["draft_tokens"], d["draft_lens"], d["uniforms"],
                         temperature=w.temperature, mode=w.mode, beta=w.beta, bias_k=w.bias_k,
                         fanout=w.fanout, seqs=seqs)
    return time.perf_counter() - t0, res


# The same oracle on every host core: sequences sharded over a spawned process pool that reads
# the batch from shared memory (the oracle itself is unchanged).
_POOL = {}


def _pool_attach(spec, w):
    from multiprocessing import shared_memory
    arrays, shms = {}, []
    for name, (shm_name, shape, dtype) in spec.items():
        shm = shared_memory.SharedMemory(name=shm_name)
        shms.append(shm)
        arrays[name] = np.ndarray(shape, dtype=np.dtype(dtype), buffer=shm.buf)
    _POOL.update(arrays=arrays, shms=shms, w=w)


def _pool_run(seqs):
    from oracle import verify as O
    a, w = _POOL["arrays"], _POOL["w"]
    O.verify_batch(a["target"], a["draft"] if w.mode == "stochastic" else None,
                   a["draft_tokens"], a["draft_lens"], a["uniforms"], temperature=w.temperature,
                   mode=w.mode, beta=w.beta, bias_k=w.bias_k, fanout=w.fanout, seqs=seqs)
    return len(seqs)


def oracle_pool_time(d, w, procs):
    import multiprocessing as mp
    from multiprocessing import shared_memory
    names = ("target", "draft", "draft_tokens", "draft_lens", "uniforms")
    shms, spec = [], {}
    try:
        for n in names:
            arr = np.ascontiguousarray(d[n])
            shm = shared_memory.SharedMemory(create=True, size=max(1, arr.nbytes))
            np.ndarray(arr.shape, dtype=arr.dtype, buffer=shm.buf)[...] = arr
            shms.append(shm)
            spec[n] = (shm.name, arr.shape, arr.dtype.str)
        parts = [p.tolist() for p in np.array_split(np.arange(w.B), procs) if len(p)]
        with mp.get_context("spawn").Pool(procs, initializer=_pool_attach,
                                          initargs=(spec, w)) as pool:
            pool.map(_pool_run, [[0]] * procs)  # imports and first touch, untimed
            t0 = time.perf_counter()
            pool.map(_pool_run, parts, chunksize=1)
            return time.perf_counter() - t0
    finally:
        for shm in shms:
            shm.close()
            shm.unlink()


# ---------------------------------------------------------------------------------------------
# reference arm: the oracle on the host cores
# ---------------------------------------------------------------------------------------------
def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    from speculative_decoding_verification_33_gb300 import workloads as W
    w_full = W.WORKLOADS[args.workload]
    w = W.small_variant(w_full, B=args.sample)  # same seeds: the first `sample` sequences
    d = W.make_inputs(w)
    toks = int(np.sum(d["draft_lens"]))
    for _ in range(args.warmup):
        oracle_time(d, w, range(w.B))
    times = [oracle_time(d, w, range(w.B))[0] for _ in range(args.steps)]
    mean = statistics.mean(times)
    value = toks / mean
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": mean * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w_full.name, "B": w_full.B, "K": w_full.K, "V": w_full.V,
                       "sample_sequences": w.B},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": f"first {w.B} of {w_full.B} sequences per step"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------------------------
# the row kernels (draft draw + exit confidence; exact-residual top-F + cache hits)
# ---------------------------------------------------------------------------------------------
ROW_FANOUT = (8, 4, 2, 1, 1, 1, 1, 1)


def row_workload(W, args):
    """The headline batch with a Saguaro bias (beta 0.5 on the 8 most likely draft ids) and
    geometric top-F widths, so both row kernels do their full work."""
    w = W.WORKLOADS[args.workload]
    return w.replace(beta=0.5, bias_k=8, fanout=ROW_FANOUT[: w.K], mode="stochastic",
                     temperature=w.temperature or 1.0)


def run_rows(args, quiet=False):
    import torch

    from speculative_decoding_verification_33_gb300 import api, build
    from speculative_decoding_verification_33_gb300 import workloads as W
    from oracle import rows as RO

    torch.cuda.set_device(dist_env()[2])
    w = row_workload(W, args)
    d = W.make_inputs(w)
    lens = d["draft_lens"]
    flush = L2Flush()
    tau = 0.1
    if args.kernel == "draft_sample":
        # every draft row the batch has (rows i < L_b), packed
        sel = [(b, i) for b in range(w.B) for i in range(int(lens[b]))]
        rows = np.stack([d["draft"][b, i] for b, i in sel])
        uni = np.ascontiguousarray(np.array([d["uniforms"][b, i] for b, i in sel], np.float32))
        R = rows.shape[0]
        D = api.to_device_logits(rows)
        U = torch.from_numpy(uni).cuda()
        out = {"tokens": torch.empty(R, dtype=torch.int32, device="cuda"),
               "conf": torch.empty(R, dtype=torch.float32, device="cuda"),
               "exit": torch.empty(R, dtype=torch.int32, device="cuda")}

        def step():
            api.draft_sample(D, U, temperature=w.temperature, beta=w.beta, bias_k=w.bias_k,
                             tau=tau, out=out)
        units, unit = R, "draft rows sampled/s"
        b_alg = R * (w.V * w.elem_bytes + 4 + 4 + 4 + 4)
    else:
        T = api.to_device_logits(d["target"])
        D = api.to_device_logits(d["draft"])
        vo = api.verify(T, D, torch.from_numpy(d["draft_tokens"]).cuda(),
                        torch.from_numpy(lens).cuda(), torch.from_numpy(d["uniforms"]).cuda(),
                        temperature=w.temperature, beta=w.beta, bias_k=w.bias_k,
                        fanout=w.fanout)
        LN = torch.from_numpy(lens).cuda()

        def step():
            return api.residual_topf(T, D, LN, w.fanout, temperature=w.temperature,
                                     beta=w.beta, bias_k=w.bias_k, verify_out=vo)
        R = int(np.sum(lens))
        units, unit = R, "draft positions/s"
        b_alg = R * (2 * w.V * w.elem_bytes + 4 * max(w.fanout)) + w.B * (4 + 4 * 5)
    for _ in range(max(args.warmup, 3)):
        flush()
        step()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    clocks = ClockSampler(dist_env()[2])
    clocks.start()
    time.sleep(0.3)
    torch.cuda.synchronize()
    for a, b in ev:
        flush()
        a.record()
        res = step()
        b.record()
    torch.cuda.synchronize()
    clk = clocks.stop()
    kms = [a.elapsed_time(b) for a, b in ev]
    mean_ms = statistics.mean(kms)
    peak, peak_src = measured_peak()
    achieved = b_alg / (mean_ms * 1e-3) / 1e9
    traffic, traffic_src = recorded_traffic(f"{args.kernel} {w.name}", build.kernel_digest("rows"))
    line = {"metric": f"{unit} and achieved HBM GB/s (% of roofline) at 1 GB300",
            "value": units / (mean_ms * 1e-3), "unit": unit, "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": mean_ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
            "config": {"workload": f"{args.kernel} {w.name}", "rows_or_positions": units,
                       "beta": w.beta, "bias_k": w.bias_k, "fanout": list(w.fanout),
                       "tau": tau, "l2": L2_NOTE},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic, "peak_source": peak_src,
                         "traffic_source": traffic_src, "algorithmic_bytes_per_launch": b_alg,
                         "kernel_ms_min": min(kms), "kernel_ms_median": statistics.median(kms)},
            "gpu_launches": args.steps,
            "clocks": clk}
    if not args.no_cpu:  # the oracle on a bounded sample, one core
        n = 32
        if args.kernel == "draft_sample":
            t0 = time.perf_counter()
            ref = [RO.draft_sample(rows[r], float(uni[r]), temperature=w.temperature,
                                   beta=w.beta, bias_k=w.bias_k, tau=tau) for r in range(n)]
            dt = time.perf_counter() - t0
            g = out["tokens"][:n].cpu().numpy()
            same = sum(int(g[r]) == o.token for r, o in enumerate(ref) if o.margin >= 1e-6)
            line["parity_sample"] = {"rows": n, "tokens_equal_unflagged": same,
                                     "flagged": sum(o.margin < 1e-6 for o in ref)}
        else:
            seqs = list(range(8))
            t0 = time.perf_counter()
            ref = RO.residual_topf(d["target"], d["draft"], lens, temperature=w.temperature,
                                   fanout=w.fanout, beta=w.beta, bias_k=w.bias_k, seqs=seqs)
            dt = time.perf_counter() - t0
            n = int(np.sum(lens[seqs]))
            g = res["r2"].cpu().numpy()[seqs]
            line["parity_sample"] = {"positions": n,
                                     "id_lists_equal": int(sum(
                                         np.array_equal(g[j, i], ref[j, i])
                                         for j in range(len(seqs))
                                         for i in range(int(lens[seqs[j]]))))}
        line["cpu_baseline"] = {"value": n / dt, "unit": unit, "cores": 1, "kind": "oracle",
                                "sample": f"first {n} {'rows' if args.kernel == 'draft_sample' else 'positions'}"}
    if args.kernel == "residual_topf":
        line["cache_hit"] = cache_hit_rates(w, vo, res)
    if not quiet:
        print(json.dumps(line), flush=True)
    return line


def cache_hit_rates(w, vo, res):
    """How often the token the verify step drew after a rejection at a_b < L_b is among the ids a
    speculation cache would have prepared for that outcome: R1, the first F_a ids of the draft
    row by logit (spec_verify's top-F output, the kernel's hit flags), and R2, the first F_a ids
    of the exact residual max(p - q', 0) (spec_residual_topf). Over every rejected sequence of
    the batch."""
    hit = res["hit"].cpu().numpy()
    acc = vo["accept_len"].cpu().numpy()
    tok = vo["tokens"].cpu().numpy()
    r2 = res["r2"].cpu().numpy()
    rej = [b for b in range(w.B) if hit[b] >= 0]
    h2 = 0
    for b in rej:
        a = int(acc[b])
        f = min(int(w.fanout[a]), r2.shape[2])
        h2 += int(tok[b, a] in r2[b, a, :f].tolist())
    n = max(1, len(rej))
    return {"rejected_sequences": len(rej), "r1_draft_topf_rate": int(np.sum(hit[rej] == 1)) / n,
            "r2_exact_residual_topf_rate": h2 / n, "fanout": list(w.fanout),
            "beta": w.beta, "bias_k": w.bias_k,
            "context": "SSD summary, Key claims: the speculation cache predicts the bonus token "
                       "from the draft logits, up to about 90% (other hardware, real models)"}


# ---------------------------------------------------------------------------------------------
# the LM head with its softmax statistics (tensor cores)
# ---------------------------------------------------------------------------------------------
def measured_tensor_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), "measured (MEASURED_PEAKS.json bf16_tflops, burst)"
    except Exception:
        return 1900.0, "fallback (1.9 PFLOP/s bf16 burst)"


def run_lmhead(args, quiet=False):
    import torch

    from speculative_decoding_verification_33_gb300 import api, build
    from speculative_decoding_verification_33_gb300 import workloads as W
    from oracle import lmhead as HO

    torch.cuda.set_device(dist_env()[2])
    w = W.HEAD_WORKLOADS[args.head]
    x = W.head_inputs(w)

    def dev(bits):
        return torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)
    H, Wt = dev(x["hidden"]), dev(x["weight"])
    ids = torch.from_numpy(x["ids"]).cuda()
    flush = L2Flush()

    def step():
        return api.lmhead_stats(H, Wt, ids, temperature=w.temperature)
    for _ in range(max(args.warmup, 3)):
        flush()
        step()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    clocks = ClockSampler(dist_env()[2])
    clocks.start()
    time.sleep(0.3)
    torch.cuda.synchronize()
    for a, b in ev:
        flush()
        a.record()
        out = step()
        b.record()
    torch.cuda.synchronize()
    clk = clocks.stop()
    kms = [a.elapsed_time(b) for a, b in ev]
    mean_ms = statistics.mean(kms)
    flops = 2.0 * w.R * w.d * w.V
    peak, peak_src = measured_tensor_peak()
    achieved = flops / (mean_ms * 1e-3) / 1e12
    traffic, traffic_src = recorded_traffic(f"lmhead {w.name}", build.kernel_digest("lmhead"))
    unit = "head rows scored/s"
    line = {"metric": f"{unit} and achieved bf16 TFLOP/s (% of roofline) at 1 GB300",
            "value": w.R / (mean_ms * 1e-3), "unit": unit, "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": mean_ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"lmhead {w.name}", "R": w.R, "d": w.d, "V": w.V,
                       "temperature": w.temperature,
                       "l2": L2_NOTE},
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak,
                         "unit": "TFLOP/s", "frac": achieved / peak, "traffic": traffic,
                         "peak_source": peak_src, "traffic_source": traffic_src,
                         "algorithmic_flops_per_launch": flops,
                         "min_bytes_per_launch": 2 * (w.R + w.V) * w.d,
                         "kernel_ms_min": min(kms), "kernel_ms_median": statistics.median(kms)},
            "gpu_launches": args.steps * 2, "clocks": clk}
    if not args.no_cpu:  # the oracle on a bounded sample of rows
        rows = np.arange(0, w.R, max(1, w.R // 8))[:8]
        t0 = time.perf_counter()
        ref = HO.head_stats(x["hidden"][rows], x["weight"], w.temperature, x["ids"][rows])
        dt = time.perf_counter() - t0
        g = out["lse"].cpu().numpy().astype(np.float64)[rows]
        line["parity_sample"] = {"rows": len(rows),
                                 "max_abs_lse_diff": float(np.max(np.abs(g - ref.lse)))}
        line["cpu_baseline"] = {"value": len(rows) / dt, "unit": unit,
                                "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
                                "sample": f"{len(rows)} rows of {w.R} (float64 numpy matmul, "
                                          "BLAS threads on the host cores)"}
    if not quiet:
        print(json.dumps(line), flush=True)
    return line


def run_hidden(args, quiet=False, oracle_seqs=8):
    """The verify step from hidden states: every row each sequence has goes through the
    tensor-core head (statistics only), the decided rows again for the draw."""
    import torch

    from speculative_decoding_verification_33_gb300 import api
    from speculative_decoding_verification_33_gb300 import workloads as W
    from oracle import lmhead as HO
    from tests import parity

    torch.cuda.set_device(dist_env()[2])
    w = W.HIDDEN_WORKLOADS["hv_B256_K8_V152064_d3584"]
    x = W.hidden_inputs(w)

    def dev(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(
            torch.bfloat16)
    Ht, Hd, Wt = dev(x["hidden_target"]), dev(x["hidden_draft"]), dev(x["weight"])
    X = torch.from_numpy(x["draft_tokens"]).cuda()
    LN = torch.from_numpy(x["draft_lens"]).cuda()
    U = torch.from_numpy(x["uniforms"]).cuda()
    out = {"accept_len": torch.empty(w.B, dtype=torch.int32, device="cuda"),
           "tokens": torch.empty(w.B, w.K + 1, dtype=torch.int32, device="cuda")}
    flush = L2Flush()

    def step():
        api.verify_hidden(Ht, Hd, Wt, X, LN, U, temperature=w.temperature, out=out)
    for _ in range(max(args.warmup, 3)):
        flush()
        step()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    clocks = ClockSampler(dist_env()[2])
    clocks.start()
    time.sleep(0.3)
    torch.cuda.synchronize()
    for a, b in ev:
        flush()
        a.record()
        step()
        b.record()
    torch.cuda.synchronize()
    clk = clocks.stop()
    kms = [a.elapsed_time(b) for a, b in ev]
    mean_ms = statistics.mean(kms)
    lens = x["draft_lens"]
    rows = int(np.sum(2 * lens + 1))
    acc = out["accept_len"].cpu().numpy()
    draws = int(np.sum(acc >= 0))
    flops = 2.0 * (rows + 2 * 64 * ((w.B + 63) // 64)) * w.d * w.V
    peak, peak_src = measured_tensor_peak()
    achieved = flops / (mean_ms * 1e-3) / 1e12
    toks = int(np.sum(lens))
    line = {"metric": "verified draft tokens/sec from hidden states (tensor-core LM head + "
                      "verify) and achieved bf16 TFLOP/s at 1 GB300",
            "value": toks / (mean_ms * 1e-3), "unit": UNIT, "n_gpus": 1, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": mean_ms, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"verify_hidden {w.name}", "B": w.B, "K": w.K, "V": w.V,
                       "d": w.d, "rows_scored": rows, "draws": draws,
                       "l2": L2_NOTE},
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak,
                         "unit": "TFLOP/s", "frac": achieved / peak, "traffic": None,
                         "peak_source": peak_src,
                         "scope": "whole step (7 launches; the two head GEMMs are the work)",
                         "algorithmic_flops_per_step": flops,
                         "kernel_ms_min": min(kms), "kernel_ms_median": statistics.median(kms)},
            "gpu_launches": args.steps * 7, "clocks": clk}
    if not args.no_cpu:  # the oracle on a bounded sample of sequences
        seqs = list(range(0, w.B, w.B // oracle_seqs))[:oracle_seqs]
        t0 = time.perf_counter()
        w64 = HO.bf16_to_f64(x["weight"])  # the head in float64 once for the sampled sequences
        res = HO.verify_hidden_batch(x["hidden_target"], x["hidden_draft"], w64,
                                     x["draft_tokens"], lens, x["uniforms"],
                                     temperature=w.temperature, mode=w.mode, seqs=seqs)
        dt = time.perf_counter() - t0
        rep = parity.compare(res, seqs, acc, out["tokens"].cpu().numpy(), margin=1e-3)
        line["parity_sample"] = {"sequences": rep.sequences, "flagged_1e-3": rep.flagged,
                                 "mismatches": len(rep.mismatches)}
        n = int(np.sum(lens[seqs]))
        line["cpu_baseline"] = {"value": n / dt, "unit": UNIT,
                                "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
                                "sample": f"{len(seqs)} of {w.B} sequences (float64 numpy "
                                          "matmul for the logits, BLAS threads)"}
    if not quiet:
        print(json.dumps(line), flush=True)
    return line


LEG_KEYS = ("metric", "value", "unit", "ms_per_step", "dtype", "config", "roofline", "clocks",
            "gpu_launches", "parity_sample", "cpu_baseline", "cache_hit")


def run_legs(args):
    """The row kernels (draft sampling, exact-residual top-F with the cache-hit rates) on the
    headline batch with a Saguaro bias, the tensor-core LM head, and the verify step from hidden
    states, each timed like the verify step (L2 flushed, CUDA events, clocks sampled), for the
    default line."""
    import copy
    legs = {}
    for kernel, fn in (("draft_sample", run_rows), ("residual_topf", run_rows),
                       ("lmhead", run_lmhead), ("verify_hidden", run_hidden)):
        sub = copy.copy(args)
        sub.kernel = kernel
        sub.steps = args.steps
        sub.warmup = 3
        t0 = time.perf_counter()
        line = fn(sub, quiet=True, **({"oracle_seqs": 2} if kernel == "verify_hidden" else {}))
        leg = {k: line[k] for k in LEG_KEYS if k in line}
        leg["steps"] = sub.steps
        leg["wall_s"] = time.perf_counter() - t0
        legs[kernel] = leg
        import torch
        torch.cuda.empty_cache()
    return legs


# ---------------------------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------------------------
def run_ours(args):
    import torch
    import torch.distributed as dist

    from speculative_decoding_verification_33_gb300 import _lib, api, build
    from speculative_decoding_verification_33_gb300 import workloads as W

    rank, world, local = dist_env()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    w = W.WORKLOADS[args.workload]
    d = W.make_inputs(w, offset=rank)
    lens = d["draft_lens"]
    toks_local = float(np.sum(lens))
    greedy = w.mode == "greedy"

    T = api.to_device_logits(d["target"])
    D = None if greedy else api.to_device_logits(d["draft"])
    tok = torch.from_numpy(d["draft_tokens"]).cuda()
    ln = torch.from_numpy(lens).cuda()
    uni = torch.from_numpy(d["uniforms"]).cuda()
    acc = torch.empty(w.B, dtype=torch.int32, device="cuda")
    otok = torch.empty(w.B, w.K + 1, dtype=torch.int32, device="cuda")
    otopf = (torch.empty(w.B, w.K, max(w.fanout), dtype=torch.int32, device="cuda")
             if w.fanout else None)
    flush = L2Flush()

    dcode = _lib.SV_DTYPE_BF16 if w.dtype == "bf16" else _lib.SV_DTYPE_F32
    prob, _keep = _lib.make_problem(w.B, w.K, w.V, dcode, w.V, w.V, w.bias_k, w.fanout,
                                    cluster_hint=args.cluster)
    plan_c, plan_n, plan_smem = _lib.plan(
        prob, _lib.SV_MODE_GREEDY if greedy else _lib.SV_MODE_STOCHASTIC)
    route, launches = _lib.route(prob, _lib.SV_MODE_GREEDY if greedy else _lib.SV_MODE_STOCHASTIC)

    def step():
        api.spec_verify(T, D, tok, ln, uni, w.temperature, w.beta, w.mode, acc, otok, otopf,
                        bias_k=w.bias_k, fanout=w.fanout, cluster_hint=args.cluster)

    for _ in range(max(args.warmup, 3)):
        if not args.l2_warm:
            flush()
        step()
    torch.cuda.synchronize()
    assert api.device_error() == 0

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    for s in range(args.steps):
        if not args.l2_warm:
            flush()
        starts[s].record()
        step()
        ends[s].record()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    wall = time.perf_counter() - wall0
    clk = clocks.stop()
    kms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    mean_ms = statistics.mean(kms)
    toks_all, ms_max = aggregate(toks_local, mean_ms)
    value = toks_all / (ms_max * 1e-3)

    g_acc = acc.cpu().numpy()
    g_tok = otok.cpu().numpy()
    # the other two rates of the metric's definition: tokens emitted (accepted drafts plus the
    # drawn token, valid sequences) and logit rows covered (every target and draft row a
    # sequence has) per second
    emitted_all, _ = aggregate(float(np.sum(np.where(g_acc >= 0, g_acc + 1, 0))), mean_ms)
    rows_local = float(np.sum(lens + 1) + (np.sum(lens) if w.mode == "stochastic" else 0))
    rows_all, _ = aggregate(rows_local, mean_ms)
    b_alg = algorithmic_bytes(w, lens, g_acc)
    b_in = input_bytes(w, lens)
    peak, peak_src = measured_peak()
    achieved = b_alg / (mean_ms * 1e-3) / 1e9
    digest = build.kernel_digest(ROUTE_SOURCES[route])
    traffic, traffic_src = recorded_traffic(w.name, digest)

    # read-only streaming probe (2 GiB), for context
    probe_gbs = None
    try:
        buf = torch.empty(1 << 29, dtype=torch.int32, device="cuda")
        buf.fill_(1)
        out = torch.zeros(1, dtype=torch.int64, device="cuda")
        for _ in range(3):
            api.hbm_read_probe(buf, out)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(10):
            api.hbm_read_probe(buf, out)
        e1.record()
        torch.cuda.synchronize()
        probe_gbs = 10 * buf.numel() * 4 / (e0.elapsed_time(e1) * 1e-3) / 1e9
        del buf
    except Exception as ex:  # pragma: no cover - reported, not fatal
        probe_gbs = f"unavailable: {ex}"

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": w.dtype,
            "data": "synthetic (seeded Zipf-prior logits, Gumbel-max drafts, NaN padding rows)",
            "config": {"workload": w.name, "B": w.B, "K": w.K, "V": w.V, "mode": w.mode,
                       "temperature": w.temperature,
                       "draft_lens": f"uniform 1..{w.K}" if w.ragged else f"all {w.K}",
                       "verified_tokens_per_rank": toks_local,
                       "l2": ("warm: no flush between steps" if args.l2_warm else
                              L2_NOTE),
                       "cluster_hint": args.cluster, "route": ROUTE_NAMES[route],
                       "ctas_per_cluster": plan_c,
                       "clusters": plan_n, "smem_per_cta": plan_smem,
                       "wall_ms_per_step_incl_flush": wall / args.steps * 1e3},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": traffic,
                         "peak_source": peak_src, "traffic_source": traffic_src,
                         "algorithmic_bytes_per_launch": b_alg,
                         "all_rows_bytes_per_launch": b_in,
                         "all_rows_gbs": b_in / (mean_ms * 1e-3) / 1e9,
                         "read_probe_gbs": probe_gbs,
                         "kernel_ms_min": min(kms), "kernel_ms_median": statistics.median(kms)},
            "gpu_launches": args.steps * launches, "clocks": clk,
            "rates": {"emitted_tokens_per_s": emitted_all / (ms_max * 1e-3),
                      "logit_rows_per_s": rows_all / (ms_max * 1e-3)}}

    # end to end through the host-buffer entry point (pinned host memory)
    if not args.no_e2e:
        def pinned_logits(a):
            return torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a).pin_memory()
        hT = pinned_logits(d["target"])
        hD = None if greedy else pinned_logits(d["draft"])
        h_tok = torch.from_numpy(d["draft_tokens"]).pin_memory()
        h_len = torch.from_numpy(lens).pin_memory()
        h_uni = torch.from_numpy(d["uniforms"]).pin_memory()
        h_acc = torch.empty(w.B, dtype=torch.int32).pin_memory()
        h_out = torch.empty(w.B, w.K + 1, dtype=torch.int32).pin_memory()
        h_topf = (torch.empty(w.B, w.K, max(w.fanout), dtype=torch.int32).pin_memory()
                  if w.fanout else None)

        def e2e_step():
            api.verify_host(hT, hD, h_tok, h_len, h_uni, h_acc, h_out, h_topf, dtype=w.dtype,
                            temperature=w.temperature, beta=w.beta, mode=w.mode,
                            bias_k=w.bias_k, fanout=w.fanout)

        for _ in range(2):
            e2e_step()
        n_e2e = max(3, min(args.steps, 20))
        if world > 1:
            dist.barrier()
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            e2e_step()
        t_e2e = (time.perf_counter() - t0) / n_e2e
        _, t_e2e_max = aggregate(0.0, t_e2e)
        h2d, d2h = host_copy_bytes(w, lens, g_acc)
        line["e2e"] = {"value": toks_all / t_e2e_max, "unit": UNIT, "h2d_bytes_per_step": h2d,
                       "d2h_bytes_per_step": d2h, "ms_per_step": t_e2e_max * 1e3,
                       "host_rows": "read in place by the kernel from pinned host memory"
                       if not top8_prepass(w) else "staged with one copy per sequence",
                       "matches_device_call": bool(np.array_equal(h_acc.numpy(), g_acc) and
                                                   np.array_equal(h_out.numpy(), g_tok))}

    # CPU baseline (the oracle, one core, the whole batch) and full-size parity
    if rank == 0 and world >= 1 and not args.no_cpu:
        from tests.parity import compare
        t_cpu, res = oracle_time(d, w, range(w.B))
        rep = compare(res, range(w.B), g_acc, g_tok,
                      otopf.cpu().numpy() if otopf is not None else None)
        line["cpu_baseline"] = {"value": toks_local / t_cpu, "unit": UNIT, "cores": 1,
                                "kind": "oracle",
                                "sample": f"all {w.B} sequences of rank 0's batch, once"}
        procs = len(os.sched_getaffinity(0))
        if procs > 1 and w.B > 1:
            t_pool = oracle_pool_time(d, w, min(procs, w.B))
            line["cpu_baseline"]["pool"] = {"value": toks_local / t_pool, "unit": UNIT,
                                            "cores": min(procs, w.B),
                                            "kind": "oracle, sequences sharded over processes"}
        line["parity"] = {"sequences": rep.sequences, "flagged": rep.flagged,
                          "mismatches": len(rep.mismatches), "invalid": rep.invalid}
    if rank == 0 and world == 1 and args.workload == 5 and args.cluster == 0 and not args.no_legs:
        del d
        torch.cuda.empty_cache()
        line["legs"] = run_legs(args)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def main(argv=None):
    args = parse_args(argv)
    if args.impl == "reference":
        run_reference(args)
    elif args.kernel == "lmhead":
        run_lmhead(args)
    elif args.kernel == "verify_hidden":
        run_hidden(args)
    elif args.kernel != "verify":
        run_rows(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()

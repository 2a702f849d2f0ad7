"""Benchmark of the DSA hot path on one GB300 (or N replicas).

Workload (the pages' 32k configuration): one sequence of S = 32768 tokens;
lightning indexer with 64 heads x 128 (bf16 q_idx [S,64,128], shared k_idx
[S,128], fp32 head weights ~ U(0,1)/8) and causal top-k K = 2048; the selected
indices drive absorbed sparse MLA forward + backward with H = 64 heads, width
576 (512 latent + 64 RoPE), value 512, softmax_scale = 192^-0.5, bf16 N(0,1)
q / kv / dO.  One step = indexer top-k -> sparse MLA forward -> sparse MLA
backward on device-resident inputs (the THD metadata is built once, as the
pages do once per pipeline stage).

Metric: sparse-MLA fwd+bwd TFLOP/s (algorithmic FLOPs over valid slots:
fwd 2*H*n*(576+512), bwd 2*H*n*(3*576+2*512)) with the indexer's top-k
tokens/s alongside.  Every input is larger than L2 (q alone is 2.4 GB), so no
L2 flush is needed between steps.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

S, HI, DI, K, H, DQK, DV = 32768, 64, 128, 2048, 64, 576, 512
SCALE = 192 ** -0.5
METRIC = "sparse-MLA fwd+bwd TFLOP/s (% bf16 peak) and indexer top-k tokens/s at S=32k,K=2048"
UNIT = "TFLOP/s"
WORKLOAD = "lightning indexer (64x128) + causal top-k K=2048 -> sparse MLA fwd+bwd H=64 width 576, S=32768, 1 sequence"


def mla_flops(n_valid: int) -> tuple[float, float]:
    return 2.0 * H * n_valid * (DQK + DV), 2.0 * H * n_valid * (3 * DQK + 2 * DV)


# L2 rates of this GPU for the two access patterns the MLA kernels live on, measured by
# standalone microbenchmarks on a GB300 (all SMs, clocks at 2070 MHz): fp32 reductions of
# 4-row x 128-byte segments at the selected rows (red.global.add.v4.f32, the backward's
# pattern, replayed over the indexer's selection at 32k) and 16-byte cp.async gathers of
# 128 random 1152-byte rows per tile by 256 threads, one tile in flight per SM.
L2_RED_TBS = 6.9
L2_GATHER_TBS = 17.5


def l2_model(n_valid: int, n_tiles: int, fwd_ms: float, bwd_ms: float) -> dict:
    """Time the MLA kernels would take if their L2 traffic alone ran at the rates above.

    Backward per valid slot: one fp32 dKV row reduced (4 * DQK bytes) and the kv row gathered
    twice (2 * 2 * DQK); per 128-slot tile, the bf16 dS tile written to and read back from the
    scratch (2 * 128 * 64 * 2 bytes).  Forward: the kv row gathered once (2 * DQK)."""
    red = 4.0 * DQK * n_valid
    gat_b = 2.0 * 2 * DQK * n_valid + 2.0 * n_tiles * 128 * 64 * 2
    gat_f = 2.0 * DQK * n_valid
    t_b = (red / (L2_RED_TBS * 1e12) + gat_b / (L2_GATHER_TBS * 1e12)) * 1e3
    t_f = gat_f / (L2_GATHER_TBS * 1e12) * 1e3
    return {"rates_tbs": {"reduction": L2_RED_TBS, "gather": L2_GATHER_TBS},
            "bwd": {"reduction_gb": round(red / 1e9, 2), "gather_gb": round(gat_b / 1e9, 2),
                    "model_ms": round(t_b, 3), "frac": round(t_b / bwd_ms, 4)},
            "fwd": {"gather_gb": round(gat_f / 1e9, 2), "model_ms": round(t_f, 3), "frac": round(t_f / fwd_ms, 4)}}


def load_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        d["source"] = "measured"
        return d
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines: list[str] = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist

        # one process per GPU over NCCL; gloo where no GPU is visible (host-side tests of the replica path)
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# CPU oracle leg (test infrastructure: the plain fp64 oracle, as it stands)
# ---------------------------------------------------------------------------
def oracle_sample(rows: int, seed: int = 0) -> dict:
    """Time the oracle on a bounded sample of the same workload: the last
    `rows` query rows (full 32k windows, full K) for indexer top-k and sparse
    MLA fwd+bwd.  Inputs are drawn with the same recipe, on the CPU."""
    import numpy as np
    import torch

    import oracle
    from sparse_attention_mla_gb300 import synth

    g = synth.generator(seed)
    k_idx = synth.randn_bf16((S, DI), g)
    q_idx = synth.randn_bf16((rows, HI, DI), g)
    w = torch.rand(rows, HI, generator=g) / 8.0
    kv = synth.randn_bf16((S, DQK), g)
    q = synth.randn_bf16((rows, H, DQK), g)
    dout = synth.randn_bf16((rows, H, DV), g)
    row_t = np.arange(S - rows, S)
    start = np.zeros(S, np.int32)
    t0 = time.perf_counter()
    idx, ln, _ = oracle.indexer_topk(q_idx, k_idx, w, start, row_t, K)
    t1 = time.perf_counter()
    oracle.sparse_mla_fwd(q, kv, idx, SCALE)
    oracle.sparse_mla_bwd(q, kv, idx, dout, SCALE)
    t2 = time.perf_counter()
    n_valid = int((idx >= 0).sum())
    fl = sum(mla_flops(n_valid))
    return {"mla_s": t2 - t1, "idx_s": t1 - t0, "mla_tflops": fl / (t2 - t1) / 1e12,
            "idx_tokens_per_s": rows / (t1 - t0), "rows": rows, "cores": os.cpu_count()}


def run_reference(args, rank, world):
    if rank != 0:
        return
    rows = os.cpu_count() or 1  # one query row per host core (the oracle is parallel over rows)
    for _ in range(args.warmup):
        oracle_sample(rows)
    vals, idx_rates, wall = [], [], []
    for i in range(args.steps):
        r = oracle_sample(rows, seed=i)
        vals.append(r["mla_tflops"])
        idx_rates.append(r["idx_tokens_per_s"])
        wall.append(r["mla_s"] + r["idx_s"])
    v = statistics.median(vals)
    sample = (f"{rows} query rows (positions {S - rows}..{S - 1}, full 32k causal windows, K=2048) per step: "
              "indexer top-k + sparse MLA fwd+bwd in the fp64 C oracle")
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 * statistics.median(wall), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "sample": sample},
        "indexer_tokens_per_s": statistics.median(idx_rates),
        "cpu_baseline": {"value": v, "unit": UNIT, "cores": os.cpu_count(), "kind": "oracle", "sample": sample},
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# CUDA leg
# ---------------------------------------------------------------------------
def run_cuda(args, rank, world, local):
    import torch

    import sparse_attention_mla_gb300 as dsa
    from sparse_attention_mla_gb300 import synth

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dsa.load_library()
    peaks = load_peaks()

    # ---- inputs (device-resident; drawn on the device with the synth recipe) ----
    ind = synth.indexer_inputs(S, HI, DI, seed=rank, device=dev)
    mla = synth.mla_inputs(S, H, DQK, DV, seed=1000 + rank, device=dev)
    cu = torch.tensor([0, S], dtype=torch.int32, device=dev)
    seq_start, _, _, _ = dsa.dsa_packed_metadata(cu, S)  # once per stage, as on the pages
    topk_idx = torch.empty(S, K, dtype=torch.int32, device=dev)
    topk_len = torch.empty(S, dtype=torch.int32, device=dev)
    out = torch.empty(S, H, DV, dtype=torch.bfloat16, device=dev)
    out_lo = torch.empty(S, H, DV, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(S, H, dtype=torch.float32, device=dev)
    dq = torch.empty(S, H, DQK, dtype=torch.bfloat16, device=dev)
    dkv = torch.empty(S, DQK, dtype=torch.float32, device=dev)
    ws_i = torch.zeros(dsa.workspace_size("indexer", S, K), dtype=torch.uint8, device=dev)
    ws_f = torch.zeros(dsa.workspace_size("fwd", S, H), dtype=torch.uint8, device=dev)
    ws_b = torch.zeros(dsa.workspace_size("bwd", S, H, K), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]

    def step(e=None):
        if e: e[0].record(stream)
        dsa.dsa_indexer_topk(ind["q_idx"], ind["k_idx"], ind["w"], seq_start, K, topk_idx=topk_idx,
                             topk_len=topk_len, workspace=ws_i)
        if e: e[1].record(stream)
        dsa.dsa_sparse_mla_fwd(mla["q"], mla["kv"], topk_idx, SCALE, topk_len=topk_len, out=out, lse=lse,
                               workspace=ws_f, out_lo=out_lo)
        if e: e[2].record(stream)
        dsa.dsa_sparse_mla_bwd(mla["q"], mla["kv"], topk_idx, SCALE, out, lse, mla["dout"], topk_len=topk_len,
                               dq=dq, dkv_accum=dkv, workspace=ws_b, out_lo=out_lo)
        if e: e[3].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    for w_ in (ws_i, ws_f, ws_b):
        st = dsa.dsa_read_device_status(w_)
        if st != 0:
            raise RuntimeError(f"device status {st} after warm-up")
    n_valid = int(topk_len.sum().item())
    n_tiles = int(((topk_len + 127) // 128).sum().item()) * ((H + 63) // 64)
    f_fwd, f_bwd = mla_flops(n_valid)

    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize(dev)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        step(ev[i])
    t_end.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    clocks = sampler.stop()
    total_ms = max_over_ranks(t_start.elapsed_time(t_end), world, dev)
    idx_ms = statistics.median(e[0].elapsed_time(e[1]) for e in ev)
    fwd_ms = statistics.median(e[1].elapsed_time(e[2]) for e in ev)
    bwd_ms = statistics.median(e[2].elapsed_time(e[3]) for e in ev)
    mla_ms_total = sum(e[1].elapsed_time(e[3]) for e in ev)
    mla_ms_total = max_over_ranks(mla_ms_total, world, dev)
    value = world * args.steps * (f_fwd + f_bwd) / (mla_ms_total * 1e-3) / 1e12
    idx_tok_s = world * S / (idx_ms * 1e-3)

    # ---- rooflines: each kernel's algorithmic work over its CUDA-event time; the dominant kernel
    # (the backward: most FLOPs and time) is `roofline` ----
    peak = peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops"))
    src = f"{peaks['source']} bf16 sustained (kernels timed inside a long step)"
    n_pairs = int((torch.arange(S, device=dev) - seq_start + 1).clamp(min=0).sum().item())
    f_idx = 2.0 * HI * DI * n_pairs
    idx_bytes = S * HI * DI * 2 + S * DI * 2 + S * HI * 4 + S * K * 4 + S * 4  # q_idx, k_idx, w, idx, len
    units = {"sparse_mla_bwd_kernel": n_valid, "sparse_mla_fwd_kernel": n_valid, "indexer_topk_kernel": S}
    per_kernel = {}
    for name, flops, ms, src_file in (("sparse_mla_bwd_kernel", f_bwd, bwd_ms, "dsa_bwd.cu"),
                                      ("sparse_mla_fwd_kernel", f_fwd, fwd_ms, "dsa_fwd.cu"),
                                      ("indexer_topk_kernel", f_idx, idx_ms, "dsa_indexer.cu")):
        ach = flops / (ms * 1e-3) / 1e12
        per_kernel[name] = {"bound": "tensor", "kernel": name, "achieved": round(ach, 2), "peak": peak,
                            "unit": "TFLOP/s", "frac": round(ach / peak, 4),
                            "traffic": traffic_per_launch(name, src_file, units[name]), "ms": round(ms, 3),
                            "peak_source": src}
    hbm = peaks.get("hbm_gbs")
    idx_gbs = idx_bytes / (idx_ms * 1e-3) / 1e9
    per_kernel["indexer_topk_kernel"].update({"causal_pairs": n_pairs, "hbm_algorithmic_bytes": idx_bytes,
                                              "hbm_achieved_gbs": round(idx_gbs, 1),
                                              "hbm_frac": round(idx_gbs / hbm, 4) if hbm else None})
    roofline = per_kernel["sparse_mla_bwd_kernel"]

    # ---- end to end through the public API with host buffers ----
    e2e = None
    if not args.no_e2e:
        # one untimed pass of the whole leg first: its 12 GB of pinned host buffers are allocated and used
        # once (right after other large jobs on the host, the first pass's copies ran at about 2/3 speed)
        run_e2e(args, dsa, torch, dev, stream, ind, mla, seq_start, f_fwd + f_bwd, world)
        e2e = run_e2e(args, dsa, torch, dev, stream, ind, mla, seq_start, f_fwd + f_bwd, world)
    cp = None if args.no_cp else run_cp_indexer(args, dsa, torch, dev, stream, ind, topk_idx, topk_len)
    kl_path = None if args.no_kl else run_kl_path(args, dsa, torch, dev, stream, ind, mla, seq_start, topk_idx,
                                                   topk_len, out, out_lo, lse, dq, dkv, ws_b, bwd_ms, n_valid)
    workloads = None
    if not args.no_workloads:
        del ws_b
        torch.cuda.empty_cache()
        workloads = {name: time_workload(name, args, dev, stream) for name in ("v32", "nope", "kpool")}

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "S": S, "K": K, "H": H, "width": DQK, "indexer_heads": HI,
                   "indexer_dim": DI, "global_batch": S * world, "seq_len": S,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "inputs larger than L2 (q 2.4 GB), no flush"},
        "mla_pct_bf16_peak": round(100 * value / world / peak, 2),
        "indexer_tokens_per_s": round(idx_tok_s, 1),
        "components_ms": {"indexer_topk": round(idx_ms, 3), "sparse_mla_fwd": round(fwd_ms, 3),
                          "sparse_mla_bwd": round(bwd_ms, 3)},
        "n_valid_slots": n_valid,
        "roofline": roofline,
        "roofline_kernels": per_kernel,
        "l2_model": l2_model(n_valid, n_tiles, fwd_ms, bwd_ms),
        "clocks": clocks,
        "gpu_launches": 3 * args.steps,  # indexer, forward, backward per step
        "e2e": e2e,
        "cp_indexer": cp,
        "kl_path": kl_path,
        "workloads": workloads,
    }
    if rank == 0 and not args.no_cpu_baseline:
        r = oracle_sample(16)
        line["cpu_baseline"] = {"value": round(r["mla_tflops"], 6), "unit": UNIT, "cores": r["cores"],
                                "kind": "oracle",
                                "sample": "16 query rows (positions 32752..32767, full windows, K=2048): indexer "
                                          "top-k then sparse MLA fwd+bwd in the fp64 C oracle; value = MLA fwd+bwd "
                                          f"TFLOP/s; indexer {r['idx_tokens_per_s']:.2f} tokens/s"}
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_kl_path(args, dsa, torch, dev, stream, ind, mla, seq_start, topk_idx, topk_len, out, out_lo, lse, dq, dkv,
                ws_b, bwd_ms, n_valid):
    """The indexer KL auxiliary loss on the same selection: the backward with its slot-probability output
    (the extra cost over the plain backward), then the KL kernel (loss and gradients) forming the slots'
    indexer scores itself; and the other order of work: the indexer returning its selection's scores, and
    the KL kernel reading them.  CUDA events on the launching stream, median over the timed steps."""
    prob = torch.empty(S, K, dtype=torch.float32, device=dev)
    ws = torch.zeros(4096, dtype=torch.uint8, device=dev)
    kl = torch.empty(S, dtype=torch.float32, device=dev)
    dqi = torch.empty_like(ind["q_idx"])
    dw = torch.empty_like(ind["w"])
    dk = torch.empty(S, DI, dtype=torch.float32, device=dev)

    def bwd():
        dsa.dsa_sparse_mla_bwd(mla["q"], mla["kv"], topk_idx, SCALE, out, lse, mla["dout"], topk_len=topk_len, dq=dq,
                               dkv_accum=dkv, workspace=ws_b, out_lo=out_lo, attn_prob=prob)

    def klk(score=None):
        dsa.dsa_indexer_kl(ind["q_idx"], ind["k_idx"], ind["w"], topk_idx, prob, 0.001, topk_len=topk_len, kl=kl,
                           dq_idx=dqi, dw=dw, dk_idx_accum=dk, workspace=ws, topk_score=score)

    isc = torch.empty(S, K, dtype=torch.float32, device=dev)
    idx_s, len_s = torch.empty_like(topk_idx), torch.empty_like(topk_len)
    wi = torch.zeros(dsa.workspace_size("indexer", S, K), dtype=torch.uint8, device=dev)

    def idx_scored():
        dsa.dsa_indexer_topk_scored(ind["q_idx"], ind["k_idx"], ind["w"], seq_start, K, topk_idx=idx_s,
                                    topk_len=len_s, topk_score=isc, workspace=wi)

    steps = (bwd, klk, idx_scored, lambda: klk(isc))
    for _ in range(args.warmup):
        for f in steps:
            f()
    torch.cuda.synchronize(dev)
    if not (torch.equal(idx_s, topk_idx) and torch.equal(len_s, topk_len)):
        raise RuntimeError("the indexer with scores selected differently")
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(steps) + 1)] for _ in range(args.steps)]
    for e in ev:
        e[0].record(stream)
        for i, f in enumerate(steps):
            f()
            e[i + 1].record(stream)
    torch.cuda.synchronize(dev)
    if any(dsa.dsa_read_device_status(w_) != 0 for w_ in (ws, ws_b, wi)):
        raise RuntimeError("device status after the KL path")
    b_ms, k_ms, i_ms, kr_ms = (statistics.median(e[i].elapsed_time(e[i + 1]) for e in ev) for i in range(len(steps)))
    f_alg = 3 * 2.0 * HI * DI * n_valid  # scores, dq_idx and dk_idx products
    return {"bwd_with_slot_prob_ms": round(b_ms, 3), "bwd_ms": round(bwd_ms, 3),
            "indexer_kl_ms": round(k_ms, 3), "indexer_kl_tflops": round(f_alg / (k_ms * 1e-3) / 1e12, 2),
            "indexer_topk_scored_ms": round(i_ms, 3), "indexer_kl_reading_scores_ms": round(kr_ms, 3),
            "note": "loss coefficient 0.001; kl per row, dq_idx, dw and the fp32 dk_idx accumulator; "
                    "indexer_kl_ms forms the slots' scores again, indexer_kl_reading_scores_ms reads those of "
                    "dsa_indexer_topk_scored (same selection)"}


def run_cp_indexer(args, dsa, torch, dev, stream, ind, topk_idx, topk_len, ranks=2):
    """The indexer in its context-parallel form: rank 0 of `ranks`, holding the load-balanced
    chunks 0 and 2R-1 of the sequence's query rows, against all keys.  Its rows must equal the
    same rows of the one-shot indexer; timed with CUDA events over K steps."""
    S_ = ind["q_idx"].shape[0]
    edges = [S_ * i // (2 * ranks) for i in range(2 * ranks + 1)]
    qi = torch.cat([torch.arange(edges[0], edges[1]), torch.arange(edges[-2], edges[-1])]).to(dev)
    q_loc, w_loc = ind["q_idx"][qi].contiguous(), ind["w"][qi].contiguous()
    cu = torch.tensor([0, S_], dtype=torch.int32, device=dev)
    st, cl, _, _ = dsa.dsa_packed_metadata_cp(cu, S_, query_indices=qi.to(torch.int32))
    ws = torch.zeros(dsa.workspace_size("indexer", q_loc.shape[0], K), dtype=torch.uint8, device=dev)
    run = lambda: dsa.dsa_indexer_topk_cp(q_loc, ind["k_idx"], w_loc, st, cl, K, workspace=ws)
    for _ in range(args.warmup):
        idx, ln = run()
    torch.cuda.synchronize(dev)
    same = bool(torch.equal(idx, topk_idx[qi]) and torch.equal(ln, topk_len[qi]))
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for a, b in ev:
        a.record(stream)
        run()
        b.record(stream)
    torch.cuda.synchronize(dev)
    if dsa.dsa_read_device_status(ws) != 0:
        raise RuntimeError("device status after the context-parallel indexer")
    ms = statistics.median(a.elapsed_time(b) for a, b in ev)
    return {"ranks": ranks, "rank": 0, "local_rows": int(q_loc.shape[0]), "ms": round(ms, 3),
            "tokens_per_s": round(q_loc.shape[0] / (ms * 1e-3), 1), "matches_one_shot_rows": same}


def run_e2e(args, dsa, torch, dev, stream, ind, mla, seq_start, flops_per_step, world):
    """Same metric through the public API with pinned host buffers: every step
    copies its inputs host->device and reads its results device->host.

    The step is pipelined the way the pages chunk long sequences (query chunks
    are independent; key gradients accumulate): the indexer runs once over all
    queries, then sparse MLA fwd+bwd run over 4096-query chunks on a compute
    stream while the next chunk's inputs and the previous chunk's results
    cross the host link on two copy streams."""
    host_in = {k: v.to("cpu").pin_memory() for k, v in list(ind.items()) + list(mla.items())}
    # two sets of device inputs, used by alternate steps: a step's input copies start while the
    # previous step still computes on the other set
    dev_sets = [{k: torch.empty_like(v, device=dev) for k, v in host_in.items()} for _ in range(2)]
    res_shapes = {"topk_idx": ((S, K), torch.int32), "topk_len": ((S,), torch.int32),
                  "out": ((S, H, DV), torch.bfloat16), "out_lo": ((S, H, DV), torch.bfloat16),
                  "lse": ((S, H), torch.float32),
                  "dq": ((S, H, DQK), torch.bfloat16), "dkv": ((S, DQK), torch.float32)}
    dres = {k: torch.empty(*s, dtype=d, device=dev) for k, (s, d) in res_shapes.items()}
    hres = {k: torch.empty(*s, dtype=d).pin_memory() for k, (s, d) in res_shapes.items()}
    h2d = sum(v.numel() * v.element_size() for v in host_in.values())
    d2h = sum(v.numel() * v.element_size() for v in hres.values())
    CH = 4096
    chunks = [(a, min(S, a + CH)) for a in range(0, S, CH)]
    comp, cin, cout = stream, torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    # every workspace is allocated once, before the timed steps
    ws_i = torch.empty(dsa.workspace_size("indexer", S, K), dtype=torch.uint8, device=dev)
    ws_f = torch.empty(dsa.workspace_size("fwd", CH, H), dtype=torch.uint8, device=dev)
    ws_b = torch.empty(dsa.workspace_size("bwd", CH, H, K), dtype=torch.uint8, device=dev)
    whole = ("k_idx", "kv", "q_idx", "w")           # the indexer's inputs and the keys: copied first
    per_chunk_in = ("q", "dout")                    # copied per query chunk
    per_chunk_out = ("out", "out_lo", "lse", "dq")  # read back per query chunk
    # ordering across steps: an input set is refilled once the step before last finished with it; a
    # result buffer is rewritten once the previous step's copy of it has left for the host
    state = {"step": 0, "set_done": [None, None], "idx_out": None, "chunk_out": [None] * len(chunks), "dkv_out": None}

    def step():
        b = state["step"] & 1
        state["step"] += 1
        dev_in = dev_sets[b]
        ev_whole = torch.cuda.Event()
        with torch.cuda.stream(cin):
            if state["set_done"][b] is not None:
                cin.wait_event(state["set_done"][b])
            for k in whole:
                dev_in[k].copy_(host_in[k], non_blocking=True)
            ev_whole.record(cin)
            ev_in = []
            for (a, e_) in chunks:
                for k in per_chunk_in:
                    dev_in[k][a:e_].copy_(host_in[k][a:e_], non_blocking=True)
                e = torch.cuda.Event()
                e.record(cin)
                ev_in.append(e)
        with torch.cuda.stream(comp):
            comp.wait_event(ev_whole)
            if state["idx_out"] is not None:
                comp.wait_event(state["idx_out"])
            dsa.dsa_indexer_topk(dev_in["q_idx"], dev_in["k_idx"], dev_in["w"], seq_start, K,
                                 topk_idx=dres["topk_idx"], topk_len=dres["topk_len"], workspace=ws_i)
            ev_idx = torch.cuda.Event()
            ev_idx.record(comp)
        with torch.cuda.stream(cout):
            cout.wait_event(ev_idx)
            hres["topk_idx"].copy_(dres["topk_idx"], non_blocking=True)
            hres["topk_len"].copy_(dres["topk_len"], non_blocking=True)
            state["idx_out"] = torch.cuda.Event()
            state["idx_out"].record(cout)
        for c, (a, e_) in enumerate(chunks):
            with torch.cuda.stream(comp):
                comp.wait_event(ev_in[c])
                if state["chunk_out"][c] is not None:
                    comp.wait_event(state["chunk_out"][c])
                if c == 0 and state["dkv_out"] is not None:
                    comp.wait_event(state["dkv_out"])
                dsa.dsa_sparse_mla_fwd(dev_in["q"][a:e_], dev_in["kv"], dres["topk_idx"][a:e_], SCALE,
                                       topk_len=dres["topk_len"][a:e_], out=dres["out"][a:e_], lse=dres["lse"][a:e_],
                                       out_lo=dres["out_lo"][a:e_], workspace=ws_f)
                dsa.dsa_sparse_mla_bwd(dev_in["q"][a:e_], dev_in["kv"], dres["topk_idx"][a:e_], SCALE,
                                       dres["out"][a:e_], dres["lse"][a:e_], dev_in["dout"][a:e_],
                                       topk_len=dres["topk_len"][a:e_], dq=dres["dq"][a:e_], dkv_accum=dres["dkv"],
                                       accumulate=c > 0, out_lo=dres["out_lo"][a:e_], workspace=ws_b)
                e = torch.cuda.Event()
                e.record(comp)
            with torch.cuda.stream(cout):
                cout.wait_event(e)
                for k in per_chunk_out:
                    hres[k][a:e_].copy_(dres[k][a:e_], non_blocking=True)
                state["chunk_out"][c] = torch.cuda.Event()
                state["chunk_out"][c].record(cout)
        state["set_done"][b] = e  # the last chunk's compute: this input set is free after it
        with torch.cuda.stream(cout):
            hres["dkv"].copy_(dres["dkv"], non_blocking=True)
            state["dkv_out"] = torch.cuda.Event()
            state["dkv_out"].record(cout)

    steps = max(1, min(args.steps, 3))
    # one untimed step per device input set, so that every buffer the timed steps use (both input sets,
    # the pinned host buffers, the results) has been through a copy before the timed region
    for _ in range(2):
        step()
    torch.cuda.synchronize(dev)
    barrier(world)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    cin.wait_stream(stream)
    cout.wait_stream(stream)
    for _ in range(steps):
        step()
    comp.wait_stream(cout)  # the timed region ends when the last step's last result is on the host
    comp.wait_stream(cin)
    t1.record(stream)
    torch.cuda.synchronize(dev)
    ms = max_over_ranks(t0.elapsed_time(t1), world, dev)
    return {"value": round(world * steps * flops_per_step / (ms * 1e-3) / 1e12, 2), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "note": "MLA fwd+bwd FLOPs over the whole step incl. indexer and host copies; query chunks of 4096 "
                    "with copies overlapping compute on two copy streams; each step copies all its inputs in "
                    "(two device input sets used by alternate steps) and all its results out; measured after "
                    "one untimed pass of the whole leg"}


def time_workload(name, args, dev, stream) -> dict:
    """One workload of the pages' table on this GPU: MLA fwd+bwd TFLOP/s and % of the sustained bf16
    peak (CUDA events on the launching stream, median over the timed steps), and the indexer's
    tokens/s where the workload has one.  Indices come from the indexer (32k path, THD packing with
    IndexShare over its layers) or are random causal sets (the others), drawn with the same seeded
    recipe as the tests; the backward gets the forward's residual of O, as in the benchmark step."""
    import torch

    import sparse_attention_mla_gb300 as dsa
    from sparse_attention_mla_gb300 import synth

    peak = load_peaks().get("bf16_tflops_sustained")
    c = synth.WORKLOADS[name]
    T, Hh, Dqk, Dv, Kw, scale = c["T"], c["H"], c["Dqk"], c["Dv"], c["K"], c["scale"]
    layers = c.get("layers", 1)
    g = synth.generator(0)
    if "nseq" in c:
        cu = synth.cu_seqlens_from_lengths(synth.thd_lengths(c["nseq"], c["lo"], c["hi"], T, g))
    else:
        cu = torch.tensor([0, T], dtype=torch.int32)
    st, _, _, _ = dsa.dsa_packed_metadata(cu.to(dev), T)
    idx_ms = None
    P = c.get("pool")
    meta = None
    if P:  # k-pool selection: the K - P + 1 best pools of 4 tokens, then the tail tokens
        meta = dsa.dsa_kpool_metadata(cu.to(dev), T, P)
        ind = synth.indexer_inputs(T, c["Hi"], c["Di"], seed=0, device=dev)
        k_pool = dsa.dsa_kpool_pool(ind["k_idx"], meta)
        wi = torch.zeros(int(dsa.load_library().dsa_kpool_topk_workspace_size(T, Kw - P + 1)), dtype=torch.uint8,
                         device=dev)
        run_idx = lambda: dsa.dsa_kpool_topk(ind["q_idx"], k_pool, ind["w"], meta, Kw - P + 1, workspace=wi)
        for _ in range(args.warmup):
            idx, ln = run_idx()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        for a, b in ev:
            a.record(stream)
            idx, ln = run_idx()
            b.record(stream)
        torch.cuda.synchronize(dev)
        idx_ms = statistics.median(a.elapsed_time(b) for a, b in ev)
        if dsa.dsa_read_device_status(wi) != 0:
            raise RuntimeError("device status after the k-pool selection")
        del ind, k_pool
    elif "Hi" in c:
        ind = synth.indexer_inputs(T, c["Hi"], c["Di"], seed=0, device=dev)
        wi = torch.zeros(dsa.workspace_size("indexer", T, Kw), dtype=torch.uint8, device=dev)
        run_idx = lambda: dsa.dsa_indexer_topk(ind["q_idx"], ind["k_idx"], ind["w"], st, Kw, workspace=wi)
        for _ in range(args.warmup):
            idx, ln = run_idx()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
        for a, b in ev:
            a.record(stream)
            idx, ln = run_idx()
            b.record(stream)
        torch.cuda.synchronize(dev)
        idx_ms = statistics.median(a.elapsed_time(b) for a, b in ev)
        del ind
    else:
        idx = synth.random_causal_topk(st.cpu(), Kw, g).to(dev)
        ln = (idx >= 0).sum(1).to(torch.int32)
    x = synth.mla_inputs(T, Hh, Dqk, Dv, seed=1000, device=dev)
    kv_rows, extra = x["kv"], 0
    if meta is not None:  # attention over [pooled kv; kv]
        extra = meta.total_pools
        kv_rows = torch.empty(extra + T, Dqk, dtype=torch.bfloat16, device=dev)
        kv_rows[extra:] = x["kv"]
    wf = torch.zeros(dsa.workspace_size("fwd", T, Hh), dtype=torch.uint8, device=dev)
    wb = torch.zeros(dsa.workspace_size("bwd", T, Hh, Kw), dtype=torch.uint8, device=dev)
    out = torch.empty(T, Hh, Dv, dtype=torch.bfloat16, device=dev)
    lo = torch.empty_like(out)
    lse = torch.empty(T, Hh, dtype=torch.float32, device=dev)
    dq = torch.empty(T, Hh, Dqk, dtype=torch.bfloat16, device=dev)
    dkv = torch.empty(extra + T, Dqk, dtype=torch.float32, device=dev)
    dkv_tok = torch.empty(T, Dqk, dtype=torch.float32, device=dev) if meta is not None else None
    evs = []

    def step(rec):
        for _ in range(layers):  # IndexShare: every layer reuses the one selection
            e = [torch.cuda.Event(enable_timing=True) for _ in range(5)] if rec else None
            if e: e[3].record(stream)
            if meta is not None:  # this layer's pooled kv rows
                dsa.dsa_kpool_pool(x["kv"], meta, out=kv_rows[:extra])
            if e: e[0].record(stream)
            dsa.dsa_sparse_mla_fwd(x["q"], kv_rows, idx, scale, topk_len=ln, out=out, lse=lse, workspace=wf,
                                   out_lo=lo, Dv=Dv)
            if e: e[1].record(stream)
            dsa.dsa_sparse_mla_bwd(x["q"], kv_rows, idx, scale, out, lse, x["dout"], topk_len=ln, dq=dq,
                                   dkv_accum=dkv, workspace=wb, out_lo=lo)
            if e: e[2].record(stream)
            if meta is not None:  # the key gradient back to the tokens
                dsa.dsa_kpool_unpool_grad(dkv, meta, dx=dkv_tok)
            if e: e[4].record(stream)
            if e: evs.append(e)

    for _ in range(args.warmup):
        step(False)
    for _ in range(args.steps):
        step(True)
    torch.cuda.synchronize(dev)
    for w_ in (wf, wb):
        if dsa.dsa_read_device_status(w_) != 0:
            raise RuntimeError(f"device status after workload {name}")
    n = int(ln.sum().item())
    fwd_ms = statistics.median(e[0].elapsed_time(e[1]) for e in evs)
    bwd_ms = statistics.median(e[1].elapsed_time(e[2]) for e in evs)
    ff = 2.0 * Hh * n * (Dqk + Dv)
    fb = 2.0 * Hh * n * (3 * Dqk + 2 * Dv)
    tf = (ff + fb) / ((fwd_ms + bwd_ms) * 1e-3) / 1e12
    line = {"workload": name, "T": T, "H": Hh, "Dqk": Dqk, "K": Kw, "layers": layers, "n_valid_slots": n,
            "mla_fwd_ms": round(fwd_ms, 3), "mla_bwd_ms": round(bwd_ms, 3), "mla_tflops": round(tf, 2),
            "mla_pct_bf16_sustained": round(100 * tf / peak, 2) if peak else None,
            "fwd_tflops": round(ff / (fwd_ms * 1e-3) / 1e12, 2), "bwd_tflops": round(fb / (bwd_ms * 1e-3) / 1e12, 2),
            "timing": f"CUDA events, {args.warmup} warm-up and {args.steps} timed steps, median"}
    if idx_ms is not None:
        line.update({"indexer_ms": round(idx_ms, 3), "indexer_tokens_per_s": round(T / (idx_ms * 1e-3), 1)})
    if meta is not None:
        line.update({"pool": P, "total_pools": meta.total_pools, "selection": "k-pool (indexer over pooled keys + tail)",
                     "kv_pool_ms": round(statistics.median(e[3].elapsed_time(e[0]) for e in evs), 3),
                     "unpool_grad_ms": round(statistics.median(e[2].elapsed_time(e[4]) for e in evs), 3)})
    del x, out, lo, dq, dkv, idx, ln, wf, wb, kv_rows, dkv_tok
    torch.cuda.empty_cache()
    return line


def run_workloads(args, local):
    """Each named workload of the pages' table on one GPU, one JSON line each (not the benchmark line)."""
    import torch

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream(dev)
    for name in args.workloads.split(","):
        print(json.dumps(time_workload(name, args, dev, stream)), flush=True)


def traffic_per_launch(kernel: str, src_file: str, units: int):
    """DRAM bytes of one launch from the committed ncu capture (profiles/traffic.json), scaled from the
    captured launch by the units processed (valid slots, or tokens for the indexer); None when the
    capture was taken on different kernel source."""
    tfile = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(tfile):
        return None
    with open(tfile) as f:
        tr = json.load(f).get(kernel)
    if not tr or tr.get("kernel_rev") != kernel_rev(src_file):
        return None
    per = tr.get("bytes_per_valid_slot", tr.get("bytes_per_token"))
    return None if per is None else per * units


def kernel_rev(src_name: str) -> str:
    """Content hash of a kernel source: ncu counters are reused only for the same code."""
    import hashlib

    h = hashlib.sha256()
    for name in (src_name, "dsa_device.cuh"):  # the kernel source and the device helpers it inlines
        with open(os.path.join(ROOT, "sparse_attention_mla_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="cuda", choices=["cuda", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cp", action="store_true", help="skip the context-parallel indexer line")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true", help="skip the V3.2, NoPE and k-pool workload timings")
    ap.add_argument("--no-kl", action="store_true", help="skip the indexer KL loss path")
    ap.add_argument("--workloads", default=None,
                    help="comma-separated workload names (tiny,v32,idx32k,nope,thd,kpool): one line per workload "
                         "instead of the benchmark line")
    ap.add_argument("--seq", type=int, default=32768,
                    help="sequence length; only for small-case profiler captures (the benchmark is 32768)")
    args = ap.parse_args()
    global S
    S = args.seq
    if args.warmup < 3 and args.impl == "cuda":
        args.warmup = 3
    if args.workloads:
        run_workloads(args, int(os.environ.get("LOCAL_RANK", "0")))
        return
    rank, world, local = dist_init()
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        run_cuda(args, rank, world, local)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()

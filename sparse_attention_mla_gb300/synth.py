"""Seeded synthetic inputs for the DSA hot path.

This module only draws random tensors and index sets with the shapes and
structure of the pages' workloads; it holds none of the method's arithmetic
(no scores, no softmax, no selection), so both the CUDA path and the CPU
oracle can take their inputs from it.

Recipe (one ``torch.Generator`` per call, seeded):
  * q, kv, dO ~ N(0, 1) drawn in fp32 then rounded to bf16 (in that order);
  * index q_idx, k_idx ~ N(0, 1) -> bf16; head weights w = U(0, 1) / 8 in fp32;
  * random causal top-k: per row t with window [start, t] of length c and
    n = min(K, c) valid slots, a uniform n-subset of the window, sorted
    ascending, then K - n copies of -1;
  * packed THD lengths: n ints U[lo, hi], rescaled by floor to sum to
    ``total``, the remainder going to the last sequence.
"""
from __future__ import annotations

import torch


def generator(seed: int, device: str | torch.device = "cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def randn_bf16(shape, g: torch.Generator, device="cpu") -> torch.Tensor:
    return torch.randn(*shape, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def thd_lengths(n: int, lo: int, hi: int, total: int, g: torch.Generator) -> list[int]:
    """n sequence lengths drawn from U[lo, hi] and rescaled to sum to ``total``."""
    raw = torch.randint(lo, hi + 1, (n,), generator=g).tolist()
    s = sum(raw)
    lens = [int(x * total // s) for x in raw]
    lens[-1] += total - sum(lens)
    return lens


def cu_seqlens_from_lengths(lengths) -> torch.Tensor:
    cu = [0]
    for x in lengths:
        cu.append(cu[-1] + int(x))
    return torch.tensor(cu, dtype=torch.int32)


def starts_from_cu(cu_seqlens: torch.Tensor, T: int) -> torch.Tensor:
    """Per-token sequence start (the structure of the packing, not a method step)."""
    cu = cu_seqlens.tolist()
    st = torch.empty(T, dtype=torch.int32)
    for a, b in zip(cu[:-1], cu[1:]):
        st[a:b] = a
    return st


def random_causal_topk(seq_start: torch.Tensor, K: int, g: torch.Generator,
                       rows: torch.Tensor | None = None) -> torch.Tensor:
    """Random causal index sets: uniform n-subset of [start(t), t], ascending, -1 suffix."""
    T = seq_start.numel()
    rows = torch.arange(T) if rows is None else rows
    out = torch.full((rows.numel(), K), -1, dtype=torch.int32)
    st = seq_start.tolist()
    for r, t in enumerate(rows.tolist()):
        b = st[t]
        c = t - b + 1
        n = min(K, c)
        if c <= K:
            sel = torch.arange(b, t + 1, dtype=torch.int32)
        else:
            sel = (torch.randperm(c, generator=g)[:n] + b).to(torch.int32).sort().values
        out[r, :n] = sel
    return out


def mla_inputs(T: int, H: int, Dqk: int, Dv: int, seed: int, device="cpu", Tk: int | None = None,
               with_grad: bool = True) -> dict:
    """q [T,H,Dqk], kv [Tk,Dqk], dO [T,H,Dv] bf16 ~ N(0,1), drawn in that order."""
    Tk = T if Tk is None else Tk
    g = generator(seed, device)
    out = {
        "q": randn_bf16((T, H, Dqk), g, device),
        "kv": randn_bf16((Tk, Dqk), g, device),
    }
    if with_grad:
        out["dout"] = randn_bf16((T, H, Dv), g, device)
    return out


def indexer_inputs(T: int, Hi: int, Di: int, seed: int, device="cpu", Tk: int | None = None) -> dict:
    """q_idx [T,Hi,Di], k_idx [Tk,Di] bf16 ~ N(0,1); w [T,Hi] fp32 ~ U(0,1)/8."""
    Tk = T if Tk is None else Tk
    g = generator(seed, device)
    q_idx = randn_bf16((T, Hi, Di), g, device)
    k_idx = randn_bf16((Tk, Di), g, device)
    w = torch.rand(T, Hi, generator=g, device=device, dtype=torch.float32) / 8.0
    return {"q_idx": q_idx, "k_idx": k_idx, "w": w}


# Workloads of the pages (shapes only).  Sizes: T tokens, H heads, Dqk/Dv widths, K top-k.
WORKLOADS = {
    "tiny": dict(T=256, H=16, Dqk=576, Dv=512, K=64, scale=192 ** -0.5),
    "v32": dict(T=4096, H=128, Dqk=576, Dv=512, K=2048, scale=192 ** -0.5),
    "idx32k": dict(T=32768, H=64, Dqk=576, Dv=512, K=2048, scale=192 ** -0.5, Hi=64, Di=128),
    "nope": dict(T=16384, H=8, Dqk=512, Dv=512, K=2051, scale=512 ** -0.5),
    "thd": dict(T=131072, H=64, Dqk=576, Dv=512, K=2048, scale=192 ** -0.5, Hi=64, Di=128,
                nseq=8, lo=4096, hi=32768, layers=4),
    # GLM-5.3-Flash k-pool selection: pools of 4 tokens, 2048 pools + the 3-token tail = 2051
    "kpool": dict(T=16384, H=8, Dqk=512, Dv=512, K=2051, scale=512 ** -0.5, Hi=64, Di=128, pool=4),
}

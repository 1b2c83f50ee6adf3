"""Seeded synthetic inputs for the KDA workloads (shared by tests, bench and smoke).

This module only draws random numbers with the distributions of each workload; it holds none of
the method's arithmetic.  Draw order from one torch CPU generator seeded per call:
q, k, v, beta-logits, g-or-a, A_log, dt_bias, dO.  Inputs are drawn in fp32 and rounded to their
storage type (bf16 for q, k, v, beta, dO; fp32 for g / a, A_log, dt_bias), so every consumer reads
the same values.

Workloads (documents packed back to back, head dim 128, chunk 64):
  m2        2048/1500 tokens, 4 heads, g form, g = logsigmoid(N(0,1))/16, q,k unit L2 per head
  R2        9000/5000/2384 tokens, 4 heads, raw form: a ~ N(0,1), A_log ~ U(0, ln 16) per head,
            dt_bias ~ U(-1, 1) per channel; R2fast: A_log ~ U(ln 8, ln 32)
  1doc      16384 tokens, 64 heads, g form, g = logsigmoid(N(0,1))/8, fused L2 norm of raw
            q,k ~ N(0,1)
  4doc      8192/4096/3072/1024 tokens, 64 heads, raw form as R2, unit q,k
  4doc-h16  the same with 16 heads (profiling case)
  longpack  120000/70000/40000/19856 tokens, 16 heads, g form /16, unit q,k; 8 fragments per doc
In every workload v, dO ~ N(0,1), beta = sigmoid(N(0,1)), zero initial state.

Conv inputs (the width-4 causal conv1d + SiLU ahead of q / k / v; conv_inputs): draw order x
~ N(0,1) [T, C] (bf16), taps w ~ N(0,1)/2 [C, 4], bias ~ N(0,1)/10 [C], halo ~ N(0,1) [N, 3, C]
(bf16, when asked for), dy ~ N(0,1) [T, C].
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

D = 128


@dataclass(frozen=True)
class Workload:
    name: str
    lens: tuple
    H: int
    gate: str            # "g" or "raw"
    l2norm: bool         # fused L2 norm in the kernel (raw q, k ~ N(0,1)); else unit q, k
    gdiv: float = 16.0   # g = logsigmoid(N(0,1)) / gdiv in g form
    A_log_range: tuple = (0.0, math.log(16.0))
    fragments: int = 0   # fragments per document for the fragment-walk workload
    notes: str = field(default="", compare=False)

    @property
    def T(self):
        return int(sum(self.lens))

    @property
    def N(self):
        return len(self.lens)

    @property
    def row(self):
        return f"{self.name}:{self.gate}:{'fused' if self.l2norm else 'off'}"


WORKLOADS = {
    "m2": Workload("m2", (2048, 1500), 4, "g", False, 16.0),
    "R2": Workload("R2", (9000, 5000, 2384), 4, "raw", False),
    "R2fast": Workload("R2fast", (9000, 5000, 2384), 4, "raw", False,
                       A_log_range=(math.log(8.0), math.log(32.0))),
    "1doc": Workload("1doc", (16384,), 64, "g", True, 8.0),
    "4doc": Workload("4doc", (8192, 4096, 3072, 1024), 64, "raw", False),
    # 4doc with 16 heads: the profiling case (inputs still larger than L2, a quarter of the units)
    "4doc-h16": Workload("4doc-h16", (8192, 4096, 3072, 1024), 16, "raw", False),
    "longpack": Workload("longpack", (120000, 70000, 40000, 19856), 16, "g", False, 16.0,
                         fragments=8),
}


def cu_from_lens(lens):
    out = [0]
    for n in lens:
        out.append(out[-1] + int(n))
    return torch.tensor(out, dtype=torch.int32)


def fragment_lens(doc_len, nfrag):
    """nfrag contiguous pieces of equal length, the remainder on the last one."""
    base = doc_len // nfrag
    return [base] * (nfrag - 1) + [doc_len - base * (nfrag - 1)]


def make_inputs(lens, H, *, gate="g", l2norm=False, gdiv=16.0,
                A_log_range=(0.0, math.log(16.0)), seed=0, with_dO=True):
    """Draws one workload's inputs on the CPU; returns a dict of tensors."""
    T = int(sum(lens))
    gen = torch.Generator("cpu").manual_seed(seed)
    q = torch.randn((T, H, D), generator=gen)
    k = torch.randn((T, H, D), generator=gen)
    if not l2norm:
        q = q / q.norm(dim=-1, keepdim=True).clamp_min(1e-12)
        k = k / k.norm(dim=-1, keepdim=True).clamp_min(1e-12)
    v = torch.randn((T, H, D), generator=gen)
    beta = torch.sigmoid(torch.randn((T, H), generator=gen))
    x = torch.randn((T, H, D), generator=gen)
    out = dict(q=q.bfloat16(), k=k.bfloat16(), v=v.bfloat16(), beta=beta.bfloat16(),
               cu_seqlens=cu_from_lens(lens))
    if gate == "g":
        out["g"] = torch.nn.functional.logsigmoid(x) / gdiv
        out["A_log"] = out["dt_bias"] = None
    else:
        lo, hi = A_log_range
        out["g"] = x  # the raw pre-activation a
        out["A_log"] = torch.rand((H,), generator=gen) * (hi - lo) + lo
        out["dt_bias"] = torch.rand((H, D), generator=gen) * 2.0 - 1.0
    if with_dO:
        out["dO"] = torch.randn((T, H, D), generator=gen).bfloat16()
    return out


def workload_inputs(name, seed=0, with_dO=True):
    w = WORKLOADS[name]
    return make_inputs(w.lens, w.H, gate=w.gate, l2norm=w.l2norm, gdiv=w.gdiv,
                       A_log_range=w.A_log_range, seed=seed, with_dO=with_dO)


def conv_inputs(lens, C, *, seed=0, halo=False, bias=True):
    """Inputs of the conv1d + SiLU on the CPU: dict x, w, bias, halo (or None), dy (fp32),
    cu_seqlens."""
    gen = torch.Generator("cpu").manual_seed(seed)
    T = int(sum(lens))
    x = torch.randn((T, C), generator=gen).bfloat16()
    w = torch.randn((C, 4), generator=gen) * 0.5
    b = torch.randn((C,), generator=gen) * 0.1 if bias else None
    h = torch.randn((len(lens), 3, C), generator=gen).bfloat16() if halo else None
    dy = torch.randn((T, C), generator=gen)
    return dict(x=x, w=w, bias=b, halo=h, dy=dy, cu_seqlens=cu_from_lens(lens))

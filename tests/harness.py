"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI binding, run the
oracle on the same (bf16/fp32-rounded) values, and score the difference."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from linear_attention_chunked_gb300 import kda

# max|x - ref| / rms(ref) bounds per output
TOL = dict(o=2e-2, ht=1e-3, dq=3e-2, dk=3e-2, dv=3e-2, dbeta=3e-2, dg=5e-2, dA_log=5e-2,
           ddt_bias=5e-2, dh0=3e-2)


def rel_err(x, ref):
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = np.sqrt(np.mean(ref * ref)) if ref.size else 0.0
    if ref.size == 0:
        return 0.0
    return float(np.max(np.abs(x - ref)) / max(rms, 1e-30))


def to_dev(inp, device="cuda"):
    return {k: (v.to(device) if torch.is_tensor(v) else v) for k, v in inp.items()}


def gpu_fwd_bwd(inp, *, gate, l2norm, h0=None, dht=None, saved_mode=True, want_bwd=True,
                out_dtype=torch.float32, group_chunks=0):
    d = to_dev(inp)
    h0d = None if h0 is None else torch.as_tensor(h0, dtype=torch.float32).cuda()
    dhtd = None if dht is None else torch.as_tensor(dht, dtype=torch.float32).cuda()
    o, ht, saved = kda.kda_fwd(d["q"], d["k"], d["v"], d["beta"], d["g"], d["cu_seqlens"],
                               gate=gate, A_log=d["A_log"], dt_bias=d["dt_bias"], h0=h0d,
                               l2norm=l2norm, save=saved_mode, out_dtype=out_dtype,
                               group_chunks=group_chunks)
    out = dict(o=o, ht=ht)
    if want_bwd:
        g = kda.kda_bwd(d["q"], d["k"], d["v"], d["beta"], d["g"], d["cu_seqlens"], d["dO"],
                        saved=saved if saved_mode else None, gate=gate, A_log=d["A_log"],
                        dt_bias=d["dt_bias"], h0=h0d, dht=dhtd, l2norm=l2norm,
                        out_dtype=out_dtype, group_chunks=group_chunks)
        out.update(g)
    torch.cuda.synchronize()
    return {k: v.float().cpu().numpy() for k, v in out.items()}


def f64(t):
    return None if t is None else t.float().double().numpy()


def oracle_fwd_bwd(inp, *, gate, l2norm, h0=None, dht=None, heads=None, want_bwd=True):
    """Oracle on the same values; `heads` restricts to a subset of heads (sampling)."""
    def sel(t, axis=1):
        if t is None:
            return None
        a = f64(t) if torch.is_tensor(t) else np.asarray(t, dtype=np.float64)
        return a if heads is None else np.take(a, heads, axis=axis)
    raw = gate == "raw"
    kw = dict(raw=raw, l2norm=l2norm,
              A_log=sel(inp["A_log"], 0) if raw else None,
              dt_bias=sel(inp["dt_bias"], 0) if raw else None,
              h0=sel(h0), )
    args = [sel(inp[n]) for n in ("q", "k", "v", "beta", "g")]
    cu = inp["cu_seqlens"].numpy()
    o, ht = oracle.kda_fwd(*args, cu, **kw)
    out = dict(o=o, ht=ht)
    if want_bwd:
        out.update(oracle.kda_bwd(*args, cu, sel(inp["dO"]), dht=sel(dht), **kw))
    return out


def compare(gpu, ref, heads=None, names=None, tol=TOL):
    """Returns {name: rel_err}; gpu arrays are sliced to `heads` on their head axis."""
    errs = {}
    for name, r in ref.items():
        if names is not None and name not in names:
            continue
        if name not in gpu:
            continue
        x = gpu[name]
        if heads is not None:
            axis = 0 if name in ("dA_log", "ddt_bias") else 1
            x = np.take(x, heads, axis=axis)
        errs[name] = rel_err(x, r)
    return errs


def assert_within(errs, tol=TOL, label=""):
    bad = {k: v for k, v in errs.items() if v > tol[k]}
    assert not bad, f"{label}: over tolerance {bad} (all: {errs})"

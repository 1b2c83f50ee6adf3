"""GPU parity of the width-4 causal conv1d + SiLU (kda_conv_fwd / kda_conv_bwd through the C ABI)
against the FP64 oracle (oracle/conv1d.py) on the same bf16 inputs.

Bounds (max|err| / rms(ref) per tensor): fp32 outputs y, dx, dhalo and the FP32-accumulated dw,
dbias are exact up to FP32 arithmetic (a 4-term dot product, sigmoid and a sum over at most a few
thousand tokens): 1e-5.  bf16 outputs are the fp32 outputs rounded to nearest (checked bitwise).
Cases: ragged documents (lengths 1, 2, 3, 5, 64, 511, 513, an empty one) so that documents start
inside and at the edge of every thread's 64-token run and block's 512-token row, with and without
halo rows and bias, SiLU on and off, and the q-sized workload (16384 tokens, 64 heads x 128
channels) on sampled channels.  Results are bitwise reproducible.
"""
import numpy as np
import pytest
import torch

from harness import rel_err
from linear_attention_chunked_gb300 import inputs, kda
from oracle import conv1d

pytestmark = pytest.mark.gpu

TOL = 1e-5


def _make(lens, C, seed, halo=False, bias=True):
    c = inputs.conv_inputs(lens, C, seed=seed, halo=halo, bias=bias)
    return c["x"], c["w"], c["bias"], c["halo"], c["dy"], c["cu_seqlens"]


def _np(t):
    return None if t is None else t.double().numpy()


def _run(x, w, b, h, dy, cu, act, out_dtype):
    d = lambda t: None if t is None else t.cuda()  # noqa: E731
    y = kda.kda_conv_fwd(d(x), d(w), d(cu), bias=d(b), halo=d(h), activation=act,
                         out_dtype=out_dtype)
    g = kda.kda_conv_bwd(d(x), d(w), d(cu), d(dy.to(out_dtype)), bias=d(b), halo=d(h),
                         activation=act)
    torch.cuda.synchronize()
    out = {"y": y.float().cpu().numpy()}
    out.update({k: v.float().cpu().numpy() for k, v in g.items()})
    return out


CASES = {
    "ragged": dict(lens=[5, 1, 2, 0, 3, 64, 511, 513, 70], C=136),
    "halo": dict(lens=[1, 2, 3, 200, 0, 515], C=64, halo=True),
    "no_bias_no_act": dict(lens=[100, 7, 300], C=24, bias=False, act=False),
}


@pytest.mark.parametrize("case", list(CASES))
def test_conv_against_oracle(case):
    c = dict(CASES[case])
    act = c.pop("act", True)
    x, w, b, h, dy, cu = _make(c["lens"], c["C"], seed=len(case), halo=c.get("halo", False),
                               bias=c.get("bias", True))
    gpu = _run(x, w, b, h, dy, cu, act, torch.float32)
    y_ref, _ = conv1d.conv_fwd(_np(x), _np(w), cu.numpy(), bias=_np(b), halo=_np(h), activation=act)
    g_ref = conv1d.conv_bwd(_np(x), _np(w), cu.numpy(), _np(dy.float()), bias=_np(b), halo=_np(h),
                            activation=act)
    errs = {"y": rel_err(gpu["y"], y_ref), "dx": rel_err(gpu["dx"], g_ref["dx"]),
            "dw": rel_err(gpu["dw"], g_ref["dw"])}
    if b is not None:
        errs["dbias"] = rel_err(gpu["dbias"], g_ref["db"])
    if h is not None:
        errs["dhalo"] = rel_err(gpu["dhalo"], g_ref["dhalo"])
    print(case, {k: f"{v:.2e}" for k, v in errs.items()})
    assert all(v <= TOL for v in errs.values()), errs
    # bf16 outputs are the fp32 outputs rounded to nearest; a second run is bitwise equal
    bf = _run(x, w, b, h, dy, cu, act, torch.bfloat16)
    assert np.array_equal(bf["y"], torch.tensor(gpu["y"]).bfloat16().float().numpy())
    again = _run(x, w, b, h, dy, cu, act, torch.float32)
    for k in gpu:
        assert np.array_equal(again[k], gpu[k]), k


def test_conv_halo_split_matches_whole_document():
    # a document cut into fragments, each fragment's halo = the three tokens before it, gives the
    # whole document's outputs; the halo gradients flow back into those tokens' dx
    lens, C = [700], 32
    x, w, b, _, dy, cu = _make(lens, C, seed=7)
    whole = _run(x, w, b, None, dy, cu, True, torch.float32)
    cuts = [0, 130, 131, 400, 700]
    fcu = torch.tensor(cuts, dtype=torch.int32)
    halo = torch.zeros((len(cuts) - 1, 3, C)).bfloat16()
    for f, s in enumerate(cuts[:-1]):
        for i in range(3):
            if s - 3 + i >= 0 and f > 0:
                halo[f, i] = x[s - 3 + i]
    frag = _run(x, w, b, halo, dy, fcu, True, torch.float32)
    assert rel_err(frag["y"], whole["y"]) <= TOL
    assert rel_err(frag["dw"], whole["dw"]) <= TOL
    dx = frag["dx"].copy()
    for f, s in enumerate(cuts[:-1]):
        for i in range(3):
            if s - 3 + i >= 0 and f > 0:
                dx[s - 3 + i] += frag["dhalo"][f, i]
    assert rel_err(dx, whole["dx"]) <= TOL


def test_conv_full_size_sampled_channels():
    # q of the 4doc workload: 16384 tokens in documents of 8192 / 4096 / 3072 / 1024, 64 heads x
    # 128 channels, the launch configuration of a full-size call; the oracle checks 3 heads' worth
    # of channels (per-channel computations are independent)
    w_ = inputs.WORKLOADS["4doc"]
    C = w_.H * 128
    x, w, b, _, dy, cu = _make(list(w_.lens), C, seed=9)
    gpu = _run(x, w, b, None, dy, cu, True, torch.float32)
    ch = np.r_[0:128, 4096:4224, C - 128:C]
    xs, ws, bs, dys = _np(x)[:, ch], _np(w)[ch], _np(b)[ch], _np(dy.float())[:, ch]
    y_ref, _ = conv1d.conv_fwd(xs, ws, cu.numpy(), bias=bs)
    g_ref = conv1d.conv_bwd(xs, ws, cu.numpy(), dys, bias=bs)
    errs = {"y": rel_err(gpu["y"][:, ch], y_ref), "dx": rel_err(gpu["dx"][:, ch], g_ref["dx"]),
            "dw": rel_err(gpu["dw"][ch], g_ref["dw"]), "dbias": rel_err(gpu["dbias"][ch], g_ref["db"])}
    print("4doc q", {k: f"{v:.2e}" for k, v in errs.items()})
    assert all(v <= TOL for v in errs.values()), errs

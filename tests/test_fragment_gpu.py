"""GPU parity of the fragment path: fragment summaries (M, B, C), the transfer walk in both
directions, and the documents finished fragment by fragment, against the unfragmented oracle."""
import numpy as np
import pytest
import torch

import oracle
from harness import TOL, assert_within, compare, f64, oracle_fwd_bwd, rel_err, to_dev
from linear_attention_chunked_gb300 import inputs, kda

pytestmark = pytest.mark.gpu


def _split(lens, nfrag):
    frag, doc_frag = [], [0]
    for L in lens:
        pieces = inputs.fragment_lens(L, nfrag)
        frag += pieces
        doc_frag.append(doc_frag[-1] + len(pieces))
    return frag, doc_frag


def run_fragment_path(inp, lens, nfrag, *, gate, l2norm, h0=None, dht=None):
    """fwd + saved bwd of the documents via summaries, walks and per-fragment finishing."""
    frag, doc_frag = _split(lens, nfrag)
    d = to_dev(inp)
    fcu = inputs.cu_from_lens(frag).cuda()
    dfr = torch.tensor(doc_frag, dtype=torch.int32, device="cuda")
    args = (d["q"], d["k"], d["v"], d["beta"], d["g"], fcu)
    kw = dict(gate=gate, A_log=d["A_log"], dt_bias=d["dt_bias"], l2norm=l2norm)
    M, B = kda.kda_fragment_summary(*args, mode=kda.KDA_FRAG_FWD, **kw)
    h0d = None if h0 is None else torch.as_tensor(h0).float().cuda()
    dhtd = None if dht is None else torch.as_tensor(dht).float().cuda()
    S_in, S_fin = kda.kda_transfer_walk(dfr, M, B, h0d)
    o, _, saved = kda.kda_fwd(*args, h0=S_in, **kw)
    C = kda.kda_fragment_summary(*args, mode=kda.KDA_FRAG_BWD, dO=d["dO"], **kw)
    dS_end, dh0 = kda.kda_transfer_walk(dfr, M, C, dhtd, reverse=True)
    g = kda.kda_bwd(*args, d["dO"], saved=saved, h0=S_in, dht=dS_end, **kw)
    torch.cuda.synchronize()
    out = dict(o=o, ht=S_fin, dh0=dh0, M=M, B=B, C=C)
    out.update({k: v for k, v in g.items() if k != "dh0"})
    return {k: v.float().cpu().numpy() for k, v in out.items()}, frag


@pytest.mark.parametrize("gate,l2norm", [("g", False), ("raw", True)])
def test_fragment_path_small(gate, l2norm):
    lens = [300, 77, 129]
    inp = inputs.make_inputs(lens, 2, gate=gate, l2norm=l2norm, gdiv=64.0, seed=11)
    rng = np.random.default_rng(3)
    h0 = rng.standard_normal((3, 2, 128, 128)).astype(np.float32) * 0.1
    dht = rng.standard_normal((3, 2, 128, 128)).astype(np.float32) * 0.1
    gpu, frag = run_fragment_path(inp, lens, 4, gate=gate, l2norm=l2norm, h0=h0, dht=dht)
    ref = oracle_fwd_bwd(inp, gate=gate, l2norm=l2norm, h0=h0, dht=dht)
    errs = compare(gpu, ref)
    print({k: f"{v:.2e}" for k, v in errs.items()})
    assert_within(errs, label=f"fragments {gate}")
    # the summaries themselves against the oracle's fragment algebra
    raw = gate == "raw"
    oargs = [f64(inp[n]) for n in ("q", "k", "v", "beta", "g")]
    okw = dict(raw=raw, l2norm=l2norm, A_log=f64(inp["A_log"]) if raw else None,
               dt_bias=f64(inp["dt_bias"]) if raw else None)
    fcu = inputs.cu_from_lens(frag).numpy()
    M, B = oracle.fragment_summary(*oargs, fcu, **okw)
    C = oracle.fragment_summary(*oargs, fcu, mode=1, dO=f64(inp["dO"]), **okw)
    # B and C are states: the final-state bound.  M is a transition product whose entries span
    # many orders of magnitude (a few slow channels near 1, the rest decayed towards 0), so it is
    # scored against its largest entry; its effect on states is covered by ht / dh0 above.
    errs = {"B": rel_err(gpu["B"], B), "C": rel_err(gpu["C"], C),
            "M": float(np.max(np.abs(gpu["M"] - M)) / np.max(np.abs(M)))}
    assert errs["B"] < TOL["ht"] and errs["C"] < TOL["ht"] and errs["M"] < 1e-4, errs


# max|err| / rms(ref) of each walk product format against the FP64 oracle walk on the same FP32
# M, B, S0: every format but plain TF32 is accurate to FP32 rounding; plain TF32 keeps 11
# significant bits per operand (unit roundoff 2^-11 ~ 4.9e-4 per product term)
WALK_TOL = {"fp32": 1e-5, "tf32": 2e-2, "tf32_hilo": 1e-5, "bf16x3": 1e-5, "bf16x3_hw": 1e-5}


def _walk_case(F=7, H=3, seed=0):
    gen = torch.Generator("cpu").manual_seed(seed)
    M = (torch.randn((F, H, 128, 128), generator=gen) * 0.05).cuda()
    B = torch.randn((F, H, 128, 128), generator=gen).cuda()
    S0 = torch.randn((4, H, 128, 128), generator=gen).cuda()
    doc_frag = [0, 2, 2, 6, 7]  # fragments per document: 2, 0 (empty), 4, 1
    return M, B, S0, doc_frag


@pytest.mark.parametrize("prec", list(WALK_TOL))
def test_walk_formats_against_oracle(prec):
    # every column of every S_in must be written (NaN prefill), the values must match the oracle
    # walk within the format's bound, both directions, with and without a start state, and a
    # second run must be bitwise equal
    M, B, S0, doc_frag = _walk_case()
    F, H = M.shape[:2]
    dfr = torch.tensor(doc_frag, dtype=torch.int32, device="cuda")
    p = kda.WALK_PRECISIONS[prec]
    for rev in (False, True):
        for s0 in (None, S0):
            S_in = torch.full((F, H, 128, 128), float("nan"), device="cuda")
            S_fin = torch.full((4, H, 128, 128), float("nan"), device="cuda")
            ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
            kda.kda_transfer_walk(dfr, M, B, s0, reverse=rev, precision=p, S_in=S_in,
                                  S_final=S_fin, ws=ws)
            assert kda.kda_read_device_status(ws) == kda.KDA_OK
            again = kda.kda_transfer_walk(dfr, M, B, s0, reverse=rev, precision=p)
            torch.cuda.synchronize()
            assert not torch.isnan(S_in).any() and not torch.isnan(S_fin).any()
            assert torch.equal(again[0], S_in) and torch.equal(again[1], S_fin)
            S_ref, fin_ref = oracle.transfer_walk(
                doc_frag, M.double().cpu().numpy(), B.double().cpu().numpy(),
                None if s0 is None else s0.double().cpu().numpy(), reverse=rev)
            e_in, e_fin = rel_err(S_in.cpu().numpy(), S_ref), rel_err(S_fin.cpu().numpy(), fin_ref)
            print(prec, "reverse" if rev else "forward", "S0" if s0 is not None else "zero",
                  f"S_in {e_in:.2e} S_final {e_fin:.2e}")
            assert e_in < WALK_TOL[prec] and e_fin < WALK_TOL[prec], (e_in, e_fin)


def test_walk_half_width_matches_full_width():
    M, B, S0, doc_frag = _walk_case(seed=1)
    dfr = torch.tensor(doc_frag, dtype=torch.int32, device="cuda")
    full = kda.kda_transfer_walk(dfr, M, B, S0, precision=kda.KDA_WALK_BF16X3)
    half = kda.kda_transfer_walk(dfr, M, B, S0, precision=kda.KDA_WALK_BF16X3_HW)
    torch.cuda.synchronize()
    for a, b in zip(full, half):
        assert rel_err(b.cpu().numpy(), a.cpu().numpy()) < 1e-6


@pytest.mark.slow
def test_longpack_sampled_heads():
    w = inputs.WORKLOADS["longpack"]
    inp = inputs.workload_inputs("longpack")
    gpu, _ = run_fragment_path(inp, w.lens, w.fragments, gate=w.gate, l2norm=w.l2norm)
    heads = [0, 9]
    ref = oracle_fwd_bwd(inp, gate=w.gate, l2norm=w.l2norm, heads=heads)
    errs = compare(gpu, ref, heads=heads)
    print("longpack", {k: f"{v:.2e}" for k, v in errs.items()})
    assert_within(errs, label="longpack")

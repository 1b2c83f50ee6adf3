"""GPU parity: the CUDA path (through the C ABI) against the FP64 oracle on the same seeded inputs.

Bounds (max|err| / rms(ref) per tensor): o 2e-2, final state 1e-3, dq/dk/dv/dbeta 3e-2,
dg/dA_log/dt_bias 5e-2 (also on fast-decay inputs).  Small cases span several chunks, ragged
tails (lengths 1, 63, 64, 65), an empty document, nonzero h0 / dht, both gate forms, the fused L2
norm and fast decay, and packs that select each value-block width of the recurrences (16, 32
and 64 columns); the full workloads run in the same launch configuration the bench times, with
heads sampled where the oracle would take too long on every head.
"""
import math

import numpy as np
import pytest
import torch

from harness import TOL, assert_within, compare, gpu_fwd_bwd, oracle_fwd_bwd, rel_err, to_dev
from linear_attention_chunked_gb300 import inputs, kda

pytestmark = pytest.mark.gpu

LN8, LN32 = math.log(8.0), math.log(32.0)

SMALL = {
    "g_edges": dict(lens=[130, 64, 1, 63, 65], H=2, gate="g", l2norm=False, gdiv=16.0),
    "g_strong": dict(lens=[200, 77], H=2, gate="g", l2norm=False, gdiv=1.0),
    "raw_empty_doc": dict(lens=[200, 0, 77], H=2, gate="raw", l2norm=False),
    "raw_fast": dict(lens=[150, 99], H=2, gate="raw", l2norm=False, A_log_range=(LN8, LN32)),
    "g_l2n": dict(lens=[96, 33], H=3, gate="g", l2norm=True, gdiv=8.0),
    "raw_l2n_fast": dict(lens=[70, 129], H=2, gate="raw", l2norm=True, A_log_range=(LN8, LN32)),
    "raw_one_head": dict(lens=[70, 64, 193], H=1, gate="raw", l2norm=False),
    # 30 (document, head) pairs: the recurrences run 32-column value blocks (16-column blocks
    # would not all fit on the SMs at once); the other small cases run 16-column blocks and the
    # many-document pack and the full workloads 64-column blocks
    "raw_30_pairs": dict(lens=[70, 1, 64, 130, 33], H=6, gate="raw", l2norm=False),
}


def _small(case, seed=1):
    c = dict(SMALL[case])
    lens, H = c.pop("lens"), c.pop("H")
    inp = inputs.make_inputs(lens, H, seed=seed, **c)
    return inp, c["gate"], c["l2norm"]


@pytest.mark.parametrize("case", list(SMALL))
@pytest.mark.parametrize("saved_mode", [True, False])
def test_small_cases(case, saved_mode):
    inp, gate, l2n = _small(case)
    N, H = inp["cu_seqlens"].numel() - 1, inp["q"].shape[1]
    rng = np.random.default_rng(7)
    h0 = rng.standard_normal((N, H, 128, 128)).astype(np.float32) * 0.1
    dht = rng.standard_normal((N, H, 128, 128)).astype(np.float32) * 0.1
    gpu = gpu_fwd_bwd(inp, gate=gate, l2norm=l2n, h0=h0, dht=dht, saved_mode=saved_mode)
    ref = oracle_fwd_bwd(inp, gate=gate, l2norm=l2n, h0=h0, dht=dht)
    assert_within(compare(gpu, ref), label=case)


@pytest.mark.parametrize("name", ["m2", "R2", "R2fast"])
def test_full_workloads_all_heads(name):
    w = inputs.WORKLOADS[name]
    inp = inputs.workload_inputs(name)
    gpu = gpu_fwd_bwd(inp, gate=w.gate, l2norm=w.l2norm)
    ref = oracle_fwd_bwd(inp, gate=w.gate, l2norm=w.l2norm)
    errs = compare(gpu, ref)
    print(name, {k: f"{v:.2e}" for k, v in errs.items()})
    assert_within(errs, label=name)


@pytest.mark.parametrize("name,saved_mode", [("1doc", True), ("4doc", True), ("4doc", False)])
def test_full_workloads_sampled_heads(name, saved_mode):
    w = inputs.WORKLOADS[name]
    inp = inputs.workload_inputs(name)
    heads = [0, 21, 42, 63]
    gpu = gpu_fwd_bwd(inp, gate=w.gate, l2norm=w.l2norm, saved_mode=saved_mode)
    ref = oracle_fwd_bwd(inp, gate=w.gate, l2norm=w.l2norm, heads=heads)
    errs = compare(gpu, ref, heads=heads)
    print(name, saved_mode, {k: f"{v:.2e}" for k, v in errs.items()})
    assert_within(errs, label=name)


def _many_docs(seed):
    # 48 short ragged documents x 4 heads: a pack with more recurrence blocks than SMs
    rng = np.random.default_rng(seed)
    lens = [int(x) for x in rng.integers(1, 200, size=48)]
    lens[:6] = [1, 63, 64, 65, 128, 0]
    return inputs.make_inputs(lens, 4, seed=seed, gate="raw", l2norm=True, A_log_range=(LN8, LN32))


@pytest.mark.parametrize("saved_mode", [True, False])
def test_many_documents(saved_mode):
    inp = _many_docs(11)
    N, H = inp["cu_seqlens"].numel() - 1, inp["q"].shape[1]
    rng = np.random.default_rng(12)
    h0 = rng.standard_normal((N, H, 128, 128)).astype(np.float32) * 0.1
    dht = rng.standard_normal((N, H, 128, 128)).astype(np.float32) * 0.1
    gpu = gpu_fwd_bwd(inp, gate="raw", l2norm=True, h0=h0, dht=dht, saved_mode=saved_mode)
    ref = oracle_fwd_bwd(inp, gate="raw", l2norm=True, h0=h0, dht=dht)
    errs = compare(gpu, ref)
    print("many documents", saved_mode, {k: f"{v:.2e}" for k, v in errs.items()})
    assert_within(errs, label="many documents")


def test_thousands_of_documents():
    # 1500 short ragged documents (empty ones included), one head: the chunk plan's block-wide
    # scan over documents (several documents per thread) and its identity launch order above
    # 1024 documents
    rng = np.random.default_rng(21)
    lens = [int(x) for x in rng.integers(0, 25, size=1500)]
    lens[:5] = [64, 0, 65, 1, 63]
    inp = inputs.make_inputs(lens, 1, seed=21, gate="raw", l2norm=False, A_log_range=(LN8, LN32))
    gpu = gpu_fwd_bwd(inp, gate="raw", l2norm=False)
    ref = oracle_fwd_bwd(inp, gate="raw", l2norm=False)
    errs = compare(gpu, ref)
    print("thousands of documents", {k: f"{v:.2e}" for k, v in errs.items()})
    assert_within(errs, label="thousands of documents")


def test_many_documents_isolation_bitwise():
    inp = _many_docs(13)
    pack = gpu_fwd_bwd(inp, gate="raw", l2norm=True)
    cu = inp["cu_seqlens"].tolist()
    for n in range(len(cu) - 1):
        a, b = cu[n], cu[n + 1]
        if a == b:
            continue
        one = {k: (v[a:b] if k in ("q", "k", "v", "beta", "g", "dO") else v)
               for k, v in inp.items()}
        one["cu_seqlens"] = torch.tensor([0, b - a], dtype=torch.int32)
        alone = gpu_fwd_bwd(one, gate="raw", l2norm=True)
        for k in ("o", "dq", "dk", "dv", "dbeta", "dg"):
            assert np.array_equal(alone[k], pack[k][a:b]), (n, k)
        for k in ("ht", "dh0"):
            assert np.array_equal(alone[k][0], pack[k][n]), (n, k)


def test_bitwise_deterministic():
    inp, gate, l2n = _small("raw_empty_doc", seed=3)
    a = gpu_fwd_bwd(inp, gate=gate, l2norm=l2n)
    b = gpu_fwd_bwd(inp, gate=gate, l2norm=l2n)
    for k in a:
        assert np.array_equal(a[k], b[k], equal_nan=True), k


def test_saved_equals_replay_bitwise():
    inp, gate, l2n = _small("raw_l2n_fast", seed=4)
    a = gpu_fwd_bwd(inp, gate=gate, l2norm=l2n, saved_mode=True)
    b = gpu_fwd_bwd(inp, gate=gate, l2norm=l2n, saved_mode=False)
    for k in a:
        assert np.array_equal(a[k], b[k]), k


@pytest.mark.parametrize("case", ["g_edges", "raw_empty_doc", "raw_l2n_fast", "raw_30_pairs"])
def test_document_isolation_bitwise(case):
    inp, gate, l2n = _small(case, seed=5)
    pack = gpu_fwd_bwd(inp, gate=gate, l2norm=l2n)
    cu = inp["cu_seqlens"].tolist()
    for n in range(len(cu) - 1):
        a, b = cu[n], cu[n + 1]
        if a == b:
            assert np.all(pack["ht"][n] == 0)
            continue
        one = {k: (v[a:b] if k in ("q", "k", "v", "beta", "g", "dO") else v)
               for k, v in inp.items()}
        one["cu_seqlens"] = torch.tensor([0, b - a], dtype=torch.int32)
        alone = gpu_fwd_bwd(one, gate=gate, l2norm=l2n)
        for k in ("o", "dq", "dk", "dv", "dbeta", "dg"):
            assert np.array_equal(alone[k], pack[k][a:b]), (n, k)
        for k in ("ht", "dh0"):
            assert np.array_equal(alone[k][0], pack[k][n]), (n, k)


def test_bounded_wait_times_out_and_reports():
    # a kernel whose mbarrier wait cannot complete gives up after 20 ms, reports KDA_ERR_TIMEOUT
    # in the status word and returns; the context stays usable for the next call
    ws = torch.zeros(4096, dtype=torch.uint8, device="cuda")
    kda.kda_selftest_wait_timeout(ws, limit_us=20000)
    assert kda.kda_read_device_status(ws) == kda.KDA_ERR_TIMEOUT
    assert kda.kda_read_device_status(ws) == kda.KDA_OK  # read clears it
    inp, gate, l2n = _small("g_edges", seed=9)
    assert_within(compare(gpu_fwd_bwd(inp, gate=gate, l2norm=l2n),
                          oracle_fwd_bwd(inp, gate=gate, l2norm=l2n)), label="after timeout")


def test_malformed_cu_seqlens_reports_device_status():
    inp, gate, l2n = _small("g_edges")
    d = to_dev(inp)
    bad = d["cu_seqlens"].clone()
    bad[2] = bad[1] - 5  # decreasing
    ws_b, _ = kda.kda_workspace_size(inp["q"].shape[0], bad.numel() - 1, 2, kda.KDA_OP_FWD)
    ws = torch.zeros(ws_b, dtype=torch.uint8, device="cuda")
    kda.kda_fwd(d["q"], d["k"], d["v"], d["beta"], d["g"], bad, save=False, ws=ws)
    assert kda.kda_read_device_status(ws) == kda.KDA_ERR_DEVICE_CHECK
    assert kda.kda_read_device_status(ws) == kda.KDA_OK  # read clears it
    kda.kda_fwd(d["q"], d["k"], d["v"], d["beta"], d["g"], d["cu_seqlens"], save=False, ws=ws)
    assert kda.kda_read_device_status(ws) == kda.KDA_OK


def test_positive_g_gate_reports_device_status():
    # g form needs a decaying gate (g <= 0): one positive value inside a document is reported as
    # KDA_ERR_DEVICE_CHECK, the recurrences write nothing (o keeps its NaN prefill), and the next
    # valid call on the same workspace reports OK and matches the oracle
    inp, gate, l2n = _small("g_edges")
    d = to_dev(inp)
    g_bad = d["g"].clone()
    g_bad[3, 1, 17] = 0.25
    ws_b, _ = kda.kda_workspace_size(inp["q"].shape[0], d["cu_seqlens"].numel() - 1, 2,
                                     kda.KDA_OP_FWD)
    ws = torch.zeros(ws_b, dtype=torch.uint8, device="cuda")
    o = torch.full(d["q"].shape, float("nan"), dtype=torch.float32, device="cuda")
    kda.kda_fwd(d["q"], d["k"], d["v"], d["beta"], g_bad, d["cu_seqlens"], save=False, ws=ws, o=o)
    assert kda.kda_read_device_status(ws) == kda.KDA_ERR_DEVICE_CHECK
    assert torch.isnan(o).all()
    o, ht, _ = kda.kda_fwd(d["q"], d["k"], d["v"], d["beta"], d["g"], d["cu_seqlens"], save=False,
                           ws=ws)
    assert kda.kda_read_device_status(ws) == kda.KDA_OK
    ref = oracle_fwd_bwd(inp, gate=gate, l2norm=l2n, want_bwd=False)
    assert rel_err(o.cpu().numpy(), ref["o"]) <= TOL["o"]


def test_host_validation_on_device():
    inp, gate, l2n = _small("g_edges")
    d = to_dev(inp)
    with pytest.raises(kda.KdaError) as e:
        kda.kda_fwd(d["q"], d["k"], d["v"], d["beta"], d["g"], d["cu_seqlens"], gate="raw")
    assert e.value.status == kda.KDA_ERR_INVALID_ARG


def test_bf16_outputs_within_rounding_of_fp32_outputs():
    # bf16 outputs are the fp32 outputs rounded to nearest: within half a bf16 ulp elementwise
    inp, gate, l2n = _small("raw_fast", seed=6)
    a = gpu_fwd_bwd(inp, gate=gate, l2norm=l2n, out_dtype=torch.float32)
    b = gpu_fwd_bwd(inp, gate=gate, l2norm=l2n, out_dtype=torch.bfloat16)
    for k in ("o", "dq", "dk", "dv", "dbeta"):
        want = torch.tensor(a[k]).bfloat16().float().numpy()
        assert np.array_equal(b[k], want), k
    for k in ("ht", "dg", "dA_log", "ddt_bias", "dh0"):
        assert np.array_equal(a[k], b[k]), k

"""GPU parity of chunk groups inside documents (kda_problem.group_chunks > 0).

With group_chunks = G the state recurrences no longer run over a document's chunks in one serial
chain: the document is cut into groups of G chunks, the groups' affine summaries (M, B; C in the
backward) run in parallel, the transfer walk composes them into each group's start state (end
gradient), and the groups are finished as documents.  The results must match the FP64 oracle of
the whole, unfragmented documents within the same bounds as the serial path, in saved and replay
mode, with nonzero h0 / dht; be bitwise reproducible; and keep every document bitwise equal to
the same document run alone with the same G.  The 1doc workload (one document of 16384 tokens,
64 heads, fused L2 norm) runs with groups of 64 chunks in the bench's launch configuration.
"""
import numpy as np
import pytest
import torch

from harness import assert_within, compare, gpu_fwd_bwd, oracle_fwd_bwd
from linear_attention_chunked_gb300 import inputs

pytestmark = pytest.mark.gpu

CASES = {
    # documents of 1 .. 6 chunks, an empty one and ragged tails: groups of 1, 2 and 3 chunks cut
    # them at every position; the last group of a document is shorter or equal
    "g1_raw": dict(lens=[300, 77, 1, 0, 129, 64, 65], H=2, gate="raw", l2norm=False, G=1),
    "g2_g": dict(lens=[300, 77, 1, 0, 129, 64, 65], H=2, gate="g", l2norm=False, G=2, gdiv=16.0),
    "g3_l2n_fast": dict(lens=[383, 200, 63], H=3, gate="raw", l2norm=True, G=3,
                        A_log_range=(np.log(8.0), np.log(32.0))),
}


def _case(name, seed=1):
    c = dict(CASES[name])
    lens, H, G = c.pop("lens"), c.pop("H"), c.pop("G")
    return inputs.make_inputs(lens, H, seed=seed, **c), c["gate"], c["l2norm"], G


@pytest.mark.parametrize("case", list(CASES))
@pytest.mark.parametrize("saved_mode", [True, False])
def test_groups_against_oracle(case, saved_mode):
    inp, gate, l2n, G = _case(case)
    N, H = inp["cu_seqlens"].numel() - 1, inp["q"].shape[1]
    rng = np.random.default_rng(5)
    h0 = rng.standard_normal((N, H, 128, 128)).astype(np.float32) * 0.1
    dht = rng.standard_normal((N, H, 128, 128)).astype(np.float32) * 0.1
    gpu = gpu_fwd_bwd(inp, gate=gate, l2norm=l2n, h0=h0, dht=dht, saved_mode=saved_mode,
                      group_chunks=G)
    ref = oracle_fwd_bwd(inp, gate=gate, l2norm=l2n, h0=h0, dht=dht)
    errs = compare(gpu, ref)
    print(case, saved_mode, {k: f"{v:.2e}" for k, v in errs.items()})
    assert_within(errs, label=f"groups {case}")


def test_groups_bitwise_deterministic_and_isolated():
    inp, gate, l2n, G = _case("g2_g", seed=3)
    a = gpu_fwd_bwd(inp, gate=gate, l2norm=l2n, group_chunks=G)
    b = gpu_fwd_bwd(inp, gate=gate, l2norm=l2n, group_chunks=G)
    for k in a:
        assert np.array_equal(a[k], b[k]), k
    cu = inp["cu_seqlens"].tolist()
    for n in range(len(cu) - 1):
        s, e = cu[n], cu[n + 1]
        if s == e:
            assert np.all(a["ht"][n] == 0)
            continue
        one = {k: (v[s:e] if k in ("q", "k", "v", "beta", "g", "dO") else v)
               for k, v in inp.items()}
        one["cu_seqlens"] = torch.tensor([0, e - s], dtype=torch.int32)
        alone = gpu_fwd_bwd(one, gate=gate, l2norm=l2n, group_chunks=G)
        for k in ("o", "dq", "dk", "dv", "dbeta", "dg"):
            assert np.array_equal(alone[k], a[k][s:e]), (n, k)
        for k in ("ht", "dh0"):
            assert np.array_equal(alone[k][0], a[k][n]), (n, k)


def test_groups_1doc_sampled_heads():
    w = inputs.WORKLOADS["1doc"]
    inp = inputs.workload_inputs("1doc")
    heads = [0, 37]
    gpu = gpu_fwd_bwd(inp, gate=w.gate, l2norm=w.l2norm, group_chunks=64)
    ref = oracle_fwd_bwd(inp, gate=w.gate, l2norm=w.l2norm, heads=heads)
    errs = compare(gpu, ref, heads=heads)
    print("1doc groups of 64 chunks", {k: f"{v:.2e}" for k, v in errs.items()})
    assert_within(errs, label="1doc groups")

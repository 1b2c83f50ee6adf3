"""Pins of the FP64 oracle to facts that do not come from the oracle itself.

Each test fixes one part of the oracle so that a plausible mistake (a dropped term, a wrong sign,
decay applied after the write instead of before it, a transposed state, a wrong gate index, a
missing chain-rule factor) fails at least one of them:

* hand-worked token steps (tests/golden/worked_examples_d2.json);
* closed forms: pure gated decay (beta = 0), plain read-out (beta = 0, g = 0), the gated
  linear-attention form of distinct one-hot keys, and exact read-back (beta = 1, q = k, |k| = 1);
* a packed sequence equals its documents run one by one;
* central finite differences of L = sum(o*dO) + sum(ht*dht) for every gradient;
* the fragment algebra: M equals the explicit product of the per-token transitions, the token
  run equals M S_in + B, composition is associative, C equals the token backward's dh0.
"""
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_examples_d2.json")


def _rand_inputs(rng, lens, H, d, *, raw=False, unit=True, gscale=0.1, fast=False):
    T = int(sum(lens))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    q = rng.standard_normal((T, H, d))
    k = rng.standard_normal((T, H, d))
    if unit:
        q /= np.linalg.norm(q, axis=-1, keepdims=True)
        k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((T, H, d))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal((T, H))))
    if raw:
        g = rng.standard_normal((T, H, d))
        A_log = rng.uniform(np.log(8), np.log(32), H) if fast else rng.uniform(0, np.log(16), H)
        dt_bias = rng.uniform(-1, 1, (H, d))
    else:
        g = -gscale * np.abs(rng.standard_normal((T, H, d)))
        A_log = dt_bias = None
    return dict(q=q, k=k, v=v, beta=beta, g_or_a=g, cu_seqlens=cu, A_log=A_log, dt_bias=dt_bias)


# ---------------------------------------------------------------------------------------------
# forward: worked examples and closed forms


def test_worked_examples_d2():
    cases = json.load(open(GOLDEN))["cases"]
    for c in cases:
        toks = c["tokens"]
        T = len(toks)
        q = np.array([t["q"] for t in toks], float)[:, None, :]
        k = np.array([t["k"] for t in toks], float)[:, None, :]
        v = np.array([t["v"] for t in toks], float)[:, None, :]
        g = np.array([t["g"] for t in toks], float)[:, None, :]
        beta = np.array([[t["beta"]] for t in toks], float)
        h0 = np.array(c["h0"], float)[None, None]
        o, ht = oracle.kda_fwd(q, k, v, beta, g, [0, T], h0=h0)
        np.testing.assert_allclose(o[:, 0, :], np.array(c["o"], float), rtol=0, atol=1e-12,
                                   err_msg=c["name"])
        np.testing.assert_allclose(ht[0, 0], np.array(c["ht"], float), rtol=0, atol=1e-12,
                                   err_msg=c["name"])


def test_zero_state_single_token_d128():
    # from S = 0 one token gives S = beta k v^T, so o = beta (q.k) v
    rng = np.random.default_rng(1)
    x = _rand_inputs(rng, [1], 3, 128)
    o, ht = oracle.kda_fwd(**x)
    qk = np.einsum("thc,thc->th", x["q"], x["k"])
    np.testing.assert_allclose(o, (x["beta"] * qk)[..., None] * x["v"], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(ht[0], x["beta"][0][:, None, None] * x["k"][0][:, :, None]
                               * x["v"][0][:, None, :], rtol=1e-13, atol=1e-15)


@pytest.mark.parametrize("zero_gate", [False, True])
def test_pure_decay_closed_form(zero_gate):
    # beta = 0: S_t = Diag(exp(gamma_t)) h0 with gamma the prefix sum of g from the document start
    rng = np.random.default_rng(2)
    lens, H, d = [7, 5], 2, 8
    x = _rand_inputs(rng, lens, H, d, gscale=0.3)
    x["beta"][:] = 0.0
    if zero_gate:
        x["g_or_a"][:] = 0.0
    h0 = rng.standard_normal((2, H, d, d))
    o, ht = oracle.kda_fwd(**x, h0=h0)
    cu = x["cu_seqlens"]
    for n in range(2):
        sl = slice(cu[n], cu[n + 1])
        gam = np.cumsum(x["g_or_a"][sl], axis=0)  # [L,H,d]
        want = np.einsum("hij,lhi->lhj", h0[n], np.exp(gam) * x["q"][sl])
        np.testing.assert_allclose(o[sl], want, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(ht[n], np.exp(gam[-1])[:, :, None] * h0[n], rtol=1e-12,
                                   atol=1e-14)
        if zero_gate:
            np.testing.assert_allclose(o[sl], np.einsum("hij,lhi->lhj", h0[n], x["q"][sl]),
                                       rtol=1e-12, atol=1e-13)


def test_one_hot_keys_gated_linear_attention():
    # distinct one-hot keys never interfere: o_t = sum_{s<=t} beta_s q_t[p_s] e^{gam_t[p_s]-gam_s[p_s]} v_s
    rng = np.random.default_rng(3)
    L, H, d = 20, 2, 32
    x = _rand_inputs(rng, [L], H, d, gscale=0.2)
    x["q"] = rng.standard_normal((L, H, d))
    perm = np.stack([rng.permutation(d)[:L] for _ in range(H)], axis=1)  # [L,H]
    k = np.zeros((L, H, d))
    for t in range(L):
        for h in range(H):
            k[t, h, perm[t, h]] = 1.0
    x["k"] = k
    o, _ = oracle.kda_fwd(**x)
    gam = np.cumsum(x["g_or_a"], axis=0)
    want = np.zeros((L, H, d))
    for h in range(H):
        for t in range(L):
            for s in range(t + 1):
                p = perm[s, h]
                w = x["beta"][s, h] * x["q"][t, h, p] * np.exp(gam[t, h, p] - gam[s, h, p])
                want[t, h] += w * x["v"][s, h]
    np.testing.assert_allclose(o, want, rtol=1e-12, atol=1e-13)
    # with g = 0 this is beta-weighted causal linear attention
    x["g_or_a"][:] = 0.0
    o0, _ = oracle.kda_fwd(**x)
    kq = np.einsum("thc,shc->hts", x["q"], x["k"])
    want0 = np.einsum("hts,sh,shj->thj", np.tril(kq), x["beta"], x["v"])
    np.testing.assert_allclose(o0, want0, rtol=1e-12, atol=1e-13)


def test_exact_read_back():
    # beta = 1, |k| = 1, q = k: the token reads back its own value whatever the history
    rng = np.random.default_rng(4)
    x = _rand_inputs(rng, [9, 6], 2, 16, gscale=0.5)
    x["beta"][:] = 1.0
    x["q"] = x["k"].copy()
    h0 = rng.standard_normal((2, 2, 16, 16))
    o, _ = oracle.kda_fwd(**x, h0=h0)
    np.testing.assert_allclose(o, x["v"], rtol=1e-11, atol=1e-12)


def test_pack_equals_documents():
    rng = np.random.default_rng(5)
    lens = [4, 0, 9, 3]
    x = _rand_inputs(rng, lens, 2, 8, raw=True)
    dO = rng.standard_normal(x["q"].shape)
    o, ht = oracle.kda_fwd(**x, raw=True, l2norm=True)
    gr = oracle.kda_bwd(**x, dO=dO, raw=True, l2norm=True)
    cu = x["cu_seqlens"]
    for n, L in enumerate(lens):
        sl = slice(cu[n], cu[n + 1])
        sub = {kk: (vv[sl] if kk in ("q", "k", "v", "beta", "g_or_a") else vv)
               for kk, vv in x.items()}
        sub["cu_seqlens"] = [0, L]
        o1, ht1 = oracle.kda_fwd(**sub, raw=True, l2norm=True)
        np.testing.assert_array_equal(o1, o[sl])
        np.testing.assert_array_equal(ht1[0], ht[n])
        if L:
            g1 = oracle.kda_bwd(**sub, dO=dO[sl], raw=True, l2norm=True)
            for name in ("dq", "dk", "dv", "dbeta", "dg"):
                np.testing.assert_array_equal(g1[name], gr[name][sl])
    # an empty document passes h0 through and has zero gradient into it beyond dht
    assert np.all(ht[1] == 0.0)


def test_l2norm_equals_prenormalised():
    rng = np.random.default_rng(6)
    x = _rand_inputs(rng, [11], 2, 16, unit=False)
    o1, ht1 = oracle.kda_fwd(**x, l2norm=True, eps=1e-6)
    y = dict(x)
    y["q"] = x["q"] / np.sqrt((x["q"] ** 2).sum(-1, keepdims=True) + 1e-6)
    y["k"] = x["k"] / np.sqrt((x["k"] ** 2).sum(-1, keepdims=True) + 1e-6)
    o2, ht2 = oracle.kda_fwd(**y)
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(ht1, ht2, rtol=1e-12, atol=1e-13)


def test_raw_gate_equals_g_form():
    # raw form = g form fed with g = -exp(A_log) * log(1 + exp(a + dt_bias))
    rng = np.random.default_rng(7)
    x = _rand_inputs(rng, [6, 5], 3, 8, raw=True)
    g = -np.exp(x["A_log"])[None, :, None] * np.log1p(np.exp(x["g_or_a"] + x["dt_bias"][None]))
    o1, ht1 = oracle.kda_fwd(**x, raw=True)
    y = dict(x, g_or_a=g, A_log=None, dt_bias=None)
    o2, ht2 = oracle.kda_fwd(**y)
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(ht1, ht2, rtol=1e-12, atol=1e-13)


# ---------------------------------------------------------------------------------------------
# backward: central finite differences


def _loss(x, dO, dht, **kw):
    o, ht = oracle.kda_fwd(**x, **kw)
    return float(np.sum(o * dO) + np.sum(ht * dht))


def _fd(x, dO, dht, name, eps=1e-6, **kw):
    base = x[name] if name in x else kw[name]
    grad = np.zeros_like(base)
    it = np.nditer(base, flags=["multi_index"])
    for _ in it:
        idx = it.multi_index
        orig = base[idx]
        base[idx] = orig + eps
        lp = _loss(x, dO, dht, **kw)
        base[idx] = orig - eps
        lm = _loss(x, dO, dht, **kw)
        base[idx] = orig
        grad[idx] = (lp - lm) / (2 * eps)
    return grad


FD_CASES = {
    "g": dict(raw=False, l2norm=False, d=4, fast=False),
    "g_d8": dict(raw=False, l2norm=False, d=8, fast=False),
    "raw": dict(raw=True, l2norm=False, d=4, fast=False),
    "l2n": dict(raw=False, l2norm=True, d=4, fast=False),
    "raw_l2n_fast": dict(raw=True, l2norm=True, d=4, fast=True),
}


@pytest.mark.parametrize("case", list(FD_CASES))
def test_gradients_finite_differences(case):
    cfg = FD_CASES[case]
    rng = np.random.default_rng(10 + list(FD_CASES).index(case))
    lens, H, d = [5, 7], 2, cfg["d"]
    x = _rand_inputs(rng, lens, H, d, raw=cfg["raw"], unit=not cfg["l2norm"], gscale=0.4,
                     fast=cfg["fast"])
    if cfg["fast"]:
        # fast decay, still resolvable by a finite difference: g of about -3 .. -6 per token
        x["g_or_a"] = 0.3 * x["g_or_a"] - 1.5
    kw = dict(raw=cfg["raw"], l2norm=cfg["l2norm"], scale=0.7)
    h0 = rng.standard_normal((2, H, d, d))
    dO = rng.standard_normal((sum(lens), H, d))
    dht = rng.standard_normal((2, H, d, d))
    kw["h0"] = h0
    if cfg["raw"]:
        kw["A_log"] = x.pop("A_log")
        kw["dt_bias"] = x.pop("dt_bias")
    else:
        x.pop("A_log"), x.pop("dt_bias")
    an = oracle.kda_bwd(**x, dO=dO, dht=dht, **kw)
    pairs = [("q", "dq"), ("k", "dk"), ("v", "dv"), ("beta", "dbeta"), ("g_or_a", "dg"),
             ("h0", "dh0")]
    if cfg["raw"]:
        pairs += [("A_log", "dA_log"), ("dt_bias", "ddt_bias")]
    for inp, gname in pairs:
        fd = _fd(x, dO, dht, inp, **kw)
        err = np.max(np.abs(fd - an[gname])) / max(np.max(np.abs(fd)), 1e-30)
        assert err < 1e-6, f"{case}: {gname} rel err {err:.3e}"


# ---------------------------------------------------------------------------------------------
# fragment algebra


def _transitions_product(x, h, t0, t1, raw=False, A_log=None, dt_bias=None):
    d = x["q"].shape[-1]
    P = np.eye(d)
    for t in range(t0, t1):
        k = x["k"][t, h]
        g = x["g_or_a"][t, h]
        if raw:
            g = -np.exp(A_log[h]) * np.log1p(np.exp(g + dt_bias[h]))
        step = (np.eye(d) - x["beta"][t, h] * np.outer(k, k)) @ np.diag(np.exp(g))
        P = step @ P
    return P


@pytest.mark.parametrize("raw", [False, True])
def test_fragment_M_is_transition_product(raw):
    rng = np.random.default_rng(20)
    lens, H, d = [6, 4, 5], 2, 8
    x = _rand_inputs(rng, lens, H, d, raw=raw, gscale=0.05)
    M, B = oracle.fragment_summary(**x, raw=raw)
    _, ht0 = oracle.kda_fwd(**x, raw=raw)
    cu = x["cu_seqlens"]
    for f in range(3):
        for h in range(H):
            P = _transitions_product(x, h, cu[f], cu[f + 1], raw, x["A_log"], x["dt_bias"])
            np.testing.assert_allclose(M[f, h], P, rtol=1e-12, atol=1e-14)
    np.testing.assert_array_equal(B, ht0)


def test_fragment_affine_map_and_walk():
    # slow decay and short fragments keep M far from 0 so the checks are not vacuous
    rng = np.random.default_rng(21)
    H, d = 2, 8
    frag = [5, 7, 4, 6, 3]           # doc 0 = fragments 0..2, doc 1 = fragments 3..4
    doc_frag = [0, 3, 5]
    x = _rand_inputs(rng, frag, H, d, gscale=1e-3)
    M, B = oracle.fragment_summary(**x)
    assert np.min(np.abs(np.linalg.det(M))) > 1e-6
    # S_out = M S_in + B against the token run from S_in
    S_in = rng.standard_normal((5, H, d, d))
    _, ht = oracle.kda_fwd(**x, h0=S_in)
    np.testing.assert_allclose(ht, np.einsum("fhij,fhjk->fhik", M, S_in) + B, rtol=1e-11,
                               atol=1e-12)
    # walk against the unfragmented documents
    h0 = rng.standard_normal((2, H, d, d))
    Sw, Sfin = oracle.transfer_walk(doc_frag, M, B, h0)
    cu_docs = [0, sum(frag[:3]), sum(frag)]
    y = dict(x, cu_seqlens=cu_docs)
    o_doc, ht_doc = oracle.kda_fwd(**y, h0=h0)
    np.testing.assert_allclose(Sfin, ht_doc, rtol=1e-11, atol=1e-12)
    o_frag, _ = oracle.kda_fwd(**x, h0=Sw)
    np.testing.assert_allclose(o_frag, o_doc, rtol=1e-11, atol=1e-12)
    # associativity: (M2 M1, M2 B1 + B2) in any grouping equals the sequential walk
    for h in range(H):
        Ms, Bs = M[:3, h], B[:3, h]
        left = (Ms[2] @ (Ms[1] @ Ms[0]), Ms[2] @ (Ms[1] @ Bs[0] + Bs[1]) + Bs[2])
        right = ((Ms[2] @ Ms[1]) @ Ms[0], (Ms[2] @ Ms[1]) @ Bs[0] + (Ms[2] @ Bs[1] + Bs[2]))
        np.testing.assert_allclose(left[0], right[0], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(left[1], right[1], rtol=1e-12, atol=1e-14)
        np.testing.assert_allclose(left[0] @ h0[0, h] + left[1], Sfin[0, h], rtol=1e-11,
                                   atol=1e-12)


def test_fragment_backward_walk():
    rng = np.random.default_rng(22)
    H, d = 2, 8
    frag = [5, 7, 4, 6, 3]
    doc_frag = [0, 3, 5]
    x = _rand_inputs(rng, frag, H, d, gscale=1e-3)
    dO = rng.standard_normal(x["q"].shape)
    M, B = oracle.fragment_summary(**x)
    C = oracle.fragment_summary(**x, mode=1, dO=dO)
    # C_f is the gradient at the fragment start with zero end gradient
    g0 = oracle.kda_bwd(**x, dO=dO)
    np.testing.assert_array_equal(C, g0["dh0"])
    # the reverse walk gives the documents' end gradients per fragment and dh0 per document
    h0 = rng.standard_normal((2, H, d, d))
    dht = rng.standard_normal((2, H, d, d))
    dS_end, dh0 = oracle.transfer_walk(doc_frag, M, C, dht, reverse=True)
    y = dict(x, cu_seqlens=[0, sum(frag[:3]), sum(frag)])
    gdoc = oracle.kda_bwd(**y, dO=dO, dht=dht, h0=h0)
    np.testing.assert_allclose(dh0, gdoc["dh0"], rtol=1e-10, atol=1e-11)
    # finishing: per-fragment backward with h0 = S_in and dht = dS_end equals the document's
    S_in, _ = oracle.transfer_walk(doc_frag, M, B, h0)
    gfr = oracle.kda_bwd(**x, dO=dO, dht=dS_end, h0=S_in)
    for name in ("dq", "dk", "dv", "dbeta", "dg"):
        np.testing.assert_allclose(gfr[name], gdoc[name], rtol=1e-10, atol=1e-11)

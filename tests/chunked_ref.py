"""FP64 numpy restatement of the chunk-parallel algebra (test-side debugging aid, not the oracle).

The CUDA library evaluates the KDA recurrence chunk by chunk (chunk C = 64 tokens, restarted at
every document start).  This module writes that decomposition out in float64 with explicit
per-channel exponent differences, so a test can check the algebra against the token-by-token
oracle (they agree to ~1e-12) and a failing GPU stage can be compared stage by stage.

Per chunk, with gam = in-chunk inclusive cumsum of g and gL = gam[-1] (per channel):
  E[r,s,c] = exp(gam[r,c] - gam[s,c])
  Akk[r,s] = sum_c k_rc k_sc E[r,s,c]   (s < r)      Aqk[r,s] = sum_c q_rc k_sc E[r,s,c]  (s <= r)
  Minv = (I + diag(beta) Akk)^-1        W = Minv diag(beta) (K*e^gam)   U = Minv diag(beta) V
  Delta = U - W S0     O = (Q*e^gam) S0 + Aqk Delta     S1 = e^gL * S0 + (K*e^(gL-gam))^T Delta
The backward is the adjoint of those lines; see chunk_bwd.
"""
import numpy as np

CHUNK = 64


def _gate(g_or_a, h, raw, A_log, dt_bias):
    if not raw:
        return g_or_a
    x = g_or_a + dt_bias[h]
    return -np.exp(A_log[h]) * (np.maximum(x, 0) + np.log1p(np.exp(-np.abs(x))))


def _norm(x, on, eps):
    if not on:
        return x, np.ones(x.shape[:-1] + (1,))
    n = np.sqrt((x * x).sum(-1, keepdims=True) + eps)
    return x / n, n


def chunk_fwd(Q, K, V, beta, g, S0):
    L = Q.shape[0]
    gam = np.cumsum(g, axis=0)
    gL = gam[-1]
    E = np.exp(gam[:, None, :] - gam[None, :, :])
    Akk = np.tril(np.einsum("rc,sc,rsc->rs", K, K, E), -1)
    Aqk = np.tril(np.einsum("rc,sc,rsc->rs", Q, K, E))
    Minv = np.linalg.inv(np.eye(L) + beta[:, None] * Akk)
    Kg, Qg, Kb = K * np.exp(gam), Q * np.exp(gam), K * np.exp(gL - gam)
    W = Minv @ (beta[:, None] * Kg)
    U = Minv @ (beta[:, None] * V)
    Delta = U - W @ S0
    O = Qg @ S0 + Aqk @ Delta
    S1 = np.exp(gL)[:, None] * S0 + Kb.T @ Delta
    return O, S1, dict(gam=gam, gL=gL, E=E, Akk=Akk, Aqk=Aqk, Minv=Minv, Kg=Kg, Qg=Qg, Kb=Kb,
                       W=W, U=U, Delta=Delta)


def chunk_bwd(Q, K, V, beta, g, S0, dO, dS1):
    """Adjoint of chunk_fwd.  Returns dQ, dK, dV, dbeta, dg, dS0."""
    _, _, c = chunk_fwd(Q, K, V, beta, g, S0)
    E, Aqk, Akk, Minv = c["E"], c["Aqk"], c["Akk"], c["Minv"]
    Kg, Qg, Kb, W, Delta, gam, gL = c["Kg"], c["Qg"], c["Kb"], c["W"], c["Delta"], c["gam"], c["gL"]
    dDelta = Aqk.T @ dO + Kb @ dS1
    dS0 = Qg.T @ dO + np.exp(gL)[:, None] * dS1 - W.T @ dDelta
    dR = Minv.T @ dDelta
    dV = beta[:, None] * dR
    P = dR @ S0.T
    dKg = -beta[:, None] * P
    dbeta = (dR * V).sum(1) - (Kg * P).sum(1)
    dQg = dO @ S0.T
    dKb = Delta @ dS1.T
    dAqk = np.tril(dO @ Delta.T)
    dM = -np.tril(dR @ Delta.T, -1)
    dAkk = beta[:, None] * dM
    dbeta += (Akk * dM).sum(1)
    dQ = dQg * np.exp(gam)
    dK = dKg * np.exp(gam) + dKb * np.exp(gL - gam)
    dgam = dQg * Qg + dKg * Kg - dKb * Kb
    dgL = (dKb * Kb).sum(0) + np.exp(gL) * (S0 * dS1).sum(1)
    # Aqk (s <= r): the r == s terms carry no gate dependence and cancel exactly in dgam
    dQ += np.einsum("rs,sc,rsc->rc", dAqk, K, E)
    dK += np.einsum("rs,rc,rsc->sc", dAqk, Q, E)
    off = np.tril(dAqk, -1)
    t = np.einsum("rs,rc,sc,rsc->rsc", off, Q, K, E)
    dgam += t.sum(1) - t.sum(0)
    # Akk (s < r)
    dK += np.einsum("rs,sc,rsc->rc", dAkk, K, E) + np.einsum("rs,rc,rsc->sc", dAkk, K, E)
    t = np.einsum("rs,rc,sc,rsc->rsc", dAkk, K, K, E)
    dgam += t.sum(1) - t.sum(0)
    dgam[-1] += dgL
    dg = np.cumsum(dgam[::-1], axis=0)[::-1]
    return dQ, dK, dV, dbeta, dg, dS0


def kda_chunked(q, k, v, beta, g_or_a, cu_seqlens, dO=None, *, raw=False, A_log=None,
                dt_bias=None, h0=None, dht=None, l2norm=False, eps=1e-6, chunk=CHUNK):
    """Forward (and backward when dO is given) by the chunked algebra, float64."""
    T, H, d = q.shape
    cu = np.asarray(cu_seqlens)
    N = cu.size - 1
    o = np.zeros((T, H, d))
    ht = np.zeros((N, H, d, d))
    grads = None
    if dO is not None:
        grads = {n: np.zeros((T, H, d)) for n in ("dq", "dk", "dv", "dg")}
        grads["dbeta"] = np.zeros((T, H))
        grads["dh0"] = np.zeros((N, H, d, d))
        if raw:
            grads["dA_log"] = np.zeros(H)
            grads["ddt_bias"] = np.zeros((H, d))
    for n in range(N):
        for h in range(H):
            b, e = int(cu[n]), int(cu[n + 1])
            qn, nq = _norm(q[b:e, h], l2norm, eps)
            kn, nk = _norm(k[b:e, h], l2norm, eps)
            gg = _gate(g_or_a[b:e, h], h, raw, A_log, dt_bias)
            S = np.zeros((d, d)) if h0 is None else h0[n, h].copy()
            states = []
            for c0 in range(0, e - b, chunk):
                c1 = min(c0 + chunk, e - b)
                states.append(S)
                O, S, _ = chunk_fwd(qn[c0:c1], kn[c0:c1], v[b + c0:b + c1, h], beta[b + c0:b + c1, h],
                                    gg[c0:c1], S)
                o[b + c0:b + c1, h] = O
            ht[n, h] = S
            if dO is None:
                continue
            dS = np.zeros((d, d)) if dht is None else dht[n, h].copy()
            ci = len(states)
            for c0 in reversed(range(0, e - b, chunk)):
                ci -= 1
                c1 = min(c0 + chunk, e - b)
                sl = slice(b + c0, b + c1)
                dQ, dK, dV, dB, dG, dS = chunk_bwd(qn[c0:c1], kn[c0:c1], v[sl, h], beta[sl, h],
                                                  gg[c0:c1], states[ci], dO[sl, h], dS)
                if l2norm:
                    dQ = (dQ - qn[c0:c1] * (qn[c0:c1] * dQ).sum(-1, keepdims=True)) / nq[c0:c1]
                    dK = (dK - kn[c0:c1] * (kn[c0:c1] * dK).sum(-1, keepdims=True)) / nk[c0:c1]
                grads["dq"][sl, h], grads["dk"][sl, h], grads["dv"][sl, h] = dQ, dK, dV
                grads["dbeta"][sl, h] = dB
                if raw:
                    x = g_or_a[sl, h] + dt_bias[h]
                    da = dG * (-np.exp(A_log[h])) / (1 + np.exp(-x))
                    grads["dA_log"][h] += (dG * gg[c0:c1]).sum()
                    grads["ddt_bias"][h] += da.sum(0)
                    dG = da
                grads["dg"][sl, h] = dG
            grads["dh0"][n, h] = dS
    return o, ht, grads

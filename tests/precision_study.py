"""Operand-precision study of the chunked algorithm's tensor-core products (CPU, numpy).

Each product class of the chunked forward and backward is evaluated with its operands rounded to
a tensor-core format, everything else in float64, and the outputs are scored against the FP64
token-by-token oracle with the parity metric (max|x - ref| / rms(ref)).  This measures the error
an operand format alone brings, the quantity that decides which formats each class may use.

Product classes (operands as the kernels form them):
  intra    Akk, Aqk across 16-row sub-chunks: (Q or K) e^(gam - gam_e) times K e^(gam_e - gam),
           split at the last row e of the source sub-chunk (diagonal 16 x 16 blocks exact)
  wu       W = Minv (beta K e^gam), U = (Minv diag(beta)) V
  chain    Delta = U - W S, S <- e^gL S + Kb^T Delta, O = Qg S + Aqk Delta
  bchain   dDelta = Aqk^T dO + Kb dS1, dS0 = e^gL dS1 + Qg^T dO - W^T dDelta
  bgemm    dR = Minv^T dDelta, P = dR S0^T, dQg = dO S0^T, dKb = Delta dS1^T, dAqk = dO Delta^T,
           dM = -dR Delta^T
Formats: split (x = hi + lo, two bf16 parts, the library's format), tf32 (11 significant bits),
bf16 (8 bits), f64 (no rounding).

Usage: python tests/precision_study.py [workload ...]   (prints one table row per class/format)
"""
from __future__ import annotations

import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(HERE))
sys.path.insert(0, HERE)

CH = 64
SUB = 16


def round_bits(x, bits):
    """Round to `bits` significant bits (round to nearest even on the scaled mantissa)."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    s = 2.0 ** bits
    return np.ldexp(np.round(m * s) / s, e)


def fmt_round(x, fmt):
    if fmt == "f64":
        return np.asarray(x, dtype=np.float64)
    if fmt == "bf16":
        return round_bits(x, 8)
    if fmt == "tf32":
        return round_bits(x, 11)
    if fmt == "split":
        hi = round_bits(x, 8)
        return hi + round_bits(x - hi, 8)
    raise ValueError(fmt)


class Rounder:
    def __init__(self, formats):
        self.formats = formats  # class -> format

    def __call__(self, cls, x):
        return fmt_round(x, self.formats.get(cls, "f64"))


def chunk_fwd(Q, K, V, beta, g, S0, R):
    L = Q.shape[0]
    gam = np.cumsum(g, axis=0)
    gL = gam[-1]
    # exp(gam_r - gam_s) for s <= r (<= 1 with a decaying gate); the upper triangle never enters
    lower = np.tril(np.ones((L, L), dtype=bool))[:, :, None]
    E = np.exp(np.where(lower, gam[:, None, :] - gam[None, :, :], -np.inf))
    Akk = np.einsum("rc,sc,rsc->rs", K, K, E)
    Aqk = np.einsum("rc,sc,rsc->rs", Q, K, E)
    # across sub-chunks: operands split at the last row of the source sub-chunk
    for i in range(0, L, SUB):
        for j in range(0, i, SUB):
            e = min(j + SUB, L) - 1
            ri, rj = slice(i, min(i + SUB, L)), slice(j, e + 1)
            A_q = R("intra", Q[ri] * np.exp(gam[ri] - gam[e]))
            A_k = R("intra", K[ri] * np.exp(gam[ri] - gam[e]))
            B_k = R("intra", K[rj] * np.exp(gam[e] - gam[rj]))
            Aqk[ri, rj] = A_q @ B_k.T
            Akk[ri, rj] = A_k @ B_k.T
    Akk = np.tril(Akk, -1)
    Aqk = np.tril(Aqk)
    Minv = np.linalg.inv(np.eye(L) + beta[:, None] * Akk)
    Kg, Qg, Kb = K * np.exp(gam), Q * np.exp(gam), K * np.exp(gL - gam)
    W = R("wu", Minv) @ R("wu", beta[:, None] * Kg)
    U = R("wu", Minv * beta[None, :]) @ V
    Delta = U - R("chain", W) @ R("chain", S0)
    O = R("chain", Qg) @ R("chain", S0) + R("chain", Aqk) @ R("chain", Delta)
    S1 = np.exp(gL)[:, None] * S0 + R("chain", Kb).T @ R("chain", Delta)
    return O, S1, dict(gam=gam, gL=gL, E=E, Akk=Akk, Aqk=Aqk, Minv=Minv, Kg=Kg, Qg=Qg, Kb=Kb,
                       W=W, U=U, Delta=Delta)


def chunk_bwd(Q, K, V, beta, g, S0, dO, dS1, R):
    _, _, c = chunk_fwd(Q, K, V, beta, g, S0, R)
    E, Aqk, Akk, Minv = c["E"], c["Aqk"], c["Akk"], c["Minv"]
    Kg, Qg, Kb, W, Delta, gam, gL = c["Kg"], c["Qg"], c["Kb"], c["W"], c["Delta"], c["gam"], c["gL"]
    dDelta = R("bchain", Aqk).T @ dO + R("bchain", Kb) @ R("bchain", dS1)
    dS0 = R("bchain", Qg).T @ dO + np.exp(gL)[:, None] * dS1 - R("bchain", W).T @ R("bchain", dDelta)
    dR = R("bgemm", Minv).T @ R("bgemm", dDelta)
    dV = beta[:, None] * dR
    P = R("bgemm", dR) @ R("bgemm", S0).T
    dKg = -beta[:, None] * P
    dbeta = (dR * V).sum(1) - (Kg * P).sum(1)
    dQg = dO @ R("bgemm", S0).T
    dKb = R("bgemm", Delta) @ R("bgemm", dS1).T
    dAqk = np.tril(dO @ R("bgemm", Delta).T)
    dM = -np.tril(R("bgemm", dR) @ R("bgemm", Delta).T, -1)
    dAkk = beta[:, None] * dM
    dbeta += (Akk * dM).sum(1)
    dQ = dQg * np.exp(gam)
    dK = dKg * np.exp(gam) + dKb * np.exp(gL - gam)
    dgam = dQg * Qg + dKg * Kg - dKb * Kb
    dgL = (dKb * Kb).sum(0) + np.exp(gL) * (S0 * dS1).sum(1)
    dQ += np.einsum("rs,sc,rsc->rc", dAqk, K, E)
    dK += np.einsum("rs,rc,rsc->sc", dAqk, Q, E)
    off = np.tril(dAqk, -1)
    t = np.einsum("rs,rc,sc,rsc->rsc", off, Q, K, E)
    dgam += t.sum(1) - t.sum(0)
    dK += np.einsum("rs,sc,rsc->rc", dAkk, K, E) + np.einsum("rs,rc,rsc->sc", dAkk, K, E)
    t = np.einsum("rs,rc,sc,rsc->rsc", dAkk, K, K, E)
    dgam += t.sum(1) - t.sum(0)
    dgam[-1] += dgL
    dg = np.cumsum(dgam[::-1], axis=0)[::-1]
    return dQ, dK, dV, dbeta, dg, dS0


def run(inp, gate, l2norm, heads, R):
    """Chunked fwd + bwd (float64 apart from the rounded operands) on the given heads."""
    q, k, v = (inp[n].double().numpy()[:, heads] for n in ("q", "k", "v"))
    beta = inp["beta"].double().numpy()[:, heads]
    ga = inp["g"].double().numpy()[:, heads]
    dO = inp["dO"].double().numpy()[:, heads]
    cu = inp["cu_seqlens"].numpy()
    raw = gate == "raw"
    A_log = inp["A_log"].double().numpy()[heads] if raw else None
    dt_bias = inp["dt_bias"].double().numpy()[heads] if raw else None
    T, H, d = q.shape
    out = {n: np.zeros((T, H, d)) for n in ("o", "dq", "dk", "dv", "dg")}
    out["dbeta"] = np.zeros((T, H))
    out["ht"] = np.zeros((len(cu) - 1, H, d, d))
    if raw:
        out["dA_log"], out["ddt_bias"] = np.zeros(H), np.zeros((H, d))
    for n in range(len(cu) - 1):
        b, e = int(cu[n]), int(cu[n + 1])
        for h in range(H):
            qh, kh = q[b:e, h], k[b:e, h]
            if l2norm:
                nq = np.sqrt((qh * qh).sum(-1, keepdims=True) + 1e-6)
                nk = np.sqrt((kh * kh).sum(-1, keepdims=True) + 1e-6)
                qh, kh = qh / nq, kh / nk
            if raw:
                x = ga[b:e, h] + dt_bias[h]
                gg = -np.exp(A_log[h]) * (np.maximum(x, 0) + np.log1p(np.exp(-np.abs(x))))
            else:
                gg = ga[b:e, h]
            S = np.zeros((d, d))
            states = []
            for c0 in range(0, e - b, CH):
                c1 = min(c0 + CH, e - b)
                states.append(S)
                O, S, _ = chunk_fwd(qh[c0:c1], kh[c0:c1], v[b + c0:b + c1, h], beta[b + c0:b + c1, h],
                                    gg[c0:c1], S, R)
                out["o"][b + c0:b + c1, h] = O
            out["ht"][n, h] = S
            dS = np.zeros((d, d))
            ci = len(states)
            for c0 in reversed(range(0, e - b, CH)):
                ci -= 1
                c1 = min(c0 + CH, e - b)
                sl = slice(b + c0, b + c1)
                dQ, dK, dV, dB, dG, dS = chunk_bwd(qh[c0:c1], kh[c0:c1], v[sl, h], beta[sl, h],
                                                  gg[c0:c1], states[ci], dO[sl, h], dS, R)
                if l2norm:
                    dQ = (dQ - qh[c0:c1] * (qh[c0:c1] * dQ).sum(-1, keepdims=True)) / nq[c0:c1]
                    dK = (dK - kh[c0:c1] * (kh[c0:c1] * dK).sum(-1, keepdims=True)) / nk[c0:c1]
                out["dq"][sl, h], out["dk"][sl, h], out["dv"][sl, h] = dQ, dK, dV
                out["dbeta"][sl, h] = dB
                if raw:
                    x = ga[sl, h] + dt_bias[h]
                    da = dG * (-np.exp(A_log[h])) / (1 + np.exp(-x))
                    out["dA_log"][h] += (dG * gg[c0:c1]).sum()
                    out["ddt_bias"][h] += da.sum(0)
                    dG = da
                out["dg"][sl, h] = dG
    return out


def main(argv):
    import oracle
    from harness import TOL, oracle_fwd_bwd, rel_err
    from linear_attention_chunked_gb300 import inputs

    names = argv or ["R2fast", "R2", "m2"]
    classes = ["intra", "wu", "chain", "bchain", "bgemm"]
    oracle.build()
    print("| workload | class | format | worst output (err / bound) | errors |")
    print("|---|---|---|---|---|")
    for name in names:
        w = inputs.WORKLOADS[name]
        inp = inputs.workload_inputs(name)
        heads = list(range(min(w.H, 2)))
        ref = oracle_fwd_bwd(inp, gate=w.gate, l2norm=w.l2norm, heads=heads)
        for cls in classes:
            for fmt in ("split", "tf32", "bf16"):
                got = run(inp, w.gate, w.l2norm, heads, Rounder({cls: fmt}))
                errs = {k: rel_err(got[k], ref[k]) for k in got if k in ref}
                worst = max(errs, key=lambda k: errs[k] / TOL[k])
                print(f"| {name} | {cls} | {fmt} | {worst} {errs[worst]:.2e} / {TOL[worst]:.0e} "
                      f"({errs[worst] / TOL[worst]:.2f}) | "
                      + ", ".join(f"{k} {v:.1e}" for k, v in sorted(errs.items())) + " |",
                      flush=True)


if __name__ == "__main__":
    main(sys.argv[1:])

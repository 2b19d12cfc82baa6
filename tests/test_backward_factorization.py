"""The chunk-form chain rule that the backward kernels compute, written out in fp64 numpy and
checked against the backward oracle (`oracle/bptt.py`, itself pinned by finite differences).

Forward per chunk (state S is d_k x d_v, G_i the cumulative log-decay through token i):
  K~ = k^ e^G, Q~ = q^ e^G, K_end = k^ e^(G_last - G), gam = e^G_last,
  L_im = sum_c k^_ic k^_mc e^(G_ic - G_mc) (m < i),  M_im = sum_c q^_ic k^_mc e^(G_ic - G_mc) (m <= i),
  T = (I + diag(beta) L)^-1,  Y = diag(beta)(V - K~ S),  E = T Y,
  O = Q~ S + M E,  S' = diag(gam) S + K_end^T E.
Backward per chunk, last chunk first:
  dE = M^T dO + K_end dS',  dY = T^T dE,  dS = Q~^T dO + diag(gam) dS' - K~^T diag(beta) dY,
  dV = diag(beta) dY,  dA = -dY E^T,  dL = diag(beta) dA,  dM = dO E^T,  dQ~ = dO S^T,
  dK~ = -diag(beta) dY S^T,  dK_end = E dS'^T,  dgam = rowsum(dS' * S),
  dbeta_i = dY_i . (V - K~ S)_i + sum_m dA_im L_im,
then the pairwise and decayed products pass their gradients to q^, k^ and G, G's reverse
cumulative sum within the chunk gives dg, and the L2 normalisation's backward gives dq, dk.
The additive write has L = 0 and no K~ S term, so dA and dK~ carry nothing back.
"""
import numpy as np
import pytest

from oracle import bptt


def chunk_backward(q, k, v, beta, g, S0, do, dS_final, *, chunk, delta_rule=True):
    T, dk = q.shape
    per_channel = g.ndim == 2
    scale = 1.0 / np.sqrt(dk)
    rk = 1.0 / np.sqrt(np.sum(k * k, axis=1) + 1e-6)
    rq = 1.0 / np.sqrt(np.sum(q * q, axis=1) + 1e-6)
    kn, qn = k * rk[:, None], q * (scale * rq)[:, None]
    gg = g if per_channel else np.repeat(g[:, None], dk, axis=1)
    starts = list(range(0, T, chunk))
    # forward, keeping each chunk's incoming state
    S = S0.copy()
    states = []
    for c0 in starts:
        sl = slice(c0, min(c0 + chunk, T))
        states.append(S.copy())
        f = chunk_forward(qn[sl], kn[sl], v[sl], beta[sl], gg[sl], S, delta_rule)
        S = f["S1"]
    dqn, dkn = np.zeros_like(qn), np.zeros_like(kn)
    dv, dbeta, dgg = np.zeros_like(v), np.zeros_like(beta), np.zeros_like(gg)
    dS1 = np.zeros_like(S0) if dS_final is None else dS_final.copy()
    for c0, S in reversed(list(zip(starts, states))):
        sl = slice(c0, min(c0 + chunk, T))
        f = chunk_forward(qn[sl], kn[sl], v[sl], beta[sl], gg[sl], S, delta_rule)
        b, dO = beta[sl], do[sl]
        dE = f["M"].T @ dO + f["Kend"] @ dS1
        dY = f["T"].T @ dE
        dS = f["Qt"].T @ dO + f["gam"][:, None] * dS1 - f["Kt"].T @ (b[:, None] * dY)
        dv[sl] = b[:, None] * dY
        # the additive write's K~ and L are the constant 0: nothing flows back through them
        dA = np.tril(-dY @ f["E"].T, -1) if delta_rule else np.zeros_like(f["L"])
        dL = b[:, None] * dA
        dM = np.tril(dO @ f["E"].T)
        dQt = dO @ S.T
        dKt = -(b[:, None] * dY) @ S.T if delta_rule else np.zeros_like(f["Kt"])
        dKend = f["E"] @ dS1.T
        dgam = np.sum(dS1 * S, axis=1)
        dbeta[sl] = np.sum(dY * f["R"], axis=1) + np.sum(dA * f["L"], axis=1)
        G, eG, kc, qc = f["G"], f["eG"], kn[sl], qn[sl]
        dG = dQt * f["Qt"] + dKt * f["Kt"] - dKend * f["Kend"]
        dGlast = np.sum(dKend * f["Kend"], axis=0) + dgam * f["gam"]
        dqc = dQt * eG
        dkc = dKt * eG + dKend * np.exp(G[-1] - G)
        dec = f["dec"]                                   # [i, m, c] = e^(G_ic - G_mc)
        PL = kc[:, None, :] * kc[None, :, :] * dec       # pair products of L
        PM = qc[:, None, :] * kc[None, :, :] * dec       # pair products of M
        dkc += np.einsum("im,mc,imc->ic", dL, kc, dec) + np.einsum("im,ic,imc->mc", dL, kc, dec)
        dqc += np.einsum("im,mc,imc->ic", dM, kc, dec)
        dkc += np.einsum("im,ic,imc->mc", dM, qc, dec)
        dG += np.einsum("im,imc->ic", dL, PL) - np.einsum("im,imc->mc", dL, PL)
        dG += np.einsum("im,imc->ic", dM, PM) - np.einsum("im,imc->mc", dM, PM)
        dG[-1] += dGlast
        dgg[sl] = np.cumsum(dG[::-1], axis=0)[::-1]      # G_i = sum_{t <= i} g_t
        dqn[sl], dkn[sl] = dqc, dkc
        dS1 = dS
    # L2 normalisation (and the query scale): x^ = x r, r = (|x|^2 + eps)^-1/2
    dk_ = rk[:, None] * dkn - (rk ** 3 * np.sum(k * dkn, axis=1))[:, None] * k
    dq_ = scale * (rq[:, None] * dqn - (rq ** 3 * np.sum(q * dqn, axis=1))[:, None] * q)
    dg = dgg if per_channel else dgg.sum(axis=1)
    return dict(dq=dq_, dk=dk_, dv=dv, dbeta=dbeta, dg=dg, dS0=dS1)


def chunk_forward(qc, kc, vc, b, gc, S, delta_rule):
    n = kc.shape[0]
    G = np.cumsum(gc, axis=0)
    eG = np.exp(G)
    dec = np.exp(G[:, None, :] - G[None, :, :])
    L = np.tril(np.einsum("ic,mc,imc->im", kc, kc, dec), -1) if delta_rule else np.zeros((n, n))
    M = np.tril(np.einsum("ic,mc,imc->im", qc, kc, dec))
    Tm = np.linalg.inv(np.eye(n) + b[:, None] * L)
    Kt = kc * eG if delta_rule else np.zeros_like(kc)
    R = vc - Kt @ S
    E = Tm @ (b[:, None] * R)
    Qt, Kend, gam = qc * eG, kc * np.exp(G[-1] - G), np.exp(G[-1])
    S1 = gam[:, None] * S + Kend.T @ E
    return dict(G=G, eG=eG, dec=dec, L=L, M=M, T=Tm, Kt=Kt, R=R, E=E, Qt=Qt, Kend=Kend, gam=gam,
                S1=S1)


def inputs(seed, T, dk, dv, per_channel):
    r = np.random.Generator(np.random.PCG64(seed))
    return dict(q=r.standard_normal((T, dk)), k=r.standard_normal((T, dk)),
                v=r.standard_normal((T, dv)), beta=r.uniform(0.1, 1.0, T),
                g=-r.uniform(0.0, 0.2, (T, dk) if per_channel else T),
                S0=r.standard_normal((dk, dv)) * 0.3, do=r.standard_normal((T, dv)),
                dS_final=r.standard_normal((dk, dv)))


@pytest.mark.parametrize("per_channel", [False, True])
@pytest.mark.parametrize("delta_rule", [True, False])
@pytest.mark.parametrize("T,chunk", [(150, 64), (40, 16), (7, 16)])
def test_chunk_chain_rule_equals_the_backward_oracle(per_channel, delta_rule, T, chunk):
    x = inputs(T + chunk + 2 * per_channel + delta_rule, T, 16, 8, per_channel)
    got = chunk_backward(x["q"], x["k"], x["v"], x["beta"], x["g"], x["S0"], x["do"],
                         x["dS_final"], chunk=chunk, delta_rule=delta_rule)
    ref = bptt.backward_seq(x["q"], x["k"], x["v"], x["beta"], x["g"], x["S0"], x["do"],
                            x["dS_final"], delta_rule=delta_rule)
    for name in ("dq", "dk", "dv", "dbeta", "dg", "dS0"):
        a, b = got[name], ref[name]
        assert a.shape == b.shape, name
        np.testing.assert_allclose(a, b, rtol=0, atol=1e-9 * max(1.0, np.abs(b).max()),
                                   err_msg=name)

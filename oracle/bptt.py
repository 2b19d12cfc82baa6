"""fp64 reverse-mode differentiation of the gated delta rule's token recurrence.

TEST INFRASTRUCTURE ONLY, like the rest of `oracle/`: it shares no code with the CUDA library.

The forward pass differentiated here is the five steps of the recurrence, one token at a
time ("You Could Have Come Up With Kimi Delta Attention", sec. 4: forget, predict, correct,
write, read; sec. 2.2 reads the write as one gradient step on 1/2 |S k - v|^2), with the
L2 normalisation of q and k and the query scale in front of them ("From Attention to Learned
Memory", sec. 1: features after normalisation; the KDA page's q^ = s q / |q|).  In the stored
orientation (state S is d_k x d_v, row = key channel) token t does

    S~ = Diag(a) S_prev,  a = exp(g_t)          v^ = S~^T k^            e = beta (v - v^)
    S  = S~ + k^ e^T                            o  = S^T q^

and the backward pass walks the tokens in reverse, applying the chain rule to each of these
assignments in turn, with every forward state kept (no recomputation, no blocking).  The
pages give the linear-attention backward in full and the delta rule's only by reference
("From Attention to Learned Memory", sec. 3); this is the plain chain rule of the recurrence
they define, pinned by central finite differences of the forward recurrence.

With delta_rule = False the prediction is left out (e = beta v), the additive write.
"""
from __future__ import annotations

from typing import Optional

import numpy as np

L2_EPS = 1e-6


def backward_seq(q, k, v, beta, g, S0, do, dS_final=None, *, scale=None, l2norm=True,
                 delta_rule=True, mutant: int = 0):
    """One sequence through one value head.

    q, k: [T, dk] (the key head's rows); v: [T, dv]; beta: [T]; g: [T] (scalar gate) or
    [T, dk]; S0: [dk, dv]; do: [T, dv] (gradient of the loss w.r.t. o); dS_final: [dk, dv]
    or None (gradient w.r.t. the final state).  Returns a dict of fp64 arrays dq, dk, dv,
    dbeta, dg (shape of g), dS0.

    `mutant` plants a mistake for the pin tests: 1 drops the prediction's path into dk,
    2 takes the forget gate's gradient against the written state instead of the previous
    one, 3 leaves out the normalisation's projection term.
    """
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    beta = np.asarray(beta, np.float64)
    g = np.asarray(g, np.float64)
    do = np.asarray(do, np.float64)
    T, dk = q.shape
    dv = v.shape[1]
    if scale is None or scale <= 0:
        scale = 1.0 / np.sqrt(dk)
    per_channel = g.ndim == 2
    rk = 1.0 / np.sqrt(np.sum(k * k, axis=1) + L2_EPS) if l2norm else np.ones(T)
    rq = 1.0 / np.sqrt(np.sum(q * q, axis=1) + L2_EPS) if l2norm else np.ones(T)
    kn = k * rk[:, None]
    qn = q * (rq * scale)[:, None]

    # forward, keeping the state before every token
    S_prev = np.empty((T, dk, dv))
    S = np.array(S0, np.float64, copy=True)
    for t in range(T):
        S_prev[t] = S
        a = np.exp(g[t]) if per_channel else np.full(dk, np.exp(g[t]))
        St = a[:, None] * S
        vhat = kn[t] @ St
        e = beta[t] * (v[t] - vhat) if delta_rule else beta[t] * v[t]
        S = St + np.outer(kn[t], e)

    dS = np.zeros((dk, dv)) if dS_final is None else np.array(dS_final, np.float64, copy=True)
    dq = np.zeros((T, dk))
    dkk = np.zeros((T, dk))
    dvv = np.zeros((T, dv))
    dbeta = np.zeros(T)
    dg = np.zeros_like(g)
    for t in range(T - 1, -1, -1):
        a = np.exp(g[t]) if per_channel else np.full(dk, np.exp(g[t]))
        St = a[:, None] * S_prev[t]
        vhat = kn[t] @ St
        e = beta[t] * (v[t] - vhat) if delta_rule else beta[t] * v[t]
        S_t = St + np.outer(kn[t], e)
        # read: o = S^T q^
        dS += np.outer(qn[t], do[t])
        dqn = S_t @ do[t]
        # write: S = S~ + k^ e^T
        dSt = dS.copy()
        dkn = dS @ e
        de = kn[t] @ dS
        # correct: e = beta (v - v^)
        dvv[t] = beta[t] * de
        if delta_rule:
            dbeta[t] = de @ (v[t] - vhat)
            dvhat = -beta[t] * de
            # predict: v^ = S~^T k^
            if mutant != 1:
                dkn += St @ dvhat
            dSt += np.outer(kn[t], dvhat)
        else:
            dbeta[t] = de @ v[t]
        # forget: S~ = Diag(a) S_prev, a = exp(g)
        da = np.sum(dSt * (S_t if mutant == 2 else S_prev[t]), axis=1)
        dS = a[:, None] * dSt
        dga = da * a
        dg[t] = dga if per_channel else np.sum(dga)
        # normalisation: k^ = k r, r = (|k|^2 + eps)^(-1/2); q^ = s q r_q
        if l2norm and mutant != 3:
            dkk[t] = rk[t] * dkn - k[t] * rk[t] ** 3 * (k[t] @ dkn)
            dq[t] = scale * (rq[t] * dqn - q[t] * rq[t] ** 3 * (q[t] @ dqn))
        else:
            dkk[t] = rk[t] * dkn
            dq[t] = scale * rq[t] * dqn
    return dict(dq=dq, dk=dkk, dv=dvv, dbeta=dbeta, dg=dg, dS0=dS)


def backward_arrays(*, offsets, slot_idx, q, k, v, beta, g, pool, d_o, d_state=None,
                    scale: float = 0.0, l2norm: bool = True, delta_rule: bool = True,
                    pairs=None):
    """The ragged batch with GQA (key head = value head // ratio) and a slot pool, as the
    forward library call: q, k [T, HK, dk]; v [T, HV, dv]; beta [T, HV]; g [T, HV] or
    [T, HV, dk]; pool [num_slots, HV, dk, dv] (the initial states); d_o [T, HV, dv];
    d_state [num_slots, HV, dk, dv] or None (gradient w.r.t. the final states).

    Returns dq, dk [T, HK, dk] (summed over the value heads of each key head), dv [T, HV, dv],
    dbeta [T, HV], dg (shape of g) and d_state0 [num_slots, HV, dk, dv] (the touched slots;
    the others zero).  `pairs`, a list of (sequence, value head), limits the work to those
    pairs (the other entries stay zero).
    """
    offsets = np.asarray(offsets, np.int64)
    slot_idx = np.asarray(slot_idx, np.int64)
    T, HK, dk = q.shape
    HV, dv = v.shape[1], v.shape[2]
    ratio = HV // HK
    out = dict(dq=np.zeros((T, HK, dk)), dk=np.zeros((T, HK, dk)), dv=np.zeros((T, HV, dv)),
               dbeta=np.zeros((T, HV)), dg=np.zeros(g.shape), d_state0=np.zeros(pool.shape))
    B = offsets.shape[0] - 1
    todo = pairs if pairs is not None else [(b, h) for b in range(B) for h in range(HV)]
    for b, h in todo:
        s, e_ = int(offsets[b]), int(offsets[b + 1])
        kh = h // ratio
        slot = int(slot_idx[b])
        dSf = None if d_state is None else d_state[slot, h]
        r = backward_seq(q[s:e_, kh], k[s:e_, kh], v[s:e_, h], beta[s:e_, h], g[s:e_, h],
                         pool[slot, h], d_o[s:e_, h], dSf, scale=scale, l2norm=l2norm,
                         delta_rule=delta_rule)
        out["dq"][s:e_, kh] += r["dq"]
        out["dk"][s:e_, kh] += r["dk"]
        out["dv"][s:e_, h] = r["dv"]
        out["dbeta"][s:e_, h] = r["dbeta"]
        out["dg"][s:e_, h] = r["dg"]
        out["d_state0"][slot, h] = r["dS0"]
    return out

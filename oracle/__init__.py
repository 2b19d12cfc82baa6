"""fp64 CPU oracle for the gated delta rule forward pass.

TEST INFRASTRUCTURE ONLY.  Only `tests/`, `__graft_entry__.smoke()` and the CPU
baseline leg of `bench.py` may import this package.  It shares no code with the
CUDA library and never imports it; the two meet only at the seeded inputs of
the `workloads` module.

Contents
  run(problem, ...)            the token-by-token recurrence in C (kda_oracle.c), fp64
  run_decode(problem, ...)     the same recurrence applied one decode step at a time
  recurrence_py(...)           a pure-numpy transcription of the same five steps, for tiny cases
  chunk_form(...)              the chunkwise closed form of "You Could Have Come Up With Kimi
                               Delta Attention", sec. 6, evaluated densely in fp64 (numpy)
  causal_linear_attention(...) brute force (Q K^T masked) V + Q S0 ("From Attention to Learned
                               Memory", sec. 1-2), the delta-free, decay-free special case
  backward(problem, ...)       reverse-mode differentiation of the recurrence in fp64
                               (`oracle/bptt.py`), pinned by finite differences
  conv.conv_gates(...)         the front end before the recurrence: causal short convolution
                               with a conv-state pool, SiLU, and the gate activations
                               (`oracle/conv.py`)

Parity status: every function here is pinned by `tests/test_oracle_pins.py`
against closed forms, invariants the pages state, brute force and the worked
example of "Linear attention visualized" (DeltaNet section, Alice/Bob memory).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_LIB_CACHE = {}

L2_EPS = 1e-6


def lib_path(mutant: int = 0) -> str:
    suffix = "" if mutant == 0 else f"_mutant{mutant}"
    return os.path.join(_HERE, "_build", f"libkda_oracle{suffix}.so")


def build(mutant: int = 0, force: bool = False) -> str:
    """Compile the C oracle with the host compiler (no fast-math)."""
    out = lib_path(mutant)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-fno-fast-math",
           "-ffp-contract=off", f"-DORACLE_MUTANT={mutant}", _SRC, "-o", tmp, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _load(mutant: int = 0):
    if mutant in _LIB_CACHE:
        return _LIB_CACHE[mutant]
    path = build(mutant)
    lib = ctypes.CDLL(path)
    f = lib.kda_oracle_run
    P = ctypes.c_void_p
    f.argtypes = [ctypes.c_int, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                  P, P, P, P, P, ctypes.c_int, ctypes.c_double, ctypes.c_int, ctypes.c_int,
                  P, P, P, ctypes.c_int]
    f.restype = ctypes.c_int
    f = lib.kda_oracle_gdp_run
    f.argtypes = [ctypes.c_int, P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                  ctypes.c_int, P, P, P, P, P, ctypes.c_int, ctypes.c_double, ctypes.c_int,
                  P, P, ctypes.c_int]
    f.restype = ctypes.c_int
    _LIB_CACHE[mutant] = lib
    return lib


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def run_arrays(*, offsets, slot_idx, q, k, v, beta, g, per_channel: bool, pool, scale: float = 0.0,
               l2norm: bool = True, delta_rule: bool = True, pair_mask=None,
               nthreads: Optional[int] = None, mutant: int = 0):
    """Run the C recurrence on plain arrays.

    q, k: [T, HK, dk]; v: [T, HV, dv]; beta: [T, HV]; g: [T, HV] or [T, HV, dk];
    pool: [num_slots, HV, dk, dv].  All floating inputs are converted to fp32 (they
    must already hold exactly representable values: bf16 inputs are widened first).
    Returns (o fp64 [T, HV, dv], pool fp64 after the call).
    """
    offsets = np.ascontiguousarray(offsets, dtype=np.int64)
    slot_idx = np.ascontiguousarray(slot_idx, dtype=np.int64)
    q = np.ascontiguousarray(q, dtype=np.float32)
    k = np.ascontiguousarray(k, dtype=np.float32)
    v = np.ascontiguousarray(v, dtype=np.float32)
    beta = np.ascontiguousarray(beta, dtype=np.float32)
    g = np.ascontiguousarray(g, dtype=np.float32)
    pool = np.array(pool, dtype=np.float64, copy=True, order="C")
    T, HK, dk = q.shape
    HV, dv = v.shape[1], v.shape[2]
    num_seqs = offsets.shape[0] - 1
    o = np.zeros((T, HV, dv), dtype=np.float64)
    if pair_mask is not None:
        pair_mask = np.ascontiguousarray(pair_mask, dtype=np.uint8).reshape(num_seqs * HV)
    if scale is None or scale <= 0:
        scale = 1.0 / np.sqrt(dk)
    lib = _load(mutant)
    rc = lib.kda_oracle_run(num_seqs, _ptr(offsets), _ptr(slot_idx), HK, HV, dk, dv, _ptr(q),
                            _ptr(k), _ptr(v), _ptr(beta), _ptr(g), int(bool(per_channel)),
                            float(scale), int(bool(l2norm)), int(bool(delta_rule)), _ptr(pool),
                            _ptr(o), _ptr(pair_mask), int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return o, pool


def run_gdp_arrays(*, offsets, slot_idx, q, k, v, beta, g, per_channel: bool, pool,
                   scale: float = 0.0, l2norm: bool = True, nthreads: Optional[int] = None,
                   mutant: int = 0):
    """Gated DeltaProduct ("Linear attention visualized", Gated Delta Product section): the C
    recurrence with n_h substeps per token.

    q: [T, HK, dk] (one query per token); k: [T, n_h, HK, dk]; v: [T, n_h, HV, dv];
    beta: [T, n_h, HV]; g: [T, HV] or [T, HV, dk] (one decay per token, applied before the
    first substep); pool: [num_slots, HV, dk, dv].  Returns (o fp64 [T, HV, dv], pool fp64).
    """
    offsets = np.ascontiguousarray(offsets, dtype=np.int64)
    slot_idx = np.ascontiguousarray(slot_idx, dtype=np.int64)
    q = np.ascontiguousarray(q, dtype=np.float32)
    k = np.ascontiguousarray(k, dtype=np.float32)
    v = np.ascontiguousarray(v, dtype=np.float32)
    beta = np.ascontiguousarray(beta, dtype=np.float32)
    g = np.ascontiguousarray(g, dtype=np.float32)
    pool = np.array(pool, dtype=np.float64, copy=True, order="C")
    T, HK, dk = q.shape
    n_h = k.shape[1]
    HV, dv = v.shape[2], v.shape[3]
    if k.shape != (T, n_h, HK, dk) or v.shape[:2] != (T, n_h) or beta.shape != (T, n_h, HV):
        raise ValueError("substep axes of k, v, beta disagree")
    num_seqs = offsets.shape[0] - 1
    o = np.zeros((T, HV, dv), dtype=np.float64)
    if scale is None or scale <= 0:
        scale = 1.0 / np.sqrt(dk)
    lib = _load(mutant)
    rc = lib.kda_oracle_gdp_run(num_seqs, _ptr(offsets), _ptr(slot_idx), HK, HV, dk, dv, n_h,
                                _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(g),
                                int(bool(per_channel)), float(scale), int(bool(l2norm)),
                                _ptr(pool), _ptr(o), int(nthreads or default_threads()))
    if rc != 0:
        raise ValueError("oracle rejected its arguments")
    return o, pool


def _widen(arr, dtype):
    # exact fp32 view of stored inputs; kept local so the oracle does not
    # depend on anything but numpy for its arithmetic
    if dtype == "bf16":
        return (np.ascontiguousarray(arr, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
    return np.ascontiguousarray(arr, dtype=np.float32)


def run(problem, *, pair_mask=None, nthreads: Optional[int] = None, mutant: int = 0,
        delta_rule: bool = True, l2norm: bool = True):
    """The oracle on a `workloads.Problem`: returns (o fp64, final pool fp64)."""
    p = problem
    return run_arrays(offsets=p.offsets, slot_idx=p.slot_idx, q=_widen(p.q, p.qkv_dtype),
                      k=_widen(p.k, p.qkv_dtype), v=_widen(p.v, p.qkv_dtype), beta=p.beta, g=p.g,
                      per_channel=(p.decay_kind == "per_channel"),
                      pool=_widen(p.pool, p.state_dtype), scale=p.scale, l2norm=l2norm,
                      delta_rule=delta_rule, pair_mask=pair_mask, nthreads=nthreads,
                      mutant=mutant)


def run_gdp(problem, *, nthreads: Optional[int] = None, mutant: int = 0):
    """The Gated DeltaProduct oracle on a `workloads.Problem` with n_h substeps."""
    p = problem
    return run_gdp_arrays(offsets=p.offsets, slot_idx=p.slot_idx, q=_widen(p.q, p.qkv_dtype),
                          k=_widen(p.k, p.qkv_dtype), v=_widen(p.v, p.qkv_dtype), beta=p.beta,
                          g=p.g, per_channel=(p.decay_kind == "per_channel"),
                          pool=_widen(p.pool, p.state_dtype), scale=p.scale, nthreads=nthreads,
                          mutant=mutant)


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """fp64 values rounded to the nearest bf16 value (8 significant bits, ties to even).

    Normal-range numbers only (the state pool never leaves it): x = m 2^e with
    m in [0.5, 1); m 2^8 is rounded half-to-even to an integer and scaled back.
    """
    x = np.asarray(x, np.float64)
    m, e = np.frexp(x)
    return np.ldexp(np.round(m * 256.0) / 256.0, e)


def run_decode(dp, *, steps: Optional[int] = None, nthreads: Optional[int] = None,
               seq_mask=None, delta_rule: bool = True):
    """The oracle on a `workloads.DecodeProblem`: each step is one token per sequence.

    Between steps the state lives in the pool, so a bf16 pool holds it rounded to
    bf16 (Modular "gated_delta" module: the pool keeps its own dtype, independent of
    the working precision); within a step the arithmetic is fp64.
    Returns (o fp64 [steps, B, HV, dv], final pool fp64, unrounded after the last
    step).  `seq_mask` limits the work to some sequences (others keep their initial
    state and zero output).
    """
    steps = dp.steps if steps is None else steps
    B = dp.num_seqs
    pool = _widen(dp.pool, dp.state_dtype).astype(np.float64)
    offsets = np.arange(B + 1, dtype=np.int64)
    outs = []
    pair_mask = None
    if seq_mask is not None:
        pair_mask = np.repeat(np.asarray(seq_mask, dtype=np.uint8), dp.num_v_heads)
    for s in range(steps):
        if s > 0 and dp.state_dtype == "bf16":
            pool = round_to_bf16(pool)
        o, pool = run_arrays(offsets=offsets, slot_idx=dp.slot_idx,
                             q=_widen(dp.q[s], dp.qkv_dtype), k=_widen(dp.k[s], dp.qkv_dtype),
                             v=_widen(dp.v[s], dp.qkv_dtype), beta=dp.beta[s], g=dp.g[s],
                             per_channel=(dp.decay_kind == "per_channel"), pool=pool,
                             scale=dp.scale, delta_rule=delta_rule, pair_mask=pair_mask,
                             nthreads=nthreads)
        outs.append(o)
    return np.stack(outs), pool


# ----------------------------------------------------------------------------------------------
# numpy restatements (tiny inputs only)
# ----------------------------------------------------------------------------------------------

def _normalise_rows(x):
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + L2_EPS)


def recurrence_py(q, k, v, beta, g, S0, *, scale=None, l2norm=True, delta_rule=True,
                  return_states=False):
    """One sequence, one head, the five steps in numpy fp64.

    q, k: [T, dk]; v: [T, dv]; beta: [T]; g: [T] or [T, dk]; S0: [dk, dv] (stored
    orientation, the transpose of the d_v x d_k state of the derivation).
    Returns o [T, dv] and the final state (and, optionally, the state after every token).
    """
    q = np.asarray(q, np.float64); k = np.asarray(k, np.float64); v = np.asarray(v, np.float64)
    beta = np.asarray(beta, np.float64); g = np.asarray(g, np.float64)
    T, dk = q.shape
    if scale is None or scale <= 0:
        scale = 1.0 / np.sqrt(dk)
    if l2norm:
        q, k = _normalise_rows(q), _normalise_rows(k)
    q = q * scale
    S = np.array(S0, np.float64, copy=True)
    o = np.zeros((T, v.shape[1]))
    states = []
    for t in range(T):
        a = np.exp(g[t]) * np.ones(dk) if g.ndim == 1 else np.exp(g[t])
        S = S * a[:, None]                       # forget (key channel = row)
        vhat = k[t] @ S                          # predict
        e = beta[t] * (v[t] - vhat) if delta_rule else beta[t] * v[t]   # correct
        S = S + np.outer(k[t], e)                # write
        o[t] = q[t] @ S                          # read after the write
        if return_states:
            states.append(S.copy())
    if return_states:
        return o, S, states
    return o, S


def chunk_form(q, k, v, beta, g, S0, *, chunk: int, scale=None, l2norm=True):
    """The chunkwise closed form of "You Could Have Come Up With Kimi Delta Attention", sec. 6.

    For one sequence and one head, chunk by chunk (sec. 6.1-6.5):
      D_{0:i}         decay from the chunk boundary through token i
      ebar_i          = beta_i (v_i - S_c D_{0:i} k_i)                       (6.2)
      rho_ij          = beta_i <k_j| D_{j+1:i} |k_i>, j < i;  R strictly lower  (6.3)
      E               = Ebar (I + R)^{-T}                                    (6.3)
      S_{c+1}         = S_c D_{0:C-1} + E K_end                              (6.4)
      chi_ij          = s <k_j| D_{j+1:i} |q_i>, j <= i                      (6.5)
      O               = s S_c Q_boundary + E A_qk^T                          (6.5)
    written in the derivation's orientation (state d_v x d_k, vectors as columns),
    with dense fp64 matrices and a library solve for the triangular system.
    Inputs/outputs use the stored orientation S0: [dk, dv].
    """
    q = np.asarray(q, np.float64); k = np.asarray(k, np.float64); v = np.asarray(v, np.float64)
    beta = np.asarray(beta, np.float64); g = np.asarray(g, np.float64)
    T, dk = q.shape
    if scale is None or scale <= 0:
        scale = 1.0 / np.sqrt(dk)
    if l2norm:
        q, k = _normalise_rows(q), _normalise_rows(k)
    if g.ndim == 1:
        g = np.repeat(g[:, None], dk, axis=1)
    S = np.array(S0, np.float64).T.copy()        # derivation orientation: d_v x d_k
    o = np.zeros((T, v.shape[1]))
    for c0 in range(0, T, chunk):
        idx = np.arange(c0, min(c0 + chunk, T))
        n = len(idx)
        alpha = np.exp(g[idx])                   # [n, dk] diagonals of D_i
        D0i = np.cumprod(alpha, axis=0)          # diag of D_{0:i}
        def Dji(j, i):                           # diag of D_{j+1:i}, j < i (identity if j == i)
            return np.prod(alpha[j + 1:i + 1], axis=0) if j < i else np.ones(dk)
        Ebar = np.stack([beta[idx[i]] * (v[idx[i]] - S @ (D0i[i] * k[idx[i]])) for i in range(n)],
                        axis=1)                  # columns ebar_i, [dv, n]
        R = np.zeros((n, n))
        for i in range(n):
            for j in range(i):
                R[i, j] = beta[idx[i]] * (k[idx[j]] @ (Dji(j, i) * k[idx[i]]))
        Akk = np.linalg.inv(np.eye(n) + R)
        E = Ebar @ Akk.T
        Kend = np.stack([Dji(j, n - 1) * k[idx[j]] for j in range(n)], axis=0)   # rows
        Aqk = np.zeros((n, n))
        for i in range(n):
            for j in range(i + 1):
                Aqk[i, j] = scale * (k[idx[j]] @ (Dji(j, i) * q[idx[i]]))
        Qb = np.stack([D0i[i] * q[idx[i]] for i in range(n)], axis=1)           # columns
        O = scale * S @ Qb + E @ Aqk.T
        o[idx] = O.T
        S = S * D0i[n - 1][None, :] + E @ Kend
    return o, S.T.copy()


def causal_linear_attention(q, k, v, S0, *, scale=None, l2norm=True):
    """Brute force o = s (Q K^T masked causally) V + s Q S0 (no decay, no delta term).

    "From Attention to Learned Memory", sec. 2: the fully parallel causal form with the
    lower-triangular mask; S0 (stored orientation [dk, dv]) is the cached prefix state.
    """
    q = np.asarray(q, np.float64); k = np.asarray(k, np.float64); v = np.asarray(v, np.float64)
    T, dk = q.shape
    if scale is None or scale <= 0:
        scale = 1.0 / np.sqrt(dk)
    if l2norm:
        q, k = _normalise_rows(q), _normalise_rows(k)
    M = np.tril(np.ones((T, T)))
    return scale * ((q @ k.T) * M) @ v + scale * q @ np.asarray(S0, np.float64)


if __name__ == "__main__":  # pragma: no cover - manual build helper
    print(build(int(sys.argv[1]) if len(sys.argv) > 1 else 0, force=True))


def backward(problem, d_o, d_state=None, *, delta_rule: bool = True, l2norm: bool = True,
             pairs=None):
    """The backward oracle on a `workloads.Problem` (the pool holds the initial states):
    gradients of the loss whose gradients w.r.t. o and the final states are d_o and d_state.
    Returns dict(dq, dk, dv, dbeta, dg, d_state0), fp64."""
    from .bptt import backward_arrays
    p = problem
    return backward_arrays(offsets=p.offsets, slot_idx=p.slot_idx, q=_widen(p.q, p.qkv_dtype),
                           k=_widen(p.k, p.qkv_dtype), v=_widen(p.v, p.qkv_dtype), beta=p.beta,
                           g=p.g, pool=_widen(p.pool, p.state_dtype).astype(np.float64),
                           d_o=d_o, d_state=d_state, scale=p.scale, l2norm=l2norm,
                           delta_rule=delta_rule, pairs=pairs)

"""Seeded synthetic inputs for the gated delta rule forward pass.

This module only draws random numbers and lays them out.  It holds none of the
recurrence's arithmetic, so both the fp64 CPU oracle and the CUDA library can
consume the exact same bytes.

Five named workloads mirror the shapes, dtypes and value distributions of the
gated-delta-rule pages ("You Could Have Come Up With Kimi Delta Attention",
sec. 4 for the KDA gate and sec. 5/6 for the decode/chunk schedules; the Modular
`gated_delta` API page for the ragged batch, GQA and slot-indexed state pool):

  tiny_gdn        1 x 64 tokens, 1 head, d=16, fp32, scalar decay, chunk 16, zero state
  gdn_prefill     4 x 4096 tokens, 16 heads, d=128, bf16 q/k/v, scalar decay, fp32 state (zero), chunk 64
  kda_prefill     2 x 16384 tokens, 32 heads, d=128, bf16, per-channel decay, fp32 state ~N(0, 0.02)
  ragged_gqa_kda  8 sequences, log-uniform lengths in [64, 8192], 16 key / 32 value heads, d=128,
                  bf16, per-channel decay, bf16 pool of 64 slots ~N(0, 0.02), distinct random slots
  kda_decode      256 sequences x 64 single-token steps, 32 heads, d=128, bf16, per-channel decay,
                  fp32 pool ~N(0, 0.02), one slot per sequence

and one for the Gated DeltaProduct extension ("Linear attention visualized", Gated Delta
Product section: n_h keys, values and gates per token, one query and one decay):

  gdp_prefill     the gdn_prefill shape (4 x 4096 tokens, 16 heads, d=128, bf16, scalar decay,
                  fp32 zero state, chunk 64) with n_h = 2 substeps per token; seed 1006

Recipe (fixed draw order so every consumer sees identical values):
  generator   numpy PCG64, seed = 1000 + workload number (1..5)
  order       lengths, q, k, v, beta logits, decay noise, state, slot permutation
              (decode: per step q, k, v, beta logits, decay noise; then state, slots)
  q, k        N(0, 1) in fp32, scaled to unit L2 norm per head row (the stated input
              distribution), then stored in the workload dtype (bf16 round-to-nearest-even)
  v           N(0, 1), stored in the workload dtype
  beta        sigmoid(N(0, 1)), fp32
  log-decay   scalar: -softplus(N(0, 1)); per channel: -exp(N(-2, 0.5)); fp32
  state       zeros (tiny_gdn, gdn_prefill) or N(0, 0.02) stored in the pool dtype
  N(mu, s)    s is the standard deviation

bf16 tensors are carried as uint16 bit patterns (numpy has no bf16 type).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np

F32 = "f32"
BF16 = "bf16"
SCALAR = "scalar"
PER_CHANNEL = "per_channel"


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (round to nearest, ties to even); returns uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    b = x.view(np.uint32)
    # add 0x7FFF plus the lowest kept bit, then truncate (no overflow for finite inputs
    # below the largest bf16 magnitude, which is all these workloads produce)
    rounded = (b + (np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1)))) >> np.uint32(16)
    return rounded.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to fp32."""
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def as_f32(arr: np.ndarray, dtype: str) -> np.ndarray:
    """Exact fp32 view of a stored tensor (bf16 bits are widened, fp32 passes through)."""
    return bf16_bits_to_f32(arr) if dtype == BF16 else np.ascontiguousarray(arr, dtype=np.float32)


def _store(x32: np.ndarray, dtype: str) -> np.ndarray:
    return f32_to_bf16_bits(x32) if dtype == BF16 else np.ascontiguousarray(x32, dtype=np.float32)


def _unit_rows(x: np.ndarray) -> np.ndarray:
    # Input distribution only: directions uniform on the sphere (a Gaussian
    # draw scaled to unit length), as the workload description states.
    n = np.sqrt(np.einsum("...i,...i->...", x, x, dtype=np.float64))[..., None]
    return (x / n).astype(np.float32)


def _sigmoid(x: np.ndarray) -> np.ndarray:
    return (1.0 / (1.0 + np.exp(-x.astype(np.float64)))).astype(np.float32)


def _neg_softplus(x: np.ndarray) -> np.ndarray:
    x = x.astype(np.float64)
    return (-(np.maximum(x, 0.0) + np.log1p(np.exp(-np.abs(x))))).astype(np.float32)


@dataclasses.dataclass
class Problem:
    """One prefill call's inputs (token-major, ragged)."""

    name: str
    num_seqs: int
    offsets: np.ndarray          # uint32 [num_seqs+1]
    num_k_heads: int
    num_v_heads: int
    d_k: int
    d_v: int
    qkv_dtype: str               # "f32" | "bf16"
    state_dtype: str
    decay_kind: str              # "scalar" | "per_channel"
    chunk: int
    q: np.ndarray                # [T, HK, d_k]  (uint16 bits for bf16)
    k: np.ndarray                # [T, HK, d_k]
    v: np.ndarray                # [T, HV, d_v]
    beta: np.ndarray             # f32 [T, HV]
    g: np.ndarray                # f32 [T, HV] or [T, HV, d_k]
    pool: np.ndarray             # [num_slots, HV, d_k, d_v]
    slot_idx: np.ndarray         # uint32 [num_seqs]
    scale: float = 0.0           # <= 0 means 1/sqrt(d_k)
    n_h: int = 1                 # substeps per token (Gated DeltaProduct): k [T, n_h, HK, d_k],
                                 # v [T, n_h, HV, d_v], beta [T, n_h, HV]; q and g stay per token

    @property
    def total_tokens(self) -> int:
        return int(self.offsets[-1])

    @property
    def num_slots(self) -> int:
        return int(self.pool.shape[0])

    @property
    def lengths(self) -> np.ndarray:
        return np.diff(self.offsets.astype(np.int64))


@dataclasses.dataclass
class DecodeProblem:
    """A run of single-token decode steps over a batch of sequences."""

    name: str
    num_seqs: int
    steps: int
    num_k_heads: int
    num_v_heads: int
    d_k: int
    d_v: int
    qkv_dtype: str
    state_dtype: str
    decay_kind: str
    q: np.ndarray                # [steps, B, HK, d_k]
    k: np.ndarray
    v: np.ndarray                # [steps, B, HV, d_v]
    beta: np.ndarray             # f32 [steps, B, HV]
    g: np.ndarray                # f32 [steps, B, HV(, d_k)]
    pool: np.ndarray             # [num_slots, HV, d_k, d_v]
    slot_idx: np.ndarray         # uint32 [B]
    scale: float = 0.0

    @property
    def num_slots(self) -> int:
        return int(self.pool.shape[0])


def _draw_tokens(rng, T, HK, HV, dk, dv, dtype, decay_kind):
    q = _unit_rows(rng.standard_normal((T, HK, dk), dtype=np.float32))
    k = _unit_rows(rng.standard_normal((T, HK, dk), dtype=np.float32))
    v = rng.standard_normal((T, HV, dv), dtype=np.float32)
    beta = _sigmoid(rng.standard_normal((T, HV), dtype=np.float32))
    if decay_kind == SCALAR:
        g = _neg_softplus(rng.standard_normal((T, HV), dtype=np.float32))
    else:
        g = (-np.exp(rng.normal(-2.0, 0.5, size=(T, HV, dk)))).astype(np.float32)
    return _store(q, dtype), _store(k, dtype), _store(v, dtype), beta, g


def _draw_state(rng, shape, dtype, zero):
    if zero:
        s = np.zeros(shape, dtype=np.float32)
    else:
        s = (rng.standard_normal(shape, dtype=np.float32) * np.float32(0.02)).astype(np.float32)
    return _store(s, dtype)


def make_problem(name: str, *, num_seqs: int, lengths, num_k_heads: int, num_v_heads: int,
                 d: int, qkv_dtype: str, state_dtype: str, decay_kind: str, chunk: int,
                 zero_state: bool, num_slots: Optional[int] = None, seed: int = 0,
                 shuffle_slots: bool = True) -> Problem:
    """Generic seeded prefill problem (used by the named workloads and by tests)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    lengths = np.asarray(lengths, dtype=np.int64)
    assert lengths.shape == (num_seqs,)
    offsets = np.zeros(num_seqs + 1, dtype=np.uint32)
    offsets[1:] = np.cumsum(lengths)
    T = int(offsets[-1])
    q, k, v, beta, g = _draw_tokens(rng, T, num_k_heads, num_v_heads, d, d, qkv_dtype, decay_kind)
    if num_slots is None:
        num_slots = num_seqs
    pool = _draw_state(rng, (num_slots, num_v_heads, d, d), state_dtype, zero_state)
    if shuffle_slots:
        slot_idx = rng.permutation(num_slots)[:num_seqs].astype(np.uint32)
    else:
        slot_idx = np.arange(num_seqs, dtype=np.uint32)
    return Problem(name, num_seqs, offsets, num_k_heads, num_v_heads, d, d, qkv_dtype,
                   state_dtype, decay_kind, chunk, q, k, v, beta, g, pool, slot_idx)


def make_gdp_problem(name: str, *, num_seqs: int, lengths, n_h: int, num_k_heads: int,
                     num_v_heads: int, d: int, qkv_dtype: str, state_dtype: str,
                     decay_kind: str, chunk: int, zero_state: bool,
                     num_slots: Optional[int] = None, seed: int = 0) -> Problem:
    """Seeded Gated DeltaProduct prefill problem: the distributions of the other workloads,
    drawn in the order lengths, q, k, v, beta logits, decay noise, state, slots, with the
    substep axis right after the token axis of k, v and beta."""
    rng = np.random.Generator(np.random.PCG64(seed))
    lengths = np.asarray(lengths, dtype=np.int64)
    assert lengths.shape == (num_seqs,) and n_h >= 1
    offsets = np.zeros(num_seqs + 1, dtype=np.uint32)
    offsets[1:] = np.cumsum(lengths)
    T, HK, HV = int(offsets[-1]), num_k_heads, num_v_heads
    q = _unit_rows(rng.standard_normal((T, HK, d), dtype=np.float32))
    k = _unit_rows(rng.standard_normal((T, n_h, HK, d), dtype=np.float32))
    v = rng.standard_normal((T, n_h, HV, d), dtype=np.float32)
    beta = _sigmoid(rng.standard_normal((T, n_h, HV), dtype=np.float32))
    if decay_kind == SCALAR:
        g = _neg_softplus(rng.standard_normal((T, HV), dtype=np.float32))
    else:
        g = (-np.exp(rng.normal(-2.0, 0.5, size=(T, HV, d)))).astype(np.float32)
    if num_slots is None:
        num_slots = num_seqs
    pool = _draw_state(rng, (num_slots, HV, d, d), state_dtype, zero_state)
    slot_idx = rng.permutation(num_slots)[:num_seqs].astype(np.uint32)
    return Problem(name, num_seqs, offsets, HK, HV, d, d, qkv_dtype, state_dtype, decay_kind,
                   chunk, _store(q, qkv_dtype), _store(k, qkv_dtype), _store(v, qkv_dtype),
                   beta, g, pool, slot_idx, n_h=n_h)


def ragged_lengths(rng, n: int, lo: int, hi: int) -> np.ndarray:
    """Log-uniform integer lengths in [lo, hi]."""
    u = rng.uniform(math.log(lo), math.log(hi), size=n)
    return np.clip(np.rint(np.exp(u)), lo, hi).astype(np.int64)


WORKLOADS = ("tiny_gdn", "gdn_prefill", "kda_prefill", "ragged_gqa_kda", "kda_decode")


def workload(name: str, replica: int = 0):
    """The named workload (Problem, or DecodeProblem for kda_decode).

    replica > 0 draws another batch of the same sizes (same sequence lengths and heads; tensors,
    and shuffled slots, from a seed offset by replica << 24): what each rank of a multi-GPU run
    processes.
    Replica 0 is the workload itself.
    """
    off = replica << 24
    if name == "tiny_gdn":
        return make_problem(name, num_seqs=1, lengths=[64], num_k_heads=1, num_v_heads=1, d=16,
                            qkv_dtype=F32, state_dtype=F32, decay_kind=SCALAR, chunk=16,
                            zero_state=True, seed=1001 + off, shuffle_slots=False)
    if name == "gdn_prefill":
        return make_problem(name, num_seqs=4, lengths=[4096] * 4, num_k_heads=16, num_v_heads=16,
                            d=128, qkv_dtype=BF16, state_dtype=F32, decay_kind=SCALAR, chunk=64,
                            zero_state=True, seed=1002 + off, shuffle_slots=False)
    if name == "kda_prefill":
        return make_problem(name, num_seqs=2, lengths=[16384] * 2, num_k_heads=32, num_v_heads=32,
                            d=128, qkv_dtype=BF16, state_dtype=F32, decay_kind=PER_CHANNEL,
                            chunk=64, zero_state=False, seed=1003 + off, shuffle_slots=False)
    if name == "ragged_gqa_kda":
        rng = np.random.Generator(np.random.PCG64(1004))
        lengths = ragged_lengths(rng, 8, 64, 8192)
        # The lengths come from their own stream; the tensors from seed 1004 + 1 << 20.
        return make_problem(name, num_seqs=8, lengths=lengths, num_k_heads=16, num_v_heads=32,
                            d=128, qkv_dtype=BF16, state_dtype=BF16, decay_kind=PER_CHANNEL,
                            chunk=64, zero_state=False, num_slots=64, seed=1004 + (1 << 20) + off,
                            shuffle_slots=True)
    if name == "gdp_prefill":
        return make_gdp_problem(name, num_seqs=4, lengths=[4096] * 4, n_h=2, num_k_heads=16,
                                num_v_heads=16, d=128, qkv_dtype=BF16, state_dtype=F32,
                                decay_kind=SCALAR, chunk=64, zero_state=True, seed=1006 + off)
    if name == "kda_decode":
        return make_decode_problem(name, num_seqs=256, steps=64, num_k_heads=32, num_v_heads=32,
                                   d=128, qkv_dtype=BF16, state_dtype=F32,
                                   decay_kind=PER_CHANNEL, zero_state=False, seed=1005 + off)
    raise KeyError(name)


def make_decode_problem(name: str, *, num_seqs: int, steps: int, num_k_heads: int,
                        num_v_heads: int, d: int, qkv_dtype: str, state_dtype: str,
                        decay_kind: str, zero_state: bool, seed: int,
                        num_slots: Optional[int] = None) -> DecodeProblem:
    rng = np.random.Generator(np.random.PCG64(seed))
    qs, ks, vs, bs, gs = [], [], [], [], []
    for _ in range(steps):
        q, k, v, beta, g = _draw_tokens(rng, num_seqs, num_k_heads, num_v_heads, d, d,
                                        qkv_dtype, decay_kind)
        qs.append(q); ks.append(k); vs.append(v); bs.append(beta); gs.append(g)
    if num_slots is None:
        num_slots = num_seqs
    pool = _draw_state(rng, (num_slots, num_v_heads, d, d), state_dtype, zero_state)
    slot_idx = rng.permutation(num_slots)[:num_seqs].astype(np.uint32)
    return DecodeProblem(name, num_seqs, steps, num_k_heads, num_v_heads, d, d, qkv_dtype,
                         state_dtype, decay_kind, np.stack(qs), np.stack(ks), np.stack(vs),
                         np.stack(bs), np.stack(gs), pool, slot_idx)


def subset_heads(p: Problem, v_heads) -> Problem:
    """A view of a problem restricted to some value heads (and the key heads they use).

    Used to sample a full-size workload: every value head is an independent
    recurrence, so checking a subset of heads checks those outputs exactly.
    The returned problem keeps the GQA ratio by taking whole key-head groups.
    """
    r = p.num_v_heads // p.num_k_heads
    kh = sorted({h // r for h in v_heads})
    vh = [kk * r + j for kk in kh for j in range(r)]
    return dataclasses.replace(
        p, num_k_heads=len(kh), num_v_heads=len(vh),
        q=np.ascontiguousarray(p.q[:, kh]), k=np.ascontiguousarray(p.k[:, kh]),
        v=np.ascontiguousarray(p.v[:, vh]), beta=np.ascontiguousarray(p.beta[:, vh]),
        g=np.ascontiguousarray(p.g[:, vh]), pool=np.ascontiguousarray(p.pool[:, vh]))

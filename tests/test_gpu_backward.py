"""The backward pass (kda_prefill_bwd through the C ABI) against the fp64 backward oracle
(`oracle/bptt.py`, pinned by finite differences of the forward recurrence).

Every gradient tensor is compared element by element: rel = max|x - ref| / max|ref| per
tensor, within the bound of the inputs' dtype (2e-3 bf16, 1e-4 fp32; the arithmetic is fp32
either way).  Small ragged GQA cases cover every chunk size, both head sizes and gate kinds,
both pool dtypes, the additive write and an empty sequence; the gdn_prefill and kda_prefill
shapes are checked on sampled (sequence, value head) pairs, whose gradients the oracle
computes one pair at a time.
"""
import numpy as np
import pytest
import torch

import gated_delta_rule_deltanet_gb300 as kda
import oracle
import workloads
from workloads import torch_io

pytestmark = pytest.mark.gpu

TOL = {"bf16": 2e-3, "f32": 1e-4}
DEV = "cuda:0"


def rel_err(x, ref):
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.all(np.isfinite(x)), "non-finite gradient"
    den = np.max(np.abs(ref))
    return float(np.max(np.abs(x - ref)) / (den if den > 0 else 1.0))


def seeds(p, seed):
    r = np.random.Generator(np.random.PCG64(seed))
    d_o = r.standard_normal((p.total_tokens, p.num_v_heads, p.d_v)).astype(np.float32)
    d_state = r.standard_normal(p.pool.shape).astype(np.float32)
    return d_o, d_state


def gpu_backward(p, d_o, d_state, **kw):
    t = torch_io.prefill_inputs(p, DEV)
    g = kda.prefill_bwd(t["q"], t["k"], t["v"], t["beta"], t["log_decay"], t["input_row_offsets"],
                        t["slot_idx"], t["state_pool"], torch.from_numpy(d_o).to(DEV),
                        torch.from_numpy(d_state).to(DEV), chunk=p.chunk, scale=p.scale, **kw)
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0
    names = ("dq", "dk", "dv", "dbeta", "dg", "d_state0")
    return {n: x.double().cpu().numpy() for n, x in zip(names, g)}


def compare(got, ref, tol, rows=None, label=""):
    errs = {}
    for name in ("dq", "dk", "dv", "dbeta", "dg", "d_state0"):
        x, r = got[name], ref[name]
        if rows is not None and name in rows:
            x, r = x[rows[name]], r[rows[name]]
        errs[name] = rel_err(x, r)
    bad = {n: e for n, e in errs.items() if e > tol}
    assert not bad, f"{label}: {errs} (tol {tol})"
    return errs


CASES = [
    # name, lengths, HK, HV, d, qkv, state, decay, chunk, delta_rule
    ("f32-d16-c16-kda", [1, 15, 0, 17, 40], 1, 2, 16, "f32", "f32", "per_channel", 16, True),
    ("f32-d16-c32-gdn", [33, 70], 2, 2, 16, "f32", "f32", "scalar", 32, True),
    ("f32-d128-c64-kda", [130, 64, 1], 1, 2, 128, "f32", "f32", "per_channel", 64, True),
    ("bf16-d128-c64-gdn", [200, 65], 2, 4, 128, "bf16", "f32", "scalar", 64, True),
    ("bf16-d128-c64-kda-bf16pool", [150, 3], 2, 2, 128, "bf16", "bf16", "per_channel", 64, True),
    ("bf16-d128-c16-kda", [90], 1, 2, 128, "bf16", "f32", "per_channel", 16, True),
    ("f32-d128-c32-gla", [100, 29], 2, 2, 128, "f32", "f32", "per_channel", 32, False),
    ("bf16-d16-c64-mamba2", [129, 0, 7], 1, 1, 16, "bf16", "f32", "scalar", 64, False),
    # the tensor-core kernels' additive-write branches (bf16, d = 128, chunk 64)
    ("bf16-d128-c64-mamba2", [129, 0, 70], 2, 4, 128, "bf16", "f32", "scalar", 64, False),
    ("bf16-d128-c64-gla", [100, 29], 2, 2, 128, "bf16", "bf16", "per_channel", 64, False),
]


@pytest.mark.parametrize("cfg", CASES, ids=[c[0] for c in CASES])
def test_backward_small(cfg):
    name, lengths, HK, HV, d, qkv, state, decay, chunk, delta = cfg
    p = workloads.make_problem(name, num_seqs=len(lengths), lengths=lengths, num_k_heads=HK,
                               num_v_heads=HV, d=d, qkv_dtype=qkv, state_dtype=state,
                               decay_kind=decay, chunk=chunk, zero_state=False,
                               num_slots=len(lengths) + 2, seed=sum(map(ord, name)))
    d_o, d_state = seeds(p, 7)
    got = gpu_backward(p, d_o, d_state, delta_rule=delta)
    ref = oracle.backward(p, d_o.astype(np.float64), d_state.astype(np.float64), delta_rule=delta)
    compare(got, ref, TOL[qkv], label=name)
    # slots no sequence names keep their zero gradient
    untouched = np.setdiff1d(np.arange(p.num_slots), np.asarray(p.slot_idx, np.int64))
    assert np.all(got["d_state0"][untouched] == 0.0)


def test_backward_without_state_gradient():
    """d_state = None is a zero gradient w.r.t. the final states."""
    p = workloads.make_problem("nostate", num_seqs=2, lengths=[70, 20], num_k_heads=1,
                               num_v_heads=2, d=128, qkv_dtype="bf16", state_dtype="f32",
                               decay_kind="per_channel", chunk=64, zero_state=False, num_slots=3,
                               seed=12)
    d_o, _ = seeds(p, 8)
    t = torch_io.prefill_inputs(p, DEV)
    g = kda.prefill_bwd(t["q"], t["k"], t["v"], t["beta"], t["log_decay"], t["input_row_offsets"],
                        t["slot_idx"], t["state_pool"], torch.from_numpy(d_o).to(DEV), None,
                        chunk=64)
    torch.cuda.synchronize()
    got = {n: x.double().cpu().numpy()
           for n, x in zip(("dq", "dk", "dv", "dbeta", "dg", "d_state0"), g)}
    ref = oracle.backward(p, d_o.astype(np.float64), None)
    compare(got, ref, TOL["bf16"], label="nostate")


@pytest.mark.parametrize("name,pairs", [("gdn_prefill", [(0, 3), (2, 15)]),
                                        ("kda_prefill", [(1, 0)])])
def test_backward_full_size_sampled(name, pairs):
    """The full shapes, every gradient of sampled (sequence, value head) pairs (their key
    heads carry no other value head's contribution: HK = HV here)."""
    p = workloads.workload(name)
    assert p.num_k_heads == p.num_v_heads
    d_o, d_state = seeds(p, 9)
    got = gpu_backward(p, d_o, d_state)
    ref = oracle.backward(p, d_o.astype(np.float64), d_state.astype(np.float64), pairs=pairs)
    offs = p.offsets.astype(np.int64)
    for b, h in pairs:
        s, e = offs[b], offs[b + 1]
        slot = int(p.slot_idx[b])
        rows = {"dq": (slice(s, e), h), "dk": (slice(s, e), h), "dv": (slice(s, e), h),
                "dbeta": (slice(s, e), h), "dg": (slice(s, e), h), "d_state0": (slot, h)}
        compare(got, ref, TOL[p.qkv_dtype], rows=rows, label=f"{name} pair {(b, h)}")


def test_backward_strong_decay_takes_the_exact_pairwise_path():
    """Per-channel decay of ~5 nats per token exceeds the anchored factors' 80-nat range
    within a 64-token chunk, so the local stage and the pairwise terms evaluate the decay
    per pair and channel; the gradients still match the oracle."""
    p = workloads.make_problem("strong", num_seqs=2, lengths=[100, 37], num_k_heads=1,
                               num_v_heads=2, d=16, qkv_dtype="f32", state_dtype="f32",
                               decay_kind="per_channel", chunk=64, zero_state=False, num_slots=3,
                               seed=33)
    p.g[...] = p.g * 40.0
    assert float(np.max(-p.g)) * 32 > 80.0
    d_o, d_state = seeds(p, 10)
    got = gpu_backward(p, d_o, d_state)
    ref = oracle.backward(p, d_o.astype(np.float64), d_state.astype(np.float64))
    compare(got, ref, TOL["f32"], label="strong decay")


def test_backward_tensor_core_path_strong_decay_falls_back_exactly():
    """bf16, d = 128, chunk 64, per-channel decay strong enough (x40) that some chunks leave the
    anchored factors' 80-nat range: the tensor-core pairwise kernel leaves those (chunk, key
    head) pairs to the exact CUDA-core kernel; every gradient still matches the oracle."""
    p = workloads.make_problem("strong128", num_seqs=2, lengths=[150, 40], num_k_heads=1,
                               num_v_heads=2, d=128, qkv_dtype="bf16", state_dtype="f32",
                               decay_kind="per_channel", chunk=64, zero_state=False, num_slots=3,
                               seed=34)
    p.g[...] = p.g * 40.0
    assert float(np.max(-p.g)) * 32 > 80.0
    d_o, d_state = seeds(p, 15)
    got = gpu_backward(p, d_o, d_state)
    ref = oracle.backward(p, d_o.astype(np.float64), d_state.astype(np.float64))
    compare(got, ref, TOL["bf16"], label="strong decay, tensor-core path")


def test_backward_ragged_gqa_workload_sampled():
    """ragged_gqa_kda (8 ragged sequences, 16 key / 32 value heads, bf16 pool): every gradient
    of one key head's two value heads on two sequences; dq and dk of that key head sum both."""
    p = workloads.workload("ragged_gqa_kda")
    ratio = p.num_v_heads // p.num_k_heads
    assert ratio == 2
    d_o, d_state = seeds(p, 12)
    got = gpu_backward(p, d_o, d_state)
    kh = 5
    seqs = [int(np.argmax(p.lengths)), int(np.argmin(p.lengths))]
    pairs = [(b, kh * ratio + r) for b in seqs for r in range(ratio)]
    ref = oracle.backward(p, d_o.astype(np.float64), d_state.astype(np.float64), pairs=pairs)
    offs = p.offsets.astype(np.int64)
    for b in seqs:
        s, e = offs[b], offs[b + 1]
        slot = int(p.slot_idx[b])
        hs = slice(kh * ratio, (kh + 1) * ratio)
        rows = {"dq": (slice(s, e), kh), "dk": (slice(s, e), kh), "dv": (slice(s, e), hs),
                "dbeta": (slice(s, e), hs), "dg": (slice(s, e), hs), "d_state0": (slot, hs)}
        compare(got, ref, TOL[p.qkv_dtype], rows=rows, label=f"ragged_gqa_kda seq {b}")


def same_as_default(full, comp):
    for k in full:
        if k == "dg":     # shared-memory atomics sum a chunk's last-token terms in any order
            assert rel_err(comp[k], full[k]) < 1e-5, k
        else:
            assert np.array_equal(full[k], comp[k]), k


COMPACT_CASES = [
    # name, lengths, HK, HV, decay, state dtype: 4 x 64 value heads give windows of two chunk
    # positions (512 slots), so the longest sequence (5 chunks) runs three windows
    ("compact-kda-gqa", [300, 0, 1, 190], 32, 64, "per_channel", "f32"),
    ("compact-gdn-bf16pool", [129, 64, 257, 2], 64, 64, "scalar", "bf16"),
]


@pytest.mark.parametrize("cfg", COMPACT_CASES, ids=[c[0] for c in COMPACT_CASES])
def test_backward_compact_equals_default(cfg):
    """The bounded-workspace form (KDA_FLAG_COMPACT: windows of chunk positions, each window's
    entering state from a checkpoint sweep, the state gradient carried between windows) runs
    the same arithmetic per chunk, so every gradient equals the default form's bit for bit
    (dg up to the order of the pair kernel's shared-memory atomic sums over a chunk's
    channels, which no two runs fix); sampled (sequence, head) pairs also match the oracle."""
    name, lengths, HK, HV, decay, state = cfg
    p = workloads.make_problem(name, num_seqs=len(lengths), lengths=lengths, num_k_heads=HK,
                               num_v_heads=HV, d=128, qkv_dtype="bf16", state_dtype=state,
                               decay_kind=decay, chunk=64, zero_state=False,
                               num_slots=len(lengths) + 1, seed=sum(map(ord, name)))
    d_o, d_state = seeds(p, 13)
    full = gpu_backward(p, d_o, d_state)
    comp = gpu_backward(p, d_o, d_state, compact=True)
    same_as_default(full, comp)
    # every value head of the sampled key heads, so that dq and dk are complete
    ratio = HV // HK
    pairs = [(b, kh * ratio + r) for b, kh in ((0, 0), (3, HK - 1), (2, HK // 2))
             for r in range(ratio)]
    ref = oracle.backward(p, d_o.astype(np.float64), d_state.astype(np.float64), pairs=pairs)
    offs = p.offsets.astype(np.int64)
    # norm-wise over the sample (the bound's reading): each gradient's sampled rows together
    got_s, ref_s = {}, {}
    for n in ("dq", "dk", "dv", "dbeta", "dg", "d_state0"):
        sel = []
        for b, h in pairs:
            s, e = offs[b], offs[b + 1]
            sel.append((int(p.slot_idx[b]), h) if n == "d_state0"
                       else (slice(s, e), h // ratio if n in ("dq", "dk") else h))
        got_s[n] = np.concatenate([np.ravel(comp[n][r]) for r in sel])
        ref_s[n] = np.concatenate([np.ravel(ref[n][r]) for r in sel])
    compare(got_s, ref_s, TOL["bf16"], label=f"{name} pairs {pairs}")


def test_backward_compact_full_size_kda_prefill():
    """kda_prefill (2 x 16384 tokens, 32 heads, per-channel decay) in the bounded workspace
    (32 windows of 8 chunk positions): equal to the default form, and a sampled pair against
    the oracle."""
    p = workloads.workload("kda_prefill")
    d_o, d_state = seeds(p, 14)
    comp = gpu_backward(p, d_o, d_state, compact=True)
    full = gpu_backward(p, d_o, d_state)
    same_as_default(full, comp)
    b, h = 0, 5
    ref = oracle.backward(p, d_o.astype(np.float64), d_state.astype(np.float64), pairs=[(b, h)])
    offs = p.offsets.astype(np.int64)
    s, e = offs[b], offs[b + 1]
    rows = {n: (slice(s, e), h) for n in ("dq", "dk", "dv", "dbeta", "dg")}
    rows["d_state0"] = (int(p.slot_idx[b]), h)
    compare(comp, ref, TOL["bf16"], rows=rows, label="kda_prefill compact")

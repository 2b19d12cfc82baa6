"""Parity of the CUDA library (through the C ABI) with the fp64 oracle.

Tolerance (per tensor): rel = max|x - ref| / max|ref|, ref the fp64 oracle on the same
inputs; <= 2e-3 for bf16 q/k/v, <= 1e-4 for fp32 q/k/v.  A bf16 state pool is compared
after discounting half a bf16 ulp of the reference (the storage rounding itself).
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
    den = np.max(np.abs(ref))
    assert np.all(np.isfinite(x)), "non-finite output"
    return float(np.max(np.abs(x - ref)) / (den if den > 0 else 1.0))


def rel_err_bf16_storage(x, ref):
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    e = np.floor(np.log2(np.maximum(np.abs(ref), 1e-300)))
    half_ulp = np.exp2(e - 8)
    den = np.max(np.abs(ref))
    return float(np.max(np.maximum(np.abs(x - ref) - half_ulp, 0.0)) / (den if den > 0 else 1.0))


def state_err(p, pool_gpu, pool_ref):
    touched = np.asarray(p.slot_idx, np.int64)
    x, r = pool_gpu[touched], pool_ref[touched]
    return rel_err_bf16_storage(x, r) if p.state_dtype == "bf16" else rel_err(x, r)


def gpu_prefill(p, chunk=None, **kw):
    t = torch_io.prefill_inputs(p, DEV)
    o = kda.prefill(**t, chunk=chunk or p.chunk, scale=p.scale, **kw)
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0
    return o.double().cpu().numpy(), torch_io.pool_to_f64(t["state_pool"]), t


def check_prefill(p, chunk=None, nthreads=None):
    o, pool, _ = gpu_prefill(p, chunk)
    o_ref, pool_ref = oracle.run(p, nthreads=nthreads)
    tol = TOL[p.qkv_dtype]
    eo, es = rel_err(o, o_ref), state_err(p, pool, pool_ref)
    assert eo <= tol and es <= tol, f"{p.name}: o err {eo:.3e}, state err {es:.3e} (tol {tol})"
    return eo, es


def small(name, lengths, HK, HV, d, qkv, state, decay, chunk, seed, zero=False, slots=None):
    return workloads.make_problem(name, num_seqs=len(lengths), lengths=lengths, num_k_heads=HK,
                                  num_v_heads=HV, d=d, qkv_dtype=qkv, state_dtype=state,
                                  decay_kind=decay, chunk=chunk, zero_state=zero,
                                  num_slots=slots, seed=seed)


def test_tiny_gdn_workload():
    check_prefill(workloads.workload("tiny_gdn"))


# ragged tails, several tiles, every chunk size, both dtypes, GQA, both decay kinds
SMALL = [
    ("f32-d16-c16", [1, 15, 16, 17, 64, 100], 1, 2, 16, "f32", "f32", "per_channel", 16),
    ("f32-d16-c32", [33, 5, 70], 2, 2, 16, "f32", "f32", "scalar", 32),
    ("f32-d128-c64", [130, 64, 1], 1, 2, 128, "f32", "f32", "per_channel", 64),
    ("f32-d128-c16", [47, 81], 2, 4, 128, "f32", "bf16", "scalar", 16),
    ("bf16-d128-c64-kda", [300, 1, 63, 65, 128], 2, 4, 128, "bf16", "f32", "per_channel", 64),
    ("bf16-d128-c32-gdn", [257, 31], 4, 4, 128, "bf16", "f32", "scalar", 32),
    ("bf16-d128-c16-kda", [100, 9], 1, 4, 128, "bf16", "bf16", "per_channel", 16),
    ("bf16-d16-c64", [129, 200], 2, 2, 16, "bf16", "bf16", "per_channel", 64),
]


@pytest.mark.parametrize("cfg", SMALL, ids=[c[0] for c in SMALL])
def test_small_configs(cfg):
    name, lengths, HK, HV, d, qkv, state, decay, chunk = cfg
    check_prefill(small(name, lengths, HK, HV, d, qkv, state, decay, chunk, seed=hash(name) % 1000,
                        slots=len(lengths) + 3))


@pytest.mark.parametrize("name", ["gdn_prefill", "kda_prefill", "ragged_gqa_kda"])
def test_full_prefill_workload(name):
    """Every output and final state of the full workload against the oracle."""
    check_prefill(workloads.workload(name))


def test_full_decode_workload():
    """256 sequences x 64 decode steps: every output of every step and the final pool."""
    dp = workloads.workload("kda_decode")
    t = torch_io.decode_inputs(dp, DEV)
    pool = t["state_pool"]
    outs = []
    for s in range(dp.steps):
        outs.append(kda.decode_step(t["q"][s], t["k"][s], t["v"][s], t["beta"][s],
                                    t["log_decay"][s], t["slot_idx"], pool))
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0
    o = torch.stack(outs).double().cpu().numpy()
    o_ref, pool_ref = oracle.run_decode(dp)
    eo = rel_err(o, o_ref)
    es = rel_err(torch_io.pool_to_f64(pool), pool_ref)
    assert eo <= TOL["bf16"] and es <= TOL["bf16"], (eo, es)


@pytest.mark.parametrize("state", ["f32", "bf16"])
@pytest.mark.parametrize("decay", ["scalar", "per_channel"])
@pytest.mark.parametrize("d", [16, 128])
def test_decode_small(state, decay, d):
    dp = workloads.make_decode_problem("dec", num_seqs=5, steps=7, num_k_heads=2, num_v_heads=4,
                                       d=d, qkv_dtype="bf16", state_dtype=state,
                                       decay_kind=decay, zero_state=False, seed=d + 3,
                                       num_slots=9)
    t = torch_io.decode_inputs(dp, DEV)
    outs = [kda.decode_step(t["q"][s], t["k"][s], t["v"][s], t["beta"][s], t["log_decay"][s],
                            t["slot_idx"], t["state_pool"]) for s in range(dp.steps)]
    o = torch.stack(outs).double().cpu().numpy()
    o_ref, pool_ref = oracle.run_decode(dp)
    pool = torch_io.pool_to_f64(t["state_pool"])
    assert rel_err(o, o_ref) <= TOL["bf16"]
    touched = dp.slot_idx.astype(np.int64)
    err = rel_err_bf16_storage if state == "bf16" else rel_err
    assert err(pool[touched], pool_ref[touched]) <= TOL["bf16"]
    untouched = np.setdiff1d(np.arange(dp.num_slots), touched)
    np.testing.assert_array_equal(pool[untouched],
                                  workloads.as_f32(dp.pool, state)[untouched].astype(np.float64))


def test_decode_steps_equal_prefill_on_gpu():
    """Two schedules of one recurrence: n decode steps == one prefill of those n tokens."""
    dp = workloads.make_decode_problem("d", num_seqs=6, steps=20, num_k_heads=2, num_v_heads=4,
                                       d=128, qkv_dtype="bf16", state_dtype="f32",
                                       decay_kind="per_channel", zero_state=False, seed=77)
    t = torch_io.decode_inputs(dp, DEV)
    pool_a = t["state_pool"].clone()
    pool_b = t["state_pool"].clone()
    o_dec = torch.stack([kda.decode_step(t["q"][s], t["k"][s], t["v"][s], t["beta"][s],
                                         t["log_decay"][s], t["slot_idx"], pool_a)
                         for s in range(dp.steps)])            # [S, B, HV, D]
    tm = lambda x: x.transpose(0, 1).reshape((-1,) + tuple(x.shape[2:])).contiguous()
    offs = torch.arange(dp.num_seqs + 1, dtype=torch.int32, device=DEV) * dp.steps
    o_pre = kda.prefill(tm(t["q"]), tm(t["k"]), tm(t["v"]), tm(t["beta"]), tm(t["log_decay"]),
                        offs, t["slot_idx"], pool_b, chunk=16)
    o_dec = o_dec.transpose(0, 1).reshape(o_pre.shape)
    assert rel_err(o_pre.cpu().numpy(), o_dec.cpu().numpy()) <= TOL["bf16"]
    assert rel_err(pool_b.cpu().numpy(), pool_a.cpu().numpy()) <= TOL["bf16"]


def test_prefill_split_resumes_from_pool():
    """S0 is the state of the cached prefix: prefill(x[:a]) then prefill(x[a:]) == prefill(x)."""
    p = small("split", [333], 2, 4, 128, "bf16", "f32", "per_channel", 64, seed=5)
    full_o, full_pool, _ = gpu_prefill(p)
    a = 150
    def part(lo, hi, pool):
        q = dict(p.__dict__)
        sub = workloads.Problem(**{**q, "offsets": np.array([0, hi - lo], np.uint32),
                                   "q": p.q[lo:hi], "k": p.k[lo:hi], "v": p.v[lo:hi],
                                   "beta": p.beta[lo:hi], "g": p.g[lo:hi], "pool": pool})
        return sub
    t1 = part(0, a, p.pool)
    o1, pool1, _ = gpu_prefill(t1)
    t2 = part(a, 333, np.ascontiguousarray(pool1.astype(np.float32)))
    o2, pool2, _ = gpu_prefill(t2)
    assert rel_err(np.concatenate([o1, o2]), full_o) <= TOL["bf16"]
    assert rel_err(pool2, full_pool) <= TOL["bf16"]


def test_untouched_slots_and_packing_order():
    """Slots not in slot_idx are bit-identical; packing order does not change any result."""
    p = small("pack", [70, 0, 200, 1, 129], 2, 4, 128, "bf16", "bf16", "per_channel", 64,
              seed=9, slots=11)
    o, pool, _ = gpu_prefill(p)
    untouched = np.setdiff1d(np.arange(p.num_slots), p.slot_idx.astype(np.int64))
    np.testing.assert_array_equal(pool[untouched],
                                  workloads.as_f32(p.pool, "bf16")[untouched].astype(np.float64))
    # the empty sequence's slot is untouched too
    empty_slot = int(p.slot_idx[1])
    np.testing.assert_array_equal(pool[empty_slot],
                                  workloads.as_f32(p.pool, "bf16")[empty_slot].astype(np.float64))
    # reverse the packing order of the sequences
    order = [4, 3, 2, 1, 0]
    L = p.lengths
    segs = [slice(int(p.offsets[b]), int(p.offsets[b + 1])) for b in order]
    cat = lambda a: np.concatenate([a[s] for s in segs])
    offs = np.concatenate([[0], np.cumsum(L[order])]).astype(np.uint32)
    rp = workloads.Problem(**{**p.__dict__, "offsets": offs, "q": cat(p.q), "k": cat(p.k),
                              "v": cat(p.v), "beta": cat(p.beta), "g": cat(p.g),
                              "slot_idx": p.slot_idx[order]})
    o2, pool2, _ = gpu_prefill(rp)
    for j, b in enumerate(order):
        np.testing.assert_allclose(o2[int(offs[j]):int(offs[j + 1])], o[segs[j]], rtol=0, atol=0)
    np.testing.assert_array_equal(pool2, pool)


def test_gqa_equals_repeated_heads():
    """Key head = value head // (HV/HK): GQA equals MHA with q, k repeated per group."""
    p = small("gqa", [90, 37], 2, 6, 128, "bf16", "f32", "per_channel", 32, seed=13)
    o, pool, _ = gpu_prefill(p)
    rep = np.repeat(np.arange(2), 3)
    m = workloads.Problem(**{**p.__dict__, "num_k_heads": 6,
                             "q": np.ascontiguousarray(p.q[:, rep]),
                             "k": np.ascontiguousarray(p.k[:, rep])})
    o2, pool2, _ = gpu_prefill(m)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(pool, pool2)


@pytest.mark.parametrize("decay", ["scalar", "per_channel"])
def test_chunk_size_invariance(decay):
    """Every valid chunk size gives the same result (up to rounding)."""
    p = small("cinv", [200, 77], 2, 2, 128, "bf16", "f32", decay, 64, seed=17)
    o64, s64, _ = gpu_prefill(p, chunk=64)
    for c in (16, 32):
        o, s, _ = gpu_prefill(p, chunk=c)
        assert rel_err(o, o64) <= TOL["bf16"] and rel_err(s, s64) <= TOL["bf16"]


def test_packed_qkv_row_strides():
    """q, k, v as column blocks of one packed [T, 2 HK D + HV D] buffer."""
    p = small("packed", [77, 130], 2, 4, 128, "bf16", "f32", "per_channel", 64, seed=21)
    o_ref, pool_ref, _ = gpu_prefill(p)
    t = torch_io.prefill_inputs(p, DEV)
    T, HK, D = t["q"].shape
    HV = t["v"].shape[1]
    packed = torch.cat([t["q"].reshape(T, -1), t["k"].reshape(T, -1), t["v"].reshape(T, -1)], 1)
    q = packed[:, :HK * D].view(T, HK, D)
    k = packed[:, HK * D:2 * HK * D].view(T, HK, D)
    v = packed[:, 2 * HK * D:].view(T, HV, D)
    o = kda.prefill(q, k, v, t["beta"], t["log_decay"], t["input_row_offsets"], t["slot_idx"],
                    t["state_pool"], chunk=64)
    np.testing.assert_array_equal(o.double().cpu().numpy(), o_ref)
    np.testing.assert_array_equal(torch_io.pool_to_f64(t["state_pool"]), pool_ref)


def test_device_errors_skip_work_without_faulting():
    """Bad offsets / slots are caught by the kernels' own checks: error word set, work skipped."""
    p = small("err", [40, 50], 1, 2, 128, "bf16", "f32", "scalar", 64, seed=23, slots=3)
    t = torch_io.prefill_inputs(p, DEV)
    before = t["state_pool"].clone()
    bad_slots = torch.tensor([0, 7], dtype=torch.int32, device=DEV)       # 7 >= num_slots
    kda.prefill(**{**t, "slot_idx": bad_slots}, chunk=64)
    assert kda.get_device_error() == 2
    assert torch.equal(t["state_pool"], before)
    bad_offs = torch.tensor([0, 60, 50], dtype=torch.int32, device=DEV)   # ends before T=90
    kda.prefill(**{**t, "input_row_offsets": bad_offs}, chunk=64)
    assert kda.get_device_error() == 1
    dup = torch.tensor([1, 1], dtype=torch.int32, device=DEV)
    kda.prefill(**{**t, "slot_idx": dup}, chunk=64, checked=True)
    assert kda.get_device_error() == 3
    assert torch.equal(t["state_pool"], before)
    # decode: a slot out of range
    dp = workloads.make_decode_problem("e", num_seqs=2, steps=1, num_k_heads=1, num_v_heads=2,
                                       d=128, qkv_dtype="bf16", state_dtype="f32",
                                       decay_kind="scalar", zero_state=False, seed=3, num_slots=2)
    td = torch_io.decode_inputs(dp, DEV)
    kda.decode_step(td["q"][0], td["k"][0], td["v"][0], td["beta"][0], td["log_decay"][0],
                    torch.tensor([1, 5], dtype=torch.int32, device=DEV), td["state_pool"])
    assert kda.get_device_error() == 2
    assert kda.get_device_error() == 0            # reading clears the word


@pytest.mark.parametrize("decay", ["scalar", "per_channel"])
@pytest.mark.parametrize("state", ["f32", "bf16"])
def test_tensor_core_path_matches_cuda_core_path(decay, state):
    """The tcgen05 path (fp16/bf16 operands) and the fp32 CUDA-core path agree to the
    tolerance, and each matches the oracle, on ragged lengths around the chunk size."""
    p = small("tc-vs-simt", [1, 63, 64, 65, 190, 128], 2, 4, 128, "bf16", state, decay, 64,
              seed=41 if decay == "scalar" else 42, slots=9)
    assert kda.uses_tensor_cores(kda.make_params(num_seqs=6, num_k_heads=2, num_v_heads=4, d=128,
                                                 num_slots=9, total_tokens=p.total_tokens))
    o_tc, s_tc, _ = gpu_prefill(p)
    o_cc, s_cc, _ = gpu_prefill(p, cuda_cores=True)
    o_ref, pool_ref = oracle.run(p)
    tol = TOL["bf16"]
    assert rel_err(o_tc, o_cc) <= tol
    assert rel_err(o_tc, o_ref) <= tol and rel_err(o_cc, o_ref) <= tol
    assert state_err(p, s_tc, pool_ref) <= tol and state_err(p, s_cc, pool_ref) <= tol


def _prefill_keep(p, **kw):
    """One call on fresh device inputs with o pre-filled by a sentinel; returns the device
    error code, o, the pool before the call and the inputs (for a second call)."""
    t = torch_io.prefill_inputs(p, DEV)
    o = torch.full((p.total_tokens, p.num_v_heads, p.d_v), 7.25, dtype=torch.float32, device=DEV)
    before = t["state_pool"].clone()
    kda.prefill(**t, chunk=p.chunk, scale=p.scale, out=o, **kw)
    torch.cuda.synchronize()
    return kda.get_device_error(), o, before, t


@pytest.mark.parametrize("path", ["default", "compact"])
@pytest.mark.parametrize("factor", [1.5, 4.0, 10.0, 33.0])
def test_strong_per_channel_decay_same_pool(path, factor):
    """Per-channel decay 1.5x-33x the kda_prefill workload's (33x: about -5 nats per token,
    some channels -20): a call either matches the oracle, or raises KDA_DEVERR_DECAY_RANGE
    with every slot and o row exactly as before, after which the fp32 CUDA-core path, run on
    that same pool, matches the oracle.  The default two-kernel path covers every one of
    these decays (16-token sub-blocks, exact fp32 pairs where fp16 cannot hold a factor);
    the compact single-kernel path raises the error at 33x."""
    p = small("strong-decay", [200, 77, 130], 1, 2, 128, "bf16", "f32", "per_channel", 64,
              seed=52, slots=5)
    p.g[:] = (p.g * factor).astype(np.float32)
    err, o, before, t = _prefill_keep(p, compact=(path == "compact"))
    o_ref, pool_ref = oracle.run(p)
    if err == 0:
        assert rel_err(o.double().cpu().numpy(), o_ref) <= TOL["bf16"]
        assert state_err(p, torch_io.pool_to_f64(t["state_pool"]), pool_ref) <= TOL["bf16"]
    else:
        assert err == 5
        assert torch.equal(t["state_pool"], before)
        assert bool(torch.all(o == 7.25))
        kda.prefill(**t, chunk=64, cuda_cores=True, out=o)
        torch.cuda.synchronize()
        assert kda.get_device_error() == 0
        assert rel_err(o.double().cpu().numpy(), o_ref) <= TOL["bf16"]
        assert state_err(p, torch_io.pool_to_f64(t["state_pool"]), pool_ref) <= TOL["bf16"]
    assert err == (5 if (path == "compact" and factor > 30) else 0)


@pytest.mark.parametrize("path", ["default", "compact"])
def test_out_of_domain_skips_only_its_sequence_and_head(path):
    """One (sequence, value head) outside the tensor-core path's domain -- a log-decay above
    zero (a gate above one) on the default path, 33x the workload's decay on the compact
    path -- raises KDA_DEVERR_DECAY_RANGE and leaves exactly that pair's slot state and o
    rows as they were; every other pair of the batch matches the oracle."""
    p = small("one-bad", [150, 90, 70], 1, 2, 128, "bf16", "f32", "per_channel", 64, seed=57,
              slots=6)
    rows = slice(int(p.offsets[1]), int(p.offsets[2]))        # sequence 1, value head 0
    if path == "default":
        p.g[rows.start + 40, 0, 5] = 0.5
    else:
        p.g[rows, 0, :] = (p.g[rows, 0, :] * 33.0).astype(np.float32)
    err, o, before, t = _prefill_keep(p, compact=(path == "compact"))
    assert err == 5
    o_ref, pool_ref = oracle.run(p)
    on = o.double().cpu().numpy()
    pool = torch_io.pool_to_f64(t["state_pool"])
    bad_slot = int(p.slot_idx[1])
    assert torch.equal(t["state_pool"][bad_slot, 0], before[bad_slot, 0])
    assert bool(torch.all(o[rows, 0] == 7.25))
    keep = np.ones(on.shape[:2], bool)
    keep[rows, 0] = False
    assert rel_err(on[keep], o_ref[keep]) <= TOL["bf16"]
    for b in range(p.num_seqs):
        for h in range(p.num_v_heads):
            if (b, h) != (1, 0):
                s = int(p.slot_idx[b])
                assert rel_err(pool[s, h], pool_ref[s, h]) <= TOL["bf16"]


@pytest.mark.parametrize("factor", [1.0, 6.0])
def test_scalar_decay_anchored_and_exact_pair_paths(factor):
    """Scalar decay: at the workload's decay the A-matrix decays come from two anchored
    per-token factors; at 6x (about -5 nats per token, beyond their fp32 range) the
    kernel uses exp(G_i - G_j) per pair.  Both match the oracle."""
    p = small("scalar-decay", [200, 64, 33], 2, 2, 128, "bf16", "f32", "scalar", 64, seed=53)
    p.g[:] = (p.g * factor).astype(np.float32)
    check_prefill(p)


@pytest.mark.parametrize("decay", ["scalar", "per_channel"])
@pytest.mark.parametrize("state", ["f32", "bf16"])
def test_compact_and_two_kernel_tensor_core_paths_agree(decay, state):
    """The two-kernel tensor-core path (default) and its single-kernel form
    (compact=True) agree to the tolerance and each matches the oracle, on ragged
    lengths around the chunk size, with GQA and shuffled slots."""
    p = small("split-vs-compact", [1, 63, 64, 65, 190, 128, 257], 2, 4, 128, "bf16", state, decay,
              64, seed=61 if decay == "scalar" else 62, slots=10)
    o_sp, s_sp, _ = gpu_prefill(p)
    o_cp, s_cp, _ = gpu_prefill(p, compact=True)
    o_ref, pool_ref = oracle.run(p)
    tol = TOL["bf16"]
    assert rel_err(o_sp, o_cp) <= tol
    assert rel_err(o_sp, o_ref) <= tol and rel_err(o_cp, o_ref) <= tol
    assert state_err(p, s_sp, pool_ref) <= tol and state_err(p, s_cp, pool_ref) <= tol


@pytest.mark.parametrize("path", ["default", "compact"])
@pytest.mark.parametrize("case", ["over_1024_sequences", "one_long_many_short"])
def test_many_sequences_in_length_order(path, case):
    """The per-sequence scans start in the plan's order of decreasing length (ranked for up to
    1024 sequences, in index order beyond): both branches, with empty sequences, ties and one
    sequence far longer than the rest, match the oracle on every output and state."""
    rng = np.random.Generator(np.random.PCG64(2718))
    if case == "over_1024_sequences":
        lengths = [int(x) for x in rng.integers(0, 24, size=1030)]
    else:
        lengths = [int(x) for x in rng.integers(1, 70, size=299)] + [2500]
        lengths[17] = 0
    p = small(f"order-{case}", lengths, 1, 2, 128, "bf16", "f32", "per_channel", 64, seed=31)
    o, pool, _ = gpu_prefill(p, compact=(path == "compact"))
    o_ref, pool_ref = oracle.run(p, nthreads=8)
    tol = TOL["bf16"]
    eo, es = rel_err(o, o_ref), state_err(p, pool, pool_ref)
    assert eo <= tol and es <= tol, f"{case} ({path}): o err {eo:.3e}, state err {es:.3e}"


def test_per_channel_log_decay_must_be_16_byte_aligned():
    """Per-channel log-decay rows are staged in 16-byte pieces: a log-decay array that is only
    4-byte aligned is refused before any work is enqueued, and the pool is untouched."""
    p = small("g-align", [70, 5], 2, 4, 128, "bf16", "f32", "per_channel", 64, seed=77)
    t = torch_io.prefill_inputs(p, DEV)
    g = t["log_decay"]
    buf = torch.empty(g.numel() + 1, dtype=g.dtype, device=DEV)
    g_off = buf[1:].view(g.shape)
    g_off.copy_(g)
    before = t["state_pool"].clone()
    t["log_decay"] = g_off
    with pytest.raises(kda.KdaError) as e:
        kda.prefill(**t, chunk=p.chunk, scale=p.scale)
    assert e.value.status == 1                  # KDA_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert torch.equal(t["state_pool"], before)

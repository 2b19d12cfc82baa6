"""kda_prefill_fwd_no_alloc: the prefill for callers that cannot allocate device memory.

Such callers (code inside an engine that owns the device memory budget, runtimes that
reserve all memory at start-up) get a prefill whose scratch is a fixed array inside the
library.  This
file is collected last so that a stop-at-first-failure run has already run every other
test; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import gated_delta_rule_deltanet_gb300 as kda
from gated_delta_rule_deltanet_gb300 import _lib
import workloads
from workloads import torch_io

TOL_BF16 = 2e-3


def rel_err(x, ref):
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    assert np.all(np.isfinite(x))
    return float(np.max(np.abs(x - ref)) / max(np.max(np.abs(ref)), 1e-30))


def problem(lengths, seed):
    return workloads.make_problem("no_alloc", num_seqs=len(lengths), lengths=lengths,
                                  num_k_heads=2, num_v_heads=4, d=128, qkv_dtype="bf16",
                                  state_dtype="f32", decay_kind="per_channel", chunk=64,
                                  zero_state=False, num_slots=len(lengths) + 2, seed=seed)


@pytest.mark.gpu
def test_no_alloc_matches_workspace_prefill_on_two_calls():
    """Calls in a row (different batches, so stale scratch from the previous call is in
    place for the next), on both prefill paths, each equal to the workspace entry point."""
    for lengths, seed, cc in [([100, 37, 64], 31, False), ([200, 1, 129, 65], 32, False),
                              ([100, 37, 64], 33, True), ([200, 1, 129, 65], 34, True)]:
        p = problem(lengths, seed)
        t = torch_io.prefill_inputs(p, "cuda:0")
        pool_ref = t["state_pool"].clone()
        o_ref = kda.prefill(**{**t, "state_pool": pool_ref}, chunk=p.chunk, cuda_cores=cc)
        out = torch.empty_like(o_ref)
        kda.prefill_no_alloc(**t, chunk=p.chunk, out=out, cuda_cores=cc)
        torch.cuda.synchronize()
        assert kda.get_device_error() == 0
        assert rel_err(out.cpu().numpy(), o_ref.cpu().numpy()) <= TOL_BF16
        assert rel_err(t["state_pool"].cpu().numpy(), pool_ref.cpu().numpy()) <= TOL_BF16


@pytest.mark.gpu
def test_no_alloc_uses_the_single_kernel_form_when_records_do_not_fit():
    """6144 tokens x 16 value heads need about 92 MB of chunk records on the two-kernel
    tensor-core path, more than the scratch holds: the no-alloc entry runs the
    single-kernel form instead and matches the regular call."""
    p = workloads.make_problem("no_alloc_big", num_seqs=3, lengths=[2048, 2048, 2048],
                               num_k_heads=16, num_v_heads=16, d=128, qkv_dtype="bf16",
                               state_dtype="f32", decay_kind="scalar", chunk=64, zero_state=False,
                               num_slots=3, seed=35)
    params = kda.make_params(num_seqs=3, num_k_heads=16, num_v_heads=16, d=128, num_slots=3,
                             total_tokens=6144, per_channel=False)
    assert kda.workspace_size(params) > _lib.KDA_NO_ALLOC_SCRATCH_BYTES
    assert kda.no_alloc_form(params) == "compact"
    t = torch_io.prefill_inputs(p, "cuda:0")
    pool_ref = t["state_pool"].clone()
    o_ref = kda.prefill(**{**t, "state_pool": pool_ref}, chunk=64)
    out = torch.empty_like(o_ref)
    kda.prefill_no_alloc(**t, chunk=64, out=out)
    torch.cuda.synchronize()
    assert kda.get_device_error() == 0
    assert rel_err(out.cpu().numpy(), o_ref.cpu().numpy()) <= TOL_BF16
    assert rel_err(t["state_pool"].cpu().numpy(), pool_ref.cpu().numpy()) <= TOL_BF16


def test_no_alloc_rejects_problems_beyond_its_scratch():
    """A problem needing more scratch than the built-in array is refused on the host,
    before anything is enqueued (so this runs without a GPU too)."""
    lib = _lib.load()
    big = kda.make_params(num_seqs=1, num_k_heads=16, num_v_heads=16, d=128, num_slots=1,
                          total_tokens=16384, chunk=64, cuda_cores=True)
    assert kda.workspace_size(big) > _lib.KDA_NO_ALLOC_SCRATCH_BYTES
    P = ctypes.c_void_p
    a = P(1 << 20)
    st = lib.kda_prefill_fwd_no_alloc(ctypes.byref(big), a, a, a, a, a, a, a, a, a, None)
    assert st == _lib.KDA_ERR_WORKSPACE
    assert kda.no_alloc_form(big) == "rejected"
    small = kda.make_params(num_seqs=1, num_k_heads=2, num_v_heads=4, d=128, num_slots=1,
                            total_tokens=300, chunk=64)
    assert kda.workspace_size(small) <= _lib.KDA_NO_ALLOC_SCRATCH_BYTES
    assert kda.no_alloc_form(small) == "two_kernel"
    small_cc = kda.make_params(num_seqs=1, num_k_heads=2, num_v_heads=4, d=128, num_slots=1,
                               total_tokens=300, chunk=64, cuda_cores=True)
    assert kda.no_alloc_form(small_cc) == "cuda_cores"

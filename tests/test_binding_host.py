"""The Python binding on CPU: every compute entry point refuses host tensors before anything
else happens (there is no CPU path to fall back to), and the library it loads is the in-tree
build."""
import os

import pytest
import torch

import gated_delta_rule_deltanet_gb300 as kda
from gated_delta_rule_deltanet_gb300 import _lib, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def host_inputs(T=8, B=2, HK=1, HV=2, D=16, slots=3):
    bf = torch.bfloat16
    return dict(q=torch.zeros(T, HK, D, dtype=bf), k=torch.zeros(T, HK, D, dtype=bf),
                v=torch.zeros(T, HV, D, dtype=bf), beta=torch.zeros(T, HV),
                log_decay=torch.zeros(T, HV),
                input_row_offsets=torch.tensor([0, T // 2, T], dtype=torch.int32),
                slot_idx=torch.arange(B, dtype=torch.int32),
                state_pool=torch.zeros(slots, HV, D, D))


CALLS = {
    "prefill": lambda t: kda.prefill(**t),
    "prefill_no_alloc": lambda t: kda.prefill_no_alloc(**t, out=torch.empty(8, 2, 16)),
    "prefill_bwd": lambda t: kda.prefill_bwd(**t, d_o=torch.zeros(8, 2, 16)),
    "gdp_prefill": lambda t: kda.gdp_prefill(**t),
    "decode_step": lambda t: kda.decode_step(
        t["q"][:2], t["k"][:2], t["v"][:2], t["beta"][:2], t["log_decay"][:2], t["slot_idx"],
        t["state_pool"]),
    "gdp_decode_step": lambda t: kda.gdp_decode_step(
        t["q"][:2], t["k"][:2], t["v"][:2], t["beta"][:2], t["log_decay"][:2], t["slot_idx"],
        t["state_pool"]),
    "verify_window": lambda t: kda.verify_window(
        t["q"], t["k"], t["v"], t["beta"], t["log_decay"], t["slot_idx"], t["state_pool"],
        window=4),
    "fold_accepted": lambda t: kda.fold_accepted(
        torch.zeros(64), torch.zeros(2, dtype=torch.int32), t["slot_idx"], t["state_pool"],
        window=4),
    "conv_gates": lambda t: kda.conv_gates(
        torch.zeros(8, 64, dtype=torch.bfloat16), torch.zeros(64, 4), torch.zeros(8, 2),
        torch.zeros(8, 2), num_k_heads=1, num_v_heads=2, d=16),
}


@pytest.mark.parametrize("name", sorted(CALLS))
def test_host_tensors_are_refused(name):
    with pytest.raises(ValueError, match="CUDA tensors"):
        CALLS[name](host_inputs())


def test_library_is_the_in_tree_build():
    lib = _lib.load()
    path = os.path.realpath(lib._name)
    assert path == os.path.realpath(build.LIB)
    assert os.path.commonpath([path, os.path.realpath(ROOT)]) == os.path.realpath(ROOT)

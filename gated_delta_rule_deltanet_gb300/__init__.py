"""GB300-native forward pass of the gated delta rule (KDA / Gated DeltaNet / DeltaNet).

The computation lives in libkda.so (hand-written CUDA for sm_103a, C ABI in
include/kda.h).  This package only builds it and marshals torch tensors into
it:

    prefill(q, k, v, beta, log_decay, input_row_offsets, slot_idx, state_pool, chunk=64)
    decode_step(q, k, v, beta, log_decay, slot_idx, state_pool)
    gdp_prefill / gdp_decode_step   (Gated DeltaProduct: n_h transitions per token)
    prefill_bwd(...)                (the backward pass of prefill)
    conv_gates(...)                 (the front end: short conv + SiLU, gate activations)

There is no CPU or eager fallback: if the library is missing, calls raise.
"""
from .kda import (decode_step, get_device_error, make_params, prefill,  # noqa: F401
                  prefill_no_alloc, no_alloc_form, set_stage_events, uses_tensor_cores,
                  workspace_size, verify_window, fold_accepted, ring_record_elems,
                  gdp_prefill, gdp_decode_step, prefill_bwd, conv_gates)
from ._lib import KdaError, KdaParams, load  # noqa: F401

__all__ = ["prefill", "decode_step", "workspace_size", "get_device_error", "make_params",
           "set_stage_events", "prefill_no_alloc", "no_alloc_form", "uses_tensor_cores", "verify_window", "fold_accepted", "ring_record_elems", "gdp_prefill", "gdp_decode_step", "prefill_bwd", "conv_gates", "KdaError", "KdaParams", "load"]

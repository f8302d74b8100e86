"""The decode step that allocates nothing, checked against the regular step and
against the oracle.

Callers that may not allocate device memory while they decode -- because an
outside allocator or a fixed budget owns the device memory, or because the
decoding thread must stay off the synchronising cudaMalloc/cudaFree paths --
use mk_decode_step_noalloc, whose scratch is a fixed array inside the library.
These tests call it through the C ABI on the same inputs as mk_decode_step,
two calls in a row, and hold both results to the parity tests' tolerance:
the no-allocation logits against the regular step's and against the oracle
teacher-forced on the same tokens.  The shapes cover batch 1 (small and
Llama-1B), a small MoE (its routing lives in the fixed array too), 5
sequences on the batched variant (h as tensor-core fragments) and 8 on the
wide tcgen05 variant (its operand buffers and attention arrival counters
live in the fixed array too).  This file is collected last so that a run
stopping at the first failure has already run every other test.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import synth
from decode_megakernel_sm_gb300 import _lib as L
from tests.harness import Run

pytestmark = pytest.mark.gpu

CASES = {
    "tiny": synth.CONFIGS["tiny"],
    "llama1b_1k": synth.CONFIGS["llama1b_1k"],
    # 16 experts, top-4, a shared expert, ragged widths
    "moe_small": synth.custom(n_layers=3, hidden=2048, n_q_heads=8, n_kv_heads=2, head_dim=128,
                              ffn=0, vocab=3001, tied=False, n_experts=16, top_k=4,
                              expert_ffn=200, shared_ffn=500, rope_theta=5e5, prefill=(70, 70),
                              steps=4),
    # five sequences, ragged lengths, the batched variant's split MLP (h as
    # fragments), which the descriptor asks for
    "batch5": synth.custom(n_layers=2, hidden=2048, n_q_heads=8, n_kv_heads=2, head_dim=64,
                           ffn=2048, vocab=5000, batch=5, prefill=(0, 300), steps=4,
                           rope_theta=5e5, batched_variant=1),
    # eight sequences: the wide tcgen05 variant
    "batch8": synth.custom(n_layers=2, hidden=2048, n_q_heads=8, n_kv_heads=2, head_dim=64,
                           ffn=2048, vocab=5000, batch=8, prefill=(0, 300), steps=4,
                           rope_theta=5e5),
}


def _noalloc(r, logits, am, status):
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = L.lib().mk_decode_step_noalloc(r.dec.h, r.d_tok.data_ptr(), r.d_pos.data_ptr(),
                                        logits.data_ptr(), am.data_ptr(), status.data_ptr(),
                                        stream)
    assert rc == L.MK_OK, L.mk_status_string(rc)
    torch.cuda.synchronize()
    assert int(status.item()) == L.MK_OK
    return logits.cpu().numpy().astype(np.float64), am.cpu().numpy()


def _oracle(r):
    if r.cfg.get("n_experts", 0) > 0:  # routing near-ties follow the regular step's routes
        return r._oracle_moe_step()
    lo, ao, _, _ = r.om.step(r.ko, r.vo, r.tokens, r.pos)
    return lo, ao


@pytest.mark.parametrize("name", list(CASES))
def test_noalloc_step_matches_regular_step_and_oracle_on_two_calls(name):
    r = Run(CASES[name], seed=13)
    try:
        V = r.cfg["vocab"]
        logits = torch.full((r.B, V), float("nan"), dtype=torch.float32, device="cuda")
        am = torch.full((r.B,), -1, dtype=torch.int32, device="cuda")
        status = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
        for _ in range(2):
            lg_ref, am_ref = r.gpu_step("mega")       # the existing entry point
            lo, ao = _oracle(r)                        # same tokens and positions
            r.check(lg_ref, am_ref, lo, ao)
            lg, a = _noalloc(r, logits, am, status)   # same inputs, same cache row P
            r.check(lg, a, lg_ref, am_ref)            # against the regular step
            r.check(lg, a, lo, ao)                    # and against the oracle
            r.tokens = [int(x) for x in am_ref]
            r.pos = [p + 1 for p in r.pos]
    finally:
        r.close()


def test_noalloc_rejects_schedules_beyond_its_array():
    # 400 layers of 4 query heads, each head split into 60 slices at 2048
    # positions: about 26 MB of split-KV partials, more than the 16 MiB
    # array holds -- refused before any launch
    cfg = synth.custom(n_layers=400, n_q_heads=4, n_kv_heads=2, ffn=256, vocab=256,
                       prefill=(8, 8), steps=2040)
    r = Run(cfg, seed=1)
    try:
        logits = torch.empty((1, 256), dtype=torch.float32, device="cuda")
        am = torch.empty(1, dtype=torch.int32, device="cuda")
        stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
        rc = L.lib().mk_decode_step_noalloc(r.dec.h, r.d_tok.data_ptr(), r.d_pos.data_ptr(),
                                            logits.data_ptr(), am.data_ptr(), None, stream)
        assert rc == L.MK_ERR_SCRATCH
        assert "16 MiB" in L.mk_status_string(rc)
    finally:
        r.close()

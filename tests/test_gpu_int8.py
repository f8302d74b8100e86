"""int8 weight streaming (mk_create_ex with MK_WEIGHTS_INT8): the device row
quantiser against the oracle's, bit for bit, and the int8 decode path against
the oracle's int8 decoder (each side quantises the same bf16 weights itself)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from decode_megakernel_sm_gb300 import (MK_ERR_UNSUPPORTED, Decoder, MkError,
                                        mk_quantize_rows_int8)
from tests.harness import Run

pytestmark = pytest.mark.gpu


def _device_quantise(w):
    rows, cols = w.shape
    q = torch.empty((rows, cols), dtype=torch.int8, device="cuda")
    s = torch.empty(rows, dtype=torch.float32, device="cuda")
    mk_quantize_rows_int8(w.data_ptr(), rows, cols, q.data_ptr(), s.data_ptr())
    torch.cuda.synchronize()
    return q.cpu().numpy(), s.cpu().numpy()


@pytest.mark.parametrize("rows,cols", [(37, 300), (64, 2048), (9, 8192)])
def test_quantiser_bit_exact_against_oracle(rows, cols):
    g = torch.Generator(device="cuda").manual_seed(rows * cols)
    w = (torch.randn((rows, cols), generator=g, device="cuda") * 0.02).to(torch.bfloat16)
    w[1] = 0  # a zero row
    # a row of exact ties: s = 1 (maximum 127), values k + 0.5
    ties = torch.zeros(cols, device="cuda")
    ties[:254] = torch.arange(-127, 127, device="cuda", dtype=torch.float32) + 0.5
    ties[-1] = 127.0
    w[2] = ties.to(torch.bfloat16)
    w[3] *= 1e4  # large magnitudes
    q, s = _device_quantise(w)
    qo, so = oracle.quantize_rows_int8(oracle._bits(w.cpu()))
    assert np.array_equal(s.view(np.uint32), so.view(np.uint32))
    assert np.array_equal(q, qo)


def _cfg(**kw):
    base = dict(n_layers=2, hidden=2048, n_q_heads=32, n_kv_heads=8, head_dim=64, ffn=2048,
                vocab=5000, rope_theta=5e5, prefill=(300, 300), steps=4)
    base.update(kw)
    return synth.custom(**base)


def run_steps(cfg, steps, seed, **kw):
    r = Run(cfg, seed, int8=True, **kw)
    try:
        for _ in range(steps):
            r.step()
    finally:
        r.close()


def test_int8_decode_against_oracle():
    r = Run(_cfg(), 71, int8=True)
    try:
        info = r.dec.info()
        assert info["n_stages"] == 4  # the int8 default ring depth
        assert info["stage_bytes"] == 32768
        for _ in range(3):
            r.step()
    finally:
        r.close()


def test_int8_untied_head_and_ragged_ffn():
    # an untied LM head, an FFN of 3008 columns (ragged MLP slices), a vocab
    # that leaves a ragged LM-head tail
    run_steps(_cfg(tied=False, ffn=3008, vocab=4099), 3, seed=73)


def test_int8_llama1b():
    run_steps(synth.CONFIGS["llama1b_1k"], 2, seed=75)


def test_int8_multistep():
    r = Run(_cfg(), seed=77, int8=True)
    try:
        r.multi_step(4)
    finally:
        r.close()


@pytest.mark.parametrize("mode", ["stream", "graph", "pdl"])
def test_int8_ablation_modes(mode):
    # the same opcode bodies, one launch per phase
    r = Run(_cfg(n_layers=1), seed=81, int8=True)
    try:
        r.step(mode)
        r.step(mode)
    finally:
        r.close()


def test_int8_paged_cache():
    run_steps(_cfg(), 2, seed=79, paged=64)


@pytest.mark.parametrize("over", [dict(batch=8, prefill=(0, 300)),
                                  dict(ffn=0, tied=False, n_experts=16, top_k=4, expert_ffn=200,
                                       shared_ffn=0),
                                  dict(ffn=2056)])
def test_int8_unsupported_shapes_are_refused(over):
    cfg = synth.with_cache(_cfg(**over))
    W = synth.make_weights(cfg, 0, "cuda")
    ks, vs = synth.make_kv(cfg, synth.make_lengths(cfg, 0), 0, "cuda")
    with pytest.raises(MkError) as e:
        Decoder(cfg, W, ks, vs, weight_format="int8")
    assert e.value.status == MK_ERR_UNSUPPORTED

"""The wide-batch variant (2 .. 32 sequences, every contraction on tcgen05 with
the accumulator in tensor memory) against the CPU oracle, through the C ABI.

The acceptance is the decode contract of tests/harness.py at every step and
for every sequence: logits within 2e-2 of the oracle's std, the argmax exact
wherever the oracle's top-2 margin exceeds 5e-2, the GPU argmax the first
maximum of its own logits, and the appended K/V rows within one bf16 ulp.
The shapes cover batches that fill 8-sequence groups exactly (16, 32) and
ones that do not (2, 5, 9, 13: zero operand rows up to the next multiple of 8),
one attention item per (sequence, kv head) (pairs at least as many as the
SMs) and split-KV slices merged by the last arriver (fewer pairs), cache
lengths of 0..2 rows (slices with no cached rows),
an FFN with an odd number of 64-column chunks and a vocabulary that is not a
multiple of 8 (the LM head's last instruction reads zero-padded rows), ring
stages of 32, 48 and 64 KB (the default; 16 KB is refused), several steps per launch, the multi-launch ablation,
a launch that times out on a dropped instruction and the steps after it,
and the full Llama-1B shape at 32 sequences.
"""
import numpy as np
import pytest

import synth
from decode_megakernel_sm_gb300 import MK_ERR_TIMEOUT, MK_ERR_UNSUPPORTED, MkError
from tests.harness import Run

pytestmark = pytest.mark.gpu


def small(batch, **kw):
    base = dict(n_layers=2, hidden=2048, n_q_heads=8, n_kv_heads=2, head_dim=64, ffn=2048,
                vocab=5000, batch=batch, prefill=(0, 300), steps=4, rope_theta=5e5)
    base.update(kw)
    return synth.custom(**base)


def run_steps(cfg, steps, seed=0, **kw):
    r = Run(cfg, seed, **kw)
    try:
        for _ in range(steps):
            r.step()
        return r.worst
    finally:
        r.close()


@pytest.mark.parametrize("batch", [2, 5, 9, 16, 32])
def test_wide_parity(batch):
    worst = run_steps(small(batch), 3, seed=batch)
    print(f"batch {batch} worst max|dlogit|/std = {worst:.2e}")


def test_wide_short_sequences():
    # cache lengths 0..2 with 4 slices per (sequence, kv head): most attention
    # items have no cached rows (only the last slice's row P)
    worst = run_steps(small(9, prefill=(0, 2)), 3, seed=11)
    print(f"batch 9, lengths 0..2 worst max|dlogit|/std = {worst:.2e}")


def test_wide_whole_sequence_attention_items():
    # 24 sequences x 8 kv heads: one attention item per pair, which writes
    # its output straight into the O-projection operand
    worst = run_steps(small(24, n_q_heads=32, n_kv_heads=8), 3, seed=24)
    print(f"batch 24, 8 kv heads worst max|dlogit|/std = {worst:.2e}")


def test_wide_ragged_ffn_vocab_and_batch():
    # 17 FFN chunks, a vocabulary of 5001 rows, 13 sequences (Bp = 16)
    cfg = small(13, ffn=1088, vocab=5001, n_layers=3, prefill=(5, 400))
    run_steps(cfg, 3, seed=7)


def test_wide_default_stage_size():
    # 64 KB stages unless the caller asks otherwise
    r = Run(small(16), seed=5)
    try:
        info = r.dec.info()
        assert info["stage_bytes"] == 65536 and info["n_stages"] >= 2
    finally:
        r.close()


@pytest.mark.parametrize("sb", [32768, 49152])
def test_wide_stage_sizes(sb):
    run_steps(small(24), 2, seed=sb % 97, stage_bytes=sb)


def test_wide_refuses_16k_stages():
    # a stage must hold a 128-row weight chunk (16 KB) and its operand chunk
    r = Run(small(16), seed=1)
    try:
        with pytest.raises(MkError) as e:
            r.dec.set_stage_bytes(16384)
        assert e.value.status == MK_ERR_UNSUPPORTED
        r.step()  # the handle keeps its ring
    finally:
        r.close()


def test_wide_missing_producer_times_out_and_recovers():
    # SM 0's first instruction (the layer-0 norm of sequence 0) never signals:
    # every QKV instruction's wait runs out, the launch ends with a timeout
    # status (its tensor memory freed), and the rebuilt schedule decodes again
    r = Run(small(16), seed=3)
    try:
        r.dec.set_wait_timeout(50_000_000)  # 50 ms
        r.dec.drop_instruction(0, 0)
        r.dec.step(r.d_tok, r.d_pos, r.d_logits, r.d_am)
        assert r.dec.sync_status() == MK_ERR_TIMEOUT
        r.dec.build_schedule(r.B, r.max_ctx)  # restores the dropped instruction
        r.step()
        r.step()
    finally:
        r.close()


def test_wide_multistep():
    r = Run(small(16, n_layers=3, steps=8), seed=5)
    try:
        r.multi_step(5)
        r.step()
    finally:
        r.close()


def test_wide_ablation_matches_megakernel():
    r = Run(small(16, steps=6), seed=8)
    try:
        for mode in ("stream", "pdl"):
            pos0, tok0 = list(r.pos), list(r.tokens)
            lg_m, am_m = r.gpu_step("mega")
            lg_a, am_a = r.gpu_step(mode)
            assert np.array_equal(am_m, am_a), mode
            assert np.abs(lg_m - lg_a).max() <= 1e-3 * lg_m.std(), mode
            r.pos, r.tokens = pos0, tok0
            r.step(mode)
    finally:
        r.close()


def test_wide_llama1b_batch32_full_config():
    # 16 layers, vocab 128256, 32 sequences with cache lengths U[512, 2048]
    cfg = dict(synth.CONFIGS["llama1b_b8"], batch=32)
    worst = run_steps(cfg, 2, seed=1)
    print(f"llama1b batch 32 worst max|dlogit|/std = {worst:.2e}")

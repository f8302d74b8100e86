"""Race stress (mk_set_race_stress): random delays before every instruction on
the producer and the consumers, and a random queue-to-CTA permutation.  Every
wait, fence and signal stays, so the results must still meet the oracle:
a missing ordering would surface here as wrong logits or cache rows."""
import pytest

import synth
from tests.harness import Run

pytestmark = pytest.mark.gpu


def _ragged():
    return synth.custom(n_layers=3, n_q_heads=6, n_kv_heads=3, ffn=1000, vocab=999,
                        prefill=(300, 300), steps=6)


@pytest.mark.parametrize("delay,seed,perm", [(3000, 1, True), (20000, 2, False), (0, 3, True)])
def test_stress_small_shape(delay, seed, perm):
    r = Run(_ragged(), seed=91 + seed, stress=(delay, seed, perm))
    try:
        r.step()
        r.multi_step(3)
    finally:
        r.close()


def test_stress_llama1b_tagged_residual_hops():
    # the split MLP at batch 1: tagged residual words and relaxed signals
    r = Run(synth.CONFIGS["llama1b_1k"], seed=95, stress=(5000, 5, True))
    try:
        r.step()
        r.multi_step(2)
    finally:
        r.close()


def test_stress_batched_and_moe():
    b8 = synth.custom(n_layers=2, hidden=2048, n_q_heads=8, n_kv_heads=2, head_dim=64, ffn=2048,
                      vocab=5000, batch=8, prefill=(0, 300), steps=3, rope_theta=5e5)
    moe = synth.custom(n_layers=3, hidden=2048, n_q_heads=8, n_kv_heads=2, head_dim=128, ffn=0,
                       vocab=3001, tied=False, n_experts=16, top_k=4, expert_ffn=200,
                       shared_ffn=500, rope_theta=5e5, prefill=(70, 70), steps=3)
    for cfg, seed in ((b8, 96), (moe, 97)):
        r = Run(cfg, seed=seed, stress=(4000, seed, True))
        try:
            r.step()
            r.step()
        finally:
            r.close()


def test_stress_int8_paged():
    cfg = synth.custom(n_layers=2, hidden=2048, n_q_heads=32, n_kv_heads=8, head_dim=64,
                       ffn=2048, vocab=5000, rope_theta=5e5, prefill=(300, 300), steps=3)
    r = Run(cfg, seed=98, int8=True, paged=64, stress=(4000, 8, True))
    try:
        r.step()
        r.step()
    finally:
        r.close()


@pytest.mark.parametrize("variant", [0, 1])
def test_stress_batch5_split_attention(variant):
    # 5 sequences: the wide variant, whose attention runs 4 split-KV slices per
    # (sequence, kv head) merged by the last arriving item (0), or the batched
    # mma.sync variant (1); one step, then a multi-step launch
    cfg = synth.custom(n_layers=2, hidden=2048, n_q_heads=8, n_kv_heads=2, head_dim=64, ffn=2048,
                       vocab=5000, batch=5, prefill=(0, 300), steps=5, rope_theta=5e5,
                       batched_variant=variant)
    r = Run(cfg, seed=99 + variant, stress=(4000, 9 + variant, True))
    try:
        r.step()
        r.multi_step(2)
    finally:
        r.close()

"""Paged KV cache (mk_set_kv_pages): the cache rows live in blocks of a pool at
shuffled block ids, addressed through a block table.  Same oracle checks as
the contiguous cache: logits, argmax, every appended K/V row."""
import pytest
import torch

import synth
from decode_megakernel_sm_gb300 import MK_ERR_INVALID_ARG
from tests.harness import Run

pytestmark = pytest.mark.gpu


def _ragged(**kw):
    return synth.custom(n_layers=3, n_q_heads=6, n_kv_heads=3, ffn=1000, vocab=999,
                        prefill=(300, 300), steps=4, **kw)


def run_steps(cfg, steps, seed, **kw):
    r = Run(cfg, seed, **kw)
    try:
        for _ in range(steps):
            r.step()
    finally:
        r.close()


@pytest.mark.parametrize("block", [16, 64, 4096])
def test_paged_ragged_shape(block):
    # blocks smaller than a ring stage half (16, 64 rows), and one block
    # holding the whole sequence
    run_steps(_ragged(), 3, seed=51, paged=block)


def test_paged_batch8_ragged_lengths():
    cfg = synth.custom(n_layers=2, hidden=2048, n_q_heads=8, n_kv_heads=2, head_dim=64, ffn=3000,
                       vocab=5000, batch=8, prefill=(0, 300), steps=3, rope_theta=5e5)
    run_steps(cfg, 3, seed=53, paged=16)


def test_paged_llama1b():
    run_steps(synth.CONFIGS["llama1b_1k"], 2, seed=55, paged=16)


def test_paged_moe_small():
    cfg = synth.custom(n_layers=3, hidden=2048, n_q_heads=8, n_kv_heads=2, head_dim=128, ffn=0,
                       vocab=3001, tied=False, n_experts=16, top_k=4, expert_ffn=200,
                       shared_ffn=500, rope_theta=5e5, prefill=(70, 70), steps=4)
    run_steps(cfg, 3, seed=57, paged=32)


def test_paged_multistep():
    r = Run(_ragged(), seed=59, paged=32)
    try:
        r.multi_step(4)
    finally:
        r.close()


def test_paged_table_rewritten_between_steps():
    # move every block of sequence 0 to a spare id (copying its rows), as an
    # allocator compacting its pool would; the next steps read and append
    # through the new table
    r = Run(_ragged(), seed=61, paged=64)
    try:
        r.step()
        used = set(int(x) for x in r.table.flatten())
        spare = [i for i in range(r.pk[0].shape[0]) if i not in used]
        for j in range(min(len(spare), r.table.shape[1])):
            old, new = int(r.table[0, j]), spare[j]
            for pool in r.pk + r.pv:
                pool[new] = pool[old]
            r.table[0, j] = new
        torch.cuda.synchronize()
        r.step()
        r.step()
    finally:
        r.close()


def test_paged_block_outside_pool_is_an_error():
    r = Run(_ragged(), seed=63, paged=16)
    try:
        P = r.pos[0]
        good = int(r.table[0, P // 16])
        r.table[0, P // 16] = r.pk[0].shape[0]  # one past the pool
        r.d_tok.copy_(torch.tensor(r.tokens, dtype=torch.int32))
        r.d_pos.copy_(torch.tensor(r.pos, dtype=torch.int32))
        r.dec.step(r.d_tok, r.d_pos, r.d_logits, r.d_am)
        assert r.dec.sync_status() == MK_ERR_INVALID_ARG
        r.table[0, P // 16] = good
        torch.cuda.synchronize()
        r.step()  # the handle recovers
    finally:
        r.close()


def test_llama1b_32k_context():
    # long context: a 32K cache, contiguous and paged (256-row blocks)
    run_steps(synth.CONFIGS["llama1b_32k"], 2, seed=65)
    run_steps(synth.CONFIGS["llama1b_32k"], 2, seed=66, paged=256)

"""GPU parity of the megakernel against the CPU oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import synth
from decode_megakernel_sm_gb300 import MK_ERR_INVALID_ARG, MK_ERR_TIMEOUT, MK_ERR_UNSUPPORTED, MK_OK, MkError
from tests.harness import Run

pytestmark = pytest.mark.gpu


def run_steps(cfg, steps, seed=0, **kw):
    r = Run(cfg, seed, **kw)
    try:
        for _ in range(steps):
            r.step()
        return r.worst
    finally:
        r.close()


def test_tiny_parity_8_steps():
    run_steps(synth.CONFIGS["tiny"], 8)


def test_ragged_small_shape_parity():
    # 3 kv heads x 2 q heads, FFN and vocab not multiples of anything, 3 layers
    cfg = synth.custom(n_layers=3, n_q_heads=6, n_kv_heads=3, ffn=1000, vocab=999,
                       prefill=(37, 37), steps=4)
    run_steps(cfg, 4, seed=3)


def test_batch1_default_stage_size():
    # one bf16 sequence: 64 KB stages unless the caller asks otherwise
    r = Run(synth.CONFIGS["tiny"], seed=5)
    try:
        info = r.dec.info()
        assert info["stage_bytes"] == 65536 and info["n_stages"] >= 2
        r.step()
    finally:
        r.close()


@pytest.mark.parametrize("sb", [16384, 32768, 49152])
def test_ring_stage_sizes(sb):
    # the same ragged shape with every stage size besides the 64 KB default:
    # fewer rows, cache positions and down rows per stage, results unchanged
    cfg = synth.custom(n_layers=3, n_q_heads=6, n_kv_heads=3, ffn=1000, vocab=999,
                       prefill=(300, 300), steps=3)
    run_steps(cfg, 3, seed=9, stage_bytes=sb)


@pytest.mark.parametrize("mask,early", [(63, 0), (63, 16384), (24, 1 << 20)])
def test_hold_policies(mask, early):
    # every op held with no early stage or with one, and the default ops
    # with every stage early: the producer's extra waits change no result
    cfg = synth.custom(n_layers=3, n_q_heads=6, n_kv_heads=3, ffn=1000, vocab=999,
                       prefill=(300, 300), steps=3)
    run_steps(cfg, 3, seed=11, hold=(mask, early))


def test_shallow_ring_and_staggered_pollers():
    # two ring stages, and four warps polling each counter 100 ns apart:
    # neither changes a result
    cfg = synth.custom(n_layers=3, n_q_heads=6, n_kv_heads=3, ffn=1000, vocab=999,
                       prefill=(300, 300), steps=3)
    r = Run(cfg, seed=13)
    try:
        r.dec.set_ring_depth(2)
        r.dec.set_poll_policy(4, 100)
        for _ in range(3):
            r.step()
        for bad in ((0, 0), (8, 0), (1, 200000)):
            with pytest.raises(MkError):
                r.dec.set_poll_policy(*bad)
        with pytest.raises(MkError):
            r.dec.set_ring_depth(1)
        r.step()  # the previous settings are kept
    finally:
        r.close()


def test_batched_split_mlp_held():
    # the batched down units gate their weight halves on the hold as well
    run_steps(_bsplit_cfg(8), 3, seed=23, hold=(63, 0))


def test_staged_partials_many_slices():
    # heads of 128 dims at 2000 positions: 31 split-KV slices, so the
    # O-projection copies its partials into a ring stage before merging them
    # (with 16 KiB stages they fill the stage to within 16 bytes)
    cfg = synth.custom(n_layers=2, hidden=2048, n_q_heads=8, n_kv_heads=2, head_dim=128,
                       ffn=2048, vocab=3000, prefill=(2000, 2000), steps=3, rope_theta=5e5)
    run_steps(cfg, 3, seed=41)
    run_steps(cfg, 2, seed=42, stage_bytes=16384)


def test_llama1b_32k_stages():
    # the bench shape with half-size stages (a deeper ring of 8-row stages)
    r = Run(synth.CONFIGS["llama1b_1k"], seed=3, stage_bytes=32768)
    try:
        r.step()
        r.step()
    finally:
        r.close()


def test_position_zero_attends_to_itself_only():
    run_steps(synth.custom(prefill=(0, 0), steps=3), 3, seed=5)


def test_last_position_below_max_ctx():
    cfg = synth.custom(prefill=(40, 40), steps=1)
    r = Run(cfg, seed=6, max_ctx=41)  # P = 40 = max_ctx - 1
    try:
        r.step()
        # P = max_ctx is rejected on the device, and the handle recovers
        r.d_pos.fill_(41)
        r.dec.step(r.d_tok, r.d_pos, r.d_logits, r.d_am)
        assert r.dec.sync_status() == MK_ERR_INVALID_ARG
        r.pos = [40]
        r.step()
    finally:
        r.close()


def test_batch8_variant_ragged_lengths():
    cfg = synth.custom(n_layers=2, hidden=2048, n_q_heads=8, n_kv_heads=2, head_dim=64, ffn=3000,
                       vocab=5000, batch=8, prefill=(0, 300), steps=3, rope_theta=5e5)
    run_steps(cfg, 3, seed=7)


def _bsplit_cfg(batch):
    # the batched (mma.sync) variant, which the descriptor asks for: this
    # shape would run on the wide-batch variant by default
    return synth.custom(n_layers=2, hidden=2048, n_q_heads=8, n_kv_heads=2, head_dim=64,
                        ffn=2048, vocab=5000, batch=batch, prefill=(0, 300), steps=3,
                        rope_theta=5e5, batched_variant=1)


@pytest.mark.parametrize("batch", [7, 5, 8])
def test_batched_split_mlp(batch):
    # batch 2..8 with an FFN of whole 512-column chunks on the batched
    # variant: gate/up slices write h as
    # tensor-core fragments, 16-row down units stream them next to their
    # weights (padded rows past the batch)
    run_steps(_bsplit_cfg(batch), 3, seed=17)


@pytest.mark.parametrize("sb", [49152, 65536])
def test_batched_split_mlp_stage_sizes(sb):
    # 48 KiB: one weight unit + its fragments per stage (8 KB idle per
    # half); 64 KiB: two of each
    run_steps(_bsplit_cfg(7), 3, seed=19, stage_bytes=sb)


def test_batched_default_stage_size():
    # the batched variant keeps 32 KB stages by default
    r = Run(_bsplit_cfg(5), seed=23)
    try:
        assert r.dec.info()["stage_bytes"] == 32768
        r.step()
    finally:
        r.close()


def test_batched_split_mlp_16k_stages():
    # one 16 KB down unit per stage
    run_steps(_bsplit_cfg(7), 3, seed=2, stage_bytes=16384)


def test_batched_split_mlp_ragged_ffn_chunks():
    # FFN of 3 chunks of 512 and a short vocabulary: down runs that start and
    # end inside chunks, two-chunk runs, and every SM's share under one chunk
    cfg = synth.custom(n_layers=2, hidden=2048, n_q_heads=8, n_kv_heads=2, head_dim=64,
                       ffn=1536, vocab=3000, batch=6, prefill=(5, 400), steps=3, rope_theta=5e5,
                       batched_variant=1)
    run_steps(cfg, 3, seed=29)


def test_llama1b_1k_parity():
    cfg = synth.CONFIGS["llama1b_1k"]
    worst = run_steps(cfg, 3, seed=0)
    print(f"llama1b_1k worst max|dlogit|/std = {worst:.2e}")


def test_llama1b_8k_parity():
    run_steps(synth.CONFIGS["llama1b_8k"], 2, seed=1)


def test_llama1b_b8_full_config_parity():
    # the full batch-8 workload: 16 layers, vocab 128256, eight sequences
    # with their own cache lengths drawn from U[512, 2048]; every step's
    # logits, argmax and appended K/V rows of every sequence against the
    # oracle
    cfg = synth.CONFIGS["llama1b_b8"]
    worst = run_steps(cfg, 3, seed=0)
    print(f"llama1b_b8 worst max|dlogit|/std = {worst:.2e}")


def _moe_small_cfg():
    # MoE variant (hidden 2048, head_dim 128, 4 q heads per kv head) at a reduced
    # size: 16 experts, top-4, shared expert, ragged FFN widths
    return synth.custom(n_layers=3, hidden=2048, n_q_heads=8, n_kv_heads=2, head_dim=128, ffn=0,
                        vocab=3001, tied=False, n_experts=16, top_k=4, expert_ffn=200,
                        shared_ffn=500, rope_theta=5e5, prefill=(70, 70), steps=4)


def test_moe_small_parity():
    run_steps(_moe_small_cfg(), 4, seed=21)


def test_moe_small_held():
    # routers, shared and routed slices all held, no early stage
    run_steps(_moe_small_cfg(), 3, seed=22, hold=(63, 0))


@pytest.mark.parametrize("shared,expert", [(0, 200), (0, 204), (8, 200)])
def test_moe_without_or_with_a_small_shared_expert(shared, expert):
    # no shared expert (or one of 8 columns): every SM's first MLP instruction
    # is a routed slice that waits on the router.  The routers' arrival counts
    # once shared a word with the dependency wait's seen-key, so an
    # instruction whose key equalled an arrival count skipped its wait on the
    # routing and read the previous step's experts; these shapes hit that
    cfg = synth.custom(n_layers=3, hidden=2048, n_q_heads=8, n_kv_heads=2, head_dim=128, ffn=0,
                       vocab=3001, tied=False, n_experts=16, top_k=4, expert_ffn=expert,
                       shared_ffn=shared, rope_theta=5e5, prefill=(70, 70), steps=4)
    run_steps(cfg, 4, seed=25)


def test_moe_full_config_parity():
    r = Run(synth.CONFIGS["moe"], seed=0)
    try:
        for _ in range(2):
            r.step()
        print(f"moe worst max|dlogit|/std = {r.worst:.2e}, near ties {r.near_ties}")
    finally:
        r.close()


def test_ablation_modes_match_megakernel():
    cfg = synth.custom(n_layers=3, n_q_heads=6, n_kv_heads=3, ffn=1000, vocab=999,
                       prefill=(20, 20), steps=6)
    r = Run(cfg, seed=11)
    try:
        for mode in ("stream", "graph", "pdl", "mega"):
            pos0, tok0 = list(r.pos), list(r.tokens)
            lg_m, am_m = r.gpu_step("mega")
            lg_a, am_a = r.gpu_step(mode)
            assert np.array_equal(am_m, am_a), mode
            assert np.abs(lg_m - lg_a).max() <= 1e-3 * lg_m.std(), mode
            r.pos, r.tokens = pos0, tok0
            r.step(mode)  # and against the oracle
    finally:
        r.close()


def test_missing_producer_times_out_and_recovers():
    r = Run(synth.CONFIGS["tiny"], seed=2)
    try:
        r.dec.set_wait_timeout(50_000_000)  # 50 ms
        r.dec.drop_instruction(0, 0)  # SM 0's first QKV slice never signals
        r.dec.step(r.d_tok, r.d_pos, r.d_logits, r.d_am)
        assert r.dec.sync_status() == MK_ERR_TIMEOUT
        r.dec.build_schedule(r.B, r.max_ctx)  # restores the dropped instruction
        r.step()
        r.step()
    finally:
        r.close()


def test_host_buffer_step_matches_and_validates():
    r = Run(synth.CONFIGS["tiny"], seed=4)
    try:
        cfg = r.cfg
        tok = torch.tensor(r.tokens, dtype=torch.int32).pin_memory()
        pos = torch.tensor(r.pos, dtype=torch.int32).pin_memory()
        lg = torch.empty((1, cfg["vocab"]), dtype=torch.float32).pin_memory()
        am = torch.empty(1, dtype=torch.int32).pin_memory()
        assert r.dec.step_host(tok, pos, lg, am) == MK_OK
        lo, ao, _, _ = r.om.step(r.ko, r.vo, r.tokens, r.pos)
        r.check(lg.numpy().astype(np.float64), am.numpy(), lo, ao)
        bad = torch.tensor([cfg["vocab"]], dtype=torch.int32)
        assert r.dec.step_host(bad, pos, lg, am) == MK_ERR_INVALID_ARG
        badp = torch.tensor([r.max_ctx], dtype=torch.int32)
        assert r.dec.step_host(tok, badp, lg, am) == MK_ERR_INVALID_ARG
    finally:
        r.close()

"""Per-phase parity: after one step, the queries after RoPE, the residual after
every O-projection and every MLP, and (dense batch 1) SiLU(gate)*up of every
layer, read back with mk_debug_read, against the same intermediates of the
oracle teacher-forced on the same tokens.  A fault in one opcode shows up at
the first phase it touches instead of only in the logits."""
import numpy as np
import pytest

import synth
from tests.harness import Run

pytestmark = pytest.mark.gpu
REL = 1e-2  # of the oracle vector's standard deviation


def _close(gpu, ref, what):
    err = np.abs(gpu.astype(np.float64) - ref).max()
    assert err <= REL * ref.std() + 1e-6, f"{what}: max|d| {err:.3g}, std {ref.std():.3g}"


def _check(cfg, seed, **kw):
    r = Run(cfg, seed, **kw)
    try:
        toks, pos = list(r.tokens), list(r.pos)
        r.gpu_step()
        tr = {}
        r.om.step(r.ko, r.vo, toks, pos, trace=tr)
        L, dense1 = cfg["n_layers"], cfg["n_experts"] == 0 and cfg["batch"] == 1
        for l in range(L):
            _close(r.dec.debug_read("q", l), tr["q"][l], f"q layer {l}")
            if dense1:
                _close(r.dec.debug_read("h", l), tr["h"][l], f"h layer {l}")
        for j in range(1, 2 * L + 1):
            _close(r.dec.debug_read("x", j), tr["x"][j - 1], f"x_{j}")
    finally:
        r.close()


def test_intermediates_small_shape():
    _check(synth.custom(n_layers=3, n_q_heads=6, n_kv_heads=3, ffn=1000, vocab=999,
                        prefill=(300, 300), steps=2), 101)


def test_intermediates_llama1b():
    _check(synth.CONFIGS["llama1b_1k"], 103)


def test_intermediates_llama1b_b8_full_config():
    # the full batch-8 workload (16 layers, lengths U[512, 2048]): q and every
    # residual of every sequence
    _check(synth.CONFIGS["llama1b_b8"], 109)


@pytest.mark.parametrize("ffn", [2048, 3000])
def test_intermediates_batch8(ffn):
    # ffn 2048: the batched split MLP; 3000: fused MLP slices with atomics
    _check(synth.custom(n_layers=2, hidden=2048, n_q_heads=8, n_kv_heads=2, head_dim=64, ffn=ffn,
                        vocab=5000, batch=8, prefill=(0, 300), steps=2, rope_theta=5e5), 105)


def test_intermediates_int8():
    _check(synth.custom(n_layers=2, hidden=2048, n_q_heads=32, n_kv_heads=8, head_dim=64,
                        ffn=2048, vocab=5000, rope_theta=5e5, prefill=(300, 300), steps=2), 107,
           int8=True)

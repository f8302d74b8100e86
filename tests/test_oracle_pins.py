"""Pins for the CPU oracle: each check compares the oracle with something other
than itself -- a closed form, an invariant, a library routine, or the
independent numpy formulation in brute_numpy.py.  No GPU needed."""
import itertools
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from tests import brute_numpy as bn

rng = np.random.default_rng(1234)


def rand_bits(shape, std=1.0):
    return bn.to_bits(rng.normal(0.0, std, size=shape))


# ---------------------------------------------------------------- bf16 ----
@pytest.mark.parametrize("bits,val", [
    (0x3F80, 1.0), (0xC000, -2.0), (0x4049, 3.140625), (0x0001, 2.0 ** -133),
    (0x7F7F, (2 - 2 ** -7) * 2.0 ** 127), (0x8000, -0.0), (0x3E80, 0.25)])
def test_bf16_widening_bit_patterns(bits, val):
    assert oracle.bf16_to_f64(bits) == val


@pytest.mark.parametrize("x,bits", [
    (1.0 + 2 ** -8, 0x3F80),             # exact tie -> even (1.0)
    (1.0 + 3 * 2 ** -8, 0x3F82),         # exact tie -> even (1 + 2^-6)
    (1.0 + 2 ** -8 + 2 ** -30, 0x3F81),  # just above the tie -> up
    (-(1.0 + 2 ** -8 + 2 ** -30), 0xBF81),
    (math.pi, 0x4049), (-0.0, 0x8000), (2.0 ** 128, 0x7F80),
    (1.5 * 2 ** -133, 0x0002), (2.5 * 2 ** -133, 0x0002),  # subnormal ties -> even
])
def test_bf16_rounding_closed_forms(x, bits):
    assert oracle.f64_to_bf16(x) == bits


def test_bf16_rounding_matches_torch_on_float32_values():
    # a float32 value rounds to bf16 in one step either way: torch's RNE must agree
    x = rng.normal(0, 3, 20000).astype(np.float32)
    x[:100] = rng.integers(-2**20, 2**20, 100) * 2.0 ** -12  # many exact ties
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.f64_to_bf16(float(v)) for v in x], np.uint16)
    assert np.array_equal(got, ref)


# -------------------------------------------------------------- RMSNorm ----
def test_rmsnorm_constant_vector_closed_form():
    n, c, eps = 64, 0.3, 1e-5
    out = oracle.rmsnorm(np.full(n, c), bn.to_bits(np.ones(n)), eps)
    assert np.allclose(out, c / math.sqrt(c * c + eps), rtol=1e-15)


def test_rmsnorm_unit_rms_times_gain():
    x = rng.normal(0, 5, 2048)
    g = rand_bits(2048, 0.5)
    out = oracle.rmsnorm(x, g, 0.0)
    unit = out / bn.widen(g)
    assert abs(np.sqrt(np.mean(unit ** 2)) - 1.0) < 1e-12
    assert np.allclose(unit * np.sqrt(np.mean(x * x)), x, rtol=1e-12)


# ----------------------------------------------------------------- RoPE ----
def test_rope_identity_at_position_zero():
    v = rng.normal(size=64)
    assert np.array_equal(oracle.rope(v, 0, 5e5), v)


def test_rope_worked_example_d4():
    # rotate-half pairs (0,2) and (1,3); frequencies 1 and theta^-1/2 = 0.01
    out = oracle.rope(np.array([1.0, 0, 0, 0]), 1, 1e4)
    assert np.allclose(out, [math.cos(1), 0, math.sin(1), 0], atol=1e-15)
    out = oracle.rope(np.array([0, 1.0, 0, 0]), 3, 1e4)
    assert np.allclose(out, [0, math.cos(0.03), 0, math.sin(0.03)], atol=1e-15)


def test_rope_preserves_pair_norms_and_relative_position():
    d, theta = 64, 5e5
    q, k = rng.normal(size=d), rng.normal(size=d)
    r = oracle.rope(q, 777, theta)
    h = d // 2
    assert np.allclose(np.hypot(r[:h], r[h:]), np.hypot(q[:h], q[h:]), rtol=1e-13)
    dots = [oracle.rope(q, m + t, theta) @ oracle.rope(k, m - 5 + t, theta)
            for m, t in [(10, 0), (10, 100), (10, 4000)]]
    assert np.allclose(dots, dots[0], rtol=1e-9)


def test_rope_matches_complex_rotation():
    d = 128
    for pos in (1, 17, 1023, 8191):
        v = rng.normal(size=d)
        assert np.allclose(oracle.rope(v, pos, 5e5), bn.rope_complex(v[None], pos, 5e5)[0],
                           atol=1e-12)


# ----------------------------------------------------------------- GEMV ----
@pytest.mark.parametrize("rows,cols", [(1, 1), (37, 129), (300, 2048)])
def test_gemv_matches_numpy_matmul(rows, cols):
    W = rand_bits((rows, cols), 0.02)
    x = rng.normal(size=cols)
    assert np.allclose(oracle.gemv(W, x), bn.widen(W) @ x, rtol=1e-12, atol=1e-14)


# ------------------------------------------------------------ attention ----
def test_attention_single_position_returns_v():
    d = 64
    K, V = rand_bits((1, d)), rand_bits((1, d))
    out = oracle.attention(rng.normal(size=d), K, V)
    assert np.array_equal(out, bn.widen(V[0]))


def test_attention_equal_scores_returns_mean_v():
    d, n = 64, 9
    K, V = rand_bits((n, d)), rand_bits((n, d))
    out = oracle.attention(np.zeros(d), K, V)
    assert np.allclose(out, bn.widen(V).mean(axis=0), rtol=1e-13, atol=1e-15)


def test_attention_matches_scipy_softmax():
    from scipy.special import softmax
    d, n = 128, 333
    K, V = rand_bits((n, d)), rand_bits((n, d))
    q = rng.normal(size=d)
    ref = softmax(bn.widen(K) @ q / math.sqrt(d)) @ bn.widen(V)
    assert np.allclose(oracle.attention(q, K, V), ref, rtol=1e-11, atol=1e-13)


def test_split_merge_equals_unsplit_for_every_split_of_a_small_context():
    d, n = 64, 7
    K, V = rand_bits((n, d)), rand_bits((n, d))
    q = rng.normal(size=d) * 3
    full = oracle.attention(q, K, V)
    for cuts in itertools.combinations_with_replacement(range(n + 1), 2):
        bounds = [0, *cuts, n]
        parts = [oracle.attention_partial(q, K, V, bounds[i], bounds[i + 1]) for i in range(3)]
        m = [p[0] for p in parts]
        l = [p[1] for p in parts]
        o = np.stack([p[2] for p in parts])
        assert np.allclose(oracle.attention_merge(m, l, o), full, rtol=1e-12, atol=1e-14), cuts


def test_empty_partial_is_neutral():
    d = 64
    K, V = rand_bits((3, d)), rand_bits((3, d))
    m, l, o = oracle.attention_partial(rng.normal(size=d), K, V, 2, 2)
    assert m == -math.inf and l == 0.0 and not o.any()


# ---------------------------------------------------------- SiLU / MLP ----
def test_silu_closed_forms():
    assert oracle.silu(0.0) == 0.0
    assert math.isclose(oracle.silu(1.0), 1.0 / (1.0 + math.exp(-1.0)), rel_tol=1e-15)
    for a in (0.3, 2.0, 7.5):
        assert math.isclose(oracle.silu(a) - oracle.silu(-a), a, rel_tol=1e-14)
    assert math.isclose(oracle.silu(40.0), 40.0, rel_tol=1e-15)


def test_swiglu_constructed_weights():
    Wg = bn.to_bits(np.array([[1.0, 0.0]]))
    Wu = bn.to_bits(np.array([[0.0, 1.0]]))
    Wd = bn.to_bits(np.array([[1.0], [2.0]]))
    a, b = 0.7, -1.3
    h = a / (1 + math.exp(-a)) * b
    assert np.allclose(oracle.swiglu(Wg, Wu, Wd, np.array([a, b])), [h, 2 * h], rtol=1e-15)


# --------------------------------------------------------------- router ----
def test_router_topk_matches_stable_argsort_and_renormalises():
    from scipy.special import softmax
    for trial in range(50):
        E, k = 128, 8
        lg = rng.normal(size=E)
        if trial % 5 == 0:  # plant exact ties
            lg[rng.integers(0, E, 10)] = lg.max()
        ids, w, margin = oracle.router_topk(lg, k)
        p = softmax(lg)
        order = np.argsort(-p, kind="stable")
        assert np.array_equal(ids, order[:k])
        assert np.allclose(w, p[order[:k]] / p[order[:k]].sum(), rtol=1e-13)
        assert math.isclose(w.sum(), 1.0, rel_tol=1e-14)
        assert math.isclose(margin, (p[order[k - 1]] - p[order[k]]) / p[order[k - 1]],
                            rel_tol=1e-9, abs_tol=1e-15)


def test_router_k_equals_e():
    ids, w, margin = oracle.router_topk(np.array([0.5, 2.0, -1.0]), 3)
    assert list(ids) == [1, 0, 2] and margin == 1.0 and math.isclose(w.sum(), 1.0)


def test_argmax_first_index_on_ties():
    assert oracle.argmax(np.array([1.0, 3.0, 3.0, 2.0])) == 1
    for _ in range(20):
        v = np.round(rng.normal(size=1000), 1)
        assert oracle.argmax(v) == int(np.argmax(v))


# -------------------------------------------------------- whole decoder ----
def _run_both(cfg, seed=0, steps=None, forced=None):
    cfg = synth.with_cache(cfg)
    W = synth.make_weights(cfg, seed)
    lengths = synth.make_lengths(cfg, seed)
    ks, vs = synth.make_kv(cfg, lengths, seed)
    kb = [bn.widen(oracle._bits(t)) for t in ks]  # independent float64 caches
    vb = [bn.widen(oracle._bits(t)) for t in vs]
    ko = [oracle._bits(t).copy() for t in ks]
    vo = [oracle._bits(t).copy() for t in vs]
    om = oracle.OracleModel(cfg, W)
    Wf = bn.weights_f64(W)
    toks = synth.make_tokens(cfg, seed)
    pos = list(lengths)
    worst = 0.0
    for _ in range(steps or cfg["steps"]):
        lo, ao, rid, _ = om.step(ko, vo, toks, pos)
        lb, ab, routes = bn.decode(cfg, Wf, kb, vb, toks, pos)
        worst = max(worst, float(np.max(np.abs(lo - lb))))
        assert np.array_equal(ao, ab)
        if rid is not None:
            assert np.array_equal(np.asarray(routes).reshape(rid.shape[1], rid.shape[0], -1),
                                  rid.transpose(1, 0, 2))
        toks = [int(a) for a in ao]
        pos = [p + 1 for p in pos]
    for l in range(cfg["n_layers"]):
        assert np.array_equal(bn.widen(ko[l]), kb[l]) and np.array_equal(bn.widen(vo[l]), vb[l])
    return worst


def test_tiny_decoder_matches_independent_numpy_formulation():
    assert _run_both(synth.CONFIGS["tiny"]) < 1e-9


def test_mha_and_batched_decoder_matches_numpy():
    cfg = synth.custom(n_q_heads=4, n_kv_heads=4, batch=3, prefill=(0, 9), steps=3,
                       hidden=128, ffn=96, vocab=300, head_dim=32)
    assert _run_both(cfg) < 1e-9


def test_moe_decoder_matches_numpy():
    cfg = synth.custom(n_layers=2, hidden=128, n_q_heads=4, n_kv_heads=2, head_dim=32, ffn=0,
                       vocab=200, tied=False, n_experts=8, top_k=3, expert_ffn=48,
                       shared_ffn=64, steps=3, prefill=(5, 5))
    assert _run_both(cfg) < 1e-9


def test_moe_single_expert_equals_dense():
    base = dict(n_layers=2, hidden=128, n_q_heads=4, n_kv_heads=2, head_dim=32, vocab=200,
                steps=2, prefill=(4, 4))
    dense = synth.with_cache(synth.custom(ffn=48, **base))
    moe = synth.with_cache(synth.custom(ffn=0, n_experts=1, top_k=1, expert_ffn=48,
                                        shared_ffn=0, **base))
    Wd = synth.make_weights(dense, 7)
    Wm = {k: v for k, v in Wd.items() if k != "layers"}
    Wm["layers"] = [{k: v for k, v in lw.items() if not k.startswith("w_")} |
                    {"router": lw["attn_norm"][None, :].clone(),
                     "ex_gate": lw["w_gate"][None], "ex_up": lw["w_up"][None],
                     "ex_down": lw["w_down"][None]} for lw in Wd["layers"]]
    outs = []
    for cfg, W in ((dense, Wd), (moe, Wm)):
        ks, vs = synth.make_kv(cfg, [4], 7)
        om = oracle.OracleModel(cfg, W)
        outs.append(om.step([oracle._bits(t).copy() for t in ks],
                            [oracle._bits(t).copy() for t in vs], [5], [4])[0])
    assert np.array_equal(outs[0], outs[1])


def test_oracle_rejects_bad_arguments():
    cfg = synth.with_cache(synth.CONFIGS["tiny"])
    W = synth.make_weights(cfg, 0)
    ks, vs = synth.make_kv(cfg, [16], 0)
    om = oracle.OracleModel(cfg, W)
    kc = [oracle._bits(t).copy() for t in ks]
    vc = [oracle._bits(t).copy() for t in vs]
    with pytest.raises(ValueError):
        om.step(kc, vc, [cfg["vocab"]], [16])
    with pytest.raises(ValueError):
        om.step(kc, vc, [1], [cfg["max_seq"]])


# ------------------------------------------------------------------- int8 ----
# Per-row int8 weights ("Gemma 4 TPU megakernel", "What's next": INT8
# weights).  Reading: s = max|w| / 127, q = round-half-even(w / s), in fp32.
def _bf16_rows(rows):
    a = np.array(rows, np.float32).view(np.uint32)
    assert np.all((a & 0xFFFF) == 0), "values must be exact in bf16"
    return (a >> 16).astype(np.uint16)


def test_int8_quantiser_worked_rows():
    W = _bf16_rows([[127, -63.5, 0.5, 1.5, -2.5, 0, 64, -127],  # s = 1: ties go to even
                    [0, 0, 0, 0, 0, 0, 0, 0],                   # zero row: s = 0
                    [254, 3, 5, 7, -3, -5, -7, 1],              # s = 2: 1.5, 2.5, 3.5, 0.5
                    [-0.25, 0.125, 0, 0, 0, 0, 0, 0.0078125]])  # negative maximum
    q, s = oracle.quantize_rows_int8(W)
    assert s.tolist() == [1.0, 0.0, 2.0, np.float32(0.25) / np.float32(127)]
    assert q[0].tolist() == [127, -64, 0, 2, -2, 0, 64, -127]
    assert q[1].tolist() == [0] * 8
    assert q[2].tolist() == [127, 2, 2, 4, -2, -2, -4, 0]
    # row 3: -0.25 is the largest magnitude -> -127; 0.125 / s = 63.5 -> 64 (even);
    # 2^-7 / s = 3.96875 -> 4
    assert q[3].tolist() == [-127, 64, 0, 0, 0, 0, 0, 4]


def test_int8_quantiser_error_bound_and_extremes():
    W = rand_bits((40, 300), std=0.02)
    W[3] = 0  # a zero row
    q, s = oracle.quantize_rows_int8(W)
    w = bn.widen(W)
    for r in range(W.shape[0]):
        if not np.any(w[r]):
            assert s[r] == 0 and not np.any(q[r])
            continue
        assert np.max(np.abs(q[r])) == 127  # the largest magnitude maps to +-127
        err = np.abs(w[r] - q[r].astype(np.float64) * np.float64(s[r]))
        # half a step, plus the fp32 rounding of s and of w / s (|w / s| <= 127)
        assert np.all(err <= np.float64(s[r]) * (0.5 + 2.0 ** -16))
        assert np.all(np.sign(q[r]) == np.sign(np.where(np.abs(w[r]) < s[r] / 2, 0, w[r])))


def test_int8_gemv_matches_numpy_on_dequantised_weights():
    rng = np.random.default_rng(9)
    q = rng.integers(-127, 128, size=(37, 160)).astype(np.int8)
    s = rng.uniform(1e-4, 1e-2, size=37).astype(np.float32)
    x = rng.standard_normal(160)
    y = oracle.gemv_q8(q, s, x)
    ref = (q.astype(np.float64) * s.astype(np.float64)[:, None]) @ x
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-14)
    # one row, one column: q * s * x
    assert oracle.gemv_q8(np.array([[-3]], np.int8), np.array([0.5], np.float32), [2.0])[0] == -3.0


def _exact_int8_weights(cfg, seed):
    """bf16 weights that per-row int8 quantisation reproduces exactly: each row
    is q * 2^-e with integer q in [-127, 127] (one entry at +-127) and e in 9..12."""
    W = synth.make_weights(cfg, seed)
    rng = np.random.default_rng(seed + 3)

    def exact(t):
        rows, cols = t.shape
        q = rng.integers(-127, 128, size=(rows, cols))
        q[np.arange(rows), rng.integers(0, cols, rows)] = 127 * rng.choice([-1, 1], rows)
        e = rng.integers(9, 13, size=rows)
        return torch.tensor(q * np.exp2(-e.astype(np.float64))[:, None],
                            dtype=torch.float32).to(torch.bfloat16)

    W["embed"] = exact(W["embed"])
    for lw in W["layers"]:
        for n in ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down"):
            lw[n] = exact(lw[n])
    return W


def _oracle_steps(cfg, W, int8, steps=3, seed=0):
    lengths = synth.make_lengths(cfg, seed)
    ks, vs = synth.make_kv(cfg, lengths, seed)
    ko = [oracle._bits(t).copy() for t in ks]
    vo = [oracle._bits(t).copy() for t in vs]
    om = oracle.OracleModel(cfg, W, int8=int8)
    toks, pos, out = synth.make_tokens(cfg, seed), list(lengths), []
    for _ in range(steps):
        lo, ao, _, _ = om.step(ko, vo, toks, pos)
        out.append(lo)
        toks = [int(a) for a in ao]
        pos = [p + 1 for p in pos]
    return out


def test_int8_decoder_equals_bf16_decoder_on_exactly_quantisable_weights():
    cfg = synth.with_cache(synth.custom(n_layers=2, hidden=128, n_q_heads=4, n_kv_heads=2,
                                        head_dim=32, ffn=96, vocab=300, batch=2,
                                        prefill=(3, 9), steps=3))
    W = _exact_int8_weights(cfg, 11)
    a = _oracle_steps(cfg, W, int8=False)
    b = _oracle_steps(cfg, W, int8=True)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_int8_decoder_differs_by_the_quantisation_error_only():
    cfg = synth.with_cache(synth.custom(n_layers=2, hidden=128, n_q_heads=4, n_kv_heads=2,
                                        head_dim=32, ffn=96, vocab=300, steps=2,
                                        prefill=(5, 5)))
    W = synth.make_weights(cfg, 13)
    a = _oracle_steps(cfg, W, int8=False, steps=1)[0]
    b = _oracle_steps(cfg, W, int8=True, steps=1)[0]
    d = np.max(np.abs(a - b)) / np.std(a)
    assert 0 < d < 0.1  # the int8 path is taken, and ~1 % weight noise stays small


def test_int8_oracle_refuses_moe():
    cfg = synth.with_cache(synth.custom(n_layers=1, hidden=128, n_q_heads=4, n_kv_heads=2,
                                        head_dim=32, ffn=0, vocab=200, tied=False, n_experts=4,
                                        top_k=2, expert_ffn=32, shared_ffn=0, prefill=(2, 2)))
    with pytest.raises(AssertionError):
        oracle.OracleModel(cfg, synth.make_weights(cfg, 0), int8=True)


# ------------------------------------------------------- traced decode step ----
def test_traced_step_equals_untraced_and_feeds_the_logits():
    cfg = synth.with_cache(synth.custom(n_layers=2, hidden=128, n_q_heads=4, n_kv_heads=2,
                                        head_dim=32, ffn=96, vocab=300, batch=2,
                                        prefill=(3, 9), steps=2))
    W = synth.make_weights(cfg, 21)
    lengths = synth.make_lengths(cfg, 21)
    ks, vs = synth.make_kv(cfg, lengths, 21)
    toks = synth.make_tokens(cfg, 21)
    om = oracle.OracleModel(cfg, W)
    runs = []
    for trace in (None, {}):
        ko = [oracle._bits(t).copy() for t in ks]
        vo = [oracle._bits(t).copy() for t in vs]
        runs.append((om.step(ko, vo, toks, list(lengths), trace=trace), trace, ko))
    (a, _, ka), (b, tr, kb) = runs
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    assert all(np.array_equal(x, y) for x, y in zip(ka, kb))
    L, H = cfg["n_layers"], cfg["hidden"]
    assert tr["q"].shape == (L, 2, cfg["n_q_heads"] * cfg["head_dim"])
    assert tr["x"].shape == (2 * L, 2, H) and tr["h"].shape == (L, 2, cfg["ffn"])
    # the last residual, normed and multiplied by the (tied) head in numpy,
    # gives the logits
    Wf = bn.weights_f64(W)
    for s in range(2):
        x = tr["x"][-1, s]
        g = bn.widen(oracle._bits(W["final_norm"]))
        xn = x / np.sqrt(np.mean(x * x) + cfg["rms_eps"]) * g
        assert np.allclose(Wf["embed"] @ xn, b[0][s], rtol=1e-12, atol=1e-12)


def test_traced_mlp_output_is_the_residual_step():
    # x after the MLP minus x after the O-projection is Wd h for the traced h
    cfg = synth.with_cache(synth.custom(n_layers=2, hidden=128, n_q_heads=4, n_kv_heads=2,
                                        head_dim=32, ffn=96, vocab=300, prefill=(5, 5)))
    W = synth.make_weights(cfg, 23)
    ks, vs = synth.make_kv(cfg, [5], 23)
    tr = {}
    oracle.OracleModel(cfg, W).step([oracle._bits(t).copy() for t in ks],
                                    [oracle._bits(t).copy() for t in vs], [7], [5], trace=tr)
    Wf = bn.weights_f64(W)
    for l in range(cfg["n_layers"]):
        d = tr["x"][2 * l + 1, 0] - tr["x"][2 * l, 0]
        assert np.allclose(Wf["layers"][l]["w_down"] @ tr["h"][l, 0], d, rtol=1e-9, atol=1e-12)

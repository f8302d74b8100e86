"""Host-only tests of libmk.so: exported symbols, the schedule builder and its
deadlock / coverage checker.  No GPU needed (no compute call is made)."""
import ctypes as C
import os
import re

import pytest

import synth
from decode_megakernel_sm_gb300 import _lib as L
from decode_megakernel_sm_gb300.decoder import desc_from_config

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_symbols():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            names |= set(re.findall(r"^(?:int|const char\*)\s+(mk_\w+)\s*\(", src, re.M))
    return names


def test_library_exports_every_declared_symbol():
    lib = L.lib()
    names = declared_symbols()
    assert len(names) >= 13
    for n in sorted(names):
        assert hasattr(lib, n), n


def test_bounds_library_exports_every_declared_symbol():
    # the bounds-checked build (MK_BOUNDS: the small variant with every
    # checked access guarded) has the same C ABI
    from decode_megakernel_sm_gb300 import build as B
    L.lib()  # builds both libraries when either is stale
    lib = C.CDLL(B.LIB_BOUNDS)
    for n in sorted(declared_symbols()):
        assert hasattr(lib, n), n
    f = lib.mk_status_string
    f.restype, f.argtypes = C.c_char_p, [C.c_int]
    assert b"bounds" in f(L.MK_ERR_BOUNDS)


def test_status_strings():
    for s in range(0, -10, -1):
        assert L.mk_status_string(s) not in ("", "unknown status")
    assert L.mk_status_string(-99) == "unknown status"


def desc(name, **over):
    cfg = synth.with_cache(dict(synth.CONFIGS[name], **over))
    return cfg, desc_from_config(cfg, cfg["batch"], cfg["max_seq"])


def queues(q, n_sm, max_pc):
    return [[q[s * max_pc + i] for i in range(max_pc)] for s in range(n_sm)]


def independent_coverage(cfg, q, n_sm, max_pc, splits):
    """Re-derive, in Python, that every unit of work appears exactly once."""
    Lc, H, Hq, Hkv, D = cfg["n_layers"], cfg["hidden"], cfg["n_q_heads"], cfg["n_kv_heads"], \
        cfg["head_dim"]
    B = cfg["batch"]
    R = Hkv * (Hq // Hkv + 2) * D
    moe = cfg["n_experts"] > 0
    Fv = cfg["shared_ffn"] + cfg["top_k"] * cfg["expert_ffn"] if moe else cfg["ffn"]
    seen = {k: set() for k in ("qkv", "attn", "oproj", "mlp", "res", "lm", "router")}
    sig = {}
    for s in range(n_sm):
        for i in range(max_pc):
            I = q[s * max_pc + i]
            if I.op == 0:
                break
            if I.sig_ctr != 0xFFFFFFFF:
                sig[I.sig_ctr] = sig.get(I.sig_ctr, 0) + 1
            if I.op == 1:
                for r in range(I.r0, I.r1):
                    assert (I.layer, r) not in seen["qkv"]
                    seen["qkv"].add((I.layer, r))
            elif I.op == 2:
                key = (I.layer, I.b, I.g, I.r0)
                assert key not in seen["attn"] and I.r1 == splits
                seen["attn"].add(key)
            elif I.op == 3:
                for r in range(I.r0, I.r1):
                    seen["oproj"].add((I.layer, I.g, r))
            elif I.op == 4:
                base = 0
                if moe and not (I.flags & 4):
                    base = cfg["shared_ffn"] + I.g * cfg["expert_ffn"]
                for c in range(I.r0, I.r1):
                    assert (I.layer, base + c) not in seen["mlp"]
                    seen["mlp"].add((I.layer, base + c))
                for r in range(I.aux & 0xFFFF, I.aux >> 16):
                    assert (I.layer, r) not in seen["res"]
                    seen["res"].add((I.layer, r))
            elif I.op == 8:  # gate/up column slice of the split MLP
                for c in range(I.r0, I.r1):
                    assert (I.layer, c) not in seen["mlp"]
                    seen["mlp"].add((I.layer, c))
            elif I.op == 9:  # down rows of the split MLP (own their residual)
                assert I.r1 - I.r0 <= 64
                for r in range(I.r0, I.r1):
                    assert (I.layer, r) not in seen["res"]
                    seen["res"].add((I.layer, r))
            elif I.op == 5:
                for r in range(I.r0, I.r1):
                    assert r not in seen["lm"]
                    seen["lm"].add(r)
            elif I.op == 6:
                for r in range(I.r0, I.r1):
                    seen["router"].add((I.layer, r))
    assert len(seen["qkv"]) == Lc * R
    assert len(seen["attn"]) == Lc * B * Hkv * splits
    assert len(seen["oproj"]) == Lc * Hq * H
    assert len(seen["mlp"]) == Lc * Fv
    assert len(seen["res"]) == Lc * H
    assert len(seen["lm"]) == cfg["vocab"]
    assert len(seen["router"]) == (Lc * cfg["n_experts"] if moe else 0)
    # every wait is for all signals of its counter
    for s in range(n_sm):
        for i in range(max_pc):
            I = q[s * max_pc + i]
            if I.op == 0:
                break
            if I.wait_ctr != 0xFFFFFFFF:
                assert I.wait_cnt == sig[I.wait_ctr] > 0


@pytest.mark.parametrize("name", list(synth.CONFIGS))
@pytest.mark.parametrize("n_sm", [1, 7, 148, 152])
def test_plan_covers_all_work_and_is_deadlock_free(name, n_sm):
    cfg, d = desc(name)
    st, q = L.mk_plan(d, cfg["batch"], cfg["max_seq"], n_sm)
    assert st["n_sm"] == n_sm
    if is_wide(cfg):
        wide_coverage(cfg, q, n_sm, st["max_pc"], st["attn_splits"])
    else:
        independent_coverage(cfg, q, n_sm, st["max_pc"], st["attn_splits"])
    assert L.mk_plan_check(q, n_sm, st["max_pc"], st["n_counters"]) == L.MK_OK


def test_split_mlp_is_used_for_dense_models():
    # batch 1, and batches of up to 8 whose FFN is whole 512-column tiles
    for name, split in (("llama1b_1k", True), ("tiny", True), ("llama1b_b8", True), ("moe", False)):
        cfg, d = desc(name)
        st, q = L.mk_plan(d, cfg["batch"], cfg["max_seq"], 152)
        ops = {q[i].op for i in range(152 * st["max_pc"])}
        assert (8 in ops and 9 in ops and 4 not in ops) == split, name
        assert (4 in ops) == (not split), name


def test_llama1b_plan_is_byte_balanced():
    cfg, d = desc("llama1b_1k")
    st, _ = L.mk_plan(d, 1, cfg["max_seq"], 152, with_queues=False)
    assert st["max_sm_bytes"] / st["mean_sm_bytes"] < 1.03
    assert 120 <= st["attn_splits"] * cfg["n_kv_heads"] <= 152


def test_checker_rejects_unsatisfiable_wait():
    cfg, d = desc("tiny")
    st, q = L.mk_plan(d, 1, cfg["max_seq"], 16)
    for i in range(len(q)):
        if q[i].op == 2:  # an attention item: wait one signal more than will ever come
            q[i].wait_cnt += 1
            break
    assert L.mk_plan_check(q, 16, st["max_pc"], st["n_counters"]) == L.MK_ERR_SCHEDULE


def test_checker_rejects_cyclic_order():
    cfg, d = desc("tiny")
    n_sm = 4
    st, q = L.mk_plan(d, 1, cfg["max_seq"], n_sm)
    mp = st["max_pc"]
    # on SM 0 move a layer-1 QKV (waits on all of layer 0's MLP) in front of
    # SM 0's own layer-0 MLP instruction: a cycle through SM 0's queue
    row = [q[i] for i in range(mp)]
    # the instruction signalling layer 0's MLP counter: fused slice (4) or down rows (9)
    i_mlp = next(i for i, I in enumerate(row) if I.op in (4, 9) and I.layer == 0)
    i_qkv = next(i for i, I in enumerate(row) if I.op == 1 and I.layer == 1)
    saved = L.mk_instr()
    C.memmove(C.byref(saved), C.byref(q[i_qkv]), C.sizeof(saved))
    for k in range(i_qkv, i_mlp, -1):
        C.memmove(C.byref(q[k]), C.byref(q[k - 1]), C.sizeof(saved))
    C.memmove(C.byref(q[i_mlp]), C.byref(saved), C.sizeof(saved))
    assert L.mk_plan_check(q, n_sm, mp, st["n_counters"]) == L.MK_ERR_SCHEDULE


def test_checker_rejects_bad_counter_id():
    cfg, d = desc("tiny")
    st, q = L.mk_plan(d, 1, cfg["max_seq"], 8)
    q[0].sig_ctr = st["n_counters"] + 5
    assert L.mk_plan_check(q, 8, st["max_pc"], st["n_counters"]) == L.MK_ERR_SCHEDULE


def test_plan_rejects_bad_arguments():
    cfg, d = desc("tiny")
    with pytest.raises(L.MkError) as e:
        L.mk_plan(d, 0, cfg["max_seq"], 8)
    assert e.value.status == L.MK_ERR_INVALID_ARG
    with pytest.raises(L.MkError) as e:
        L.mk_plan(d, 1, cfg["max_seq"] + 1, 8)
    assert e.value.status == L.MK_ERR_INVALID_ARG
    with pytest.raises(L.MkError) as e:
        L.mk_plan(d, 2, cfg["max_seq"], 8)  # batch above max_batch
    assert e.value.status == L.MK_ERR_INVALID_ARG
    _, d2 = desc("tiny", head_dim=96)
    with pytest.raises(L.MkError) as e:
        L.mk_plan(d2, 1, 64, 8)
    assert e.value.status == L.MK_ERR_UNSUPPORTED
    _, d3 = desc("tiny", batched_variant=2)  # 0 or 1 only
    with pytest.raises(L.MkError) as e:
        L.mk_plan(d3, 1, 64, 8)
    assert e.value.status == L.MK_ERR_INVALID_ARG


@pytest.mark.parametrize("variant", [0, 1])
def test_batched_variant_picks_the_plan(variant):
    # 2..8 sequences on a shape the wide variant takes: its plan (NORM
    # instructions, tensor-core tiles) unless the descriptor asks for the
    # batched mma.sync variant (whole-tile split MLP, no NORM instructions)
    cfg, d = desc("llama1b_b8", batch=4, batched_variant=variant)
    st, q = L.mk_plan(d, 4, cfg["max_seq"], 152)
    ops = {q[i].op for i in range(152 * st["max_pc"])}
    assert (10 in ops) == (variant == 0)
    assert is_wide(cfg) == (variant == 0)


def test_split_mlp_residual_hop_is_tagged():
    # dense batch 1: the down rows publish x_{2l+2} as tagged words and signal
    # without release; its readers (next QKV, LM head) poll the words
    cfg, d = desc("llama1b_1k")
    st, q = L.mk_plan(d, 1, cfg["max_seq"], 152)
    n = 152 * st["max_pc"]
    ops = [q[i] for i in range(n) if q[i].op != 0]
    F_TAG_WAIT, F_RELAXED_SIG = 16, 32
    assert all(I.flags & F_RELAXED_SIG for I in ops if I.op == 9)
    assert all(I.flags & F_TAG_WAIT for I in ops if I.op == 5)
    assert all(bool(I.flags & F_TAG_WAIT) == (I.layer > 0) for I in ops if I.op == 1)
    assert not any(I.flags & (F_TAG_WAIT | F_RELAXED_SIG) for I in ops if I.op in (2, 3, 8))


def test_checker_rejects_plain_wait_on_relaxed_signals():
    # relaxed signals order no data: a consumer that waits on such a counter
    # and then reads untagged data could read stale values, so the checker
    # counts only release signals for plain waits and reports the deadlock
    cfg, d = desc("tiny")
    st, q = L.mk_plan(d, 1, cfg["max_seq"], 8)
    assert L.mk_plan_check(q, 8, st["max_pc"], st["n_counters"]) == L.MK_OK
    i = next(i for i in range(len(q)) if q[i].op == 1 and q[i].layer == 1)
    q[i].flags &= ~16
    assert L.mk_plan_check(q, 8, st["max_pc"], st["n_counters"]) == L.MK_ERR_SCHEDULE


def test_batched_split_mlp_cuts_whole_tiles():
    # 7 sequences on the batched (mma.sync) variant, asked for by the descriptor
    cfg, d = desc("llama1b_b8", batch=7, batched_variant=1)
    st, q = L.mk_plan(d, cfg["batch"], cfg["max_seq"], 152)
    ops = [q[i] for i in range(152 * st["max_pc"]) if q[i].op in (8, 9)]
    assert all(I.r0 % 16 == 0 and I.r1 % 16 == 0 for I in ops if I.op == 8)
    # down instructions: runs of chunk-major (row block, 512-column chunk)
    # units, at most 32 units and two chunks each, covering every unit of a
    # layer exactly once, with every SM's share within one unit of the mean
    down = [I for I in ops if I.op == 9]
    nrb, nkc = cfg["hidden"] // 16, cfg["ffn"] // 512
    units = sorted(u for I in down if I.layer == 0 for u in range(I.r0, I.r1))
    assert units == list(range(nrb * nkc))
    assert all(I.r1 - I.r0 <= 32 and (I.r1 - 1) // nrb <= I.r0 // nrb + 1 for I in down)
    per_sm = [sum(q[sm * st["max_pc"] + k].r1 - q[sm * st["max_pc"] + k].r0
                  for k in range(st["max_pc"])
                  if q[sm * st["max_pc"] + k].op == 9 and q[sm * st["max_pc"] + k].layer == 0)
              for sm in range(152)]
    assert max(per_sm) - min(per_sm) <= 1
    assert not any(I.flags & (16 | 32) for I in ops)  # no tagged hops at batch > 1


def test_default_hold_marks_gate_up_and_down():
    # the default fetch policy holds the first gate/up and the first down
    # instruction of each layer on every SM, and nothing else
    cfg, d = desc("llama1b_1k")
    st, q = L.mk_plan(d, 1, cfg["max_seq"], 152)
    mp = st["max_pc"]
    for sm in range(152):
        run = [q[sm * mp + k] for k in range(mp) if q[sm * mp + k].op != 0]
        for k, I in enumerate(run):
            first = k > 0 and (run[k - 1].op != I.op or run[k - 1].layer != I.layer)
            assert bool(I.flags & 8) == (first and I.op in (8, 9)), (sm, k, I.op)


# ---- int8 weights: argument checks taken before any CUDA call
def test_create_ex_refuses_bad_format_and_unsupported_int8_shapes():
    lib = L.lib()
    zero_w, zero_kv = L.mk_weights(), L.mk_kv()
    h = C.c_void_p()
    _, d = desc("llama1b_1k")
    assert lib.mk_create_ex(C.byref(d), C.byref(zero_w), C.byref(zero_kv), 7,
                            C.byref(h)) == L.MK_ERR_INVALID_ARG
    assert h.value is None
    for name, over in (("llama1b_b8", {}), ("moe", {}), ("llama1b_1k", {"ffn": 2056}),
                       ("llama1b_1k", {"head_dim": 128, "n_q_heads": 16})):
        _, d = desc(name, **over)
        assert lib.mk_create_ex(C.byref(d), C.byref(zero_w), C.byref(zero_kv),
                                L.MK_WEIGHTS_INT8, C.byref(h)) == L.MK_ERR_UNSUPPORTED, name


def test_quantize_rows_refuses_bad_arguments():
    lib = L.lib()
    p = C.c_void_p(16)  # never dereferenced: the checks come first
    assert lib.mk_quantize_rows_int8(p, -1, 8, p, p, None) == L.MK_ERR_INVALID_ARG
    assert lib.mk_quantize_rows_int8(p, 4, 0, p, p, None) == L.MK_ERR_INVALID_ARG
    assert lib.mk_quantize_rows_int8(None, 4, 8, p, p, None) == L.MK_ERR_INVALID_ARG
    assert lib.mk_quantize_rows_int8(p, 4, 8, None, p, None) == L.MK_ERR_INVALID_ARG
    assert lib.mk_quantize_rows_int8(p, 4, 8, p, None, None) == L.MK_ERR_INVALID_ARG


def is_wide(cfg):
    # the wide-batch (tcgen05) variant's plan: 9..32 sequences, or 2..8 on a
    # shape it takes unless the batched (mma.sync) variant is asked for
    b, dense = cfg["batch"], cfg["n_experts"] == 0
    shape = (cfg["ffn"] % 64 == 0 and cfg["hidden"] % 64 == 0 and cfg["head_dim"] == 64 and
             cfg["n_q_heads"] == 4 * cfg["n_kv_heads"])
    return dense and (b > 8 or (b >= 2 and shape and not cfg.get("batched_variant", 0)))


def wide_coverage(cfg, q, n_sm, max_pc, splits):
    """The wide-batch plan (2..32 sequences), re-derived in Python: every norm
    row, QKV row, attention item, O-projection (head, row), FFN column, down
    (row, 64-column chunk) and LM-head row exactly once, within the tile
    limits the tensor-core bodies rely on (at most 128 weight rows per
    instruction, starting on a multiple of 8), and the LM-head slices: one
    per SM, its instructions consecutive, the first and the last marked."""
    Lc, H, Hq, Hkv, D = cfg["n_layers"], cfg["hidden"], cfg["n_q_heads"], cfg["n_kv_heads"], \
        cfg["head_dim"]
    B, F, V = cfg["batch"], cfg["ffn"], cfg["vocab"]
    HPG, Bp = Hq // Hkv, (B + 7) // 8 * 8
    R = Hkv * (HPG + 2) * D
    seen = {k: set() for k in ("norm", "qkv", "attn", "oproj", "up", "down", "lm")}
    slices = {}
    for s in range(n_sm):
        lm_run = []
        for i in range(max_pc):
            I = q[s * max_pc + i]
            if I.op == 0:
                break
            rows = I.r1 - I.r0
            if I.op == 10:
                key = (I.layer, I.g, I.r0)
                assert key not in seen["norm"] and rows == 1 and I.r0 < Bp
                seen["norm"].add(key)
            elif I.op == 1:
                assert I.r0 % 8 == 0 and 0 < rows <= 128
                for r in range(I.r0, I.r1):
                    assert (I.layer, r) not in seen["qkv"]
                    seen["qkv"].add((I.layer, r))
            elif I.op == 2:
                key = (I.layer, I.b, I.g, I.r0)
                assert key not in seen["attn"] and I.r1 == splits
                seen["attn"].add(key)
            elif I.op == 3:  # a kv group's heads
                assert I.r0 % 8 == 0 and 0 < rows <= 128 and I.g < Hkv
                assert bool(I.flags & 1) == (I.g == 0)
                for h in range(I.g * HPG, (I.g + 1) * HPG):
                    for r in range(I.r0, I.r1):
                        assert (I.layer, h, r) not in seen["oproj"]
                        seen["oproj"].add((I.layer, h, r))
            elif I.op == 8:
                assert I.r0 % 4 == 0 and 0 < 2 * rows <= 128
                for c in range(I.r0, I.r1):
                    assert (I.layer, c) not in seen["up"]
                    seen["up"].add((I.layer, c))
            elif I.op == 9:  # rows x FFN chunks [b, g)
                assert I.r0 % 8 == 0 and 0 < rows <= 128 and I.b < I.g <= F // 64
                for r in range(I.r0, I.r1):
                    for k in range(I.b, I.g):
                        assert (I.layer, r, k) not in seen["down"]
                        seen["down"].add((I.layer, r, k))
            elif I.op == 5:
                assert I.r0 % 8 == 0 and 0 < rows <= 128
                lm_run.append((i, I))
                for r in range(I.r0, I.r1):
                    assert r not in seen["lm"]
                    seen["lm"].add(r)
            else:
                raise AssertionError(f"op {I.op} in a wide plan")
        if lm_run:
            idx = [i for i, _ in lm_run]
            assert idx == list(range(idx[0], idx[0] + len(idx)))  # consecutive
            assert len({I.aux for _, I in lm_run}) == 1
            assert [I.b for _, I in lm_run] == ([3] if len(lm_run) == 1 else
                                               [1] + [0] * (len(lm_run) - 2) + [2])
            assert lm_run[0][1].aux not in slices
            slices[lm_run[0][1].aux] = s
    assert len(seen["norm"]) == (2 * Lc + 1) * Bp
    assert len(seen["qkv"]) == Lc * R
    assert len(seen["attn"]) == Lc * B * Hkv * splits
    assert len(seen["oproj"]) == Lc * Hq * H
    assert len(seen["up"]) == Lc * F
    assert len(seen["down"]) == Lc * H * (F // 64)
    assert len(seen["lm"]) == V
    assert sorted(slices) == list(range(len(slices)))


@pytest.mark.parametrize("batch", [2, 7, 9, 16, 32])
@pytest.mark.parametrize("n_sm", [1, 7, 148, 152])
def test_wide_plan_covers_all_work_and_is_deadlock_free(batch, n_sm):
    cfg, d = desc("llama1b_b8", batch=batch)
    st, q = L.mk_plan(d, batch, cfg["max_seq"], n_sm)
    # as many slices as keep the items at one per SM, at most 4, at least 16
    # positions each
    pairs = batch * cfg["n_kv_heads"]
    assert st["attn_splits"] == min(min(4, max(1, n_sm // pairs)), max(1, cfg["max_seq"] // 16))
    wide_coverage(cfg, q, n_sm, st["max_pc"], st["attn_splits"])
    assert st["n_lm"] == min(n_sm, cfg["vocab"] // 8)
    assert L.mk_plan_check(q, n_sm, st["max_pc"], st["n_counters"]) == L.MK_OK


def test_wide_plan_ragged_shape():
    # 17 FFN chunks, a vocabulary that is not a multiple of 8, 13 sequences
    cfg, d = desc("llama1b_b8", batch=13, n_layers=3, ffn=1088, vocab=5001)
    st, q = L.mk_plan(d, 13, cfg["max_seq"], 152)
    wide_coverage(cfg, q, 152, st["max_pc"], st["attn_splits"])
    assert L.mk_plan_check(q, 152, st["max_pc"], st["n_counters"]) == L.MK_OK


def test_wide_shapes_outside_the_variant_are_refused():
    # the wide variant needs a dense FFN of whole 64-column chunks
    cfg, d = desc("llama1b_b8", batch=16, ffn=1000)
    with pytest.raises(L.MkError):
        L.mk_plan(d, 16, cfg["max_seq"], 152)

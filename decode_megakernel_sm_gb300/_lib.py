"""ctypes binding of libmk.so (include/mk.h).  Argument marshalling only:
every step of the decode path runs in the library's CUDA kernels.  There is
no fallback -- if the library is missing and cannot be built, import of the
entry points raises."""
from __future__ import annotations

import ctypes as C
import os
import threading

from . import build as _build

MK_OK = 0
MK_ERR_INVALID_ARG = -1
MK_ERR_CUDA = -2
MK_ERR_UNSUPPORTED = -3
MK_ERR_SCHEDULE = -4
MK_ERR_TIMEOUT = -5
MK_ERR_NOT_READY = -6
MK_ERR_DEVICE = -7
MK_ERR_SCRATCH = -8
MK_ERR_BOUNDS = -9
MK_ABL_STREAM, MK_ABL_GRAPH, MK_ABL_PDL = 0, 1, 2
MK_WEIGHTS_BF16, MK_WEIGHTS_INT8 = 0, 1

OP_NAMES = {0: "HALT", 1: "QKV", 2: "ATTN", 3: "OPROJ", 4: "MLP", 5: "LMHEAD", 6: "ROUTER", 8: "MLP_UP", 9: "MLP_DOWN", 10: "NORM",
            7: "NOP"}


class mk_model_desc(C.Structure):
    _fields_ = [(n, C.c_int) for n in ("n_layers", "hidden", "n_q_heads", "n_kv_heads",
                                        "head_dim", "ffn", "vocab")] + \
               [("rms_eps", C.c_float), ("rope_theta", C.c_float)] + \
               [(n, C.c_int) for n in ("tied_lm_head", "n_experts", "top_k", "expert_ffn",
                                        "shared_ffn", "max_batch", "max_seq",
                                        "batched_variant")]


WEIGHT_LISTS = ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "w_gate", "w_up", "w_down",
                "router", "ex_gate", "ex_up", "ex_down", "sh_gate", "sh_up", "sh_down")


class mk_weights(C.Structure):
    _fields_ = [("embed", C.c_void_p), ("lm_head", C.c_void_p), ("final_norm", C.c_void_p)] + \
               [(n, C.POINTER(C.c_void_p)) for n in WEIGHT_LISTS]


class mk_kv(C.Structure):
    _fields_ = [("k", C.POINTER(C.c_void_p)), ("v", C.POINTER(C.c_void_p))]


class mk_info(C.Structure):
    _fields_ = [(n, C.c_int) for n in ("n_sm", "stage_bytes", "n_stages", "smem_bytes", "max_pc",
                                        "n_instr", "n_counters", "attn_splits",
                                        "launches_per_step", "ablation_launches", "batch",
                                        "max_ctx")] + \
               [("packed_bytes", C.c_size_t), ("scratch_bytes", C.c_size_t),
                ("weight_bytes_per_step", C.c_double)]


class mk_instr(C.Structure):
    _fields_ = [("op", C.c_uint8), ("flags", C.c_uint8), ("layer", C.c_uint16),
                ("b", C.c_uint16), ("g", C.c_uint16), ("r0", C.c_uint32), ("r1", C.c_uint32),
                ("wait_ctr", C.c_uint32), ("wait_cnt", C.c_uint32), ("sig_ctr", C.c_uint32),
                ("aux", C.c_uint32)]


class mk_plan_stats(C.Structure):
    _fields_ = [(n, C.c_int) for n in ("n_sm", "max_pc", "n_instr", "n_counters", "attn_splits",
                                        "n_lm")] + \
               [("max_sm_bytes", C.c_double), ("mean_sm_bytes", C.c_double)]


class MkError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {mk_status_string(status)} ({status})")


_lock = threading.Lock()
_lib = None

SIGNATURES = {
    "mk_create": (C.c_int, [C.POINTER(mk_model_desc), C.POINTER(mk_weights), C.POINTER(mk_kv),
                            C.POINTER(C.c_void_p)]),
    "mk_create_ex": (C.c_int, [C.POINTER(mk_model_desc), C.POINTER(mk_weights), C.POINTER(mk_kv),
                               C.c_int, C.POINTER(C.c_void_p)]),
    "mk_quantize_rows_int8": (C.c_int, [C.c_void_p, C.c_long, C.c_int, C.c_void_p, C.c_void_p,
                                        C.c_void_p]),
    "mk_build_schedule": (C.c_int, [C.c_void_p, C.c_int, C.c_int]),
    "mk_decode_step": (C.c_int, [C.c_void_p] * 6),
    "mk_decode_steps": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_int, C.c_void_p,
                                  C.c_void_p, C.c_void_p]),
    "mk_decode_step_host": (C.c_int, [C.c_void_p] * 5),
    "mk_decode_step_ablation": (C.c_int, [C.c_void_p, C.c_int] + [C.c_void_p] * 5),
    "mk_decode_step_noalloc": (C.c_int, [C.c_void_p] * 7),
    "mk_sync_status": (C.c_int, [C.c_void_p, C.c_void_p]),
    "mk_set_wait_timeout": (C.c_int, [C.c_void_p, C.c_uint64]),
    "mk_get_info": (C.c_int, [C.c_void_p, C.POINTER(mk_info)]),
    "mk_debug_drop_instruction": (C.c_int, [C.c_void_p, C.c_int, C.c_int]),
    "mk_get_routes": (C.c_int, [C.c_void_p, C.POINTER(C.c_int32), C.c_size_t]),
    "mk_set_trace": (C.c_int, [C.c_void_p, C.c_int]),
    "mk_set_l2_prefetch": (C.c_int, [C.c_void_p, C.c_uint64]),
    "mk_set_residual_copies": (C.c_int, [C.c_void_p, C.c_int]),
    "mk_set_stage_bytes": (C.c_int, [C.c_void_p, C.c_int]),
    "mk_set_ring_depth": (C.c_int, [C.c_void_p, C.c_int]),
    "mk_set_kv_pages": (C.c_int, [C.c_void_p, C.c_int, C.c_int, C.c_void_p, C.c_int]),
    "mk_set_race_stress": (C.c_int, [C.c_void_p, C.c_uint, C.c_uint, C.c_int]),
    "mk_debug_read": (C.c_int, [C.c_void_p, C.c_int, C.c_int, C.c_void_p, C.c_size_t]),
    "mk_set_poll_policy": (C.c_int, [C.c_void_p, C.c_int, C.c_uint]),
    "mk_set_hold_policy": (C.c_int, [C.c_void_p, C.c_uint, C.c_uint64]),
    "mk_get_trace": (C.c_int, [C.c_void_p, C.POINTER(C.c_uint64), C.c_size_t]),
    "mk_destroy": (C.c_int, [C.c_void_p]),
    "mk_status_string": (C.c_char_p, [C.c_int]),
    "mk_plan": (C.c_int, [C.POINTER(mk_model_desc), C.c_int, C.c_int, C.c_int,
                          C.POINTER(mk_plan_stats), C.POINTER(mk_instr), C.c_size_t]),
    "mk_plan_check": (C.c_int, [C.POINTER(mk_instr), C.c_int, C.c_int, C.c_int]),
}


def lib():
    """Load libmk.so (building it in-tree first if it is missing or stale); with
    MK_LIB=bounds in the environment, the bounds-checked libmk_bounds.so."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB_BOUNDS if os.environ.get("MK_LIB") == "bounds" else _build.LIB
            if not _build.up_to_date():
                try:
                    _build.build()
                except Exception as e:  # no silent fallback: the CUDA path is the product
                    raise RuntimeError(f"libmk.so is missing and could not be built: {e}") from e
            L = C.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                f = getattr(L, name)
                f.restype = res
                f.argtypes = args
            _lib = L
    return _lib


def lib_path() -> str:
    return os.path.abspath(_build.LIB)


def mk_status_string(status: int) -> str:
    return lib().mk_status_string(status).decode()


def _check(status: int, what: str):
    if status != MK_OK:
        raise MkError(status, what)


def mk_create(desc: mk_model_desc, weights: mk_weights, kv: mk_kv) -> int:
    h = C.c_void_p()
    _check(lib().mk_create(C.byref(desc), C.byref(weights), C.byref(kv), C.byref(h)), "mk_create")
    return h.value


def mk_create_ex(desc: mk_model_desc, weights: mk_weights, kv: mk_kv, weight_format: int) -> int:
    h = C.c_void_p()
    _check(lib().mk_create_ex(C.byref(desc), C.byref(weights), C.byref(kv), weight_format,
                              C.byref(h)), "mk_create_ex")
    return h.value


def mk_quantize_rows_int8(d_w, rows: int, cols: int, d_codes, d_scales, stream=None):
    _check(lib().mk_quantize_rows_int8(d_w, rows, cols, d_codes, d_scales, stream),
           "mk_quantize_rows_int8")


def mk_build_schedule(h, batch: int, max_ctx: int):
    _check(lib().mk_build_schedule(h, batch, max_ctx), "mk_build_schedule")


def mk_decode_step(h, d_tokens, d_positions, d_logits, d_argmax, stream=None):
    _check(lib().mk_decode_step(h, d_tokens, d_positions, d_logits, d_argmax, stream),
           "mk_decode_step")


def mk_decode_steps(h, d_tokens, d_positions, n_steps: int, d_logits, d_argmax, stream=None):
    _check(lib().mk_decode_steps(h, d_tokens, d_positions, int(n_steps), d_logits, d_argmax,
                                 stream), "mk_decode_steps")


def mk_decode_step_host(h, h_tokens, h_positions, h_logits, h_argmax) -> int:
    """Host-buffer step; returns the status (device errors are statuses, not raises)."""
    return lib().mk_decode_step_host(h, h_tokens, h_positions, h_logits, h_argmax)


def mk_decode_step_ablation(h, mode, d_tokens, d_positions, d_logits, d_argmax, stream=None):
    _check(lib().mk_decode_step_ablation(h, mode, d_tokens, d_positions, d_logits, d_argmax,
                                         stream), "mk_decode_step_ablation")


def mk_decode_step_noalloc(h, d_tokens, d_positions, d_logits, d_argmax, d_status=None,
                           stream=None) -> int:
    """The decode step with its scratch in the library's fixed device array (no
    allocation anywhere); returns the status of the call itself."""
    return lib().mk_decode_step_noalloc(h, d_tokens, d_positions, d_logits, d_argmax, d_status,
                                        stream)


def mk_sync_status(h, stream=None) -> int:
    return lib().mk_sync_status(h, stream)


def mk_set_wait_timeout(h, ns: int):
    _check(lib().mk_set_wait_timeout(h, ns), "mk_set_wait_timeout")


def mk_get_info(h) -> dict:
    info = mk_info()
    _check(lib().mk_get_info(h, C.byref(info)), "mk_get_info")
    return {n: getattr(info, n) for n, _ in mk_info._fields_}


def mk_get_routes(h, n_layers: int, top_k: int):
    """Expert ids chosen at the last step, numpy int32 [n_layers][top_k]."""
    import numpy as np
    out = np.zeros((n_layers, top_k), np.int32)
    _check(lib().mk_get_routes(h, out.ctypes.data_as(C.POINTER(C.c_int32)), out.size),
           "mk_get_routes")
    return out


def mk_debug_drop_instruction(h, sm: int, pc: int):
    _check(lib().mk_debug_drop_instruction(h, sm, pc), "mk_debug_drop_instruction")


def mk_set_l2_prefetch(h, bytes_ahead: int):
    _check(lib().mk_set_l2_prefetch(h, int(bytes_ahead)), "mk_set_l2_prefetch")


def mk_set_residual_copies(h, copies: int):
    _check(lib().mk_set_residual_copies(h, int(copies)), "mk_set_residual_copies")


def mk_set_poll_policy(h, pollers: int, stagger_ns: int):
    _check(lib().mk_set_poll_policy(h, int(pollers), int(stagger_ns)), "mk_set_poll_policy")


MK_DBG_Q, MK_DBG_X, MK_DBG_H = 0, 1, 2


def mk_debug_read(h, what: int, layer: int, out) -> None:
    """out: a C-contiguous float32 numpy array of the intermediate's size."""
    _check(lib().mk_debug_read(h, int(what), int(layer), out.ctypes.data_as(C.c_void_p),
                               out.size), "mk_debug_read")


def mk_set_race_stress(h, max_delay_ns: int, seed: int, permute_queues: bool):
    _check(lib().mk_set_race_stress(h, int(max_delay_ns), int(seed), int(bool(permute_queues))),
           "mk_set_race_stress")


def mk_set_kv_pages(h, block: int, n_blocks: int, d_table, table_stride: int):
    _check(lib().mk_set_kv_pages(h, int(block), int(n_blocks), d_table, int(table_stride)),
           "mk_set_kv_pages")


def mk_set_ring_depth(h, max_stages: int):
    _check(lib().mk_set_ring_depth(h, int(max_stages)), "mk_set_ring_depth")


def mk_set_stage_bytes(h, stage_bytes: int):
    _check(lib().mk_set_stage_bytes(h, int(stage_bytes)), "mk_set_stage_bytes")


def mk_set_hold_policy(h, mask: int, early_bytes: int):
    _check(lib().mk_set_hold_policy(h, int(mask), int(early_bytes)), "mk_set_hold_policy")


def mk_set_trace(h, on: bool):
    _check(lib().mk_set_trace(h, 1 if on else 0), "mk_set_trace")


def mk_get_trace(h, n_sm: int, max_pc: int):
    """Returns a numpy uint64 array [n_sm][max_pc][8] of %globaltimer stamps."""
    import numpy as np
    out = np.zeros((n_sm, max_pc, 8), np.uint64)
    _check(lib().mk_get_trace(h, out.ctypes.data_as(C.POINTER(C.c_uint64)), out.size),
           "mk_get_trace")
    return out


def mk_destroy(h):
    _check(lib().mk_destroy(h), "mk_destroy")


def mk_plan(desc: mk_model_desc, batch: int, max_ctx: int, n_sm: int, with_queues=True):
    """Host-only schedule build; returns (stats dict, queue array or None)."""
    st = mk_plan_stats()
    _check(lib().mk_plan(C.byref(desc), batch, max_ctx, n_sm, C.byref(st), None, 0), "mk_plan")
    stats = {n: getattr(st, n) for n, _ in mk_plan_stats._fields_}
    if not with_queues:
        return stats, None
    q = (mk_instr * (st.n_sm * st.max_pc))()
    _check(lib().mk_plan(C.byref(desc), batch, max_ctx, n_sm, None, q, len(q)), "mk_plan")
    return stats, q


def mk_plan_check(q, n_sm: int, max_pc: int, n_counters: int) -> int:
    return lib().mk_plan_check(q, n_sm, max_pc, n_counters)

"""Plain CPU reference decoder (the oracle) -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the cpu_baseline / reference
leg of ``bench.py`` may import this package.  The product package
``decode_megakernel_sm_gb300`` never imports it, and this package never
imports the product.  The arithmetic lives in ``oracle.c`` (fp64, bf16 inputs
widened exactly); this module only compiles it with gcc and marshals numpy
arrays through ctypes.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, OpenMP)."""
    stale = (not os.path.exists(_LIB_PATH)) or (
        os.path.getmtime(_LIB_PATH) < max(os.path.getmtime(_SRC),
                                          os.path.getmtime(os.path.join(_HERE, "oracle.h"))))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-std=c11", "-O2", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class OrcConfig(C.Structure):
    _fields_ = [(n, C.c_int) for n in ("n_layers", "hidden", "n_q_heads", "n_kv_heads",
                                        "head_dim", "ffn", "vocab")] + \
               [("rms_eps", C.c_double), ("rope_theta", C.c_double)] + \
               [(n, C.c_int) for n in ("n_experts", "top_k", "expert_ffn", "shared_ffn",
                                        "max_seq")]


_WFIELDS = ("attn_norm", "wq", "wk", "wv", "wo", "mlp_norm", "w_gate", "w_up", "w_down",
            "router", "ex_gate", "ex_up", "ex_down", "sh_gate", "sh_up", "sh_down")


class OrcWeights(C.Structure):
    _fields_ = [("embed", C.c_void_p), ("lm_head", C.c_void_p), ("final_norm", C.c_void_p)] + \
               [(n, C.POINTER(C.c_void_p)) for n in _WFIELDS] + [("q8", C.c_void_p)]


class OrcQmat(C.Structure):
    _fields_ = [("codes", C.c_void_p), ("scales", C.c_void_p)]


_QFIELDS = ("wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down")


class OrcQ8(C.Structure):
    _fields_ = [(n, C.POINTER(OrcQmat)) for n in _QFIELDS] + [("lm_head", OrcQmat)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = C.CDLL(_LIB_PATH)
            dp = C.POINTER(C.c_double)
            u16p = C.POINTER(C.c_uint16)
            ip = C.POINTER(C.c_int)
            L.orc_bf16_to_f64.restype = C.c_double
            L.orc_bf16_to_f64.argtypes = [C.c_uint16]
            L.orc_f64_to_bf16.restype = C.c_uint16
            L.orc_f64_to_bf16.argtypes = [C.c_double]
            L.orc_rmsnorm.argtypes = [dp, u16p, C.c_int, C.c_double, dp]
            L.orc_rope.argtypes = [dp, C.c_int, C.c_int, C.c_double]
            L.orc_gemv.argtypes = [u16p, C.c_int, C.c_int, dp, dp]
            L.orc_attention.argtypes = [dp, u16p, u16p, C.c_int, C.c_int, dp]
            L.orc_attention_partial.argtypes = [dp, u16p, u16p, C.c_int, C.c_int, C.c_int, dp,
                                                dp, dp]
            L.orc_attention_merge.argtypes = [C.c_int, dp, dp, dp, C.c_int, dp]
            L.orc_silu.restype = C.c_double
            L.orc_silu.argtypes = [C.c_double]
            L.orc_swiglu.argtypes = [u16p, u16p, u16p, C.c_int, C.c_int, dp, dp]
            L.orc_router_topk.restype = C.c_double
            L.orc_router_topk.argtypes = [dp, C.c_int, C.c_int, ip, dp]
            L.orc_argmax.restype = C.c_int
            L.orc_argmax.argtypes = [dp, C.c_int]
            L.orc_quantize_rows_int8.argtypes = [u16p, C.c_int, C.c_int, C.c_void_p, C.c_void_p]
            L.orc_gemv_q8.argtypes = [C.c_void_p, C.c_void_p, C.c_int, C.c_int, dp, dp]
            L.orc_decode_step_trace.restype = C.c_int
            L.orc_decode_step_trace.argtypes = [C.POINTER(OrcConfig), C.POINTER(OrcWeights),
                                                C.POINTER(C.c_void_p), C.POINTER(C.c_void_p),
                                                C.c_int, ip, ip, dp, ip, ip, dp, ip, ip, dp, dp,
                                                dp]
            L.orc_decode_step.restype = C.c_int
            L.orc_decode_step.argtypes = [C.POINTER(OrcConfig), C.POINTER(OrcWeights),
                                          C.POINTER(C.c_void_p), C.POINTER(C.c_void_p),
                                          C.c_int, ip, ip, dp, ip, ip, dp, ip, ip]
            L.orc_set_threads.argtypes = [C.c_int]
            L.orc_get_threads.restype = C.c_int
            _lib = L
    return _lib


def _dp(a):
    return a.ctypes.data_as(C.POINTER(C.c_double))


def _u16(a):
    assert a.dtype == np.uint16 and a.flags.c_contiguous
    return a.ctypes.data_as(C.POINTER(C.c_uint16))


def _ip(a):
    assert a.dtype == np.int32 and a.flags.c_contiguous
    return a.ctypes.data_as(C.POINTER(C.c_int))


def f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


# ---- single operations (used by the pin tests) ------------------------------------------
def bf16_to_f64(bits: int) -> float:
    return lib().orc_bf16_to_f64(bits)


def f64_to_bf16(x: float) -> int:
    return lib().orc_f64_to_bf16(x)


def rmsnorm(x, gain_bits, eps):
    x = f64(x)
    out = np.empty_like(x)
    lib().orc_rmsnorm(_dp(x), _u16(gain_bits), x.size, eps, _dp(out))
    return out


def rope(v, pos, theta):
    v = f64(v).copy()
    lib().orc_rope(_dp(v), v.size, pos, theta)
    return v


def gemv(W_bits, x):
    rows, cols = W_bits.shape
    x = f64(x)
    y = np.empty(rows)
    lib().orc_gemv(_u16(W_bits), rows, cols, _dp(x), _dp(y))
    return y


def quantize_rows_int8(W_bits):
    """Per-row int8 codes [rows][cols] (int8) and scales [rows] (float32) of a
    bf16 matrix given as uint16 bits."""
    W = np.ascontiguousarray(W_bits, np.uint16)
    rows, cols = W.shape
    q = np.empty((rows, cols), np.int8)
    s = np.empty(rows, np.float32)
    lib().orc_quantize_rows_int8(_u16(W), rows, cols, q.ctypes.data_as(C.c_void_p),
                                 s.ctypes.data_as(C.c_void_p))
    return q, s


def gemv_q8(codes, scales, x):
    q = np.ascontiguousarray(codes, np.int8)
    s = np.ascontiguousarray(scales, np.float32)
    xx = f64(x)
    y = np.empty(q.shape[0])
    lib().orc_gemv_q8(q.ctypes.data_as(C.c_void_p), s.ctypes.data_as(C.c_void_p), q.shape[0],
                      q.shape[1], _dp(xx), _dp(y))
    return y


def attention(q, K_bits, V_bits):
    q = f64(q)
    out = np.empty(q.size)
    lib().orc_attention(_dp(q), _u16(K_bits), _u16(V_bits), K_bits.shape[0], q.size, _dp(out))
    return out


def attention_partial(q, K_bits, V_bits, p0, p1):
    q = f64(q)
    m, l = C.c_double(), C.c_double()
    o = np.empty(q.size)
    lib().orc_attention_partial(_dp(q), _u16(K_bits), _u16(V_bits), p0, p1, q.size,
                                C.byref(m), C.byref(l), _dp(o))
    return m.value, l.value, o


def attention_merge(m, l, o):
    m, l, o = f64(m), f64(l), f64(o)
    out = np.empty(o.shape[1])
    lib().orc_attention_merge(m.size, _dp(m), _dp(l), _dp(o), o.shape[1], _dp(out))
    return out


def silu(a):
    return lib().orc_silu(a)


def swiglu(wg_bits, wu_bits, wd_bits, xn):
    F, H = wg_bits.shape
    xn = f64(xn)
    y = np.empty(H)
    lib().orc_swiglu(_u16(wg_bits), _u16(wu_bits), _u16(wd_bits), F, H, _dp(xn), _dp(y))
    return y


def router_topk(logits, k):
    logits = f64(logits)
    ids = np.empty(k, np.int32)
    w = np.empty(k)
    margin = lib().orc_router_topk(_dp(logits), logits.size, k, _ip(ids), _dp(w))
    return ids, w, margin


def argmax(v):
    v = f64(v)
    return lib().orc_argmax(_dp(v), v.size)


def set_threads(n: int):
    lib().orc_set_threads(n)


def get_threads() -> int:
    return lib().orc_get_threads()


# ---- whole decode step -------------------------------------------------------------------
def _bits(t):
    """numpy uint16 view of a bf16 array (numpy uint16 or a CPU torch bf16 tensor)."""
    if isinstance(t, np.ndarray):
        assert t.dtype == np.uint16
        return np.ascontiguousarray(t)
    import torch  # only for the bf16 -> uint16 reinterpretation of CPU tensors
    assert t.dtype == torch.bfloat16 and t.device.type == "cpu"
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


class OracleModel:
    """Holds host copies of the weights and runs ``orc_decode_step``.

    ``weights`` is the dict produced by ``synth.make_weights`` (bf16 tensors
    on any device are accepted; they are copied to host once).  ``int8``:
    quantise every streamed matrix with ``orc_quantize_rows_int8`` and decode
    with the int8 weights (dense models)."""

    def __init__(self, cfg: dict, weights: dict, int8: bool = False):
        self.cfg = cfg
        self._keep = []
        c = OrcConfig()
        for n in ("n_layers", "hidden", "n_q_heads", "n_kv_heads", "head_dim", "ffn", "vocab",
                  "n_experts", "top_k", "expert_ffn", "shared_ffn"):
            setattr(c, n, int(cfg.get(n, 0)))
        c.rms_eps = float(cfg["rms_eps"])
        c.rope_theta = float(cfg["rope_theta"])
        c.max_seq = int(cfg["max_seq"])
        self.c = c
        w = OrcWeights()
        embed = self._host(weights["embed"])
        w.embed = embed.ctypes.data
        w.lm_head = embed.ctypes.data if weights.get("lm_head") is None else \
            self._host(weights["lm_head"]).ctypes.data
        w.final_norm = self._host(weights["final_norm"]).ctypes.data
        L = cfg["n_layers"]
        for n in _WFIELDS:
            arr = (C.c_void_p * L)()
            for l in range(L):
                t = weights["layers"][l].get(n)
                arr[l] = None if t is None else self._host(t).ctypes.data
            self._keep.append(arr)
            setattr(w, n, C.cast(arr, C.POINTER(C.c_void_p)))
        w.q8 = None
        if int8:
            assert cfg.get("n_experts", 0) == 0, "int8 weights: dense models"
            q8 = OrcQ8()
            for n in _QFIELDS:
                mats = (OrcQmat * L)()
                for l in range(L):
                    mats[l] = self._qmat(weights["layers"][l][n])
                self._keep.append(mats)
                setattr(q8, n, C.cast(mats, C.POINTER(OrcQmat)))
            lm = weights["embed"] if weights.get("lm_head") is None else weights["lm_head"]
            q8.lm_head = self._qmat(lm)
            self._keep.append(q8)
            w.q8 = C.addressof(q8)
        self.w = w

    def _qmat(self, t):
        q, s = quantize_rows_int8(self._host(t))
        self._keep += [q, s]
        return OrcQmat(q.ctypes.data, s.ctypes.data)

    def _host(self, t):
        if not isinstance(t, np.ndarray):
            t = t.detach().to("cpu")
        a = _bits(t)
        self._keep.append(a)
        return a

    def step(self, kc, vc, tokens, positions, forced_routes=None, forced_mask=None,
             trace=None):
        """kc/vc: lists (per layer) of uint16 arrays [B][Hkv][max_seq][d], updated in
        place.  Returns (logits [B][V] float64, argmax [B] int32, route_ids, margins).
        trace: a dict that receives the intermediates q [L][B][Hq*d] (after RoPE),
        x [2L][B][H] (residual after each O-projection and each MLP) and, for dense
        models, h [L][B][F]."""
        cfg = self.cfg
        B = len(tokens)
        L = cfg["n_layers"]
        kp = (C.c_void_p * L)(*[a.ctypes.data for a in kc])
        vp = (C.c_void_p * L)(*[a.ctypes.data for a in vc])
        tok = np.ascontiguousarray(tokens, np.int32)
        pos = np.ascontiguousarray(positions, np.int32)
        logits = np.empty((B, cfg["vocab"]))
        am = np.empty(B, np.int32)
        moe = cfg.get("n_experts", 0) > 0
        rid = np.zeros((L, B, max(cfg.get("top_k", 0), 1)), np.int32) if moe else None
        rmg = np.zeros((L, B)) if moe else None
        fr = None if forced_routes is None else np.ascontiguousarray(forced_routes, np.int32)
        fm = None if forced_mask is None else np.ascontiguousarray(forced_mask, np.int32)
        if trace is not None:
            H, Hq, d = cfg["hidden"], cfg["n_q_heads"], cfg["head_dim"]
            tq = np.zeros((L, B, Hq * d))
            tx = np.zeros((2 * L, B, H))
            th = np.zeros((L, B, max(cfg.get("ffn", 0), 1)))
            rc = lib().orc_decode_step_trace(
                C.byref(self.c), C.byref(self.w), C.cast(kp, C.POINTER(C.c_void_p)),
                C.cast(vp, C.POINTER(C.c_void_p)), B, _ip(tok), _ip(pos), _dp(logits), _ip(am),
                None if rid is None else _ip(rid), None if rmg is None else _dp(rmg),
                None if fr is None else _ip(fr), None if fm is None else _ip(fm), _dp(tq),
                _dp(tx), _dp(th) if not moe else None)
            trace.update(q=tq, x=tx, h=None if moe else th)
        else:
            rc = lib().orc_decode_step(
                C.byref(self.c), C.byref(self.w), C.cast(kp, C.POINTER(C.c_void_p)),
                C.cast(vp, C.POINTER(C.c_void_p)), B, _ip(tok), _ip(pos), _dp(logits), _ip(am),
                None if rid is None else _ip(rid), None if rmg is None else _dp(rmg),
                None if fr is None else _ip(fr), None if fm is None else _ip(fm))
        if rc != 0:
            raise ValueError("oracle: invalid argument")
        return logits, am, rid, rmg

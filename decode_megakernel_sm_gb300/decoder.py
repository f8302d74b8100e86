"""Decoder: a thin object over the C ABI that keeps the caller's tensors alive
and marshals torch CUDA tensors to device pointers.  No arithmetic here."""
from __future__ import annotations

import ctypes as C

import torch

from . import _lib as L


def desc_from_config(cfg: dict, max_batch: int, max_seq: int) -> L.mk_model_desc:
    d = L.mk_model_desc()
    for n in ("n_layers", "hidden", "n_q_heads", "n_kv_heads", "head_dim", "ffn", "vocab",
              "n_experts", "top_k", "expert_ffn", "shared_ffn"):
        setattr(d, n, int(cfg.get(n, 0)))
    d.rms_eps = float(cfg["rms_eps"])
    d.rope_theta = float(cfg["rope_theta"])
    d.tied_lm_head = 1 if cfg.get("tied", True) else 0
    d.max_batch = int(max_batch)
    d.max_seq = int(max_seq)
    d.batched_variant = int(cfg.get("batched_variant", 0))
    return d


def _ptr(t, dtype=None):
    if t is None:
        return None
    if not (isinstance(t, torch.Tensor) and t.is_cuda and t.is_contiguous()):
        raise ValueError("expected a contiguous CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"expected {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return C.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return C.c_void_p(stream.cuda_stream)
    return C.c_void_p(stream)


class Decoder:
    """One megakernel handle for a model whose weights and KV cache are CUDA tensors.

    weights: dict as produced by ``synth.make_weights`` (bf16, [out][in]);
    kcache / vcache: per-layer bf16 tensors [max_batch][Hkv][max_seq][head_dim]."""

    def __init__(self, cfg: dict, weights: dict, kcache, vcache, max_batch=None, max_seq=None,
                 weight_format: str = "bf16"):
        """kcache / vcache may also be paged pools [n_blocks][Hkv][block][head_dim]:
        then pass max_batch and max_seq, and call set_kv_pages before the first step.
        weight_format "int8": the library quantises every streamed matrix per row
        (mk_create_ex with MK_WEIGHTS_INT8)."""
        if max_batch is None or max_seq is None:
            max_batch, _, max_seq, _ = kcache[0].shape
        self.cfg = cfg
        self.desc = desc_from_config(cfg, max_batch, max_seq)
        nl = cfg["n_layers"]
        bf = torch.bfloat16
        w = L.mk_weights()
        w.embed = _ptr(weights["embed"], bf)
        w.lm_head = _ptr(weights.get("lm_head"), bf)
        w.final_norm = _ptr(weights["final_norm"], bf)
        self._arrays = []
        for name in L.WEIGHT_LISTS:
            ts = [lw.get(name) for lw in weights["layers"]]
            if all(t is None for t in ts):
                continue
            arr = (C.c_void_p * nl)(*[_ptr(t, bf) for t in ts])
            self._arrays.append(arr)
            setattr(w, name, C.cast(arr, C.POINTER(C.c_void_p)))
        ka = (C.c_void_p * nl)(*[_ptr(t, bf) for t in kcache])
        va = (C.c_void_p * nl)(*[_ptr(t, bf) for t in vcache])
        self._arrays += [ka, va]
        kv = L.mk_kv(C.cast(ka, C.POINTER(C.c_void_p)), C.cast(va, C.POINTER(C.c_void_p)))
        self.kcache, self.vcache = kcache, vcache  # the library writes row P in place
        fmt = {"bf16": L.MK_WEIGHTS_BF16, "int8": L.MK_WEIGHTS_INT8}[weight_format]
        self.weight_format = weight_format
        self.h = L.mk_create_ex(self.desc, w, kv, fmt)
        self.batch = 0

    # -- schedule ---------------------------------------------------------
    def build_schedule(self, batch: int, max_ctx: int):
        L.mk_build_schedule(self.h, batch, max_ctx)
        self.batch = batch

    def info(self) -> dict:
        return L.mk_get_info(self.h)

    def set_wait_timeout(self, ns: int):
        L.mk_set_wait_timeout(self.h, int(ns))

    def set_residual_copies(self, copies: int):
        """Takes effect at the next build_schedule."""
        L.mk_set_residual_copies(self.h, copies)

    def set_stage_bytes(self, stage_bytes: int):
        """Ring stage size (16, 32, 48 or 64 KiB); takes effect at the next step."""
        L.mk_set_stage_bytes(self.h, stage_bytes)

    def set_poll_policy(self, pollers: int, stagger_ns: int):
        """Warps polling each dependency counter, and their stagger."""
        L.mk_set_poll_policy(self.h, pollers, stagger_ns)

    def set_kv_pages(self, block: int, table):
        """Paged KV cache: table is an int32 CUDA tensor [max_batch][stride] of block ids
        into the pools given at construction (block 0: back to contiguous)."""
        if block == 0:
            L.mk_set_kv_pages(self.h, 0, 0, None, 0)
            self._kv_table = None
            return
        n_blocks = self.kcache[0].shape[0]
        L.mk_set_kv_pages(self.h, block, n_blocks, _ptr(table, torch.int32), table.shape[1])
        self._kv_table = table  # kept alive: the kernel reads it every step

    def debug_read(self, what: str, layer: int):
        """An intermediate of the most recent step as a float32 numpy array:
        "q" [batch][Hq*d] of layer `layer`, "x" [batch][H] the residual x_layer
        (1 .. 2L), "h" [batch][F] of layer `layer` (dense batch 1)."""
        import numpy as np
        c = self.cfg
        width = {"q": c["n_q_heads"] * c["head_dim"], "x": c["hidden"], "h": c["ffn"]}[what]
        out = np.empty((self.batch, width), np.float32)
        L.mk_debug_read(self.h, {"q": L.MK_DBG_Q, "x": L.MK_DBG_X, "h": L.MK_DBG_H}[what], layer,
                        out)
        return out

    def set_race_stress(self, max_delay_ns: int, seed: int = 0, permute_queues: bool = True):
        """Test aid: random delays before every instruction and a random
        queue-to-CTA permutation; results must not change (0 delay and no
        permutation: off)."""
        L.mk_set_race_stress(self.h, max_delay_ns, seed, permute_queues)

    def set_ring_depth(self, max_stages: int):
        """At most max_stages ring stages (0: as many as fit)."""
        L.mk_set_ring_depth(self.h, max_stages)

    def set_hold_policy(self, mask: int, early_bytes: int = 128 << 10):
        """Takes effect at the next build_schedule."""
        L.mk_set_hold_policy(self.h, mask, early_bytes)

    def set_l2_prefetch(self, bytes_ahead: int):
        L.mk_set_l2_prefetch(self.h, bytes_ahead)

    def set_trace(self, on: bool):
        L.mk_set_trace(self.h, on)

    def get_trace(self):
        """(stamps [n_sm][max_pc][8], host copy of the queues) of the last traced launch."""
        info = self.info()
        tr = L.mk_get_trace(self.h, info["n_sm"], info["max_pc"])
        _, q = L.mk_plan(self.desc, info["batch"], info["max_ctx"], info["n_sm"])
        return tr, q, info["n_sm"], info["max_pc"]

    def routes(self):
        """MoE: expert ids chosen at the last step, [n_layers][top_k]."""
        return L.mk_get_routes(self.h, self.cfg["n_layers"], self.cfg["top_k"])

    def drop_instruction(self, sm: int, pc: int):
        L.mk_debug_drop_instruction(self.h, sm, pc)

    # -- steps ------------------------------------------------------------
    def step(self, tokens, positions, logits, argmax, stream=None):
        """Device-buffer step (asynchronous): int32 tokens/positions [B], fp32 logits
        [B][V], int32 argmax [B]."""
        i32 = torch.int32
        L.mk_decode_step(self.h, _ptr(tokens, i32), _ptr(positions, i32),
                         _ptr(logits, torch.float32), _ptr(argmax, i32), _stream(stream))

    def steps(self, tokens, positions, n_steps, logits, argmax, stream=None):
        """n_steps greedy steps in one launch (asynchronous): int32 tokens/positions [B]
        for the first step, fp32 logits [B][V] of the last step, int32 argmax
        [n_steps][B] of every step."""
        i32 = torch.int32
        if argmax.numel() < n_steps * len(tokens):
            raise ValueError("argmax needs n_steps x batch entries")
        L.mk_decode_steps(self.h, _ptr(tokens, i32), _ptr(positions, i32), n_steps,
                          _ptr(logits, torch.float32), _ptr(argmax, i32), _stream(stream))

    def step_ablation(self, mode, tokens, positions, logits, argmax, stream=None):
        i32 = torch.int32
        L.mk_decode_step_ablation(self.h, mode, _ptr(tokens, i32), _ptr(positions, i32),
                                  _ptr(logits, torch.float32), _ptr(argmax, i32),
                                  _stream(stream))

    def step_host(self, tokens, positions, logits, argmax) -> int:
        """Host-buffer step (synchronous).  Accepts CPU int32 / fp32 tensors (pinned
        for speed); logits may be None.  Returns the status."""
        def hp(t, dt):
            if t is None:
                return None
            if t.device.type != "cpu" or t.dtype != dt or not t.is_contiguous():
                raise ValueError("expected a contiguous CPU tensor of " + str(dt))
            return t.data_ptr()
        return L.mk_decode_step_host(self.h, hp(tokens, torch.int32), hp(positions, torch.int32),
                                     hp(logits, torch.float32), hp(argmax, torch.int32))

    def sync_status(self, stream=None) -> int:
        return L.mk_sync_status(self.h, _stream(stream))

    def close(self):
        if self.h:
            L.mk_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

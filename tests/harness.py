"""Parity harness: run the CUDA decode path and the CPU oracle on the same seeded
inputs, teacher-forcing the oracle with the GPU's emitted tokens.

MoE routing: where the oracle's k-th vs (k+1)-th router probability margin is
below 1e-4 (relative) the oracle adopts the GPU's expert ids for that layer;
everywhere else the chosen expert sets must be identical.

Acceptance per step and sequence (the decode contract):
  * max |logit_gpu - logit_oracle| <= 2e-2 * std(logit_oracle);
  * argmax_gpu == argmax_oracle wherever the oracle's top-2 margin > 5e-2;
  * argmax_gpu is exactly the first index of the maximum of the GPU's own logits;
  * the K/V rows appended at P match the oracle's bf16 rows to one bf16 ulp.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import synth
from decode_megakernel_sm_gb300 import Decoder

TOL = 2e-2
MARGIN = 5e-2
ROUTE_TIE = 1e-4


class Run:
    def __init__(self, cfg: dict, seed: int = 0, max_ctx: int | None = None,
                 stage_bytes: int | None = None, hold: tuple | None = None,
                 paged: int | None = None, int8: bool = False, stress: tuple | None = None):
        cfg = cfg if "max_seq" in cfg else synth.with_cache(cfg)
        self.cfg = cfg
        self.W = synth.make_weights(cfg, seed, "cuda")
        self.lengths = synth.make_lengths(cfg, seed)
        self.ks, self.vs = synth.make_kv(cfg, self.lengths, seed, "cuda")
        torch.cuda.synchronize()
        self.ko = [oracle._bits(t.cpu()).copy() for t in self.ks]
        self.vo = [oracle._bits(t.cpu()).copy() for t in self.vs]
        # int8: each side quantises the same bf16 weights itself (the library
        # on the device, the oracle on the host)
        self.om = oracle.OracleModel(cfg, self.W, int8=int8)
        fmt = "int8" if int8 else "bf16"
        self.paged = paged
        if paged:
            # the same rows in pools of `paged`-row blocks, at shuffled block
            # ids (plus a few spare blocks), addressed through a block table
            B, Hkv, S, D = self.ks[0].shape
            pk, pv, self.table = synth.paged_pools(self.ks, self.vs, paged, seed)
            self.pk, self.pv = pk, pv
            self.dec = Decoder(cfg, self.W, pk, pv, max_batch=B, max_seq=S, weight_format=fmt)
            self.dec.set_kv_pages(paged, self.table)
        else:
            self.dec = Decoder(cfg, self.W, self.ks, self.vs, weight_format=fmt)
        if stage_bytes is not None:
            self.dec.set_stage_bytes(stage_bytes)
        if stress is not None:  # (max delay ns, seed, permute queues)
            self.dec.set_race_stress(*stress)
        if hold is not None:
            self.dec.set_hold_policy(*hold)
        self.B = cfg["batch"]
        self.max_ctx = max_ctx or cfg["max_seq"]
        self.dec.build_schedule(self.B, self.max_ctx)
        self.tokens = synth.make_tokens(cfg, seed)
        self.pos = list(self.lengths)
        dev = "cuda"
        self.d_tok = torch.tensor(self.tokens, dtype=torch.int32, device=dev)
        self.d_pos = torch.tensor(self.pos, dtype=torch.int32, device=dev)
        self.d_logits = torch.empty((self.B, cfg["vocab"]), dtype=torch.float32, device=dev)
        self.d_am = torch.empty(self.B, dtype=torch.int32, device=dev)
        self.worst = 0.0
        self.near_ties = 0

    def gpu_step(self, mode: str = "mega"):
        self.d_tok.copy_(torch.tensor(self.tokens, dtype=torch.int32))
        self.d_pos.copy_(torch.tensor(self.pos, dtype=torch.int32))
        if mode == "mega":
            self.dec.step(self.d_tok, self.d_pos, self.d_logits, self.d_am)
        else:
            self.dec.step_ablation({"stream": 0, "graph": 1, "pdl": 2}[mode], self.d_tok,
                                   self.d_pos, self.d_logits, self.d_am)
        status = self.dec.sync_status()
        assert status == 0, f"device status {status}"
        return self.d_logits.cpu().numpy().astype(np.float64), self.d_am.cpu().numpy()

    def check(self, lg, am, lo, ao):
        for b in range(self.B):
            std = lo[b].std()
            d = np.abs(lg[b] - lo[b]).max()
            self.worst = max(self.worst, d / std)
            assert d <= TOL * std, f"b={b}: max|dlogit| {d:.3e} > {TOL} * std {std:.3e}"
            assert am[b] == int(np.argmax(lg[b])), "argmax is not the first max of the logits"
            s = np.sort(lo[b])
            if s[-1] - s[-2] > MARGIN:
                assert am[b] == ao[b], f"b={b}: argmax {am[b]} vs oracle {ao[b]}"

    def check_kv(self, back: int = 0):
        """The K/V rows appended at the current positions (and the `back`
        positions before them)."""
        for l in range(self.cfg["n_layers"]):
            for b in range(self.B):
                for P in range(self.pos[b] - back, self.pos[b] + 1):
                    for kind, ora in ((0, self.ko[l]), (1, self.vo[l])):
                        g = self.gpu_row(l, kind, b, P)
                        o = (ora[b, :, P, :].astype(np.uint32) << 16).view(np.float32)
                        # one bf16 ulp, plus fp32-vs-fp64 accumulation noise at the row's scale
                        tol = 2.0 ** -7 * np.abs(o) + 1e-3 * np.sqrt(np.mean(o * o))
                        assert np.all(np.abs(g - o) <= tol), \
                            f"layer {l} b {b} row {P}: appended K/V row differs by " \
                            f"{np.abs(g - o).max()}"

    def gpu_row(self, l: int, kind: int, b: int, P: int):
        """Cache row P of sequence b, all kv heads ([Hkv][D] fp32), as the GPU holds it."""
        if self.paged:
            pool = (self.pk, self.pv)[kind][l]
            blk = int(self.table[b, P // self.paged])
            return pool[blk, :, P % self.paged, :].float().cpu().numpy()
        return (self.ks, self.vs)[kind][l][b, :, P, :].float().cpu().numpy()

    def step(self, mode: str = "mega", check_kv: bool = True):
        lg, am = self.gpu_step(mode)
        if self.cfg.get("n_experts", 0) > 0:
            lo, ao = self._oracle_moe_step()
        else:
            lo, ao, _, _ = self.om.step(self.ko, self.vo, self.tokens, self.pos)
        self.check(lg, am, lo, ao)
        if check_kv:
            self.check_kv()
        self.tokens = [int(a) for a in am]
        self.pos = [p + 1 for p in self.pos]
        return lg, am

    def _oracle_moe_step(self):
        gpu_ids = self.dec.routes()  # [L][K]
        lo, ao, rid, margin = self.om.step(self.ko, self.vo, self.tokens, self.pos)
        L = self.cfg["n_layers"]
        tie = margin[:, 0] < ROUTE_TIE
        if tie.any():  # redo the step with the GPU's choice at the near-tied layers
            self.near_ties += int(tie.sum())
            forced = gpu_ids.reshape(L, 1, -1)
            lo, ao, rid, margin = self.om.step(self.ko, self.vo, self.tokens, self.pos,
                                               forced_routes=forced,
                                               forced_mask=tie.astype(np.int32).reshape(L, 1))
        for l in range(L):
            assert sorted(rid[l, 0]) == sorted(gpu_ids[l]), \
                f"layer {l}: experts {sorted(gpu_ids[l])} vs oracle {sorted(rid[l, 0])}"
        return lo, ao

    def multi_step(self, n: int, oracle: bool = True):
        """n greedy steps in one launch.  With `oracle`: teacher-force the
        oracle with the GPU's argmax of every step, check each step's argmax
        where the oracle's top-2 margin is clear, then the last step's logits
        and every appended K/V row.  Returns (logits of the last step,
        argmax [n][B])."""
        self.d_tok.copy_(torch.tensor(self.tokens, dtype=torch.int32))
        self.d_pos.copy_(torch.tensor(self.pos, dtype=torch.int32))
        d_am = torch.full((n, self.B), -1, dtype=torch.int32, device="cuda")
        self.dec.steps(self.d_tok, self.d_pos, n, self.d_logits, d_am)
        status = self.dec.sync_status()
        assert status == 0, f"device status {status}"
        lg = self.d_logits.cpu().numpy().astype(np.float64)
        am = d_am.cpu().numpy()
        if oracle:
            for t in range(n):
                lo, ao, _, _ = self.om.step(self.ko, self.vo, self.tokens, self.pos)
                for b in range(self.B):
                    s = np.sort(lo[b])
                    if s[-1] - s[-2] > MARGIN:
                        assert am[t][b] == ao[b], f"step {t} b={b}: argmax {am[t][b]} vs oracle {ao[b]}"
                if t < n - 1:
                    self.tokens = [int(a) for a in am[t]]
                    self.pos = [p + 1 for p in self.pos]
            self.check(lg, am[n - 1], lo, ao)
            self.check_kv(back=n - 1)
        else:
            self.pos = [p + n - 1 for p in self.pos]
        self.tokens = [int(a) for a in am[n - 1]]
        self.pos = [p + 1 for p in self.pos]
        return lg, am

    def close(self):
        self.dec.close()

"""Seeded synthetic inputs shared by the oracle tests and the CUDA path.

This module holds workload shapes and random-number recipes only -- none of
the decoder's arithmetic.  Every tensor is drawn from its own torch generator
seeded from (seed, tensor name), so any tensor can be regenerated alone and
the order of generation does not matter.  Generation runs on whatever device
is asked for; the oracle always receives the very same bf16 bytes that the
GPU path consumes (tests copy them device -> host).

Recipe (no dataset or public suite stands behind these workloads):
  * weights: bf16 ~ N(0, 0.02); norm gains: bf16 1 + N(0, 0.02);
  * KV cache prefill: bf16 ~ N(0, 1) at rows [0, len_b), zeros elsewhere;
  * initial tokens: uniform in [0, vocab);
  * batch lengths: uniform integers in [lo, hi] inclusive.
Seeds: weights ``seed``, KV ``seed + 1``, tokens ``seed + 2``, lengths ``seed + 3``.
"""
from __future__ import annotations

import zlib

import torch

# Workload shapes (decoder configurations) with their decode lengths.
CONFIGS = {
    "tiny": dict(
        name="tiny", n_layers=2, hidden=256, n_q_heads=4, n_kv_heads=2, head_dim=64, ffn=1024,
        vocab=1024, rms_eps=1e-5, rope_theta=1e4, tied=True, n_experts=0, top_k=0,
        expert_ffn=0, shared_ffn=0, batch=1, prefill=(16, 16), steps=8),
    "llama1b_1k": dict(
        name="llama1b_1k", n_layers=16, hidden=2048, n_q_heads=32, n_kv_heads=8, head_dim=64,
        ffn=8192, vocab=128256, rms_eps=1e-5, rope_theta=5e5, tied=True, n_experts=0, top_k=0,
        expert_ffn=0, shared_ffn=0, batch=1, prefill=(1024, 1024), steps=128),
    "llama1b_8k": dict(
        name="llama1b_8k", n_layers=16, hidden=2048, n_q_heads=32, n_kv_heads=8, head_dim=64,
        ffn=8192, vocab=128256, rms_eps=1e-5, rope_theta=5e5, tied=True, n_experts=0, top_k=0,
        expert_ffn=0, shared_ffn=0, batch=1, prefill=(8192, 8192), steps=128),
    # long-context decode (the paged / long-context next step): a 32K cache,
    # where the attention's share of the bytes passes a third
    "llama1b_32k": dict(
        name="llama1b_32k", n_layers=16, hidden=2048, n_q_heads=32, n_kv_heads=8, head_dim=64,
        ffn=8192, vocab=128256, rms_eps=1e-5, rope_theta=5e5, tied=True, n_experts=0, top_k=0,
        expert_ffn=0, shared_ffn=0, batch=1, prefill=(32768, 32768), steps=128),
    "llama1b_b8": dict(
        name="llama1b_b8", n_layers=16, hidden=2048, n_q_heads=32, n_kv_heads=8, head_dim=64,
        ffn=8192, vocab=128256, rms_eps=1e-5, rope_theta=5e5, tied=True, n_experts=0, top_k=0,
        expert_ffn=0, shared_ffn=0, batch=8, prefill=(512, 2048), steps=64),
    # A small case of the same kernel for detailed profiler captures: four
    # layers of the Llama-1B shape and a 32000-row head (about 620 MB of bf16
    # weights, well above the 129 MB L2).
    "llama1b_4l": dict(
        name="llama1b_4l", n_layers=4, hidden=2048, n_q_heads=32, n_kv_heads=8, head_dim=64,
        ffn=8192, vocab=32000, rms_eps=1e-5, rope_theta=5e5, tied=True, n_experts=0, top_k=0,
        expert_ffn=0, shared_ffn=0, batch=1, prefill=(1024, 1024), steps=128),
    "moe": dict(
        name="moe", n_layers=24, hidden=2048, n_q_heads=16, n_kv_heads=4, head_dim=128, ffn=0,
        vocab=65536, rms_eps=1e-5, rope_theta=5e5, tied=False, n_experts=128, top_k=8,
        expert_ffn=768, shared_ffn=2048, batch=1, prefill=(1024, 1024), steps=64),
}


def with_cache(cfg: dict, extra_steps: int = 0) -> dict:
    """Copy of cfg with max_seq = longest prefill + decode steps (+ extra), rounded up to 64."""
    c = dict(cfg)
    need = cfg["prefill"][1] + cfg["steps"] + extra_steps
    c["max_seq"] = int((need + 63) // 64 * 64)
    return c


def paged_pools(ks, vs, block: int, seed: int, spare: int = 5):
    """The rows of contiguous caches ks[l] / vs[l] ([B][Hkv][S][D]) as pools
    [n_blocks][Hkv][block][D] at shuffled block ids, and the int32 block table
    [B][ceil(S / block)] that addresses them (plus `spare` unused blocks)."""
    B, Hkv, S, D = ks[0].shape
    nb = -(-S // block)
    n_blocks = B * nb + spare
    perm = torch.randperm(n_blocks, generator=torch.Generator().manual_seed(seed + 99))
    table = perm[:B * nb].reshape(B, nb).to(torch.int32)
    pk, pv = [], []
    for kt, vt in zip(ks, vs):
        pool_k = torch.zeros((n_blocks, Hkv, block, D), dtype=kt.dtype, device=kt.device)
        pool_v = torch.zeros_like(pool_k)
        for b in range(B):
            for j in range(nb):
                rows = slice(j * block, min(S, (j + 1) * block))
                n = rows.stop - rows.start
                pool_k[int(table[b, j]), :, :n] = kt[b, :, rows]
                pool_v[int(table[b, j]), :, :n] = vt[b, :, rows]
        pk.append(pool_k)
        pv.append(pool_v)
    return pk, pv, table.to(ks[0].device)


def custom(**kw) -> dict:
    """A small decoder shape for tests; unspecified fields come from 'tiny'."""
    c = dict(CONFIGS["tiny"])
    c.update(kw)
    c.setdefault("name", "custom")
    return c


def _gen(seed: int, name: str, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed((seed * 1_000_003 + zlib.crc32(name.encode())) % (2**63))
    return g


def _normal(shape, seed, name, device, std=1.0, mean=0.0):
    g = _gen(seed, name, device)
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    if mean != 0.0:
        t.add_(mean)
    return t.to(torch.bfloat16)


def make_weights(cfg: dict, seed: int = 0, device="cpu", std: float = 0.02) -> dict:
    """bf16 weights in the [out][in] row-major layout of each projection."""
    H, Hq, Hkv, d = cfg["hidden"], cfg["n_q_heads"], cfg["n_kv_heads"], cfg["head_dim"]
    F, V, L = cfg["ffn"], cfg["vocab"], cfg["n_layers"]
    E, Fe, Fs = cfg["n_experts"], cfg["expert_ffn"], cfg["shared_ffn"]
    W = {
        "embed": _normal((V, H), seed, "embed", device, std),
        "lm_head": None if cfg["tied"] else _normal((V, H), seed, "lm_head", device, std),
        "final_norm": _normal((H,), seed, "final_norm", device, std, 1.0),
        "layers": [],
    }
    for l in range(L):
        p = f"l{l}."
        lw = {
            "attn_norm": _normal((H,), seed, p + "attn_norm", device, std, 1.0),
            "wq": _normal((Hq * d, H), seed, p + "wq", device, std),
            "wk": _normal((Hkv * d, H), seed, p + "wk", device, std),
            "wv": _normal((Hkv * d, H), seed, p + "wv", device, std),
            "wo": _normal((H, Hq * d), seed, p + "wo", device, std),
            "mlp_norm": _normal((H,), seed, p + "mlp_norm", device, std, 1.0),
        }
        if E == 0:
            lw["w_gate"] = _normal((F, H), seed, p + "w_gate", device, std)
            lw["w_up"] = _normal((F, H), seed, p + "w_up", device, std)
            lw["w_down"] = _normal((H, F), seed, p + "w_down", device, std)
        else:
            lw["router"] = _normal((E, H), seed, p + "router", device, std)
            lw["ex_gate"] = _normal((E, Fe, H), seed, p + "ex_gate", device, std)
            lw["ex_up"] = _normal((E, Fe, H), seed, p + "ex_up", device, std)
            lw["ex_down"] = _normal((E, H, Fe), seed, p + "ex_down", device, std)
            if Fs > 0:
                lw["sh_gate"] = _normal((Fs, H), seed, p + "sh_gate", device, std)
                lw["sh_up"] = _normal((Fs, H), seed, p + "sh_up", device, std)
                lw["sh_down"] = _normal((H, Fs), seed, p + "sh_down", device, std)
        W["layers"].append(lw)
    return W


def make_lengths(cfg: dict, seed: int = 0) -> list:
    """Prefilled cache length per sequence: uniform integers in cfg['prefill'] (inclusive)."""
    lo, hi = cfg["prefill"]
    B = cfg["batch"]
    if lo == hi:
        return [lo] * B
    g = _gen(seed + 3, "lengths", "cpu")
    return torch.randint(lo, hi + 1, (B,), generator=g).tolist()


def make_kv(cfg: dict, lengths, seed: int = 0, device="cpu"):
    """Per-layer bf16 K and V caches [B][Hkv][max_seq][d]; rows < length are N(0,1)."""
    B, Hkv, d, S = len(lengths), cfg["n_kv_heads"], cfg["head_dim"], cfg["max_seq"]
    ks, vs = [], []
    for l in range(cfg["n_layers"]):
        pair = []
        for kind in ("k", "v"):
            t = torch.zeros((B, Hkv, S, d), dtype=torch.bfloat16, device=device)
            for b, n in enumerate(lengths):
                if n > 0:
                    t[b, :, :n, :] = _normal((Hkv, n, d), seed + 1, f"{kind}{l}.{b}", device)
            pair.append(t)
        ks.append(pair[0])
        vs.append(pair[1])
    return ks, vs


def make_tokens(cfg: dict, seed: int = 0, batch: int | None = None) -> list:
    B = cfg["batch"] if batch is None else batch
    g = _gen(seed + 2, "tokens", "cpu")
    return torch.randint(0, cfg["vocab"], (B,), generator=g).tolist()

"""An independent numpy float64 formulation of the decoder, used to pin the oracle.

It shares nothing with oracle/oracle.c: rotary embedding is a complex
multiplication, attention is a batched matrix softmax with the key/value heads
repeated for grouped-query attention, softmax / sigmoid come from scipy, the
projections are numpy matmuls, top-k is a stable argsort, and bf16 rounding is
numpy's round-half-to-even on the frexp significand.
"""
import numpy as np
from scipy.special import expit, softmax


def widen(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(
        np.float64)


def round_bf16(x):
    m, e = np.frexp(np.asarray(x, np.float64))
    return np.ldexp(np.round(m * 256.0), e - 8)


def to_bits(x):
    return (np.asarray(round_bf16(x), np.float32).view(np.uint32) >> 16).astype(np.uint16)


def rms(x, g, eps):
    return x / np.sqrt(np.mean(x * x) + eps) * g


def rope_complex(v, pos, theta):
    """v: [heads, d]; rotate (v[:, i], v[:, i + d/2]) as one complex number."""
    d = v.shape[-1]
    h = d // 2
    inv = theta ** (-np.arange(h) * 2.0 / d)
    z = (v[:, :h] + 1j * v[:, h:]) * np.exp(1j * pos * inv)
    return np.concatenate([z.real, z.imag], axis=-1)


def swiglu(Wg, Wu, Wd, xn):
    a = Wg @ xn
    return Wd @ (a * expit(a) * (Wu @ xn))


def decode(cfg, W, K, V, tokens, positions, forced=None):
    """W: dict of float64 arrays (same keys as synth.make_weights); K, V: per-layer
    float64 [B][Hkv][S][d], updated in place with the bf16-rounded new rows."""
    H, Hq, Hkv, d = cfg["hidden"], cfg["n_q_heads"], cfg["n_kv_heads"], cfg["head_dim"]
    eps, theta = cfg["rms_eps"], cfg["rope_theta"]
    grp = Hq // Hkv
    B = len(tokens)
    logits = np.zeros((B, cfg["vocab"]))
    routes = []
    for b in range(B):
        P = positions[b]
        x = W["embed"][tokens[b]].copy()
        for l, lw in enumerate(W["layers"]):
            xn = rms(x, lw["attn_norm"], eps)
            q = rope_complex((lw["wq"] @ xn).reshape(Hq, d), P, theta)
            k = rope_complex((lw["wk"] @ xn).reshape(Hkv, d), P, theta)
            v = (lw["wv"] @ xn).reshape(Hkv, d)
            K[l][b, :, P, :] = round_bf16(k)
            V[l][b, :, P, :] = round_bf16(v)
            Kc = np.repeat(K[l][b, :, :P + 1, :], grp, axis=0)
            Vc = np.repeat(V[l][b, :, :P + 1, :], grp, axis=0)
            s = np.einsum("hd,hcd->hc", q, Kc) / np.sqrt(d)
            o = np.einsum("hc,hcd->hd", softmax(s, axis=-1), Vc).reshape(-1)
            x = x + lw["wo"] @ o
            xn = rms(x, lw["mlp_norm"], eps)
            if cfg["n_experts"] == 0:
                x = x + swiglu(lw["w_gate"], lw["w_up"], lw["w_down"], xn)
            else:
                p = softmax(lw["router"] @ xn)
                ids = np.argsort(-p, kind="stable")[:cfg["top_k"]]
                if forced is not None and forced.get((l, b)) is not None:
                    ids = np.asarray(forced[(l, b)])
                routes.append(ids)
                wsel = p[ids] / p[ids].sum()
                y = np.zeros(H)
                for j, e in enumerate(ids):
                    y += wsel[j] * swiglu(lw["ex_gate"][e], lw["ex_up"][e], lw["ex_down"][e], xn)
                if cfg["shared_ffn"] > 0:
                    y += swiglu(lw["sh_gate"], lw["sh_up"], lw["sh_down"], xn)
                x = x + y
        logits[b] = W["lm_head"] @ rms(x, W["final_norm"], eps)
    return logits, np.argmax(logits, axis=-1), routes


def weights_f64(weights):
    """synth weights (CPU bf16 tensors) -> float64 numpy dict for decode()."""
    import torch

    def cv(t):
        return None if t is None else t.detach().cpu().to(torch.float64).numpy()

    W = {"embed": cv(weights["embed"]), "final_norm": cv(weights["final_norm"])}
    W["lm_head"] = W["embed"] if weights["lm_head"] is None else cv(weights["lm_head"])
    W["layers"] = [{k: cv(v) for k, v in lw.items()} for lw in weights["layers"]]
    return W

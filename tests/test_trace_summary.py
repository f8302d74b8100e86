"""Host-side trace analysis on synthetic stamps (no GPU)."""
import numpy as np

from decode_megakernel_sm_gb300 import trace as T

OPS = {"QKV": 1, "ATTN": 2, "OPROJ": 3, "MLP_UP": 8, "MLP_DOWN": 9}


def _rows(n_layers=4, n_sm=3):
    # phase i of layer l: prologue ends at t + 1000 + 100 s, body ends at
    # t + 5000 + 100 s (s = SM), t = 100 us * l + 10 us * i
    rows = []
    for l in range(n_layers):
        for i, op in enumerate(OPS.values()):
            t = l * 100_000 + i * 10_000
            for s in range(n_sm):
                m0, te = t + 1000 + 100 * s, t + 5000 + 100 * s
                rows.append((s, 0, op, l, 0, t, t, te, m0, m0, 0, te))
    return rows


def test_hops_measure_last_producer_to_consumer_prologue():
    h = T._hops(_rows())
    # within a layer: last body end of phase i is t_i + 5.2 us; the next
    # phase's prologues end at t_i + 10 us + 1.0 / 1.1 / 1.2 us
    for k in ("QKV->ATTN", "ATTN->OPROJ", "OPROJ->MLP_UP", "MLP_UP->MLP_DOWN"):
        assert np.allclose([h[k]["min_us"], h[k]["median_us"], h[k]["max_us"]], [5.8, 5.9, 6.0])
        assert np.isclose(h[k]["consumer_ring_and_epilogue_us"], 4.0)
    # the down rows feed the next layer's QKV, 100 us later
    assert np.allclose(h["MLP_DOWN->QKV"]["median_us"], 55.9)

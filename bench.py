"""Decode throughput of the GB300 megakernel (one JSON line on rank 0).

Workload (default): the Llama-3.2-1B-shaped decoder at batch 1 -- 16 layers,
hidden 2048, 32 query / 8 kv heads of 64, SwiGLU FFN 8192, vocab 128256, tied
LM head, bf16 weights ~N(0, 0.02) from a seed, bf16 KV cache prefilled with
1024 positions -- decoding greedily: step t feeds the previous step's argmax
device-to-device and writes cache row 1024 + (t mod 128), so the timed steps
cycle over the 128-step decode window of the workload.  A step is one pass
of the persistent kernel over the whole forward pass; by default one launch
runs up to 16 such steps back to back (mk_decode_steps: each step decodes the
previous step's argmax on the device; the launch size divides --steps), and
--multi-step 0 launches once per step.  Besides the mean, the line gives the
median and p10 / p90 of the per-step time of every launch.
The end-to-end figure goes through the host-buffer call, one step per call.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
  python bench.py --impl reference ...   (the CPU oracle on the host cores)

Multi-GPU: replicas only (the path has no exchange step): under torchrun each
rank decodes its own copy of the workload; value = all ranks' tokens / the
slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode tok/s at batch 1 (Llama-1B shape); % of 8 TB/s HBM roofline"
WINDOW = None  # decode window (steps) of the workload, from the config


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1024)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="mk", choices=["mk", "reference"])
    ap.add_argument("--config", default="llama1b_1k")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ablation", action="store_true", help="also time the per-phase launches")
    ap.add_argument("--multi-step", type=int, default=None,
                    help="greedy steps per launch (mk_decode_steps); 0: one launch per step; "
                         "default: the largest of 16, 8, 4, 2 that divides both the decode "
                         "window and --steps (else one launch per step)")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--l2-ahead", type=int, default=None,
                    help="bytes each SM warms in L2 ahead of its ring (library default if unset)")
    ap.add_argument("--kc", type=int, default=None,
                    help="partial copies of each residual vector (library default if unset)")
    ap.add_argument("--hold", type=int, default=None,
                    help="hold-policy mask (library default if unset)")
    ap.add_argument("--pollers", type=int, default=None,
                    help="warps polling each dependency counter (library default if unset)")
    ap.add_argument("--poll-stagger", type=int, default=0, help="ns between pollers (with --pollers)")
    ap.add_argument("--batch", type=int, default=None,
                    help="sequences per step (default: the workload's own; at most its batch capacity)")
    ap.add_argument("--weights", default="bf16", choices=["bf16", "int8"],
                    help="streamed weight format (int8: per-row int8 codes + fp32 scales)")
    ap.add_argument("--paged", type=int, default=0,
                    help="paged KV cache with blocks of this many rows (0: contiguous)")
    ap.add_argument("--ring-depth", type=int, default=None,
                    help="at most this many ring stages (library default if unset)")
    ap.add_argument("--hold-early", type=int, default=128 << 10,
                    help="bytes of a held instruction's copies issued early (with --hold)")
    ap.add_argument("--batched-variant", type=int, default=0, choices=[0, 1],
                    help="2..8 sequences: 0 the tcgen05 wide-batch kernel where the shape allows "
                         "it (default), 1 the warp-level mma.sync batched kernel")
    ap.add_argument("--stage-bytes", type=int, default=None,
                    help="ring stage size in bytes (default: the library's)")
    ap.add_argument("--trace", default=None,
                    help="write a per-instruction timeline of 3 traced steps to this path")
    return ap.parse_args()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def job_rate(elapsed_s, units_per_rank, ws, device):
    """The slowest rank's elapsed time (max over ranks) and the whole job's
    rate: all ranks' units over that time.  Every rank runs the same units
    (weak scaling); ws == 1 needs no process group."""
    import torch
    t = torch.tensor([float(elapsed_s)], dtype=torch.float64, device=device)
    if ws > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    slowest = float(t.item())
    return slowest, ws * units_per_rank / slowest


def workload_desc(cfg):
    lo, hi = cfg["prefill"]
    kv = f"KV prefill {lo}" if lo == hi else f"KV prefill U[{lo},{hi}]"
    mlp = (f"{cfg['n_experts']} experts x F{cfg['expert_ffn']} top-{cfg['top_k']} + shared "
           f"F{cfg['shared_ffn']}" if cfg["n_experts"] else f"SwiGLU F{cfg['ffn']}")
    return (f"{cfg['name']}: {cfg['n_layers']}L H{cfg['hidden']} {cfg['n_q_heads']}q/"
            f"{cfg['n_kv_heads']}kv d{cfg['head_dim']} {mlp} V{cfg['vocab']}"
            f"{' tied' if cfg['tied'] else ''}, "
            f"{'int8 weights (per-row fp32 scales)' if cfg.get('int8') else 'bf16 weights'}, "
            f"batch {cfg['batch']}, {kv}"
            f"{' in blocks of %d rows (paged)' % cfg['kv_pages'] if cfg.get('kv_pages') else ''}, "
            f"{cfg['steps']} greedy steps")


def step_bytes(cfg, positions, weight_bytes):
    """Algorithmic HBM bytes of one step: every weight once (routed MoE: the
    active experts), K and V rows [0, P] read, the new K/V row written, the
    logits written."""
    Hkv, d, L, B, V = cfg["n_kv_heads"], cfg["head_dim"], cfg["n_layers"], cfg["batch"], \
        cfg["vocab"]
    kv_row = L * Hkv * d * 2 * 2  # K and V, all layers, bytes per position
    kv = sum((p + 1) * kv_row for p in positions) + B * kv_row
    return weight_bytes + kv + B * V * 4


def kernel_src_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "decode_megakernel_sm_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        j = json.load(open(p))
        return float(j["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def traffic_record(config, steps_per_launch=1):
    """DRAM bytes per launch of `steps_per_launch` steps from the committed ncu
    summary (profiles/traffic.json), if it was taken on the current kernel
    sources: the capture of launches of that size when there is one, else a
    capture of another launch size of the same workload scaled by its steps
    (the step-to-step L2 reuse is a few MB of a 2.5 GB step).  Returns
    (bytes, how) or (None, reason)."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        j = json.load(open(p))
    except Exception:
        return None, "no profiles/traffic.json"
    src = kernel_src_hash()
    exact = j.get(config if steps_per_launch == 1 else f"{config}@{steps_per_launch}")
    if exact and exact.get("kernel_src_sha") == src:
        return float(exact["dram_bytes_per_launch"]), f"ncu, launches of {steps_per_launch} step(s)"
    near = []  # captures of other launch sizes, nearest size first
    for key, e in j.items():
        if key.split("@")[0] != config or e.get("kernel_src_sha") != src:
            continue
        spl = int(key.split("@")[1]) if "@" in key else 1
        near.append((abs(spl - steps_per_launch), -spl, spl, e))
    if near:
        _, _, spl, e = min(near, key=lambda x: x[:2])
        per_step = float(e["dram_bytes_per_launch"]) / spl
        return per_step * steps_per_launch, (f"ncu, launches of {spl} step(s), scaled to "
                                             f"{steps_per_launch}")
    return None, "no capture on this kernel source"


class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_uuid=None):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "50"]
        if device_uuid:
            cmd += ["-i", device_uuid]
        try:
            self.p = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                      text=True)
        except Exception:
            self.p = None

    def stop(self):
        if self.p is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.p.terminate()
        out, _ = self.p.communicate(timeout=10)
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx = float(f[1])
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm)}


def _to_host(W):
    return {k: (None if v is None else
                [{n: t.cpu() for n, t in lw.items()} for lw in v] if k == "layers" else v.cpu())
            for k, v in W.items()}


def cpu_baseline(cfg, W, ks, vs, lengths, tokens, budget_s=20.0):
    """The oracle as it stands, on the host cores, on a bounded sample of decode
    steps of the same workload (at least one step)."""
    import oracle
    t0 = time.perf_counter()
    om = oracle.OracleModel(cfg, W, int8=bool(cfg.get("int8")))
    ko = [oracle._bits(t.cpu()).copy() for t in ks]
    vo = [oracle._bits(t.cpu()).copy() for t in vs]
    prep = time.perf_counter() - t0
    pos = list(lengths)
    n, t_run = 0, 0.0
    while True:
        t1 = time.perf_counter()
        _, am, _, _ = om.step(ko, vo, tokens, pos)
        t_run += time.perf_counter() - t1
        n += 1
        tokens = [int(a) for a in am]
        pos = [p + 1 for p in pos]
        if t_run + t_run / n > budget_s or n >= cfg["steps"]:
            break
    B = cfg["batch"]
    return {"value": n * B / t_run, "unit": "tok/s", "cores": oracle.get_threads(),
            "kind": "oracle",
            "sample": f"{n} greedy decode step(s) of the same workload from position "
                      f"{lengths[0]} ({t_run:.1f} s; host copy of the weights {prep:.1f} s "
                      f"excluded)"}


def run_reference(args, cfg):
    """--impl reference: the CPU oracle timed on the host cores."""
    import numpy as np
    import torch
    import oracle
    import synth
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    W = synth.make_weights(cfg, args.seed, "cpu")
    lengths = synth.make_lengths(cfg, args.seed)
    ks, vs = synth.make_kv(cfg, lengths, args.seed, "cpu")
    om = oracle.OracleModel(cfg, W, int8=bool(cfg.get("int8")))
    ko = [oracle._bits(t).copy() for t in ks]
    vo = [oracle._bits(t).copy() for t in vs]
    tokens = synth.make_tokens(cfg, args.seed)
    P0 = list(lengths)
    t1 = time.perf_counter()
    om.step(ko, vo, tokens, P0)
    t_one = time.perf_counter() - t1
    budget = 120.0
    k = max(1, min(args.steps, int(budget / max(t_one, 1e-6))))
    w = min(args.warmup, 1)
    for i in range(w):
        om.step(ko, vo, tokens, [p + i for p in P0])
    t0 = time.perf_counter()
    toks = tokens
    for i in range(k):
        _, am, _, _ = om.step(ko, vo, toks, [p + (i % cfg["steps"]) for p in P0])
        toks = [int(a) for a in am]
    el = time.perf_counter() - t0
    B = cfg["batch"]
    val = k * B / el
    line = {
        "impl": "reference", "metric": METRIC, "value": val, "unit": "tok/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / k * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64 (int8 weights)" if cfg.get("int8") else "f64",
        "data": "synthetic", "config": {"workload": workload_desc(cfg)},
        "cpu_baseline": {"value": val, "unit": "tok/s", "cores": oracle.get_threads(),
                         "kind": "oracle",
                         "sample": f"{k} of {args.steps} requested steps (bounded to ~{budget:.0f}"
                                   f" s of CPU work), {w} warm-up"},
        "e2e": {"value": val, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    import synth
    base = synth.CONFIGS[args.config]
    cfg = synth.with_cache(base)
    if args.weights == "int8":
        cfg = dict(cfg, int8=True)
    if args.batch is not None:
        cfg = dict(cfg, batch=args.batch)
    if args.batched_variant:
        cfg = dict(cfg, batched_variant=1)
    if args.impl == "reference":
        run_reference(args, cfg)
        return
    import numpy as np
    import torch
    import torch.distributed as dist
    from decode_megakernel_sm_gb300 import Decoder, MK_ABL_GRAPH, MK_ABL_PDL, MK_ABL_STREAM

    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    if ws > 1:
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    B, V = cfg["batch"], cfg["vocab"]
    W = synth.make_weights(cfg, args.seed, dev)
    lengths = synth.make_lengths(cfg, args.seed)
    ks, vs = synth.make_kv(cfg, lengths, args.seed, dev)
    tokens0 = synth.make_tokens(cfg, args.seed)
    torch.cuda.synchronize()
    if args.paged:  # the same rows in shuffled blocks of a pool, through a block table
        pk, pv, table = synth.paged_pools(ks, vs, args.paged, args.seed)
        dec = Decoder(cfg, W, pk, pv, max_batch=B, max_seq=cfg["max_seq"],
                      weight_format=args.weights)
        dec.set_kv_pages(args.paged, table)
        cfg = dict(cfg, kv_pages=args.paged)
    else:
        dec = Decoder(cfg, W, ks, vs, weight_format=args.weights)
    # the library holds its own packed copy: keep only a host copy (for the CPU
    # baseline) and free the device one
    want_cpu = rank == 0 and ws == 1 and not args.no_cpu_baseline
    W = _to_host(W) if want_cpu else None
    torch.cuda.empty_cache()
    if args.kc is not None:
        dec.set_residual_copies(args.kc)
    if args.pollers is not None:
        dec.set_poll_policy(args.pollers, args.poll_stagger)
    if args.ring_depth is not None:
        dec.set_ring_depth(args.ring_depth)
    if args.hold is not None:
        dec.set_hold_policy(args.hold, args.hold_early)
    if args.stage_bytes is not None:
        dec.set_stage_bytes(args.stage_bytes)
    dec.build_schedule(B, cfg["max_seq"])
    if args.l2_ahead is not None:
        dec.set_l2_prefetch(args.l2_ahead)
    info = dec.info()
    stream = torch.cuda.current_stream()
    window = cfg["steps"]
    P0 = torch.tensor(lengths, dtype=torch.int32)
    pos_table = (P0[None, :] + torch.arange(window, dtype=torch.int32)[:, None]).to(dev)
    tok0 = torch.tensor(tokens0, dtype=torch.int32, device=dev)
    am = [torch.empty(B, dtype=torch.int32, device=dev) for _ in range(2)]
    logits = torch.empty((B, V), dtype=torch.float32, device=dev)

    ns = args.multi_step
    if ns is None:  # the longest launch (<= 16 steps) that divides the window and --steps
        ns = next((k for k in (16, 8, 4, 2) if window % k == 0 and args.steps % k == 0), 0)
    if ns:
        if ns < 1 or window % ns or args.steps % ns:
            raise SystemExit(f"--multi-step {ns} must divide the decode window ({window}) "
                             f"and --steps ({args.steps})")
        am_ms = [torch.empty((ns, B), dtype=torch.int32, device=dev) for _ in range(2)]

    def run(n, fn=None, marks=None):
        """n steps; with `marks`, an event is recorded after every launch."""
        if ns and fn is None:  # launches of ns steps, each fed the last argmax of the one before
            for k in range((n + ns - 1) // ns):
                tok = tok0 if k == 0 else am_ms[(k - 1) % 2][ns - 1]
                dec.steps(tok, pos_table[(k * ns) % window], ns, logits, am_ms[k % 2], stream)
                if marks is not None:
                    marks.append(torch.cuda.Event(enable_timing=True))
                    marks[-1].record(stream)
            return
        for t in range(n):
            tok = tok0 if t == 0 else am[(t - 1) % 2]
            if fn is None:
                dec.step(tok, pos_table[t % window], logits, am[t % 2], stream)
            else:
                fn(tok, pos_table[t % window], logits, am[t % 2])
            if marks is not None:
                marks.append(torch.cuda.Event(enable_timing=True))
                marks[-1].record(stream)

    def barrier():
        if ws > 1:
            dist.barrier()
        torch.cuda.synchronize()

    run(max(args.warmup, 3))
    st = dec.sync_status(stream)
    if st != 0:
        raise SystemExit(f"device status {st} during warm-up")
    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    barrier()
    clocks = ClockSampler(uuid)
    time.sleep(0.15)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    marks = []
    e0.record(stream)
    run(args.steps, marks=marks)
    e1.record(stream)
    barrier()
    ms = e0.elapsed_time(e1)
    # per-step time of every launch (launch time / its steps): median, p10, p90
    spl_ = ns if ns else 1
    per = [a.elapsed_time(b) / spl_ for a, b in zip([e0] + marks[:-1], marks)]
    qs = np.quantile(np.array(per), [0.1, 0.5, 0.9]) if per else [None] * 3
    ck = clocks.stop()
    st = dec.sync_status(stream)
    if st != 0:
        raise SystemExit(f"device status {st} in the timed region")
    el_s, value = job_rate(ms / 1e3, args.steps * B, ws, dev)
    ms_max = el_s * 1e3
    ms_step = ms_max / args.steps

    # roofline of the (only) kernel: algorithmic bytes / average launch time
    per_step = [step_bytes(cfg, [lengths[b] + (t % window) for b in range(B)],
                           info["weight_bytes_per_step"]) for t in range(args.steps)]
    alg = sum(per_step) / len(per_step)
    peak, peak_kind = measured_peak()
    achieved = alg / (ms / args.steps / 1e3) / 1e9
    spl = ns if ns else 1  # steps per launch
    traffic, traffic_how = traffic_record(
        args.config + ("+int8" if args.weights == "int8" else "") +
        (f"+b{B}" if args.batch is not None else "") +
        ("+mma" if args.batched_variant else "") +
        (f"+paged{args.paged}" if args.paged else ""), spl)
    roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": achieved / peak, "traffic": traffic, "traffic_source": traffic_how,
            "traffic_over_algorithmic": (traffic / (alg * spl)) if traffic else None,
            "peak_source": peak_kind, "algorithmic_bytes_per_launch": alg * spl,
            "kernel": "mk::mk_decode_kernel (persistent, %d step(s) per launch)" % spl}

    line = {
        "metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step,
        "ms_per_step_dist": {"p10": float(qs[0]), "median": float(qs[1]), "p90": float(qs[2]),
                             "over": f"{len(per)} launches of {spl_} step(s)"},
        "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "int8 weights x f32" if args.weights == "int8" else "bf16", "data": "synthetic",
        "config": {"workload": workload_desc(cfg), "batch": B, "prefill": list(cfg["prefill"]),
                   "decode_window": window, "parallelism": f"replicas x{ws}",
                   "l2": "inputs larger than L2 (%.2f GB of weights streamed per step)"
                         % (info["weight_bytes_per_step"] / 1e9)},
        "gpu_launches": args.steps // ns if ns else args.steps, "roofline": roof, "clocks": ck,
        "kernel": {"n_sm": info["n_sm"], "ring_stages": info["n_stages"],
                   "stage_bytes": info["stage_bytes"], "instructions": info["n_instr"],
                   "attn_splits": info["attn_splits"],
                   "batched_variant": int(cfg.get("batched_variant", 0))},
    }

    if args.ablation:
        abl = {}
        for name, mode in (("stream", MK_ABL_STREAM), ("graph", MK_ABL_GRAPH),
                           ("pdl", MK_ABL_PDL)):
            n = min(args.steps, 256)
            fn = (lambda m: (lambda t, p, lg, a: dec.step_ablation(m, t, p, lg, a, stream)))(mode)
            run(3, fn)
            barrier()
            e0.record(stream)
            run(n, fn)
            e1.record(stream)
            barrier()
            abl[name] = e0.elapsed_time(e1) / n
            if dec.sync_status(stream) != 0:
                abl[name] = None
        line["ablation_ms_per_step"] = abl
        line["ablation_launches_per_step"] = info["ablation_launches"]
        # what each extra launch costs beyond the megakernel's step time: launch,
        # drain and refill of the pipeline at every (layer, phase) boundary
        line["ablation_overhead_us_per_launch"] = {
            k: (None if v is None else (v - ms_step) * 1e3 / info["ablation_launches"])
            for k, v in abl.items()}

    if args.trace:
        from decode_megakernel_sm_gb300.trace import chrome_trace, summarize
        dec.set_trace(True)
        run(3)
        barrier()
        tr, q, n_sm, max_pc = dec.get_trace()
        dec.set_trace(False)
        summ = summarize(tr, q, n_sm, max_pc)
        chrome_trace(tr, q, n_sm, max_pc, args.trace)
        with open(args.trace + ".summary.json", "w") as f:
            json.dump(summ, f, indent=1)

    if not args.no_e2e:
        # the public host-buffer call: pinned inputs in, logits + argmax out, every step
        n = min(args.steps, 256)
        htok = torch.tensor(tokens0, dtype=torch.int32).pin_memory()
        hpos = torch.empty(B, dtype=torch.int32).pin_memory()
        hlg = torch.empty((B, V), dtype=torch.float32).pin_memory()
        ham = torch.empty(B, dtype=torch.int32).pin_memory()
        for t in range(3):
            hpos.copy_(pos_table[t % window].cpu())
            dec.step_host(htok, hpos, hlg, ham)
        barrier()
        host_pos = pos_table.cpu()
        t0 = time.perf_counter()
        for t in range(n):
            hpos.copy_(host_pos[t % window])
            stt = dec.step_host(htok, hpos, hlg, ham)
            if stt != 0:
                raise SystemExit(f"host step status {stt}")
            htok.copy_(ham)
        _, e2e_rate = job_rate(time.perf_counter() - t0, n * B, ws, dev)
        line["e2e"] = {"value": e2e_rate, "unit": "tok/s",
                       "h2d_bytes_per_step": 2 * B * 4, "d2h_bytes_per_step": B * V * 4 + B * 4,
                       "steps": n}

    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(cfg, W, ks, vs, lengths, tokens0)

    if rank == 0:
        print(json.dumps(line), flush=True)
    dec.close()
    if ws > 1:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()

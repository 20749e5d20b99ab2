"""Benchmark: batch-invariant decode step, Llama-3-8B shapes, one GB300 per rank.

Workload (one step): a decode step of a ragged batch of B requests (B = 64 by
default; contexts uniform in [128, 8192], paged KV with page 16, K/V ~ N(0, 1)
bf16) through the whole path — embedding, one 8B-shaped decoder layer (d 4096,
32/8 heads, head dim 128, SwiGLU 14336), final RMSNorm, the 128256-wide LM
head in fp32 and greedy argmax — via bi_forward_step.  Weights are random
N(0, 0.02) bf16 (synthetic data; no trained weights).  The step reads ~2.6 GB,
far more than L2, so no flush is needed between steps.

Prints one JSON line (rank 0).  `value` is decode tokens/s of the invariant
mode at batch B, summed over ranks (each rank is an independent replica with
its own batch: weak scaling, no collective on the data path).  `sweep` holds
invariant vs variant tokens/s and the HBM-roofline fraction of the whole step
for B in 1..64.  `roofline` is for the dominant kernel (the tcgen05 GEMM),
timed with CUDA events on its launching stream.  `cpu_baseline` is the CPU
oracle on a bounded sample of the same workload.

--impl reference times the CPU oracle (the slow, plain definition) on the same
workload as the reference arm.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode tokens/s (8B-shape, bs 1-64, invariant vs variant); % HBM roofline"
WORKLOAD = "llama3-8b-shape decode step: 1 decoder layer + final norm + LM head + argmax"
CTX_LO, CTX_HI = 128, 8192
DATA_SEED = 43          # 42 + config index
WEIGHT_SEED = 1234


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--batch", type=int, default=64)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--no-sweep", action="store_true")
    p.add_argument("--no-cpu", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=15.0)
    p.add_argument("--ncu-target", choices=["gemm-decode64", "gemm-prefill8192", "prefill-attn16", "gemm-o-m1", "decode-attn16"],
                   default=None,
                   help="launch only the named GEMMs (twice: warm-up, then the pass to capture) for an ncu "
                        "capture; prints no measurement")
    p.add_argument("--floor", action="store_true",
                   help="print the GEMM floor microbenchmarks (ns per MMA per tcgen05 form, per-SM ingest) and the "
                        "floor they give each decode projection at M = 1, against its measured time")
    return p.parse_args()


def run_config(batch: int, world: int) -> dict:
    """The workload both arms report (the same keys and values)."""
    from invariant_fixed_order_gb300 import roofline
    cfg, ctx, _ = make_workload(batch, 0)
    step_gb = roofline.decode_step_bytes(cfg, [int(s) for s in ctx]) / 1e9
    return {"workload": WORKLOAD, "batch_per_gpu": batch, "context": [CTX_LO, CTX_HI], "mode": "invariant",
            "parallelism": f"replicas{world}", "l2": "inputs larger than L2 (step reads %.2f GB)" % step_gb}


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            j = json.load(fh)
        return float(j["hbm_gbs"]), float(j["bf16_tflops"]), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


def sustained_bf16_peak() -> float:
    """The bf16 GEMM rate measured back to back for seconds under the power cap (the denominator for kernels
    timed over long runs), else the fallback's sustained figure."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            return float(json.load(fh)["bf16_tflops_sustained"])
    except Exception:
        return 1700.0


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200",
                 "-i", str(gpu_index)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        loaded = [s for s in sm if s > 0]
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# workload
# ---------------------------------------------------------------------------

def make_workload(B: int, rank: int):
    from invariant_fixed_order_gb300 import synth
    from invariant_fixed_order_gb300.config import LLAMA3_8B_1L
    cfg = LLAMA3_8B_1L
    ctx = synth.uniform_ints(B, CTX_LO, CTX_HI, DATA_SEED + 1000 * rank)
    ids = synth.token_ids(B, cfg.V, DATA_SEED + 1000 * rank + 1)
    return cfg, ctx, ids


class GpuWorkload:
    def __init__(self, B: int, rank: int, device: str):
        import torch
        from invariant_fixed_order_gb300 import synth
        from invariant_fixed_order_gb300.engine import Engine
        self.cfg, self.ctx, self.ids = make_workload(B, rank)
        cfg = self.cfg
        self.B = B
        self.max_pages = CTX_HI // 16 + 1
        pages_needed = int(sum((int(s) + 15) // 16 for s in self.ctx))
        self.eng = Engine(cfg, seed=WEIGHT_SEED, num_pages=pages_needed + 64, max_pages=self.max_pages, max_T=B,
                          max_B=B, max_R=B, max_seq=self.max_pages * 16, device=device)
        # per-request pages and KV history (positions 0 .. s-2; the step appends s-1)
        self.table = np.zeros((B, self.max_pages), np.int32)
        for i, s in enumerate(self.ctx):
            pages = self.eng.pool.alloc((int(s) + 15) // 16)
            self.table[i, :len(pages)] = pages
            n = int(s) - 1
            if n > 0:
                k, v = synth.kv_history(n, cfg.Hkv, cfg.Dh, DATA_SEED * 7919 + i, device=device)
                pos = np.arange(n)
                pg = torch.from_numpy(self.table[i, pos // 16].astype(np.int64)).to(device)
                sl = torch.from_numpy((pos % 16).astype(np.int64)).to(device)
                self.eng.k[0][pg, :, sl, :] = k
                self.eng.v[0][pg, :, sl, :] = v
        self.d_table = torch.from_numpy(self.table).to(device)
        self.d_ids = torch.from_numpy(self.ids).to(device)
        self.logits = torch.empty(B, cfg.V, dtype=torch.float32, device=device)
        self.tokens = torch.empty(B, dtype=torch.int32, device=device)
        torch.cuda.synchronize()

    def step(self, b: int, mode: int, stream=None):
        """Decode step over the first b requests."""
        self.eng.step([1] * b, [int(s) - 1 for s in self.ctx[:b]], self.d_ids[:b], self.d_table[:b],
                      list(range(b)), mode=mode, stream=stream, logits_out=self.logits[:b], tokens_out=self.tokens)

    def step_layer(self, b: int, mode: int, stream=None):
        """The layer alone (embedding + layer, no logit rows) over the first b requests."""
        self.eng.step([1] * b, [int(s) - 1 for s in self.ctx[:b]], self.d_ids[:b], self.d_table[:b], [],
                      mode=mode, stream=stream, want_logits=False)

    def layer_bytes(self, b: int) -> int:
        from invariant_fixed_order_gb300 import roofline
        return roofline.decode_layer_bytes(self.cfg, [int(s) for s in self.ctx[:b]])

    def step_bytes(self, b: int) -> int:
        from invariant_fixed_order_gb300 import roofline
        return roofline.decode_step_bytes(self.cfg, [int(s) for s in self.ctx[:b]])


def time_steps(fn, steps: int, warmup: int, stream) -> float:
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def gemm_roofline(w: GpuWorkload, steps: int, stream, hbm_peak: float) -> dict:
    """Times every GEMM of the step standalone (same shapes, same weights) with
    CUDA events on the launching stream; algorithmic bytes per launch are the
    weights, the activations in and the outputs (plus the residual read)."""
    import torch
    from invariant_fixed_order_gb300 import bi
    cfg, B = w.cfg, w.B
    L = w.eng.layers[0]
    dev = w.d_ids.device
    x = torch.randn(B, cfg.d, device=dev).to(torch.bfloat16)
    h = torch.randn(B, cfg.F, device=dev).to(torch.bfloat16)
    qkv = torch.empty(B, cfg.qkv_dim, dtype=torch.float32, device=dev)
    res = torch.randn(B, cfg.d, device=dev).to(torch.bfloat16)
    hout = torch.empty(B, cfg.F, dtype=torch.bfloat16, device=dev)
    logits = torch.empty(B, cfg.V, dtype=torch.float32, device=dev)
    shapes = [
        ("qkv", lambda: bi.gemm(x, L["w_qkv"], out=qkv, c_dtype=bi.F32, stream=stream),
         cfg.qkv_dim * cfg.d * 2 + B * cfg.d * 2 + B * cfg.qkv_dim * 4),
        ("o", lambda: bi.gemm(x, L["w_o"], out=res, residual=res, ep=bi.EP_RESIDUAL, stream=stream),
         cfg.d * cfg.d * 2 + B * cfg.d * 2 + B * cfg.d * 4),
        ("gate_up", lambda: bi.gemm(x, L["w_gu"], out=hout, ep=bi.EP_SWIGLU, stream=stream),
         2 * cfg.F * cfg.d * 2 + B * cfg.d * 2 + B * cfg.F * 2),
        ("down", lambda: bi.gemm(h, L["w_down"], out=res, residual=res, ep=bi.EP_RESIDUAL, stream=stream),
         cfg.d * cfg.F * 2 + B * cfg.F * 2 + B * cfg.d * 4),
        ("lm_head", lambda: bi.gemm(x, w.eng.head["w_lm"], out=logits, c_dtype=bi.F32, stream=stream),
         cfg.V * cfg.d * 2 + B * cfg.d * 2 + B * cfg.V * 4),
    ]
    per = {}
    tot_bytes, tot_ms = 0, 0.0
    for name, fn, nbytes in shapes:
        ms = time_steps(fn, max(steps, 10), 3, stream)
        per[name] = {"us": round(ms * 1e3, 2), "GBps": round(nbytes / (ms * 1e-3) / 1e9, 1),
                     "frac": round(nbytes / (ms * 1e-3) / 1e9 / hbm_peak, 3)}
        tot_bytes += nbytes
        tot_ms += ms
    n = len(shapes)
    achieved = (tot_bytes / n) / (tot_ms / n * 1e-3) / 1e9
    return {"per_launch_bytes": tot_bytes / n, "per_launch_ms": tot_ms / n, "achieved": achieved, "per_gemm": per}


def attention_time(w: GpuWorkload, steps: int, stream) -> dict:
    import torch
    from invariant_fixed_order_gb300 import bi
    cfg, B = w.cfg, w.B
    dev = w.d_ids.device
    q = torch.randn(B, cfg.H, cfg.Dh, device=dev).to(torch.bfloat16)
    sl = torch.from_numpy(np.asarray(w.ctx, np.int32)).to(dev)
    ws = torch.empty(bi.decode_attention_workspace_size(B, cfg.H, cfg.Dh, w.max_pages * 16, bi.VARIANT),
                     dtype=torch.uint8, device=dev)
    out = torch.empty(B, cfg.H, cfg.Dh, dtype=torch.bfloat16, device=dev)
    fn = lambda: bi.decode_attention(q, w.eng.k[0], w.eng.v[0], w.d_table, sl, int(max(w.ctx)), ws=ws, out=out,
                                     stream=stream)
    ms = time_steps(fn, max(steps, 10), 3, stream)
    kv = sum(2 * int(s) * cfg.Hkv * cfg.Dh * 2 for s in w.ctx)
    return {"us": round(ms * 1e3, 2), "GBps": round(kv / (ms * 1e-3) / 1e9, 1), "kv_bytes": kv}


def gemm_chain(steps: int, stream) -> dict:
    """The cost of one dependent MMA in the layer projections' form: one output tile (M = 1, N = 128, a single
    CTA pair) at K = 1024 ... 65536.  Every K step of the tile's accumulator is one 256x128x16 pair MMA that
    must follow the previous one, so the time's slope against K / 16 is the cost of a dependent MMA (the weights,
    at most 16 MB, stay in L2 across the timed repeats: this measures the chain, not HBM).  The layer's floor
    under one MMA form and no split of K follows: each projection's chain length (K / 16 per output tile, times
    the waves of output tiles over the 76 CTA pairs) times that cost."""
    import torch
    from invariant_fixed_order_gb300 import bi
    from invariant_fixed_order_gb300.config import LLAMA3_8B
    g = torch.Generator(device="cuda").manual_seed(5)
    ks = [1024, 2048, 4096, 8192, 16384, 32768, 65536]
    us = []
    for K in ks:
        A = torch.randn(1, K, device="cuda", generator=g).to(torch.bfloat16)
        W = (torch.randn(128, K, device="cuda", generator=g) * 0.02).to(torch.bfloat16)
        C = torch.empty(1, 128, dtype=torch.float32, device="cuda")
        us.append(time_steps(lambda: bi.gemm(A, W, out=C, c_dtype=bi.F32, stream=stream), max(steps, 20), 3,
                             stream) * 1e3)
    slope, icpt = np.polyfit(np.asarray(ks, np.float64) / 16.0, np.asarray(us), 1)
    c = LLAMA3_8B
    pairs = 76
    chains = {"qkv": (c.d // 16) * -(-(c.qkv_dim // 128) // pairs), "o": (c.H * c.Dh // 16) * -(-(c.d // 128) // pairs),
              "gate_up": (c.d // 16) * -(-(2 * c.F // 128) // pairs), "down": (c.F // 16) * -(-(c.d // 128) // pairs)}
    floor = {k: round(v * slope + icpt, 1) for k, v in chains.items()}  # slope: us per dependent MMA
    return {"shape": "M=1, N=128: one output tile, CTA-pair form 256x128x16", "k": ks, "us": [round(x, 2) for x in us],
            "ns_per_dependent_mma": round(slope * 1e3, 2), "fixed_us": round(icpt, 2),
            "layer_chain_mmas": chains, "layer_chain_floor_us": floor,
            "layer_chain_floor_total_us": round(sum(floor.values()), 1)}


def gemm_floor(stream) -> dict:
    """What bounds a decode projection at M = 1 (one token), measured.  libbi_probe.so times one tcgen05 MMA
    per instruction form (operands resident in shared memory, unrolled issue) and how fast one SM takes in a
    stream (TMA boxes, bulk copies; one CTA per SM).  At M = 1 the projections take the CTA-pair MMA with
    M = 128; a 64-deep K tile costs each SM of a pair four such MMAs and bringing in 10 KB (its 64 W rows and
    the 16-row A box); a projection's tiles run K / 64 such K tiles in a row, in waves over the 76 pairs.  The floor is that chain at the larger of
    the two costs per K tile (no launch overhead); each projection is also timed standalone at M = 1 with
    the L2 flushed before every launch."""
    import ctypes
    import torch
    from invariant_fixed_order_gb300 import bi
    from invariant_fixed_order_gb300 import build as B
    from invariant_fixed_order_gb300.config import LLAMA3_8B
    lib = ctypes.CDLL(B.PROBE_LIB)
    dp = ctypes.POINTER(ctypes.c_double)
    lib.bip_mma_ns.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, dp]
    lib.bip_ingest.argtypes = [ctypes.c_int, ctypes.c_int, dp, dp]

    def mma(cg, m, n, nacc=1):
        v = ctypes.c_double()
        rc = lib.bip_mma_ns(cg, m, n, nacc, ctypes.byref(v))
        if rc != 0:
            raise RuntimeError(f"bip_mma_ns({cg}, {m}, {n}, {nacc}) returned {rc}")
        return round(v.value, 2)

    forms = {"single 128x16": mma(1, 128, 16), "single 128x32": mma(1, 128, 32), "single 128x64": mma(1, 128, 64),
             "single 128x128": mma(1, 128, 128), "single 64x16": mma(1, 64, 16), "pair 256x64": mma(2, 256, 64),
             "pair 256x128": mma(2, 256, 128), "pair 256x256": mma(2, 256, 256), "pair 128x128": mma(2, 128, 128),
             "single 128x64, 4 accumulators alternating": mma(1, 128, 64, 4),
             "pair 256x128, 2 accumulators alternating": mma(2, 256, 128, 2)}
    ingest = {}
    for mode, name in ((0, "tma 2-D boxes, 128 rows x 128 B contiguous"), (1, "bulk 1-D copies of 16 KB"),
                       (2, "tma 3-D weight-ring boxes: 64 rows x 4 K tiles of a 128 KB-row matrix")):
        rows = []
        for ctas in (1, 32, 64, 96, 128, 152):
            a, t = ctypes.c_double(), ctypes.c_double()
            rc = lib.bip_ingest(mode, ctas, ctypes.byref(a), ctypes.byref(t))
            if rc != 0:
                raise RuntimeError(f"bip_ingest({mode}, {ctas}) returned {rc}")
            rows.append({"ctas": ctas, "gbps_per_cta": round(a.value, 1), "gbps_total": round(t.value, 1)})
        ingest[name] = rows
    per_cta = {r["ctas"]: r["gbps_per_cta"] for r in ingest["tma 3-D weight-ring boxes: 64 rows x 4 K tiles of a "
                                                            "128 KB-row matrix"]}
    c = LLAMA3_8B
    pairs = 76
    shapes = {"qkv": (c.qkv_dim, c.d, bi.EP_NONE), "o": (c.d, c.H * c.Dh, bi.EP_RESIDUAL),
              "gate_up": (2 * c.F, c.d, bi.EP_SWIGLU), "down": (c.d, c.F, bi.EP_RESIDUAL)}
    g = torch.Generator(device="cuda").manual_seed(9)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    proj = {}
    for name, (N, K, ep) in shapes.items():
        tiles = N // 128
        waves = -(-tiles // pairs)
        sms = 2 * min(tiles, pairs)
        ktiles = (K // 64) * waves
        mma_ns = 4 * forms["pair 128x128"]
        ingest_ns = 10240 / per_cta[min((1, 32, 64, 96, 128, 152), key=lambda x: abs(x - sms))]
        floor_us = ktiles * max(mma_ns, ingest_ns) / 1e3
        W = (torch.randn(N, K, device="cuda", generator=g) * 0.02).to(torch.bfloat16)
        A = torch.randn(1, K, device="cuda", generator=g).to(torch.bfloat16)
        R = torch.randn(1, N, device="cuda", generator=g).to(torch.bfloat16)

        def run(flush_only=False):
            flush.zero_()
            if flush_only:
                return
            if ep == bi.EP_RESIDUAL:
                bi.gemm(A, W, residual=R, ep=ep, stream=stream)
            elif ep == bi.EP_SWIGLU:
                bi.gemm(A, W, ep=ep, stream=stream)
            else:
                bi.gemm(A, W, stream=stream)
        t = min(time_steps(run, 30, 5, stream) for _ in range(3))
        t0 = min(time_steps(lambda: run(True), 30, 5, stream) for _ in range(3))
        measured = (t - t0) * 1e3
        proj[name] = {"tiles": tiles, "sms": sms, "k_tiles_in_a_row": ktiles, "mma_ns_per_k_tile": round(mma_ns, 1),
                      "ingest_ns_per_k_tile": round(ingest_ns, 1), "floor_us": round(floor_us, 1),
                      "measured_us": round(measured, 1), "measured_over_floor": round(measured / floor_us, 2)}
        del W
    chain = gemm_chain(20, stream)
    return {"mma_ns": forms, "ingest": ingest, "projections_m1": proj,
            "chain_through_the_kernel": {k: chain[k] for k in ("ns_per_dependent_mma", "fixed_us")}}


def logits_ops_time(w: GpuWorkload, steps: int, stream, hbm_peak: float) -> dict:
    """Logprobs (log_softmax) and seeded sampling over the step's B logit rows, standalone with CUDA events.
    log_softmax algorithmic bytes: the logits read once and the logprobs written once."""
    import torch
    from invariant_fixed_order_gb300 import bi
    cfg, B = w.cfg, w.B
    dev = w.d_ids.device
    x = (torch.randn(B, cfg.V, device=dev) * 3.0).float()
    lp = torch.empty_like(x)
    lws = torch.empty(bi.log_softmax_workspace_size(B, cfg.V), dtype=torch.uint8, device=dev)
    ms_ls = time_steps(lambda: bi.log_softmax(x, out=lp, ws=lws, stream=stream), max(steps, 10), 3, stream)
    g = torch.Generator().manual_seed(DATA_SEED)
    seeds = torch.randint(0, 2 ** 31 - 1, (B,), generator=g, dtype=torch.int32).to(dev)
    pos = torch.from_numpy(np.asarray(w.ctx, np.int32)).to(dev)
    temps = torch.full((B,), 0.8, device=dev)
    tok = torch.empty(B, dtype=torch.int32, device=dev)
    ws = torch.empty(bi.sample_workspace_size(B, cfg.V), dtype=torch.uint8, device=dev)
    ms_s = time_steps(lambda: bi.sample(x, seeds, pos, temps, out=tok, ws=ws, stream=stream), max(steps, 10), 3,
                      stream)
    ls_bytes = 2 * B * cfg.V * 4
    return {"rows": B, "V": cfg.V,
            "log_softmax": {"us": round(ms_ls * 1e3, 2), "GBps": round(ls_bytes / (ms_ls * 1e-3) / 1e9, 1),
                            "frac": round(ls_bytes / (ms_ls * 1e-3) / 1e9 / hbm_peak, 3)},
            "sample": {"us": round(ms_s * 1e3, 2), "Gcols_per_s": round(B * cfg.V / (ms_s * 1e-3) / 1e9, 2)}}


def prefill_measure(device: str, steps: int, bf16_peak: float, stream) -> dict:
    """One prefill step of 64 requests (chunks of 256-2048 tokens, contexts from
    position 0) through the same 1-layer + LM-head path, plus the gate/up GEMM
    of that step timed alone for the tensor-core rate."""
    import torch
    from invariant_fixed_order_gb300 import bi, roofline, synth
    from invariant_fixed_order_gb300.config import LLAMA3_8B_1L
    from invariant_fixed_order_gb300.engine import Engine
    cfg = LLAMA3_8B_1L
    lens = [int(x) for x in synth.uniform_ints(64, 256, 2048, DATA_SEED + 1)]
    T = sum(lens)
    max_pages = 2048 // 16 + 1
    eng = Engine(cfg, seed=WEIGHT_SEED, num_pages=sum((L + 15) // 16 for L in lens) + 64, max_pages=max_pages,
                 max_T=T, max_B=64, max_R=64, max_seq=max_pages * 16, device=device)
    table = np.zeros((64, max_pages), np.int32)
    for i, L in enumerate(lens):
        pg = eng.pool.alloc((L + 15) // 16)
        table[i, :len(pg)] = pg
    d_table = torch.from_numpy(table).to(device)
    ids = torch.from_numpy(synth.token_ids(T, cfg.V, DATA_SEED + 2)).to(device)
    rows = list(np.cumsum(lens) - 1)
    logits = torch.empty(64, cfg.V, dtype=torch.float32, device=device)
    tokens = torch.empty(64, dtype=torch.int32, device=device)
    fn = lambda: eng.step(lens, [0] * 64, ids, d_table, rows, logits_out=logits, tokens_out=tokens)
    ms = time_steps(fn, max(2, steps // 10), 1, stream)
    eng.check()
    gemm_fl = roofline.layer_flops(cfg, T) + roofline.gemm_flops(64, cfg.V, cfg.d)
    attn_fl = 4 * cfg.H * cfg.Dh * sum(L * (L + 1) // 2 for L in lens)
    # the step's causal attention alone, on the K/V the step just appended
    q = (torch.randn(T, cfg.H, cfg.Dh, device=device) * 0.5).to(torch.bfloat16)
    cu_q = torch.from_numpy(np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)).to(device)
    pos0 = torch.zeros(64, dtype=torch.int32, device=device)
    aout = torch.empty(T, cfg.H, cfg.Dh, dtype=torch.bfloat16, device=device)
    ams = time_steps(lambda: bi.prefill_attention(q, cu_q, pos0, eng.k[0], eng.v[0], d_table, out=aout,
                                                  stream=stream), 3, 1, stream)
    # the step's largest GEMM alone: gate/up over all T tokens
    y = torch.randn(T, cfg.d, device=device).to(torch.bfloat16)
    hbuf = torch.empty(T, cfg.F, dtype=torch.bfloat16, device=device)
    gms = time_steps(lambda: bi.gemm(y, eng.layers[0]["w_gu"], out=hbuf, ep=bi.EP_SWIGLU, stream=stream), 3, 1,
                     stream)
    gu_tf = roofline.gemm_flops(T, 2 * cfg.F, cfg.d) / (gms * 1e-3) / 1e12
    at_tf = attn_fl / (ams * 1e-3) / 1e12
    sus = sustained_bf16_peak()
    eng.close()
    # fractions of the burst peak (a kernel timed alone) and of the sustained one (these run back to back for
    # tens of milliseconds, long enough for the power cap to lower the clocks)
    return {"requests": 64, "tokens": T, "chunk": [256, 2048], "ms_per_step": round(ms, 3),
            "tokens_per_s": round(T / (ms * 1e-3), 1), "gemm_tflop": round(gemm_fl / 1e12, 2),
            "attention_tflop": round(attn_fl / 1e12, 3),
            "attention": {"us": round(ams * 1e3, 1), "tflops": round(at_tf, 1), "frac": round(at_tf / bf16_peak, 3),
                          "frac_sustained": round(at_tf / sus, 3)},
            "gate_up_gemm": {"us": round(gms * 1e3, 1), "tflops": round(gu_tf, 1),
                             "frac": round(gu_tf / bf16_peak, 3), "peak_tflops": bf16_peak,
                             "frac_sustained": round(gu_tf / sus, 3), "peak_sustained_tflops": sus}}


def model32_measure(device: str, steps: int, hbm_peak: float, stream) -> dict:
    """The full 32-layer Llama-3-8B-shaped model (random-init weights): one decode step (every layer, final
    norm, LM head, greedy argmax) by CUDA-graph replay at bs 1, 16 and 64, invariant vs batch-variant.
    Contexts U[128, 4096] (the prompt lengths of the 32-layer configuration), KV history N(0, 1) in every
    layer, pages from the engine's shuffled pool.  Roofline bytes: every layer's weights, the LM head, each
    request's KV in every layer and the activations (roofline.decode_step_bytes)."""
    import torch
    from invariant_fixed_order_gb300 import bi, roofline, synth
    from invariant_fixed_order_gb300.config import LLAMA3_8B
    from invariant_fixed_order_gb300.engine import Engine
    from invariant_fixed_order_gb300.graphs import DecodeGraphs
    cfg = LLAMA3_8B
    B = 64
    ctx = [int(x) for x in synth.uniform_ints(B, 128, 4096, DATA_SEED + 2)]
    ids = synth.token_ids(B, cfg.V, DATA_SEED + 3)
    max_pages = 4096 // 16 + 1
    pages = sum((s + 15) // 16 for s in ctx)
    eng = Engine(cfg, seed=WEIGHT_SEED, num_pages=pages + 8, max_pages=max_pages, max_T=B, max_B=B, max_R=B,
                 max_seq=max_pages * 16, device=device)
    table = np.zeros((B, max_pages), np.int32)
    for i, s in enumerate(ctx):
        pg = eng.pool.alloc((s + 15) // 16)
        table[i, :len(pg)] = pg
    g = torch.Generator(device=device).manual_seed(DATA_SEED * 7919)
    for layer in range(cfg.n_layers):  # the KV history of every layer: N(0, 1) bf16
        for t in (eng.k[layer], eng.v[layer]):
            t.copy_(torch.randn(t.shape, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16))
    positions = [s - 1 for s in ctx]
    out = {"layers": cfg.n_layers, "context": [128, 4096], "path": "bi_forward_step by CUDA-graph replay",
           "weights_gb": round(roofline.step_weight_bytes(cfg) / 1e9, 2), "rows": []}
    rows = {b: {"bs": b} for b in (1, 16, 64)}
    for name, mode in (("invariant", bi.INVARIANT), ("variant", bi.VARIANT)):
        graphs = DecodeGraphs(eng, max(ctx), ladder=(1, 16, 64), mode=mode)
        for b in (1, 16, 64):
            graphs.step(ids[:b], positions[:b], table[:b], bucket=b)
            t = time_steps(graphs.buckets[b][0].replay, max(steps, 10), 3, stream)
            nbytes = roofline.decode_step_bytes(cfg, ctx[:b])
            rows[b][name + "_tok_s"] = round(b / (t * 1e-3), 1)
            rows[b][name + "_ms"] = round(t, 3)
            rows[b][name + "_hbm_frac"] = round(nbytes / (t * 1e-3) / 1e9 / hbm_peak, 3)
            rows[b]["step_gb"] = round(nbytes / 1e9, 2)
        graphs.close()
    eng.check()
    eng.close()
    out["rows"] = [rows[b] for b in (1, 16, 64)]
    return out


def gemm_traffic(per_launch_bytes_of: str):
    """Per-launch DRAM traffic of gemm_tc_kernel from the committed ncu summary,
    if it was captured on the current kernel source (else None)."""
    import hashlib
    try:
        with open(os.path.join(ROOT, "profiles", "gemm_tc_kernel_traffic.json")) as fh:
            j = json.load(fh)
        with open(os.path.join(ROOT, "invariant_fixed_order_gb300", "csrc", "k_gemm.cu"), "rb") as fh:
            sha = hashlib.sha256(fh.read()).hexdigest()
        if j.get("k_gemm_sha256") != sha or j.get("workload") != per_launch_bytes_of:
            return None
        return j["per_launch_dram_bytes"]
    except Exception:
        return None


# ---------------------------------------------------------------------------
# CPU oracle timing
# ---------------------------------------------------------------------------

class OracleSample:
    """The CPU oracle on the same workload: shapes, contexts, token ids and
    distributions as the GPU run (values drawn by the CPU generator)."""

    def __init__(self, B: int, rank: int):
        import oracle
        import torch
        from invariant_fixed_order_gb300 import synth
        oracle.build()
        self.cfg, self.ctx, self.ids = make_workload(B, rank)
        cfg = self.cfg
        wl = synth.layer_weights(cfg, WEIGHT_SEED, "cpu", 0)
        hd = synth.head_weights(cfg, WEIGHT_SEED, "cpu")
        self.w = {k: synth.to_f32_numpy(v) for k, v in wl.items()}
        self.gamma_final = synth.to_f32_numpy(hd["gamma_final"])
        self.w_lm = synth.to_f32_numpy(hd["w_lm"])
        self.x = synth.to_f32_numpy(hd["embed"][torch.from_numpy(self.ids.astype(np.int64))])
        del wl, hd
        self.dims = oracle.Dims(cfg.d, cfg.H, cfg.Hkv, cfg.Dh, cfg.F, cfg.eps, cfg.rope_theta)
        self.B = B
        self.next = 0

    def run(self, target_s: float) -> dict:
        """One decode step (layer + LM head + argmax) per request, in request
        order (wrapping around), until ~target_s of oracle time."""
        import oracle
        from invariant_fixed_order_gb300 import synth
        cfg = self.cfg
        done, t_total = 0, 0.0
        while t_total < target_s and done < 4 * self.B:
            i = self.next % self.B
            self.next += 1
            n = int(self.ctx[i]) - 1
            k, v = synth.kv_history(max(n, 1), cfg.Hkv, cfg.Dh, DATA_SEED * 7919 + i, device="cpu")
            kf, vf = synth.to_f32_numpy(k), synth.to_f32_numpy(v)
            t0 = time.perf_counter()
            x_out, _, _, _ = oracle.layer_forward(self.dims, self.w, [1], [n], [kf], [vf], self.x[i:i + 1])
            oracle.lm_head(self.dims, self.gamma_final, self.w_lm, x_out, [0])
            t_total += time.perf_counter() - t0
            done += 1
        return {"value": done / t_total, "unit": "tokens/s", "cores": oracle.num_threads(), "kind": "oracle",
                "sample": f"{done} single-request decode steps (1 layer + LM head + argmax) of requests drawn in "
                          f"order from the {self.B}-request batch, {t_total:.1f} s of oracle time; ms_per_step is "
                          f"a whole {self.B}-request step at that rate"}


# ---------------------------------------------------------------------------
# arms
# ---------------------------------------------------------------------------

def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    per_step = max(1.0, min(20.0, 150.0 / max(args.steps + args.warmup, 1)))
    sample = OracleSample(args.batch, 0)
    rates = []
    for i in range(args.warmup + args.steps):
        r = sample.run(per_step)
        if i >= args.warmup:
            rates.append(r)
    value = statistics.median(x["value"] for x in rates)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * args.batch / value,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": run_config(args.batch, args.gpus),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": rates[0]["cores"], "kind": "oracle",
                             "sample": rates[0]["sample"] + " (one timed step)"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ours(args):
    import torch
    rank, world, local_rank = dist_env()
    torch.cuda.set_device(local_rank)
    device = f"cuda:{local_rank}"
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device(device))
    from __graft_entry__ import build
    build()
    from invariant_fixed_order_gb300 import bi
    hbm_peak, _, peak_kind = peaks()

    stream = torch.cuda.current_stream()
    sampler = ClockSampler(local_rank)
    w = GpuWorkload(args.batch, rank, device)
    B = args.batch

    def barrier():
        if world > 1:
            torch.distributed.barrier()

    # ---- the decode step as a CUDA graph (graphs.DecodeGraphs, the serving path), one bucket per sweep size ----
    from invariant_fixed_order_gb300.graphs import DecodeGraphs
    positions = [int(s) - 1 for s in w.ctx]
    ladder = sorted({b for b in (1, 2, 4, 8, 16, 32, 64) if b <= B} | {B})
    graphs = DecodeGraphs(w.eng, int(max(w.ctx)), ladder=tuple(ladder), mode=bi.INVARIANT)
    graphs.step(w.ids, positions, w.table, bucket=B)  # writes the bucket's inputs once (resident from here on)
    replay = graphs.buckets[B][0].replay

    # ---- main timed region: K invariant steps at batch B, replayed with inputs resident ----
    for _ in range(max(args.warmup, 3)):
        replay()
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        replay()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    ms = e0.elapsed_time(e1) / args.steps
    if world > 1:
        from invariant_fixed_order_gb300 import replicas
        ms = replicas.max_over_ranks(ms, device=device)
    w.eng.check()
    value = world * B / (ms * 1e-3)
    # embedding gather + first norm, FFN norm, 4 GEMMs (RoPE + K/V append inside the QKV GEMM's epilogue),
    # decode split, merge, final norm of the gathered rows, LM GEMM (greedy argmax fused into its epilogue):
    # 10 kernels per step (a graph replay launches the same kernels)
    launches_per_step = 10
    # the same step launched eagerly through bi_forward_step, for comparison
    eager_ms = time_steps(lambda: w.step(B, bi.INVARIANT), max(args.steps, 10), 3, stream)

    # ---- e2e: host buffers in, tokens back, through the public API (pinned copies + graph replay) ----
    bufs = graphs.buckets[B][1]
    pin_ids = torch.from_numpy(w.ids).pin_memory()
    pin_table = torch.from_numpy(w.table).pin_memory()
    pin_meta = torch.from_numpy(DecodeGraphs._meta(np.asarray(positions, np.int32), B)).pin_memory()
    pin_tok = torch.empty(B, dtype=torch.int32).pin_memory()

    def e2e_step():
        bufs["ids"].copy_(pin_ids, non_blocking=True)
        bufs["table"].copy_(pin_table, non_blocking=True)
        bufs["meta"].copy_(pin_meta, non_blocking=True)
        replay()
        pin_tok.copy_(bufs["tokens"], non_blocking=True)

    for _ in range(3):
        e2e_step()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        e2e_step()
    torch.cuda.synchronize()
    e2e_ms = (time.perf_counter() - t0) * 1e3 / args.steps
    h2d = (pin_ids.numel() + pin_table.numel() + pin_meta.numel()) * 4
    d2h = B * 4

    # ---- e2e through the C ABI alone: bi_forward_step launched eagerly, its per-token metadata staged by the
    # library from host arrays (q_len, pos0, logit rows), token ids and page table copied in from pinned host
    # memory, tokens copied back; no graph ----
    d_ids_c = torch.empty_like(w.d_ids)
    d_table_c = torch.empty_like(w.d_table)
    tok_c = torch.empty(B, dtype=torch.int32, device=device)
    rows = list(range(B))

    def e2e_cabi_step():
        d_ids_c.copy_(pin_ids, non_blocking=True)
        d_table_c.copy_(pin_table, non_blocking=True)
        w.eng.step([1] * B, positions, d_ids_c, d_table_c, rows, mode=bi.INVARIANT, want_logits=False,
                   tokens_out=tok_c, stream=stream)
        pin_tok.copy_(tok_c, non_blocking=True)

    for _ in range(3):
        e2e_cabi_step()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        e2e_cabi_step()
    torch.cuda.synchronize()
    e2e_cabi_ms = (time.perf_counter() - t0) * 1e3 / args.steps
    h2d_cabi = (pin_ids.numel() + pin_table.numel() + 3 * B + B) * 4  # ids, table, the library's metadata

    # ---- sweep: invariant vs variant over batch sizes ----
    sweep = []
    if not args.no_sweep:
        for b in (1, 2, 4, 8, 16, 32, 64):
            if b > B:
                break
            row = {"bs": b}
            graphs.step(w.ids[:b], positions[:b], w.table[:b], bucket=b)
            t = time_steps(graphs.buckets[b][0].replay, max(args.steps, 10), 3, stream)
            row["invariant_graph_tok_s"] = round(b / (t * 1e-3), 1)
            row["invariant_graph_us"] = round(t * 1e3, 1)
            row["invariant_graph_hbm_frac"] = round(w.step_bytes(b) / (t * 1e-3) / 1e9 / hbm_peak, 3)
            for name, mode in (("invariant", bi.INVARIANT), ("variant", bi.VARIANT)):
                t = time_steps(lambda: w.step(b, mode), max(args.steps, 10), 3, stream)
                row[name + "_tok_s"] = round(b / (t * 1e-3), 1)
                row[name + "_us"] = round(t * 1e3, 1)
                row[name + "_hbm_frac"] = round(w.step_bytes(b) / (t * 1e-3) / 1e9 / hbm_peak, 3)
            # the layer alone against the layer's own bytes (weights once + this batch's KV + activations)
            t = time_steps(lambda: w.step_layer(b, bi.INVARIANT), max(args.steps, 10), 3, stream)
            row["invariant_layer_us"] = round(t * 1e3, 1)
            row["invariant_layer_hbm_frac"] = round(w.layer_bytes(b) / (t * 1e-3) / 1e9 / hbm_peak, 3)
            sweep.append(row)
    w.eng.check()

    # ---- dominant kernel (GEMM) and attention, timed standalone with events ----
    graphs.close()
    g = gemm_roofline(w, args.steps, stream, hbm_peak)
    att = attention_time(w, args.steps, stream)
    lops = logits_ops_time(w, args.steps, stream, hbm_peak)
    chain = gemm_chain(args.steps, stream) if not args.no_sweep else None
    step_bytes = w.step_bytes(B)
    del w
    torch.cuda.empty_cache()
    _, bf16_peak, _ = peaks()
    pre = prefill_measure(device, args.steps, bf16_peak, stream) if not args.no_sweep else None
    torch.cuda.empty_cache()
    m32 = model32_measure(device, args.steps, hbm_peak, stream) if not args.no_sweep else None
    torch.cuda.empty_cache()
    clocks = sampler.stop()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = OracleSample(B, rank).run(args.cpu_seconds)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": run_config(B, world),
            "step_hbm_frac": round(step_bytes / (ms * 1e-3) / 1e9 / hbm_peak, 3),
            "path": "bi_forward_step captured in a CUDA graph (graphs.DecodeGraphs), replayed with inputs resident",
            "roofline": {"bound": "hbm", "kernel": "gemm_tc_kernel", "achieved": round(g["achieved"], 1),
                         "peak": hbm_peak, "unit": "GB/s", "frac": round(g["achieved"] / hbm_peak, 3),
                         "traffic": gemm_traffic(f"decode bs{B}"), "peak_kind": peak_kind,
                         "per_gemm": g["per_gemm"],
                         "per_launch_bytes": int(g["per_launch_bytes"])},
            "attention": att,
            "logits_ops": lops,
            "eager": {"ms_per_step": round(eager_ms, 4), "value": round(world * B / (eager_ms * 1e-3), 1),
                      "step_hbm_frac": round(step_bytes / (eager_ms * 1e-3) / 1e9 / hbm_peak, 3)},
            "e2e": {"value": round(world * B / (e2e_ms * 1e-3), 1), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h,
                    "path": "pinned host ids, page table and step metadata copied into the CUDA graph's buffers, "
                            "graph replay, tokens copied back"},
            "e2e_c_abi": {"value": round(world * B / (e2e_cabi_ms * 1e-3), 1), "unit": "tokens/s",
                          "h2d_bytes_per_step": h2d_cabi, "d2h_bytes_per_step": d2h,
                          "path": "bi_forward_step launched eagerly through the C ABI with host q_len/pos0/logit "
                                  "rows (staged by the library), pinned host ids and page table copied in, tokens "
                                  "copied back"},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks,
            "sweep": sweep,
        }
        if chain is not None:
            line["gemm_chain"] = chain
        if pre is not None:
            line["prefill"] = pre
        if m32 is not None:
            line["model32"] = m32
        if cpu is not None:
            line["cpu_baseline"] = cpu
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def ncu_target(which: str) -> None:
    """The GEMM launches the committed profiles capture: the five decode-step
    GEMMs at M = 64, or the prefill gate/up GEMM at M = 8192 (random weights)."""
    import torch
    from __graft_entry__ import build
    build()
    from invariant_fixed_order_gb300 import bi
    from invariant_fixed_order_gb300.config import LLAMA3_8B
    c = LLAMA3_8B
    g = torch.Generator(device="cuda").manual_seed(0)

    def rnd(*shape, std=1.0):
        return (torch.randn(*shape, device="cuda", generator=g) * std).to(torch.bfloat16)

    if which == "prefill-attn16":
        # causal prefill attention of 16 prompts of U[256, 2048] tokens on random K/V (launched twice)
        from invariant_fixed_order_gb300 import synth
        lens = [int(x) for x in synth.uniform_ints(16, 256, 2048, DATA_SEED + 1)]
        T = sum(lens)
        max_pages = 2048 // 16 + 1
        n_pages = sum((L + 15) // 16 for L in lens)
        kc = rnd(n_pages, c.Hkv, 16, c.Dh)
        vc = rnd(n_pages, c.Hkv, 16, c.Dh)
        table = torch.zeros(16, max_pages, dtype=torch.int32, device="cuda")
        p0 = 0
        for i, L in enumerate(lens):
            n = (L + 15) // 16
            table[i, :n] = torch.arange(p0, p0 + n, dtype=torch.int32, device="cuda")
            p0 += n
        q = rnd(T, c.H, c.Dh)
        cu_q = torch.tensor([0] + list(np.cumsum(lens)), dtype=torch.int32, device="cuda")
        pos0 = torch.zeros(16, dtype=torch.int32, device="cuda")
        for _ in range(2):
            bi.prefill_attention(q, cu_q, pos0, kc, vc, table)
        torch.cuda.synchronize()
        print(json.dumps({"ncu_target": which, "done": True}))
        return
    if which == "decode-attn16":
        # decode attention of 16 requests with contexts U[128, 8192] (the bench's distribution) over paged K/V in
        # a shuffled pool (launched twice)
        from invariant_fixed_order_gb300 import synth
        ctx = [int(x) for x in synth.uniform_ints(16, 128, 8192, DATA_SEED)]
        max_pages = 8192 // 16 + 1
        n_pages = sum((s + 15) // 16 for s in ctx)
        kc = rnd(n_pages, c.Hkv, 16, c.Dh)
        vc = rnd(n_pages, c.Hkv, 16, c.Dh)
        perm = np.random.default_rng(DATA_SEED).permutation(n_pages).astype(np.int32)
        table = np.zeros((16, max_pages), np.int32)
        p0 = 0
        for i, s in enumerate(ctx):
            n = (s + 15) // 16
            table[i, :n] = perm[p0:p0 + n]
            p0 += n
        q = rnd(16, c.H, c.Dh)
        sl = torch.tensor(ctx, dtype=torch.int32, device="cuda")
        d_table = torch.from_numpy(table).cuda()
        for _ in range(2):
            bi.decode_attention(q, kc, vc, d_table, sl, max(ctx))
        torch.cuda.synchronize()
        print(json.dumps({"ncu_target": which, "kv_bytes": sum(2 * s * c.Hkv * c.Dh * 2 for s in ctx), "done": True}))
        return
    if which == "gemm-o-m1":
        # the decode-step o projection at M = 1 with its residual epilogue (launched twice)
        A, W = rnd(1, c.H * c.Dh), rnd(c.d, c.H * c.Dh, std=0.02)
        res = rnd(1, c.d)
        for _ in range(2):
            bi.gemm(A, W, out=res, residual=res, ep=bi.EP_RESIDUAL)
        torch.cuda.synchronize()
        print(json.dumps({"ncu_target": which, "done": True}))
        return
    if which == "gemm-decode64":
        shapes = [(c.qkv_dim, c.d, bi.F32, bi.EP_NONE), (c.d, c.H * c.Dh, bi.BF16, bi.EP_RESIDUAL),
                  (2 * c.F, c.d, bi.BF16, bi.EP_SWIGLU), (c.d, c.F, bi.BF16, bi.EP_RESIDUAL),
                  (c.V, c.d, bi.F32, bi.EP_NONE)]
        for _ in range(2):
            for N, K, dt, ep in shapes:
                A, W = rnd(64, K), rnd(N, K, std=0.02)
                res = rnd(64, N) if ep == bi.EP_RESIDUAL else None
                bi.gemm(A, W, c_dtype=dt, residual=res, out=res, ep=ep)
    else:
        A, W = rnd(8192, c.d), rnd(2 * c.F, c.d, std=0.02)
        for _ in range(2):
            bi.gemm(A, W, ep=bi.EP_SWIGLU)
    torch.cuda.synchronize()
    print(json.dumps({"ncu_target": which, "done": True}))


def main():
    args = parse()
    if args.floor:
        import torch
        from __graft_entry__ import build
        build()
        print(json.dumps({"gemm_floor": gemm_floor(torch.cuda.current_stream())}))
        return
    if args.ncu_target:
        ncu_target(args.ncu_target)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()

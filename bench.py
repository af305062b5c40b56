#!/usr/bin/env python
"""Throughput of the token early-exit step on one GB300 (or N replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

A step is one pass of the whole hot path over one batch of synthetic input:
  decode-1b (default): cosine gate (batch-min) -> compaction with gather ->
      exit scatter (the three in one launch) -> KV fill of 8 layers (identity
      map, int4 Wk/Wv), for a 64-token Llama-3.2-1B-shaped decode batch;
  decode-tiny: the same on the tiny fp32 workload;
  router-32 / router-4096: router gate -> compaction with gather, 32 or 4096
      tokens, d = 4096;
  router-65536: the same at 65,536 tokens (inputs far larger than L2), with the
      cosine gate and the exit scatter at that batch timed alongside;
  prefill-16k / prefill-120k: the RidgeFill KV fill of every layer after the
      split for all filled rows;
  river-1b / river-tiny: River-LLM's Exit River -- 64 exited tokens through the
      W4A16 copies of 8 Llama-3.2-1B-shaped layers (attention over a 4096-slot
      cache, FFN), one call;
  ridge-4096: RidgeFill's closed-form map fitted on the GPU from 16,384 bf16
      calibration rows at d = 4096 (the Gram GEMMs, the Cholesky and the solves).
L2 is flushed (a write larger than L2) between timed steps, outside the timed
events, except where every input is larger than L2 (router-65536). Under torchrun each rank runs its own replica (independent batches,
no collective on the data path: weak scaling); rank 0 prints one JSON line.
The reference arm (--impl reference) times the CPU oracle on a bounded sample
of the same workload on the host cores.
"""
from __future__ import annotations

import os

# The CPU oracle (single-threaded C++) is timed on one core; pin every BLAS /
# OpenMP pool to one thread too (numpy only marshals arrays for it), whatever
# the environment says.
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ[_v] = "1"

import argparse  # noqa: E402
import hashlib  # noqa: E402
import json  # noqa: E402
import statistics  # noqa: E402
import subprocess  # noqa: E402
import tempfile  # noqa: E402
import sys  # noqa: E402
import time  # noqa: E402

import numpy as np  # noqa: E402
import torch  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from workloads import configs, gen  # noqa: E402

METRIC = "tokens/s through exit gate+compact+KV fill"
RIVER_METRIC = "tokens/s through the Exit River (W4A16 exit layers)"
RIDGE_METRIC = "calibration rows/s through the ridge fit (RidgeFill's closed-form map)"
RIDGE_SHAPE = (16384, 4096)       # calibration rows, d (d_out = d)
RIDGE_SAMPLE = (2048, 256)        # the oracle's bounded sample (the float64 fit at d = 4096 takes minutes)
WORKLOADS = ("decode-1b", "decode-tiny", "router-32", "router-4096", "router-65536", "prefill-16k", "prefill-120k", "river-1b", "ridge-4096",
             "river-tiny")


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        j = json.load(open(p))
        return {"hbm_gbs": j["hbm_gbs"], "bf16_tflops": j["bf16_tflops"],
                "bf16_tflops_sustained": j.get("bf16_tflops_sustained", j["bf16_tflops"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def traffic(key):
    """DRAM bytes per call of the dominant kernel, from the ncu capture recorded in
    profiles/traffic.json, or None when there is none or the kernel's source has
    changed since it was taken."""
    if key is None:
        return None
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    e = json.load(open(p)).get(key)
    if not e:
        return None
    src = os.path.join(ROOT, e["source"])
    if not os.path.exists(src) or hashlib.sha256(open(src, "rb").read()).hexdigest() != e["sha256"]:
        return None
    return int(e["dram_bytes_per_launch"]) * int(e.get("launches_per_call", 1))


# --------------------------------------------------------------------------- workloads

# --------------------------------------------------------------------------- workload descriptions

def decode_config(c, case):
    return {"workload": c.name, "tokens_per_step": c.batch, "d": c.d, "fill_layers": len(c.fill_layers),
            "kv_heads": c.n_kv_heads, "head_dim": c.head_dim, "cache_len": c.cache_len, "gate": "cosine",
            "rule": c.rule, "tau": c.tau, "map": c.map, "weights": c.weights, "case": case,
            "l2": "flushed between timed steps"}


def router_config(c, n, theta, flush):
    return {"workload": f"{c.name}-n{n}", "tokens_per_step": n, "d": c.d, "bottleneck": c.bottleneck,
            "theta": theta, "gate": "router", "rule": "per_token", "gather": True,
            "l2": "flushed between timed steps" if flush else "inputs larger than L2 (no flush)"}


def router_flush(c, n, dev):
    """h alone twice L2 or more: no flush between steps (its lines are gone anyway)."""
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size if dev.type == "cuda" else 126 << 20
    return n * c.d * 2 < 2 * l2


def prefill_config(c, rows, n_layers):
    name = c.name if (rows, n_layers) == (c.filled_rows, len(c.fill_layers)) else \
        f"{c.name}-reduced-{rows}rows-{n_layers}layers"
    return {"workload": name, "tokens_per_step": rows, "d": c.d, "fill_layers": n_layers,
            "kv_heads": c.n_kv_heads, "head_dim": c.head_dim, "prompt_tokens": c.tokens,
            "exact_tail": c.exact_tail, "map": "ridge (N(0,1/d)+0.5I)", "weights": "bf16 dense",
            "l2": "inputs larger than L2; flushed between timed steps"}


def river_cfg(cfg, rows=None, layers=None):
    import dataclasses
    if not (rows or layers):
        return cfg
    return dataclasses.replace(cfg, batch=rows or cfg.batch,
                               river_layers=cfg.river_layers[:layers] if layers else cfg.river_layers,
                               name=f"{cfg.name}-reduced-{rows or cfg.batch}tokens-"
                                    f"{layers or len(cfg.river_layers)}layers")


def river_bytes(cfg, pos):
    """Algorithmic bytes of one Exit River call: the int4 weights (codes, scales,
    zeros) and norm weights of every layer, the K/V rows 0..pos that the
    attention reads, the slots written, h in and out."""
    L = len(cfg.river_layers)
    d, f, qw, kvw, g = cfg.d, cfg.d_ff, cfg.qw, cfg.kvw, cfg.group
    mats = [(d, qw), (d, kvw), (d, kvw), (qw, d), (d, f), (d, f), (f, d)]
    w_layer = sum(k * n // 2 + 2 * (k // g) * n * 2 for k, n in mats) + 2 * d * 2
    p = pos.cpu().numpy().astype(np.int64)
    kv_read = int((p + 1).sum()) * kvw * 2 * 2
    kv_write = cfg.batch * kvw * 2 * 2
    return L * (w_layer + kv_read + kv_write) + 2 * cfg.batch * d * 2


def river_config(c, nbytes):
    return {"workload": c.name, "tokens_per_step": c.batch, "d": c.d, "river_layers": len(c.river_layers),
            "q_heads": c.n_q_heads, "kv_heads": c.n_kv_heads, "head_dim": c.head_dim, "d_ff": c.d_ff,
            "cache_len": c.cache_len, "positions": "U[0, cache_len) per sequence",
            "weights": "int4 group-64 (W4A16), every matrix", "algorithmic_bytes_per_step": nbytes,
            "l2": "inputs larger than L2 (the KV cache read); flushed between timed steps"}


def unit_for(name):
    return "rows/s" if name.startswith("ridge") else "tokens/s"


def metric_for(name):
    return RIVER_METRIC if name.startswith("river") else RIDGE_METRIC if name.startswith("ridge") else METRIC


def ridge_config(n, d):
    return {"workload": f"ridge-fit-d{d}-n{n}", "rows": n, "d": d, "d_out": d, "lambda": 0.5, "inputs": "bf16",
            "solve": "fp32 blocked Cholesky", "l2": "flushed between timed steps"}


def reference_config(name, dev, seed=0, rows=None, layers=None):
    """The ``config`` of a workload as the GPU arm reports it, from the
    configurations and the generator alone."""
    if name in ("decode-1b", "decode-tiny"):
        cfg = configs.LLAMA1B_DECODE if name == "decode-1b" else configs.TINY_DECODE
        return decode_config(cfg, "exit" if cfg.rule == "batch_all" else "default")
    if name in ("router-32", "router-4096", "router-65536"):
        n = {"router-32": 32, "router-4096": 4096}.get(name) or (rows or 65536)
        return router_config(configs.ROUTER_4096, n, 0.5, router_flush(configs.ROUTER_4096, n, dev))
    if name == "ridge-4096":
        return ridge_config(*RIDGE_SHAPE)
    if name in ("prefill-16k", "prefill-120k"):
        cfg = configs.PREFILL_16K if name == "prefill-16k" else configs.PREFILL_120K
        return prefill_config(cfg, cfg.filled_rows if rows is None else rows,
                              len(cfg.fill_layers) if layers is None else layers)
    cfg = river_cfg(configs.LLAMA1B_RIVER if name == "river-1b" else configs.TINY_RIVER, rows, layers)
    return river_config(cfg, river_bytes(cfg, gen.river_positions(cfg, seed, dev)))


class Decode:
    """gate -> compact (+gather) -> kv_fill -> scatter on one decode batch."""

    def __init__(self, tee, cfg, dev, seed=0, case=None):
        self.tee, self.cfg, self.dev = tee, cfg, dev
        case = case or ("exit" if cfg.rule == "batch_all" else "default")
        self.case = case
        self.x = gen.decode_inputs(cfg, seed=seed, device=dev, case=case)
        self.ws = tee.Workspace(dev)
        self.fill = tee.KVFill(self.x["layers"], d=cfg.d, n_kv_heads=cfg.n_kv_heads, head_dim=cfg.head_dim,
                               rope_base=cfg.rope_base, eps=cfg.eps, dtype=self.x["h_cur"].dtype,
                               max_pos=cfg.cache_len, int4=cfg.weights == "int4", group=cfg.group,
                               early_weights=True)   # the step's kernels never write the weights
        n, d = cfg.batch, cfg.d
        dt = self.x["h_cur"].dtype
        self.g_out = {"score": torch.empty(n, device=dev), "mask": torch.empty(n, dtype=torch.uint8, device=dev),
                      "flag": torch.empty(1, dtype=torch.int32, device=dev)}
        self.c_out = {k: torch.empty(n, dtype=torch.int32, device=dev)
                      for k in ("cont_rows", "exit_rows", "cont_pos", "exit_pos")}
        self.c_out["counts"] = torch.empty(2, dtype=torch.int32, device=dev)
        self.c_out["h_cont"] = torch.empty(n, d, dtype=dt, device=dev)
        self.c_out.update(self.g_out)   # the front writes score, mask and flag into the same dict
        self.out = torch.zeros(n, d, dtype=dt, device=dev)
        # the end-to-end run: host buffers in, host buffers out, one library call a step
        self.step_host = tee.DecodeStep(self.fill, n_max=n, d=d, threshold=cfg.tau, dtype=dt, rule=cfg.rule,
                                        k_cache=self.x["k_cache"], v_cache=self.x["v_cache"])
        self.units = n
        self.kernel = "kv_fill"
        # the decode kernels with a recorded ncu capture: int4 (identity map, bf16) and the tiny fp32 one
        self.traffic_key = ("kv_fill/decode" if cfg.weights == "int4" and cfg.map == "identity" and cfg.dtype == "bf16"
                            else "kv_fill/decode-tiny" if cfg is configs.TINY_DECODE else None)
        # algorithmic bytes of the fill call: weights + the h rows + K/V written
        L = len(cfg.fill_layers)
        kvw = cfg.kvw
        if cfg.weights == "int4":
            wbytes = 2 * (d * kvw // 2 + 2 * (d // cfg.group) * kvw * 2)
        else:
            wbytes = 2 * d * kvw * dt.itemsize
        if cfg.map != "identity":
            wbytes += d * d * dt.itemsize
        wbytes += d * dt.itemsize  # gamma
        self.n_exit_expected = None
        self._fill_bytes_per_item_layer = 2 * kvw * dt.itemsize
        self._fill_weight_bytes = L * wbytes
        self._h_row_bytes = d * dt.itemsize
        self.bound = "hbm"

    def fill_bytes(self, n_exit):
        L = len(self.cfg.fill_layers)
        return self._fill_weight_bytes + n_exit * (self._h_row_bytes + L * self._fill_bytes_per_item_layer)

    def parts(self):
        tee, cfg, x = self.tee, self.cfg, self.x

        def front():
            # cosine gate, compaction (continuing rows gathered) and the exit scatter
            # of the exiting rows to their slots of the output: one launch
            tee.exit_gate_compact_scatter(x["h_cur"], x["h_prev"], cfg.tau, self.out, rule=cfg.rule, ws=self.ws,
                                          res=self.c_out)

        def fill():
            self.fill(x["h_cur"], x["k_cache"], x["v_cache"], rows=self.c_out["exit_rows"], pos=x["pos"],
                      seq=x["seq"], n_dev=self.c_out["counts"][1:], n_max=cfg.batch, ws=self.ws)
        # The fill's early launch (TEE_FILL_EARLY_WEIGHTS) streams its weights while the
        # front runs.
        return [front, fill], 1

    def step(self):
        for f in self.parts()[0]:
            f()

    def host_io(self):
        """Pinned host copies of the step's inputs and outputs for the end-to-end run."""
        x = self.x
        self.h_in = {k: x[k].cpu().pin_memory() for k in ("h_prev", "h_cur", "pos", "seq")}
        self.h_out = {"score": torch.empty(self.cfg.batch).pin_memory(),
                      "mask": torch.empty(self.cfg.batch, dtype=torch.uint8).pin_memory(),
                      "counts": torch.empty(2, dtype=torch.int32).pin_memory(),
                      "out": torch.empty_like(self.out, device="cpu").pin_memory()}
        bi = sum(t.numel() * t.element_size() for t in self.h_in.values())
        bo = sum(t.numel() * t.element_size() for t in self.h_out.values())
        return bi, bo

    def e2e_step(self):
        # tee_decode_step_run_host: the inputs' copies, the front, the fill and the
        # results' copies in one call
        hi, ho = self.h_in, self.h_out
        self.step_host.run_host(hi["h_prev"], hi["h_cur"], hi["pos"], hi["seq"], score=ho["score"], mask=ho["mask"],
                                counts=ho["counts"], out=ho["out"])

    def n_exit(self):
        return int(self.c_out["counts"][1].item())

    def config(self):
        return decode_config(self.cfg, self.case)



class Router:
    """Router gate -> compaction with gather at one checkpoint."""

    def __init__(self, tee, cfg, dev, seed=0, n=4096, theta=0.5):
        self.tee, self.cfg, self.dev, self.n, self.theta = tee, cfg, dev, n, theta
        k = cfg.checkpoints[0]
        self.w = gen.router_weights(cfg, k, seed=seed, device=dev)
        self.h = gen.router_hidden(cfg, n, k, seed=seed, device=dev)
        self.ws = tee.Workspace(dev)
        self.g_out = {"score": torch.empty(n, device=dev), "mask": torch.empty(n, dtype=torch.uint8, device=dev),
                      "flag": torch.empty(1, dtype=torch.int32, device=dev)}
        self.c_out = {k2: torch.empty(n, dtype=torch.int32, device=dev) for k2 in ("cont_rows", "exit_rows")}
        self.c_out["counts"] = torch.empty(2, dtype=torch.int32, device=dev)
        self.c_out["h_cont"] = torch.empty(n, cfg.d, dtype=self.h.dtype, device=dev)
        self.units = n
        self.kernel = "exit_gate(router)"
        self.traffic_key = f"exit_gate(router)/n{n}"   # recorded ncu captures: 4096 and 65,536 tokens
        self.bound = "hbm"
        self.flush = router_flush(cfg, n, dev)

    def fill_bytes(self, n_exit):
        d, b = self.cfg.d, self.cfg.bottleneck
        return self.n * d * 2 + b * d * 2 + b * 2 + self.n * 5

    def kernels(self):
        """Each kernel of the path at this batch as its own call: (name, call, algorithmic bytes).
        Besides the step's router gate and compaction, the cosine gate (a second
        hidden state of the same shape) and the exit scatter of the exiting rows."""
        if self.n < 16384:
            return []
        tee, n, d = self.tee, self.n, self.cfg.d
        gen_ = torch.Generator(device=self.dev)
        gen_.manual_seed(1)
        h_prev = (self.h.float() + 0.3 * torch.randn(n, d, device=self.dev, generator=gen_)).to(self.h.dtype)
        c_out = dict(self.c_out)
        pos = torch.arange(n, dtype=torch.int32, device=self.dev)
        c_out["cont_pos"] = torch.empty(n, dtype=torch.int32, device=self.dev)
        c_out["exit_pos"] = torch.empty(n, dtype=torch.int32, device=self.dev)
        self.tee.exit_gate(self.h, self.theta, w_down=self.w["w_down"], w_up=self.w["w_up"], eps=self.cfg.eps,
                           ws=self.ws, out=self.g_out)
        tee.exit_compact(self.g_out["mask"], pos_in=pos, h=self.h, ws=self.ws, out=c_out)
        torch.cuda.synchronize(self.dev)
        n_cont, n_exit = [int(v) for v in c_out["counts"].tolist()]
        out = torch.empty(n, d, dtype=self.h.dtype, device=self.dev)
        g_out = {k: torch.empty_like(v) for k, v in self.g_out.items()}
        self._keep = (h_prev, c_out, pos, out, g_out)
        return [
            ("exit_gate(cosine, per_token)",
             lambda: tee.exit_gate(self.h, 0.95, h_prev=h_prev, ws=self.ws, out=g_out), 2 * n * d * 2 + 5 * n),
            ("exit_gate(router)",
             lambda: tee.exit_gate(self.h, self.theta, w_down=self.w["w_down"], w_up=self.w["w_up"],
                                   eps=self.cfg.eps, ws=self.ws, out=g_out), self.fill_bytes(0)),
            ("exit_compact(gather, positions)",
             lambda: tee.exit_compact(self.g_out["mask"], pos_in=pos, h=self.h, ws=self.ws, out=c_out),
             n + 4 * n + 16 * n + 8 + 2 * n_cont * d * 2),
            ("exit_scatter",
             lambda: tee.exit_scatter(c_out["counts"], c_out["exit_rows"], c_out["exit_pos"], self.h, out,
                                      ws=self.ws), 2 * n_exit * d * 2 + 8 * n_exit + 8),
        ]

    def parts(self):
        def gate():
            self.tee.exit_gate(self.h, self.theta, w_down=self.w["w_down"], w_up=self.w["w_up"], eps=self.cfg.eps,
                               ws=self.ws, out=self.g_out)

        def compact():
            self.tee.exit_compact(self.g_out["mask"], h=self.h, ws=self.ws, out=self.c_out, with_pos=False)
        return [gate, compact], 0

    def step(self):
        for f in self.parts()[0]:
            f()

    def host_io(self):
        self.h_in = {"h": self.h.cpu().pin_memory()}
        self.h_out = {"mask": torch.empty(self.n, dtype=torch.uint8).pin_memory(),
                      "counts": torch.empty(2, dtype=torch.int32).pin_memory()}
        return (sum(t.numel() * t.element_size() for t in self.h_in.values()),
                sum(t.numel() * t.element_size() for t in self.h_out.values()))

    def e2e_step(self):
        self.h.copy_(self.h_in["h"], non_blocking=True)
        self.step()
        self.h_out["mask"].copy_(self.g_out["mask"], non_blocking=True)
        self.h_out["counts"].copy_(self.c_out["counts"], non_blocking=True)

    def n_exit(self):
        return int(self.c_out["counts"][1].item())

    def config(self):
        return router_config(self.cfg, self.n, self.theta, self.flush)



class Prefill:
    """RidgeFill KV fill of every layer after the split, for all filled rows."""

    def __init__(self, tee, cfg, dev, seed=0, rows=None, layers=None):
        self.tee, self.cfg, self.dev = tee, cfg, dev
        self.rows = cfg.filled_rows if rows is None else rows
        self.x = gen.prefill_inputs(cfg, seed=seed, device=dev, rows=rows, layers=layers)
        self.n_layers = len(self.x["layers"])
        self.ws = tee.Workspace(dev)
        self.fill = tee.KVFill(self.x["layers"], d=cfg.d, n_kv_heads=cfg.n_kv_heads, head_dim=cfg.head_dim,
                               rope_base=cfg.rope_base, eps=cfg.eps, dtype=torch.bfloat16, max_pos=cfg.tokens)
        self.units = self.rows
        self.kernel = "kv_fill"
        full = (self.rows, self.n_layers) == (cfg.filled_rows, len(cfg.fill_layers))
        self.traffic_key = "kv_fill/prefill-16k" if full and cfg is configs.PREFILL_16K else None
        self.bound = "tensor"
        d, kvw = cfg.d, cfg.kvw
        self.flops = float(self.n_layers) * self.rows * (2 * d * d + 4 * d * kvw)

    def fill_bytes(self, n_exit):
        return self.flops  # tensor-bound: FLOPs

    def parts(self):
        def fill():
            self.fill(self.x["h_split"], self.x["k_cache"], self.x["v_cache"], ws=self.ws)
        return [fill], 0

    def step(self):
        for f in self.parts()[0]:
            f()

    def host_io(self):
        # inputs: the split-layer rows; output read back: the K/V of the last filled row of each layer
        self.h_in = {"h_split": self.x["h_split"].cpu().pin_memory()}
        kc = self.x["k_cache"]
        self.h_out = {"k_last": torch.empty(kc.shape[0], kc.shape[2], kc.shape[4], dtype=kc.dtype).pin_memory()}
        return (sum(t.numel() * t.element_size() for t in self.h_in.values()),
                sum(t.numel() * t.element_size() for t in self.h_out.values()))

    def e2e_step(self):
        self.x["h_split"].copy_(self.h_in["h_split"], non_blocking=True)
        self.step()
        self.h_out["k_last"].copy_(self.x["k_cache"][:, 0, :, self.rows - 1], non_blocking=True)

    def n_exit(self):
        return self.rows

    def config(self):
        return prefill_config(self.cfg, self.rows, self.n_layers)



class River:
    """The Exit River: the exited tokens through the W4A16 copies of the
    remaining layers (attention over the shared cache + FFN), one call."""

    def __init__(self, tee, cfg, dev, seed=0, rows=None, layers=None):
        cfg = river_cfg(cfg, rows, layers)
        self.tee, self.cfg, self.dev = tee, cfg, dev
        self.x = gen.river_inputs(cfg, seed, dev)
        self.ws = tee.Workspace(dev)
        self.river = tee.ExitRiver(self.x["layers"], d=cfg.d, n_q_heads=cfg.n_q_heads, n_kv_heads=cfg.n_kv_heads,
                                   head_dim=cfg.head_dim, d_ff=cfg.d_ff, rope_base=cfg.rope_base, eps=cfg.eps,
                                   max_pos=cfg.cache_len)
        self.out = torch.empty(cfg.batch, cfg.d, dtype=torch.bfloat16, device=dev)
        self.units = cfg.batch
        self.kernel = "exit_river (all launches of the call)"
        self.metric = RIVER_METRIC
        self.traffic_key = None
        self.bound = "hbm"
        self._bytes = river_bytes(cfg, self.x["pos"])

    def fill_bytes(self, n_exit):
        return self._bytes

    def parts(self):
        x = self.x

        def river():
            self.river(x["h"], x["k_cache"], x["v_cache"], x["pos"], seq=x["seq"], out=self.out, ws=self.ws)
        return [river], 0

    def step(self):
        for f in self.parts()[0]:
            f()

    def host_io(self):
        x = self.x
        self.h_in = {k: x[k].cpu().pin_memory() for k in ("h", "pos", "seq")}
        self.h_out = {"out": torch.empty_like(self.out, device="cpu").pin_memory()}
        return (sum(t.numel() * t.element_size() for t in self.h_in.values()),
                sum(t.numel() * t.element_size() for t in self.h_out.values()))

    def e2e_step(self):
        for k, t in self.h_in.items():
            self.x[k].copy_(t, non_blocking=True)
        self.step()
        self.h_out["out"].copy_(self.out, non_blocking=True)

    def n_exit(self):
        return self.cfg.batch

    def config(self):
        return river_config(self.cfg, self._bytes)



class Ridge:
    """RidgeFill's map W = (X^T X + 0.5 I)^-1 X^T Y fitted on the GPU (tee_ridge_fit)."""

    def __init__(self, tee, dev, seed=0):
        n, d = RIDGE_SHAPE
        self.tee, self.dev, self.n, self.d = tee, dev, n, d
        self.x = gen.ridge_inputs(n, d, seed, dev)
        self.w = torch.empty(d, d, device=dev)
        self.ws = tee.Workspace(dev)
        self.units = n
        self.kernel = "ridge_fit (all launches of the call)"
        self.metric = RIDGE_METRIC
        self.traffic_key = None
        self.bound = "tensor"

    def fill_bytes(self, n_exit):
        """Algorithmic FLOPs: the two Gram products (2 n d^2 each), the Cholesky (d^3 / 3)
        and the two triangular solves (d^2 d_out each)."""
        n, d = self.n, self.d
        return 4.0 * n * d * d + d ** 3 / 3.0 + 2.0 * d ** 3

    def parts(self):
        def fit():
            self.tee.ridge_fit(self.x["x"], self.x["y"], 0.5, ws=self.ws, out=self.w)
        return [fit], 0

    def step(self):
        for f in self.parts()[0]:
            f()

    def host_io(self):
        self.h_in = {k: self.x[k].cpu().pin_memory() for k in ("x", "y")}
        self.h_out = {"w": torch.empty_like(self.w, device="cpu").pin_memory()}
        return (sum(t.numel() * t.element_size() for t in self.h_in.values()),
                sum(t.numel() * t.element_size() for t in self.h_out.values()))

    def e2e_step(self):
        for k, t in self.h_in.items():
            self.x[k].copy_(t, non_blocking=True)
        self.step()
        self.h_out["w"].copy_(self.w, non_blocking=True)

    def n_exit(self):
        return self.n

    def config(self):
        return ridge_config(self.n, self.d)


# --------------------------------------------------------------------------- the oracle (CPU baseline)

def _host(x):
    """Tensors (and dicts / lists of them) -> numpy on the host: float64 for
    floating point, as stored for integers."""
    if torch.is_tensor(x):
        return x.detach().double().cpu().numpy() if x.dtype.is_floating_point else x.detach().cpu().numpy()
    if isinstance(x, dict):
        return {k: _host(v) for k, v in x.items()}
    if isinstance(x, (list, tuple)):
        return [_host(v) for v in x]
    return x


def oracle_sample(name, dev, seed=0, rows=None, layers=None):
    """A bounded sample of the workload for the CPU oracle: (run, description).

    The inputs come from the seeded generator alone (drawn with torch on
    ``dev``, a GPU or the CPU, and copied to the host as float64); nothing
    here builds, loads or calls the CUDA library. ``run()`` computes the
    sample with the C++ oracle and returns the tokens it stands for."""
    import oracle
    if name == "ridge-4096":
        n_s, d_s = RIDGE_SAMPLE
        x = gen.ridge_inputs(n_s, d_s, seed, dev)
        xh, yh = _host(x["x"]), _host(x["y"])

        def run():
            oracle.ridge_fit(xh, yh, 0.5)
            return n_s
        return run, (f"the oracle's fit of {n_s} rows at d = d_out = {d_s} (rows/s at that d; the float64 fit at "
                     f"d = 4096 is a multi-minute job)")
    if name in ("decode-1b", "decode-tiny"):
        cfg = configs.LLAMA1B_DECODE if name == "decode-1b" else configs.TINY_DECODE
        case = "exit" if cfg.rule == "batch_all" else "default"
        x = gen.decode_inputs(cfg, seed=seed, device=dev, case=case, with_cache=False)
        hp, hc, layers_h = _host(x["h_prev"]), _host(x["h_cur"]), _host(x["layers"])
        pos = x["pos"].cpu().numpy()

        def run():
            s, m, f = oracle.cosine_gate(hp, hc, cfg.tau, cfg.rule)
            part = oracle.stable_partition(m)
            oracle.gather_rows(hc, part["cont_rows"])
            r = part["exit_rows"]
            for L in layers_h:
                if len(r):
                    oracle.fill_rows(hc[r], L, pos[r], cfg.n_kv_heads, cfg.head_dim, cfg.rope_base, cfg.eps,
                                     cfg.group)
            oracle.exit_scatter(np.zeros_like(hc), hc, r, r)
            return cfg.batch
        return run, "one full decode step (all tokens)"
    if name in ("router-32", "router-4096", "router-65536"):
        cfg = configs.ROUTER_4096
        n = {"router-32": 32, "router-4096": 4096}.get(name) or (rows or 65536)
        k, m, theta = cfg.checkpoints[0], min(256, n), 0.5
        w = _host(gen.router_weights(cfg, k, seed=seed, device=dev))
        h = _host(gen.router_hidden(cfg, n, k, seed=seed, device=dev)[:m])

        def run():
            p, mask, _ = oracle.router_gate(h, w["w_down"], w["w_up"], theta, "per_token", eps=cfg.eps)
            part = oracle.stable_partition(mask)
            oracle.gather_rows(h, part["cont_rows"])
            return m
        return run, f"router gate + compaction with gather on the first {m} of {n} tokens"
    if name in ("prefill-16k", "prefill-120k"):
        cfg = configs.PREFILL_16K if name == "prefill-16k" else configs.PREFILL_120K
        n_rows = cfg.filled_rows if rows is None else rows
        x = gen.prefill_inputs(cfg, seed=seed, device=dev, rows=rows, layers=layers, with_cache=False)
        sample = np.arange(16) * (n_rows // 16)
        h = _host(x["h_split"][torch.as_tensor(sample, device=dev)])
        layers_h = []
        for L in x["layers"]:   # one layer at a time to the host
            layers_h.append(_host(L))
        del x

        def run():
            for L in layers_h:
                oracle.fill_rows(h, L, sample, cfg.n_kv_heads, cfg.head_dim, cfg.rope_base, cfg.eps)
            return len(sample)
        return run, (f"fill of 16 evenly spaced rows across all {len(layers_h)} layers "
                     "(per-row time extrapolated)")
    if name in ("river-1b", "river-tiny"):
        import dataclasses
        from oracle import river
        cfg = configs.LLAMA1B_RIVER if name == "river-1b" else configs.TINY_RIVER
        if rows or layers:
            cfg = dataclasses.replace(cfg, batch=rows or cfg.batch,
                                      river_layers=cfg.river_layers[:layers] if layers else cfg.river_layers)
        x = gen.river_inputs(cfg, seed, dev)
        L = _host(x["layers"][0])
        L["cache_layer"] = 0
        p = int(x["pos"][0].item())
        j0 = cfg.river_layers[0]
        kc = np.ascontiguousarray(_host(x["k_cache"][j0:j0 + 1, :1, :, :p + 1]))
        vc = np.ascontiguousarray(_host(x["v_cache"][j0:j0 + 1, :1, :, :p + 1]))
        h = _host(x["h"][:1])
        del x
        frac = 1.0 / len(cfg.river_layers)

        def run():
            river.exit_layer(h, L, [p], [0], kc, vc, cfg.n_q_heads, cfg.n_kv_heads, cfg.head_dim, cfg.rope_base,
                             cfg.eps, cfg.group)
            return frac
        return run, (f"one token through one of the {len(cfg.river_layers)} exit layers "
                     f"(position {p}; counted as 1/{len(cfg.river_layers)} token)")
    raise SystemExit(f"unknown workload {name}")


def make(name, tee, dev, seed, rows=None, layers=None):
    if name == "river-1b":
        return River(tee, configs.LLAMA1B_RIVER, dev, seed, rows, layers)
    if name == "river-tiny":
        return River(tee, configs.TINY_RIVER, dev, seed, rows, layers)
    if name == "decode-1b":
        return Decode(tee, configs.LLAMA1B_DECODE, dev, seed)
    if name == "decode-tiny":
        return Decode(tee, configs.TINY_DECODE, dev, seed)
    if name == "ridge-4096":
        return Ridge(tee, dev, seed)
    if name == "router-32":
        return Router(tee, configs.ROUTER_4096, dev, seed, n=32)
    if name == "router-4096":
        return Router(tee, configs.ROUTER_4096, dev, seed)
    if name == "router-65536":
        return Router(tee, configs.ROUTER_4096, dev, seed, n=rows or 65536)
    if name == "prefill-16k":
        return Prefill(tee, configs.PREFILL_16K, dev, seed, rows, layers)
    if name == "prefill-120k":
        return Prefill(tee, configs.PREFILL_120K, dev, seed, rows, layers)
    raise SystemExit(f"unknown workload {name}")


# --------------------------------------------------------------------------- helpers

class Clocks:
    """nvidia-smi samples (every 200 ms) taken during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index, self.proc, self.path = index, None, None

    def start(self):
        try:
            # the raw samples: $TEE_CLOCKS_DIR if set, else the system's temporary folder
            d = os.environ.get("TEE_CLOCKS_DIR") or tempfile.gettempdir()
            os.makedirs(d, exist_ok=True)
            self.path = os.path.join(d, f"clocks_rank{self.index}.csv")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for ln in open(self.path):
            f = [v.strip() for v in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append((float(f[1]), float(f[2]), f[5:9]))
            except ValueError:
                continue
        if not rows:
            return None
        mx = max(r[1] for r in rows)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[2]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": mx, "reasons": reasons,
                "samples": len(rows)}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def max_over_ranks(x: float, world: int, dev) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, world: int, t_ms: float) -> float:
    """Whole-job units/s: every rank processes its own batch (weak scaling), and the
    step time is the slowest rank's."""
    return world * units_per_rank / (t_ms * 1e-3)


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def time_oracle(run, budget_s):
    """Repeat the oracle sample until ``budget_s`` of CPU time; units/s."""
    run()  # warm
    units, t0 = 0, time.perf_counter()
    while True:
        units += run()
        el = time.perf_counter() - t0
        if el >= budget_s:
            return units / el, el


# --------------------------------------------------------------------------- arms

def run_reference(args):
    """The reference arm: the C++ CPU oracle, single-threaded, on a bounded
    sample of the workload. Its inputs come from the seeded generator only
    (drawn on the GPU with torch when one is present, else on the CPU); the
    CUDA library is neither built nor loaded."""
    world, rank, local = dist_env()
    if rank != 0:
        return 0
    dev = torch.device("cuda", local) if torch.cuda.is_available() else torch.device("cpu")
    run, sample = oracle_sample(args.workload, dev, args.seed, args.rows, args.layers)
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    units = 0
    for _ in range(args.steps):
        units += run()
    el = time.perf_counter() - t0
    v = units / el
    line = {"metric": metric_for(args.workload), "value": v,
            "unit": unit_for(args.workload), "n_gpus": 0, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * el / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": reference_config(args.workload, dev, args.seed, args.rows, args.layers),
            "cpu_baseline": {"value": v, "unit": unit_for(args.workload), "cores": 1, "kind": "oracle",
                             "impl": "C++17, single-threaded, float64", "host_cores": os.cpu_count(),
                             "sample": sample},
            "e2e": {"value": v, "unit": unit_for(args.workload), "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def run_gpu(args):
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    import __graft_entry__
    __graft_entry__.build()
    import token_early_exit_gb300 as tee
    from token_early_exit_gb300 import _lib
    lib = _lib.load()

    w = make(args.workload, tee, dev, args.seed + rank, args.rows, args.layers)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    for _ in range(args.warmup):
        w.step()
    torch.cuda.synchronize(dev)
    n_exit = w.n_exit()

    # The step (and, separately, the dominant call) replay as CUDA graphs. Each graph
    # holds the L2 flush, then a timing event, the work, and a second timing event:
    # the events run on the device inside the graph, so the interval is the work
    # alone (kernels and the gaps between them), without the graph's own launch.
    fns, kidx = w.parts()

    def capture(calls):
        a = torch.cuda.Event(enable_timing=True, external=True)
        b = torch.cuda.Event(enable_timing=True, external=True)
        g = torch.cuda.CUDAGraph()
        l0 = lib.tee_launch_count()
        with torch.cuda.graph(g):
            if getattr(w, "flush", True):
                flush.zero_()
            a.record()
            for f in calls:
                f()
            b.record()
        return g, a, b, lib.tee_launch_count() - l0

    g_step, sa, sb, k_step = capture(fns)
    g_kern, ka, kb, k_kern = (capture([fns[kidx]]) if len(fns) > 1 else (None, None, None, 0))
    # the floor of this timing method: one trivial kernel between the same two events
    one = torch.zeros(1, device=dev)
    g_floor, fa, fb, _ = capture([lambda: one.add_(1.0)])
    for _ in range(2):
        g_step.replay()
        if g_kern is not None:
            g_kern.replay()
        g_floor.replay()
    torch.cuda.synchronize(dev)

    clocks = Clocks(dev.index)
    barrier(world)
    torch.cuda.synchronize(dev)
    clocks.start()
    step_ms, kern_ms = [], []
    for i in range(args.steps):
        g_step.replay()
        torch.cuda.synchronize(dev)
        step_ms.append(sa.elapsed_time(sb))
        if g_kern is not None:
            g_kern.replay()
            torch.cuda.synchronize(dev)
            kern_ms.append(ka.elapsed_time(kb))
    launches = args.steps * (k_step + k_kern)
    barrier(world)
    clk = clocks.stop()
    floor_ms = []
    for _ in range(args.steps):
        g_floor.replay()
        torch.cuda.synchronize(dev)
        floor_ms.append(fa.elapsed_time(fb))
    floor_ms = statistics.median(floor_ms)
    if g_kern is None:
        kern_ms = step_ms
    # each kernel of the path as its own call, where the workload lists them
    per_kernel = {}
    for name, call, nbytes in (w.kernels() if hasattr(w, "kernels") else []):
        g1, a1, b1, k1 = capture([call])
        g1.replay()
        torch.cuda.synchronize(dev)
        ts = []
        for _ in range(args.steps):
            g1.replay()
            torch.cuda.synchronize(dev)
            ts.append(a1.elapsed_time(b1))
        km = statistics.median(ts)
        gbs = nbytes / (km * 1e-3) / 1e9
        per_kernel[name] = {"us": km * 1e3, "algorithmic_bytes": nbytes, "GB/s": gbs,
                            "frac": gbs / peaks()["hbm_gbs"], "launches": int(k1),
                            "traffic": traffic(f"{name}/n{w.n}" if hasattr(w, "n") else None)}
    t_step = statistics.mean(step_ms)
    t_step = max_over_ranks(t_step, world, dev)
    value = job_throughput(w.units, world, t_step)

    # end to end: pinned host inputs -> device -> step -> result back to the host, per step
    bi, bo = w.host_io()
    for _ in range(2):
        w.e2e_step()
    torch.cuda.synchronize(dev)
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        w.e2e_step()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    t_e2e = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, dev)

    pk = peaks()
    k_ms = statistics.mean(kern_ms)
    work = w.fill_bytes(n_exit)
    if w.bound == "hbm":
        achieved = work / (k_ms * 1e-3) / 1e9
        peak = pk["hbm_gbs"]
        roof = {"bound": "hbm", "kernel": w.kernel, "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": traffic(w.traffic_key), "algorithmic_bytes": work, "kernel_ms": k_ms,
                "event_floor_ms": floor_ms, "peak_source": pk["source"]}
    else:
        achieved = work / (k_ms * 1e-3) / 1e12
        peak = pk["bf16_tflops_sustained"] if k_ms > 50 else pk["bf16_tflops"]
        roof = {"bound": "tensor", "kernel": w.kernel, "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": traffic(w.traffic_key), "algorithmic_flops": work, "kernel_ms": k_ms,
                "event_floor_ms": floor_ms, "peak_source": pk["source"]}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        run, sample = oracle_sample(args.workload, dev, args.seed, args.rows, args.layers)
        v, el = time_oracle(run, args.cpu_seconds)
        cpu = {"value": v, "unit": unit_for(args.workload), "cores": 1, "kind": "oracle", "impl": "C++17, single-threaded, float64",
               "host_cores": os.cpu_count(), "sample": sample, "seconds": round(el, 2)}

    line = {"metric": getattr(w, "metric", METRIC), "value": value, "unit": unit_for(args.workload), "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": t_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16" if w.config().get("workload") != configs.TINY_DECODE.name else "f32",
            "data": "synthetic", "config": w.config(), "exits_per_step": n_exit,
            "roofline": roof, "cpu_baseline": cpu,
            "e2e": {"value": job_throughput(w.units, world, t_e2e), "unit": unit_for(args.workload), "h2d_bytes_per_step": bi,
                    "d2h_bytes_per_step": bo, "ms_per_step": t_e2e},
            "gpu_launches": int(launches), "launches_per_step": int(k_step), "clocks": clk,
            **({"kernels": per_kernel} if per_kernel else {}),
            "timing": "CUDA-graph replay per step; " + ("L2 flushed inside the graph before the step; "
                                                           if getattr(w, "flush", True) else
                                                           "no flush (every input is larger than L2); ") +
                      "timed by device events recorded inside the graph around the step; roofline.event_floor_ms "
                      "is the same interval around one trivial kernel (part of every kernel_ms)",
            "step_ms": {"median": statistics.median(step_ms), "min": min(step_ms), "max": max(step_ms)}}
    if rank == 0:
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("tee", "reference"), default="tee")
    ap.add_argument("--workload", choices=WORKLOADS, default="decode-1b")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--rows", type=int, default=None,
                    help="prefill workloads: fewer filled rows; router-65536: fewer tokens (profiling)")
    ap.add_argument("--layers", type=int, default=None, help="prefill workloads: fewer filled layers (profiling)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
